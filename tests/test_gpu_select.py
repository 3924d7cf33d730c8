"""GPU parity of the comparison selectors (Top-k, Top-p) and of the decode over a given mask.

The masks come from ffd_select_blocks and are compared with the oracle's selection
(oracle/selectors.py) on the oracle's fp64 thumbnail scores. The GPU scores are fp32, so a block
whose decision sits within a small band of the rule's cut may go either way (see _topk_check and
_topp_check); every other block must match. The attention over a mask is compared with the oracle
run on the GPU's own mask.
"""
import numpy as np
import pytest
import torch

import ffd_synth
import oracle
from oracle import selectors as SEL
import sparse_quantized_attention_gb300 as ffd
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu

SCORE_BAND = 1e-4   # fp32 vs fp64 provisional scores (128-term dot products of values < 2^8)
MASS_BAND = 1e-4    # cumulative softmax mass


def _setup(w, lens=None, scale=1.0):
    inp = ffd_synth.make_inputs(w, seq_lens=lens, signal_scale=scale)
    dev = H.to_device(inp)
    qc = H.quantize(dev)
    qk = oracle.quantize(inp.k_bits)
    ref = oracle.decode(inp.q_bits, inp.seq_lens, inp.block_table, qk, inp.v_bits,
                        sink=w.sink, local=w.local, delta=5.0, sm_scale=H.SM, want_s_hat=True)
    return inp, dev, qc, qk, ref


def _select(inp, dev, qc, selector, budget):
    w = inp.workload
    p = H.params_for(inp, 5.0)
    ws = ffd.alloc_select_workspace(p)
    mask = torch.full((w.batch, w.num_kv_heads, inp.max_blocks), 7, dtype=torch.uint8,
                      device="cuda")
    ffd.ffd_select_blocks(p, selector, budget, dev["q"], qc, dev["seq_lens"],
                          dev["block_table"], mask, ws)
    assert ffd.ffd_get_error(ws) == 0
    return mask.cpu().numpy()


def _topk_check(s_hat, n, w, k, got):
    want, imp = SEL.select_topk(s_hat, n, w.sink, w.local, k)
    forced = SEL.forced_blocks(n, w.sink, w.local)
    assert np.all(got[forced] == 1)
    elig = np.nonzero(~forced)[0]
    kk = min(k, len(elig))
    assert int(got[elig].sum()) == kk, "Top-k keeps exactly k non-forced blocks"
    if 0 < kk < len(elig):
        kth = np.sort(imp[elig])[::-1][kk - 1]
        clear = np.abs(imp[elig] - kth) > SCORE_BAND * max(1.0, abs(kth))
        assert np.array_equal(got[elig][clear], want[elig][clear])
    else:
        assert np.array_equal(got, want)
    return int((got != want).sum())


def _topp_check(s_hat, n, w, p, got):
    want, mass, before = SEL.select_topp(s_hat, n, w.sink, w.local, p)
    forced = SEL.forced_blocks(n, w.sink, w.local)
    G, nb = mass.shape
    clear_keep = forced.copy()
    ambiguous = np.zeros(nb, bool)
    for i in range(G):
        kept = before[i] < p
        amb = np.abs(before[i] - p) <= MASS_BAND
        # nearly equal masses on both sides of the cut may trade places
        tol = MASS_BAND * mass[i] + 1e-9
        for c in np.nonzero(kept)[0]:
            close = np.abs(mass[i] - mass[i, c]) <= np.maximum(tol, tol[c])
            if np.any(close & ~kept):
                amb[c] = True
                amb |= close & ~kept
        clear_keep |= kept & ~amb
        ambiguous |= amb
    must_drop = ~clear_keep & ~ambiguous
    assert np.all(got[clear_keep] == 1), "a clearly selected block was dropped"
    assert np.all(got[must_drop] == 0), "a clearly unselected block was kept"
    return int((got != want).sum())


CASES = [
    ("tiny-4k", lambda: (ffd_synth.WORKLOADS[0], None, 1.0)),
    ("tiny-4k-peaked", lambda: (ffd_synth.WORKLOADS[0], None, ffd_synth.peaked_scale())),
    ("ragged-paged-g7", lambda: (ffd_synth.custom(3, 14, 2, 6000, sink=16, local=200,
                                                  random_pages=True, seed=21),
                                 [6000, 1, 2500], ffd_synth.peaked_scale())),
    ("llama-32k-peaked", lambda: (ffd_synth.WORKLOADS[1], None, ffd_synth.peaked_scale())),
    ("batched-paged-peaked", lambda: (ffd_synth.WORKLOADS[4], None, ffd_synth.peaked_scale())),
    # the workload and inputs the benchmark's selector rows time
    ("qwen-128k-peaked", lambda: (ffd_synth.WORKLOADS[2], None, ffd_synth.peaked_scale())),
]


@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
def test_selector_masks_and_masked_attention(name, make):
    w, lens, scale = make()
    inp, dev, qc, qk, ref = _setup(w, lens, scale)
    p = H.params_for(inp, 5.0)
    stats = []
    for selector, budget in [(ffd.SELECT_TOPK, 0), (ffd.SELECT_TOPK, 3), (ffd.SELECT_TOPK, 17),
                             (ffd.SELECT_TOPK, 1 << 20), (ffd.SELECT_TOPP, 0.5),
                             (ffd.SELECT_TOPP, 0.9), (ffd.SELECT_TOPP, 0.99),
                             (ffd.SELECT_TOPP, 1.0)]:
        got = _select(inp, dev, qc, selector, budget)
        diffs = 0
        for (b, h), s_hat in ref.s_hat.items():
            n = int(inp.seq_lens[b])
            nb = (n + 63) // 64
            assert np.all(got[b, h, nb:] == 0)
            if n == 0:
                continue
            if selector == ffd.SELECT_TOPK:
                diffs += _topk_check(s_hat, n, w, int(budget), got[b, h, :nb])
            else:
                diffs += _topp_check(s_hat, n, w, budget, got[b, h, :nb])
        stats.append((selector, budget, int(got.sum()), diffs))
        # attention over the GPU's mask, against the oracle on the same mask
        out = torch.empty((w.batch, w.num_q_heads, 128), dtype=torch.float32, device="cuda")
        used = torch.zeros_like(torch.from_numpy(got)).cuda()
        ws = ffd.alloc_workspace(p)
        ffd.ffd_decode_attention_masked(p, dev["q"], qc, dev["v"], dev["seq_lens"],
                                        dev["block_table"], torch.from_numpy(got).cuda(), out,
                                        ws, keep_mask=used)
        assert ffd.ffd_get_error(ws) == 0
        assert np.array_equal(used.cpu().numpy(), got)
        want = oracle.decode(inp.q_bits, inp.seq_lens, inp.block_table, qk, inp.v_bits,
                             sink=w.sink, local=w.local, delta=5.0, sm_scale=H.SM, mask_in=got)
        H.compare_outputs(out.cpu().numpy(), want.out, f"{name} selector {selector} {budget}")
    print(name, stats)


def test_masked_decode_with_the_top_delta_mask_repeats_the_step():
    """Given the mask the Top-delta step chose, the masked decode produces the same output bit
    for bit (the same blocks through the same refinement)."""
    w = ffd_synth.custom(2, 28, 4, 9000, sink=64, local=1024, random_pages=True, seed=22)
    inp = ffd_synth.make_inputs(w, seq_lens=[9000, 3333], signal_scale=ffd_synth.peaked_scale())
    dev = H.to_device(inp)
    qc = H.quantize(dev)
    step = H.decode(inp, dev, qc, 5.0)
    assert step["err"] == 0
    p = H.params_for(inp, 5.0)
    out = torch.empty((w.batch, w.num_q_heads, 128), dtype=torch.float32, device="cuda")
    mt = torch.empty((w.batch, w.num_q_heads), dtype=torch.float32, device="cuda")
    ws = ffd.alloc_workspace(p)
    ffd.ffd_decode_attention_masked(p, dev["q"], qc, dev["v"], dev["seq_lens"],
                                    dev["block_table"], torch.from_numpy(step["mask"]).cuda(),
                                    out, ws, m_tilde=mt)
    assert ffd.ffd_get_error(ws) == 0
    assert np.array_equal(out.cpu().numpy(), step["out"])
    assert np.array_equal(mt.cpu().numpy(), step["m_tilde"])


def test_masked_decode_with_an_empty_mask_gives_zero():
    w = ffd_synth.custom(2, 8, 2, 700, sink=16, local=64, seed=23)
    inp = ffd_synth.make_inputs(w, seq_lens=[700, 130])
    dev = H.to_device(inp)
    qc = H.quantize(dev)
    p = H.params_for(inp, 5.0)
    keep = np.zeros((w.batch, w.num_kv_heads, inp.max_blocks), np.uint8)
    keep[1, 1, 2] = 1  # one block of one unit
    out = torch.full((w.batch, w.num_q_heads, 128), float("nan"), device="cuda")
    ws = ffd.alloc_workspace(p)
    ffd.ffd_decode_attention_masked(p, dev["q"], qc, dev["v"], dev["seq_lens"],
                                    dev["block_table"], torch.from_numpy(keep).cuda(), out, ws)
    assert ffd.ffd_get_error(ws) == 0
    got = out.cpu().numpy()
    assert np.all(got[0] == 0) and np.all(got[1, :4] == 0)
    want = oracle.decode(inp.q_bits, inp.seq_lens, inp.block_table, oracle.quantize(inp.k_bits),
                         inp.v_bits, sink=w.sink, local=w.local, delta=5.0, sm_scale=H.SM,
                         mask_in=keep)
    H.compare_outputs(got, want.out, "one kept block")
