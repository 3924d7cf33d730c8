"""GPU parity of attention with run-time termination (ffd_art_attention) against the CPU statement
(oracle/art.py) on the same seeded inputs.

* tau = phi = 0 never terminates: every unit uses block 0 plus every listed block, and the output
  is the softmax over them (max-abs 2e-3, relative L2 1e-3 against fp64).
* Huge thresholds always hold: a unit stops after 1 + patience blocks (or at its last block).
* Thresholds in between: the GPU's fp32 metrics may fall on either side of a threshold that one of
  them lies within a small band of; a unit with no metric in that band before its stop must stop
  exactly where the oracle does. Every unit's output is compared with the oracle stopped after the
  same number of blocks.
"""
import math

import numpy as np
import pytest
import torch

import ffd_synth
import oracle
from oracle import art as ART
import sparse_quantized_attention_gb300 as ffd
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu

DS_BAND = (2e-5, 1e-3)   # d_scale: absolute, relative band around tau
DD_BAND = (1e-7, 1e-3)   # d_direction


def _setup(w, lens=None, scale=1.0):
    inp = ffd_synth.make_inputs(w, seq_lens=lens, signal_scale=scale)
    dev = H.to_device(inp)
    qc = H.quantize(dev)
    return inp, dev, qc, oracle.quantize(inp.k_bits)


def _run(inp, dev, qc, tau, phi, patience, keep=None):
    w = inp.workload
    p = H.params_for(inp, 5.0)
    ws = ffd.alloc_art_workspace(p)
    out = torch.full((w.batch, w.num_q_heads, 128), float("nan"), device="cuda")
    used = torch.full((w.batch, w.num_kv_heads), -1, dtype=torch.int32, device="cuda")
    keep_t = None if keep is None else torch.from_numpy(keep).cuda()
    ffd.ffd_art_attention(p, tau, phi, patience, dev["q"], qc, dev["v"], dev["seq_lens"],
                          dev["block_table"], out, ws, keep_in=keep_t, blocks_used=used)
    assert ffd.ffd_get_error(ws) == 0
    return out.cpu().numpy().astype(np.float64), used.cpu().numpy()


def _oracle(inp, qk, b, h, keep_row, tau, phi, patience, stop_after=None):
    w = inp.workload
    G = w.num_q_heads // w.num_kv_heads
    n = int(inp.seq_lens[b])
    nb = (n + 63) // 64
    kr = np.ones(nb, np.uint8) if keep_row is None else keep_row[:nb]
    return ART.art_unit(inp.q_bits[b, h * G:(h + 1) * G], n, inp.block_table[b], qk, inp.v_bits,
                        h, kr, H.SM, tau, phi, patience, stop_after=stop_after), kr


def _close(got, want):
    err = np.abs(got - want).max() if want.size else 0.0
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)
    assert err <= H.OUT_MAX_ABS and (rel <= H.OUT_REL_L2 or np.linalg.norm(want) == 0), (err, rel)


def _random_keep(inp, seed, frac=0.4):
    w = inp.workload
    rng = np.random.default_rng(seed)
    return (rng.random((w.batch, w.num_kv_heads, inp.max_blocks)) < frac).astype(np.uint8)


CASES = {
    # name: (workload, seq_lens, signal scale). The literal scale spreads the attention, so the
    # metrics are of order 1e-2 and thresholds between them are well conditioned; the peaked
    # scale concentrates it on a few tokens (metrics near 1e-5 and 1e-9, below fp32 resolution
    # of a threshold), so that case only runs the tests that do not place thresholds.
    "qwen-shape-4k": (ffd_synth.custom(1, 28, 4, 4000, seed=51), None, 1.0),
    "qwen-shape-4k-peaked": (ffd_synth.custom(1, 28, 4, 4000, seed=51), None,
                             ffd_synth.peaked_scale()),
    "ragged-g8": (ffd_synth.custom(4, 16, 2, 700, seed=52), [700, 129, 1, 0], 1.0),
    "g1-random-pages": (ffd_synth.custom(2, 4, 4, 2000, random_pages=True, seed=53),
                        [2000, 1337], 1.0),
}


@pytest.fixture(scope="module", params=sorted(CASES))
def case(request):
    w, lens, scale = CASES[request.param]
    return _setup(w, lens, scale) + (scale != 1.0,)


@pytest.mark.parametrize("masked", [False, True])
def test_without_termination_uses_every_listed_block(case, masked):
    inp, dev, qc, qk, _ = case
    w = inp.workload
    G = w.num_q_heads // w.num_kv_heads
    keep = _random_keep(inp, 5) if masked else None
    out, used = _run(inp, dev, qc, 0.0, 0.0, 1, keep)
    for b in range(w.batch):
        for h in range(w.num_kv_heads):
            res, kr = _oracle(inp, qk, b, h, None if keep is None else keep[b, h], 0.0, 0.0, 1)
            nb = (int(inp.seq_lens[b]) + 63) // 64
            assert used[b, h] == len(ART.art_order(nb, kr)) == res.used
            _close(out[b, h * G:(h + 1) * G], res.out)


@pytest.mark.parametrize("patience", [1, 2, 3])
def test_huge_thresholds_stop_after_patience(case, patience):
    """Stops after 1 + patience blocks: the second block of a pair the sequencer takes together
    (patience 1, 3) and the first one (patience 2)."""
    inp, dev, qc, qk, _ = case
    w = inp.workload
    G = w.num_q_heads // w.num_kv_heads
    out, used = _run(inp, dev, qc, 1e30, 1e30, patience)
    for b in range(w.batch):
        nb = (int(inp.seq_lens[b]) + 63) // 64
        for h in range(w.num_kv_heads):
            assert used[b, h] == min(nb, 1 + patience)
            res, _ = _oracle(inp, qk, b, h, None, 1e30, 1e30, patience)
            assert res.used == used[b, h]
            _close(out[b, h * G:(h + 1) * G], res.out)


def _ambiguous(res, tau, phi):
    """True when a metric up to the oracle's stop lies within the band of its threshold."""
    for ds, dd in zip(res.d_scale, res.d_dir):
        if abs(ds - tau) <= DS_BAND[0] + DS_BAND[1] * tau:
            return True
        if abs(dd - phi) <= DD_BAND[0] + DD_BAND[1] * phi:
            return True
    return False


@pytest.mark.parametrize("q", [0.3, 0.6])
@pytest.mark.parametrize("patience", [1, 2])
def test_thresholds_stop_where_the_oracle_stops(case, q, patience):
    inp, dev, qc, qk, peaked = case
    if peaked:
        pytest.skip("thresholds below fp32 resolution of the metrics")
    w = inp.workload
    G = w.num_q_heads // w.num_kv_heads
    keep = _random_keep(inp, 9, frac=0.6)
    # thresholds at quantiles of the first unit with enough blocks
    full = None
    for b in range(w.batch):
        full, _ = _oracle(inp, qk, b, 0, keep[b, 0], 0.0, 0.0, 1)
        if len(full.d_scale) >= 4:
            break
    if full is None or len(full.d_scale) < 4:
        pytest.skip("no unit with enough blocks")
    def between(vals):  # midway between the two metrics around quantile q
        s = np.sort(np.asarray(vals))
        k = min(max(int(q * len(s)), 1), len(s) - 1)
        return float(0.5 * (s[k - 1] + s[k]))
    tau, phi = between(full.d_scale), between(full.d_dir)
    out, used = _run(inp, dev, qc, tau, phi, patience, keep)
    exact = 0
    for b in range(w.batch):
        for h in range(w.num_kv_heads):
            res, _ = _oracle(inp, qk, b, h, keep[b, h], tau, phi, patience)
            if not _ambiguous(res, tau, phi):
                assert used[b, h] == res.used, (b, h)
                exact += 1
            at, _ = _oracle(inp, qk, b, h, keep[b, h], tau, phi, patience,
                            stop_after=int(used[b, h]))
            assert at.used == used[b, h]
            _close(out[b, h * G:(h + 1) * G], at.out)
    assert exact >= 1


def test_bad_block_table_entry_raises_and_contributes_nothing():
    """A block-table entry outside [0, P) sets the bounds bit; that block adds nothing and still
    counts as visited; the other blocks give the softmax over themselves."""
    w = ffd_synth.custom(1, 8, 2, 1000, seed=57)
    inp, dev, qc, qk = _setup(w)
    G = w.num_q_heads // w.num_kv_heads
    nb = (int(inp.seq_lens[0]) + 63) // 64
    bad = 5
    bt = dev["block_table"].clone()
    bt[0, bad] = inp.num_pages  # one past the last page
    p = H.params_for(inp, 5.0)
    ws = ffd.alloc_art_workspace(p)
    out = torch.zeros((1, w.num_q_heads, 128), device="cuda")
    used = torch.zeros((1, w.num_kv_heads), dtype=torch.int32, device="cuda")
    ffd.ffd_art_attention(p, 0.0, 0.0, 1, dev["q"], qc, dev["v"], dev["seq_lens"], bt, out, ws,
                          blocks_used=used)
    assert ffd.ffd_get_error(ws) == 5  # FFD_ERR_BOUNDS
    got = out.cpu().numpy().astype(np.float64)
    keep = np.ones(nb, np.uint8)
    keep[bad] = 0
    for h in range(w.num_kv_heads):
        assert used[0, h] == nb
        res, _ = _oracle(inp, qk, 0, h, keep, 0.0, 0.0, 1)
        _close(got[0, h * G:(h + 1) * G], res.out)


@pytest.fixture(scope="module")
def full_size():
    """The 128K Qwen2.5-7B-shaped workload (batch 4, 28/4 heads), peaked, with the Top-delta mask
    of the decode step as ART's block list: the launch the benchmark's ART rows time."""
    w = ffd_synth.WORKLOADS[2]
    inp = ffd_synth.make_inputs(w, signal_scale=ffd_synth.peaked_scale())
    dev = H.to_device(inp)
    qc = H.quantize(dev)
    mask = H.decode(inp, dev, qc, 5.0)["mask"]
    yield inp, dev, qc, oracle.quantize(inp.k_bits), mask
    del dev, qc
    torch.cuda.empty_cache()


@pytest.mark.parametrize("tau,phi,patience", [(0.0, 0.0, 1), (1e-2, 1e-3, 2)])
def test_full_size_sampled_units(full_size, tau, phi, patience):
    inp, dev, qc, qk, mask = full_size
    w = inp.workload
    G = w.num_q_heads // w.num_kv_heads
    out, used = _run(inp, dev, qc, tau, phi, patience, mask)
    # sampled units: the one that keeps the most blocks, and two fixed ones
    kept = mask.reshape(w.batch * w.num_kv_heads, -1).sum(axis=1)
    units = sorted({int(np.argmax(kept)), 0, w.batch * w.num_kv_heads - 1})
    for u in units:
        b, h = divmod(u, w.num_kv_heads)
        res, kr = _oracle(inp, qk, b, h, mask[b, h], tau, phi, patience)
        if tau == 0.0:
            nb = (int(inp.seq_lens[b]) + 63) // 64
            assert used[b, h] == len(ART.art_order(nb, kr)) == res.used
        elif not _ambiguous(res, tau, phi):
            assert used[b, h] == res.used, (b, h)
        at, _ = _oracle(inp, qk, b, h, mask[b, h], tau, phi, patience, stop_after=int(used[b, h]))
        _close(out[b, h * G:(h + 1) * G], at.out)


def test_closed_form_metrics_decide_the_stop():
    """Identical keys give equal weights, so the probe is the mean of the V rows seen. Order:
    block 0 (V = 2 e1), block 2 (V = 3 e2), block 1 (V = 3 e2). After the second block P = e1 +
    1.5 e2 with d_scale = | |P| - 2 | / 2 and d_direction = 1 - 1 / |P|; thresholds just above
    both stop there (patience 1), just below them the unit runs to its end."""
    def bf(x):
        return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).cuda()
    k = np.zeros((3, 1, 64, 128), np.float32) + 0.25
    v = np.zeros((3, 1, 64, 128), np.float32)
    v[0, 0, :, 0] = 2.0
    v[1:, 0, :, 1] = 3.0
    q = np.random.default_rng(6).standard_normal((1, 2, 128)).astype(np.float32)
    kd, vd, qd = bf(k), bf(v), bf(q)
    qc = ffd.alloc_quantized_cache(3, 1)
    ffd.ffd_quantize_keys(kd, qc)
    sl = torch.tensor([192], dtype=torch.int32, device="cuda")
    bt = torch.tensor([[0, 1, 2]], dtype=torch.int32, device="cuda")
    p = ffd.make_params(1, 2, 1, 3, 3, sink=16, local=64, delta=5.0, sm_scale=H.SM)
    n2 = math.sqrt(1.0 + 1.5 ** 2)
    ds, dd = abs(n2 - 2.0) / 2.0, 1.0 - 1.0 / n2
    for scale, want_used in ((1.001, 2), (0.999, 3)):
        ws = ffd.alloc_art_workspace(p)
        out = torch.zeros((1, 2, 128), device="cuda")
        used = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
        ffd.ffd_art_attention(p, ds * scale, dd * scale, 1, qd, qc, vd, sl, bt, out, ws,
                              blocks_used=used)
        assert ffd.ffd_get_error(ws) == 0
        assert int(used[0, 0]) == want_used
        got = out.cpu().numpy()
        want = np.zeros(128)
        if want_used == 2:
            want[0], want[1] = 1.0, 1.5
        else:
            want[0], want[1] = 2.0 / 3.0, 2.0
        np.testing.assert_allclose(got[0], np.stack([want, want]), rtol=0, atol=1e-5)
