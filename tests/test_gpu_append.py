"""Append-time quantisation (ffd_append_kv) and the CUDA-graph-captured decode step.

The appended token's records must be bit for bit what quantising the whole cache gives (the
oracle's quantiser on the full keys); its value and raw key rows must land in the right page row.
The graph test captures append + decode once and replays it over several generated tokens,
comparing every replay with the same calls made eagerly and with the oracle.
"""
import dataclasses

import numpy as np
import pytest
import torch

import ffd_synth
import oracle
import sparse_quantized_attention_gb300 as ffd
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu


def _rows(inp, positions):
    """(page, row) of token positions[b] of every sequence b."""
    bt = inp.block_table
    return [(int(bt[b, p // 64]), p % 64) for b, p in enumerate(positions)]


def _new_tokens(bits, rows, Hkv):
    """bf16 bits [B, Hkv, 128] of the cache rows named by rows."""
    return np.stack([bits[pg, :, r, :] for pg, r in rows]).reshape(len(rows), Hkv, 128)


def _blank_rows(bits, rows, rng):
    """A copy of the cache with the named rows overwritten by unrelated values."""
    out = bits.copy()
    for pg, r in rows:
        noise = torch.from_numpy(rng.standard_normal(out[pg, :, r, :].shape).astype(np.float32) * 9)
        out[pg, :, r, :] = noise.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return out


APPEND_CASES = [
    ("tiny-4k", lambda: (ffd_synth.WORKLOADS[0], None)),
    ("ragged-paged-g7", lambda: (ffd_synth.custom(3, 14, 2, 3000, sink=16, local=200,
                                                  random_pages=True, seed=11), [3000, 1, 1729])),
    ("page-boundary", lambda: (ffd_synth.custom(2, 8, 2, 4096, sink=64, local=256,
                                                random_pages=True, seed=12), [65, 4096])),
    ("batched-paged-32x", lambda: (ffd_synth.WORKLOADS[4], None)),
]


@pytest.mark.parametrize("name,make", APPEND_CASES, ids=[c[0] for c in APPEND_CASES])
def test_append_matches_whole_cache_quantisation(name, make):
    w, lens = make()
    inp = ffd_synth.make_inputs(w, seq_lens=lens)
    Hkv = w.num_kv_heads
    pos = [int(n) - 1 for n in inp.seq_lens]
    rows = _rows(inp, pos)
    rng = np.random.default_rng(1)
    k_old = _blank_rows(inp.k_bits, rows, rng)
    v_old = _blank_rows(inp.v_bits, rows, rng)
    k_dev = H.bits_to_bf16(k_old)
    v_dev = H.bits_to_bf16(v_old)
    qc = ffd.alloc_quantized_cache(inp.num_pages, Hkv)
    ffd.ffd_quantize_keys(k_dev, qc)
    k_new = H.bits_to_bf16(_new_tokens(inp.k_bits, rows, Hkv))
    v_new = H.bits_to_bf16(_new_tokens(inp.v_bits, rows, Hkv))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    positions = torch.tensor(pos, dtype=torch.int32, device="cuda")
    bt = torch.from_numpy(inp.block_table).cuda()
    ffd.ffd_append_kv(k_new, v_new, positions, bt, qc, v_dev, k_cache=k_dev, error_word=err)
    assert ffd.ffd_get_error(err) == 0
    ref = oracle.quantize(inp.k_bits)
    H.assert_cache_equal(H.cache_to_host(qc), ref)
    assert np.array_equal(v_dev.view(torch.int16).cpu().numpy().view(np.uint16), inp.v_bits)
    assert np.array_equal(k_dev.view(torch.int16).cpu().numpy().view(np.uint16), inp.k_bits)
    # the step that follows the append sees the new token
    dev = H.to_device(inp)
    dev["v"] = v_dev
    got = H.decode(inp, dev, qc, 5.0)
    H.check_decode(inp, ref, got, 5.0, what=f"{name} after append")


def test_append_skips_and_reports_bad_rows():
    w = ffd_synth.custom(3, 8, 2, 1000, sink=16, local=64, random_pages=True, seed=13)
    inp = ffd_synth.make_inputs(w)
    Hkv = w.num_kv_heads
    k_dev = H.bits_to_bf16(inp.k_bits)
    v_dev = H.bits_to_bf16(inp.v_bits)
    qc = ffd.alloc_quantized_cache(inp.num_pages, Hkv)
    ffd.ffd_quantize_keys(k_dev, qc)
    before = [t.clone() for t in qc] + [v_dev.clone()]
    k_new = torch.randn((3, Hkv, 128), device="cuda").to(torch.bfloat16)
    v_new = torch.randn((3, Hkv, 128), device="cuda").to(torch.bfloat16)
    bt = torch.from_numpy(inp.block_table).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def unchanged():
        return all(torch.equal(a, b) for a, b in zip(before, list(qc) + [v_dev]))

    # negative positions: nothing appended, nothing reported
    ffd.ffd_append_kv(k_new, v_new, torch.full((3,), -1, dtype=torch.int32, device="cuda"), bt,
                      qc, v_dev, error_word=err)
    assert ffd.ffd_get_error(err) == 0 and unchanged()
    # a position past the block table's row
    past = torch.tensor([-1, 64 * inp.max_blocks, -1], dtype=torch.int32, device="cuda")
    ffd.ffd_append_kv(k_new, v_new, past, bt, qc, v_dev, error_word=err)
    assert ffd.ffd_get_error(err) == 5 and unchanged()
    # a block-table entry outside the page pool
    bt2 = bt.clone()
    bt2[2, 3] = inp.num_pages + 7
    ffd.ffd_append_kv(k_new, v_new, torch.tensor([-1, -1, 3 * 64 + 5], dtype=torch.int32,
                                                 device="cuda"), bt2, qc, v_dev, error_word=err)
    assert ffd.ffd_get_error(err) == 5 and unchanged()
    # a key outside the fp16 range is written and reported
    k_bad = k_new.clone()
    k_bad[0, 1, 9] = 1.0e6
    ffd.ffd_append_kv(k_bad, v_new, torch.tensor([999, -1, -1], dtype=torch.int32,
                                                 device="cuda"), bt, qc, v_dev, error_word=err)
    assert ffd.ffd_get_error(err) == 6


def test_graph_captured_append_and_decode_step():
    """Append + decode captured once in a CUDA graph and replayed for several generated tokens:
    every replay equals the eager calls bit for bit, and the oracle within tolerance."""
    w = ffd_synth.custom(3, 14, 2, 5000, sink=64, local=512, random_pages=True, seed=14)
    steps = 3
    lens = [5000, 1200, 64 * 20]
    inp = ffd_synth.make_inputs(w, seq_lens=[n + steps for n in lens])
    Hkv, B = w.num_kv_heads, w.batch
    final_rows = [_rows(inp, [n + t for n in lens]) for t in range(steps)]
    rng = np.random.default_rng(2)
    blank = [r for rows in final_rows for r in rows]
    k_dev = H.bits_to_bf16(_blank_rows(inp.k_bits, blank, rng))
    v_dev = H.bits_to_bf16(_blank_rows(inp.v_bits, blank, rng))
    qc = ffd.alloc_quantized_cache(inp.num_pages, Hkv)
    ffd.ffd_quantize_keys(k_dev, qc)
    bt = torch.from_numpy(inp.block_table).cuda()
    q = H.bits_to_bf16(inp.q_bits)
    p = H.params_for(inp, 5.0)
    # buffers the graph reads: refilled before every replay
    k_new = torch.empty((B, Hkv, 128), dtype=torch.bfloat16, device="cuda")
    v_new = torch.empty_like(k_new)
    positions = torch.empty(B, dtype=torch.int32, device="cuda")
    seq_lens = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty((B, w.num_q_heads, 128), dtype=torch.float32, device="cuda")
    mask = torch.zeros((B, Hkv, inp.max_blocks), dtype=torch.uint8, device="cuda")
    ws = ffd.alloc_workspace(p)
    # the eager twin: its own cache copies, the same calls
    qc_e = ffd.QuantizedCache(qc.thumb.clone(), qc.resid.clone())
    v_e = v_dev.clone()
    out_e = torch.empty_like(out)
    mask_e = torch.zeros_like(mask)
    ws_e = ffd.alloc_workspace(p)

    def step(cache, vcache, o, m, wsp):
        ffd.ffd_append_kv(k_new, v_new, positions, bt, cache, vcache)
        ffd.ffd_decode_attention(p, q, cache, vcache, seq_lens, bt, o, wsp, keep_mask=m)

    def fill(t):
        rows = final_rows[t]
        k_new.copy_(H.bits_to_bf16(_new_tokens(inp.k_bits, rows, Hkv)))
        v_new.copy_(H.bits_to_bf16(_new_tokens(inp.v_bits, rows, Hkv)))
        positions.copy_(torch.tensor([n + t for n in lens], dtype=torch.int32))
        seq_lens.copy_(torch.tensor([n + t + 1 for n in lens], dtype=torch.int32))

    fill(0)
    step(qc, v_dev, out, mask, ws)  # first calls outside capture (one-time set-up)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(qc, v_dev, out, mask, ws)
    ref_q = oracle.quantize(inp.k_bits)
    for t in range(steps):
        fill(t)
        graph.replay()
        step(qc_e, v_e, out_e, mask_e, ws_e)
        torch.cuda.synchronize()
        assert ffd.ffd_get_error(ws) == 0 and ffd.ffd_get_error(ws_e) == 0
        assert torch.equal(out, out_e), f"replay {t}: output differs from the eager step"
        assert torch.equal(mask, mask_e), f"replay {t}: mask differs from the eager step"
        step_inp = dataclasses.replace(inp, seq_lens=np.array([n + t + 1 for n in lens],
                                                              dtype=np.int32))
        got = {"out": out.cpu().numpy(), "mask": mask.cpu().numpy(),
               "m_tilde": np.full((B, w.num_q_heads), np.nan, np.float32), "err": 0}
        H.check_decode(step_inp, ref_q, dict(got, m_tilde=_m_tilde(step_inp, qc, v_dev)),
                       5.0, what=f"graph replay {t}")


def _m_tilde(inp, qc, v_dev):
    """m~ of one eager decode (the graph does not ask for it)."""
    dev = H.to_device(inp)
    dev["v"] = v_dev
    return H.decode(inp, dev, qc, 5.0)["m_tilde"]
