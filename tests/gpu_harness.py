"""Glue for the GPU parity tests: move seeded inputs to the device, call the CUDA library through
its C ABI binding, and compare with the CPU oracle on the same bytes.

Tolerances (from the library's parity contract):
  * codes, residuals and scales: bit-exact;
  * block masks: bit-exact except blocks whose best provisional score lies within 1e-4 of
    m~ - delta (either answer is correct there);
  * outputs: max-abs error <= 2e-3 and relative L2 error <= 1e-3 against the fp64 oracle run with
    the GPU's own mask (so a legitimately different borderline block is compared like for like).
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import sparse_quantized_attention_gb300 as ffd

SM = float(np.float32(1.0 / math.sqrt(128.0)))
MASK_BAND = 1e-4
OUT_MAX_ABS = 2e-3
OUT_REL_L2 = 1e-3


def bits_to_bf16(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def to_device(inp, device="cuda") -> dict:
    return {
        "q": bits_to_bf16(inp.q_bits, device),
        "k": bits_to_bf16(inp.k_bits, device),
        "v": bits_to_bf16(inp.v_bits, device),
        "seq_lens": torch.from_numpy(inp.seq_lens).to(device),
        "block_table": torch.from_numpy(inp.block_table).to(device),
    }


def quantize(dev: dict) -> ffd.QuantizedCache:
    P, Hkv = dev["k"].shape[0], dev["k"].shape[1]
    qc = ffd.alloc_quantized_cache(P, Hkv, device=dev["k"].device)
    err = torch.zeros(1, dtype=torch.int32, device=dev["k"].device)
    ffd.ffd_quantize_keys(dev["k"], qc, error_word=err)
    assert ffd.ffd_get_error(err) == 0
    return qc


def cache_to_host(qc: ffd.QuantizedCache) -> oracle.QuantizedKeys:
    """Unpack the library's (page, KV head) records into the method's arrays (record layout in
    include/ffd.h; the residual codes' 16-byte chunk j of token r is stored at j ^ (r % 8))."""
    th = qc.thumb.cpu().numpy()
    rr = qc.resid.cpu().numpy()
    P, Hkv = th.shape[:2]
    rows = np.arange(64)[:, None]
    chunks = np.arange(8)[None, :] ^ (rows % 8)
    stored = rr[..., :8192].reshape(P, Hkv, 64, 8, 16)
    return oracle.QuantizedKeys(
        thumb=np.ascontiguousarray(th[..., :2048]).reshape(P, Hkv, 64, 32),
        t_scale=np.ascontiguousarray(th[..., 2048:2560]).view(np.uint16).reshape(P, Hkv, 64, 4),
        t_zero=np.ascontiguousarray(th[..., 2560:3072]).view(np.uint16).reshape(P, Hkv, 64, 4),
        resid=np.ascontiguousarray(stored[:, :, rows, chunks, :]).reshape(P, Hkv, 64, 128)
        .view(np.int8),
        r_scale=np.ascontiguousarray(rr[..., 8192:]).view(np.uint16).reshape(P, Hkv, 64, 4))


def assert_cache_equal(gpu: oracle.QuantizedKeys, ref: oracle.QuantizedKeys):
    for name in ("thumb", "t_scale", "t_zero", "resid", "r_scale"):
        a, b = getattr(gpu, name), getattr(ref, name)
        if not np.array_equal(a, b):
            bad = np.argwhere(a != b)
            raise AssertionError(f"{name}: {len(bad)} mismatches, first at {bad[0].tolist()}: "
                                 f"gpu {a[tuple(bad[0])]} oracle {b[tuple(bad[0])]}")


def params_for(inp, delta, num_splits=0, schedule=0):
    w = inp.workload
    return ffd.make_params(w.batch, w.num_q_heads, w.num_kv_heads, inp.num_pages,
                           inp.max_blocks, sink=w.sink, local=w.local, delta=delta,
                           sm_scale=SM, num_splits=num_splits, schedule=schedule)


def decode(inp, dev, qc, delta, num_splits=0, schedule=0) -> dict:
    w = inp.workload
    p = params_for(inp, delta, num_splits, schedule)
    d = dev["q"].device
    out = torch.empty((w.batch, w.num_q_heads, 128), dtype=torch.float32, device=d)
    mask = torch.full((w.batch, w.num_kv_heads, inp.max_blocks), 7, dtype=torch.uint8, device=d)
    mt = torch.empty((w.batch, w.num_q_heads), dtype=torch.float32, device=d)
    ws = ffd.alloc_workspace(p, device=d)
    ffd.ffd_decode_attention(p, dev["q"], qc, dev["v"], dev["seq_lens"], dev["block_table"],
                             out, ws, keep_mask=mask, m_tilde=mt)
    err = ffd.ffd_get_error(ws)
    return {"out": out.cpu().numpy(), "mask": mask.cpu().numpy(), "m_tilde": mt.cpu().numpy(),
            "err": err}


def dense(inp, dev, num_splits=0) -> np.ndarray:
    w = inp.workload
    p = params_for(inp, 5.0, num_splits)
    out = torch.empty((w.batch, w.num_q_heads, 128), dtype=torch.float32, device=dev["q"].device)
    ws = ffd.alloc_workspace(p, dense=True, device=dev["q"].device)
    ffd.ffd_dense_decode(p, dev["q"], dev["k"], dev["v"], dev["seq_lens"], dev["block_table"],
                         out, ws)
    assert ffd.ffd_get_error(ws) == 0
    return out.cpu().numpy()


def compare_outputs(gpu_out: np.ndarray, ref_out: np.ndarray, what: str) -> dict:
    diff = np.abs(gpu_out.astype(np.float64) - ref_out)
    max_abs = float(diff.max()) if diff.size else 0.0
    denom = float(np.linalg.norm(ref_out))
    rel = float(np.linalg.norm(gpu_out.astype(np.float64) - ref_out)) / denom if denom else 0.0
    assert max_abs <= OUT_MAX_ABS, f"{what}: max-abs error {max_abs:.3e} > {OUT_MAX_ABS}"
    assert rel <= OUT_REL_L2, f"{what}: relative L2 error {rel:.3e} > {OUT_REL_L2}"
    return {"max_abs": max_abs, "rel_l2": rel}


def check_decode(inp, qk_ref: oracle.QuantizedKeys, gpu: dict, delta: float, units=None,
                 what: str = "") -> dict:
    """Compare one GPU decode with the oracle on the listed (sequence, KV head) units."""
    w = inp.workload
    G = w.num_q_heads // w.num_kv_heads
    ref = oracle.decode(inp.q_bits, inp.seq_lens, inp.block_table, qk_ref, inp.v_bits,
                        sink=w.sink, local=w.local, delta=delta, sm_scale=SM, units=units)
    assert gpu["err"] == 0, f"{what}: device error {gpu['err']}"
    stats = {"borderline": 0, "mask_diffs": 0, "kept": 0, "blocks": 0}
    rerun = []
    for (b, h) in ref.units:
        n = int(inp.seq_lens[b])
        nb = (n + 63) // 64
        gm = gpu["mask"][b, h]
        assert np.all(gm[nb:] == 0), f"{what}: mask tail not cleared at {(b, h)}"
        om = ref.margin[b, h, :nb]
        clear = np.isnan(om) | (np.abs(om) >= MASK_BAND)
        diff = gm[:nb] != ref.mask[b, h, :nb]
        if np.any(diff & clear):
            bad = np.nonzero(diff & clear)[0]
            raise AssertionError(f"{what}: mask mismatch at unit {(b, h)} blocks {bad[:8]} "
                                 f"margins {om[bad[:8]]}")
        stats["borderline"] += int((~clear).sum())
        stats["mask_diffs"] += int(diff.sum())
        stats["kept"] += int(gm[:nb].sum())
        stats["blocks"] += nb
        if diff.any():
            rerun.append((b, h))
        # m~ within fp32 accumulation error
        mt_ref = ref.m_tilde[b, h * G:(h + 1) * G]
        mt_gpu = gpu["m_tilde"][b, h * G:(h + 1) * G]
        fin = np.isfinite(mt_ref)
        assert np.array_equal(np.isfinite(mt_gpu), fin), f"{what}: m~ finiteness at {(b, h)}"
        np.testing.assert_allclose(mt_gpu[fin], mt_ref[fin], rtol=1e-5, atol=2e-5,
                                   err_msg=f"{what}: m~ at {(b, h)}")
    ref_out = ref.out
    if rerun:
        again = oracle.decode(inp.q_bits, inp.seq_lens, inp.block_table, qk_ref, inp.v_bits,
                              sink=w.sink, local=w.local, delta=delta, sm_scale=SM,
                              units=rerun, mask_in=gpu["mask"])
        for (b, h) in rerun:
            ref_out[b, h * G:(h + 1) * G] = again.out[b, h * G:(h + 1) * G]
    sel = np.zeros(gpu["out"].shape[:2], bool)
    for (b, h) in ref.units:
        sel[b, h * G:(h + 1) * G] = True
    stats.update(compare_outputs(gpu["out"][sel], ref_out[sel], what))
    return stats
