"""CPU oracle for FFD sparse decode attention -- TEST INFRASTRUCTURE ONLY.

The arithmetic lives in ``ffd_oracle.c`` (plain C: fp32 bit-defined quantiser, fp64 attention).
This module only compiles it with gcc, loads it with ctypes and loops over independent
(sequence, KV-head) units on host threads (ctypes drops the GIL during each call).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference leg may
import this package. The product library never does, and shares no code with it.

Source of every definition: "Faster Than Flash: Exploiting Attention Sparsity for Efficient
Long-Context Decoding", Methodology section (see ``ffd_oracle.c`` for the per-step citations).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ffd_oracle.c")
_LIB = os.path.join(_HERE, "libffd_oracle.so")
_lock = threading.Lock()
_lib = None

D = 128
BLK = 64
NGROUP = 4


def build(force: bool = False) -> str:
    """Compile ffd_oracle.c into libffd_oracle.so (gcc, no fp contraction, IEEE semantics)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           "-fexcess-precision=standard", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            L.ffdo_f16_from_f32.argtypes = [ctypes.c_float]
            L.ffdo_f16_from_f32.restype = ctypes.c_uint16
            L.ffdo_f32_from_f16.argtypes = [ctypes.c_uint16]
            L.ffdo_f32_from_f16.restype = ctypes.c_float
            L.ffdo_quantize_group.argtypes = [P, P, P, P, P, P]
            L.ffdo_quantize_group.restype = i32
            L.ffdo_quantize_tiles.argtypes = [i64, i64, P, P, P, P, P, P]
            L.ffdo_quantize_tiles.restype = i64
            L.ffdo_dequant_token.argtypes = [P, P, P, P, P, P, P]
            L.ffdo_dequant_token.restype = None
            L.ffdo_decode_unit.argtypes = [i32, i32, i32, i32, f64, f64, P, P, i32, i32, i32,
                                           P, P, P, P, P, P, P, P, P, P, P, P]
            L.ffdo_decode_unit.restype = i32
            L.ffdo_dense_unit.argtypes = [i32, i32, f64, P, P, i32, i32, i32, P, P, P]
            L.ffdo_dense_unit.restype = i32
            _lib = L
    return _lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# ------------------------------------------------------------------------------------------ #
# Number formats                                                                             #
# ------------------------------------------------------------------------------------------ #

def f16_from_f32(x: float) -> int:
    return int(lib().ffdo_f16_from_f32(float(x)))


def f32_from_f16(h: int) -> float:
    return float(lib().ffdo_f32_from_f16(int(h)))


# ------------------------------------------------------------------------------------------ #
# Methodology §1: quantisation                                                                #
# ------------------------------------------------------------------------------------------ #

@dataclass
class QuantizedKeys:
    """The stored key format, one entry per page and KV head ("tile").

    thumb u8 [P,Hkv,64,32]; t_scale, t_zero u16 (f16 bits) [P,Hkv,64,4];
    resid i8 [P,Hkv,64,128]; r_scale u16 (f16 bits) [P,Hkv,64,4]."""
    thumb: np.ndarray
    t_scale: np.ndarray
    t_zero: np.ndarray
    resid: np.ndarray
    r_scale: np.ndarray
    range_violations: int = 0


def quantize_group(x: np.ndarray):
    """Quantise one group of 32 fp32 values; returns (c2, t_scale, t_zero, c8, r_scale, bad)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.shape == (32,)
    c2 = np.zeros(32, np.uint8)
    c8 = np.zeros(32, np.int8)
    ts = np.zeros(1, np.uint16)
    tz = np.zeros(1, np.uint16)
    rs = np.zeros(1, np.uint16)
    bad = lib().ffdo_quantize_group(_p(x), _p(c2), _p(ts), _p(tz), _p(c8), _p(rs))
    return c2, int(ts[0]), int(tz[0]), c8, int(rs[0]), bad


def quantize(k_bits: np.ndarray, threads: int | None = None) -> QuantizedKeys:
    """Quantise a whole paged key cache given as bf16 bit patterns uint16 [P,Hkv,64,128]."""
    k_bits = np.ascontiguousarray(k_bits, dtype=np.uint16)
    P, Hkv, blk, d = k_bits.shape
    assert blk == BLK and d == D
    tiles = P * Hkv
    q = QuantizedKeys(
        thumb=np.zeros((P, Hkv, BLK, D // 4), np.uint8),
        t_scale=np.zeros((P, Hkv, BLK, NGROUP), np.uint16),
        t_zero=np.zeros((P, Hkv, BLK, NGROUP), np.uint16),
        resid=np.zeros((P, Hkv, BLK, D), np.int8),
        r_scale=np.zeros((P, Hkv, BLK, NGROUP), np.uint16),
    )
    L = lib()
    nthr = max(1, min(threads or default_threads(), tiles))
    bounds = np.linspace(0, tiles, nthr + 1).astype(np.int64)

    def run(k):
        return L.ffdo_quantize_tiles(int(bounds[k]), int(bounds[k + 1]), _p(k_bits), _p(q.thumb),
                                     _p(q.t_scale), _p(q.t_zero), _p(q.resid), _p(q.r_scale))

    with ThreadPoolExecutor(nthr) as ex:
        q.range_violations = int(sum(ex.map(run, range(nthr))))
    return q


def dequant_token(qk: QuantizedKeys, page: int, h: int, slot: int):
    """(x^2, K^) of one cached token, fp32 [128] each."""
    xh2 = np.zeros(D, np.float32)
    kh = np.zeros(D, np.float32)
    th = np.ascontiguousarray(qk.thumb[page, h, slot])
    ts = np.ascontiguousarray(qk.t_scale[page, h, slot])
    tz = np.ascontiguousarray(qk.t_zero[page, h, slot])
    rs = np.ascontiguousarray(qk.resid[page, h, slot])
    rc = np.ascontiguousarray(qk.r_scale[page, h, slot])
    lib().ffdo_dequant_token(_p(th), _p(ts), _p(tz), _p(rs), _p(rc), _p(xh2), _p(kh))
    return xh2, kh


# ------------------------------------------------------------------------------------------ #
# Methodology §2-§3: decode                                                                   #
# ------------------------------------------------------------------------------------------ #

@dataclass
class DecodeResult:
    out: np.ndarray        # float64 [B,Hq,128]
    m_tilde: np.ndarray    # float64 [B,Hq]
    mask: np.ndarray       # uint8 [B,Hkv,max_blocks] (blocks >= nb stay 0)
    margin: np.ndarray     # float64 [B,Hkv,max_blocks] (NaN = forced or beyond nb)
    units: list            # the (b, h) units computed
    s_hat: dict | None = None  # (b, h) -> float64 [G, n]


def decode(q_bits, seq_lens, block_table, qk: QuantizedKeys, v_bits, *, sink: int, local: int,
           delta: float, sm_scale: float, units=None, mask_in=None, want_s_hat=False,
           threads: int | None = None) -> DecodeResult:
    """FFD decode of every (sequence b, KV head h) unit listed in ``units`` (default: all).

    q_bits uint16 [B,Hq,128] (bf16 bits); seq_lens int32 [B]; block_table int32 [B,max_blocks];
    v_bits uint16 [P,Hkv,64,128]. ``mask_in`` (uint8 [B,Hkv,max_blocks]) replaces the Top-delta
    block rule for the listed units."""
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    v_bits = np.ascontiguousarray(v_bits, dtype=np.uint16)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    block_table = np.ascontiguousarray(block_table, dtype=np.int32)
    B, Hq, _ = q_bits.shape
    P, Hkv = v_bits.shape[0], v_bits.shape[1]
    G = Hq // Hkv
    maxb = block_table.shape[1]
    res = DecodeResult(out=np.zeros((B, Hq, D)), m_tilde=np.full((B, Hq), -np.inf),
                       mask=np.zeros((B, Hkv, maxb), np.uint8),
                       margin=np.full((B, Hkv, maxb), np.nan),
                       units=list(units) if units is not None else
                       [(b, h) for b in range(B) for h in range(Hkv)],
                       s_hat={} if want_s_hat else None)
    L = lib()
    arrays = [np.ascontiguousarray(a) for a in (qk.thumb, qk.t_scale, qk.t_zero, qk.resid,
                                                qk.r_scale)]

    def run(unit):
        b, h = unit
        n = int(seq_lens[b])
        nb = (n + BLK - 1) // BLK
        q = np.ascontiguousarray(q_bits[b, h * G:(h + 1) * G])
        pages = np.ascontiguousarray(block_table[b, :max(nb, 1)])
        out = np.zeros((G, D))
        mt = np.zeros(G)
        mk = np.zeros(max(nb, 1), np.uint8)
        mg = np.zeros(max(nb, 1))
        sh = np.zeros((G, max(n, 1))) if want_s_hat else None
        mi = None
        if mask_in is not None:
            mi = np.ascontiguousarray(mask_in[b, h, :max(nb, 1)], dtype=np.uint8)
        rc = L.ffdo_decode_unit(G, n, int(sink), int(local), float(delta), float(sm_scale),
                                _p(q), _p(pages), P, Hkv, h, *[_p(a) for a in arrays],
                                _p(v_bits), _p(mi), _p(out), _p(mt), _p(mk), _p(mg), _p(sh))
        if rc != 0:
            raise ValueError(f"oracle decode unit {unit}: page index out of range")
        return unit, n, nb, out, mt, mk, mg, sh

    nthr = max(1, min(threads or default_threads(), len(res.units)))
    with ThreadPoolExecutor(nthr) as ex:
        for (b, h), n, nb, out, mt, mk, mg, sh in ex.map(run, res.units):
            res.out[b, h * G:(h + 1) * G] = out
            res.m_tilde[b, h * G:(h + 1) * G] = mt
            res.mask[b, h, :nb] = mk[:nb]
            res.margin[b, h, :nb] = mg[:nb]
            if want_s_hat:
                res.s_hat[(b, h)] = sh[:, :n]
    return res


def dense(q_bits, seq_lens, block_table, k_bits, v_bits, *, sm_scale: float, units=None,
          threads: int | None = None) -> np.ndarray:
    """Dense softmax attention over the bf16 keys; float64 [B,Hq,128] (zeros outside units)."""
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    k_bits = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v_bits = np.ascontiguousarray(v_bits, dtype=np.uint16)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    block_table = np.ascontiguousarray(block_table, dtype=np.int32)
    B, Hq, _ = q_bits.shape
    P, Hkv = k_bits.shape[0], k_bits.shape[1]
    G = Hq // Hkv
    units = list(units) if units is not None else [(b, h) for b in range(B) for h in range(Hkv)]
    out = np.zeros((B, Hq, D))
    L = lib()

    def run(unit):
        b, h = unit
        n = int(seq_lens[b])
        nb = (n + BLK - 1) // BLK
        q = np.ascontiguousarray(q_bits[b, h * G:(h + 1) * G])
        pages = np.ascontiguousarray(block_table[b, :max(nb, 1)])
        o = np.zeros((G, D))
        rc = L.ffdo_dense_unit(G, n, float(sm_scale), _p(q), _p(pages), P, Hkv, h, _p(k_bits),
                               _p(v_bits), _p(o))
        if rc != 0:
            raise ValueError(f"oracle dense unit {unit}: page index out of range")
        return unit, o

    nthr = max(1, min(threads or default_threads(), len(units)))
    with ThreadPoolExecutor(nthr) as ex:
        for (b, h), o in ex.map(run, units):
            out[b, h * G:(h + 1) * G] = o
    return out
