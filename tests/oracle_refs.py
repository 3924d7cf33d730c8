"""Test-side reference computations used to pin the oracle.

Everything here is an independent restatement through numpy / scipy (vectorised bit unpacking,
library softmax, set-based index enumeration), so that a mistake inside the oracle's C loops
(a dropped term, a wrong index, a transposed operand) shows up as a disagreement.
"""
from __future__ import annotations

import numpy as np
import scipy.special

D = 128
BLK = 64


def f16_bits_to_f64(bits) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def bf16_bits_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def unpack_codes(thumb: np.ndarray) -> np.ndarray:
    """[..., 32] packed bytes -> [..., 128] 2-bit codes; channel c sits in byte c//4 at bit
    2*(c%4)."""
    t = np.asarray(thumb, dtype=np.uint8)
    shifts = np.array([0, 2, 4, 6], dtype=np.uint8)
    codes = (t[..., :, None] >> shifts) & 3          # [..., 32, 4]
    return codes.reshape(t.shape[:-1] + (D,))


def reconstruct(qk, page: int, h: int):
    """(x^2, K^) of every row of one page/head tile as fp32 values, computed as exact fp64
    products and sums rounded once to fp32 (which is what a single fused multiply-add gives)."""
    codes = unpack_codes(qk.thumb[page, h]).astype(np.float64)            # [64,128]
    sf = np.repeat(f16_bits_to_f64(qk.t_scale[page, h]), 32, axis=-1)      # [64,128]
    zf = np.repeat(f16_bits_to_f64(qk.t_zero[page, h]), 32, axis=-1)
    sr = np.repeat(f16_bits_to_f64(qk.r_scale[page, h]), 32, axis=-1)
    x2 = (codes * sf + zf).astype(np.float32)
    kh = (qk.resid[page, h].astype(np.float64) * sr + x2.astype(np.float64)).astype(np.float32)
    return x2, kh


def sequence_rows(qk, block_table, b: int, h: int, n: int):
    """(x^2, K^) [n,128] of the logical tokens 0..n-1 of sequence b, head h."""
    nb = (n + BLK - 1) // BLK
    x2s, khs = [], []
    for blk in range(nb):
        x2, kh = reconstruct(qk, int(block_table[b, blk]), h)
        x2s.append(x2)
        khs.append(kh)
    if not x2s:
        return np.zeros((0, D), np.float32), np.zeros((0, D), np.float32)
    return np.concatenate(x2s)[:n], np.concatenate(khs)[:n]


def v_rows(v_bits, block_table, b: int, h: int, n: int) -> np.ndarray:
    nb = (n + BLK - 1) // BLK
    if nb == 0:
        return np.zeros((0, D))
    rows = [bf16_bits_to_f64(v_bits[int(block_table[b, blk]), h]) for blk in range(nb)]
    return np.concatenate(rows)[:n]


def k_rows(k_bits, block_table, b: int, h: int, n: int) -> np.ndarray:
    return v_rows(k_bits, block_table, b, h, n)


def softmax_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, sm: float) -> np.ndarray:
    """Plain softmax attention through scipy: q [G,128], k/v [m,128] -> [G,128]."""
    if k.shape[0] == 0:
        return np.zeros((q.shape[0], D))
    s = sm * (q @ k.T)
    p = scipy.special.softmax(s, axis=-1)
    return p @ v


def forced_blocks(n: int, S: int, L: int) -> set:
    """Blocks that hold a sink token (j < S) or a local token (j >= n - L), by enumeration."""
    toks = set(range(min(S, n))) | set(range(max(0, n - L), n))
    return {j // BLK for j in toks}


def bruteforce_mask(q, x2, kh, n, S, L, delta, sm):
    """Top-delta block mask straight from the definition, token by token.
    Returns (mask[nb] bool, m_tilde[G], s_hat[G,n], margin[nb])."""
    G = q.shape[0]
    toks = sorted(set(range(min(S, n))) | set(range(max(0, n - L), n)))
    if toks:
        m_tilde = (sm * (q @ kh[toks].T)).max(axis=1)
    else:
        m_tilde = np.full(G, -np.inf)
    s_hat = sm * (q @ x2.T) if n else np.zeros((G, 0))
    nb = (n + BLK - 1) // BLK
    forced = forced_blocks(n, S, L)
    mask = np.zeros(nb, bool)
    margin = np.full(nb, np.nan)
    for blk in range(nb):
        cols = list(range(blk * BLK, min(n, blk * BLK + BLK)))
        d = s_hat[:, cols] - (m_tilde - delta)[:, None]
        margin[blk] = d.max()
        mask[blk] = (blk in forced) or bool((d >= 0).any())
    return mask, m_tilde, s_hat, margin
