"""Comparison block selectors (Top-k, Top-p) on the thumbnail scores: the plain CPU statement.

TEST INFRASTRUCTURE ONLY, like the rest of this package: only the tests, the package smoke check
and the benchmark's CPU legs use it; the product library never loads it.

Source: "Faster Than Flash" (technical summaries), Problem statement, the "selection dilemma":
a fixed-budget Top-k does not adapt to attention entropy that varies from head to head and step
to step, and a distribution-adaptive Top-p needs a global softmax and a sort, which breaks a
streaming pipeline. FFD's Top-delta rule (Methodology §2) is measured against these two. The
pages define neither rule in detail; the readings taken here:

  * Both rules rank the same 64-token blocks as Top-delta, on the same provisional scores
    s^_ij = sm * q_i . x^2_j (thumbnail only), and keep the same always-kept blocks (those holding
    a sink or local token), so that the three rules differ only in how they choose the rest.
  * Top-k: a block's importance is the largest s^_ij over the heads i of the GQA group and its
    tokens j < n. The k non-forced blocks of largest importance are kept (ties: lower block index
    first); with fewer than k non-forced blocks, all are kept.
  * Top-p: per query head i, P_ij = softmax over all tokens j < n of s^_ij (the global softmax),
    and block c has mass m_ic = sum of P_ij over its tokens. Blocks are ranked by mass
    (descending; ties: lower block index first) and a block is kept when the masses ranked
    before it sum to less than p: the shortest prefix whose mass reaches p. The kept set is the
    union of these prefixes over the heads of the group, plus the forced blocks.

Everything here is fp64 and written for a reader, not for speed.
"""
from __future__ import annotations

import numpy as np

BLK = 64


def forced_blocks(n: int, sink: int, local: int) -> np.ndarray:
    """Blocks holding a sink token (j < S) or a local token (j >= n - L), as a bool [nb]."""
    nb = (n + BLK - 1) // BLK
    out = np.zeros(nb, bool)
    for j in range(n):
        if j < sink or j >= n - local:
            out[j // BLK] = True
    return out


def block_importance(s_hat: np.ndarray, n: int) -> np.ndarray:
    """max over heads and tokens j < n of the block, of s^_ij; s_hat is [G, n]."""
    nb = (n + BLK - 1) // BLK
    return np.array([s_hat[:, c * BLK:min(n, (c + 1) * BLK)].max() for c in range(nb)])


def block_mass(s_hat: np.ndarray, n: int) -> np.ndarray:
    """m_ic = sum over the tokens of block c of softmax_j(s^_ij), per head: [G, nb]."""
    G = s_hat.shape[0]
    nb = (n + BLK - 1) // BLK
    out = np.zeros((G, nb))
    for i in range(G):
        row = s_hat[i, :n]
        w = np.exp(row - row.max())
        P = w / w.sum()
        for c in range(nb):
            out[i, c] = P[c * BLK:min(n, (c + 1) * BLK)].sum()
    return out


def _rank(values: np.ndarray, eligible: np.ndarray) -> list:
    """Indices of the eligible entries, largest value first, ties by lower index."""
    idx = [c for c in range(len(values)) if eligible[c]]
    return sorted(idx, key=lambda c: (-values[c], c))


def select_topk(s_hat: np.ndarray, n: int, sink: int, local: int, k: int):
    """Top-k keep mask [nb] (uint8) and the importance of every block."""
    forced = forced_blocks(n, sink, local)
    imp = block_importance(s_hat, n)
    keep = forced.copy()
    for c in _rank(imp, ~forced)[:max(0, k)]:
        keep[c] = True
    return keep.astype(np.uint8), imp


def select_topp(s_hat: np.ndarray, n: int, sink: int, local: int, p: float):
    """Top-p keep mask [nb] (uint8), the per-head block masses [G, nb] and, per head, the mass
    ranked before each block ([G, nb]: the exclusive prefix sum in the head's ranking)."""
    forced = forced_blocks(n, sink, local)
    mass = block_mass(s_hat, n)
    G, nb = mass.shape
    before = np.zeros((G, nb))
    keep = forced.copy()
    for i in range(G):
        acc = 0.0
        for c in _rank(mass[i], np.ones(nb, bool)):
            before[i, c] = acc
            if acc < p:
                keep[c] = True
            acc += mass[i, c]
    return keep.astype(np.uint8), mass, before
