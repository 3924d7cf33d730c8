"""Run-time termination of the attention over a unit's blocks (ART), the plain CPU statement.

TEST INFRASTRUCTURE ONLY, like the rest of this package: only the tests, the package smoke check and
the benchmark's CPU legs use it; the product library never loads it.

Source: "ART: Attention Run-time Termination" (technical summary page), §2.2 "stability-based
termination criterion" (the partial output O(t) is watched as KV blocks are added; the magnitude
change d_scale, an L2-norm difference between consecutive probe vectors, and the direction change
d_direction, the deviation of their cosine similarity, must both fall below thresholds tau and phi),
§2.3 "patience" (the criterion must hold p times in a row before the computation stops) and §2.4
(the block traversal can be reordered, for instance most recent first, because online softmax is
permutation invariant; block 0, an attention sink, is always evaluated first). The pages of the
FFD method call ART an orthogonal layer; here it runs over the blocks that a selection kept.

Readings (the page leaves these open):
  * the probe of head i after t blocks is its whole normalised partial output o_i / l_i;
  * d_scale = | |P_i(t)| - |P_i(t-1)| | / |P_i(t-1)| and d_direction = 1 - cos(P_i(t), P_i(t-1)),
    each taken as the maximum over the heads of the GQA group (the group shares the blocks);
  * the criterion is strict (d_scale < tau and d_direction < phi), first checked after the second
    block; the computation stops after the block at which it has held `patience` times in a row;
  * the order is block 0, then the kept blocks from the most recent to the oldest.

Everything here is fp64; keys are the reconstructed K^ of the quantised cache (thumbnail plus
residual), scores s = sm_scale * q . K^, as in the FFD decode step.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import dequant_token

BLK = 64


def _bf16(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def art_order(nb: int, keep) -> list:
    """Block 0 first, then the kept blocks from the most recent to the oldest."""
    if nb == 0:
        return []
    return [0] + [c for c in range(nb - 1, 0, -1) if keep[c]]


@dataclass
class ArtResult:
    out: np.ndarray            # [G, 128] normalised output after the last block used
    used: int                  # blocks used (a prefix of art_order)
    d_scale: list = field(default_factory=list)   # metric after block t (t >= 2), in order
    d_dir: list = field(default_factory=list)


def art_unit(q_bits: np.ndarray, n: int, pages, qk, v_bits: np.ndarray, h: int, keep,
             sm_scale: float, tau: float, phi: float, patience: int,
             stop_after: int | None = None) -> ArtResult:
    """ART over one (sequence, KV head) unit. q_bits [G, 128] bf16 bits of the group's queries;
    pages: the sequence's block-table row; keep [nb]: blocks the selection kept (block 0 is
    evaluated whatever it says). With stop_after, exactly that many blocks are used (the criterion
    is still evaluated and reported)."""
    q = _bf16(q_bits)
    G = q.shape[0]
    nb = (n + BLK - 1) // BLK
    order = art_order(nb, keep)
    m = np.full(G, -np.inf)
    lsum = np.zeros(G)
    o = np.zeros((G, 128))
    prev = None
    streak = 0
    res = ArtResult(out=np.zeros((G, 128)), used=0)
    for c in order:
        rows = range(c * BLK, min(n, (c + 1) * BLK))
        keys = np.stack([dequant_token(qk, int(pages[c]), h, j % BLK)[1] for j in rows])
        vals = _bf16(np.stack([v_bits[int(pages[c]), h, j % BLK] for j in rows]))
        s = sm_scale * (q @ keys.astype(np.float64).T)          # [G, rows]
        m_new = np.maximum(m, s.max(axis=1))
        alpha = np.where(np.isfinite(m), np.exp(m - m_new), 0.0)
        p = np.exp(s - m_new[:, None])
        lsum = lsum * alpha + p.sum(axis=1)
        o = o * alpha[:, None] + p @ vals
        m = m_new
        res.used += 1
        cur = o / lsum[:, None]
        if prev is not None:
            nc = np.linalg.norm(cur, axis=1)
            npv = np.linalg.norm(prev, axis=1)
            ds = np.where(npv > 0, np.abs(nc - npv) / np.where(npv > 0, npv, 1.0), nc)
            cosv = np.where((nc > 0) & (npv > 0),
                            (cur * prev).sum(axis=1) / np.where((nc > 0) & (npv > 0), nc * npv, 1.0),
                            np.where((nc == 0) & (npv == 0), 1.0, 0.0))
            d_scale, d_dir = float(ds.max()), float((1.0 - cosv).max())
            res.d_scale.append(d_scale)
            res.d_dir.append(d_dir)
            streak = streak + 1 if (d_scale < tau and d_dir < phi) else 0
        prev = cur
        if stop_after is not None:
            if res.used >= stop_after:
                break
        elif streak >= patience:
            break
    res.out = o / lsum[:, None] if res.used else np.zeros((G, 128))
    return res
