"""Seeded synthetic decode workloads for FFD sparse decode attention.

This module only draws inputs; it holds none of the method's arithmetic. The same bytes feed the
CUDA library and the CPU oracle. Inputs stand in for the pages' workloads (7B-class GQA models
decoding RULER / LongBench prompts at 16K-256K context, "Faster Than Flash", Main results), which
need datasets and trained weights that are not used here.

Recipe (per configuration; fp32 sampling, then one round-to-nearest-even cast to bf16):
  * q ~ N(0, 1) [B, Hq, 128] (torch generator); K, V ~ N(0, 1) [P, Hkv, 64, 128] in a paged
    layout (page = 64), drawn from numpy PCG64 streams per chunk of 64 pages.
  * q_hat(b, h) = normalise(sum of the bf16 query rows of KV head h's GQA group), fp32.
  * Sink tokens j < S: K_j <- K_j + 3 * a * q_hat.
  * Needles: positions uniform without replacement in [S, n - L); K_j <- 4 * a * q_hat + eps,
    eps ~ N(0, 0.1^2) per channel.
  * a = 1 for the literal workloads; a = sqrt(128) for the "peaked" variant, which states the
    sink shift and needle magnitude in score units so that attention is concentrated and most
    blocks fall below the Top-delta threshold.
  * Block tables: identity (sequence b owns pages b*max_blocks ...), or a random permutation of
    the page pool for the batched paged workload. Unused entries are -1.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

D = 128
PAGE = 64


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    seq_len: int | tuple          # fixed length, or (lo, hi) inclusive uniform per sequence
    sink: int
    local: int
    deltas: tuple
    needles: int | tuple          # per KV head: fixed count, or (lo, hi) inclusive uniform
    random_pages: bool = False
    seed: int = 0


WORKLOADS = {
    0: Workload("tiny-b1-h8x2-4k", 1, 8, 2, 4096, 64, 256, (5.0,), 6, seed=1000),
    1: Workload("llama3.1-8b-b1-h32x8-32k", 1, 32, 8, 32768, 64, 1024, (5.0, 7.0), 16,
                seed=1001),
    2: Workload("qwen2.5-7b-b4-h28x4-128k", 4, 28, 4, 131072, 64, 1024, (5.0,), (4, 64),
                seed=1002),
    3: Workload("llama3.1-8b-b1-h32x8-256k", 1, 32, 8, 262144, 64, 1024, (5.0, 7.0), 16,
                seed=1003),
    4: Workload("paged-b32-h32x8-4k..16k", 32, 32, 8, (4096, 16384), 64, 512, (5.0,), 16,
                random_pages=True, seed=1004),
}


@dataclass
class Inputs:
    """One decode step's inputs as raw bit patterns (bf16 -> uint16)."""
    workload: Workload
    q_bits: np.ndarray          # uint16 [B, Hq, 128]
    k_bits: np.ndarray          # uint16 [P, Hkv, 64, 128]
    v_bits: np.ndarray          # uint16 [P, Hkv, 64, 128]
    seq_lens: np.ndarray        # int32 [B]
    block_table: np.ndarray     # int32 [B, max_blocks]
    needle_pos: dict = field(default_factory=dict)  # (b, h) -> np.ndarray of token positions
    signal_scale: float = 1.0

    @property
    def num_pages(self) -> int:
        return int(self.k_bits.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])


def _bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


_CHUNK_PAGES = 64


def _normal_pages(seed: int, stream: int, P: int, Hkv: int) -> torch.Tensor:
    """N(0,1) fp32 [P, Hkv, 64, 128]; page chunk c draws from its own PCG64 stream
    (seed, stream, c), so the values do not depend on how many threads draw them."""
    out = np.empty((P, Hkv, PAGE, D), np.float32)
    chunks = range(0, P, _CHUNK_PAGES)

    def fill(p0):
        rng = np.random.Generator(np.random.PCG64([seed, stream, p0 // _CHUNK_PAGES]))
        p1 = min(P, p0 + _CHUNK_PAGES)
        out[p0:p1] = rng.standard_normal((p1 - p0, Hkv, PAGE, D), dtype=np.float32)

    with ThreadPoolExecutor(max(1, min(16, os.cpu_count() or 1))) as ex:
        list(ex.map(fill, chunks))
    return torch.from_numpy(out)


def make_inputs(w: Workload, *, seed: int | None = None, signal_scale: float = 1.0,
                seq_lens=None) -> Inputs:
    """Draw one step's inputs for workload ``w``. ``seq_lens`` overrides the drawn lengths."""
    g = torch.Generator().manual_seed(w.seed if seed is None else seed)
    B, Hq, Hkv = w.batch, w.num_q_heads, w.num_kv_heads
    assert Hq % Hkv == 0
    G = Hq // Hkv

    if seq_lens is not None:
        lens = np.asarray(seq_lens, dtype=np.int64)
        assert lens.shape == (B,)
    elif isinstance(w.seq_len, tuple):
        lo, hi = w.seq_len
        lens = torch.randint(lo, hi + 1, (B,), generator=g).numpy().astype(np.int64)
    else:
        lens = np.full(B, w.seq_len, np.int64)
    nbs = [(int(n) + PAGE - 1) // PAGE for n in lens]
    if isinstance(w.seq_len, tuple) and seq_lens is None:
        max_blocks = (w.seq_len[1] + PAGE - 1) // PAGE
    else:
        max_blocks = max(nbs)
    max_blocks = max(1, max_blocks)

    if w.random_pages:
        P = max(1, sum(nbs))
        perm = torch.randperm(P, generator=g).numpy().astype(np.int32)
        bt = np.full((B, max_blocks), -1, np.int32)
        off = 0
        for b, nb in enumerate(nbs):
            bt[b, :nb] = perm[off:off + nb]
            off += nb
    else:
        P = B * max_blocks
        bt = np.full((B, max_blocks), -1, np.int32)
        for b, nb in enumerate(nbs):
            bt[b, :nb] = np.arange(b * max_blocks, b * max_blocks + nb, dtype=np.int32)

    q = torch.randn((B, Hq, D), generator=g, dtype=torch.float32)
    q_bits = _bf16_bits(q)
    qf = q.to(torch.bfloat16).to(torch.float32)
    base_seed = w.seed if seed is None else seed
    k = _normal_pages(base_seed, 1, P, Hkv)
    v = _normal_pages(base_seed, 2, P, Hkv)

    a = float(signal_scale)
    needle_pos = {}
    for b in range(B):
        n = int(lens[b])
        for h in range(Hkv):
            s = qf[b, h * G:(h + 1) * G].sum(dim=0)
            qhat = s / torch.linalg.vector_norm(s)
            # sink shift
            for j in range(min(w.sink, n)):
                page = int(bt[b, j // PAGE])
                k[page, h, j % PAGE] += 3.0 * a * qhat
            # needles
            if isinstance(w.needles, tuple):
                cnt = int(torch.randint(w.needles[0], w.needles[1] + 1, (1,), generator=g))
            else:
                cnt = int(w.needles)
            span = n - w.local - w.sink
            cnt = max(0, min(cnt, span))
            if cnt > 0:
                pos = (torch.randperm(span, generator=g)[:cnt] + w.sink).numpy()
                noise = 0.1 * torch.randn((cnt, D), generator=g, dtype=torch.float32)
                for t, j in enumerate(pos):
                    page = int(bt[b, int(j) // PAGE])
                    k[page, h, int(j) % PAGE] = 4.0 * a * qhat + noise[t]
                needle_pos[(b, h)] = np.sort(pos)
            else:
                needle_pos[(b, h)] = np.zeros(0, np.int64)

    return Inputs(workload=w, q_bits=q_bits, k_bits=_bf16_bits(k), v_bits=_bf16_bits(v),
                  seq_lens=lens.astype(np.int32), block_table=bt, needle_pos=needle_pos,
                  signal_scale=a)


def custom(batch, num_q_heads, num_kv_heads, seq_len, *, sink=64, local=256, needles=4,
           random_pages=False, seed=7) -> Workload:
    """A workload with explicit shape, for tests (edge cases, ragged lengths)."""
    return Workload(f"custom-b{batch}-h{num_q_heads}x{num_kv_heads}", batch, num_q_heads,
                    num_kv_heads, seq_len, sink, local, (5.0,), needles,
                    random_pages=random_pages, seed=seed)


def peaked_scale() -> float:
    return math.sqrt(D)
