"""The algorithmic bytes behind the bench's roofline, on the CPU.

Per token and KV head the step reads 48 B of thumbnail record (32 B of 2-bit codes, four fp16
scales and four fp16 zeros) and, for a kept token, 392 B more (128 B of int8 residual codes, four
fp16 residual scales, 256 B of bf16 V); per step q, out, seq_lens and the block table. The 128K
workload with every block kept is 922 865 680 B, the figure the roofline divides by the measured
launch time. The per-unit count used for the CPU baseline's sample adds up to the same step.
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import ffd_synth  # noqa: E402


def _literal(wid):
    w = ffd_synth.WORKLOADS[wid]
    max_blocks = (w.seq_len + 63) // 64
    seq_lens = np.full(w.batch, w.seq_len, np.int32)
    keep = np.ones((w.batch, w.num_kv_heads, max_blocks), np.uint8)
    return w, seq_lens, max_blocks, keep


def test_128k_step_bytes_by_hand():
    w, seq_lens, max_blocks, keep = _literal(2)
    assert (w.batch, w.num_q_heads, w.num_kv_heads, w.seq_len) == (4, 28, 4, 131072)
    tok_heads = 4 * 131072 * 4
    by = bench.step_bytes(w, seq_lens, max_blocks, bench.kept_tokens(seq_lens, keep))
    assert by["thumbs"] == 48 * tok_heads
    assert by["refine"] == (128 + 8 + 256) * tok_heads
    assert by["q"] == 4 * 28 * 128 * 2 and by["out"] == 4 * 28 * 128 * 4
    assert by["meta"] == 4 * 4 + 4 * 4 * 2048
    assert by["step"] == 922_865_680
    assert by["dense_step"] == 512 * tok_heads + by["q"] + by["out"] + by["meta"]


def test_kept_tokens_counts_the_ragged_last_block():
    seq_lens = np.array([130, 64, 0], np.int32)  # blocks of 64, 64, 2 | 64 | none
    keep = np.zeros((3, 2, 3), np.uint8)
    keep[0, 0, 2] = 1        # the 2-token tail
    keep[0, 1, :] = 1        # 130 tokens
    keep[1, 0, 0] = 1        # 64 tokens
    keep[2, :, :] = 1        # an empty sequence keeps nothing
    assert bench.kept_tokens(seq_lens, keep) == 2 + 130 + 64


def test_unit_bytes_add_up_to_the_step():
    w, seq_lens, max_blocks, keep = _literal(1)
    rng = np.random.default_rng(3)
    keep = (rng.random(keep.shape) < 0.3).astype(np.uint8)
    by = bench.step_bytes(w, seq_lens, max_blocks, bench.kept_tokens(seq_lens, keep))
    units = [(b, h) for b in range(w.batch) for h in range(w.num_kv_heads)]
    assert bench.unit_bytes(w, seq_lens, keep, units) + by["meta"] == by["step"]
