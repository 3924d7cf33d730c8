"""Pins of the CPU statement of ART run-time termination (oracle/art.py): the no-termination limit
against the decode oracle, hand-built stable outputs, the traversal order, strictness, patience and
monotonicity. No GPU needed."""
import math

import numpy as np
import pytest
import torch

import ffd_synth
import oracle
from oracle import art as ART

SM = float(np.float32(1.0 / math.sqrt(128.0)))


def _bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


@pytest.fixture(scope="module")
def small():
    w = ffd_synth.custom(1, 6, 2, 700, sink=16, local=64, seed=41)
    inp = ffd_synth.make_inputs(w, signal_scale=ffd_synth.peaked_scale())
    return w, inp, oracle.quantize(inp.k_bits)


def test_order_is_block_zero_then_most_recent_first():
    assert ART.art_order(5, [1, 1, 0, 1, 1]) == [0, 4, 3, 1]
    assert ART.art_order(3, [0, 0, 0]) == [0]
    assert ART.art_order(0, []) == []


@pytest.mark.parametrize("h", [0, 1])
def test_without_termination_equals_the_softmax_over_the_blocks(small, h):
    """tau = phi = 0: nothing is ever stable, every listed block is used, and the result is the
    softmax over them (the decode oracle with that mask, which sums in token order)."""
    w, inp, qk = small
    G = w.num_q_heads // w.num_kv_heads
    n = int(inp.seq_lens[0])
    nb = (n + 63) // 64
    keep = np.zeros(nb, np.uint8)
    keep[[0, 3, 4, nb - 1]] = 1
    res = ART.art_unit(inp.q_bits[0, h * G:(h + 1) * G], n, inp.block_table[0], qk, inp.v_bits,
                       h, keep, SM, 0.0, 0.0, 1)
    assert res.used == 4
    mask = np.zeros((1, w.num_kv_heads, inp.max_blocks), np.uint8)
    mask[0, h, :nb] = keep
    ref = oracle.decode(inp.q_bits, inp.seq_lens, inp.block_table, qk, inp.v_bits, sink=w.sink,
                        local=w.local, delta=5.0, sm_scale=SM, units=[(0, h)], mask_in=mask)
    np.testing.assert_allclose(res.out, ref.out[0, h * G:(h + 1) * G], rtol=0, atol=1e-12)


def test_two_blocks_by_hand(small):
    """stop_after = 2 uses block 0 and the most recent kept block: the softmax over their tokens,
    written out directly."""
    w, inp, qk = small
    G, h = w.num_q_heads // w.num_kv_heads, 0
    n = int(inp.seq_lens[0])
    nb = (n + 63) // 64
    res = ART.art_unit(inp.q_bits[0, :G], n, inp.block_table[0], qk, inp.v_bits, h,
                       np.ones(nb, np.uint8), SM, 1.0, 1.0, 100, stop_after=2)
    toks = list(range(0, 64)) + list(range(64 * (nb - 1), n))
    pg = inp.block_table[0]
    K = np.stack([oracle.dequant_token(qk, int(pg[j // 64]), h, j % 64)[1] for j in toks])
    V = np.stack([inp.v_bits[int(pg[j // 64]), h, j % 64] for j in toks])
    V = (V.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    q = (inp.q_bits[0, :G].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    s = SM * q @ K.astype(np.float64).T
    p = np.exp(s - s.max(axis=1, keepdims=True))
    want = (p @ V) / p.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(res.out, want, rtol=0, atol=1e-12)
    assert res.used == 2 and len(res.d_scale) == 1


def _uniform_cache(nb, value, G=2):
    """One KV head, every key and value the same: every partial output equals `value`."""
    k = np.zeros((nb, 1, 64, 128), np.float32) + 0.25
    v = np.zeros((nb, 1, 64, 128), np.float32) + value
    q = np.random.default_rng(0).standard_normal((G, 128)).astype(np.float32)
    return _bits(q), _bits(k), _bits(v)


@pytest.mark.parametrize("patience", [1, 2, 3])
def test_stable_output_stops_after_patience(patience):
    nb = 8
    q, k, v = _uniform_cache(nb, 0.5)
    qk = oracle.quantize(k)
    res = ART.art_unit(q, 64 * nb, np.arange(nb), qk, v, 0, np.ones(nb, np.uint8), SM,
                       1e-9, 1e-9, patience)
    assert res.used == 1 + patience  # first check after block 2
    assert max(res.d_scale) == 0.0 and max(res.d_dir) <= 1e-15
    np.testing.assert_allclose(res.out, 0.5, rtol=0, atol=1e-15)


def test_criterion_is_strict_and_monotone(small):
    w, inp, qk = small
    G = w.num_q_heads // w.num_kv_heads
    n = int(inp.seq_lens[0])
    nb = (n + 63) // 64
    keep = np.ones(nb, np.uint8)
    full = ART.art_unit(inp.q_bits[0, :G], n, inp.block_table[0], qk, inp.v_bits, 0, keep, SM,
                        0.0, 0.0, 1)
    assert full.used == nb
    # a threshold equal to every metric is never passed (strict comparisons)
    tau_eq = max(full.d_scale)
    phi_eq = max(full.d_dir)
    res = ART.art_unit(inp.q_bits[0, :G], n, inp.block_table[0], qk, inp.v_bits, 0, keep, SM,
                       min(full.d_scale), min(full.d_dir), 1)
    t = [i for i in range(len(full.d_scale))
         if full.d_scale[i] < min(full.d_scale) and full.d_dir[i] < min(full.d_dir)]
    assert not t and res.used == nb
    # looser thresholds never stop later
    prev_used = nb + 1
    for scale in (1e-4, 1e-3, 1e-2, 1e-1, 1.0):
        r = ART.art_unit(inp.q_bits[0, :G], n, inp.block_table[0], qk, inp.v_bits, 0, keep, SM,
                         scale * tau_eq, scale * phi_eq, 2)
        assert r.used <= prev_used
        prev_used = r.used


def test_metrics_in_closed_form():
    """Identical keys make every softmax weight equal, so the probe after t blocks is the mean of
    the V rows seen. Block 0 holds V = 2 e1 and block 1 holds V = 3 e2: P(1) = 2 e1,
    P(2) = e1 + 1.5 e2, hence d_scale = | |P(2)| - 2 | / 2 and d_direction = 1 - 2 / (2 |P(2)|)."""
    G = 2
    k = np.zeros((2, 1, 64, 128), np.float32) + 0.25
    v = np.zeros((2, 1, 64, 128), np.float32)
    v[0, 0, :, 0] = 2.0
    v[1, 0, :, 1] = 3.0
    q = np.random.default_rng(5).standard_normal((G, 128)).astype(np.float32)
    qk = oracle.quantize(_bits(k))
    res = ART.art_unit(_bits(q), 128, np.arange(2), qk, _bits(v), 0, np.ones(2, np.uint8), SM,
                       0.0, 0.0, 1)
    n2 = math.sqrt(1.0 + 1.5 ** 2)
    assert res.used == 2 and len(res.d_scale) == 1
    assert res.d_scale[0] == pytest.approx(abs(n2 - 2.0) / 2.0, rel=1e-12)
    assert res.d_dir[0] == pytest.approx(1.0 - 1.0 / n2, rel=1e-12)
    want = np.zeros(128)
    want[0], want[1] = 1.0, 1.5
    np.testing.assert_allclose(res.out, np.stack([want, want]), rtol=0, atol=1e-12)
