"""Pins of the CPU oracle to things other than itself (runs on the CPU, no GPU).

Each test compares the oracle with an independent source: numpy's IEEE half conversion, a
brute-force nearest-level search, hand-derived golden values, closed forms (one-hot attention,
identical keys), a library softmax, set-based enumeration of the Top-delta rule, and invariances
that the method's definition implies ("Faster Than Flash", Methodology §1-§3).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import ffd_synth
import oracle
from tests import oracle_refs as R

SM = float(np.float32(1.0 / math.sqrt(128.0)))
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(x) -> np.ndarray:
    """fp32 values -> nearest bf16 values (as fp32)."""
    t = torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16).to(torch.float32)
    return t.numpy()


# ------------------------------------------------------------------------------------------- #
# Number formats                                                                              #
# ------------------------------------------------------------------------------------------- #

def test_f16_from_f32_matches_numpy():
    rng = np.random.default_rng(0)
    vals = [np.float32(v) for v in
            rng.standard_normal(3000) * np.exp2(rng.integers(-30, 18, 3000))]
    # exact midpoints between adjacent binary16 values (ties), normal and subnormal
    for h in rng.integers(0, 0x7BFF, 2000):
        a = float(np.uint16(h).view(np.float16))
        b = float(np.uint16(h + 1).view(np.float16))
        vals.append(np.float32((a + b) / 2))
        vals.append(np.float32(-(a + b) / 2))
    vals += [np.float32(v) for v in (0.0, -0.0, 65504.0, 65519.0, 65520.0, 1e6, 2.0 ** -24,
                                     2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -14, 6.0e-8, 1.0 / 3)]
    for v in vals:
        want = int(np.array([v], np.float32).astype(np.float16).view(np.uint16)[0])
        assert oracle.f16_from_f32(float(v)) == want, v


def test_f32_from_f16_all_patterns():
    for h in range(65536):
        f = np.uint16(h).view(np.float16)
        if np.isnan(f):
            assert math.isnan(oracle.f32_from_f16(h))
        else:
            assert oracle.f32_from_f16(h) == float(np.float32(f)), hex(h)


# ------------------------------------------------------------------------------------------- #
# Methodology §1: quantiser                                                                   #
# ------------------------------------------------------------------------------------------- #

def test_golden_quant_groups():
    with open(os.path.join(GOLDEN, "quant_groups.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        x = np.full(32, case.get("fill", 0.0), np.float32)
        x[:len(case["x"])] = case["x"]
        c2, ts, tz, c8, rs, bad = oracle.quantize_group(x)
        assert bad == 0
        assert list(c2) == case["c2"], case["name"]
        assert list(c8) == case["c8"], case["name"]
        assert ts == int(case["t_scale"], 16), case["name"]
        assert tz == int(case["t_zero"], 16), case["name"]
        assert rs == int(case["r_scale"], 16), case["name"]


def _random_groups(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for k in range(n):
        kind = k % 5
        if kind == 0:
            x = rng.standard_normal(32)
        elif kind == 1:
            x = rng.standard_normal(32) * 1e-3 + rng.standard_normal()
        elif kind == 2:
            x = rng.uniform(-50, 50, 32)
        elif kind == 3:
            x = rng.standard_normal(32)
            x[rng.integers(32)] = rng.choice([-1, 1]) * rng.uniform(5, 40)
        else:
            x = rng.integers(-4, 5, 32) * rng.choice([0.5, 0.25, 1.0])
        out.append(_bf16(x))
    return out


def test_quantizer_nearest_level_bruteforce():
    """c2 is the nearest of the 4 thumbnail levels and c8 the nearest of the 255 residual levels,
    found here by exhaustive search (exact fp64 distances), except at numerical ties."""
    checked2 = checked8 = 0
    for x in _random_groups(1500, 1):
        c2, ts, tz, c8, rs, bad = oracle.quantize_group(x)
        assert bad == 0
        sf = float(R.f16_bits_to_f64(ts))
        zf = float(R.f16_bits_to_f64(tz))
        sr = float(R.f16_bits_to_f64(rs))
        # scale / zero against numpy's own half rounding
        assert tz == int(np.float32(x.min()).astype(np.float16).view(np.uint16))
        step = np.float32(np.float32(x.max()) - np.float32(x.min())) / np.float32(3.0)
        assert ts == int(np.float32(step).astype(np.float16).view(np.uint16))
        if sf == 0.0:
            assert not c2.any()
        levels = np.array([c * sf + zf for c in range(4)])
        x2 = np.empty(32, np.float32)
        for c in range(32):
            d = np.abs(float(x[c]) - levels)
            order = np.argsort(d)
            if sf > 0 and d[order[1]] - d[order[0]] > 1e-6 * sf:
                assert c2[c] == order[0], (x, c)
                checked2 += 1
            x2[c] = np.float32(c2[c] * sf + zf)
        r = (x - x2).astype(np.float32)
        assert rs == int((np.float32(np.abs(r).max()) / np.float32(127.0))
                         .astype(np.float16).view(np.uint16))
        if sr == 0.0:
            assert not c8.any()
            continue
        ks = np.arange(-127, 128)
        for c in range(32):
            d = np.abs(float(r[c]) - ks * sr)
            order = np.argsort(d)
            if d[order[1]] - d[order[0]] > 1e-6 * sr:
                assert c8[c] == ks[order[0]], (x, c)
                checked8 += 1
    assert checked2 > 40000 and checked8 > 40000


def test_quantizer_error_bounds_near_fp16():
    """|x - x^2| <= scale/2; |x - K^| <= max(r_scale/2, max|r| - 127 r_scale) (+1 ulp), and when
    r_scale is an fp16 normal number also <= range/1500: the residual rebuilds the key to about
    2^-11 of the group's range (Methodology §1, "near FP16 precision"). Below fp16's normal range
    r_scale itself is coarse and the +-127 clamp can cost up to about one r_scale."""
    normal = 0
    for x in _random_groups(1500, 2):
        c2, ts, tz, c8, rs, _ = oracle.quantize_group(x)
        sf = float(R.f16_bits_to_f64(ts))
        zf = float(R.f16_bits_to_f64(tz))
        sr = float(R.f16_bits_to_f64(rs))
        x2 = np.float32(c2 * sf + zf)
        kh = (c8.astype(np.float64) * sr + x2.astype(np.float64)).astype(np.float32)
        err = np.abs(x.astype(np.float64) - kh)
        ulp = 2.0 ** -23 * float(np.abs(x).max())
        assert np.all(np.abs(x - x2) <= 0.5 * sf * (1 + 2e-3) + 1e-30)
        rmax = float(np.abs((x - x2).astype(np.float32)).max())
        assert np.all(err <= max(0.5 * sr, rmax - 127 * sr) * (1 + 1e-6) + ulp), (x, kh)
        if sr >= 2.0 ** -14:
            normal += 1
            assert np.all(err <= float(x.max() - x.min()) / 1500 + ulp), (x, kh)
    assert normal > 1000


def test_thumb_packing_and_tile_layout():
    """The tile quantiser stores each token's groups at the documented positions: channel c of
    token j in byte c//4 at bit 2*(c%4); scales per group of 32 channels."""
    rng = np.random.default_rng(3)
    k = _bf16(rng.standard_normal((3, 2, 64, 128)) * rng.uniform(0.1, 4, (3, 2, 64, 1)))
    bits = torch.as_tensor(k).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    qk = oracle.quantize(bits, threads=2)
    codes = R.unpack_codes(qk.thumb)
    for p, h, j in [(0, 0, 0), (2, 1, 63), (1, 0, 17), (1, 1, 40)]:
        for g in range(4):
            c2, ts, tz, c8, rs, _ = oracle.quantize_group(k[p, h, j, 32 * g:32 * g + 32])
            assert list(codes[p, h, j, 32 * g:32 * g + 32]) == list(c2)
            assert list(qk.resid[p, h, j, 32 * g:32 * g + 32]) == list(c8)
            assert (qk.t_scale[p, h, j, g], qk.t_zero[p, h, j, g], qk.r_scale[p, h, j, g]) == \
                (ts, tz, rs)


def test_dequant_matches_numpy_reconstruction():
    rng = np.random.default_rng(4)
    k = _bf16(rng.standard_normal((2, 2, 64, 128)))
    bits = torch.as_tensor(k).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    qk = oracle.quantize(bits, threads=1)
    for p in range(2):
        for h in range(2):
            x2n, khn = R.reconstruct(qk, p, h)
            for j in (0, 5, 63):
                x2, kh = oracle.dequant_token(qk, p, h, j)
                assert np.array_equal(x2, x2n[j]) and np.array_equal(kh, khn[j])


# ------------------------------------------------------------------------------------------- #
# Methodology §2-§3: decode                                                                   #
# ------------------------------------------------------------------------------------------- #

def _setup(batch=2, hq=4, hkv=2, seq_lens=(300, 129), sink=4, local=16, needles=3,
           peaked=True, random_pages=True, seed=11):
    w = ffd_synth.custom(batch, hq, hkv, max(seq_lens), sink=sink, local=local, needles=needles,
                         random_pages=random_pages, seed=seed)
    inp = ffd_synth.make_inputs(w, signal_scale=ffd_synth.peaked_scale() if peaked else 1.0,
                                seq_lens=list(seq_lens))
    qk = oracle.quantize(inp.k_bits, threads=2)
    return w, inp, qk


def _decode(inp, qk, w, delta, **kw):
    return oracle.decode(inp.q_bits, inp.seq_lens, inp.block_table, qk, inp.v_bits,
                         sink=w.sink, local=w.local, delta=delta, sm_scale=SM, threads=2, **kw)


def _q(inp, b, h, G):
    return R.bf16_bits_to_f64(inp.q_bits[b, h * G:(h + 1) * G])


def test_delta_inf_is_dense_softmax_over_khat():
    """delta = +inf keeps every block, so the output is plain softmax attention over the
    reconstructed keys K^ -- here through scipy on an independent reconstruction."""
    w, inp, qk = _setup(peaked=False)
    res = _decode(inp, qk, w, math.inf)
    G = w.num_q_heads // w.num_kv_heads
    for b in range(w.batch):
        n = int(inp.seq_lens[b])
        nb = (n + 63) // 64
        for h in range(w.num_kv_heads):
            assert res.mask[b, h, :nb].all()
            _, kh = R.sequence_rows(qk, inp.block_table, b, h, n)
            ref = R.softmax_attention(_q(inp, b, h, G), kh.astype(np.float64),
                                      R.v_rows(inp.v_bits, inp.block_table, b, h, n), SM)
            np.testing.assert_allclose(res.out[b, h * G:(h + 1) * G], ref, rtol=0, atol=1e-12)


def test_dense_oracle_is_softmax_over_bf16_keys():
    w, inp, qk = _setup(peaked=False)
    out = oracle.dense(inp.q_bits, inp.seq_lens, inp.block_table, inp.k_bits, inp.v_bits,
                       sm_scale=SM, threads=2)
    G = w.num_q_heads // w.num_kv_heads
    for b in range(w.batch):
        n = int(inp.seq_lens[b])
        for h in range(w.num_kv_heads):
            ref = R.softmax_attention(_q(inp, b, h, G),
                                      R.k_rows(inp.k_bits, inp.block_table, b, h, n),
                                      R.v_rows(inp.v_bits, inp.block_table, b, h, n), SM)
            np.testing.assert_allclose(out[b, h * G:(h + 1) * G], ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("shape", [
    dict(batch=1, hq=1, hkv=1, seq_lens=(1,), sink=1, local=1),
    dict(batch=1, hq=2, hkv=1, seq_lens=(63,), sink=0, local=8),
    dict(batch=2, hq=4, hkv=2, seq_lens=(64, 65), sink=4, local=0),
    dict(batch=2, hq=4, hkv=1, seq_lens=(200, 256), sink=8, local=16),
    dict(batch=3, hq=6, hkv=2, seq_lens=(130, 300, 77), sink=3, local=40),
])
@pytest.mark.parametrize("delta", [0.0, 2.0, 5.0, 7.0])
def test_mask_and_pseudo_max_bruteforce(shape, delta):
    """Stage 1 and stage 2 against the rule written out token by token on tiny inputs: m~ from
    the sink / local token sets, s^ from the thumbnail, block kept iff forced or some head and
    token pass s^ >= m~ - delta."""
    w, inp, qk = _setup(needles=2, **shape)
    res = _decode(inp, qk, w, delta, want_s_hat=True)
    G = w.num_q_heads // w.num_kv_heads
    for b in range(w.batch):
        n = int(inp.seq_lens[b])
        nb = (n + 63) // 64
        for h in range(w.num_kv_heads):
            x2, kh = R.sequence_rows(qk, inp.block_table, b, h, n)
            mask, mt, sh, mg = R.bruteforce_mask(_q(inp, b, h, G), x2.astype(np.float64),
                                                 kh.astype(np.float64), n, w.sink, w.local,
                                                 delta, SM)
            np.testing.assert_allclose(res.m_tilde[b, h * G:(h + 1) * G], mt, rtol=1e-13,
                                       atol=1e-13)
            np.testing.assert_allclose(res.s_hat[(b, h)], sh, rtol=1e-13, atol=1e-13)
            clear = ~(np.abs(mg) < 1e-9)
            assert np.array_equal(res.mask[b, h, :nb].astype(bool)[clear], mask[clear])


def test_forced_blocks_only_with_negative_delta():
    """With the threshold out of reach only blocks holding sink or local tokens stay, and the
    output is softmax attention over exactly those blocks' tokens (whole blocks)."""
    w, inp, qk = _setup(peaked=False, sink=4, local=16)
    res = _decode(inp, qk, w, -1e9)
    G = w.num_q_heads // w.num_kv_heads
    for b in range(w.batch):
        n = int(inp.seq_lens[b])
        nb = (n + 63) // 64
        forced = R.forced_blocks(n, w.sink, w.local)
        for h in range(w.num_kv_heads):
            assert set(np.nonzero(res.mask[b, h, :nb])[0]) == forced
            _, kh = R.sequence_rows(qk, inp.block_table, b, h, n)
            v = R.v_rows(inp.v_bits, inp.block_table, b, h, n)
            toks = [j for j in range(n) if j // 64 in forced]
            ref = R.softmax_attention(_q(inp, b, h, G), kh[toks].astype(np.float64), v[toks], SM)
            np.testing.assert_allclose(res.out[b, h * G:(h + 1) * G], ref, rtol=0, atol=1e-12)


def test_selection_monotone_in_delta():
    w, inp, qk = _setup(batch=1, hq=8, hkv=2, seq_lens=(4096,), sink=64, local=256, needles=6)
    prev = None
    for delta in (-1e9, 0.0, 2.0, 5.0, 7.0, 20.0, math.inf):
        m = _decode(inp, qk, w, delta).mask.astype(bool)
        if prev is not None:
            assert np.all(m >= prev)
        prev = m
    assert prev.all()


def test_block_order_invariance():
    """Softmax attention does not depend on the order of the blocks: exchanging two non-forced
    blocks between logical positions (through the block table) changes nothing but the order in
    which the mask lists them; moving pages to other physical slots changes nothing at all."""
    w, inp, qk = _setup(batch=1, hq=4, hkv=2, seq_lens=(1000,), sink=4, local=16, needles=4)
    for delta in (5.0, math.inf):
        base = _decode(inp, qk, w, delta)
        bt = inp.block_table.copy()
        bt[0, [3, 9]] = bt[0, [9, 3]]
        inp2 = ffd_synth.Inputs(**{**inp.__dict__, "block_table": bt})
        sw = _decode(inp2, qk, w, delta)
        np.testing.assert_allclose(sw.out, base.out, rtol=0, atol=1e-14)
        exp_mask = base.mask.copy()
        exp_mask[0, :, [3, 9]] = exp_mask[0, :, [9, 3]]
        assert np.array_equal(sw.mask, exp_mask)
    # physical relocation: reverse the page pool
    P = inp.num_pages
    perm = np.arange(P)[::-1].copy()
    inv = np.argsort(perm)
    qk2 = oracle.QuantizedKeys(*(np.ascontiguousarray(a[perm]) for a in
                                 (qk.thumb, qk.t_scale, qk.t_zero, qk.resid, qk.r_scale)))
    bt = np.where(inp.block_table >= 0, inv[np.maximum(inp.block_table, 0)], -1).astype(np.int32)
    inp3 = ffd_synth.Inputs(**{**inp.__dict__, "block_table": bt,
                               "v_bits": np.ascontiguousarray(inp.v_bits[perm])})
    base = _decode(inp, qk, w, 5.0)
    mv = _decode(inp3, qk2, w, 5.0)
    assert np.array_equal(mv.out, base.out) and np.array_equal(mv.mask, base.mask)


def test_needle_gives_one_hot_attention():
    """One key whose score exceeds all others by > 50 takes all the attention: out = V_needle to
    within e^-50 (closed form of softmax)."""
    w, inp, qk = _setup(batch=1, hq=1, hkv=1, seq_lens=(500,), sink=4, local=16, needles=0,
                        peaked=False)
    q = R.bf16_bits_to_f64(inp.q_bits[0, 0])
    j = 200
    kj = _bf16(q * (60.0 / SM / float(q @ q)))
    page = int(inp.block_table[0, j // 64])
    k_bits = inp.k_bits.copy()
    k_bits[page, 0, j % 64] = torch.as_tensor(kj).to(torch.bfloat16).view(torch.int16).numpy() \
        .view(np.uint16)
    qk = oracle.quantize(k_bits, threads=1)
    res = _decode(inp, qk, w, 5.0)
    vj = R.bf16_bits_to_f64(inp.v_bits[page, 0, j % 64])
    assert res.mask[0, 0, j // 64] == 1
    np.testing.assert_allclose(res.out[0, 0], vj, rtol=0, atol=1e-12)


def test_identical_keys_give_mean_of_kept_values():
    w, inp, qk = _setup(batch=1, hq=2, hkv=1, seq_lens=(333,), sink=4, local=16, peaked=False)
    k_bits = inp.k_bits.copy()
    k_bits[:, :, :, :] = k_bits[0, 0, 0]
    qk = oracle.quantize(k_bits, threads=1)
    for delta in (5.0, -1e9):
        res = _decode(inp, qk, w, delta)
        n = 333
        v = R.v_rows(inp.v_bits, inp.block_table, 0, 0, n)
        kept = [j for j in range(n) if res.mask[0, 0, j // 64]]
        for i in range(2):
            np.testing.assert_allclose(res.out[0, i], v[kept].mean(axis=0), rtol=0, atol=1e-12)


def test_degenerate_lengths_and_windows():
    w, inp, qk = _setup(batch=3, hq=2, hkv=1, seq_lens=(0, 5, 70), sink=0, local=0)
    res = _decode(inp, qk, w, 5.0)
    assert np.all(res.out[0] == 0) and np.all(np.isneginf(res.m_tilde[0]))
    # no sink / local tokens: the pseudo-max is -inf, so the threshold keeps every block and the
    # result equals delta = +inf
    inf = _decode(inp, qk, w, math.inf)
    np.testing.assert_array_equal(res.out, inf.out)
    assert res.mask[2, 0, :2].all() and res.mask[1, 0, 0]


def test_sm_scale_is_applied_to_every_score():
    """Doubling q and halving sm leaves every fp64 score bit-identical (powers of two)."""
    w, inp, qk = _setup(batch=1, hq=4, hkv=1, seq_lens=(400,), sink=4, local=16)
    a = _decode(inp, qk, w, 5.0, want_s_hat=True)
    q2 = (torch.as_tensor(inp.q_bits.view(np.int16)).view(torch.bfloat16) * 2).view(torch.int16) \
        .numpy().view(np.uint16)
    inp2 = ffd_synth.Inputs(**{**inp.__dict__, "q_bits": q2})
    b = oracle.decode(inp2.q_bits, inp2.seq_lens, inp2.block_table, qk, inp2.v_bits,
                      sink=w.sink, local=w.local, delta=5.0, sm_scale=SM / 2, threads=1,
                      want_s_hat=True)
    assert np.array_equal(a.out, b.out) and np.array_equal(a.mask, b.mask)
    assert np.array_equal(a.s_hat[(0, 0)], b.s_hat[(0, 0)])


def test_literal_workload_keeps_every_block():
    """Under the literal configuration-0 recipe background scores are ~N(0,1) and the pseudo-max
    is ~4, so with delta = 5 every 64-token block holds a token above m~ - delta."""
    w = ffd_synth.WORKLOADS[0]
    inp = ffd_synth.make_inputs(w)
    qk = oracle.quantize(inp.k_bits)
    res = oracle.decode(inp.q_bits, inp.seq_lens, inp.block_table, qk, inp.v_bits, sink=w.sink,
                        local=w.local, delta=5.0, sm_scale=SM)
    assert res.mask.all()
    assert np.all((res.m_tilde > 2.5) & (res.m_tilde < 6))


def _plant(inp, b, h, j, vec):
    """Overwrite the bf16 key of token j (sequence b, KV head h) with ``vec``."""
    page = int(inp.block_table[b, j // 64])
    inp.k_bits[page, h, j % 64] = torch.as_tensor(_bf16(vec)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def test_keep_rule_is_inclusive():
    """A block whose best provisional score equals m~ - delta exactly is kept (the rule is >=).
    delta is chosen as m~ - s^max of one block; both differences are exact in fp64 by Sterbenz's
    lemma (the operands are within a factor of two), so the block's margin is exactly 0."""
    w, inp, qk = _setup(batch=1, hq=1, hkv=1, seq_lens=(2000,), sink=16, local=64, needles=0,
                        peaked=False)
    probe = _decode(inp, qk, w, 5.0, want_s_hat=True)
    mt = float(probe.m_tilde[0, 0])
    sh = probe.s_hat[(0, 0)][0]
    forced = R.forced_blocks(2000, w.sink, w.local)
    tested = 0
    for blk in range(31):
        if blk in forced:
            continue
        smax = float(sh[blk * 64:(blk + 1) * 64].max())
        if not (mt / 2 <= smax <= mt):
            continue
        delta = mt - smax
        if mt - delta != smax:
            continue
        res = _decode(inp, qk, w, delta)
        assert res.margin[0, 0, blk] == 0.0
        assert res.mask[0, 0, blk] == 1
        tested += 1
        if tested == 3:
            break
    assert tested >= 1


@pytest.mark.parametrize("where", ["last_sink", "first_local", "before_local", "first_mid"])
def test_pseudo_max_window_edges(where):
    """m~ takes exactly the tokens j < S and j >= n - L: a planted peak on the window's edge
    raises it, one just outside does not."""
    n, S, L = 1000, 10, 100
    w, inp, qk = _setup(batch=1, hq=1, hkv=1, seq_lens=(n,), sink=S, local=L, needles=0,
                        peaked=False)
    q = R.bf16_bits_to_f64(inp.q_bits[0, 0])
    j = {"last_sink": S - 1, "first_local": n - L, "before_local": n - L - 1, "first_mid": S}[where]
    _plant(inp, 0, 0, j, q * (30.0 / SM / float(q @ q)))
    qk = oracle.quantize(inp.k_bits, threads=1)
    res = _decode(inp, qk, w, 5.0, want_s_hat=True)
    x2, kh = R.sequence_rows(qk, inp.block_table, 0, 0, n)
    s_peak = SM * float(q @ kh[j].astype(np.float64))
    inside = where in ("last_sink", "first_local")
    assert (abs(res.m_tilde[0, 0] - s_peak) < 1e-9) == inside
    _, mt, _, _ = R.bruteforce_mask(q[None], x2.astype(np.float64), kh.astype(np.float64), n, S,
                                    L, 5.0, SM)
    assert abs(res.m_tilde[0, 0] - mt[0]) < 1e-12


@pytest.mark.parametrize("target", [2.6, 2.8, 3.0])
def test_each_head_uses_its_own_threshold(target):
    """Heads of one GQA group carry their own pseudo-max and threshold: with head 1's query
    scaled by 4 (exact in bf16) its scores and m~ are 4x head 0's, and the block mask is the
    union of two different per-head masks, checked against the token-by-token definition.
    delta is set so that head 0's threshold m~_0 - delta sits at ``target`` (background block
    maxima are ~2-3 there), which makes the mask non-trivial whatever the random draw."""
    w, inp, qk = _setup(batch=1, hq=2, hkv=1, seq_lens=(3000,), sink=16, local=64, needles=0,
                        peaked=False)
    qb = torch.as_tensor(inp.q_bits.view(np.int16)).view(torch.bfloat16).clone()
    qb[0, 1] = qb[0, 0] * 4
    inp.q_bits[:] = qb.view(torch.int16).numpy().view(np.uint16)
    delta = float(_decode(inp, qk, w, 5.0).m_tilde[0, 0]) - target
    res = _decode(inp, qk, w, delta)
    x2, kh = R.sequence_rows(qk, inp.block_table, 0, 0, 3000)
    q = R.bf16_bits_to_f64(inp.q_bits[0])
    mask, mt, sh, mg = R.bruteforce_mask(q, x2.astype(np.float64), kh.astype(np.float64), 3000,
                                         16, 64, delta, SM)
    np.testing.assert_allclose(res.m_tilde[0], mt, rtol=1e-13)
    assert abs(mt[1] - 4 * mt[0]) < 1e-9
    # the test is sensitive: thresholding head 1 with head 0's m~ would keep other blocks
    forced = R.forced_blocks(3000, 16, 64)
    wrong = np.array([blk in forced or bool((sh[:, blk * 64:(blk + 1) * 64] >= mt[0] - delta)
                                            .any()) for blk in range(47)])
    assert not np.array_equal(wrong, mask)
    clear = ~(np.abs(mg) < 1e-9)
    assert np.array_equal(res.mask[0, 0, :47].astype(bool)[clear], mask[clear])
    assert 0 < mask.sum() < 47


def test_signed_zero_extremes_count_as_plus_zero():
    """Whichever zero comes first, a zero minimum gives zero = +0 (bits 0x0000)."""
    for first in (-0.0, 0.0):
        x = np.zeros(32, np.float32)
        x[0] = first
        x[1] = -first
        x[2:] = 1.0
        c2, ts, tz, c8, rs, _ = oracle.quantize_group(x)
        assert tz == 0x0000 and ts == int(np.float32(1 / 3).astype(np.float16).view(np.uint16))
