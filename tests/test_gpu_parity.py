"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle on seeded inputs.

Runs on a GB300 (`pytest -m gpu`). The five workloads run at their full sizes: every output, every
mask bit and every quantised byte is compared.
"""
import math

import numpy as np
import pytest
import torch

import ffd_synth
import oracle
import sparse_quantized_attention_gb300 as ffd
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu

_cache = {}


def _workload(cid, peaked=False):
    key = (cid, peaked)
    if key not in _cache:
        _cache.clear()
        torch.cuda.empty_cache()
        w = ffd_synth.WORKLOADS[cid]
        inp = ffd_synth.make_inputs(w, signal_scale=ffd_synth.peaked_scale() if peaked else 1.0)
        dev = H.to_device(inp)
        qc = H.quantize(dev)
        ref = oracle.quantize(inp.k_bits)
        _cache[key] = (inp, dev, qc, ref)
    return _cache[key]


@pytest.mark.parametrize("cid", [0, 1, 2, 3, 4])
def test_quantize_bit_exact(cid):
    inp, dev, qc, ref = _workload(cid)
    H.assert_cache_equal(H.cache_to_host(qc), ref)


CASES = [(0, 5.0, False), (0, 5.0, True), (1, 5.0, False), (1, 7.0, False), (1, 5.0, True),
         (2, 5.0, False), (2, 5.0, True), (3, 5.0, False), (3, 7.0, False), (3, 7.0, True),
         (4, 5.0, False), (4, 5.0, True)]


@pytest.mark.parametrize("cid,delta,peaked", CASES)
def test_decode_parity_full_size(cid, delta, peaked):
    inp, dev, qc, ref = _workload(cid, peaked)
    gpu = H.decode(inp, dev, qc, delta)
    st = H.check_decode(inp, ref, gpu, delta, what=f"cfg{cid} delta={delta} peaked={peaked}")
    print(f"cfg{cid} delta={delta} peaked={peaked}: kept {st['kept']}/{st['blocks']} blocks, "
          f"borderline {st['borderline']}, mask diffs {st['mask_diffs']}, "
          f"max-abs {st['max_abs']:.2e}, rel-L2 {st['rel_l2']:.2e}")


@pytest.mark.parametrize("cid", [0, 1, 2, 3, 4])
def test_dense_parity(cid):
    inp, dev, qc, ref = _workload(cid)
    w = inp.workload
    units = [(b, h) for b in range(w.batch) for h in range(w.num_kv_heads)]
    if cid == 4:
        units = units[::9]
    want = oracle.dense(inp.q_bits, inp.seq_lens, inp.block_table, inp.k_bits, inp.v_bits,
                        sm_scale=H.SM, units=units)
    got = H.dense(inp, dev)
    G = w.num_q_heads // w.num_kv_heads
    sel = np.zeros(got.shape[:2], bool)
    for (b, h) in units:
        sel[b, h * G:(h + 1) * G] = True
    st = H.compare_outputs(got[sel], want[sel], f"dense cfg{cid}")
    print(f"dense cfg{cid}: max-abs {st['max_abs']:.2e} rel-L2 {st['rel_l2']:.2e}")


# ------------------------------------------------------------------------------------------- #
# Edge cases: ragged and tiny lengths, every GQA group size, empty windows, split counts       #
# ------------------------------------------------------------------------------------------- #

EDGE = [
    dict(batch=4, hq=1, hkv=1, seq_lens=(0, 1, 63, 64), sink=4, local=8),
    dict(batch=3, hq=2, hkv=1, seq_lens=(65, 127, 129), sink=0, local=16),
    dict(batch=2, hq=3, hkv=1, seq_lens=(300, 1000), sink=16, local=0),
    dict(batch=2, hq=8, hkv=2, seq_lens=(777, 2049), sink=64, local=256),
    dict(batch=2, hq=5, hkv=1, seq_lens=(4000, 333), sink=3, local=70),
    dict(batch=1, hq=12, hkv=2, seq_lens=(5000,), sink=0, local=0),
    dict(batch=2, hq=7, hkv=1, seq_lens=(6000, 6001), sink=64, local=1024),
    dict(batch=3, hq=16, hkv=2, seq_lens=(2000, 64, 3100), sink=128, local=100),
]


@pytest.mark.parametrize("shape", EDGE, ids=[f"edge{i}" for i in range(len(EDGE))])
@pytest.mark.parametrize("delta", [0.0, 5.0, math.inf])
@pytest.mark.parametrize("peaked", [False, True])
def test_decode_edge_cases(shape, delta, peaked):
    shape = dict(shape)
    lens = shape.pop("seq_lens")
    w = ffd_synth.custom(shape.pop("batch"), shape.pop("hq"), shape.pop("hkv"), max(lens),
                         random_pages=True, needles=3, seed=len(lens) * 101 + max(lens),
                         **shape)
    inp = ffd_synth.make_inputs(w, seq_lens=list(lens),
                                signal_scale=ffd_synth.peaked_scale() if peaked else 1.0)
    dev = H.to_device(inp)
    qc = H.quantize(dev)
    ref = oracle.quantize(inp.k_bits)
    H.assert_cache_equal(H.cache_to_host(qc), ref)
    for splits in (0, 1, 3):
        gpu = H.decode(inp, dev, qc, delta, num_splits=splits)
        H.check_decode(inp, ref, gpu, delta, what=f"{w.name} splits={splits}")


@pytest.mark.parametrize("shape", EDGE, ids=[f"edge{i}" for i in range(len(EDGE))])
def test_dense_edge_cases(shape):
    """The dense comparison kernel at every GQA group size 1 ... 8 (odd ones included), ragged and
    empty sequences, random block tables, and split counts 0 (one per SM), 1 and 3."""
    shape = dict(shape)
    lens = shape.pop("seq_lens")
    w = ffd_synth.custom(shape.pop("batch"), shape.pop("hq"), shape.pop("hkv"), max(lens),
                         random_pages=True, needles=3, seed=len(lens) * 211 + max(lens),
                         **shape)
    inp = ffd_synth.make_inputs(w, seq_lens=list(lens))
    dev = H.to_device(inp)
    want = oracle.dense(inp.q_bits, inp.seq_lens, inp.block_table, inp.k_bits, inp.v_bits,
                        sm_scale=H.SM)
    for splits in (0, 1, 3):
        got = H.dense(inp, dev, num_splits=splits)
        H.compare_outputs(got, want, f"dense {w.name} splits={splits}")


def test_split_count_invariance_and_determinism():
    inp, dev, qc, ref = _workload(1)
    base = H.decode(inp, dev, qc, 5.0)
    again = H.decode(inp, dev, qc, 5.0)
    assert np.array_equal(base["out"], again["out"]) and np.array_equal(base["mask"], again["mask"])
    for splits in (1, 2, 5, 64, 512):
        other = H.decode(inp, dev, qc, 5.0, num_splits=splits)
        assert np.array_equal(other["mask"], base["mask"])
        np.testing.assert_allclose(other["out"], base["out"], rtol=0, atol=2e-6)


def test_quantize_special_groups():
    """Golden groups, signed zeros, constant groups, fp16-subnormal ranges and ties, on the GPU."""
    rng = np.random.default_rng(5)
    k = rng.standard_normal((4, 2, 64, 128)).astype(np.float32)
    k[0, 0, 0, :32] = [-1, 0, 1, 2] * 8
    k[0, 0, 1, :32] = 0.0
    k[0, 0, 1, :6] = [0, 3, 0.25, 1.5, 2.5, 0.5]
    k[0, 0, 2, :32] = -1
    k[0, 0, 2, :3] = [-1, 1, 0]
    k[0, 0, 3, :32] = 0.30078125
    k[0, 1, 0, :32] = -0.0
    k[0, 1, 0, 5] = 0.0
    k[0, 1, 1, :32] = rng.standard_normal(32) * 1e-6
    k[0, 1, 2, :32] = 1.0 + rng.integers(0, 4, 32) * 2.0 ** -7
    k[1] = rng.standard_normal((2, 64, 128)) * np.exp2(rng.integers(-20, 12, (2, 64, 1)))
    k[2] = np.round(rng.standard_normal((2, 64, 128)) * 4) / 4
    bits = torch.from_numpy(k).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    qc_ref = oracle.quantize(bits)
    dev_k = H.bits_to_bf16(bits)
    qc = ffd.alloc_quantized_cache(4, 2)
    ffd.ffd_quantize_keys(dev_k, qc)
    H.assert_cache_equal(H.cache_to_host(qc), qc_ref)


def test_quantize_selected_pages_and_errors():
    rng = np.random.default_rng(6)
    k = torch.from_numpy(rng.standard_normal((6, 2, 64, 128)).astype(np.float32)) \
        .to(torch.bfloat16)
    bits = k.view(torch.int16).numpy().view(np.uint16)
    ref = oracle.quantize(bits)
    dev_k = k.cuda()
    qc = ffd.alloc_quantized_cache(6, 2)
    for t in qc:
        t.zero_()
    ids = torch.tensor([4, 1], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ffd.ffd_quantize_keys(dev_k, qc, page_ids=ids, error_word=err)
    assert ffd.ffd_get_error(err) == 0
    host = H.cache_to_host(qc)
    for name in ("thumb", "t_scale", "t_zero", "resid", "r_scale"):
        got, want = getattr(host, name), getattr(ref, name)
        assert np.array_equal(got[[1, 4]], want[[1, 4]])
        assert not got[[0, 2, 3, 5]].any()
    # an out-of-range page id is skipped and reported
    ffd.ffd_quantize_keys(dev_k, qc, page_ids=torch.tensor([2, 9], dtype=torch.int32,
                                                            device="cuda"), error_word=err)
    assert ffd.ffd_get_error(err) == 5  # FFD_ERR_BOUNDS
    assert ffd.ffd_get_error(err) == 0  # cleared
    # a key outside the fp16 range is reported
    k2 = dev_k.clone()
    k2[3, 1, 5, 77] = 1.0e6
    ffd.ffd_quantize_keys(k2, qc, error_word=err)
    assert ffd.ffd_get_error(err) == 6  # FFD_ERR_RANGE


def test_decode_reports_bad_block_table_entry():
    w = ffd_synth.custom(2, 4, 2, 700, sink=16, local=64, seed=3)
    inp = ffd_synth.make_inputs(w, seq_lens=[700, 500])
    dev = H.to_device(inp)
    qc = H.quantize(dev)
    bt = dev["block_table"].clone()
    bt[1, 3] = inp.num_pages + 5   # a page that does not exist
    dev2 = dict(dev, block_table=bt)
    got = H.decode(inp, dev2, qc, 5.0)
    assert got["err"] == 5          # FFD_ERR_BOUNDS, read and cleared
    assert got["mask"][1, 0, 3] == 0
    # sequence 0 is untouched by the bad entry
    ref = oracle.quantize(inp.k_bits)
    again = H.decode(inp, dev, qc, 5.0)
    np.testing.assert_array_equal(got["out"][0], again["out"][0])
    H.check_decode(inp, ref, again, 5.0, what="clean rerun")
