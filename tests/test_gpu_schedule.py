"""The scan-then-refine schedule of the decode step against the CPU oracle.

FFD_SCHEDULE_SCAN_REFINE computes the same step as the fused schedule in another order: every CTA
scans an equal share of all thumbnails and keeps, per block and head, the maximum provisional
score; after a grid-wide barrier the kept blocks of all CTAs are shared out equally for the
refinement. Its masks must equal the fused schedule's bit for bit (both compare the same fp32
scores with the thresholds), and its outputs must meet the parity tolerances against the fp64
oracle, at full size on the five workloads and on the edge shapes (every GQA group size, ragged
and empty sequences, delta = 0 / 5 / +inf, split counts).
"""
import math

import numpy as np
import pytest

import ffd_synth
import oracle
from tests import gpu_harness as H
from tests.test_gpu_parity import CASES, EDGE, _workload

pytestmark = pytest.mark.gpu

SCAN_REFINE = 1


@pytest.mark.parametrize("cid,delta,peaked", CASES)
def test_scan_refine_full_size(cid, delta, peaked):
    inp, dev, qc, ref = _workload(cid, peaked)
    fused = H.decode(inp, dev, qc, delta)
    got = H.decode(inp, dev, qc, delta, schedule=SCAN_REFINE)
    assert got["err"] == 0 and fused["err"] == 0
    assert np.array_equal(got["mask"], fused["mask"]), "masks differ between the schedules"
    np.testing.assert_allclose(got["m_tilde"], fused["m_tilde"], rtol=0, atol=0)
    st = H.check_decode(inp, ref, got, delta, what=f"scan-refine cfg{cid} delta={delta}")
    print(f"scan-refine cfg{cid} delta={delta} peaked={peaked}: kept {st['kept']}/{st['blocks']}"
          f", max-abs {st['max_abs']:.2e}, rel-L2 {st['rel_l2']:.2e}")


@pytest.mark.parametrize("shape", EDGE, ids=[f"edge{i}" for i in range(len(EDGE))])
@pytest.mark.parametrize("delta", [0.0, 5.0, math.inf])
@pytest.mark.parametrize("peaked", [False, True])
def test_scan_refine_edge_cases(shape, delta, peaked):
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
    for splits in (0, 1, 3):
        got = H.decode(inp, dev, qc, delta, num_splits=splits, schedule=SCAN_REFINE)
        H.check_decode(inp, ref, got, delta, what=f"scan-refine {w.name} splits={splits}")


def test_scan_refine_repeats_and_alternates_buffers():
    """Calls on one workspace alternate the per-unit kept-count buffers: three calls in a row, and
    a fused call in between, give the same result."""
    inp, dev, qc, ref = _workload(1, True)
    first = H.decode(inp, dev, qc, 5.0, schedule=SCAN_REFINE)
    p = H.params_for(inp, 5.0, schedule=SCAN_REFINE)
    import sparse_quantized_attention_gb300 as ffd
    import torch
    ws = ffd.alloc_workspace(p)
    outs = []
    scheds = (SCAN_REFINE, SCAN_REFINE, 0, SCAN_REFINE)
    for sched in scheds:
        q = H.params_for(inp, 5.0, schedule=sched)
        out = torch.empty((inp.workload.batch, inp.workload.num_q_heads, 128),
                          dtype=torch.float32, device="cuda")
        ffd.ffd_decode_attention(q, dev["q"], qc, dev["v"], dev["seq_lens"],
                                 dev["block_table"], out, ws)
        assert ffd.ffd_get_error(ws) == 0
        outs.append(out.cpu().numpy())
    for sched, o in zip(scheds, outs):
        if sched == SCAN_REFINE:
            # the same kept list, shares and group of every block: the same sums in the same order
            np.testing.assert_array_equal(o, first["out"])
        else:
            # the fused schedule splits the units differently: equal up to rounding
            np.testing.assert_allclose(o, first["out"], rtol=0, atol=H.OUT_MAX_ABS)


def test_scan_refine_reports_bad_block_table_entry():
    w = ffd_synth.custom(2, 4, 2, 700, sink=16, local=64, seed=3)
    inp = ffd_synth.make_inputs(w, seq_lens=[700, 500])
    dev = H.to_device(inp)
    qc = H.quantize(dev)
    bt = dev["block_table"].clone()
    bt[1, 3] = inp.num_pages + 5
    got = H.decode(inp, dict(dev, block_table=bt), qc, 5.0, schedule=SCAN_REFINE)
    assert got["err"] == 5
    assert got["mask"][1, 0, 3] == 0
    again = H.decode(inp, dev, qc, 5.0, schedule=SCAN_REFINE)
    # the other sequence is untouched up to rounding: the kept blocks of all units are shared out
    # to the CTAs in equal runs, so the dropped block moves the runs' boundaries and with them the
    # order in which sequence 0's blocks are summed
    np.testing.assert_allclose(got["out"][0], again["out"][0], rtol=0, atol=2e-6)
    H.check_decode(inp, oracle.quantize(inp.k_bits), again, 5.0, what="clean rerun")


@pytest.mark.gpu
def test_suggest_schedule_on_this_device():
    import torch
    import sparse_quantized_attention_gb300 as ffd
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    total = 64 * sms
    assert ffd.ffd_suggest_schedule(total, total // 2 - 1) == ffd.SCHEDULE_SCAN_REFINE
    assert ffd.ffd_suggest_schedule(total, total // 2) == ffd.SCHEDULE_FUSED
    assert ffd.ffd_suggest_schedule(total - 1, 0) == ffd.SCHEDULE_FUSED  # too few blocks per SM
    assert ffd.ffd_suggest_schedule(1 << 40, 1 << 20) == ffd.SCHEDULE_SCAN_REFINE
