"""Failure detection on the GPU without a fault: a device wait that runs out.

Every wait inside the library's kernels (a copy landing, another warp's or another CTA's result)
is bounded; past the bound the CTA sets FFD_ERRBIT_TIMEOUT in the workspace's error word, stops
waiting, drains its own copies and ends, so the context stays usable. Here the wait is made to run
out on purpose, with no fault: the workspace's per-unit counters are pre-filled with large negative
values, so the count of published stage-1 slots that the scan warps wait for (the pseudo-max of a
unit, Methodology §2) never reaches its target. The bound is set to 1 ms for this call; the call
must end quickly, report FFD_ERR_TIMEOUT, and the next call on a zero-filled workspace must be
correct again.
"""
import numpy as np
import pytest
import torch

import ffd_synth
import oracle
import sparse_quantized_attention_gb300 as ffd
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu


def _decode(p, inp, dev, qc, ws):
    w = inp.workload
    out = torch.empty((w.batch, w.num_q_heads, 128), dtype=torch.float32, device="cuda")
    mask = torch.zeros((w.batch, w.num_kv_heads, inp.max_blocks), dtype=torch.uint8,
                       device="cuda")
    mt = torch.empty((w.batch, w.num_q_heads), dtype=torch.float32, device="cuda")
    ffd.ffd_decode_attention(p, dev["q"], qc, dev["v"], dev["seq_lens"], dev["block_table"],
                             out, ws, keep_mask=mask, m_tilde=mt)
    return out, mask, mt


@pytest.mark.parametrize("num_splits", [0, 4])
def test_wait_runs_out_and_the_next_call_is_correct(num_splits):
    w = ffd_synth.custom(2, 8, 2, 3000, sink=64, local=256, seed=11)
    inp = ffd_synth.make_inputs(w)
    dev = H.to_device(inp)
    qc = H.quantize(dev)
    p = ffd.make_params(w.batch, w.num_q_heads, w.num_kv_heads, inp.num_pages, inp.max_blocks,
                        sink=w.sink, local=w.local, delta=5.0, sm_scale=H.SM,
                        num_splits=num_splits, wait_limit_us=1000)
    ws = ffd.alloc_workspace(p)
    ws.fill_(0x80)   # every counter reads as -2^31 + ...: no count of slots ever reaches its target
    ws[:256].zero_()  # the error word starts clear
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    _decode(p, inp, dev, qc, ws)
    e1.record()
    torch.cuda.synchronize()
    assert ffd.ffd_get_error(ws) == 7          # FFD_ERR_TIMEOUT, read and cleared
    assert e0.elapsed_time(e1) < 1000.0        # ms: the waits ended near their 1 ms bound
    # the context is usable and a zero-filled workspace decodes correctly
    ws.zero_()
    out, mask, mt = _decode(p, inp, dev, qc, ws)
    got = {"out": out.cpu().numpy(), "mask": mask.cpu().numpy(), "m_tilde": mt.cpu().numpy(),
           "err": ffd.ffd_get_error(ws)}
    H.check_decode(inp, oracle.quantize(inp.k_bits), got, 5.0, what="after a timeout")


def test_default_bound_does_not_fire():
    """wait_limit_us = 0 keeps the 2 s default: a normal call reports nothing."""
    w = ffd_synth.custom(1, 4, 1, 2000, sink=16, local=64, seed=12)
    inp = ffd_synth.make_inputs(w)
    dev = H.to_device(inp)
    qc = H.quantize(dev)
    p = ffd.make_params(w.batch, w.num_q_heads, w.num_kv_heads, inp.num_pages, inp.max_blocks,
                        sink=w.sink, local=w.local, delta=5.0, sm_scale=H.SM)
    assert p.wait_limit_us == 0
    ws = ffd.alloc_workspace(p)
    _decode(p, inp, dev, qc, ws)
    assert ffd.ffd_get_error(ws) == 0
