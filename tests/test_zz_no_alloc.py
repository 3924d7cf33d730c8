"""The allocation-free decode entry point, checked against the workspace entry point.

ffd_decode_attention_static serves callers that cannot allocate device memory for a workspace
(a plain C host that links only libffd.so, or a serving loop whose device memory is all committed
to its KV-cache pool): it runs the same kernels with a 4 MiB static scratch array inside the
library. This file is collected last, so a failure here leaves every other test already run; it
also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import ffd_synth
import oracle
import sparse_quantized_attention_gb300 as ffd
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu


def _static_decode(inp, dev, qc, delta):
    w = inp.workload
    p = H.params_for(inp, delta)
    d = dev["q"].device
    out = torch.full((w.batch, w.num_q_heads, 128), float("nan"), dtype=torch.float32, device=d)
    mask = torch.full((w.batch, w.num_kv_heads, inp.max_blocks), 7, dtype=torch.uint8, device=d)
    mt = torch.full((w.batch, w.num_q_heads), float("nan"), dtype=torch.float32, device=d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    ffd.ffd_decode_attention_static(p, dev["q"], qc, dev["v"], dev["seq_lens"],
                                    dev["block_table"], out, keep_mask=mask, m_tilde=mt,
                                    error_word=err)
    return {"out": out.cpu().numpy(), "mask": mask.cpu().numpy(), "m_tilde": mt.cpu().numpy(),
            "err": ffd.ffd_get_error(err)}


CASES = [
    ("tiny-4k", lambda: (ffd_synth.WORKLOADS[0], None, 1.0)),
    ("tiny-4k-peaked", lambda: (ffd_synth.WORKLOADS[0], None, ffd_synth.peaked_scale())),
    ("ragged-paged-g7", lambda: (ffd_synth.custom(3, 14, 2, 3000, sink=16, local=200,
                                                  random_pages=True, seed=5),
                                 [3000, 1, 777], ffd_synth.peaked_scale())),
    ("batched-paged-32x-4k-16k", lambda: (ffd_synth.WORKLOADS[4], None, 1.0)),
]


@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
def test_static_scratch_matches_workspace_path_twice(name, make):
    w, lens, scale = make()
    inp = ffd_synth.make_inputs(w, seq_lens=lens, signal_scale=scale)
    dev = H.to_device(inp)
    qc = H.quantize(dev)
    ref = H.decode(inp, dev, qc, 5.0)
    assert ref["err"] == 0
    for call in range(2):  # the second call finds the first call's scratch contents
        got = _static_decode(inp, dev, qc, 5.0)
        assert got["err"] == 0, f"{name} call {call}: device error {got['err']}"
        assert np.array_equal(got["mask"], ref["mask"]), f"{name} call {call}: masks differ"
        np.testing.assert_allclose(got["m_tilde"], ref["m_tilde"], rtol=0, atol=0)
        H.compare_outputs(got["out"], ref["out"].astype(np.float64), f"{name} call {call}")
    # and both agree with the oracle
    H.check_decode(inp, oracle.quantize(inp.k_bits), got, 5.0, what=f"{name} static")


def test_static_scratch_rejects_oversized_problem():
    """A problem whose scratch would exceed the 4 MiB array is refused before any work."""
    w = ffd_synth.WORKLOADS[0]
    inp = ffd_synth.make_inputs(w)
    dev = H.to_device(inp)
    qc = H.quantize(dev)
    big = ffd.make_params(4096, 64, 8, inp.num_pages, inp.max_blocks, sink=64, local=256)
    assert ffd.ffd_decode_workspace_size(big) > 4 << 20
    out = torch.empty((4096, 64, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(ffd.FFDError) as e:
        ffd.ffd_decode_attention_static(big, dev["q"], qc, dev["v"], dev["seq_lens"],
                                        dev["block_table"], out)
    assert e.value.status == 3  # FFD_ERR_WORKSPACE


def test_static_scratch_without_error_word_matches_workspace_path():
    """error_word NULL: device errors go to the scratch's own word (cleared every call) and are not
    reported; the results equal the workspace path's, in both schedules."""
    w = ffd_synth.custom(3, 14, 2, 3000, sink=16, local=200, random_pages=True, seed=9)
    inp = ffd_synth.make_inputs(w, seq_lens=[3000, 1, 777], signal_scale=ffd_synth.peaked_scale())
    dev = H.to_device(inp)
    qc = H.quantize(dev)
    for schedule in (0, 1):
        ref = H.decode(inp, dev, qc, 5.0, schedule=schedule)
        p = H.params_for(inp, 5.0, schedule=schedule)
        out = torch.full((w.batch, w.num_q_heads, 128), float("nan"), dtype=torch.float32,
                         device="cuda")
        mask = torch.full((w.batch, w.num_kv_heads, inp.max_blocks), 7, dtype=torch.uint8,
                          device="cuda")
        ffd.ffd_decode_attention_static(p, dev["q"], qc, dev["v"], dev["seq_lens"],
                                        dev["block_table"], out, keep_mask=mask)
        torch.cuda.synchronize()
        assert np.array_equal(mask.cpu().numpy(), ref["mask"])
        H.compare_outputs(out.cpu().numpy(), ref["out"].astype(np.float64),
                          f"static, no error word, schedule {schedule}")


def test_static_scratch_reports_bad_block_table_entry():
    """An out-of-range block-table entry through the static entry point: FFD_ERR_BOUNDS from the
    caller's error word, the entry's block dropped, and a clean call afterwards is correct."""
    w = ffd_synth.custom(2, 4, 2, 700, sink=16, local=64, seed=3)
    inp = ffd_synth.make_inputs(w, seq_lens=[700, 500])
    dev = H.to_device(inp)
    qc = H.quantize(dev)
    bt = dev["block_table"].clone()
    bt[1, 3] = inp.num_pages + 5
    got = _static_decode(inp, dict(dev, block_table=bt), qc, 5.0)
    assert got["err"] == 5  # FFD_ERR_BOUNDS
    assert got["mask"][1, 0, 3] == 0
    again = _static_decode(inp, dev, qc, 5.0)
    assert again["err"] == 0
    H.check_decode(inp, oracle.quantize(inp.k_bits), again, 5.0, what="static clean rerun")
