"""Rows of a sequence's last page past its length hold whatever the cache holds there. They must
not reach the output: NaN in those V rows (and, for the dense path, K rows) must give results
bit-identical to a clean cache, for the decode step, the dense kernel, attention over a given mask
and ART. (A zero probability times a NaN is a NaN, so the kernels must zero those rows, not rely
on the probability alone.)"""
import numpy as np
import pytest
import torch

import ffd_synth
import sparse_quantized_attention_gb300 as ffd
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu

LENS = [700, 129, 1000]  # partial last pages: 60, 1 and 40 rows


@pytest.fixture(scope="module")
def setup():
    w = ffd_synth.custom(3, 16, 2, 700, seed=61)
    inp = ffd_synth.make_inputs(w, seq_lens=LENS)
    dev = H.to_device(inp)
    qc = H.quantize(dev)  # keys quantised while the cache is clean
    dirty = {k: v.clone() for k, v in dev.items()}
    nan = torch.tensor(float("nan"), dtype=torch.bfloat16, device="cuda")
    for b, n in enumerate(LENS):
        page = int(inp.block_table[b, (n - 1) // 64])
        rows = n % 64
        if rows:
            dirty["v"][page, :, rows:, :] = nan
            dirty["k"][page, :, rows:, :] = nan
    return inp, dev, dirty, qc


def _decode(inp, d, qc, keep_in=None):
    w = inp.workload
    p = H.params_for(inp, 5.0)
    out = torch.empty((w.batch, w.num_q_heads, 128), device="cuda")
    ws = ffd.alloc_workspace(p)
    if keep_in is None:
        ffd.ffd_decode_attention(p, d["q"], qc, d["v"], d["seq_lens"], d["block_table"], out, ws)
    else:
        ffd.ffd_decode_attention_masked(p, d["q"], qc, d["v"], d["seq_lens"], d["block_table"],
                                        keep_in, out, ws)
    assert ffd.ffd_get_error(ws) == 0
    return out.cpu().numpy()


def test_decode_ignores_rows_past_the_sequence(setup):
    inp, clean, dirty, qc = setup
    a, b = _decode(inp, clean, qc), _decode(inp, dirty, qc)
    assert np.isfinite(b).all()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_masked_decode_ignores_rows_past_the_sequence(setup):
    inp, clean, dirty, qc = setup
    w = inp.workload
    keep = torch.ones((w.batch, w.num_kv_heads, inp.max_blocks), dtype=torch.uint8, device="cuda")
    a, b = _decode(inp, clean, qc, keep), _decode(inp, dirty, qc, keep)
    assert np.isfinite(b).all()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_dense_ignores_rows_past_the_sequence(setup):
    inp, clean, dirty, _ = setup
    a, b = H.dense(inp, clean), H.dense(inp, dirty)
    assert np.isfinite(b).all()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_art_ignores_rows_past_the_sequence(setup):
    inp, clean, dirty, qc = setup
    w = inp.workload
    p = H.params_for(inp, 5.0)
    res = []
    for d in (clean, dirty):
        ws = ffd.alloc_art_workspace(p)
        out = torch.empty((w.batch, w.num_q_heads, 128), device="cuda")
        ffd.ffd_art_attention(p, 0.0, 0.0, 1, d["q"], qc, d["v"], d["seq_lens"],
                              d["block_table"], out, ws)
        assert ffd.ffd_get_error(ws) == 0
        res.append(out.cpu().numpy())
    assert np.isfinite(res[1]).all()
    assert np.array_equal(res[0].view(np.uint32), res[1].view(np.uint32))
