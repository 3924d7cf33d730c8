"""The library's CTA count (num_splits 0): one CTA per SM, or one per four blocks of
batch * num_kv_heads * max_blocks_per_seq when that is fewer. The workspace sizes tell which count
the library took (they hold a split record per unit and CTA, so they grow with the count), and a
step with the default count gives, bit for bit, the step with that count given explicitly."""
import numpy as np
import pytest
import torch

from sparse_quantized_attention_gb300 import ffd
from tests import gpu_harness as H
from tests.test_gpu_parity import _workload

pytestmark = pytest.mark.gpu


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _expected(batch, hkv, max_blocks):
    return min(_sms(), max(1, -(-batch * hkv * max_blocks // 4)))


@pytest.mark.parametrize("batch,hkv,max_blocks", [(1, 2, 64), (1, 8, 512), (4, 4, 2048), (3, 1, 1),
                                                  (2, 8, 30)])
def test_default_cta_count(batch, hkv, max_blocks):
    want = _expected(batch, hkv, max_blocks)
    for size in (ffd.ffd_decode_workspace_size, ffd.ffd_dense_workspace_size):
        def ws(splits):
            return size(ffd.make_params(batch, 4 * hkv, hkv, 100, max_blocks, sink=64,
                                        local=128, num_splits=splits))
        assert ws(0) == ws(want)
        if want < _sms():
            assert ws(want + 1) > ws(0)


def test_default_count_step_equals_explicit_count():
    inp, dev, qc, _ = _workload(0)  # 4K tokens, 2 KV heads: 128 blocks, 32 CTAs
    w = inp.workload
    want = _expected(w.batch, w.num_kv_heads, inp.max_blocks)
    assert want < _sms()
    for schedule in (0, 1):
        a = H.decode(inp, dev, qc, 5.0, schedule=schedule)
        b = H.decode(inp, dev, qc, 5.0, num_splits=want, schedule=schedule)
        assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["mask"], b["mask"])
    assert np.array_equal(H.dense(inp, dev), H.dense(inp, dev, num_splits=want))
