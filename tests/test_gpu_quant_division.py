"""The quantiser divides the group range by 3 and the residual maximum by 127 with a precomputed
reciprocal and one fused multiply-add correction instead of an IEEE division; the records stay
bit-exact only if that quotient is the IEEE one. This checks it for every finite non-negative
fp32 value (the domain of both dividends) on the GPU, against CUDA's __fdiv_rn."""
import ctypes
import os
import subprocess

import pytest

from sparse_quantized_attention_gb300 import _build

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.gpu
def test_division_by_constant_equals_ieee_division(tmp_path):
    lib = str(tmp_path / "libdivcheck.so")
    subprocess.run([_build.nvcc(), *_build.ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
                    "-I", _build.INCLUDE, "-I", _build.CSRC, "-shared", "-cudart", "static",
                    os.path.join(HERE, "quant_division_check.cu"), "-o", lib], check=True)
    dll = ctypes.CDLL(lib)
    bad = (ctypes.c_ulonglong * 2)()
    first = (ctypes.c_uint * 2)()
    assert dll.ffd_check_division(bad, first) == 0
    assert (bad[0], bad[1]) == (0, 0), (list(bad), [hex(v) for v in first])
