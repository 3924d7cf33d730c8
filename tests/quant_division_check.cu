// Exhaustive check of the quantiser's division by a constant (quant.cuh, div_const) against the
// IEEE division __fdiv_rn, for b = 3 and b = 127 and every finite non-negative fp32 x. Built and
// loaded by tests/test_gpu_quant_division.py.
#include <cuda_runtime.h>
#include <stdint.h>

#include "quant.cuh"

namespace {

__global__ void check_kernel(unsigned long long *bad, unsigned int *first) {
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < 0x7F800000ull;
         i += stride) {
        const float x = __uint_as_float((unsigned int)i);
        const float a3 = ffd::quant::div_const(x, 3.0f, ffd::quant::kThird);
        const float a127 = ffd::quant::div_const(x, 127.0f, ffd::quant::kInv127);
        if (__float_as_uint(a3) != __float_as_uint(__fdiv_rn(x, 3.0f))) {
            atomicAdd(&bad[0], 1ull);
            atomicMin(&first[0], (unsigned int)i);
        }
        if (__float_as_uint(a127) != __float_as_uint(__fdiv_rn(x, 127.0f))) {
            atomicAdd(&bad[1], 1ull);
            atomicMin(&first[1], (unsigned int)i);
        }
    }
}

}  // namespace

// Mismatch counts and the first mismatching bit pattern per divisor (0xffffffff: none), into
// host arrays of two entries each. Returns a cudaError_t.
extern "C" int ffd_check_division(unsigned long long *host_bad, unsigned int *host_first) {
    unsigned long long *bad = nullptr;
    unsigned int *first = nullptr;
    cudaError_t e = cudaMalloc(&bad, 2 * sizeof(unsigned long long));
    if (e != cudaSuccess) return (int)e;
    e = cudaMalloc(&first, 2 * sizeof(unsigned int));
    if (e == cudaSuccess) e = cudaMemset(bad, 0, 2 * sizeof(unsigned long long));
    if (e == cudaSuccess) e = cudaMemset(first, 0xff, 2 * sizeof(unsigned int));
    if (e == cudaSuccess) {
        check_kernel<<<1216, 256>>>(bad, first);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaMemcpy(host_bad, bad, 2 * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(host_first, first, 2 * sizeof(unsigned int), cudaMemcpyDeviceToHost);
    cudaFree(bad);
    cudaFree(first);
    return (int)e;
}
