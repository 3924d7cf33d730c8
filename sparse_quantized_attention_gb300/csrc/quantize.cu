// quantize.cu -- split bf16 keys into the 2-bit thumbnail and the int8 residual.
//
// Source: "Faster Than Flash", Methodology §1 (content-aware scanning via low-bit quantization:
// the K cache is kept as 2-bit thumbnails for score estimation plus 8-bit residuals that rebuild
// the keys close to fp16 precision). The exact format, and the record layout each (page, KV head)
// tile is written in, are the ones stated in include/ffd.h.
//
// One warp quantises one token of one KV head: lane l holds channels 4l .. 4l+3, so a group of
// 32 channels is 8 lanes and group reductions are 3 shuffles. Every arithmetic step is a single
// IEEE fp32 operation with an explicit rounding intrinsic, so the outputs are bit-defined.
#include "common.cuh"

namespace ffd {

__device__ __forceinline__ float group8_min(float v) {
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float group8_max(float v) {
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__global__ void __launch_bounds__(256) quantize_keys_kernel(
    int P, int Hkv, int num_rows, const int32_t *__restrict__ page_ids,
    const __nv_bfloat16 *__restrict__ k, uint8_t *__restrict__ thumb, uint8_t *__restrict__ resid,
    int *err) {
    const int lane = threadIdx.x & 31;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (warp >= num_rows) return;  // warp-uniform
    // warp -> (tile, slot); tile -> (page, head)
    const int slot = warp % kPage;
    const int tile_local = warp / kPage;
    int page = tile_local / Hkv;
    const int h = tile_local % Hkv;
    if (page_ids) {
        page = page_ids[page];
        if (page < 0 || page >= P) {
            if (lane == 0 && slot == 0 && h == 0) raise_error(err, FFD_ERRBIT_BOUNDS);
            return;
        }
    }
    const int64_t tile = (int64_t)page * Hkv + h;
    const int64_t row = tile * kPage + slot;

    // 4 consecutive channels per lane (8 bytes of bf16)
    const uint2 raw = *reinterpret_cast<const uint2 *>(k + row * kD + 4 * lane);
    float x[4];
    x[0] = __uint_as_float(raw.x << 16);
    x[1] = __uint_as_float(raw.x & 0xffff0000u);
    x[2] = __uint_as_float(raw.y << 16);
    x[3] = __uint_as_float(raw.y & 0xffff0000u);

    bool bad = false;
#pragma unroll
    for (int c = 0; c < 4; c++) bad |= !(fabsf(x[c]) < 65504.0f);
    if (bad) raise_error(err, FFD_ERRBIT_RANGE);

    float mn = fminf(fminf(x[0], x[1]), fminf(x[2], x[3]));
    float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
    mn = group8_min(mn);
    mx = group8_max(mx);
    if (mn == 0.0f) mn = 0.0f;  // a signed-zero extreme counts as +0
    if (mx == 0.0f) mx = 0.0f;

    const __half zf16 = __float2half_rn(mn);
    const __half sf16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), 3.0f));
    const float zf = __half2float(zf16);
    const float sf = __half2float(sf16);

    uint32_t codes = 0;
    float r[4];
    float amax = 0.0f;
#pragma unroll
    for (int c = 0; c < 4; c++) {
        float code = 0.0f;
        if (sf != 0.0f) {
            code = rintf(__fdiv_rn(__fsub_rn(x[c], zf), sf));
            code = fminf(fmaxf(code, 0.0f), 3.0f);
        }
        codes |= (uint32_t)code << (2 * c);
        const float xh = __fmaf_rn(code, sf, zf);
        r[c] = __fsub_rn(x[c], xh);
        amax = fmaxf(amax, fabsf(r[c]));
    }
    amax = group8_max(amax);
    const __half sr16 = __float2half_rn(__fdiv_rn(amax, 127.0f));
    const float sr = __half2float(sr16);
    uint32_t packed = 0;
#pragma unroll
    for (int c = 0; c < 4; c++) {
        float q8 = 0.0f;
        if (sr != 0.0f) {
            q8 = rintf(__fdiv_rn(r[c], sr));
            q8 = fminf(fmaxf(q8, -127.0f), 127.0f);
        }
        packed |= ((uint32_t)(int)q8 & 0xffu) << (8 * c);
    }

    uint8_t *trec = thumb + tile * kThumbRec;
    uint8_t *rrec = resid + tile * kResidRec;
    trec[slot * kThumbRow + lane] = (uint8_t)codes;
    *reinterpret_cast<uint32_t *>(rrec + resid_offset(slot, 4 * lane)) = packed;
    if ((lane & 7) == 0) {
        const int g = lane >> 3;
        reinterpret_cast<__half *>(trec + kThumbScaleOff)[slot * kGroups + g] = sf16;
        reinterpret_cast<__half *>(trec + kThumbZeroOff)[slot * kGroups + g] = zf16;
        reinterpret_cast<__half *>(rrec + kResidScaleOff)[slot * kGroups + g] = sr16;
    }
}

cudaError_t launch_quantize(int P, int Hkv, const int32_t *page_ids, int num_pages_listed,
                            const void *k, uint8_t *thumb, uint8_t *resid, int *err,
                            cudaStream_t stream) {
    const int64_t rows = (int64_t)num_pages_listed * Hkv * kPage;
    if (rows == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = (rows * 32 + threads - 1) / threads;
    quantize_keys_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
        P, Hkv, (int)rows, page_ids, static_cast<const __nv_bfloat16 *>(k), thumb, resid, err);
    return cudaGetLastError();
}

}  // namespace ffd
