// quantize.cu -- split bf16 keys into the 2-bit thumbnail and the int8 residual.
//
// Source: "Faster Than Flash", Methodology §1 (content-aware scanning via low-bit quantization:
// the K cache is kept as 2-bit thumbnails for score estimation plus 8-bit residuals that rebuild
// the keys close to fp16 precision). The exact format, and the record layout each (page, KV head)
// tile is written in, are the ones stated in include/ffd.h.
//
// One CTA of 256 threads quantises one (page, KV head) tile: thread t owns token t / 4 and
// channel group t % 4, so the 32 channels that share a scale live in one thread and no group
// reduction crosses lanes. The thread loads its 64 bytes of keys with four 16-byte loads and
// writes its codes, its two 16-byte residual chunks and its three scales with vector stores; a
// warp covers 8 whole tokens, so every store of the tile's records is a full 32-byte sector.
//
// The per-group arithmetic (bit-defined, with no IEEE division per channel) is in quant.cuh.
#include "common.cuh"
#include "quant.cuh"

namespace ffd {

using namespace quant;

// Five CTAs per SM (48 registers a thread, a few bytes of spill): the kernel is issue-bound, and
// the fifth CTA's warps fill the issue slots that the loads' latency leaves empty with four.
__global__ void __launch_bounds__(256, 5) quantize_keys_kernel(
    int P, int Hkv, const int32_t *__restrict__ page_ids, const __nv_bfloat16 *__restrict__ k,
    uint8_t *__restrict__ thumb, uint8_t *__restrict__ resid, int *err) {
    int page = blockIdx.x / Hkv;
    const int h = blockIdx.x - page * Hkv;
    if (page_ids) {
        page = page_ids[page];
        if (page < 0 || page >= P) {
            if (threadIdx.x == 0 && h == 0) raise_error(err, FFD_ERRBIT_BOUNDS);
            return;  // CTA-uniform
        }
    }
    const int64_t tile = (int64_t)page * Hkv + h;
    const int row = threadIdx.x >> 2;
    const int g = threadIdx.x & 3;
    uint32_t u[16];
    load_words(k + (tile * kPage + row) * kD + 32 * g, u);
    GroupCodes o;
    quantize_group(u, o);
    if (o.bad) raise_error(err, FFD_ERRBIT_RANGE);
    store_group(o, thumb + tile * kThumbRec, resid + tile * kResidRec, row, g);
}

// Append: four threads per (sequence, KV head), one channel group each. The new token of
// sequence b goes to row p % 64 of page block_table[b][p / 64], p = positions[b].
__global__ void __launch_bounds__(128) append_kv_kernel(
    int B, int Hkv, int P, int max_blocks, const int32_t *__restrict__ positions,
    const int32_t *__restrict__ block_table, const __nv_bfloat16 *__restrict__ k_new,
    const __nv_bfloat16 *__restrict__ v_new, uint8_t *__restrict__ thumb,
    uint8_t *__restrict__ resid, __nv_bfloat16 *__restrict__ v_cache,
    __nv_bfloat16 *__restrict__ k_cache, int *err) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    const int th = t >> 2;  // (sequence, KV head) index b * Hkv + h
    const int g = t & 3;
    if (th >= B * Hkv) return;
    const int b = th / Hkv;
    append_group(b, th - b * Hkv, g, Hkv, P, max_blocks, positions, block_table, k_new, v_new,
                 thumb, resid, v_cache, k_cache, err);
}

cudaError_t launch_append(int B, int Hkv, int P, int max_blocks, const int32_t *positions,
                          const int32_t *block_table, const void *k_new, const void *v_new,
                          uint8_t *thumb, uint8_t *resid, void *v_cache, void *k_cache, int *err,
                          cudaStream_t stream) {
    const int64_t threads = (int64_t)B * Hkv * 4;
    const unsigned blocks = (unsigned)((threads + 127) / 128);
    append_kv_kernel<<<blocks, 128, 0, stream>>>(
        B, Hkv, P, max_blocks, positions, block_table, static_cast<const __nv_bfloat16 *>(k_new),
        static_cast<const __nv_bfloat16 *>(v_new), thumb, resid,
        static_cast<__nv_bfloat16 *>(v_cache), static_cast<__nv_bfloat16 *>(k_cache), err);
    return cudaGetLastError();
}

cudaError_t launch_quantize(int P, int Hkv, const int32_t *page_ids, int num_pages_listed,
                            const void *k, uint8_t *thumb, uint8_t *resid, int *err,
                            cudaStream_t stream) {
    const int64_t tiles = (int64_t)num_pages_listed * Hkv;
    if (tiles == 0) return cudaSuccess;
    if (tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
    quantize_keys_kernel<<<(unsigned)tiles, 256, 0, stream>>>(
        P, Hkv, page_ids, static_cast<const __nv_bfloat16 *>(k), thumb, resid, err);
    return cudaGetLastError();
}

}  // namespace ffd
