// common.cuh -- shapes, argument bundles and small device helpers shared by the FFD kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ffd.h"

namespace ffd {

constexpr int kD = 128;          // head dimension
constexpr int kPage = 64;        // tokens per page == tokens per selection block
constexpr int kGroups = 4;       // channel groups per token (one scale/zero each)
constexpr int kGroupSize = 32;   // channels per group
constexpr int kThumbRow = kD / 4;  // bytes of 2-bit codes per token
constexpr int kMaxG = 8;         // largest supported GQA group
constexpr int kPartStride = 132; // floats per split partial: o[128], m, l, 2 pad
constexpr int kRefineGroups = 2; // decode refine groups = split records per (CTA, unit)
// Cache records (layout in ffd.h): thumbnail = codes [64][32] | scale [64][4] f16 | zero [64][4]
// f16; residual = codes [64][128] (16-byte chunk j of token r at j ^ (r % 8)) | scale [64][4] f16.
constexpr int kThumbRec = FFD_THUMB_RECORD_BYTES;
constexpr int kThumbScaleOff = 2048;
constexpr int kThumbZeroOff = 2560;
constexpr int kResidRec = FFD_RESID_RECORD_BYTES;
constexpr int kResidScaleOff = 8192;
static_assert(kThumbRec == 3072 && kResidRec == 8704, "record sizes");

// Byte offset of residual channel c of token r inside its record.
__host__ __device__ inline int resid_offset(int r, int c) {
    return r * 128 + ((((c >> 4) ^ (r & 7)) << 4) | (c & 15));
}

// Everything a decode launch needs; passed by value to the kernels.
struct DecodeArgs {
    int B, Hq, Hkv, G, P, max_blocks, S, L;
    int nf;          // stage-1 slots per (sequence, KV head)
    float delta, sm_scale;
    const __nv_bfloat16 *q;
    const uint8_t *thumb;    // thumbnail records, kThumbRec bytes per (page, KV head)
    const uint8_t *resid;    // residual records, kResidRec bytes per (page, KV head)
    const __nv_bfloat16 *k;  // dense path only
    const __nv_bfloat16 *v;
    const int32_t *seq_lens, *block_table;
    float *out;
    uint8_t *keep_mask;
    const uint8_t *keep_in;  // optional [B][Hkv][max_blocks] given block mask (replaces Top-delta)
    float *m_tilde;
    int *err;        // device error word
    float *ws_m1;    // [B*Hkv][nf][kMaxG] stage-1 block maxima over the sink / local tokens
    float *ws_mt;    // [B*Hkv][kMaxG] m~ per unit and head (scan-then-refine schedule)
    int2 *ws_kept;   // [blocks of all units] (u * max_blocks + block, page) of the kept blocks,
                     // per CTA range
    int *ws_keptn;   // [CTAs] kept blocks per CTA range
    int *ws_ukept;   // [2][B*Hkv] kept blocks per unit (two buffers, alternate calls)
    unsigned int *ws_grid;  // grid-barrier arrivals (grows by the CTA count each call)
    float *ws_part;  // main-kernel split records: [B*Hkv + CTAs][kRefineGroups][G][kPartStride]
    int *ws_cnt;     // [4][B*Hkv]: merge tickets, stage-1 slots, merge reports, merger
                     // declarations; zero between calls
    cudaEvent_t prof_start, prof_stop;  // optional: recorded around the main kernel
    uint64_t wait_ns;  // bound of every device wait (mbarrier, counter) before FFD_ERRBIT_TIMEOUT
};

// Sink / local block bookkeeping of one sequence (Methodology §2: the pseudo-max uses the sink
// tokens j < S and the local tokens n-L <= j < n; the blocks holding them are always kept).
struct ForcedBlocks {
    int nb;           // ceil(n / 64)
    int ns;           // blocks holding a sink token: 0 .. ns-1
    int local_first;  // first block holding a local token (nb when there is none)
    int lo;           // first local block not already counted as a sink block
    int count;        // number of distinct forced blocks

    __host__ __device__ ForcedBlocks(int n, int S, int L) {
        nb = (n + kPage - 1) / kPage;
        int sink_tokens = n < S ? n : S;
        ns = (sink_tokens + kPage - 1) / kPage;
        if (L > 0 && n > 0) {
            int first_tok = n - L > 0 ? n - L : 0;
            local_first = first_tok / kPage;
        } else {
            local_first = nb;
        }
        lo = local_first > ns ? local_first : ns;
        count = ns + (nb - lo);
    }
    __host__ __device__ bool forced(int blk) const { return blk < ns || blk >= local_first; }
    // The slot-th forced block, 0 <= slot < count.
    __host__ __device__ int block(int slot) const { return slot < ns ? slot : lo + slot - ns; }
};

// Upper bound of ForcedBlocks::count over all sequence lengths.
__host__ __device__ inline int max_forced_blocks(int S, int L, int max_blocks) {
    int c = (S + kPage - 1) / kPage + (L > 0 ? (L + kPage - 1) / kPage + 1 : 0);
    return c < max_blocks ? c : max_blocks;
}

// Host: raise a kernel's dynamic shared-memory limit to `bytes` on the current device. The
// attribute is per device, so the sizes already set are remembered per device in `done`.
constexpr int kMaxDevicesTracked = 64;
template <class Kernel>
inline cudaError_t raise_smem_limit(Kernel *kernel, int bytes, int (&done)[kMaxDevicesTracked]) {
    int dev = 0;
    const cudaError_t q = cudaGetDevice(&dev);
    if (q != cudaSuccess) return q;
    const bool tracked = dev >= 0 && dev < kMaxDevicesTracked;
    if (tracked && done[dev] >= bytes) return cudaSuccess;
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && tracked) done[dev] = bytes;
    return e;
}

__device__ __forceinline__ void raise_error(int *word, int bit) {
    if (word) atomicOr(word, bit);
}

// seq_lens[b], checked against the block table's row length: a length outside
// [0, 64 * max_blocks] raises FFD_ERRBIT_BOUNDS and is clamped, so no kernel reads past a row.
__device__ __forceinline__ int checked_seq_len(const DecodeArgs &a, int b) {
    int n = a.seq_lens[b];
    const int cap = a.max_blocks * kPage;
    if (n < 0 || n > cap) {
        if (threadIdx.x == 0) raise_error(a.err, FFD_ERRBIT_BOUNDS);
        n = n < 0 ? 0 : cap;
    }
    return n;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace ffd
