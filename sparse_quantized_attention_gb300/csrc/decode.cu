// decode.cu -- FFD decode attention on GB300: stage 1 (pseudo-max) and the fused, persistent
// stage-2/3 kernel (Top-delta scan of the 2-bit thumbnails, refinement of the kept blocks with the
// int8 residual and V, online softmax, split merge).
//
// Source: "Faster Than Flash", Methodology §2 (keep token j when s_ij >= m~_i - delta; m~_i from
// the sink and local tokens only) and §3 (stage 1 pseudo-max estimation; stage 2 streams the 2-bit
// keys, computes provisional scores and filters blocks; stage 3 loads the 8-bit residuals and V of
// the selected blocks and computes exact attention, reusing the scan results).
//
// Tensor-core operands (mma.sync m16n8k16, bf16 in, fp32 accumulate; 16 tokens x 8 heads):
//   * A = keys of 16 tokens, B = the GQA group's queries (heads as N, padded to 8).
//   * 2-bit codes enter as bf16 bit patterns (code << s) with s <= 6: exponent field 0, so the
//     value is exactly code * 2^s * 2^-133. B holds q * 2^(kKq - s), so every product is exactly
//     code * q * 2^(kKq-133) and one LOP3 turns two codes into an operand register.
//   * int8 residual codes enter as (c8 + 128) with the same scaling; the +128 is removed in the
//     epilogue with the per-group query sums.
//   * PV: O^T(d x heads) += V^T(d x tokens) P^T(tokens x heads); V^T comes from the 128B-swizzled
//     TMA tile by ldmatrix.trans, P^T from the score accumulators by movmatrix; P is split into
//     bf16 hi + lo parts so that the product keeps ~2^-17 relative precision.
// Channel order inside each 16-channel MMA step is permuted (the same permutation on A and B);
// a dot product does not depend on it.
#include <string.h>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "ptx.cuh"

namespace ffd {

constexpr int kSub = 6;              // blocks per sub-chunk (scan / refine pipeline unit)
constexpr int kRing = 6;             // refine ring slots (residual + V of one kept block each)
constexpr int kPageSlots = 8;        // sub-chunks whose block-table entries are resolved ahead
constexpr int kGroups3 = 3;          // consumer groups: group grp takes the blocks k with k%3==grp
static_assert(kSub == 2 * kGroups3, "each consumer group refines two blocks of a sub-chunk");
constexpr int kConsumerWarps = 12;   // warp c = 4 grp + mt works on m-tile mt (16 tokens)
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kMainThreads = kConsumers + 128;  // + the producer warpgroup (one TMA warp)
constexpr int kProducerRegs = 32;    // setmaxnreg budgets: 128 x 32 + 384 x 160 <= 512 x 128
constexpr int kConsumerRegs = 160;
static_assert(128 * kProducerRegs + kConsumers * kConsumerRegs <= kMainThreads * 128,
              "register reallocation exceeds the launch allocation");
constexpr int kKq = 100;             // q enters the MMA scaled by 2^kKq (|q| < 2^27 required)
constexpr float kUnscale = 8589934592.0f;      // 2^(133 - kKq)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kQMax = 134217728.0f;          // 2^27
constexpr float kRescaleMargin = 30.0f;        // lazy softmax rescaling, natural-log units

// ring slot: residual tile (64 x 128 B, swizzled), V tile (2 boxes of 64 x 128 B, swizzled),
// residual scales (64 x 8 B)
constexpr int kSlotV = 8192;
constexpr int kSlotRScale = 8192 + 16384;
constexpr int kSlotTx = 8192 + 16384 + 512;
constexpr int kSlotBytes = 25600;
constexpr int kThumbBlock = 3072;    // codes 2048 B + scales 512 B + zeros 512 B
constexpr int kShatBuf = kSub * 4 * 32 * 16;  // provisional scores of one sub-chunk
constexpr int kCombineWarpBytes = kMaxG * kD * 4;  // one warp's O^T in the combine

constexpr int kOffRing = 0;
constexpr int kOffThumb = kOffRing + kRing * kSlotBytes;
constexpr int kOffShat = kOffThumb + 2 * kSub * kThumbBlock;  // also the combine buffer
constexpr int kOffUnit = kOffShat + 2 * kShatBuf;
constexpr int kOffMisc = kOffUnit + 4608;
constexpr int kMiscBytes = 1536;
constexpr int kSmemBytes = kOffMisc + kMiscBytes + 1024;  // + slack to align the base to 1 KB
static_assert(6 * kCombineWarpBytes <= 2 * kShatBuf, "combine buffer inside the score buffers");

// One sub-chunk as the page warp hands it to the TMA producer.
struct PageSlot {
    int32_t row[kSub];   // first token row of each block's tile: (page * Hkv + h) * 64
    uint32_t bad;        // entries outside [0, P), one bit per block (row 0, never loaded)
    int32_t cnt;         // blocks; 0 marks the end of this CTA's schedule
    int32_t pad[2];
};

struct Misc {
    uint32_t vote_mask[4];            // blocks of sub-chunk t voted kept, in vote_mask[t % 4]
    uint32_t bad[2];
    uint32_t merge_flag;
    uint32_t aborted;
    float cm[kConsumerWarps][kMaxG];  // combine: per-warp softmax maxima
    float cl[kConsumerWarps][kMaxG];  // combine: per-warp softmax sums
    PageSlot ps[kPageSlots];          // sub-chunk t in ps[t % kPageSlots]
    uint64_t pages_full[kPageSlots];
    uint64_t pages_empty[kPageSlots];
    uint64_t thumb_full[2];
    uint64_t decision[2];
    uint64_t ring_seen[2];            // the ring warp has read the decision of sub-chunk t
    uint64_t ring_full[kRing];
    uint64_t ring_empty[kRing];
};
static_assert(sizeof(Misc) <= kMiscBytes, "misc region");

// Query operands of the (sequence, KV head) unit being processed, laid out so that a lane loads
// its 16 B-fragment registers with four conflict-free 128-bit loads.
struct UnitOps {
    uint4 bt[4][32];   // thumbnail B fragments: [bt0[0..3], bt0[4..7], bt1[0..3], bt1[4..7]][lane]
    uint4 br[4][32];   // residual B fragments, same arrangement
    float4 qs[kMaxG];  // per-group query sums, [head].{group 0..3}
    float thr[kMaxG];  // m~ - delta (+inf for heads >= G)
    float mt[kMaxG];   // m~
    int n;             // sequence length
    int pad[15];
};
static_assert(sizeof(UnitOps) <= 4608, "unit operand slot");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

struct MainParams {
    CUtensorMap tm_resid;
    CUtensorMap tm_v;
    DecodeArgs a;
};

// ------------------------------------------------------------------------------------------
// Work schedule. Stage 1 handles each unit's forced blocks (those holding a sink or a local
// token); the main kernel takes the blocks between them, the unit's "middle" range, which is
// contiguous. The middle blocks of all (sequence, KV head) units, concatenated unit by unit, are
// cut into `ncta` contiguous ranges of equal length; each range is walked in sub-chunks of at
// most kSub blocks that never cross a unit. Producer and consumers walk the same sequence.
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ int len_of(const DecodeArgs &a, int b) {
    const int n = a.seq_lens[b];
    const int cap = a.max_blocks * kPage;
    return n < 0 ? 0 : (n > cap ? cap : n);
}

// First middle block and middle block count of sequence b.
__device__ __forceinline__ int mid_range(const DecodeArgs &a, int b, int &lo) {
    const ForcedBlocks fb(len_of(a, b), a.S, a.L);
    lo = fb.ns;
    return fb.local_first > fb.ns ? fb.local_first - fb.ns : 0;
}

__device__ __forceinline__ int64_t total_mid_blocks(const DecodeArgs &a) {
    int64_t T = 0;
    for (int bb = 0; bb < a.B; bb++) {
        int lo;
        T += (int64_t)a.Hkv * mid_range(a, bb, lo);
    }
    return T;
}

struct Sub {
    int b, h, j0, cnt;  // unit (b, h), first block, block count
    int jr;             // index of the first block within the unit's middle range
    int nmid;           // middle blocks of the unit
    int64_t x0;         // global index of the sub-chunk's first block
    bool last;          // last sub-chunk of this CTA's segment of the unit
};

struct Sched {
    int64_t x, x1, T;
    int b, h, j, nbb, lob;  // j: index within the middle range [lob, lob + nbb)

    __device__ void init(const DecodeArgs &a, int cta, int ncta) {
        T = total_mid_blocks(a);
        x = T * cta / ncta;
        x1 = T * (cta + 1) / ncta;
        int64_t pre = 0;
        b = h = j = nbb = lob = 0;
        for (; b < a.B; b++) {
            int lo;
            const int nb = mid_range(a, b, lo);
            const int64_t span = (int64_t)a.Hkv * nb;
            if (x < pre + span) {
                nbb = nb;
                lob = lo;
                h = (int)((x - pre) / nb);
                j = (int)((x - pre) % nb);
                break;
            }
            pre += span;
        }
    }

    __device__ bool next(const DecodeArgs &a, Sub &s) {
        if (x >= x1) return false;
        int cnt = kSub;
        if (nbb - j < cnt) cnt = nbb - j;
        if (x1 - x < cnt) cnt = (int)(x1 - x);
        s.b = b;
        s.h = h;
        s.j0 = lob + j;
        s.jr = j;
        s.nmid = nbb;
        s.cnt = cnt;
        s.x0 = x;
        s.last = (j + cnt == nbb) || (x + cnt == x1);
        x += cnt;
        j += cnt;
        if (j == nbb) {
            j = 0;
            if (++h == a.Hkv) {
                h = 0;
                for (b++; b < a.B; b++) {
                    nbb = mid_range(a, b, lob);
                    if (nbb > 0) break;
                }
            }
        }
        return true;
    }
};

// CTA whose range holds global block x (ranges are non-empty because ncta <= T).
__device__ __forceinline__ int cta_of(int64_t x, int64_t T, int ncta) {
    return (int)(((x + 1) * ncta - 1) / T);
}

// ------------------------------------------------------------------------------------------
// Query operands. Thread (g = lane/4, tig = lane%4) holds the B fragments of head g and, for the
// epilogue, the per-group query sums of heads 2*tig and 2*tig+1.
// ------------------------------------------------------------------------------------------
struct ThumbOps {
    uint32_t bt0[8], bt1[8];  // chunk kc = channels 16kc .. 16kc+15, head g
    float qs[2][4];           // sum of q over group gg for heads 2tig, 2tig+1
};
struct ResidOps {
    uint32_t br0[8], br1[8];  // chunk 2gg + half, head g
    float qs[2][4];
};

// Per-group query sums of heads 2tig, 2tig+1, from this thread's partial sums of head g over the
// channels c = tig (mod 4): quad reduction, then fetch from the quads of heads 2tig and 2tig+1.
__device__ __forceinline__ void group_sums(float (&part)[4], int tig, float (&qs)[2][4]) {
#pragma unroll
    for (int gg = 0; gg < 4; gg++) {
        part[gg] += __shfl_xor_sync(0xffffffffu, part[gg], 1);
        part[gg] += __shfl_xor_sync(0xffffffffu, part[gg], 2);
    }
#pragma unroll
    for (int gg = 0; gg < 4; gg++) {
        qs[0][gg] = __shfl_sync(0xffffffffu, part[gg], 8 * tig);
        qs[1][gg] = __shfl_sync(0xffffffffu, part[gg], 8 * tig + 4);
    }
}

__device__ __forceinline__ const __nv_bfloat16 *q_row(const DecodeArgs &a, int b, int h, int g) {
    return a.q + ((size_t)b * a.Hq + h * a.G + (g < a.G ? g : 0)) * kD;
}

__device__ __forceinline__ void load_thumb_ops(const DecodeArgs &a, int b, int h, int lane,
                                               ThumbOps &Q) {
    const int g = lane >> 2, tig = lane & 3;
    const bool hv = g < a.G;
    const __nv_bfloat16 *qrow = q_row(a, b, h, g);
    float big = 0.0f;
    auto ld = [&](int c) {
        const float v = hv ? __bfloat162float(qrow[c]) : 0.0f;
        big = fmaxf(big, fabsf(v));
        return v;
    };
    const float st = __int_as_float((127 + kKq - 2 * tig) << 23);  // 2^(kKq - 2 tig)
    float part[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int kc = 0; kc < 8; kc++) {
        const float x0 = ld(16 * kc + tig), x1 = ld(16 * kc + 8 + tig);
        const float x2 = ld(16 * kc + 4 + tig), x3 = ld(16 * kc + 12 + tig);
        Q.bt0[kc] = pack_bf16x2(x0 * st, x1 * st);
        Q.bt1[kc] = pack_bf16x2(x2 * st, x3 * st);
        part[kc >> 1] += (x0 + x1) + (x2 + x3);
    }
    group_sums(part, tig, Q.qs);
    if (!(big < kQMax)) raise_error(a.err, FFD_ERRBIT_RANGE);
}

__device__ __forceinline__ void load_resid_ops(const DecodeArgs &a, int b, int h, int lane,
                                               ResidOps &Q) {
    const int g = lane >> 2, tig = lane & 3;
    const bool hv = g < a.G;
    const __nv_bfloat16 *qrow = q_row(a, b, h, g);
    const float sr = __int_as_float((127 + kKq) << 23);  // 2^kKq
    float part[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int gg = 0; gg < 4; gg++) {
        const int base = 32 * gg + 8 * tig;
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; e++) y[e] = hv ? __bfloat162float(qrow[base + e]) : 0.0f;
        Q.br0[2 * gg] = pack_bf16x2(y[0] * sr, y[2] * sr);
        Q.br1[2 * gg] = pack_bf16x2(y[1] * sr, y[3] * sr);
        Q.br0[2 * gg + 1] = pack_bf16x2(y[4] * sr, y[6] * sr);
        Q.br1[2 * gg + 1] = pack_bf16x2(y[5] * sr, y[7] * sr);
        part[gg] = ((y[0] + y[1]) + (y[2] + y[3])) + ((y[4] + y[5]) + (y[6] + y[7]));
    }
    group_sums(part, tig, Q.qs);
}

// D[gg] = sum over group gg of q . code (scaled by 2^(kKq-133)) for rows (g, g+8) x heads.
__device__ __forceinline__ void thumb_mma(float (&D)[4][4], const uint32_t (&w0)[8],
                                          const uint32_t (&w1)[8], uint32_t m0,
                                          const ThumbOps &Q) {
#pragma unroll
    for (int gg = 0; gg < 4; gg++) D[gg][0] = D[gg][1] = D[gg][2] = D[gg][3] = 0.0f;
#pragma unroll
    for (int kc = 0; kc < 8; kc++) {
        const uint32_t a0 = w0[kc] & m0, a1 = w1[kc] & m0;
        const uint32_t a2 = (w0[kc] >> 8) & m0, a3 = (w1[kc] >> 8) & m0;
        mma_bf16(D[kc >> 1], a0, a1, a2, a3, Q.bt0[kc], Q.bt1[kc]);
    }
}

// D[gg] = sum over group gg of q . (c8 + 128) (scaled by 2^(kKq-133)).
// x0[gg] / x1[gg]: bytes 32gg + 8tig .. +7 of rows g / g+8.
__device__ __forceinline__ void resid_mma(float (&D)[4][4], const uint2 (&x0)[4],
                                          const uint2 (&x1)[4], const ResidOps &Q) {
#pragma unroll
    for (int gg = 0; gg < 4; gg++) D[gg][0] = D[gg][1] = D[gg][2] = D[gg][3] = 0.0f;
#pragma unroll
    for (int gg = 0; gg < 4; gg++) {
#pragma unroll
        for (int half = 0; half < 2; half++) {
            const uint32_t v0 = half ? x0[gg].y : x0[gg].x;
            const uint32_t v1 = half ? x1[gg].y : x1[gg].x;
            const uint32_t a0 = (v0 & 0x00FF00FFu) ^ 0x00800080u;
            const uint32_t a1 = (v1 & 0x00FF00FFu) ^ 0x00800080u;
            const uint32_t a2 = ((v0 >> 8) & 0x00FF00FFu) ^ 0x00800080u;
            const uint32_t a3 = ((v1 >> 8) & 0x00FF00FFu) ^ 0x00800080u;
            mma_bf16(D[gg], a0, a1, a2, a3, Q.br0[2 * gg + half], Q.br1[2 * gg + half]);
        }
    }
}

__device__ __forceinline__ void unpack4h(uint2 v, float (&f)[4]) {
    const float2 lo = __half22float2(*reinterpret_cast<const __half2 *>(&v.x));
    const float2 hi = __half22float2(*reinterpret_cast<const __half2 *>(&v.y));
    f[0] = lo.x;
    f[1] = lo.y;
    f[2] = hi.x;
    f[3] = hi.y;
}

// Provisional score s^ = sm * sum_g (scale_g q_g.c_g + zero_g sum(q_g)) of accumulator entry e.
__device__ __forceinline__ float est_score(const float (&D)[4][4], int e, const float (&sf)[4],
                                           const float (&zf)[4], const float (&qs)[4], float sm) {
    float acc = 0.0f;
#pragma unroll
    for (int gg = 0; gg < 4; gg++)
        acc = fmaf(sf[gg] * kUnscale, D[gg][e], fmaf(zf[gg], qs[gg], acc));
    return acc * sm;
}

// Residual correction sm * sum_g r_scale_g q_g . c8_g of accumulator entry e.
__device__ __forceinline__ float corr_score(const float (&D)[4][4], int e, const float (&sr)[4],
                                            const float (&qs)[4], float sm) {
    float acc = 0.0f;
#pragma unroll
    for (int gg = 0; gg < 4; gg++)
        acc = fmaf(sr[gg], fmaf(kUnscale, D[gg][e], -128.0f * qs[gg]), acc);
    return acc * sm;
}

// Pseudo-max of heads 2tig, 2tig+1 from the stage-1 block maxima (-inf when there are none).
__device__ __forceinline__ void load_mtilde(const DecodeArgs &a, int u, int tig, float &m0,
                                            float &m1) {
    m0 = -INFINITY;
    m1 = -INFINITY;
    for (int s = 0; s < a.nf; s++) {
        const float *p = a.ws_m1 + ((size_t)u * a.nf + s) * kMaxG;
        m0 = fmaxf(m0, p[2 * tig]);
        m1 = fmaxf(m1, p[2 * tig + 1]);
    }
}

// ------------------------------------------------------------------------------------------
// Split merge: out_i = sum_r e^(m_r - M) num_r / sum_r e^(m_r - M) den_r over a unit's records
// (stage-1 slots of the forced blocks, and main-kernel records of CTAs cf..cl when it has a
// middle range); records hold (num[128], m, den) per head.
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ const float *s1_record(const DecodeArgs &a, int u, int slot, int i) {
    return a.ws_s1 + (((size_t)u * a.nf + slot) * a.G + i) * kPartStride;
}

__device__ __forceinline__ const float *main_record(const DecodeArgs &a, int u, int c, int i) {
    return a.ws_part + ((size_t)(u + c) * a.G + i) * kPartStride;
}

// Called after a __threadfence() that follows the atomic ticket showing this CTA came last.
// Warp w of nwarps merges heads w, w + nwarps, ...: lane r owns record r's maximum, weight and
// denominator; every lane accumulates 4 of the 128 channels over all records, whose loads do not
// depend on each other.
__device__ __forceinline__ void merge_unit(const DecodeArgs &a, int b, int h, bool with_main,
                                           int cf, int cl, int warp, int nwarps, int lane) {
    const int u = b * a.Hkv + h;
    const int n1 = a.nf, nr = n1 + (with_main ? cl - cf + 1 : 0);
    for (int i = warp; i < a.G; i += nwarps) {
        auto rec = [&](int r) {
            return r < n1 ? s1_record(a, u, r, i) : main_record(a, u, cf + r - n1, i);
        };
        float M = -INFINITY;
        for (int r = lane; r < nr; r += 32) M = fmaxf(M, __ldcg(rec(r) + kD));
        M = warp_max(M);
        float num[4] = {0.0f, 0.0f, 0.0f, 0.0f}, den = 0.0f;
        if (M != -INFINITY) {
            for (int r0 = 0; r0 < nr; r0 += 32) {
                const int r = r0 + lane;
                float f = 0.0f;
                if (r < nr) {
                    const float *p = rec(r);
                    const float mr = __ldcg(p + kD);
                    if (mr != -INFINITY) {
                        f = exp2f((mr - M) * kLog2e);
                        den = fmaf(f, __ldcg(p + kD + 1), den);
                    }
                }
                const int cnt = nr - r0 < 32 ? nr - r0 : 32;
#pragma unroll 4
                for (int j = 0; j < cnt; j++) {
                    const float fj = __shfl_sync(0xffffffffu, f, j);
                    const float *p = rec(r0 + j);
#pragma unroll
                    for (int k = 0; k < 4; k++) {
                        const float x = __ldcg(p + lane + 32 * k);
                        num[k] = fj > 0.0f ? fmaf(fj, x, num[k]) : num[k];
                    }
                }
            }
            den = warp_sum(den);
        }
        float *o = a.out + ((size_t)b * a.Hq + h * a.G + i) * kD;
#pragma unroll
        for (int k = 0; k < 4; k++) o[lane + 32 * k] = den > 0.0f ? num[k] / den : 0.0f;
        if (a.m_tilde) {
            float m = -INFINITY;
            for (int sl = lane; sl < a.nf; sl += 32)
                m = fmaxf(m, __ldcg(a.ws_m1 + ((size_t)u * a.nf + sl) * kMaxG + i));
            m = warp_max(m);
            if (lane == 0) a.m_tilde[(size_t)b * a.Hq + h * a.G + i] = m;
        }
    }
}

// ------------------------------------------------------------------------------------------
// Stage 1: one CTA per (forced-block slot, unit); warp w takes 16 tokens of the block.
//   * exact scores s = sm q . K^ (thumbnail + residual, on tensor cores);
//   * per-head maximum over the block's sink / local tokens -> ws_m1 (the pseudo-max m~ is the
//     maximum over the unit's slots);
//   * softmax partial of the whole block (forced blocks are always kept) -> ws_s1, with PV on
//     CUDA cores (V read straight from global memory; the CTA keeps 2 KB of shared memory, so it
//     runs beside the persistent main kernel);
//   * a unit without middle blocks is merged here by the last of its slot CTAs (atomic ticket).
// Slot 0 of every unit also clears the keep-mask tail past the sequence.
// ------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(128, 1) stage1_kernel(const DecodeArgs a) {
    grid_launch_dependents();
    __shared__ float red_m[4][kMaxG], red_x[4][kMaxG], red_l[4][kMaxG];
    __shared__ float pbuf[kPage][kMaxG];
    __shared__ uint32_t merge_flag;
    const int u = blockIdx.y, b = u / a.Hkv, h = u % a.Hkv;
    const int slot = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, tig = lane & 3;
    const int raw_n = a.seq_lens[b];
    const int n = len_of(a, b);
    const int nb = (n + kPage - 1) / kPage;
    if (slot == 0) {
        if (tid == 0 && h == 0 && raw_n != n) raise_error(a.err, FFD_ERRBIT_BOUNDS);
        if (a.keep_mask)
            for (int blk = nb + tid; blk < a.max_blocks; blk += blockDim.x)
                a.keep_mask[(size_t)u * a.max_blocks + blk] = 0;
    }
    const ForcedBlocks fb(n, a.S, a.L);
    int page = -1;
    const int blk = slot < fb.count ? fb.block(slot) : 0;
    if (slot < fb.count) {
        page = a.block_table[(size_t)b * a.max_blocks + blk];
        if (page < 0 || page >= a.P) {
            if (tid == 0) raise_error(a.err, FFD_ERRBIT_BOUNDS);
            page = -1;
        }
        if (a.keep_mask && tid == 0) a.keep_mask[(size_t)u * a.max_blocks + blk] = page >= 0;
    }
    float *mdst = a.ws_m1 + ((size_t)u * a.nf + slot) * kMaxG;
    float *rdst = a.ws_s1 + ((size_t)u * a.nf + slot) * a.G * kPartStride;
    if (page < 0) {  // empty slot (uniform across the CTA)
        if (tid < kMaxG) mdst[tid] = -INFINITY;
        if (tid < a.G) {
            rdst[tid * kPartStride + kD] = -INFINITY;
            rdst[tid * kPartStride + kD + 1] = 0.0f;
        }
    } else {
        ThumbOps Q;
        ResidOps QR;
        load_thumb_ops(a, b, h, lane, Q);
        load_resid_ops(a, b, h, lane, QR);
        const size_t tile = (size_t)page * a.Hkv + h;
        const int r0 = 16 * warp + g, r1 = r0 + 8;
        uint32_t w0[8], w1[8];
        {
            const uint4 *c0 = reinterpret_cast<const uint4 *>(a.thumb + (tile * kPage + r0) * kThumbRow);
            const uint4 *c1 = reinterpret_cast<const uint4 *>(a.thumb + (tile * kPage + r1) * kThumbRow);
            const uint4 p0 = c0[0], p1 = c0[1], p2 = c1[0], p3 = c1[1];
            w0[0] = p0.x; w0[1] = p0.y; w0[2] = p0.z; w0[3] = p0.w;
            w0[4] = p1.x; w0[5] = p1.y; w0[6] = p1.z; w0[7] = p1.w;
            w1[0] = p2.x; w1[1] = p2.y; w1[2] = p2.z; w1[3] = p2.w;
            w1[4] = p3.x; w1[5] = p3.y; w1[6] = p3.z; w1[7] = p3.w;
        }
        uint2 x0[4], x1[4];
#pragma unroll
        for (int gg = 0; gg < 4; gg++) {
            x0[gg] = *reinterpret_cast<const uint2 *>(a.resid + (tile * kPage + r0) * kD + 32 * gg + 8 * tig);
            x1[gg] = *reinterpret_cast<const uint2 *>(a.resid + (tile * kPage + r1) * kD + 32 * gg + 8 * tig);
        }
        float sf0[4], sf1[4], zf0[4], zf1[4], sr0[4], sr1[4];
        const uint2 *ts = reinterpret_cast<const uint2 *>(a.t_scale);
        const uint2 *tz = reinterpret_cast<const uint2 *>(a.t_zero);
        const uint2 *rs = reinterpret_cast<const uint2 *>(a.r_scale);
        unpack4h(ts[tile * kPage + r0], sf0);
        unpack4h(ts[tile * kPage + r1], sf1);
        unpack4h(tz[tile * kPage + r0], zf0);
        unpack4h(tz[tile * kPage + r1], zf1);
        unpack4h(rs[tile * kPage + r0], sr0);
        unpack4h(rs[tile * kPage + r1], sr1);

        float D[4][4], Dr[4][4];
        thumb_mma(D, w0, w1, 0x00030003u << (2 * tig), Q);
        resid_mma(Dr, x0, x1, QR);
        const float sm = a.sm_scale;
        const int t0 = blk * kPage + r0, t1 = blk * kPage + r1;
        const bool in0 = t0 < n, in1 = t1 < n;
        const float s00 = in0 ? est_score(D, 0, sf0, zf0, Q.qs[0], sm) + corr_score(Dr, 0, sr0, Q.qs[0], sm) : -INFINITY;
        const float s01 = in0 ? est_score(D, 1, sf0, zf0, Q.qs[1], sm) + corr_score(Dr, 1, sr0, Q.qs[1], sm) : -INFINITY;
        const float s10 = in1 ? est_score(D, 2, sf1, zf1, Q.qs[0], sm) + corr_score(Dr, 2, sr1, Q.qs[0], sm) : -INFINITY;
        const float s11 = in1 ? est_score(D, 3, sf1, zf1, Q.qs[1], sm) + corr_score(Dr, 3, sr1, Q.qs[1], sm) : -INFINITY;
        // pseudo-max candidates: sink and local tokens only
        const bool v0 = in0 && (t0 < a.S || t0 >= n - a.L);
        const bool v1 = in1 && (t1 < a.S || t1 >= n - a.L);
        float mx0 = fmaxf(v0 ? s00 : -INFINITY, v1 ? s10 : -INFINITY);
        float mx1 = fmaxf(v0 ? s01 : -INFINITY, v1 ? s11 : -INFINITY);
        // block maximum over all its tokens (softmax reference of the partial)
        float bx0 = fmaxf(s00, s10), bx1 = fmaxf(s01, s11);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
            bx0 = fmaxf(bx0, __shfl_xor_sync(0xffffffffu, bx0, o));
            bx1 = fmaxf(bx1, __shfl_xor_sync(0xffffffffu, bx1, o));
        }
        if (g == 0) {
            red_m[warp][2 * tig] = mx0;
            red_m[warp][2 * tig + 1] = mx1;
            red_x[warp][2 * tig] = bx0;
            red_x[warp][2 * tig + 1] = bx1;
        }
        __syncthreads();
        const float M0 = fmaxf(fmaxf(red_x[0][2 * tig], red_x[1][2 * tig]),
                               fmaxf(red_x[2][2 * tig], red_x[3][2 * tig]));
        const float M1 = fmaxf(fmaxf(red_x[0][2 * tig + 1], red_x[1][2 * tig + 1]),
                               fmaxf(red_x[2][2 * tig + 1], red_x[3][2 * tig + 1]));
        const float p00 = in0 ? exp2f((s00 - M0) * kLog2e) : 0.0f;
        const float p01 = in0 ? exp2f((s01 - M1) * kLog2e) : 0.0f;
        const float p10 = in1 ? exp2f((s10 - M0) * kLog2e) : 0.0f;
        const float p11 = in1 ? exp2f((s11 - M1) * kLog2e) : 0.0f;
        pbuf[r0][2 * tig] = p00;
        pbuf[r0][2 * tig + 1] = p01;
        pbuf[r1][2 * tig] = p10;
        pbuf[r1][2 * tig + 1] = p11;
        float l0 = p00 + p10, l1 = p01 + p11;
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, o);
            l1 += __shfl_xor_sync(0xffffffffu, l1, o);
        }
        if (g == 0) {
            red_l[warp][2 * tig] = l0;
            red_l[warp][2 * tig + 1] = l1;
        }
        __syncthreads();
        // PV: thread = channel d
        float acc[kMaxG];
#pragma unroll
        for (int i = 0; i < kMaxG; i++) acc[i] = 0.0f;
        const __nv_bfloat16 *vcol = a.v + tile * kPage * kD + tid;
        for (int tt = 0; tt < kPage; tt++) {
            const float vv = __bfloat162float(vcol[(size_t)tt * kD]);
#pragma unroll
            for (int i = 0; i < kMaxG; i++) acc[i] = fmaf(pbuf[tt][i], vv, acc[i]);
        }
#pragma unroll
        for (int i = 0; i < kMaxG; i++)
            if (i < a.G) rdst[i * kPartStride + tid] = acc[i];
        if (tid < kMaxG)
            mdst[tid] = tid < a.G ? fmaxf(fmaxf(red_m[0][tid], red_m[1][tid]),
                                          fmaxf(red_m[2][tid], red_m[3][tid]))
                                  : -INFINITY;
        if (tid < a.G) {
            rdst[tid * kPartStride + kD] = fmaxf(fmaxf(red_x[0][tid], red_x[1][tid]),
                                                 fmaxf(red_x[2][tid], red_x[3][tid]));
            rdst[tid * kPartStride + kD + 1] =
                (red_l[0][tid] + red_l[1][tid]) + (red_l[2][tid] + red_l[3][tid]);
        }
    }
    // a unit with no middle blocks is merged by the last of its stage-1 CTAs
    int lo;
    if (mid_range(a, b, lo) > 0) return;  // uniform: the main kernel merges this unit
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        uint32_t last = 1;
        if (a.nf > 1) {
            int *cnt = a.ws_cnt + a.B * a.Hkv + u;
            last = atomicAdd(cnt, 1) == a.nf - 1;
            if (last) *cnt = 0;  // ready for the next call
        }
        merge_flag = last;
    }
    __syncthreads();
    if (merge_flag) {
        __threadfence();
        merge_unit(a, b, h, false, 0, -1, warp, blockDim.x / 32, lane);
    }
}
// ------------------------------------------------------------------------------------------
// Main kernel: persistent, one CTA per SM. Warpgroup 0 issues the copies: the ring warp (0), the
// page warp (1) and the thumbnail warp (2); warps 4-15 consume.
// ------------------------------------------------------------------------------------------
struct Smem {
    uint8_t *ring, *thumb, *shat;
    UnitOps *unit;
    Misc *misc;
};

// Bounded wait: after kWaitTimeoutNs the CTA records FFD_ERRBIT_TIMEOUT, marks itself aborted and
// stops waiting (its results are then garbage, but every thread still reaches every barrier).
__device__ __forceinline__ void wait_bar(const DecodeArgs &a, Misc *m, uint64_t *bar,
                                         uint32_t parity) {
    if (*reinterpret_cast<volatile uint32_t *>(&m->aborted)) return;
    if (mbar_try_wait(bar, parity)) return;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
            raise_error(a.err, FFD_ERRBIT_TIMEOUT);
            *reinterpret_cast<volatile uint32_t *>(&m->aborted) = 1;
            return;
        }
    }
}

// Page warp: walks the CTA's schedule ahead of the producer and resolves the block-table entries
// of every sub-chunk (one lane per block) into the page ring, so that no global-load latency sits
// on the TMA issue path; a slot with cnt == 0 ends the schedule. Entries outside [0, P) are
// flagged (FFD_ERRBIT_BOUNDS) and their blocks are never loaded.
__device__ __forceinline__ void pager(const DecodeArgs &a, const Smem &S, int cta, int ncta,
                                      int lane) {
    Misc *m = S.misc;
    Sched sch;
    sch.init(a, cta, ncta);
    Sub s;
    for (int t = 0;; t++) {
        const bool more = sch.next(a, s);
        const int ps = t % kPageSlots, round = t / kPageSlots;
        if (round > 0) wait_bar(a, m, &m->pages_empty[ps], (round - 1) & 1);
        PageSlot &P = m->ps[ps];
        if (!more) {  // end marker
            if (lane == 0) {
                P.cnt = 0;
                mbar_arrive(&m->pages_full[ps]);
            }
            return;
        }
        int page = 0;
        if (lane < s.cnt) page = a.block_table[(size_t)s.b * a.max_blocks + s.j0 + lane];
        const bool bad = lane < s.cnt && (page < 0 || page >= a.P);
        const uint32_t badmask = __ballot_sync(0xffffffffu, bad);
        // every row in the ring is in range (a bad entry reads as page 0 and is never loaded)
        if (lane < s.cnt) P.row[lane] = ((bad ? 0 : page) * a.Hkv + s.h) * kPage;
        if (lane == 0) {
            P.bad = badmask;
            P.cnt = s.cnt;
            if (badmask) raise_error(a.err, FFD_ERRBIT_BOUNDS);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&m->pages_full[ps]);
    }
}

__device__ __forceinline__ const PageSlot &page_slot(const DecodeArgs &a, Misc *m, int t) {
    wait_bar(a, m, &m->pages_full[t % kPageSlots], (t / kPageSlots) & 1);
    return m->ps[t % kPageSlots];
}

// Wait for a copy this CTA issued, ignoring the abort flag (still bounded in time): no CTA exits
// with a copy into its shared memory in flight.
__device__ __forceinline__ void drain_bar(const DecodeArgs &a, uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
            raise_error(a.err, FFD_ERRBIT_TIMEOUT);
            return;
        }
    }
}

// Thumbnail warp: the 2-bit codes, scales and zeros of sub-chunk t go to buffer t&1 once the ring
// warp has taken the decision of sub-chunk t-2 (so that buffer is free, and no decision can run
// two phases ahead of the ring warp); lane k issues block k's copies.
__device__ __forceinline__ void thumb_issuer(const DecodeArgs &a, const Smem &S, int lane) {
    Misc *m = S.misc;
    uint32_t pend0 = 0, pend1 = 0;  // phases of thumb_full[0/1] armed by this warp
    for (int t = 0;; t++) {
        const int buf = t & 1;
        if (t >= 2) wait_bar(a, m, &m->ring_seen[buf], ((t - 2) >> 1) & 1);
        const PageSlot &P = page_slot(a, m, t);
        const int cnt = P.cnt;
        if (cnt == 0 || *reinterpret_cast<volatile uint32_t *>(&m->aborted)) break;
        const uint32_t bad = P.bad;
        if (lane == 0) {
            m->bad[buf] = bad;
            mbar_arrive_expect_tx(&m->thumb_full[buf],
                                  (uint32_t)((cnt - __popc(bad)) * kThumbBlock));
        }
        pend0 += buf == 0;
        pend1 += buf == 1;
        __syncwarp();
        if (lane < cnt && !((bad >> lane) & 1u)) {
            const size_t row = (size_t)P.row[lane];
            uint8_t *d = S.thumb + buf * (kSub * kThumbBlock) + lane * kThumbBlock;
            tma_load_1d(d, a.thumb + row * kThumbRow, 2048, &m->thumb_full[buf]);
            tma_load_1d(d + 2048, a.t_scale + row * kGroups, 512, &m->thumb_full[buf]);
            tma_load_1d(d + 2560, a.t_zero + row * kGroups, 512, &m->thumb_full[buf]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&m->pages_empty[t % kPageSlots]);
    }
    // leave no copy in flight
    if (lane == 0) {
        if (pend0) drain_bar(a, &m->thumb_full[0], (pend0 - 1) & 1);
        if (pend1) drain_bar(a, &m->thumb_full[1], (pend1 - 1) & 1);
    }
}

// Ring warp: residual tile, V tile and residual scales of every kept block of sub-chunk t, once
// the consumers have decided it; lanes 0-3 issue one block's four copies side by side.
__device__ __forceinline__ void ring_issuer(const MainParams &prm, const Smem &S, int lane) {
    const DecodeArgs &a = prm.a;
    Misc *m = S.misc;
    if (lane == 0) {
        prefetch_tensormap(&prm.tm_resid);
        prefetch_tensormap(&prm.tm_v);
    }
    int kb = 0;
    for (int t = 0;; t++) {
        const PageSlot &P = page_slot(a, m, t);
        const int cnt = P.cnt;
        if (cnt == 0 || *reinterpret_cast<volatile uint32_t *>(&m->aborted)) break;
        wait_bar(a, m, &m->decision[t & 1], (t >> 1) & 1);
        const uint32_t mask = *reinterpret_cast<volatile uint32_t *>(&m->vote_mask[t & 3]) &
                              ~P.bad & ((1u << cnt) - 1u);
        __syncwarp();
        if (lane == 0) {
            // every consumer has read the votes of sub-chunk t-2 (it voted on t since), and none
            // votes on t+2 before this arrival releases its thumbnails
            m->vote_mask[(t + 2) & 3] = 0;
            mbar_arrive(&m->ring_seen[t & 1]);
        }
        for (int k = 0; k < cnt; k++) {
            if (!(mask & (1u << k))) continue;
            const int slot = kb % kRing, round = kb / kRing;
            kb++;
            if (round > 0) wait_bar(a, m, &m->ring_empty[slot], (round - 1) & 1);
            const int row = P.row[k];
            uint8_t *d = S.ring + slot * kSlotBytes;
            uint64_t *bar = &m->ring_full[slot];
            if (lane == 0) mbar_arrive_expect_tx(bar, kSlotTx);
            __syncwarp();
            if (lane == 0) tma_load_2d(d, &prm.tm_resid, 0, row, bar);
            else if (lane == 1) tma_load_2d(d + kSlotV, &prm.tm_v, 0, row, bar);
            else if (lane == 2) tma_load_2d(d + kSlotV + 8192, &prm.tm_v, 64, row, bar);
            else if (lane == 3)
                tma_load_1d(d + kSlotRScale, a.r_scale + (size_t)row * kGroups, 512, bar);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&m->pages_empty[t % kPageSlots]);
    }
    // leave no copy in flight: wait for the last fill of every ring slot
    if (lane == 0)
        for (int s = 0; s < kRing && s < kb; s++) {
            const int last = kb - 1 - ((kb - 1 - s) % kRing);
            drain_bar(a, &m->ring_full[s], (last / kRing) & 1);
        }
}

// Consumer warp 0 computes the unit's query operands and thresholds into the unit slot; every
// consumer warp then reads them from shared memory.
__device__ __forceinline__ void setup_unit(const DecodeArgs &a, const Smem &S, const Sub &s,
                                           int warp, int lane) {
    if (warp == 0) {
        UnitOps &U = *S.unit;
        const int g = lane >> 2, tig = lane & 3;
        ThumbOps T;
        ResidOps Rr;
        load_thumb_ops(a, s.b, s.h, lane, T);
        load_resid_ops(a, s.b, s.h, lane, Rr);
#pragma unroll
        for (int r = 0; r < 2; r++) {
            U.bt[r][lane] = make_uint4(T.bt0[4 * r], T.bt0[4 * r + 1], T.bt0[4 * r + 2], T.bt0[4 * r + 3]);
            U.bt[2 + r][lane] = make_uint4(T.bt1[4 * r], T.bt1[4 * r + 1], T.bt1[4 * r + 2], T.bt1[4 * r + 3]);
            U.br[r][lane] = make_uint4(Rr.br0[4 * r], Rr.br0[4 * r + 1], Rr.br0[4 * r + 2], Rr.br0[4 * r + 3]);
            U.br[2 + r][lane] = make_uint4(Rr.br1[4 * r], Rr.br1[4 * r + 1], Rr.br1[4 * r + 2], Rr.br1[4 * r + 3]);
        }
        if (g == 0) {
            U.qs[2 * tig] = make_float4(T.qs[0][0], T.qs[0][1], T.qs[0][2], T.qs[0][3]);
            U.qs[2 * tig + 1] = make_float4(T.qs[1][0], T.qs[1][1], T.qs[1][2], T.qs[1][3]);
        }
        if (lane < kMaxG) {
            float m = -INFINITY;
            const int u = s.b * a.Hkv + s.h;
            for (int sl = 0; sl < a.nf; sl++)
                m = fmaxf(m, a.ws_m1[((size_t)u * a.nf + sl) * kMaxG + lane]);
            U.mt[lane] = m;
            U.thr[lane] = lane < a.G ? m - a.delta : INFINITY;
        }
        if (lane == 0) U.n = len_of(a, s.b);
    }
    named_barrier_sync(1, kConsumers);
}

__device__ __forceinline__ void load_frags(const uint4 (&src)[4][32], int lane, uint32_t (&f0)[8],
                                           uint32_t (&f1)[8]) {
    const uint4 p0 = src[0][lane], p1 = src[1][lane], p2 = src[2][lane], p3 = src[3][lane];
    f0[0] = p0.x; f0[1] = p0.y; f0[2] = p0.z; f0[3] = p0.w;
    f0[4] = p1.x; f0[5] = p1.y; f0[6] = p1.z; f0[7] = p1.w;
    f1[0] = p2.x; f1[1] = p2.y; f1[2] = p2.z; f1[3] = p2.w;
    f1[4] = p3.x; f1[5] = p3.y; f1[6] = p3.z; f1[7] = p3.w;
}

// Provisional scores of one m-tile (rows r0 = 16 mt + g and r1 = r0 + 8 of a thumbnail block in
// shared memory), for heads 2tig, 2tig+1: {(r0,h0), (r0,h1), (r1,h0), (r1,h1)}.
__device__ __forceinline__ float4 scan_tile(const uint8_t *base, int r0, int r1, uint32_t m0,
                                            const ThumbOps &Q, float sm) {
    const uint4 *c0 = reinterpret_cast<const uint4 *>(base + r0 * kThumbRow);
    const uint4 *c1 = reinterpret_cast<const uint4 *>(base + r1 * kThumbRow);
    const uint4 p0 = c0[0], p1 = c0[1], p2 = c1[0], p3 = c1[1];
    const uint32_t w0[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
    const uint32_t w1[8] = {p2.x, p2.y, p2.z, p2.w, p3.x, p3.y, p3.z, p3.w};
    float D[4][4];
    thumb_mma(D, w0, w1, m0, Q);
    float sf0[4], sf1[4], zf0[4], zf1[4];
    const uint2 *ts = reinterpret_cast<const uint2 *>(base + 2048);
    const uint2 *tz = reinterpret_cast<const uint2 *>(base + 2560);
    unpack4h(ts[r0], sf0);
    unpack4h(ts[r1], sf1);
    unpack4h(tz[r0], zf0);
    unpack4h(tz[r1], zf1);
    float4 e;
    e.x = est_score(D, 0, sf0, zf0, Q.qs[0], sm);
    e.y = est_score(D, 1, sf0, zf0, Q.qs[1], sm);
    e.z = est_score(D, 2, sf1, zf1, Q.qs[0], sm);
    e.w = est_score(D, 3, sf1, zf1, Q.qs[1], sm);
    return e;
}

__device__ __forceinline__ bool tile_passes(float4 e, bool v0, bool v1, float thr0, float thr1) {
    return (v0 && (e.x >= thr0 || e.y >= thr1)) || (v1 && (e.z >= thr0 || e.w >= thr1));
}

// Scan of sub-chunk t: provisional scores of this warp's m-tiles and its vote (an OR into
// vote_mask, then one arrival on the decision barrier; no warp waits for the others here).
// Returns the sub-chunk's never-loaded blocks. The warp's blocks are k = grp and grp + 3,
// scanned side by side (two independent dependency chains). The second tile is computed even past the sub-chunk's end (its shared-memory reads stay
// inside the buffer) and then ignored, so both chains stay in one basic block.
__device__ __forceinline__ uint32_t scan_sub(const DecodeArgs &a, const Smem &S, const Sub &s,
                                             int t, int warp, int lane) {
    Misc *m = S.misc;
    const UnitOps &U = *S.unit;
    const int g = lane >> 2, tig = lane & 3, grp = warp >> 2, mt = warp & 3;
    const int buf = t & 1;
    wait_bar(a, m, &m->thumb_full[buf], (t >> 1) & 1);
    const uint32_t bad = m->bad[buf];
    uint32_t votes = 0;
    const int kA = grp, kB = grp + kGroups3;
    if (kA < s.cnt) {
        const uint32_t m0 = 0x00030003u << (2 * tig);
        const float sm = a.sm_scale;
        const float thr0 = U.thr[2 * tig], thr1 = U.thr[2 * tig + 1];
        const int n = U.n;
        ThumbOps Q;
        load_frags(U.bt, lane, Q.bt0, Q.bt1);
        {
            const float4 q0 = U.qs[2 * tig], q1 = U.qs[2 * tig + 1];
            Q.qs[0][0] = q0.x; Q.qs[0][1] = q0.y; Q.qs[0][2] = q0.z; Q.qs[0][3] = q0.w;
            Q.qs[1][0] = q1.x; Q.qs[1][1] = q1.y; Q.qs[1][2] = q1.z; Q.qs[1][3] = q1.w;
        }
        const int r0 = 16 * mt + g, r1 = r0 + 8;
        const uint8_t *tb = S.thumb + buf * (kSub * kThumbBlock);
        float4 *shat = reinterpret_cast<float4 *>(S.shat + buf * kShatBuf);
        const float4 eA = scan_tile(tb + kA * kThumbBlock, r0, r1, m0, Q, sm);
        const float4 eB = scan_tile(tb + kB * kThumbBlock, r0, r1, m0, Q, sm);
        const int tA = (s.j0 + kA) * kPage, tB = (s.j0 + kB) * kPage;
        const bool pA = tile_passes(eA, tA + r0 < n, tA + r1 < n, thr0, thr1);
        const bool pB = kB < s.cnt && tile_passes(eB, tB + r0 < n, tB + r1 < n, thr0, thr1);
        if (__any_sync(0xffffffffu, pA)) votes |= 1u << kA;
        if (__any_sync(0xffffffffu, pB)) votes |= 1u << kB;
        shat[(kA * 4 + mt) * 32 + lane] = eA;
        if (kB < s.cnt) shat[(kB * 4 + mt) * 32 + lane] = eB;
    }
    if (lane == 0) {
        if (votes) atomicOr(&m->vote_mask[t & 3], votes);
        mbar_arrive(&m->decision[buf]);  // releases the vote; the decision completes at 12 votes
    }
    return bad;
}

// Kept blocks of sub-chunk t: every warp's vote, less the blocks that were never loaded.
__device__ __forceinline__ uint32_t kept_mask(const DecodeArgs &a, Misc *m, const Sub &s, int t,
                                              uint32_t bad) {
    wait_bar(a, m, &m->decision[t & 1], (t >> 1) & 1);
    return *reinterpret_cast<volatile uint32_t *>(&m->vote_mask[t & 3]) & ~bad &
           ((1u << s.cnt) - 1u);
}

// Refine-side state of the unit being refined: its query operands, and this warp's running
// softmax state (max, sum, O^T accumulators) for heads 2tig, 2tig+1.
struct RefineState {
    float m0, m1, l0, l1;
    float o[8][4];
};

// Fresh softmax state for a unit: the reference starts at its pseudo-max m~.
__device__ __forceinline__ void reset_refine(RefineState &R, const UnitOps &U, int lane) {
    R.m0 = U.mt[2 * (lane & 3)];
    R.m1 = U.mt[2 * (lane & 3) + 1];
    R.l0 = R.l1 = 0.0f;
#pragma unroll
    for (int md = 0; md < 8; md++) R.o[md][0] = R.o[md][1] = R.o[md][2] = R.o[md][3] = 0.0f;
}

// Stage 3 on this warp's m-tile of one kept block held in a ring slot.
__device__ __forceinline__ void refine_tile(const DecodeArgs &a, const uint8_t *slot,
                                            const UnitOps &U, const float4 est, int blk,
                                            RefineState &R, int mt, int lane) {
    const int g = lane >> 2, tig = lane & 3;
    ResidOps Q;
    load_frags(U.br, lane, Q.br0, Q.br1);
    {
        const float4 q0 = U.qs[2 * tig], q1 = U.qs[2 * tig + 1];
        Q.qs[0][0] = q0.x; Q.qs[0][1] = q0.y; Q.qs[0][2] = q0.z; Q.qs[0][3] = q0.w;
        Q.qs[1][0] = q1.x; Q.qs[1][1] = q1.y; Q.qs[1][2] = q1.z; Q.qs[1][3] = q1.w;
    }
    const int n = U.n;
    const int r0 = 16 * mt + g, r1 = r0 + 8;
    uint2 x0[4], x1[4];
#pragma unroll
    for (int gg = 0; gg < 4; gg++) {
        const int o = 32 * gg + 8 * tig;
        x0[gg] = *reinterpret_cast<const uint2 *>(slot + r0 * 128 +
                                                  ((((o >> 4) ^ (r0 & 7)) << 4) | (o & 15)));
        x1[gg] = *reinterpret_cast<const uint2 *>(slot + r1 * 128 +
                                                  ((((o >> 4) ^ (r1 & 7)) << 4) | (o & 15)));
    }
    float Dr[4][4];
    resid_mma(Dr, x0, x1, Q);
    float sr0[4], sr1[4];
    const uint2 *rs = reinterpret_cast<const uint2 *>(slot + kSlotRScale);
    unpack4h(rs[r0], sr0);
    unpack4h(rs[r1], sr1);
    const float sm = a.sm_scale;
    const bool v0 = blk * kPage + r0 < n, v1 = blk * kPage + r1 < n;
    const float s00 = v0 ? est.x + corr_score(Dr, 0, sr0, Q.qs[0], sm) : -INFINITY;
    const float s01 = v0 ? est.y + corr_score(Dr, 1, sr0, Q.qs[1], sm) : -INFINITY;
    const float s10 = v1 ? est.z + corr_score(Dr, 2, sr1, Q.qs[0], sm) : -INFINITY;
    const float s11 = v1 ? est.w + corr_score(Dr, 3, sr1, Q.qs[1], sm) : -INFINITY;

    // online softmax, heads 2tig (0) and 2tig+1 (1). The running reference m starts at the
    // pseudo-max m~ (an exact score of an always-kept token) and is raised only when a score
    // exceeds it by more than kRescaleMargin: exp(s - m) then stays below e^kRescaleMargin and the
    // common tile needs no max reduction and no rescaling of O.
    const bool over = s00 > R.m0 + kRescaleMargin || s10 > R.m0 + kRescaleMargin ||
                      s01 > R.m1 + kRescaleMargin || s11 > R.m1 + kRescaleMargin;
    if (__any_sync(0xffffffffu, over)) {
        float mx0 = fmaxf(s00, s10), mx1 = fmaxf(s01, s11);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
        }
        const float mn0 = fmaxf(R.m0, mx0), mn1 = fmaxf(R.m1, mx1);
        const float al0 = R.m0 == -INFINITY ? 0.0f : exp2f((R.m0 - mn0) * kLog2e);
        const float al1 = R.m1 == -INFINITY ? 0.0f : exp2f((R.m1 - mn1) * kLog2e);
        R.m0 = mn0;
        R.m1 = mn1;
        R.l0 *= al0;
        R.l1 *= al1;
#pragma unroll
        for (int md = 0; md < 8; md++) {
            R.o[md][0] *= al0;
            R.o[md][1] *= al1;
            R.o[md][2] *= al0;
            R.o[md][3] *= al1;
        }
    }
    const float p00 = s00 == -INFINITY ? 0.0f : exp2f((s00 - R.m0) * kLog2e);
    const float p01 = s01 == -INFINITY ? 0.0f : exp2f((s01 - R.m1) * kLog2e);
    const float p10 = s10 == -INFINITY ? 0.0f : exp2f((s10 - R.m0) * kLog2e);
    const float p11 = s11 == -INFINITY ? 0.0f : exp2f((s11 - R.m1) * kLog2e);
    R.l0 += p00 + p10;
    R.l1 += p01 + p11;
    // P^T fragments, bf16 hi + lo
    const uint32_t h0 = pack_bf16x2(p00, p01), h1 = pack_bf16x2(p10, p11);
    const uint32_t l0 = pack_bf16x2(p00 - __uint_as_float(h0 << 16),
                                    p01 - __uint_as_float(h0 & 0xffff0000u));
    const uint32_t l1 = pack_bf16x2(p10 - __uint_as_float(h1 << 16),
                                    p11 - __uint_as_float(h1 & 0xffff0000u));
    const uint32_t bh0 = movmatrix_trans(h0), bh1 = movmatrix_trans(h1);
    const uint32_t bl0 = movmatrix_trans(l0), bl1 = movmatrix_trans(l1);
    // V^T fragments by ldmatrix.trans from the swizzled tile (16-byte chunk c of row r is stored
    // at chunk c ^ (r % 8))
    const int mi = lane >> 3, jr = lane & 7;
    const int tok = 16 * mt + ((mi >> 1) << 3) + jr;
    const uint32_t vrow = smem_u32(slot + kSlotV) + tok * 128;
#pragma unroll
    for (int md = 0; md < 8; md++) {
        const int chunk = 2 * (md & 3) + (mi & 1);
        const uint32_t addr = vrow + (md >> 2) * 8192 + ((chunk ^ jr) << 4);
        uint32_t v0r, v1r, v2r, v3r;
        ldmatrix_x4_trans(v0r, v1r, v2r, v3r, addr);
        mma_bf16(R.o[md], v0r, v1r, v2r, v3r, bh0, bh1);
        mma_bf16(R.o[md], v0r, v1r, v2r, v3r, bl0, bl1);
    }
}

// Merge another warp's softmax state (reference maxima pm0/pm1, sums pl0/pl1, O^T in `src`)
// into this warp's state.
__device__ __forceinline__ void absorb(RefineState &R, float pm0, float pm1, float pl0, float pl1,
                                       const float *src, int lane) {
    const float M0 = fmaxf(R.m0, pm0), M1 = fmaxf(R.m1, pm1);
    const float fa0 = R.m0 == -INFINITY ? 0.0f : exp2f((R.m0 - M0) * kLog2e);
    const float fa1 = R.m1 == -INFINITY ? 0.0f : exp2f((R.m1 - M1) * kLog2e);
    const float fb0 = pm0 == -INFINITY ? 0.0f : exp2f((pm0 - M0) * kLog2e);
    const float fb1 = pm1 == -INFINITY ? 0.0f : exp2f((pm1 - M1) * kLog2e);
#pragma unroll
    for (int md = 0; md < 8; md++) {
        R.o[md][0] = fmaf(R.o[md][0], fa0, fb0 * src[(md * 4 + 0) * 32 + lane]);
        R.o[md][1] = fmaf(R.o[md][1], fa1, fb1 * src[(md * 4 + 1) * 32 + lane]);
        R.o[md][2] = fmaf(R.o[md][2], fa0, fb0 * src[(md * 4 + 2) * 32 + lane]);
        R.o[md][3] = fmaf(R.o[md][3], fa1, fb1 * src[(md * 4 + 3) * 32 + lane]);
    }
    R.l0 = fmaf(R.l0, fa0, fb0 * pl0);
    R.l1 = fmaf(R.l1, fa1, fb1 * pl1);
    R.m0 = M0;
    R.m1 = M1;
}

// Combine the 12 consumer warps' softmax states into this CTA's record for the unit (three
// pairwise rounds through the score buffers, which are free at a unit's end); the last CTA of the
// unit (atomic ticket, no waiting) then merges all records of the unit into the output.
__device__ __forceinline__ void combine_unit(const DecodeArgs &a, const Smem &S, const Sub &s,
                                             RefineState &R, int cta, int ncta, int64_t T,
                                             int warp, int lane) {
    Misc *m = S.misc;
    const int g = lane >> 2, tig = lane & 3, tid = warp * 32 + lane;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {  // this warp's sums over its 16-token rows
        R.l0 += __shfl_xor_sync(0xffffffffu, R.l0, o);
        R.l1 += __shfl_xor_sync(0xffffffffu, R.l1, o);
    }
    float *buf = reinterpret_cast<float *>(S.shat);
    constexpr int kWarpFloats = kCombineWarpBytes / 4;
    named_barrier_sync(1, kConsumers);  // every warp is done reading its scores
    // rounds: warps [half, 2 half) hand their state to warps [0, half)
    const int halves[3] = {6, 3, 1};
#pragma unroll
    for (int r = 0; r < 3; r++) {
        const int half = halves[r];
        const int top = r == 0 ? 12 : (r == 1 ? 6 : 3);
        if (warp >= half && warp < top) {
            float *dst = buf + (warp - half) * kWarpFloats;
#pragma unroll
            for (int md = 0; md < 8; md++)
#pragma unroll
                for (int e = 0; e < 4; e++) dst[(md * 4 + e) * 32 + lane] = R.o[md][e];
            if (g == 0) {
                m->cm[warp][2 * tig] = R.m0;
                m->cm[warp][2 * tig + 1] = R.m1;
                m->cl[warp][2 * tig] = R.l0;
                m->cl[warp][2 * tig + 1] = R.l1;
            }
        }
        named_barrier_sync(1, kConsumers);
        // round 2 hands 3 warps to 1: warps 1 and 2 both go to warp 0
        for (int p = warp + half; p < top && warp < half; p += half) {
            absorb(R, m->cm[p][2 * tig], m->cm[p][2 * tig + 1], m->cl[p][2 * tig],
                   m->cl[p][2 * tig + 1], buf + (p - half) * kWarpFloats, lane);
            if (r < 2) break;
        }
        named_barrier_sync(1, kConsumers);
    }
    const int u = s.b * a.Hkv + s.h;
    if (warp == 0) {
        float *rec = a.ws_part + (size_t)(u + cta) * a.G * kPartStride;
        const int h0 = 2 * tig, h1 = 2 * tig + 1;
#pragma unroll
        for (int md = 0; md < 8; md++) {
            const int d = 16 * md + g;
            if (h0 < a.G) {
                rec[h0 * kPartStride + d] = R.o[md][0];
                rec[h0 * kPartStride + d + 8] = R.o[md][2];
            }
            if (h1 < a.G) {
                rec[h1 * kPartStride + d] = R.o[md][1];
                rec[h1 * kPartStride + d + 8] = R.o[md][3];
            }
        }
        if (g == 0) {
            if (h0 < a.G) {
                rec[h0 * kPartStride + kD] = R.m0;
                rec[h0 * kPartStride + kD + 1] = R.l0;
            }
            if (h1 < a.G) {
                rec[h1 * kPartStride + kD] = R.m1;
                rec[h1 * kPartStride + kD + 1] = R.l1;
            }
        }
        __threadfence();
    }
    named_barrier_sync(1, kConsumers);
    const int64_t first = s.x0 - s.jr;  // global index of the unit's first middle block
    const int cf = cta_of(first, T, ncta), cl = cta_of(first + s.nmid - 1, T, ncta);
    if (tid == 0) {
        uint32_t last = 1;
        if (cl > cf) {
            int *cnt = a.ws_cnt + u;
            const int old = atomicAdd(cnt, 1);
            last = old == cl - cf;
            if (last) *cnt = 0;  // ready for the next call
        }
        m->merge_flag = last;
    }
    named_barrier_sync(1, kConsumers);
    if (m->merge_flag) {
        __threadfence();
        merge_unit(a, s.b, s.h, true, cf, cl, warp, kConsumerWarps, lane);
    }
    named_barrier_sync(1, kConsumers);
}

// Consumer warps (c = 0..11). Within a unit, sub-chunk t+1 is scanned before sub-chunk t is
// refined, so the refine loads of t+1 can be issued while t is being refined. At a unit's end
// the last sub-chunk is refined and combined first; the next unit's scan follows.
__device__ __forceinline__ void consumer(const MainParams &prm, const Smem &S, int cta, int ncta,
                                         int warp, int lane) {
    const DecodeArgs &a = prm.a;
    Misc *m = S.misc;
    const int grp = warp >> 2, mt = warp & 3;
    Sched sch;
    sch.init(a, cta, ncta);
    Sub cur, nxt;
    if (!sch.next(a, cur)) return;
    grid_dependency_wait();  // stage-1 results are visible from here on
    setup_unit(a, S, cur, warp, lane);
    uint32_t bad_cur = scan_sub(a, S, cur, 0, warp, lane);
    RefineState R;
    reset_refine(R, *S.unit, lane);
    int t = 0, kb = 0;
    while (true) {
        const bool has_nxt = sch.next(a, nxt);
        uint32_t bad_nxt = 0;
        if (has_nxt && !cur.last) bad_nxt = scan_sub(a, S, nxt, t + 1, warp, lane);
        const float4 *shat = reinterpret_cast<const float4 *>(S.shat + (t & 1) * kShatBuf);
        const uint32_t mask_cur = kept_mask(a, m, cur, t, bad_cur);
        if (warp == 0 && a.keep_mask && lane < cur.cnt)
            a.keep_mask[((size_t)cur.b * a.Hkv + cur.h) * a.max_blocks + cur.j0 + lane] =
                (mask_cur >> lane) & 1u;
        // this group's blocks k = grp and grp + 3; kept block number kb + (kept blocks before k)
        // is the ring position the producer gave it
#pragma unroll
        for (int q = 0; q < 2; q++) {
            const int k = grp + q * kGroups3;
            if (k >= cur.cnt || !((mask_cur >> k) & 1u)) continue;
            const int kbk = kb + __popc(mask_cur & ((1u << k) - 1u));
            const int slot = kbk % kRing;
            wait_bar(a, m, &m->ring_full[slot], (kbk / kRing) & 1);
            refine_tile(a, S.ring + slot * kSlotBytes, *S.unit, shat[(k * 4 + mt) * 32 + lane],
                        cur.j0 + k, R, mt, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(&m->ring_empty[slot]);
        }
        kb += __popc(mask_cur);
        if (cur.last) {
            combine_unit(a, S, cur, R, cta, ncta, sch.T, warp, lane);
            if (has_nxt) {  // a new unit only follows the last sub-chunk of the previous one
                setup_unit(a, S, nxt, warp, lane);
                bad_nxt = scan_sub(a, S, nxt, t + 1, warp, lane);
                reset_refine(R, *S.unit, lane);
            }
        }
        if (!has_nxt) break;
        cur = nxt;
        bad_cur = bad_nxt;
        t++;
    }
}

__global__ void __launch_bounds__(kMainThreads, 1)
    main_kernel(const __grid_constant__ MainParams prm) {
    const DecodeArgs &a = prm.a;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    Smem S;
    S.ring = base + kOffRing;
    S.thumb = base + kOffThumb;
    S.shat = base + kOffShat;
    S.unit = reinterpret_cast<UnitOps *>(base + kOffUnit);
    S.misc = reinterpret_cast<Misc *>(base + kOffMisc);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // every CTA range must hold at least one block: use at most T CTAs
    const int64_t T = total_mid_blocks(a);
    const int ncta = (int)(T < (int64_t)gridDim.x ? T : (int64_t)gridDim.x);
    const int cta = blockIdx.x;
    if (cta >= ncta) return;

    if (threadIdx.x == 0) {
        Misc *m = S.misc;
        m->aborted = 0;
        for (int i = 0; i < 4; i++) m->vote_mask[i] = 0;
        for (int i = 0; i < 2; i++) {
            mbar_init(&m->thumb_full[i], 1);
            mbar_init(&m->decision[i], kConsumerWarps);
            mbar_init(&m->ring_seen[i], 1);
        }
        for (int i = 0; i < kRing; i++) {
            mbar_init(&m->ring_full[i], 1);
            mbar_init(&m->ring_empty[i], 4);
        }
        for (int i = 0; i < kPageSlots; i++) {
            mbar_init(&m->pages_full[i], 1);
            mbar_init(&m->pages_empty[i], 2);  // thumbnail warp and ring warp
        }
        fence_barrier_init();
    }
    __syncthreads();
    if (warp < 4) {  // producer warpgroup: ring warp, page warp, thumbnail warp, one idle warp
        regs_decrease<kProducerRegs>();
        if (warp == 0) ring_issuer(prm, S, lane);
        else if (warp == 1) pager(a, S, cta, ncta, lane);
        else if (warp == 2) thumb_issuer(a, S, lane);
    } else {
        regs_increase<kConsumerRegs>();
        consumer(prm, S, cta, ncta, warp - 4, lane);
    }
}

// ------------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D map over [rows][inner] elements with a box of 64 rows x box_inner elements, 128B swizzle.
static bool make_map(CUtensorMap *map, CUtensorMapDataType type, void *ptr, uint64_t inner,
                     uint64_t rows, uint64_t row_bytes, uint32_t box_inner) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, (cuuint32_t)kPage};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, type, 2, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_decode(const DecodeArgs &a, int main_ctas, cudaStream_t stream) {
    static bool attr_done = false;
    if (!attr_done) {
        const cudaError_t e = cudaFuncSetAttribute(
            main_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    MainParams prm;
    memset(&prm, 0, sizeof prm);
    prm.a = a;
    const uint64_t rows = (uint64_t)a.P * a.Hkv * kPage;
    if (!make_map(&prm.tm_resid, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<int8_t *>(a.resid),
                  kD, rows, kD, kD) ||
        !make_map(&prm.tm_v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<__nv_bfloat16 *>(a.v),
                  kD, rows, kD * 2, 64))
        return cudaErrorInvalidValue;

    stage1_kernel<<<dim3(a.nf > 0 ? a.nf : 1, a.B * a.Hkv), 128, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (a.prof_start) cudaEventRecord(a.prof_start, stream);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(main_ctas);
    cfg.blockDim = dim3(kMainThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, main_kernel, prm);
    if (e != cudaSuccess) return e;
    if (a.prof_stop) cudaEventRecord(a.prof_stop, stream);
    return cudaGetLastError();
}

}  // namespace ffd
