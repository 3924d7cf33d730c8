// select.cu -- the comparison block selectors Top-k and Top-p on the FFD thumbnails.
//
// Source: "Faster Than Flash", Problem statement (the selection dilemma: a fixed-budget Top-k does
// not adapt to the attention entropy, a distribution-adaptive Top-p needs a global softmax and a
// sort, which breaks a streaming pipeline). Both rank the same 64-token blocks as Top-delta, on
// the same provisional scores s^_ij = sm * q_i . x^2_j (Methodology §3, stage 2), and keep the same
// always-kept sink and local blocks (Methodology §2). Definitions (the pages give none in detail):
//   Top-k: importance of block c = max over the group's heads i and its tokens j < n of s^_ij;
//          keep the k non-forced blocks of largest importance (ties: lower block index first).
//   Top-p: per head i, P_ij = softmax over all j < n of s^_ij, block mass m_ic = sum of P_ij over
//          the block; rank blocks by mass (descending, ties: lower index first) and keep a block
//          when the masses ranked before it sum to less than p; union over the heads.
//
// Two passes, as the rules require (the whole sequence must be scored before anything is chosen):
//   block_stats_kernel  streams every thumbnail record once and writes, per block, its importance
//                       and, per head, the block's (max s^, sum of e^(s^ - max)) pair;
//   select_kernel       one CTA per (sequence, KV head), and for Top-p per query head too: for
//                       Top-k a radix select of the k-th (importance, index) key in shared
//                       memory; for Top-p the global softmax normalisation and a mass-weighted
//                       radix select of the cut (no sort: four passes over 8-bit digits of the
//                       blocks' mass keys, each a count and mass histogram); then the kept bytes.
// The chosen mask then goes to the decode kernel as a given mask (ffd_decode_attention_masked).
#include "common.cuh"
#include "ptx.cuh"
#include "scan.cuh"

namespace ffd {

namespace {

constexpr int kStatBlocks = 32;    // blocks per CTA of the statistics pass
constexpr int kStatWarps = 4;      // its warps; warp w takes blocks w, w + 4, ...
constexpr int kSelThreads = 1024;  // threads of the selection CTA
constexpr int kSelMaxBlocks = 16384;
constexpr float kLog2e = 1.4426950408889634f;  // 1 / ln 2

__device__ __forceinline__ int stat_len(const DecodeArgs &a, int b) {
    int n = a.seq_lens[b];
    const int cap = a.max_blocks * kPage;
    if (n < 0 || n > cap) {
        if (threadIdx.x == 0 && blockIdx.x == 0) raise_error(a.err, FFD_ERRBIT_BOUNDS);
        n = n < 0 ? 0 : cap;
    }
    return n;
}

// Pass 1. CTA (x, u) takes blocks kStatBlocks x .. of unit u: it writes their initial keep-mask
// bytes (1 for a sink or local block, 0 otherwise, 0 past the sequence); then each warp takes
// every fourth of those blocks on its own, with no CTA barrier: lane 0 brings the block's
// thumbnail record into the warp's two shared-memory stages by one bulk copy (the next block's
// copy is in flight while the current one is scored), and the warp scores all 64 rows for every
// head of the group (four scan_tile m-tiles). Block importance -> imp[u][c]; per head (max,
// sum e^(s^ - max)) -> ml[u][c][G].
__global__ void __launch_bounds__(128) block_stats_kernel(DecodeArgs a, float *imp, float2 *ml) {
    __shared__ __align__(128) uint8_t recs[kStatWarps][2][kThumbRec];
    __shared__ __align__(8) uint64_t full[kStatWarps][2];
    const int u = blockIdx.y;
    const int b = u / a.Hkv, h = u - b * a.Hkv;
    const int n = stat_len(a, b);
    const int nb = (n + kPage - 1) / kPage;
    const int c0 = blockIdx.x * kStatBlocks;
    const size_t row = (size_t)u * a.max_blocks;
    {
        const ForcedBlocks fb(n, a.S, a.L);
        for (int k = threadIdx.x; k < kStatBlocks; k += blockDim.x) {
            const int c = c0 + k;
            if (c < a.max_blocks) a.keep_mask[row + c] = c < nb && fb.forced(c);
        }
    }
    const int cend = nb < c0 + kStatBlocks ? nb : c0 + kStatBlocks;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (c0 + warp >= cend) return;  // warp-uniform; no CTA barrier follows
    const int g = lane >> 2, tig = lane & 3;
    const uint32_t m0 = 0x00030003u << (2 * tig);
    const int h0 = 2 * tig, h1 = 2 * tig + 1;
    const bool w0 = h0 < a.G, w1 = h1 < a.G;
    const int32_t *bt = a.block_table + (size_t)b * a.max_blocks;
    if (lane == 0) {
        mbar_init(&full[warp][0], 1);
        mbar_init(&full[warp][1], 1);
        fence_barrier_init();
    }
    __syncwarp();
    // The copy of block c into stage st (false, nothing issued, for a page outside [0, P)).
    auto issue = [&](int c, int st) -> bool {
        int page = 0;
        if (lane == 0) page = bt[c];
        page = __shfl_sync(0xffffffffu, page, 0);
        if (page < 0 || page >= a.P) {
            if (lane == 0) raise_error(a.err, FFD_ERRBIT_BOUNDS);
            return false;
        }
        if (lane == 0) {
            mbar_arrive_expect_tx(&full[warp][st], kThumbRec);
            tma_load_1d(recs[warp][st], a.thumb + ((size_t)page * a.Hkv + h) * kThumbRec,
                        kThumbRec, &full[warp][st]);
        }
        return true;
    };
    uint32_t phases = 0u;  // bit st: parity of stage st's next completion
    auto wait_stage = [&](int st) -> bool {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&full[warp][st], (phases >> st) & 1u)) {
            if (globaltimer_ns() - t0 > a.wait_ns) {
                phases ^= 1u << st;
                if (lane == 0) raise_error(a.err, FFD_ERRBIT_TIMEOUT);
                return false;
            }
        }
        phases ^= 1u << st;
        return true;
    };
    ThumbOps Q;
    load_thumb_ops(a, b, h, lane, Q);  // overlaps the first copies
    // scores as scan_tile_raw's times sm * 2^(133 - kKq): bit for bit scan_tile's
    float qsr[2][4];
#pragma unroll
    for (int i = 0; i < 2; i++)
#pragma unroll
        for (int gg = 0; gg < 4; gg++) qsr[i][gg] = Q.qs[i][gg] * (1.0f / kUnscale);
    const float post = a.sm_scale * kUnscale;
    int c = c0 + warp, st = 0;
    uint32_t have = (issue(c, 0) ? 1u : 0u);
    if (c + kStatWarps < cend && issue(c + kStatWarps, 1)) have |= 2u;
    bool ok = true;
    for (; c < cend; c += kStatWarps, st ^= 1) {
        const bool good = (have >> st) & 1u;
        if (good) {
            ok = __all_sync(0xffffffffu, wait_stage(st));
            if (!ok) break;
        }
        const int rows = n - c * kPage < kPage ? n - c * kPage : kPage;
        float x[4][4];
#pragma unroll
        for (int mt = 0; mt < 4; mt++) {
            const int r0 = 16 * mt + g, r1 = r0 + 8;
            float4 e = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            if (good) {
                e = scan_tile_raw(recs[warp][st], r0, r1, m0, Q, qsr);
                e.x *= post;
                e.y *= post;
                e.z *= post;
                e.w *= post;
            }
            const bool v0 = r0 < rows, v1 = r1 < rows;
            x[mt][0] = v0 && w0 ? e.x : -INFINITY;
            x[mt][1] = v0 && w1 ? e.y : -INFINITY;
            x[mt][2] = v1 && w0 ? e.z : -INFINITY;
            x[mt][3] = v1 && w1 ? e.w : -INFINITY;
        }
        __syncwarp();  // every lane has read the stage: it can be refilled
        have &= ~(1u << st);
        if (c + 2 * kStatWarps < cend && issue(c + 2 * kStatWarps, st)) have |= 1u << st;
        // per head: max over the block's 64 rows (lanes with the same tig), then the sum
        float mh0 = -INFINITY, mh1 = -INFINITY;
#pragma unroll
        for (int mt = 0; mt < 4; mt++) {
            mh0 = fmaxf(mh0, fmaxf(x[mt][0], x[mt][2]));
            mh1 = fmaxf(mh1, fmaxf(x[mt][1], x[mt][3]));
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            mh0 = fmaxf(mh0, __shfl_xor_sync(0xffffffffu, mh0, o));
            mh1 = fmaxf(mh1, __shfl_xor_sync(0xffffffffu, mh1, o));
        }
        const float b0 = mh0 == -INFINITY ? 0.0f : mh0, b1 = mh1 == -INFINITY ? 0.0f : mh1;
        float l0 = 0.0f, l1 = 0.0f;
#pragma unroll
        for (int mt = 0; mt < 4; mt++) {
            l0 += ex2_approx((x[mt][0] - b0) * kLog2e) + ex2_approx((x[mt][2] - b0) * kLog2e);
            l1 += ex2_approx((x[mt][1] - b1) * kLog2e) + ex2_approx((x[mt][3] - b1) * kLog2e);
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, o);
            l1 += __shfl_xor_sync(0xffffffffu, l1, o);
        }
        // importance: max over every head (the quads' heads, then across quads)
        float im = fmaxf(mh0, mh1);
        im = fmaxf(im, __shfl_xor_sync(0xffffffffu, im, 1));
        im = fmaxf(im, __shfl_xor_sync(0xffffffffu, im, 2));
        const size_t slot = row + c;
        if (lane == 0) imp[slot] = im;
        if (g == 0) {
            if (w0) ml[slot * a.G + h0] = make_float2(mh0, l0);
            if (w1) ml[slot * a.G + h1] = make_float2(mh1, l1);
        }
    }
    // copies still in flight into this warp's stages are waited for (bounded) before it exits
    for (int k = 0; k < 2; k++)
        if ((have >> k) & 1u) __all_sync(0xffffffffu, wait_stage(k));
}

// Float -> unsigned key whose unsigned order is the float's order (NaN never occurs here).
__device__ __forceinline__ uint32_t ordered(float f) {
    const uint32_t x = __float_as_uint(f);
    return (x & 0x80000000u) ? ~x : (x | 0x80000000u);
}

// Float -> float of an ordered key (the inverse of ordered).
__device__ __forceinline__ float unordered(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

__device__ __forceinline__ float block_max_reduce(float v, float *red) {
    v = warp_max(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = -INFINITY;
    for (int w = 0; w < kSelThreads / 32; w++) r = fmaxf(r, red[w]);
    __syncthreads();
    return r;
}

__device__ __forceinline__ float block_sum_reduce(float v, float *red) {
    v = warp_sum(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = 0.0f;
    for (int w = 0; w < kSelThreads / 32; w++) r += red[w];
    __syncthreads();
    return r;
}

// Pass 2: CTA (u, i) of kSelThreads threads: unit u, and for Top-p its head i (Top-k has one CTA
// per unit). It only raises keep-mask bytes to 1 (pass 1 wrote the initial mask), so the heads of
// a unit OR their choices without further synchronisation. Shared memory: keys [N] u64, mass [N]
// f32, N = the block count rounded up to a power of two.
__global__ void __launch_bounds__(kSelThreads) select_kernel(DecodeArgs a, int selector, float budget,
                                                             int N, const float *imp,
                                                             const float2 *ml) {
    extern __shared__ __align__(16) unsigned char smem[];
    uint64_t *key = reinterpret_cast<uint64_t *>(smem);
    float *mass = reinterpret_cast<float *>(key + N);
    __shared__ float red[kSelThreads / 32];
    const int u = blockIdx.x, hh = blockIdx.y;
    const int b = u / a.Hkv;
    int n = a.seq_lens[b];
    const int cap = a.max_blocks * kPage;
    n = n < 0 ? 0 : (n > cap ? cap : n);
    const int nb = (n + kPage - 1) / kPage;
    const ForcedBlocks fb(n, a.S, a.L);
    const size_t row = (size_t)u * a.max_blocks;
    uint8_t *keep = a.keep_mask + row;

    if (selector == FFD_SELECT_TOPK) {
        for (int c = threadIdx.x; c < N; c += blockDim.x) {
            const float v = c < nb ? imp[row + c] : -INFINITY;
            const bool eligible = c < nb && !fb.forced(c) && v != -INFINITY;
            key[c] = eligible ? ((uint64_t)(~ordered(v)) << 32) | (uint32_t)c : ~0ull;
        }
        // the k smallest keys (unique: the block index is in the low bits) by a radix select of
        // the k-th smallest, 8 bits a pass from the top, instead of a full sort
        const int k = (int)budget;
        __shared__ unsigned int hist[256];
        __shared__ uint64_t s_prefix;
        __shared__ int s_elig, s_kk;
        if (threadIdx.x == 0) {
            s_prefix = 0;
            s_elig = 0;
            s_kk = k;
        }
        __syncthreads();
        int mine = 0;
        for (int c = threadIdx.x; c < N; c += blockDim.x) mine += key[c] != ~0ull;
        mine = __reduce_add_sync(0xffffffffu, mine);
        if ((threadIdx.x & 31) == 0 && mine) atomicAdd(&s_elig, mine);
        __syncthreads();
        const int elig = s_elig;
        if (k <= 0) return;
        uint64_t kth = ~0ull - 1;  // k >= eligible blocks: every eligible key
        if (k < elig) {
            for (int shift = 56; shift >= 0; shift -= 8) {
                for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
                __syncthreads();
                const uint64_t hi_mask = shift == 56 ? 0ull : (~0ull << (shift + 8));
                const uint64_t prefix = s_prefix;
                for (int c = threadIdx.x; c < N; c += blockDim.x) {
                    const uint64_t x = key[c];
                    if ((x & hi_mask) == prefix) atomicAdd(&hist[(x >> shift) & 255u], 1u);
                }
                __syncthreads();
                if (threadIdx.x < 32) {  // the bin holding the kk-th key: 8 bins per lane
                    const int lane = threadIdx.x;
                    unsigned int cnt8[8], tot = 0;
#pragma unroll
                    for (int j = 0; j < 8; j++) {
                        cnt8[j] = hist[8 * lane + j];
                        tot += cnt8[j];
                    }
                    unsigned int incl = tot;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const unsigned int y = __shfl_up_sync(0xffffffffu, incl, o);
                        if (lane >= o) incl += y;
                    }
                    const unsigned int kk = (unsigned int)s_kk;
                    const unsigned int before = incl - tot;
                    if (before < kk && kk <= incl) {  // exactly one lane
                        unsigned int acc = before;
                        int d = 0;
                        for (; d < 8; d++) {
                            if (acc + cnt8[d] >= kk) break;
                            acc += cnt8[d];
                        }
                        s_prefix = prefix | ((uint64_t)(8 * lane + d) << shift);
                        s_kk = (int)(kk - acc);
                    }
                }
                __syncthreads();
            }
            kth = s_prefix;
        }
        for (int c = threadIdx.x; c < N; c += blockDim.x) {
            const uint64_t x = key[c];
            if (x != ~0ull && x <= kth) keep[(uint32_t)x] = 1;
        }
        return;
    }
    // Top-p, head hh: global softmax normalisation over the blocks, M = max, L = sum e^(m - M) l
    float lm = -INFINITY;
    for (int c = threadIdx.x; c < nb; c += blockDim.x)
        if (ml[(row + c) * a.G + hh].y > 0.0f) lm = fmaxf(lm, ml[(row + c) * a.G + hh].x);
    const float M = block_max_reduce(lm, red);
    float ls = 0.0f;
    for (int c = threadIdx.x; c < nb; c += blockDim.x) {
        const float2 v = ml[(row + c) * a.G + hh];
        const float w = v.y > 0.0f ? v.y * ex2_approx((v.x - M) * kLog2e) : 0.0f;
        mass[c] = w;
        ls += w;
    }
    const float Ltot = block_sum_reduce(ls, red);
    const float inv = Ltot > 0.0f ? 1.0f / Ltot : 0.0f;
    for (int c = threadIdx.x; c < nb; c += blockDim.x) mass[c] *= inv;
    __syncthreads();
    if (!(budget > 0.0f)) return;  // only the forced blocks (pass 1 kept them)
    // The cut: blocks ranked by (mass descending, index ascending) are kept while the mass ranked
    // before them is below p. With keys k = ordered(mass), the boundary key K* is found 8 bits at
    // a time from the top: among the blocks whose key matches the digits found so far, a count and
    // a mass histogram of the next digit; every block in a digit bucket above the boundary bucket
    // B is kept (all of them lie before the cut), every block below it is dropped, and the search
    // continues inside B with `before` raised by the mass of the buckets above it. B is the lowest
    // non-empty bucket whose higher buckets leave the running mass below p. The masses are summed
    // in 2^-31 fixed point (exact and order-independent; the cut moves by at most nb 2^-32), and
    // the lanes of a warp that hit the same bucket add once (match + reduce) before the atomics.
    __shared__ unsigned int hcnt[256];
    __shared__ unsigned int hmass[256];
    __shared__ unsigned long long s_before;
    __shared__ int s_bucket;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float kFx = 2147483648.0f;  // 2^31
    const unsigned long long p_fx = (unsigned long long)((double)budget * 2147483648.0);
    uint32_t prefix = 0u, known = 0u;
    unsigned long long before = 0ull;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += blockDim.x) {
            hcnt[i] = 0u;
            hmass[i] = 0u;
        }
        __syncthreads();
        for (int cb = warp * 32; cb < nb; cb += blockDim.x) {  // warp-converged
            const int c = cb + lane;
            const float mc = c < nb ? mass[c] : 0.0f;
            const uint32_t k = ordered(mc);
            const bool valid = c < nb && (k & known) == prefix;
            const unsigned int active = __ballot_sync(0xffffffffu, valid);
            if (valid) {
                const uint32_t d = (k >> shift) & 255u;
                const unsigned int peers = __match_any_sync(active, d);
                const unsigned int sum = __reduce_add_sync(peers, __float2uint_rn(mc * kFx));
                if (lane == __ffs(peers) - 1) {
                    atomicAdd(&hcnt[d], (unsigned int)__popc(peers));
                    atomicAdd(&hmass[d], sum);
                }
            }
        }
        __syncthreads();
        if (warp == 0) {  // lane L holds digits 8L .. 8L+7
            unsigned long long mz[8];
            unsigned int cz[8];
            unsigned long long tot = 0ull;
#pragma unroll
            for (int j = 0; j < 8; j++) {
                mz[j] = hmass[8 * lane + j];
                cz[j] = hcnt[8 * lane + j];
                tot += mz[j];
            }
            // mass of the digits above this lane's: suffix over the higher lanes
            unsigned long long above = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long y = __shfl_down_sync(0xffffffffu, above, o);
                if (lane + o < 32) above += y;
            }
            above -= tot;
            int best = 256;  // the lowest qualifying non-empty digit of this lane
            unsigned long long best_before = 0ull;
            unsigned long long run = above;  // mass of the digits above digit 8L + j
#pragma unroll
            for (int j = 7; j >= 0; j--) {
                if (cz[j] > 0u && before + run < p_fx) {
                    best = 8 * lane + j;
                    best_before = before + run;
                }
                run += mz[j];
            }
            int lo = best;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
            if (best == lo && lo < 256) {  // exactly one lane
                s_bucket = lo;
                s_before = best_before;
            }
            if (lane == 0 && lo == 256) s_bucket = 256;  // no block in range: nothing more to keep
        }
        __syncthreads();
        const int B = s_bucket;
        if (B == 256) return;  // the blocks matching the prefix are all past the cut
        before = s_before;
        prefix |= (uint32_t)B << shift;
        known |= 255u << shift;
        __syncthreads();  // the histograms are cleared again only after every thread read B
    }
    // keys above K* = prefix are kept; among the blocks of key K* (equal masses w), in index order,
    // the j-th is kept while before + j w < p: a CTA-wide count of the ties before each block
    const unsigned long long w_fx = __float2uint_rn(unordered(prefix) * kFx);
    const int per = (nb + (int)blockDim.x - 1) / (int)blockDim.x;
    const int c0 = threadIdx.x * per, c1 = c0 + per < nb ? c0 + per : nb;
    int ties = 0;
    for (int c = c0; c < c1; c++) ties += ordered(mass[c]) == prefix;
    int incl = ties;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    __shared__ int wties[kSelThreads / 32];
    if (lane == 31) wties[warp] = incl;
    __syncthreads();
    int rank = incl - ties;
    for (int v = 0; v < warp; v++) rank += wties[v];
    for (int c = c0; c < c1; c++) {
        const uint32_t k = ordered(mass[c]);
        if (k > prefix) {
            keep[c] = 1;
        } else if (k == prefix) {
            if (before + (unsigned long long)rank * w_fx < p_fx) keep[c] = 1;
            rank++;
        }
    }
}

}  // namespace

size_t select_smem_bytes(int max_blocks) {
    int N = 1;
    while (N < max_blocks) N <<= 1;
    return (size_t)N * (8 + 4);
}

int select_max_blocks() { return kSelMaxBlocks; }

cudaError_t launch_select(const DecodeArgs &a, int selector, float budget, float *imp, float2 *ml,
                          cudaStream_t stream) {
    const int units = a.B * a.Hkv;
    dim3 g1((a.max_blocks + kStatBlocks - 1) / kStatBlocks, units);
    block_stats_kernel<<<g1, 128, 0, stream>>>(a, imp, ml);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    int N = 1;
    while (N < a.max_blocks) N <<= 1;
    const size_t smem = select_smem_bytes(a.max_blocks);
    static int smem_set[kMaxDevicesTracked];
    if (smem > 48 * 1024) {
        e = raise_smem_limit(select_kernel, (int)smem, smem_set);
        if (e != cudaSuccess) return e;
    }
    const dim3 g2(units, selector == FFD_SELECT_TOPP ? a.G : 1);
    select_kernel<<<g2, kSelThreads, smem, stream>>>(a, selector, budget, N, imp, ml);
    return cudaGetLastError();
}

}  // namespace ffd
