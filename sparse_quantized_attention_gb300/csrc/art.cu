// art.cu -- run-time termination of the attention over a unit's kept blocks (ART).
//
// Source: "ART: Attention Run-time Termination" (technical summary page), §2.2 (the partial
// output is watched as KV blocks are added; its magnitude change and direction change between
// consecutive probes must both fall below the thresholds tau and phi), §2.3 (the criterion must
// hold `patience` times in a row) and §2.4 (the traversal can be reordered because online softmax
// is permutation invariant; block 0, an attention sink, is evaluated first). The FFD pages call
// ART an orthogonal layer; here it runs over the blocks an FFD step kept (or over every block).
// Readings, shared with the CPU statement:
//   * the probe of head i is its whole normalised partial output P_i = o_i / l_i;
//   * d_scale = max_i | |P_i(t)| - |P_i(t-1)| | / |P_i(t-1)|,
//     d_direction = max_i (1 - cos(P_i(t), P_i(t-1))) over the heads of the GQA group;
//   * the criterion is strict, first checked after the second block; the computation stops after
//     the block at which it has held `patience` times in a row;
//   * the order is block 0, then the kept blocks from the most recent to the oldest.
//
// The criterion makes one unit's traversal sequential, so the parallelism is across units, the
// regime the page reports its gains in (large batches): one CTA of 128 threads (one refine group
// of the decode kernel) walks one (sequence, KV head) unit. A block's three records (thumbnail
// 3 KB, residual 8.5 KB, V 16 KB as a swizzled tensor tile) are brought into shared memory by
// bulk copies into a ring of kArtStages stages: the next kArtStages - 1 blocks' copies are in
// flight while the current block is processed, so the walk runs at the rate of the arithmetic
// rather than of the copy latency. Per block, warp mt computes the exact scores of rows 16mt .. 16mt+15 for every head
// (the thumbnail + residual tensor-core tile of scan.cuh), and the group's online softmax and P.V
// on the tensor cores (softmax_pv of splitkv.cuh, P as bf16 hi + lo parts) fold the block in; warp
// mt then holds O^T for channels 32mt .. 32mt+31. The probe needs, per head, l, then |P|^2, then
// for the direction |P/|P| - P'/|P'||^2 = 2 (1 - cos), which keeps its precision when the two
// directions are close: three CTA reductions per block. Every thread takes the same decision from
// the reduced values, so no broadcast is needed.
#include "common.cuh"
#include "ptx.cuh"
#include "scan.cuh"
#include "splitkv.cuh"

namespace ffd {

namespace {

constexpr int kArtThreads = 128;
// One block's records in shared memory: the V tile first (1 KB aligned for the 128-byte swizzle).
constexpr int kArtV = 0;
constexpr int kArtThumb = kPage * kD * 2;
constexpr int kArtResid = kArtThumb + kThumbRec;
constexpr int kArtStage = 28672;  // 28 KB: a multiple of 1 KB
static_assert(kArtResid + kResidRec <= kArtStage && kArtStage % 1024 == 0, "stage layout");
constexpr uint32_t kArtStageTx = kThumbRec + kResidRec + kPage * kD * 2;
constexpr int kArtStages = 5;
constexpr int kArtPx = kArtStages * kArtStage;       // two P^T fragment buffers
constexpr int kArtSmem = kArtPx + 2 * kPxBuf + 1024;  // + slack to align the base to 1 KB

// The shared control block softmax_pv expects (one refine group), and the probe reductions.
struct ArtCtl {
    uint32_t over[1][2][4];
    float wmax[1][2][4][kMaxG];
    float red_l[4][kMaxG];  // [warp][head]: l partial sums
    float red_n[4][kMaxG];  // [warp][head]: |o|^2 partial sums
    float red_d[4][kMaxG];  // [warp][head]: direction-change partial sums
    int list[kArtThreads];    // kept blocks of the current chunk, most recent first
    int wc[4];
    uint64_t full[kArtStages];
};

struct ArtParams {
    CUtensorMap tm_v;
    DecodeArgs a;
    float tau, phi;
    int patience;
    int32_t *used;
};

// Sum over the 8 lanes of a warp that share tig (one head pair).
__device__ __forceinline__ float quad_col_sum(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    v += __shfl_xor_sync(0xffffffffu, v, 16);
    return v;
}

// d_scale and 1 - cos of one head (a zero probe on one side only counts as orthogonal).
__device__ __forceinline__ void head_metrics(float nc, float np, float dd, float &ds, float &dr) {
    ds = np > 0.0f ? fabsf(nc - np) / np : nc;
    dr = (nc > 0.0f && np > 0.0f) ? 0.5f * dd : ((nc == 0.0f && np == 0.0f) ? 0.0f : 1.0f);
}

__global__ void __launch_bounds__(kArtThreads) art_kernel(const __grid_constant__ ArtParams prm) {
    const DecodeArgs &a = prm.a;
    extern __shared__ uint8_t art_raw[];
    uint8_t *base = align_shared<1024>(art_raw);
    __shared__ ArtCtl ctl;
    const int u = blockIdx.x;
    const int b = u / a.Hkv, h = u - b * a.Hkv;
    const int G = a.G;
    const int n = checked_seq_len(a, b);
    const int nb = (n + kPage - 1) / kPage;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int g = lane >> 2, tig = lane & 3;
    const int r0 = 16 * warp + g, r1 = r0 + 8;
    const int h0 = 2 * tig, h1 = h0 + 1;
    const bool w0 = h0 < G, w1 = h1 < G;
    ThumbOps Q;
    ResidOps QR;
    load_thumb_ops(a, b, h, lane, Q);
    load_resid_ops(a, b, h, lane, QR);
    const int32_t *bt = a.block_table + (size_t)b * a.max_blocks;
    const uint8_t *keep = a.keep_in ? a.keep_in + (size_t)u * a.max_blocks : nullptr;
    if (t == 0) {
        for (int i = 0; i < kArtStages; i++) mbar_init(&ctl.full[i], 1);
        fence_barrier_init();
        prefetch_tensormap(&prm.tm_v);
    }
    __syncthreads();
    // Copies of block c's records into stage st; false (nothing issued) for a page outside
    // [0, P). Every thread evaluates it (block-uniform result); thread 0 issues.
    auto issue = [&](int c, int st) -> bool {
        const int page = bt[c];
        if (page < 0 || page >= a.P) {
            if (t == 0) raise_error(a.err, FFD_ERRBIT_BOUNDS);
            return false;
        }
        if (t == 0) {
            const size_t tile = (size_t)page * a.Hkv + h;
            uint8_t *d = base + st * kArtStage;
            mbar_arrive_expect_tx(&ctl.full[st], kArtStageTx);
            tma_load_3d(d + kArtV, &prm.tm_v, 0, (int)(tile * kPage), 0, &ctl.full[st]);
            tma_load_1d(d + kArtThumb, a.thumb + tile * kThumbRec, kThumbRec, &ctl.full[st]);
            tma_load_1d(d + kArtResid, a.resid + tile * kResidRec, kResidRec, &ctl.full[st]);
        }
        return true;
    };
    // Bounded wait for stage st's copies; the result is block-uniform.
    uint32_t phases = 0u;  // bit st: parity of stage st's next completion
    auto wait_stage = [&](int st) -> bool {
        const uint64_t t0 = globaltimer_ns();
        bool ok = true;
        while (!mbar_try_wait(&ctl.full[st], (phases >> st) & 1u)) {
            if (globaltimer_ns() - t0 > a.wait_ns) {
                ok = false;
                break;
            }
        }
        phases ^= 1u << st;
        ok = __syncthreads_and(ok) != 0;
        if (!ok && t == 0) raise_error(a.err, FFD_ERRBIT_TIMEOUT);
        return ok;
    };
    int hi = nb - 1;       // top block of the next chunk of the kept-block list
    int pos = 0, cnt = 0;  // read position and length of the current chunk
    // The next block of the traversal after block 0: the kept blocks from the most recent down,
    // listed 128 candidates at a time (block-uniform; the barriers are reached by every thread).
    auto advance = [&]() -> int {
        while (pos == cnt && hi >= 1) {
            const int idx = hi - t;
            const bool k = idx >= 1 && (keep == nullptr || keep[idx] != 0);
            const unsigned bal = __ballot_sync(0xffffffffu, k);
            __syncthreads();  // earlier reads of the list are done
            if (lane == 0) ctl.wc[warp] = __popc(bal);
            __syncthreads();
            int off = 0;
            for (int w = 0; w < warp; w++) off += ctl.wc[w];
            if (k) ctl.list[off + __popc(bal & ((1u << lane) - 1u))] = idx;
            cnt = (ctl.wc[0] + ctl.wc[1]) + (ctl.wc[2] + ctl.wc[3]);
            pos = 0;
            hi -= kArtThreads;
            __syncthreads();
        }
        return pos < cnt ? ctl.list[pos++] : -1;
    };

    RefineState R;
    R.m0 = R.m1 = kNoReference;  // the first block raises it through the rescale path
    R.nl0 = R.nl1 = -kNoReference * kLog2e;
    R.l0 = R.l1 = 0.0f;
#pragma unroll
    for (int i = 0; i < 2; i++) R.o[i][0] = R.o[i][1] = R.o[i][2] = R.o[i][3] = 0.0f;
    float px[2][4];                // the previous probe's direction o' / |o'|, this thread's entries
    float pn0 = 0.0f, pn1 = 0.0f;  // the previous probe's norms |P| (heads h0, h1)
    float L0 = 0.0f, L1 = 0.0f;    // the current l (heads h0, h1)
#pragma unroll
    for (int i = 0; i < 2; i++) px[i][0] = px[i][1] = px[i][2] = px[i][3] = 0.0f;
    int used = 0, streak = 0, pb = 0;

    // the ring: stage k holds the k-th next block of the traversal (blk[k] < 0: none), issued
    // (bit k of inflight) unless its page was out of range
    int blk[kArtStages];
    uint32_t inflight = 0u;
#pragma unroll
    for (int k = 0; k < kArtStages; k++) {
        blk[k] = k == 0 ? (nb > 0 ? 0 : -1) : (blk[k - 1] >= 0 ? advance() : -1);  // block 0 first
        if (blk[k] >= 0 && issue(blk[k], k)) inflight |= 1u << k;
    }
    int st = 0;
    while (blk[st] >= 0) {
        const int c = blk[st];
        const bool have = (inflight >> st) & 1u;
        if (have) {
            inflight &= ~(1u << st);
            if (!wait_stage(st)) break;  // timed out: the error word says so
        }
        if (have) {  // block-uniform
            uint8_t *sg = base + st * kArtStage;
            const int rows = n - c * kPage < kPage ? n - c * kPage : kPage;
            const float4 e = exact_tile(sg + kArtThumb, sg + kArtResid, r0, r1, tig, Q, QR,
                                        a.sm_scale);
            const bool v0 = r0 < rows, v1 = r1 < rows;
            if (rows < kPage) {  // the sequence's partial last block: V rows past it read as 0
                for (int k = t; k < (kPage - rows) * 16; k += kArtThreads) {
                    const int r = rows + (k >> 4), half = (k >> 3) & 1;
                    *reinterpret_cast<uint4 *>(sg + kArtV + half * 8192 + r * 128 + (k & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async();  // before the stage's next bulk copy
                __syncthreads();
            }
            softmax_pv(&ctl, base + kArtPx + pb * kPxBuf, sg + kArtV, v0 && w0 ? e.x : -INFINITY,
                       v0 && w1 ? e.y : -INFINITY, v1 && w0 ? e.z : -INFINITY,
                       v1 && w1 ? e.w : -INFINITY, R, 0, warp, pb, lane);
            pb ^= 1;
        }
        used++;
        // the probe, per head: l (this warp's rows, then the 4 warps), then |P|^2 of P = o / l
        // (o is the whole numerator in every warp, |P| stays below max |V|, so nothing overflows
        // however far the lazy softmax reference lags)
        {
            const float l0 = quad_col_sum(R.l0), l1 = quad_col_sum(R.l1);
            if (g == 0) {
                ctl.red_l[warp][h0] = l0;
                ctl.red_l[warp][h1] = l1;
            }
        }
        __syncthreads();
        L0 = (ctl.red_l[0][h0] + ctl.red_l[1][h0]) + (ctl.red_l[2][h0] + ctl.red_l[3][h0]);
        L1 = (ctl.red_l[0][h1] + ctl.red_l[1][h1]) + (ctl.red_l[2][h1] + ctl.red_l[3][h1]);
        const float il0 = L0 > 0.0f ? __frcp_rn(L0) : 0.0f, il1 = L1 > 0.0f ? __frcp_rn(L1) : 0.0f;
        float cur[2][4];
#pragma unroll
        for (int i = 0; i < 2; i++) {
            cur[i][0] = R.o[i][0] * il0;
            cur[i][2] = R.o[i][2] * il0;
            cur[i][1] = R.o[i][1] * il1;
            cur[i][3] = R.o[i][3] * il1;
        }
        {
            const float q0 = quad_col_sum((cur[0][0] * cur[0][0] + cur[0][2] * cur[0][2]) +
                                          (cur[1][0] * cur[1][0] + cur[1][2] * cur[1][2]));
            const float q1 = quad_col_sum((cur[0][1] * cur[0][1] + cur[0][3] * cur[0][3]) +
                                          (cur[1][1] * cur[1][1] + cur[1][3] * cur[1][3]));
            if (g == 0) {
                ctl.red_n[warp][h0] = q0;
                ctl.red_n[warp][h1] = q1;
            }
        }
        __syncthreads();
        const float N0 = (ctl.red_n[0][h0] + ctl.red_n[1][h0]) + (ctl.red_n[2][h0] + ctl.red_n[3][h0]);
        const float N1 = (ctl.red_n[0][h1] + ctl.red_n[1][h1]) + (ctl.red_n[2][h1] + ctl.red_n[3][h1]);
        const float nc0 = sqrtf(N0), nc1 = sqrtf(N1);  // |P|
        const float rn0 = N0 > 0.0f ? rsqrtf(N0) : 0.0f, rn1 = N1 > 0.0f ? rsqrtf(N1) : 0.0f;
        bool stop = false;
        if (used >= 2) {
            float d0 = 0.0f, d1 = 0.0f;
#pragma unroll
            for (int i = 0; i < 2; i++) {
                const float a0 = cur[i][0] * rn0 - px[i][0], a2 = cur[i][2] * rn0 - px[i][2];
                const float a1 = cur[i][1] * rn1 - px[i][1], a3 = cur[i][3] * rn1 - px[i][3];
                d0 = fmaf(a0, a0, fmaf(a2, a2, d0));
                d1 = fmaf(a1, a1, fmaf(a3, a3, d1));
            }
            d0 = quad_col_sum(d0);
            d1 = quad_col_sum(d1);
            if (g == 0) {
                ctl.red_d[warp][h0] = d0;
                ctl.red_d[warp][h1] = d1;
            }
            __syncthreads();
            const float D0 = (ctl.red_d[0][h0] + ctl.red_d[1][h0]) +
                             (ctl.red_d[2][h0] + ctl.red_d[3][h0]);
            const float D1 = (ctl.red_d[0][h1] + ctl.red_d[1][h1]) +
                             (ctl.red_d[2][h1] + ctl.red_d[3][h1]);
            float ds0 = 0.0f, dr0 = 0.0f, ds1 = 0.0f, dr1 = 0.0f;
            if (w0) head_metrics(nc0, pn0, D0, ds0, dr0);
            if (w1) head_metrics(nc1, pn1, D1, ds1, dr1);
            float ds = fmaxf(ds0, ds1), dr = fmaxf(dr0, dr1);
            ds = fmaxf(ds, __shfl_xor_sync(0xffffffffu, ds, 1));
            dr = fmaxf(dr, __shfl_xor_sync(0xffffffffu, dr, 1));
            ds = fmaxf(ds, __shfl_xor_sync(0xffffffffu, ds, 2));
            dr = fmaxf(dr, __shfl_xor_sync(0xffffffffu, dr, 2));
            streak = (ds < prm.tau && dr < prm.phi) ? streak + 1 : 0;
            stop = streak >= prm.patience;
        }
        if (stop) break;
#pragma unroll
        for (int i = 0; i < 2; i++) {
            px[i][0] = cur[i][0] * rn0;
            px[i][2] = cur[i][2] * rn0;
            px[i][1] = cur[i][1] * rn1;
            px[i][3] = cur[i][3] * rn1;
        }
        pn0 = nc0;
        pn1 = nc1;
        // every read of stage st is behind the barriers above: refill it with the block
        // kArtStages - 1 after the next (the last block in the ring decides whether there is one)
        const int last = blk[(st + kArtStages - 1) % kArtStages];
        blk[st] = last >= 0 ? advance() : -1;
        if (blk[st] >= 0 && issue(blk[st], st)) inflight |= 1u << st;
        st = st + 1 == kArtStages ? 0 : st + 1;
    }
    // copies still in flight into this CTA's shared memory are waited for (bounded) before it
    // exits: the ring's blocks after a stop or a timed-out wait
    for (int k = 0; k < kArtStages; k++)
        if ((inflight >> k) & 1u) wait_stage(k);
    // out = o / l: this thread's channels 32mt + 16i + {g, g+8} of heads h0, h1
    const float i0 = L0 > 0.0f ? 1.0f / L0 : 0.0f, i1 = L1 > 0.0f ? 1.0f / L1 : 0.0f;
    float *ob = a.out + ((size_t)b * a.Hq + h * G) * kD;
#pragma unroll
    for (int i = 0; i < 2; i++) {
        const int ch = 32 * warp + 16 * i + g;
        if (w0) {
            ob[h0 * kD + ch] = R.o[i][0] * i0;
            ob[h0 * kD + ch + 8] = R.o[i][2] * i0;
        }
        if (w1) {
            ob[h1 * kD + ch] = R.o[i][1] * i1;
            ob[h1 * kD + ch + 8] = R.o[i][3] * i1;
        }
    }
    if (prm.used && t == 0) prm.used[u] = used;
}

}  // namespace

cudaError_t launch_art(const DecodeArgs &a, float tau, float phi, int patience, int32_t *used,
                       cudaStream_t stream) {
    static int smem_set[kMaxDevicesTracked];
    const cudaError_t ea = raise_smem_limit(art_kernel, kArtSmem, smem_set);
    if (ea != cudaSuccess) return ea;
    ArtParams prm;
    memset(&prm, 0, sizeof prm);
    prm.a = a;
    prm.tau = tau;
    prm.phi = phi;
    prm.patience = patience;
    prm.used = used;
    if (!make_tile_map(&prm.tm_v, const_cast<__nv_bfloat16 *>(a.v),
                       (uint64_t)a.P * a.Hkv * kPage))
        return cudaErrorInvalidValue;
    art_kernel<<<a.B * a.Hkv, kArtThreads, kArtSmem, stream>>>(prm);
    return cudaGetLastError();
}

}  // namespace ffd
