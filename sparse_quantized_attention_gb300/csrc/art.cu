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
// regime the page reports its gains in (large batches): one CTA of 128 threads walks one
// (sequence, KV head) unit. Per block, warp mt computes the exact scores (thumbnail + residual, on
// the tensor cores) of rows 16mt .. 16mt+15 for every head, thread t owns the online-softmax
// probabilities of head t % 8 on rows t/8 + 16j, and thread t accumulates output channel t of
// every head over the block's V rows. A block's three records (thumbnail 3 KB, residual 8.5 KB,
// V 16 KB) are brought into shared memory by bulk copies, double-buffered: the next block's copies
// are in flight while the current block is processed. 1 - cos is formed as |P/|P| - Q/|Q||^2 / 2,
// which keeps its precision when the two directions are close.
#include "common.cuh"
#include "ptx.cuh"
#include "scan.cuh"

namespace ffd {

namespace {

constexpr float kLog2eArt = 1.4426950408889634f;
constexpr int kArtThreads = 128;

// One block's records in shared memory (each part 128-byte aligned).
struct alignas(128) ArtStage {
    uint8_t thumb[kThumbRec];
    uint8_t resid[kResidRec];
    __nv_bfloat16 v[kPage * kD];
};
constexpr uint32_t kArtStageTx = kThumbRec + kResidRec + kPage * kD * 2;
static_assert(kThumbRec % 128 == 0 && (kThumbRec + kResidRec) % 128 == 0, "stage alignment");
constexpr size_t kArtSmem = 2 * sizeof(ArtStage);

// Sums of eight per-thread values over the 32 lanes of a warp, transposed: on return lane L holds
// the sum for value L / 4 (each value reaches four lanes). Nine shuffles instead of forty.
__device__ __forceinline__ float warp_sum8_t(const float (&v)[kMaxG], int lane) {
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float w[4], x[2];
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const float send = b4 ? v[k] : v[k + 4];
        const float keep = b4 ? v[k + 4] : v[k];
        w[k] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int k = 0; k < 2; k++) {
        const float send = b3 ? w[k] : w[k + 2];
        const float keep = b3 ? w[k + 2] : w[k];
        x[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    const float send = b2 ? x[0] : x[1];
    float y = (b2 ? x[1] : x[0]) + __shfl_xor_sync(0xffffffffu, send, 4);
    y += __shfl_xor_sync(0xffffffffu, y, 1);
    y += __shfl_xor_sync(0xffffffffu, y, 2);
    return y;
}

// CTA sums of eight per-thread values; red is a [4 warps][kMaxG] buffer of its own. On return
// every thread holds all eight sums.
__device__ __forceinline__ void cta_sum8(float (&v)[kMaxG], float (*red)[kMaxG]) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float y = warp_sum8_t(v, lane);
    if ((lane & 3) == 0) red[warp][lane >> 2] = y;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kMaxG; i++) v[i] = (red[0][i] + red[1][i]) + (red[2][i] + red[3][i]);
}

__global__ void __launch_bounds__(kArtThreads) art_kernel(DecodeArgs a, float tau, float phi,
                                                          int patience, int32_t *used_out) {
    __shared__ __align__(16) float sp[kPage][kMaxG];  // the block's scores, then its probabilities
    __shared__ float red_m[4][kMaxG], red_l[4][kMaxG], red_n[4][kMaxG], red_d[4][kMaxG];
    __shared__ int s_list[kArtThreads];  // kept blocks of the current chunk, most recent first
    __shared__ int s_wc[4];
    __shared__ __align__(8) uint64_t full[2];
    extern __shared__ __align__(128) uint8_t art_dyn[];
    ArtStage *stage = reinterpret_cast<ArtStage *>(art_dyn);
    const int u = blockIdx.x;
    const int b = u / a.Hkv, h = u - b * a.Hkv;
    const int G = a.G;
    const int n = checked_seq_len(a, b);
    const int nb = (n + kPage - 1) / kPage;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int g = lane >> 2, tig = lane & 3;
    const int r0 = 16 * warp + g, r1 = r0 + 8;
    const int hp = t & 7, rp = t >> 3;  // probability phase: head hp, rows rp + 16 j
    ThumbOps Q;
    ResidOps QR;
    load_thumb_ops(a, b, h, lane, Q);
    load_resid_ops(a, b, h, lane, QR);
    const int32_t *bt = a.block_table + (size_t)b * a.max_blocks;
    const uint8_t *keep = a.keep_in ? a.keep_in + (size_t)u * a.max_blocks : nullptr;
    if (t == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        fence_barrier_init();
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
            mbar_arrive_expect_tx(&full[st], kArtStageTx);
            tma_load_1d(stage[st].thumb, a.thumb + tile * kThumbRec, kThumbRec, &full[st]);
            tma_load_1d(stage[st].resid, a.resid + tile * kResidRec, kResidRec, &full[st]);
            tma_load_1d(stage[st].v, a.v + tile * kPage * kD, kPage * kD * 2, &full[st]);
        }
        return true;
    };
    // Bounded wait for stage st's copies; the result is block-uniform.
    uint32_t phases = 0u;  // bit st: parity of stage st's next completion
    auto wait_stage = [&](int st) -> bool {
        const uint64_t t0 = globaltimer_ns();
        bool ok = true;
        while (!mbar_try_wait(&full[st], (phases >> st) & 1u)) {
            if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
                ok = false;
                break;
            }
        }
        phases ^= 1u << st;
        ok = __syncthreads_and(ok) != 0;
        if (!ok && t == 0) raise_error(a.err, FFD_ERRBIT_TIMEOUT);
        return ok;
    };

    float m[kMaxG], l[kMaxG], o[kMaxG], prev[kMaxG], pn[kMaxG], rpn[kMaxG];
#pragma unroll
    for (int i = 0; i < kMaxG; i++) {
        m[i] = -INFINITY;
        l[i] = 0.0f;
        o[i] = 0.0f;
        prev[i] = 0.0f;
        pn[i] = 0.0f;   // squared norm of the previous probe
        rpn[i] = 0.0f;  // 1 / its norm
    }
    int used = 0, streak = 0;
    int hi = nb - 1;       // top block of the next chunk of the kept-block list
    int pos = 0, cnt = 0;  // read position and length of the current chunk
    // The next block of the traversal after block 0: the kept blocks from the most recent down,
    // listed 128 candidates at a time (block-uniform; the barriers are reached by every thread).
    auto advance = [&]() -> int {
        while (pos == cnt && hi >= 1) {
            const int idx = hi - t;
            const bool k = idx >= 1 && (keep == nullptr || keep[idx] != 0);
            const unsigned bal = __ballot_sync(0xffffffffu, k);
            __syncthreads();  // earlier reads of s_list / s_wc are done
            if (lane == 0) s_wc[warp] = __popc(bal);
            __syncthreads();
            int off = 0;
            for (int w = 0; w < warp; w++) off += s_wc[w];
            if (k) s_list[off + __popc(bal & ((1u << lane) - 1u))] = idx;
            cnt = (s_wc[0] + s_wc[1]) + (s_wc[2] + s_wc[3]);
            pos = 0;
            hi -= kArtThreads;
            __syncthreads();
        }
        return pos < cnt ? s_list[pos++] : -1;
    };
    int c = nb > 0 ? 0 : -1;  // block 0 first
    int st = 0;
    bool have = c >= 0 && issue(c, 0);
    int cn = c >= 0 ? advance() : -1;
    bool have_n = cn >= 0 && issue(cn, 1);
    while (c >= 0) {
        const bool bad = !have;
        if (have && !wait_stage(st)) break;  // timed out: the error word says so
        const ArtStage &sg = stage[st];
        // scores of the block's rows for every head (-inf for rows past n and heads past G)
        float4 e = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        if (!bad) e = exact_tile(sg.thumb, sg.resid, r0, r1, tig, Q, QR, a.sm_scale);
        const int rows = n - c * kPage < kPage ? n - c * kPage : kPage;
        const bool v0 = r0 < rows, v1 = r1 < rows;
        const int h0 = 2 * tig, h1 = h0 + 1;
        sp[r0][h0] = v0 && h0 < G ? e.x : -INFINITY;
        sp[r0][h1] = v0 && h1 < G ? e.y : -INFINITY;
        sp[r1][h0] = v1 && h0 < G ? e.z : -INFINITY;
        sp[r1][h1] = v1 && h1 < G ? e.w : -INFINITY;
        __syncthreads();
        // block maxima per head: thread t covers head hp on rows rp + 16 j
        float s4[4];
        float bm = -INFINITY;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            s4[j] = sp[rp + 16 * j][hp];
            bm = fmaxf(bm, s4[j]);
        }
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
        if (lane < 8) red_m[warp][lane] = bm;
        __syncthreads();
        float alpha[kMaxG], mine = -INFINITY;
#pragma unroll
        for (int i = 0; i < kMaxG; i++) {
            const float mn = fmaxf(fmaxf(m[i], fmaxf(red_m[0][i], red_m[1][i])),
                                   fmaxf(red_m[2][i], red_m[3][i]));
            alpha[i] = m[i] == -INFINITY ? 0.0f : exp2f((m[i] - mn) * kLog2eArt);
            m[i] = mn;
            if (i == hp) mine = mn;
        }
        // probabilities and their sums per head
        float ps[kMaxG];
#pragma unroll
        for (int i = 0; i < kMaxG; i++) ps[i] = 0.0f;
        float mysum = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const float p = s4[j] == -INFINITY ? 0.0f : exp2f((s4[j] - mine) * kLog2eArt);
            sp[rp + 16 * j][hp] = p;
            mysum += p;
        }
#pragma unroll
        for (int i = 0; i < kMaxG; i++) ps[i] = i == hp ? mysum : 0.0f;
        // lanes L and L ^ 8, L ^ 16, L ^ 24 share a head: the transposed sum collects them too
        cta_sum8(ps, red_l);  // its barrier also orders the probability stores before PV
        // output channel t of every head: o = alpha o + sum_r p[r] V[r][t]
        float acc[kMaxG];
#pragma unroll
        for (int i = 0; i < kMaxG; i++) acc[i] = 0.0f;
        if (!bad) {
            const __nv_bfloat16 *vt = sg.v + t;
#pragma unroll 4
            for (int r = 0; r < rows; r++) {
                const float vv = __bfloat162float(vt[(size_t)r * kD]);
                const float4 p0 = *reinterpret_cast<const float4 *>(&sp[r][0]);
                const float4 p1 = *reinterpret_cast<const float4 *>(&sp[r][4]);
                acc[0] = fmaf(p0.x, vv, acc[0]);
                acc[1] = fmaf(p0.y, vv, acc[1]);
                acc[2] = fmaf(p0.z, vv, acc[2]);
                acc[3] = fmaf(p0.w, vv, acc[3]);
                acc[4] = fmaf(p1.x, vv, acc[4]);
                acc[5] = fmaf(p1.y, vv, acc[5]);
                acc[6] = fmaf(p1.z, vv, acc[6]);
                acc[7] = fmaf(p1.w, vv, acc[7]);
            }
        }
        float cur[kMaxG], nn[kMaxG];
#pragma unroll
        for (int i = 0; i < kMaxG; i++) {
            o[i] = fmaf(alpha[i], o[i], acc[i]);
            l[i] = fmaf(alpha[i], l[i], ps[i]);
            cur[i] = l[i] > 0.0f ? o[i] * __frcp_rn(l[i]) : 0.0f;
            nn[i] = cur[i] * cur[i];
        }
        used++;
        // the probe and the stability criterion (every thread takes the same decision)
        cta_sum8(nn, red_n);
        float rn[kMaxG];  // 1 / |P_i(t)|
#pragma unroll
        for (int i = 0; i < kMaxG; i++) rn[i] = nn[i] > 0.0f ? rsqrtf(nn[i]) : 0.0f;
        bool stop = false;
        if (used >= 2) {
            float dd[kMaxG];
#pragma unroll
            for (int i = 0; i < kMaxG; i++) {
                const float x = cur[i] * rn[i] - prev[i] * rpn[i];
                dd[i] = x * x;
            }
            cta_sum8(dd, red_d);
            // head lane & 7 on every lane (the same values in every warp), then the maxima
            const int i = lane & 7;
            float nni = 0.0f, pni = 0.0f, ddi = 0.0f;
#pragma unroll
            for (int k = 0; k < kMaxG; k++)
                if (k == i) nni = nn[k], pni = pn[k], ddi = dd[k];
            float ds = 0.0f, dr = 0.0f;
            if (i < G) {
                const float nc = sqrtf(nni), np = sqrtf(pni);
                ds = np > 0.0f ? fabsf(nc - np) / np : nc;
                // 1 - cos; a zero probe on one side only counts as orthogonal
                dr = (nc > 0.0f && np > 0.0f) ? 0.5f * ddi
                                              : ((nc == 0.0f && np == 0.0f) ? 0.0f : 1.0f);
            }
#pragma unroll
            for (int off = 1; off < 8; off <<= 1) {
                ds = fmaxf(ds, __shfl_xor_sync(0xffffffffu, ds, off));
                dr = fmaxf(dr, __shfl_xor_sync(0xffffffffu, dr, off));
            }
            streak = (ds < tau && dr < phi) ? streak + 1 : 0;
            stop = streak >= patience;
        }
        if (stop) break;
#pragma unroll
        for (int i = 0; i < kMaxG; i++) {
            prev[i] = cur[i];
            pn[i] = nn[i];
            rpn[i] = rn[i];
        }
        // every read of stage st is behind the barriers above: refill it with the block after cn
        const int cn2 = cn >= 0 ? advance() : -1;
        const bool have_n2 = cn2 >= 0 && issue(cn2, st);
        c = cn;
        have = have_n;
        cn = cn2;
        have_n = have_n2;
        st ^= 1;
    }
    // copies still in flight into this CTA's shared memory are waited for (bounded) before it
    // exits: the next block's, after a stop or a timed-out wait
    if (c >= 0 && cn >= 0 && have_n) wait_stage(st ^ 1);
#pragma unroll
    for (int i = 0; i < kMaxG; i++)
        if (i < G)
            a.out[((size_t)b * a.Hq + h * G + i) * kD + t] = l[i] > 0.0f ? o[i] / l[i] : 0.0f;
    if (used_out && t == 0) used_out[u] = used;
}

}  // namespace

cudaError_t launch_art(const DecodeArgs &a, float tau, float phi, int patience, int32_t *used,
                       cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(art_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kArtSmem);
    if (e != cudaSuccess) return e;
    art_kernel<<<a.B * a.Hkv, kArtThreads, kArtSmem, stream>>>(a, tau, phi, patience, used);
    return cudaGetLastError();
}

}  // namespace ffd
