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
// The criterion makes one unit's traversal sequential, but only through the probe: a block's own
// softmax state (its maximum m, its sum l and its numerator o per head) does not depend on the
// others, and the state after t blocks is the log-sum-exp merge of the per-block states. So one CTA
// per (sequence, KV head) unit runs kArtGroups refine groups of four warps, group g scoring
// traversal positions g, g + kArtGroups, ...: each block's thumbnail, residual and V records land
// in the group's two stages by bulk and tensor copies, its exact scores come from the thumbnail +
// residual tensor-core tile (`exact_tile`, scan.cuh) and `softmax_pv` (splitkv.cuh) forms the
// block's state from a fresh reference, which the group writes to one of its two state slots.
// One more warp, the sequencer, merges the states in traversal order into the running state it
// holds in registers (four lanes per head, 32 channels each), takes the probe and its two metrics
// with warp shuffles alone, and stops the walk. The sequential path per block is a merge
// and a few warp reductions; the scoring, softmax and P.V of the next blocks run beside it. The
// direction change is formed as |P/|P| - P'/|P'||^2 = 2 (1 - cos), which keeps its precision when
// the two directions are close. The traversal list is built once at the start, in the workspace.
#include "common.cuh"
#include "ptx.cuh"
#include "scan.cuh"
#include "splitkv.cuh"

namespace ffd {

namespace {

constexpr int kArtGroups = 3;                        // refine groups (4 warps each)
constexpr int kArtSeqWarp = 4 * kArtGroups;          // the sequencer warp
constexpr int kArtThreads = 32 * (kArtSeqWarp + 1);
// One block's records in shared memory: the V tile first (1 KB aligned for the 128-byte swizzle).
constexpr int kArtV = 0;
constexpr int kArtThumb = kPage * kD * 2;
constexpr int kArtResid = kArtThumb + kThumbRec;
constexpr int kArtStage = 28672;  // 28 KB: a multiple of 1 KB
static_assert(kArtResid + kResidRec <= kArtStage && kArtStage % 1024 == 0, "stage layout");
constexpr uint32_t kArtStageTx = kThumbRec + kResidRec + kPage * kD * 2;
constexpr int kArtStages = 2 * kArtGroups;                      // two per group
constexpr int kArtPx = kArtStages * kArtStage;                  // [group][2] P^T fragments
constexpr int kArtState = kArtPx + kArtGroups * 2 * kPxBuf;     // [slot][kMaxG][kPartStride]
constexpr int kArtSlots = 2 * kArtGroups;                       // two per group
constexpr int kArtSmem = kArtState + kArtSlots * kMaxG * kPartStride * 4 + 1024;  // + align slack
static_assert(kArtSmem <= 232448, "shared memory per CTA");

// The shared control block softmax_pv and write_record expect (one entry per refine group).
struct ArtCtl {
    uint32_t over[kArtGroups][2][4];
    float wmax[kArtGroups][2][4][kMaxG];
    float lsum[kArtGroups][4][kMaxG];
    uint32_t aborted;
    int32_t stop_at;  // traversal positions >= stop_at are not needed (the sequencer stopped)
    int32_t wc[kArtSeqWarp + 1];
    uint64_t full[kArtStages];
    uint64_t state_full[kArtSlots], state_empty[kArtSlots];
};

struct ArtParams {
    CUtensorMap tm_v;
    DecodeArgs a;
    float tau, phi;
    int patience;
    int32_t *used;
    int32_t *list;  // [B * Hkv][max_blocks] traversal lists
};

// d_scale and 1 - cos of one head (a zero probe on one side only counts as orthogonal).
__device__ __forceinline__ void head_metrics(float nc, float np, float dd, float &ds, float &dr) {
    ds = np > 0.0f ? fabsf(nc - np) / np : nc;
    dr = (nc > 0.0f && np > 0.0f) ? 0.5f * dd : ((nc == 0.0f && np == 0.0f) ? 0.0f : 1.0f);
}

__device__ __forceinline__ bool stopped_before(const ArtCtl &c, int p) {
    return *reinterpret_cast<const volatile int32_t *>(&c.stop_at) <= p;
}

// Bounded wait on an mbarrier phase. False after the wait ran out (the error bit and the abort
// flag are then set), after an abort, or, for p >= 0, as soon as traversal position p is no longer
// needed.
__device__ __forceinline__ bool art_wait(const DecodeArgs &a, ArtCtl &c, uint64_t *bar,
                                         uint32_t parity, int p) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (p >= 0 && stopped_before(c, p)) return false;
        if (*reinterpret_cast<volatile uint32_t *>(&c.aborted)) return false;
        if (globaltimer_ns() - t0 > a.wait_ns) {
            raise_error(a.err, FFD_ERRBIT_TIMEOUT);
            *reinterpret_cast<volatile uint32_t *>(&c.aborted) = 1;
            return false;
        }
    }
    return true;
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
    const int32_t *bt = a.block_table + (size_t)b * a.max_blocks;
    const uint8_t *keep = a.keep_in ? a.keep_in + (size_t)u * a.max_blocks : nullptr;
    int32_t *list = prm.list + (size_t)u * a.max_blocks;
    if (t == 0) {
        for (int i = 0; i < kArtStages; i++) mbar_init(&ctl.full[i], 1);
        for (int i = 0; i < kArtSlots; i++) {
            mbar_init(&ctl.state_full[i], 1);
            mbar_init(&ctl.state_empty[i], 1);
        }
        ctl.aborted = 0;
        ctl.stop_at = 0x7fffffff;
        fence_barrier_init();
        prefetch_tensormap(&prm.tm_v);
    }
    // The traversal list: block 0, then the kept blocks from the most recent down, kArtThreads
    // candidates at a time (ballot and a prefix over the warps' counts).
    int nl = 0;
    if (nb > 0) {
        if (t == 0) list[0] = 0;
        nl = 1;
        for (int hi = nb - 1; hi >= 1; hi -= kArtThreads) {
            const int idx = hi - t;
            const bool k = idx >= 1 && (keep == nullptr || keep[idx] != 0);
            const unsigned bal = __ballot_sync(0xffffffffu, k);
            if (lane == 0) ctl.wc[warp] = __popc(bal);
            __syncthreads();
            int off = nl;
            for (int w = 0; w < warp; w++) off += ctl.wc[w];
            if (k) list[off + __popc(bal & ((1u << lane) - 1u))] = idx;
            for (int w = 0; w <= kArtSeqWarp; w++) nl += ctl.wc[w];
            __syncthreads();  // wc is rewritten by the next chunk
        }
    }
    __syncthreads();  // the list (this CTA's own global writes) and the barriers are ready

    if (warp < kArtSeqWarp) {
        // ---- refine group g: traversal positions g, g + kArtGroups, ..., each into a state slot
        const int g = warp >> 2, mt = warp & 3;
        const int qg = lane >> 2, tig = lane & 3;
        const int r0 = 16 * mt + qg, r1 = r0 + 8;
        const bool w0 = 2 * tig < G, w1 = 2 * tig + 1 < G;
        const uint32_t bar_id = 2 + g;
        ThumbOps Q;
        ResidOps QR;
        load_thumb_ops(a, b, h, lane, Q);
        load_resid_ops(a, b, h, lane, QR);
        // Copies of traversal position p into the group's stage s; false (nothing issued) for a
        // page outside [0, P). Group-uniform; one thread of the group issues.
        int issued = 0;  // bit s: a copy into the group's stage s is in flight
        auto issue = [&](int p, int s) -> bool {
            const int page = bt[list[p]];
            if (page < 0 || page >= a.P) {
                if (mt == 0 && lane == 0) raise_error(a.err, FFD_ERRBIT_BOUNDS);
                return false;
            }
            if (mt == 0 && lane == 0) {
                const size_t tile = (size_t)page * a.Hkv + h;
                uint8_t *d = base + (g * 2 + s) * kArtStage;
                uint64_t *fb = &ctl.full[g * 2 + s];
                mbar_arrive_expect_tx(fb, kArtStageTx);
                tma_load_3d(d + kArtV, &prm.tm_v, 0, (int)(tile * kPage), 0, fb);
                tma_load_1d(d + kArtThumb, a.thumb + tile * kThumbRec, kThumbRec, fb);
                tma_load_1d(d + kArtResid, a.resid + tile * kResidRec, kResidRec, fb);
            }
            issued |= 1 << s;
            return true;
        };
        uint32_t have = 0u;  // bit s: stage s holds (or will hold) a loaded block
        if (g < nl && issue(g, 0)) have |= 1u;
        if (g + kArtGroups < nl && issue(g + kArtGroups, 1)) have |= 2u;
        int pb = 0;
        uint32_t fph = 0u;  // bit s: parity of the group's stage s's next completion
        for (int p = g, j = 0; p < nl; p += kArtGroups, j++) {
            const int s = j & 1;
            const bool good = (have >> s) & 1u;
            // the block's copies, unless the sequencer has stopped before it (the flag is only
            // ever lowered; a group that sees it late computes one block more, harmlessly); one
            // decision for the group
            bool go = !stopped_before(ctl, p);
            if (good && go) {
                go = art_wait(a, ctl, &ctl.full[g * 2 + s], (fph >> s) & 1u, p);
                if (go) {
                    fph ^= 1u << s;
                    issued &= ~(1 << s);
                }
            }
            if (named_barrier_or(bar_id, 128, !go)) break;
            RefineState R;
            R.m0 = R.m1 = kNoReference;  // the block's own maximum comes through the rescale path
            R.nl0 = R.nl1 = -kNoReference * kLog2e;
            R.l0 = R.l1 = 0.0f;
#pragma unroll
            for (int i = 0; i < 2; i++) R.o[i][0] = R.o[i][1] = R.o[i][2] = R.o[i][3] = 0.0f;
            if (good) {
                uint8_t *sg = base + (g * 2 + s) * kArtStage;
                const int c = list[p];
                const int rows = n - c * kPage < kPage ? n - c * kPage : kPage;
                const float4 e = exact_tile(sg + kArtThumb, sg + kArtResid, r0, r1, tig, Q, QR,
                                            a.sm_scale);
                const bool v0 = r0 < rows, v1 = r1 < rows;
                if (rows < kPage) {  // the sequence's partial last block: V rows past it read 0
                    for (int k = 32 * mt + lane; k < (kPage - rows) * 16; k += 128) {
                        const int r = rows + (k >> 4), half = (k >> 3) & 1;
                        *reinterpret_cast<uint4 *>(sg + kArtV + half * 8192 + r * 128 +
                                                   (k & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async();  // before the stage's next bulk copy
                    named_barrier_sync(bar_id, 128);
                }
                softmax_pv(&ctl, base + kArtPx + (g * 2 + pb) * kPxBuf, sg + kArtV,
                           v0 && w0 ? e.x : -INFINITY, v0 && w1 ? e.y : -INFINITY,
                           v1 && w0 ? e.z : -INFINITY, v1 && w1 ? e.w : -INFINITY, R, g, mt, pb,
                           lane);
                pb ^= 1;
            } else {
                R.m0 = R.m1 = -INFINITY;  // a block not loaded adds nothing
            }
            // the block's state goes to slot g * 2 + s once the sequencer has taken its previous one;
            // the same barrier tells that every read of the stage is done, so it is refilled
            const int slot = g * 2 + s;
            const bool ok =
                j < 2 || art_wait(a, ctl, &ctl.state_empty[slot], ((j >> 1) - 1) & 1, p);
            if (named_barrier_or(bar_id, 128, !ok)) break;
            have &= ~(1u << s);
            const int pn = p + 2 * kArtGroups;
            if (pn < nl && issue(pn, s)) have |= 1u << s;  // unneeded after a stop: drained
            write_record(a, &ctl, R, reinterpret_cast<float *>(base + kArtState) +
                                         slot * kMaxG * kPartStride,
                         g, mt, lane);
            named_barrier_sync(bar_id, 128);
            if (mt == 0 && lane == 0) mbar_arrive(&ctl.state_full[slot]);
        }
        // leave no copy in flight: the group's stages still being filled
        for (int s = 0; s < 2; s++) {
            if (!((issued >> s) & 1)) continue;
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(&ctl.full[g * 2 + s], (fph >> s) & 1u)) {
                if (globaltimer_ns() - t0 > a.wait_ns) {
                    if (mt == 0 && lane == 0) raise_error(a.err, FFD_ERRBIT_TIMEOUT);
                    break;
                }
            }
        }
        return;
    }

    // ---- the sequencer: the running state, lane L holding head L / 4, channels 32 (L % 4) .. +31
    const int hh = lane >> 2, cq = 32 * (lane & 3);
    const bool hv = hh < G;
    float o[32], px[32];
    float M = -INFINITY, Ls = 0.0f, pn = 0.0f;
#pragma unroll
    for (int k = 0; k < 32; k++) o[k] = px[k] = 0.0f;
    int used = 0, streak = 0;
    for (int p = 0; p < nl; p++) {
        const int g = p % kArtGroups, j = p / kArtGroups, slot = g * 2 + (j & 1);
        if (!__all_sync(0xffffffffu, art_wait(a, ctl, &ctl.state_full[slot], (j >> 1) & 1, -1)))
            break;  // warp-uniform
        const float *rec = reinterpret_cast<const float *>(base + kArtState) +
                           (slot * kMaxG + (hv ? hh : 0)) * kPartStride;
        // merge the block's state: M' = max(M, m), o = e^(M - M') o + e^(m - M') o_b, same for l
        const float mb = rec[kD];
        if (hv && mb != -INFINITY) {  // a block not loaded adds nothing
            const float lb = rec[kD + 1];
            const float Mn = fmaxf(M, mb);
            const float fa = M == -INFINITY ? 0.0f : exp2f((M - Mn) * kLog2e);
            const float fb = exp2f((mb - Mn) * kLog2e);
#pragma unroll
            for (int k = 0; k < 32; k += 4) {
                const float4 v = *reinterpret_cast<const float4 *>(rec + cq + k);
                o[k] = fmaf(fb, v.x, fa * o[k]);
                o[k + 1] = fmaf(fb, v.y, fa * o[k + 1]);
                o[k + 2] = fmaf(fb, v.z, fa * o[k + 2]);
                o[k + 3] = fmaf(fb, v.w, fa * o[k + 3]);
            }
            Ls = fmaf(fb, lb, fa * Ls);
            M = Mn;
        }
        __syncwarp();  // every lane has read the slot
        if (lane == 0) mbar_arrive(&ctl.state_empty[slot]);
        used++;
        // the probe P = o / l of this lane's head: |P| over the head's four lanes, then the
        // direction change against the last probe
        const float il = Ls > 0.0f ? __frcp_rn(Ls) : 0.0f;
        float q = 0.0f;
#pragma unroll
        for (int k = 0; k < 32; k++) {
            const float c = o[k] * il;
            q = fmaf(c, c, q);
        }
        q += __shfl_xor_sync(0xffffffffu, q, 1);
        q += __shfl_xor_sync(0xffffffffu, q, 2);
        const float nc = sqrtf(q);
        const float rn = q > 0.0f ? rsqrtf(q) : 0.0f;
        if (used >= 2) {
            float d = 0.0f;
#pragma unroll
            for (int k = 0; k < 32; k++) {
                const float e = o[k] * il * rn - px[k];
                d = fmaf(e, e, d);
            }
            d += __shfl_xor_sync(0xffffffffu, d, 1);
            d += __shfl_xor_sync(0xffffffffu, d, 2);
            float ds = 0.0f, dr = 0.0f;
            if (hv) head_metrics(nc, pn, d, ds, dr);
#pragma unroll
            for (int o2 = 4; o2 < 32; o2 <<= 1) {
                ds = fmaxf(ds, __shfl_xor_sync(0xffffffffu, ds, o2));
                dr = fmaxf(dr, __shfl_xor_sync(0xffffffffu, dr, o2));
            }
            streak = (ds < prm.tau && dr < prm.phi) ? streak + 1 : 0;
        }
        pn = nc;
#pragma unroll
        for (int k = 0; k < 32; k++) px[k] = o[k] * il * rn;
        if (used >= 2 && streak >= prm.patience) break;
    }
    // the groups stop fetching and scoring past the stop (also after an abort)
    if (lane == 0) *reinterpret_cast<volatile int32_t *>(&ctl.stop_at) = used;
    // out = o / l: this lane's 32 channels of its head
    if (hv) {
        float *ob = a.out + ((size_t)b * a.Hq + h * G + hh) * kD + cq;
        const float iv = Ls > 0.0f ? 1.0f / Ls : 0.0f;
#pragma unroll
        for (int k = 0; k < 32; k += 4)
            *reinterpret_cast<float4 *>(ob + k) =
                make_float4(o[k] * iv, o[k + 1] * iv, o[k + 2] * iv, o[k + 3] * iv);
    }
    if (prm.used && lane == 0) prm.used[u] = used;
}

}  // namespace

size_t art_list_bytes(int units, int max_blocks) {
    return (size_t)units * max_blocks * sizeof(int32_t);
}

cudaError_t launch_art(const DecodeArgs &a, float tau, float phi, int patience, int32_t *used,
                       int32_t *list, cudaStream_t stream) {
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
    prm.list = list;
    if (!make_tile_map(&prm.tm_v, const_cast<__nv_bfloat16 *>(a.v),
                       (uint64_t)a.P * a.Hkv * kPage))
        return cudaErrorInvalidValue;
    art_kernel<<<a.B * a.Hkv, kArtThreads, kArtSmem, stream>>>(prm);
    return cudaGetLastError();
}

}  // namespace ffd
