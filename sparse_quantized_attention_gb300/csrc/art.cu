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
// Four more warps, the sequencer, merge the states in traversal order into the running state
// they hold in registers (two heads a warp, sixteen lanes a head, eight channels a lane), take
// the probe and its two metrics, and stop the walk. They take the blocks two at a time: the
// states after the first and after the second block are merged in order and the two probes are
// formed side by side, so the sequential path is one merge pair, a few warp reductions and one
// named barrier per two blocks; the scoring, softmax and P.V of the next blocks run beside it.
// The direction change is formed as |P/|P| - P'/|P'||^2 = 2 (1 - cos), which keeps its precision
// when the two directions are close; |P| = |o| / l and P/|P| = o / |o|, so l enters the scale
// change only. The traversal list is built once at the start, in the workspace; each group reads
// its list entries and block-table pages an iteration ahead of their use.
#include "common.cuh"
#include "ptx.cuh"
#include "scan.cuh"
#include "splitkv.cuh"

namespace ffd {

namespace {

constexpr int kArtGroups = 3;                        // refine groups (4 warps each)
constexpr int kArtSeqWarp = 4 * kArtGroups;          // the first sequencer warp
constexpr int kArtSeqWarps = 4;                      // sequencer warps: two heads each
constexpr int kArtWarps = kArtSeqWarp + kArtSeqWarps;
constexpr int kArtThreads = 32 * kArtWarps;
constexpr int kArtSeqBar = 1;                        // named barrier of the sequencer warps
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
    int32_t wc[kArtWarps];
    float seq_met[2][kArtSeqWarps][4];  // the sequencer warps' metrics of a pair of blocks
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
            for (int w = 0; w < kArtWarps; w++) nl += ctl.wc[w];
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
        // Copies of a traversal position's block, on `page`, into the group's stage s; false
        // (nothing issued) for a page outside [0, P). Group-uniform; one thread of the group
        // issues.
        int issued = 0;  // bit s: a copy into the group's stage s is in flight
        auto issue = [&](int page, int s) -> bool {
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
        // The list and block-table reads run ahead of their use, so that neither waits in the
        // loop: cs0 / cs1 is the block in stage 0 / 1, nx_c the block of the next position to
        // copy.
        int cs0 = g < nl ? list[g] : 0, cs1 = g + kArtGroups < nl ? list[g + kArtGroups] : 0;
        int nx_c = g + 2 * kArtGroups < nl ? list[g + 2 * kArtGroups] : 0;
        uint32_t have = 0u;  // bit s: stage s holds (or will hold) a loaded block
        if (g < nl && issue(bt[cs0], 0)) have |= 1u;
        if (g + kArtGroups < nl && issue(bt[cs1], 1)) have |= 2u;
        int pb = 0;
        uint32_t fph = 0u;  // bit s: parity of the group's stage s's next completion
        for (int p = g, j = 0; p < nl; p += kArtGroups, j++) {
            const int s = j & 1;
            const int pn = p + 2 * kArtGroups;  // the position this iteration copies into stage s
            const int pn_page = pn < nl ? bt[nx_c] : -1;
            const int nn_c = pn + kArtGroups < nl ? list[pn + kArtGroups] : 0;
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
                const int c = s ? cs1 : cs0;
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
            if (pn < nl && issue(pn_page, s)) have |= 1u << s;  // unneeded after a stop: drained
            if (s) cs1 = nx_c;
            else cs0 = nx_c;
            nx_c = nn_c;
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

    // ---- the sequencer: warp sw holds the running state of heads 2 sw and 2 sw + 1, lane L head
    // 2 sw + L / 16 and channels 8 (L % 16) .. +7. The warps take the blocks two at a time: the
    // state after the first (a) and after the second (b) are merged in order, as one block at a
    // time would, and the two probes' metrics are formed side by side; the four warps exchange
    // their heads' maxima through shared memory at one named barrier (which also tells that every
    // warp has read the slots), and the stop decisions, at a and then at b, are the same in all.
    const int sw = warp - kArtSeqWarp;
    const int hh = 2 * sw + (lane >> 4), cq = 8 * (lane & 15);
    const bool hv = hh < G;
    float o[8], px[8];
    float M = -INFINITY, Ls = 0.0f, pn = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; k++) o[k] = px[k] = 0.0f;
    int used = 0, streak = 0;
    // merge one block's state (rec) into (Mx, Lx, ox): M' = max(M, m), o = e^(M - M') o +
    // e^(m - M') o_b, same for l; while the running maximum holds the state is not rescaled
    auto merge = [&](const float *rec, float &Mx, float &Lx, float (&ox)[8]) {
        const float mb = rec[kD];
        if (!hv || mb == -INFINITY) return;  // a block not loaded adds nothing
        const float lb = rec[kD + 1];
        if (mb > Mx) {
            const float fa = Mx == -INFINITY ? 0.0f : exp2f((Mx - mb) * kLog2e);
#pragma unroll
            for (int k = 0; k < 8; k++) ox[k] = fa * ox[k];
            Lx = fa * Lx;
            Mx = mb;
        }
        const float fb = exp2f((mb - Mx) * kLog2e);
#pragma unroll
        for (int k = 0; k < 8; k += 4) {
            const float4 v = *reinterpret_cast<const float4 *>(rec + cq + k);
            ox[k] = fmaf(fb, v.x, ox[k]);
            ox[k + 1] = fmaf(fb, v.y, ox[k + 1]);
            ox[k + 2] = fmaf(fb, v.z, ox[k + 2]);
            ox[k + 3] = fmaf(fb, v.w, ox[k + 3]);
        }
        Lx = fmaf(fb, lb, Lx);
    };
    const float *states = reinterpret_cast<const float *>(base + kArtState);
    for (int p = 0; p < nl; p += 2) {
        const bool two = p + 1 < nl;
        const int ja = p / kArtGroups, sa = (p % kArtGroups) * 2 + (ja & 1);
        const int jb = (p + 1) / kArtGroups, sb = ((p + 1) % kArtGroups) * 2 + (jb & 1);
        bool ok = art_wait(a, ctl, &ctl.state_full[sa], (ja >> 1) & 1, -1);
        if (two && ok) ok = art_wait(a, ctl, &ctl.state_full[sb], (jb >> 1) & 1, -1);
        ok = __all_sync(0xffffffffu, ok);
        float Ma = M, La = Ls, oa[8];
#pragma unroll
        for (int k = 0; k < 8; k++) oa[k] = o[k];
        if (ok) merge(states + (sa * kMaxG + (hv ? hh : 0)) * kPartStride, Ma, La, oa);
        float Mb = Ma, Lb = La, ob[8];
#pragma unroll
        for (int k = 0; k < 8; k++) ob[k] = oa[k];
        if (ok && two) merge(states + (sb * kMaxG + (hv ? hh : 0)) * kPartStride, Mb, Lb, ob);
        // the probes P = o / l of this lane's head: |P| = |o| / l and the direction o / |o|
        // (l cancels), |o|^2 over the head's sixteen lanes; then the direction changes, a against
        // the last probe, b against a
        float qa = 0.0f, qb = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; k++) {
            qa = fmaf(oa[k], oa[k], qa);
            qb = fmaf(ob[k], ob[k], qb);
        }
#pragma unroll
        for (int o2 = 1; o2 < 16; o2 <<= 1) {
            qa += __shfl_xor_sync(0xffffffffu, qa, o2);
            qb += __shfl_xor_sync(0xffffffffu, qb, o2);
        }
        const float nca = sqrtf(qa) * (La > 0.0f ? __frcp_rn(La) : 0.0f);
        const float ncb = sqrtf(qb) * (Lb > 0.0f ? __frcp_rn(Lb) : 0.0f);
        const float rna = qa > 0.0f ? rsqrtf(qa) : 0.0f, rnb = qb > 0.0f ? rsqrtf(qb) : 0.0f;
        float da = 0.0f, db = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; k++) {
            const float ca = oa[k] * rna, cb = ob[k] * rnb;
            const float ea = ca - px[k], eb = cb - ca;
            da = fmaf(ea, ea, da);
            db = fmaf(eb, eb, db);
            px[k] = two ? cb : ca;  // the direction of the last probe taken
        }
#pragma unroll
        for (int o2 = 1; o2 < 16; o2 <<= 1) {
            da += __shfl_xor_sync(0xffffffffu, da, o2);
            db += __shfl_xor_sync(0xffffffffu, db, o2);
        }
        float dsa = 0.0f, dra = 0.0f, dsb = 0.0f, drb = 0.0f;
        if (hv) {
            head_metrics(nca, pn, da, dsa, dra);
            head_metrics(ncb, nca, db, dsb, drb);
        }
        dsa = fmaxf(dsa, __shfl_xor_sync(0xffffffffu, dsa, 16));
        dra = fmaxf(dra, __shfl_xor_sync(0xffffffffu, dra, 16));
        dsb = fmaxf(dsb, __shfl_xor_sync(0xffffffffu, dsb, 16));
        drb = fmaxf(drb, __shfl_xor_sync(0xffffffffu, drb, 16));
        float *met = ctl.seq_met[(p >> 1) & 1][sw];
        if (lane == 0) {
            met[0] = dsa;
            met[1] = dra;
            met[2] = dsb;
            met[3] = drb;
        }
        // every sequencer warp has read the slots and written its maxima (one decision for all)
        if (named_barrier_or(kArtSeqBar, 32 * kArtSeqWarps, !ok)) break;
        if (sw == 0 && lane == 0) {
            mbar_arrive(&ctl.state_empty[sa]);
            if (two) mbar_arrive(&ctl.state_empty[sb]);
        }
        float m4[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            m4[i] = ctl.seq_met[(p >> 1) & 1][0][i];
#pragma unroll
            for (int w = 1; w < kArtSeqWarps; w++) m4[i] = fmaxf(m4[i], ctl.seq_met[(p >> 1) & 1][w][i]);
        }
        // block a: the criterion is first checked after the second block
        bool stop = false;
        if (used + 1 >= 2) {
            streak = (m4[0] < prm.tau && m4[1] < prm.phi) ? streak + 1 : 0;
            stop = streak >= prm.patience;
        }
        if (stop || !two) {  // the state after a is the last one
            M = Ma;
            Ls = La;
#pragma unroll
            for (int k = 0; k < 8; k++) o[k] = oa[k];
            pn = nca;
            used += 1;
            if (stop) break;
            continue;
        }
        streak = (m4[2] < prm.tau && m4[3] < prm.phi) ? streak + 1 : 0;
        M = Mb;
        Ls = Lb;
#pragma unroll
        for (int k = 0; k < 8; k++) o[k] = ob[k];
        pn = ncb;
        used += 2;
        if (streak >= prm.patience) break;
    }
    // the groups stop fetching and scoring past the stop (also after an abort)
    if (sw == 0 && lane == 0) *reinterpret_cast<volatile int32_t *>(&ctl.stop_at) = used;
    // out = o / l: this lane's 8 channels of its head
    if (hv) {
        float *ob = a.out + ((size_t)b * a.Hq + h * G + hh) * kD + cq;
        const float iv = Ls > 0.0f ? 1.0f / Ls : 0.0f;
#pragma unroll
        for (int k = 0; k < 8; k += 4)
            *reinterpret_cast<float4 *>(ob + k) =
                make_float4(o[k] * iv, o[k + 1] * iv, o[k + 2] * iv, o[k + 3] * iv);
    }
    if (prm.used && sw == 0 && lane == 0) prm.used[u] = used;
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
