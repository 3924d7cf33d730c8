// sparse.cu -- the scan-then-refine schedule of the FFD decode step: one cooperative launch in two
// phases, for steps where most blocks are dropped.
//
// Source: "Faster Than Flash", Methodology §2 (keep token j when s_ij >= m~_i - delta, m~_i the
// maximum exact score over the sink and local tokens; the blocks holding those are always kept)
// and §3 (stage 1 pseudo-max, stage 2 scan of the 2-bit keys and block filter, stage 3 exact
// attention over the selected blocks). The arithmetic is the fused kernel's (decode.cu); only the
// order of the work differs:
//   phase A  stage 1 (every refine group of the grid takes its (unit, forced block) pairs), then
//            each CTA scans an equal contiguous range of all blocks: every compute warp scores
//            whole blocks (all 64 rows, every head of the group) and keeps, per block and head, the
//            maximum provisional score. A block is kept when it holds a sink or local token or when
//            some head's maximum reaches m~ - delta, which is the Top-delta rule (some token and
//            head reach the threshold exactly when the maximum over them does). The kept blocks go,
//            in block order, to the CTA's list;
//   grid-wide barrier;
//   phase B  the kept blocks of all CTAs, in order, are cut into equal contiguous shares, one per
//            CTA, so the refinement is balanced by kept work rather than by block count: each kept
//            block's thumbnail record, residual record and V tile land in a ring slot by bulk and
//            tensor copies, and a refine group computes its exact scores (thumbnail + residual, on
//            the tensor cores), the softmax and P.V; the split records of each unit are merged as in
//            the fused kernel.
// The fused kernel overlaps the scan with the refinement, which suits steps that keep most blocks;
// this one scans with every compute warp and balances the refinement, which suits sparse steps.
#include <string.h>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "ptx.cuh"
#include "scan.cuh"
#include "splitkv.cuh"
#include "stage1.cuh"

namespace ffd {
namespace {

constexpr int kSpGroups = 3;                // compute groups of 4 warps (warps 4 .. 15)
constexpr int kSpWarps = 4 * kSpGroups;     // compute warps
constexpr int kSpThreads = 128 + 32 * kSpWarps;  // a producer warpgroup + the compute warps
constexpr int kSpActive = 32 + 32 * kSpWarps;    // warp 0 and the compute warps
// Registers: the launch gives 128 a thread (512 threads fill the 64K file), kept through phase A
// (warp 0 stages thumbnails, warps 1-3 run stage 1, the compute warps scan). Phase B: the
// producer warpgroup drops to 56 (warps 1-3 leave) and the compute warpgroups (the refinement)
// rise to 152, which again fills the file; each SM sub-partition holds one warp of each
// warpgroup (56 + 3 * 152 = 512 registers a lane).
constexpr int kSpProducerRegs = 56, kSpComputeRegs = 152;
static_assert(128 * kSpProducerRegs + 32 * kSpWarps * kSpComputeRegs == 65536, "register split");
// named barriers: 1 the producer and compute warps, 2 + g refine group g, kSpComputeBar the compute
// warps, kSpScanBar every warp that scans (warps 1 .. 15: the stage-1 warps join the scan)
constexpr int kSpActiveBar = 1;
constexpr int kSpComputeBar = 2 + kSpGroups;
constexpr int kSpScanBar = 3 + kSpGroups;
constexpr int kSpScanners = 32 * (3 + kSpWarps);

// Phase A: thumbnail stages (block li of the range uses stage li % kSpStages; the scanning warps
// take blocks in order from a shared counter), and the per-block head maxima of one chunk of the
// range. 48 stages keep 96 to 144 KB of thumbnails in flight per SM, which covers the copy latency
// at the HBM rate.
constexpr int kSpStages = 48;
constexpr int kSpIssue = 16;                // stages armed at a time by the producer warp
static_assert(kSpStages % kSpIssue == 0 && 32 % kSpIssue == 0, "issue batches");
constexpr int kSpChunk = 512;               // range blocks whose maxima are held at once
constexpr int kSpOffStages = 0;
constexpr int kSpOffBmax = kSpOffStages + kSpStages * kThumbRec;    // float [kSpChunk][kMaxG]
constexpr int kSpOffBunit = kSpOffBmax + kSpChunk * kMaxG * 4;       // int2 [kSpChunk]: (u, blk)
constexpr int kSpOffWcnt = kSpOffBunit + kSpChunk * 8;               // int [kSpChunk / 32 + 1]
constexpr int kSpPhaseA = kSpOffWcnt + (kSpChunk / 32 + 1) * 4;

// Phase B: ring slots (residual record, V tile with the 128-byte swizzle, thumbnail record);
// kept block j of the CTA's share uses slot j % kSpRing and refine group j % kSpGroups.
constexpr int kSpRing = 6;
static_assert(kSpRing % kSpGroups == 0, "a ring slot always serves the same refine group");
constexpr int kSpSlotV = 9216;
constexpr int kSpSlotThumb = kSpSlotV + 16384;
constexpr int kSpSlotBytes = kSpSlotThumb + kThumbRec;
constexpr int kSpSlotTx = kResidRec + 16384 + kThumbRec;
static_assert(kResidRec <= kSpSlotV && kSpSlotV % 1024 == 0, "slot layout");
constexpr int kSpPhaseB = ((kSpRing * kSpSlotBytes + 1023) / 1024) * 1024;

constexpr int kSpOffShared = kSpPhaseA > kSpPhaseB ? kSpPhaseA : kSpPhaseB;
constexpr int kSpOffPx = ((kSpOffShared + 1023) / 1024) * 1024;      // [group][2][kPxBuf]
// the refine groups' records of a unit's segment, combined into the CTA's one record
constexpr int kSpOffComb = kSpOffPx + kSpGroups * 2 * kPxBuf;        // float [group][kMaxG][stride]
// each refine group's copy of the current unit's query rows (bf16 [kMaxG][kD])
constexpr int kSpOffQ = kSpOffComb + kSpGroups * kMaxG * kPartStride * 4;
constexpr int kSpOffMisc = kSpOffQ + kSpGroups * kMaxG * kD * 2;
constexpr int kSpMaxCtas = 256;
constexpr int kSpMiscBytes = 5120;
constexpr int kSpSmemBytes = kSpOffMisc + kSpMiscBytes + 1024;       // + slack to align to 1 KB
static_assert(kSpSmemBytes <= 232448, "shared memory per CTA");

struct SpDesc {       // a phase-A stage: the block it holds (page -1: not loaded)
    int32_t u, blk, rows, page;
};

struct SpMisc {
    uint32_t aborted;
    uint32_t merge_flag[kSpGroups];
    uint32_t over[kSpGroups][2][4];       // softmax_pv
    float wmax[kSpGroups][2][4][kMaxG];   // softmax_pv, stage 1
    float lsum[kSpGroups][4][kMaxG];      // write_record
    int32_t ured[kSpGroups][4];           // per-group sums (a unit's first kept index)
    int32_t pref[kSpMaxCtas + 1];         // phase B: prefix of the CTAs' kept counts
    int32_t kept;                         // phase A: kept blocks of this CTA so far
    int32_t scan_next;                    // phase A: next block of the chunk to score
    SpDesc desc[kSpStages];
    int32_t armed_a[kSpStages];           // uses armed per phase-A stage
    int32_t armed_b[kSpRing];             // uses armed per phase-B ring slot
    uint64_t a_full[kSpStages], a_empty[kSpStages];
    uint64_t b_full[kSpRing], b_empty[kSpRing];
};
static_assert(sizeof(SpMisc) <= kSpMiscBytes, "control block");

struct SpParams {
    CUtensorMap tm_v;
    DecodeArgs a;
};

// Blocks of all units and this CTA's phase-A range [x, x1) of them (equal contiguous ranges).
struct SpRange {
    int T, ncta, x, x1;
};

__device__ __forceinline__ SpRange sp_range(const DecodeArgs &a) {
    SpRange r;
    r.T = 0;
    for (int b = 0; b < a.B; b++) r.T += a.Hkv * ((len_of(a, b) + kPage - 1) / kPage);
    r.ncta = r.T < (int)gridDim.x ? r.T : (int)gridDim.x;
    const int c = blockIdx.x;
    r.x = c < r.ncta ? (int)((int64_t)r.T * c / r.ncta) : 0;
    r.x1 = c < r.ncta ? (int)((int64_t)r.T * (c + 1) / r.ncta) : 0;
    return r;
}

// Unit and block of global block index x (units in order, each unit's blocks in order).
__device__ __forceinline__ int2 sp_locate(const DecodeArgs &a, int x) {
    int pre = 0;
    for (int b = 0; b < a.B; b++) {
        const int nb = (len_of(a, b) + kPage - 1) / kPage;
        if (x < pre + a.Hkv * nb) {
            const int h = (x - pre) / nb;
            return make_int2(b * a.Hkv + h, (x - pre) - h * nb);
        }
        pre += a.Hkv * nb;
    }
    return make_int2(0, 0);  // not reached for x < T
}

// ------------------------------------------------------------------------------------------
// Phase A
// ------------------------------------------------------------------------------------------
// Where range block x lies: its unit, block, rows and page (-1 for a block-table entry outside
// [0, P)).
struct SpLook {
    int u, blk, rows, page;
};
__device__ __forceinline__ SpLook sp_lookup(const DecodeArgs &a, int x) {
    const int2 ub = sp_locate(a, x);
    const int b = ub.x / a.Hkv;
    SpLook l;
    l.u = ub.x;
    l.blk = ub.y;
    l.page = a.block_table[(size_t)b * a.max_blocks + ub.y];
    if (l.page < 0 || l.page >= a.P) l.page = -1;
    const int n = len_of(a, b);
    l.rows = n - ub.y * kPage < kPage ? n - ub.y * kPage : kPage;
    return l;
}

// Producer warp: range block li (global x + li) goes to stage li % kSpStages once the stage's
// previous block has been scored. The lanes look up 32 blocks at once, those after the ones being
// armed, so that the lookups overlap the waits; the blocks are armed kSpIssue at a time (lane k of
// a batch arms its own block), so a batch waits for blocks kSpStages earlier while the other
// stages stay in flight. A block whose block-table entry lies outside [0, P) is flagged
// (FFD_ERRBIT_BOUNDS) and not loaded.
__device__ __forceinline__ void sp_stage_issuer(const DecodeArgs &a, SpMisc *m, uint8_t *base,
                                                const SpRange &r, int lane) {
    const int len = r.x1 - r.x;
    SpLook cur = lane < len ? sp_lookup(a, r.x + lane) : SpLook{0, 0, 0, -1};
    for (int li0 = 0; li0 < len; li0 += 32) {
        const SpLook nxt =
            li0 + 32 + lane < len ? sp_lookup(a, r.x + li0 + 32 + lane) : SpLook{0, 0, 0, -1};
#pragma unroll 1
        for (int half = 0; half < 32 / kSpIssue; half++) {
            const int li = li0 + lane;
            if (lane / kSpIssue == half && li < len) {
                const int b = cur.u / a.Hkv, h = cur.u - b * a.Hkv;
                const int st = li % kSpStages, use = li / kSpStages;
                if (use > 0) wait_bar(a, m, &m->a_empty[st], (use - 1) & 1);
                // after an abort nothing more is armed: the stage may still be filling
                if (!aborted(m)) {
                    m->desc[st] = SpDesc{cur.u, cur.blk, cur.rows, cur.page};
                    if (cur.page < 0) {
                        raise_error(a.err, FFD_ERRBIT_BOUNDS);
                        mbar_arrive(&m->a_full[st]);
                    } else {
                        mbar_arrive_expect_tx(&m->a_full[st], kThumbRec);
                        tma_load_1d(base + kSpOffStages + st * kThumbRec,
                                    a.thumb + ((size_t)cur.page * a.Hkv + h) * kThumbRec,
                                    kThumbRec, &m->a_full[st]);
                    }
                    m->armed_a[st] = use + 1;
                }
            }
            __syncwarp();
        }
        cur = nxt;
    }
    // leave no copy in flight: the last armed use of every stage
    __syncwarp();
    for (int st = lane; st < kSpStages; st += 32)
        if (m->armed_a[st] > 0) drain_bar(a, &m->a_full[st], (m->armed_a[st] - 1) & 1);
}

// Bounded wait until the producer has armed use `target - 1` of stage st (the stage's previous
// block has then been scored, so the parity wait that follows is unambiguous).
__device__ __forceinline__ void wait_armed(const DecodeArgs &a, SpMisc *m, int st, int target) {
    const volatile int32_t *armed = &m->armed_a[st];
    if (*armed >= target) return;
    const uint64_t t0 = globaltimer_ns();
    while (*armed < target) {
        if (aborted(m)) return;
        if (globaltimer_ns() - t0 > a.wait_ns) {
            raise_error(a.err, FFD_ERRBIT_TIMEOUT);
            *reinterpret_cast<volatile uint32_t *>(&m->aborted) = 1;
            return;
        }
        __nanosleep(32);  // leave the issue slots to the warps that are scoring
    }
}

// A scanning warp takes blocks li of chunk [c0, c1) in order from m->scan_next and scores each:
// for each head of the group the maximum provisional score over the block's tokens (-inf for a
// block not loaded, and for heads past G), into bmax[li - c0]; (u * max_blocks + block, page) into
// bunit (-1 for a block not loaded). The maximum is taken over scan_tile_raw's scores and scaled
// once.
__device__ __forceinline__ void sp_scan_chunk(const DecodeArgs &a, SpMisc *m, uint8_t *base,
                                              int c0, int c1, int lane, ThumbOps &Q,
                                              float (&qsr)[2][4], int &qu) {
    const int g = lane >> 2, tig = lane & 3;
    const uint32_t m0 = 0x00030003u << (2 * tig);
    float *bmax = reinterpret_cast<float *>(base + kSpOffBmax);
    int2 *bunit = reinterpret_cast<int2 *>(base + kSpOffBunit);
    const float post = a.sm_scale * kUnscale;  // exact: kUnscale is a power of two
    // the next block is taken while the current one is scored (a warp holds at most two blocks,
    // fewer than the stages, so the producer never waits on a block nobody can score)
    int li_next = 0;
    if (lane == 0) li_next = c0 + atomicAdd(&m->scan_next, 1);
    for (;;) {
        const int li = __shfl_sync(0xffffffffu, li_next, 0);
        if (li >= c1) break;
        const int st = li % kSpStages, use = li / kSpStages;
        wait_armed(a, m, st, use + 1);
        wait_bar(a, m, &m->a_full[st], use & 1);
        if (lane == 0) li_next = c0 + atomicAdd(&m->scan_next, 1);
        SpDesc d = m->desc[st];
        if (d.u < 0 || d.u >= a.B * a.Hkv) d.page = -1;  // only after a wait ran out
        float mh0 = -INFINITY, mh1 = -INFINITY;
        if (d.page >= 0) {  // warp-uniform
            if (d.u != qu) {  // the unit's query operands (thumbnail B fragments, query sums)
                const int b = d.u / a.Hkv;
                load_thumb_ops(a, b, d.u - b * a.Hkv, lane, Q);
#pragma unroll
                for (int i = 0; i < 2; i++)
#pragma unroll
                    for (int gg = 0; gg < 4; gg++) qsr[i][gg] = Q.qs[i][gg] * (1.0f / kUnscale);
                qu = d.u;
            }
            const uint8_t *rec = base + kSpOffStages + st * kThumbRec;
#pragma unroll
            for (int mt = 0; mt < 4; mt++) {
                const float4 e = scan_tile_raw(rec, 16 * mt + g, 16 * mt + g + 8, m0, Q, qsr);
                const bool v0 = 16 * mt + g < d.rows, v1 = 16 * mt + g + 8 < d.rows;
                mh0 = fmaxf(mh0, fmaxf(v0 ? e.x : -INFINITY, v1 ? e.z : -INFINITY));
                mh1 = fmaxf(mh1, fmaxf(v0 ? e.y : -INFINITY, v1 ? e.w : -INFINITY));
            }
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                mh0 = fmaxf(mh0, __shfl_xor_sync(0xffffffffu, mh0, o));
                mh1 = fmaxf(mh1, __shfl_xor_sync(0xffffffffu, mh1, o));
            }
            mh0 *= post;
            mh1 *= post;
        }
        __syncwarp();  // every lane has read the stage
        if (lane == 0) mbar_arrive(&m->a_empty[st]);
        if (g == 0) {
            bmax[(li - c0) * kMaxG + 2 * tig] = 2 * tig < a.G ? mh0 : -INFINITY;
            bmax[(li - c0) * kMaxG + 2 * tig + 1] = 2 * tig + 1 < a.G ? mh1 : -INFINITY;
        }
        if (lane == 0)
            bunit[li - c0] = d.page < 0 ? make_int2(-1, 0) : make_int2(d.u * a.max_blocks + d.blk, d.page);
    }
}

// Votes of chunk [c0, c1) and its kept blocks, in block order, appended to the CTA's list at
// ws_kept[x + kept]. The compute warps take windows of 32 blocks (lane = block); pass 1 counts
// each window's kept blocks, pass 2 writes them after the preceding windows'. The thresholds
// m~ - delta of a unit come from ws_mt once its stage-1 slots are all in (slot counter nf + 1).
__device__ __forceinline__ void sp_vote_chunk(const DecodeArgs &a, SpMisc *m, uint8_t *base,
                                              int x, int c0, int c1, int cw, int lane,
                                              int ubuf) {
    const float *bmax = reinterpret_cast<const float *>(base + kSpOffBmax);
    const int2 *bunit = reinterpret_cast<const int2 *>(base + kSpOffBunit);
    int *wcnt = reinterpret_cast<int *>(base + kSpOffWcnt);
    const int nwin = (c1 - c0 + 31) / 32;
    constexpr int kWin = (kSpChunk / 32 + kSpWarps - 1) / kSpWarps;  // windows per warp, at most
    uint32_t keepbits[kWin];
#pragma unroll
    for (int nw = 0; nw < kWin; nw++) {
        const int w = cw + nw * kSpWarps;
        keepbits[nw] = 0u;
        if (w >= nwin) continue;  // warp-uniform
        const int li = c0 + 32 * w + lane;
        bool keep = false;
        if (li < c1) {
            const int2 ub = bunit[li - c0];
            if (ub.x >= 0) {
                const int u = ub.x / a.max_blocks, blk = ub.x - u * a.max_blocks;
                const int n = len_of(a, u / a.Hkv);
                const ForcedBlocks fb(n, a.S, a.L);
                keep = fb.forced(blk);
                if (!keep) {
                    wait_count(a, m, slot_counter(a, u), a.nf + 1);
                    // the unit's eight thresholds at once (heads past G are not compared)
                    const float4 *mt = reinterpret_cast<const float4 *>(a.ws_mt + (size_t)u * kMaxG);
                    const float4 t0 = __ldcg(mt), t1 = __ldcg(mt + 1);
                    const float th[kMaxG] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
#pragma unroll
                    for (int i = 0; i < kMaxG; i++)
                        keep |= i < a.G && bmax[(li - c0) * kMaxG + i] >= th[i] - a.delta;
                }
            }
            if (a.keep_mask && ub.x >= 0)
                a.keep_mask[ub.x] = keep ? 1 : 0;  // u * max_blocks + block
            else if (a.keep_mask) {  // a block not loaded: its unit is located again
                const int2 u2 = sp_locate(a, x + li);
                a.keep_mask[(size_t)u2.x * a.max_blocks + u2.y] = 0;
            }
        }
        const uint32_t bits = __ballot_sync(0xffffffffu, keep);
        keepbits[nw] = bits;
        if (lane == 0) wcnt[w] = __popc(bits);
    }
    named_barrier_sync(kSpComputeBar, 32 * kSpWarps);
    if (cw == 0) {  // exclusive prefix over the windows, after the kept blocks of earlier chunks
        int run = m->kept;
        for (int w0 = 0; w0 < nwin; w0 += 32) {
            const int c = w0 + lane < nwin ? wcnt[w0 + lane] : 0;
            int inc = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += y;
            }
            if (w0 + lane < nwin) wcnt[w0 + lane] = run + inc - c;
            run += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0) {
            m->kept = run;
            m->scan_next = 0;  // every scanner has left the chunk's loop
        }
    }
    named_barrier_sync(kSpComputeBar, 32 * kSpWarps);
#pragma unroll
    for (int nw = 0; nw < kWin; nw++) {
        const int w = cw + nw * kSpWarps;
        if (w >= nwin) continue;
        const uint32_t bits = keepbits[nw];
        if ((bits >> lane) & 1u) {
            const int li = c0 + 32 * w + lane;
            const int2 ub = bunit[li - c0];
            a.ws_kept[x + wcnt[w] + __popc(bits & ((1u << lane) - 1u))] = ub;
            atomicAdd(a.ws_ukept + (size_t)ubuf * a.B * a.Hkv + ub.x / a.max_blocks, 1);
        }
    }
    named_barrier_sync(kSpScanBar, kSpScanners);  // the chunk's buffers may be refilled
}

// ------------------------------------------------------------------------------------------
// Phase B
// ------------------------------------------------------------------------------------------
// Kept block k of all CTAs' lists (k < K): its (u * max_blocks + block, page). pref[c] = kept
// blocks of the CTAs before c; CTA c's list starts at its range start.
__device__ __forceinline__ int2 sp_kept(const DecodeArgs &a, const SpMisc *m, const SpRange &r,
                                        int k) {
    int lo = 0, hi = r.ncta - 1;  // the last CTA c with pref[c] <= k
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (m->pref[mid] <= k) lo = mid;
        else hi = mid - 1;
    }
    const int xs = (int)((int64_t)r.T * lo / r.ncta);
    const int2 e = a.ws_kept[xs + (k - m->pref[lo])];
    // every entry was written this call unless a wait ran out somewhere: checked all the same
    return e.x >= 0 && e.x < a.B * a.Hkv * a.max_blocks && e.y >= 0 && e.y < a.P ? e
                                                                               : make_int2(0, 0);
}

// Producer warp: kept block j of the share [s0, s1) goes to slot j % kSpRing once it is free
// (its previous block refined). The lanes look up 32 kept blocks at once (entry and page), the
// next 32 while the current ones are armed; lane k of a batch of kSpRing arms block j0 + k.
__device__ __forceinline__ int2 sp_ring_lookup(const DecodeArgs &a, const SpMisc *m,
                                               const SpRange &r, int k) {
    const int2 e = sp_kept(a, m, r, k);
    return make_int2((e.x / a.max_blocks) % a.Hkv, e.y);  // (KV head, page)
}

__device__ __forceinline__ void sp_ring_issuer(const SpParams &prm, SpMisc *m, uint8_t *base,
                                               const SpRange &r, int s0, int s1, int lane) {
    const DecodeArgs &a = prm.a;
    const int len = s1 - s0;
    int2 cur = lane < len ? sp_ring_lookup(a, m, r, s0 + lane) : make_int2(0, 0);
    for (int jb = 0; jb < len; jb += 32) {
        const int2 nxt = jb + 32 + lane < len ? sp_ring_lookup(a, m, r, s0 + jb + 32 + lane)
                                              : make_int2(0, 0);
        const int je = len < jb + 32 ? len : jb + 32;
        for (int j0 = jb; j0 < je; j0 += kSpRing) {
            const int j = j0 + lane;
            const int src = (j - jb) & 31;
            const int h = __shfl_sync(0xffffffffu, cur.x, src);
            const int page = __shfl_sync(0xffffffffu, cur.y, src);
            if (lane < kSpRing && j < je) {
                const int slot = j % kSpRing, use = j / kSpRing;
                if (use > 0) wait_bar(a, m, &m->b_empty[slot], (use - 1) & 1);
                if (!aborted(m)) {  // after an abort nothing more is armed
                    const size_t tile = (size_t)page * a.Hkv + h;
                    uint8_t *d = base + slot * kSpSlotBytes;
                    mbar_arrive_expect_tx(&m->b_full[slot], kSpSlotTx);
                    tma_load_1d(d, a.resid + tile * kResidRec, kResidRec, &m->b_full[slot]);
                    tma_load_3d(d + kSpSlotV, &prm.tm_v, 0, (int)(tile * kPage), 0,
                                &m->b_full[slot]);
                    tma_load_1d(d + kSpSlotThumb, a.thumb + tile * kThumbRec, kThumbRec,
                                &m->b_full[slot]);
                    m->armed_b[slot] = use + 1;
                }
            }
            __syncwarp();
        }
        cur = nxt;
    }
    // leave no copy in flight: the last armed use of every slot
    __syncwarp();
    for (int slot = lane; slot < kSpRing; slot += 32)
        if (m->armed_b[slot] > 0) drain_bar(a, &m->b_full[slot], (m->armed_b[slot] - 1) & 1);
}

// Kept blocks before unit u in the kept order (the units' counts, summed by refine group grp).
__device__ __forceinline__ int sp_unit_first(const DecodeArgs &a, SpMisc *m, const int *ukept,
                                             int u, int grp, int mt, int lane) {
    int s = 0;
    for (int v = 32 * mt + lane; v < u; v += 128) s += __ldcg(ukept + v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) m->ured[grp][mt] = s;
    named_barrier_sync(2 + grp, 128);
    const int t = m->ured[grp][0] + m->ured[grp][1] + m->ured[grp][2] + m->ured[grp][3];
    named_barrier_sync(2 + grp, 128);
    return t;
}

// Refine group grp: walks the share's kept blocks in order (every group sees every unit change,
// and every CTA-wide barrier below) and refines blocks j = grp (mod kSpGroups) from ring slot
// j % kSpRing. At the end of a unit's segment the three groups' softmax states go to shared memory
// and group 0 combines them into the CTA's one record of the unit (records, tickets and merge
// reads are a third of one record per group), then takes the unit's ticket and merges when last.
// After an abort a group stops computing but keeps walking, so that the barriers still match.
__device__ __forceinline__ void sp_combine(const DecodeArgs &a, const float *rec, float *dst,
                                           int tid) {
    for (int i = 0; i < a.G; i++) {
        const float *r0 = rec + (size_t)i * kPartStride;
        const float *r1 = r0 + kMaxG * kPartStride, *r2 = r1 + kMaxG * kPartStride;
        const float m0 = r0[kD], m1 = r1[kD], m2 = r2[kD];
        const float M = fmaxf(m0, fmaxf(m1, m2));  // finite: references never go to -inf
        const float f0 = exp2f((m0 - M) * kLog2e), f1 = exp2f((m1 - M) * kLog2e);
        const float f2 = exp2f((m2 - M) * kLog2e);
        float *d = dst + (size_t)i * kPartStride;
        d[tid] = fmaf(f2, r2[tid], fmaf(f1, r1[tid], f0 * r0[tid]));
        if (tid == 0) {
            d[kD] = M;
            d[kD + 1] = fmaf(f2, r2[kD + 1], fmaf(f1, r1[kD + 1], f0 * r0[kD + 1]));
        }
    }
}

__device__ __forceinline__ void sp_refiner(const DecodeArgs &a, SpMisc *m, uint8_t *base,
                                           const SpRange &r, int K, int nctab, int s0, int s1,
                                           const int *ukept, int grp, int mt, int lane) {
    const int g = lane >> 2, tig = lane & 3;
    const int r0 = 16 * mt + g, r1 = r0 + 8;
    const int cta = blockIdx.x;
    float *comb = reinterpret_cast<float *>(base + kSpOffComb);
    ThumbOps Q;
    ResidOps QR;
    RefineState R;
    int cu = -1, seg0 = 0, n = 0, pb = 0;
    bool dead = false;  // group-uniform: stopped computing after an abort
    auto end_segment = [&](int k_end) {
        if (!dead) write_record(a, m, R, comb + grp * kMaxG * kPartStride, grp, mt, lane);
        // every group's record is in; one decision for the whole CTA
        const bool live = !named_barrier_or(kSpComputeBar, 32 * kSpWarps, aborted(m));
        if (grp == 0 && live)
            sp_combine(a, comb, unit_record<1>(a, cu, cta, 0), 32 * mt + lane);
        named_barrier_sync(kSpComputeBar, 32 * kSpWarps);  // the shared records are free again
        if (grp == 0 && live) {
            const int b = cu / a.Hkv;
            Sub s;
            s.b = b;
            s.h = cu - b * a.Hkv;
            s.cnt = k_end - seg0;
            s.x0 = seg0;
            const int first = sp_unit_first(a, m, ukept, cu, grp, mt, lane);
            s.j0 = seg0 - first;
            s.nblk = __ldcg(ukept + cu);
            s.first = s.last = true;
            finish_unit<SpMisc, 1>(a, m, s, cta, nctab, K, grp, mt, lane);
        }
    };
    for (int j0 = 0; j0 < s1 - s0; j0 += 32) {
        // the (unit, block) of 32 consecutive kept blocks, one per lane
        const int jl = j0 + lane < s1 - s0 ? j0 + lane : s1 - s0 - 1;
        const int2 mine = sp_kept(a, m, r, s0 + jl);
        const int mu = mine.x / a.max_blocks, mblk = mine.x - mu * a.max_blocks;
        const int cnt = s1 - s0 - j0 < 32 ? s1 - s0 - j0 : 32;
        for (int i = 0; i < cnt; i++) {
            const int j = j0 + i;
            const int u = __shfl_sync(0xffffffffu, mu, i);
            const int blk = __shfl_sync(0xffffffffu, mblk, i);
            if (u != cu) {  // CTA-uniform
                if (cu >= 0) end_segment(s0 + j);
                cu = u;
                seg0 = s0 + j;
                const int b = u / a.Hkv, h = u - b * a.Hkv;
                // the group's query rows, staged once (the previous unit's readers have all passed
                // end_segment's barriers)
                __nv_bfloat16 *sq = reinterpret_cast<__nv_bfloat16 *>(base + kSpOffQ) + grp * kMaxG * kD;
                stage_query(a, b, h, sq, 32 * mt + lane, 128);
                named_barrier_sync(2 + grp, 128);
                thumb_ops_from_row(sq + (g < a.G ? g : 0) * kD, g < a.G, lane, a.err, Q);
                resid_ops_from_row(sq + (g < a.G ? g : 0) * kD, g < a.G, lane, QR);
                n = len_of(a, b);
                const float mt0 = __ldcg(a.ws_mt + (size_t)u * kMaxG + 2 * tig);
                const float mt1 = __ldcg(a.ws_mt + (size_t)u * kMaxG + 2 * tig + 1);
                R.m0 = mt0 == -INFINITY ? kNoReference : mt0;
                R.m1 = mt1 == -INFINITY ? kNoReference : mt1;
                R.nl0 = -R.m0 * kLog2e;
                R.nl1 = -R.m1 * kLog2e;
                R.l0 = R.l1 = 0.0f;
#pragma unroll
                for (int q = 0; q < 2; q++) R.o[q][0] = R.o[q][1] = R.o[q][2] = R.o[q][3] = 0.0f;
            }
            if (j % kSpGroups != grp || dead) continue;
            const int slot = j % kSpRing;
            wait_bar(a, m, &m->b_full[slot], (j / kSpRing) & 1);
            // a slot that never filled (a wait ran out) must not split the group's barriers
            dead = named_barrier_or(2 + grp, 128, aborted(m));
            if (dead) continue;
            uint8_t *d = base + slot * kSpSlotBytes;
            const int rows = n - blk * kPage < kPage ? n - blk * kPage : kPage;
            if (rows < kPage) {  // the sequence's partial last block: V rows past it are zeroed
                for (int c = 32 * mt + lane; c < (kPage - rows) * 16; c += 128) {
                    const int rr = rows + (c >> 4), half = (c >> 3) & 1;
                    *reinterpret_cast<uint4 *>(d + kSpSlotV + half * 8192 + rr * 128 +
                                               (c & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async();  // before the slot's next bulk copy
                named_barrier_sync(2 + grp, 128);
            }
            const float4 e = exact_tile(d + kSpSlotThumb, d, r0, r1, tig, Q, QR, a.sm_scale);
            const bool v0 = r0 < rows, v1 = r1 < rows;
            softmax_pv(m, base + kSpOffPx + (grp * 2 + pb) * kPxBuf, d + kSpSlotV,
                       v0 ? e.x : -INFINITY, v0 ? e.y : -INFINITY, v1 ? e.z : -INFINITY,
                       v1 ? e.w : -INFINITY, R, grp, mt, pb, lane);
            pb ^= 1;
            __syncwarp();
            if (lane == 0) mbar_arrive(&m->b_empty[slot]);
        }
    }
    if (cu >= 0) end_segment(s1);
}

// A unit none of whose blocks was kept (every block-table entry out of range): its zero output,
// its m~, and its counters cleared for the next call. CTA c takes units c, c + grid, ...
__device__ __forceinline__ void sp_empty_units(const DecodeArgs &a, const int *ukept, int lane) {
    for (int u = blockIdx.x; u < a.B * a.Hkv; u += gridDim.x) {
        const int b = u / a.Hkv, h = u - b * a.Hkv;
        if (len_of(a, b) == 0 || __ldcg(ukept + u) > 0) continue;
        for (int idx = lane; idx < a.G * kD; idx += 32)
            a.out[((size_t)b * a.Hq + h * a.G) * kD + idx] = 0.0f;
        if (a.m_tilde && lane < a.G)
            a.m_tilde[(size_t)b * a.Hq + h * a.G + lane] = __ldcg(a.ws_mt + (size_t)u * kMaxG + lane);
        if (lane == 0) *slot_counter(a, u) = 0;
    }
}

// ------------------------------------------------------------------------------------------
// The kernel: one CTA per SM, all resident (cooperative launch).
// ------------------------------------------------------------------------------------------
// Thread 0's half of the grid-wide barrier between the phases (bounded). The generation counter
// only grows: call g waits for it to reach (g + 1) * gridDim.x.
__device__ __forceinline__ void sp_grid_barrier(const DecodeArgs &a, SpMisc *m) {
    __threadfence();
    const unsigned int arrived = atomicAdd(a.ws_grid, 1u);
    const unsigned int target = (arrived / gridDim.x + 1u) * gridDim.x;
    const uint64_t t0 = globaltimer_ns();
    while ((int)((unsigned int)ld_acquire_gpu(reinterpret_cast<const int *>(a.ws_grid)) - target) <
           0) {
        if (globaltimer_ns() - t0 > a.wait_ns) {
            raise_error(a.err, FFD_ERRBIT_TIMEOUT);
            m->aborted = 1;
            break;
        }
        __nanosleep(64);
    }
    __threadfence();
}

// This CTA's share [s0, s1) of the K kept blocks, from the prefix of the CTAs' kept counts.
struct SpShare {
    int K, nctab, s0, s1;
};
__device__ __forceinline__ SpShare sp_share(const SpRange &r, const SpMisc *m) {
    SpShare sh;
    sh.K = r.ncta > 0 ? m->pref[r.ncta] : 0;
    sh.nctab = sh.K < (int)gridDim.x ? sh.K : (int)gridDim.x;
    const int c = blockIdx.x;
    sh.s0 = c < sh.nctab ? (int)((int64_t)sh.K * c / sh.nctab) : 0;
    sh.s1 = c < sh.nctab ? (int)((int64_t)sh.K * (c + 1) / sh.nctab) : 0;
    return sh;
}

// ------------------------------------------------------------------------------------------
// The kernel: one CTA per SM, all resident (cooperative launch). Each role runs in its own branch
// from the register split on, meeting the other at barrier 1 (phase A done, grid barrier passed,
// prefix ready).
// ------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kSpThreads, 1) sparse_kernel(const __grid_constant__ SpParams prm) {
    const DecodeArgs &a = prm.a;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = align_shared<1024>(smem_raw);
    SpMisc *m = reinterpret_cast<SpMisc *>(base + kSpOffMisc);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int units = a.B * a.Hkv;
    if (threadIdx.x == 0) {
        m->aborted = 0;
        m->kept = 0;
        m->scan_next = 0;
        for (int i = 0; i < kSpStages; i++) {
            mbar_init(&m->a_full[i], 1);
            mbar_init(&m->a_empty[i], 1);  // the compute warp that scored the block
            m->desc[i] = SpDesc{-1, 0, 0, -1};  // read as "not loaded" if a wait runs out first
            m->armed_a[i] = 0;
        }
        for (int i = 0; i < kSpRing; i++) {
            mbar_init(&m->b_full[i], 1);
            mbar_init(&m->b_empty[i], 4);  // the refine group that took the block
            m->armed_b[i] = 0;
        }
        fence_barrier_init();
    }
    // calls alternate between two per-unit kept-count buffers: this call's generation of the grid
    // barrier (every CTA reads it before the last one arrives)
    const unsigned int gen = *reinterpret_cast<volatile unsigned int *>(a.ws_grid) / gridDim.x;
    const int ubuf = gen & 1;
    int *ukept = a.ws_ukept + (size_t)ubuf * units;
    __syncthreads();
    const SpRange r = sp_range(a);

    if (warp < 4) {
        // ---- phase A: stage the range's thumbnails (warp 0); stage 1 (warps 1-3)
        if (warp == 0) {
            if (lane == 0) prefetch_tensormap(&prm.tm_v);
            if (blockIdx.x < r.ncta) sp_stage_issuer(a, m, base, r, lane);
        } else {
            pseudo_max_warp(a, blockIdx.x * 3 + warp - 1, gridDim.x * 3, lane);
            // then scan with the compute warps (the vote is theirs)
            ThumbOps Q;
            float qsr[2][4];
            int qu = -1;
            for (int c0 = 0; c0 < r.x1 - r.x; c0 += kSpChunk) {
                const int c1 = r.x1 - r.x < c0 + kSpChunk ? r.x1 - r.x : c0 + kSpChunk;
                sp_scan_chunk(a, m, base, c0, c1, lane, Q, qsr, qu);
                named_barrier_sync(kSpScanBar, kSpScanners);  // the chunk's maxima are in
                named_barrier_sync(kSpScanBar, kSpScanners);  // the chunk's votes are in
            }
        }
        regs_decrease<kSpProducerRegs>();  // the whole warpgroup
        if (warp != 0) return;
        named_barrier_sync(kSpActiveBar, kSpActive);
        if (lane == 0) sp_grid_barrier(a, m);
        __syncwarp();
        named_barrier_sync(kSpActiveBar, kSpActive);
        named_barrier_sync(kSpActiveBar, kSpActive);  // the prefix is in
        // ---- phase B: stream the kept blocks of this CTA's share
        const SpShare sh = sp_share(r, m);
        if (sh.s1 > sh.s0 && !aborted(m)) sp_ring_issuer(prm, m, base, r, sh.s0, sh.s1, lane);
        // clear the other kept-count buffer for the next call, and close the units with no kept
        // block
        for (int u = blockIdx.x * 32 + lane; u < units; u += gridDim.x * 32)
            a.ws_ukept[(size_t)(ubuf ^ 1) * units + u] = 0;
        sp_empty_units(a, ukept, lane);
    } else {
        const int cw = warp - 4, grp = cw >> 2, mt = cw & 3;
        // ---- phase A: score and vote the range chunk by chunk
        ThumbOps Q;
        float qsr[2][4];
        int qu = -1;
        for (int c0 = 0; c0 < r.x1 - r.x; c0 += kSpChunk) {
            const int c1 = r.x1 - r.x < c0 + kSpChunk ? r.x1 - r.x : c0 + kSpChunk;
            sp_scan_chunk(a, m, base, c0, c1, lane, Q, qsr, qu);
            named_barrier_sync(kSpScanBar, kSpScanners);  // the chunk's maxima are in
            sp_vote_chunk(a, m, base, r.x, c0, c1, cw, lane, ubuf);
        }
        if (cw == 0 && lane == 0 && blockIdx.x < r.ncta) a.ws_keptn[blockIdx.x] = m->kept;
        named_barrier_sync(kSpActiveBar, kSpActive);
        regs_increase<kSpComputeRegs>();  // once the producer warpgroup has released its share
        named_barrier_sync(kSpActiveBar, kSpActive);  // the grid barrier is passed
        if (cw == 0) {  // prefix of the CTAs' kept counts (all loads first)
            int v[kSpMaxCtas / 32];
#pragma unroll
            for (int k = 0; k < kSpMaxCtas / 32; k++)
                v[k] = 32 * k + lane < r.ncta ? __ldcg(a.ws_keptn + 32 * k + lane) : 0;
            int run = 0;
#pragma unroll
            for (int k = 0; k < kSpMaxCtas / 32; k++) {
                int inc = v[k];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, inc, o);
                    if (lane >= o) inc += y;
                }
                if (32 * k + lane < r.ncta) m->pref[32 * k + lane] = run + inc - v[k];
                run += __shfl_sync(0xffffffffu, inc, 31);
            }
            if (lane == 0) m->pref[r.ncta] = run;
        }
        named_barrier_sync(kSpActiveBar, kSpActive);
        // ---- phase B: refine the kept blocks of this CTA's share
        const SpShare sh = sp_share(r, m);
        if (sh.s1 > sh.s0 && !aborted(m))
            sp_refiner(a, m, base, r, sh.K, sh.nctab, sh.s0, sh.s1, ukept, grp, mt, lane);
    }
}

}  // namespace

size_t sparse_smem_bytes() { return kSpSmemBytes; }

cudaError_t launch_sparse(const DecodeArgs &a, int ctas, cudaStream_t stream) {
    static int smem_set[kMaxDevicesTracked];
    const cudaError_t ea = raise_smem_limit(sparse_kernel, kSpSmemBytes, smem_set);
    if (ea != cudaSuccess) return ea;
    if (ctas > kSpMaxCtas) ctas = kSpMaxCtas;
    SpParams prm;
    memset(&prm, 0, sizeof prm);
    prm.a = a;
    const uint64_t rows = (uint64_t)a.P * a.Hkv * kPage;
    if (!make_tile_map(&prm.tm_v, const_cast<__nv_bfloat16 *>(a.v), rows))
        return cudaErrorInvalidValue;
    if (a.prof_start) cudaEventRecord(a.prof_start, stream);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(kSpThreads);
    cfg.dynamicSmemBytes = kSpSmemBytes;
    cfg.stream = stream;
    // CTAs wait for each other (stage-1 slots, the grid barrier, merge tickets): all resident
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, sparse_kernel, prm);
    if (e != cudaSuccess) return e;
    if (a.prof_stop) cudaEventRecord(a.prof_stop, stream);
    return cudaGetLastError();
}

}  // namespace ffd
