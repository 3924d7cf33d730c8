// decode.cu -- FFD decode attention on GB300: stage 1 (pseudo-max of every (sequence, KV head)
// unit) and the persistent, warp-specialised main kernel (Top-delta scan of the 2-bit thumbnails,
// refinement of the kept blocks with the int8 residual and V, online softmax, split merge).
//
// Source: "Faster Than Flash", Methodology §2 (keep token j when s_ij >= m~_i - delta; m~_i from
// the sink and local tokens only) and §3 (stage 1 pseudo-max estimation; stage 2 streams the 2-bit
// keys, computes provisional scores and filters blocks; stage 3 loads the 8-bit residuals and V of
// the selected blocks and computes exact attention, reusing the scan results). The blocks that
// hold a sink or local token are always kept.
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
#include "scan.cuh"
#include "splitkv.cuh"
#include "stage1.cuh"

namespace ffd {

// ---- main kernel: roles ---------------------------------------------------------------------
// Warpgroup 0: ring warp (0), page warp (1), thumbnail warp (2), one idle warp.
// Warpgroup 1: scan warps 4-7; scan warp mt takes rows 16mt .. 16mt+15 of every block.
// Warpgroups 2..: kRefineGroups refine groups (group grp = warps 8 + 4grp .. 11 + 4grp); kept
// block number kb goes to group kb % kRefineGroups. In a group, warp mt computes the scores of
// rows 16mt .. 16mt+15 and the output channels 32mt .. 32mt+31 (the probabilities are exchanged
// through shared memory).
constexpr int kRing = 5;             // refine ring slots (residual + V of one kept block each)
// Kept block kb takes ring slot kb % kRing and refine group kb % kRefineGroups; the blocks that a
// group's fill barrier of one slot sees are kb, kb + kFillPeriod, ... (the lcm of the two).
constexpr int kFillPeriod = kRing / gcd_c(kRing, kRefineGroups) * kRefineGroups;
constexpr int kThumbBufs = 3;        // thumbnail buffers (sub-chunks in flight ahead of the ring)
constexpr int kShatBufs = 2;         // provisional-score buffers (scan ahead of refinement)
constexpr int kDepth = 8;            // ring of per-sub-chunk decision slots
constexpr int kPageSlots = 8;        // sub-chunks whose block-table entries are resolved ahead
constexpr int kMainThreads = 256 + 128 * kRefineGroups;
constexpr int kLaunchRegs = (65536 / kMainThreads) & ~7;  // per thread at launch (one CTA/SM)
// setmaxnreg shares of the producer, scan and refine warpgroups (multiples of 8); their sum must
// fit the launch allocation, or an increase would wait forever
constexpr int kProducerRegs = kRefineGroups == 2 ? 32 : 24;
constexpr int kScanRegs = kRefineGroups == 2 ? 128 : 96;
constexpr int kRefineRegs = kRefineGroups == 2 ? 176 : 120;
static_assert(128 * kProducerRegs + 128 * kScanRegs + 128 * kRefineGroups * kRefineRegs <=
                  kMainThreads * kLaunchRegs,
              "register reallocation exceeds the launch allocation");
static_assert(kScanRegs <= kLaunchRegs && kProducerRegs <= kLaunchRegs &&
                  kRefineRegs >= kLaunchRegs, "register shares");

static_assert(kDepth > kThumbBufs + 1 && kDepth > kShatBufs + kThumbBufs, "decision ring depth");

// ring slot: the block's residual record (codes 64 x 128 B, already in the swizzled order, then
// the scales 64 x 8 B; one bulk copy), V tile (channels 0-63 of the 64 rows, then channels 64-127,
// each 64 x 128 B, swizzled; one 3-D copy)
constexpr int kSlotRScale = kResidScaleOff;
constexpr int kSlotV = 9216;
constexpr int kSlotTx = kResidRec + 16384;
constexpr int kSlotBytes = kSlotV + 16384;
static_assert(kResidRec <= kSlotV, "residual record inside the slot");
constexpr int kThumbBlock = kThumbRec;  // the block's thumbnail record: codes, scales, zeros
constexpr int kThumbBuf = kSub * kThumbBlock;
constexpr int kShatBuf = kSub * 4 * 32 * 16;  // provisional scores of one sub-chunk
constexpr int kUnitBytes = 4352;

constexpr int kOffRing = 0;
constexpr int kOffThumb = kOffRing + kRing * kSlotBytes;
constexpr int kOffShat = kOffThumb + kThumbBufs * kThumbBuf;
constexpr int kOffPx = kOffShat + kShatBufs * kShatBuf;      // [group][2][kPxBuf]
constexpr int kOffUnit = kOffPx + kRefineGroups * 2 * kPxBuf;  // [2] unit operand slots
constexpr int kOffMisc = kOffUnit + 2 * kUnitBytes;
constexpr int kMiscBytes = 2560;
constexpr int kSmemBytes = kOffMisc + kMiscBytes + 1024;  // + slack to align the base to 1 KB
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(kSlotBytes % 1024 == 0 && kSlotV % 1024 == 0, "swizzled TMA tiles need 1 KB");

// One sub-chunk as the page warp hands it to the copy warps.
struct PageSlot {
    int32_t row[kSub];   // first token row of each block's tile: (page * Hkv + h) * 64
    uint32_t bad;        // entries outside [0, P), one bit per block (row 0, never loaded)
    uint32_t forced;     // blocks holding a sink or local token (kept whatever the scan says)
    int32_t cnt;         // blocks; 0 marks the end of this CTA's schedule
    int32_t tail;        // rows of block cnt - 1 when it is the sequence's partial last block, else 0
};

struct Misc {
    uint32_t vote[kDepth];        // OR of the scan votes of sub-chunk t, in slot t % kDepth
    uint32_t final_mask[kDepth];  // kept blocks of sub-chunk t, published by the ring warp
    uint32_t aborted;
    uint32_t merge_flag[kRefineGroups];
    uint32_t over[kRefineGroups][2][4];      // [group][buffer][warp]: a score passed m + margin
    float wmax[kRefineGroups][2][4][kMaxG];  // [group][buffer][warp][head]: block row maxima
    float lsum[kRefineGroups][4][kMaxG];     // [group][warp][head]: softmax sums at unit end
    PageSlot ps[kPageSlots];      // sub-chunk t in ps[t % kPageSlots]
    uint64_t pages_full[kPageSlots];
    uint64_t pages_empty[kPageSlots];
    uint64_t thumb_full[kThumbBufs];
    uint64_t decision[kDepth];    // the 4 scan warps voted on sub-chunk t
    uint64_t ring_seen[kDepth];   // the ring warp published the kept blocks of sub-chunk t
    uint64_t shat_free[kShatBufs];
    uint64_t ring_full[kRefineGroups][kRing];  // [group of the block][slot]
    uint64_t ring_empty[kRing];
    uint64_t unit_ready[2];
    uint64_t unit_free[2];
    uint64_t tail_full;  // the ring warp's own copies of a partial last block
    uint32_t tails;      // partial last blocks the ring warp has copied so far
};
static_assert(sizeof(Misc) <= kMiscBytes, "misc region");

// Query operands of one (sequence, KV head) unit, laid out so that a lane loads its 16
// B-fragment registers with four conflict-free 128-bit loads.
struct UnitOps {
    uint4 bt[4][32];   // thumbnail B fragments: [bt0[0..3], bt0[4..7], bt1[0..3], bt1[4..7]][lane]
    uint4 br[4][32];   // residual B fragments, same arrangement
    float4 qs[kMaxG];  // per-group query sums, [head].{group 0..3}
    float thr[kMaxG];  // m~ - delta (+inf for heads >= G)
    float mt[kMaxG];   // m~
    int n;             // sequence length
};
static_assert(sizeof(UnitOps) <= kUnitBytes, "unit operand slot");

struct MainParams {
    CUtensorMap tm_v;
    DecodeArgs a;
};

struct Smem {
    uint8_t *ring, *thumb, *shat, *px;
    UnitOps *unit;
    Misc *misc;
};

__device__ __forceinline__ void load_frags(const uint4 (&src)[4][32], int lane, uint32_t (&f0)[8],
                                           uint32_t (&f1)[8]) {
    const uint4 p0 = src[0][lane], p1 = src[1][lane], p2 = src[2][lane], p3 = src[3][lane];
    f0[0] = p0.x; f0[1] = p0.y; f0[2] = p0.z; f0[3] = p0.w;
    f0[4] = p1.x; f0[5] = p1.y; f0[6] = p1.z; f0[7] = p1.w;
    f1[0] = p2.x; f1[1] = p2.y; f1[2] = p2.z; f1[3] = p2.w;
    f1[4] = p3.x; f1[5] = p3.y; f1[6] = p3.z; f1[7] = p3.w;
}

__device__ __forceinline__ bool tile_passes(float4 e, bool v0, bool v1, float thr0, float thr1) {
    return (v0 && (e.x >= thr0 || e.y >= thr1)) || (v1 && (e.z >= thr0 || e.w >= thr1));
}


// ------------------------------------------------------------------------------------------
// Main kernel: waits and the copy warps.
// ------------------------------------------------------------------------------------------
// Page warp: walks the CTA's schedule ahead of the copy warps and resolves the block-table entries
// of every sub-chunk (one lane per block) into the page ring, so that no global-load latency sits
// on a TMA issue path; a slot with cnt == 0 ends the schedule. Entries outside [0, P) are flagged
// (FFD_ERRBIT_BOUNDS) and their blocks are never loaded.
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
        const int n = len_of(a, s.b);
        const ForcedBlocks fb(n, a.S, a.L);
        // with a caller-given mask (comparison selectors) the mask alone decides: the scan's
        // thresholds are +inf and the given blocks take the place of the forced ones
        const bool given = a.keep_in && lane < s.cnt &&
                           a.keep_in[((size_t)s.b * a.Hkv + s.h) * a.max_blocks + s.j0 + lane];
        const uint32_t forced = __ballot_sync(
            0xffffffffu, a.keep_in ? given : (lane < s.cnt && fb.forced(s.j0 + lane)));
        // every row in the ring is in range (a bad entry reads as page 0 and is never loaded)
        if (lane < s.cnt) P.row[lane] = ((bad ? 0 : page) * a.Hkv + s.h) * kPage;
        if (lane == 0) {
            P.bad = badmask;
            P.forced = forced;
            P.cnt = s.cnt;
            P.tail = s.j0 + s.cnt == s.nblk ? (n & (kPage - 1)) : 0;
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

// Thumbnail warp: the thumbnail records of sub-chunk t go to buffer t % kThumbBufs
// once the ring warp has published sub-chunk t - kThumbBufs (so the scan warps are done with that
// buffer, and no decision runs more than kThumbBufs sub-chunks ahead of the ring warp); lane k
// issues block k's copy.
__device__ __forceinline__ void thumb_issuer(const DecodeArgs &a, const Smem &S, int lane) {
    Misc *m = S.misc;
    int t = 0;
    for (;; t++) {
        const int buf = t % kThumbBufs;
        if (t >= kThumbBufs) {
            const int tp = t - kThumbBufs;
            wait_bar(a, m, &m->ring_seen[tp % kDepth], (tp / kDepth) & 1);
        }
        const PageSlot &P = page_slot(a, m, t);
        const int cnt = P.cnt;
        if (cnt == 0 || aborted(m)) break;
        const uint32_t bad = P.bad;
        if (lane == 0)
            mbar_arrive_expect_tx(&m->thumb_full[buf],
                                  (uint32_t)((cnt - __popc(bad)) * kThumbBlock));
        __syncwarp();
        if (lane < cnt && !((bad >> lane) & 1u)) {
            const size_t tile = (size_t)(P.row[lane] / kPage);
            uint8_t *d = S.thumb + buf * kThumbBuf + lane * kThumbBlock;
            tma_load_1d(d, a.thumb + tile * kThumbRec, kThumbRec, &m->thumb_full[buf]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&m->pages_empty[t % kPageSlots]);
    }
    // leave no copy in flight: wait for the last fill of every buffer (t fills were armed)
    if (lane == 0)
        for (int j = 0; j < kThumbBufs && j < t; j++)
            drain_bar(a, &m->thumb_full[j], ((t - 1 - j) / kThumbBufs) & 1);
}

// Ring warp: publishes the kept blocks of sub-chunk t (scan votes, plus the forced blocks, less
// the never-loaded ones), then issues the residual record and the V tile of each kept block into
// the next ring slot as it frees up; lanes 0 and 1 issue the two copies side by side. A sequence's
// partial last block is copied under the warp's own barrier instead: the warp waits for it, zeroes
// the V rows past the sequence (they hold whatever the cache holds, and a zero probability times a
// NaN would poison P.V) and then completes the slot's fill barrier itself.
__device__ __forceinline__ void ring_issuer(const MainParams &prm, const Smem &S, int lane) {
    const DecodeArgs &a = prm.a;
    Misc *m = S.misc;
    if (lane == 0) prefetch_tensormap(&prm.tm_v);
    int kb = 0;
    for (int t = 0;; t++) {
        const PageSlot &P = page_slot(a, m, t);
        const int cnt = P.cnt;
        if (cnt == 0 || aborted(m)) break;
        const int ds = t % kDepth;
        wait_bar(a, m, &m->decision[ds], (t / kDepth) & 1);
        if (aborted(m)) break;  // a wait ran out: nothing more is issued
        const uint32_t mask = (*reinterpret_cast<volatile uint32_t *>(&m->vote[ds]) | P.forced) &
                              ~P.bad & ((1u << cnt) - 1u);
        __syncwarp();
        if (lane == 0) {
            m->final_mask[ds] = mask;
            // the scan of sub-chunk t + kThumbBufs votes into this slot only after its
            // thumbnails, which wait for this arrival; the slot's last reader was this warp
            m->vote[(t + kThumbBufs) % kDepth] = 0;
            mbar_arrive(&m->ring_seen[ds]);
        }
        const int tail_k = P.tail ? cnt - 1 : -1;  // the partial last block, if any
        for (int k = 0; k < cnt; k++) {
            if (!(mask & (1u << k))) continue;
            const int slot = kb % kRing, round = kb / kRing;
            kb++;
            if (round > 0) wait_bar(a, m, &m->ring_empty[slot], (round - 1) & 1);
            if (aborted(m)) {  // the slot may still be filling: arm nothing more
                kb--;
                break;
            }
            const int row = P.row[k];
            uint8_t *d = S.ring + slot * kSlotBytes;
            uint64_t *bar = &m->ring_full[(kb - 1) % kRefineGroups][slot];  // kb advanced above
            const bool tail = k == tail_k;
            uint64_t *cb = tail ? &m->tail_full : bar;
            if (lane == 0) mbar_arrive_expect_tx(cb, kSlotTx);
            __syncwarp();
            if (lane == 0) tma_load_1d(d, a.resid + (size_t)(row / kPage) * kResidRec, kResidRec, cb);
            else if (lane == 1) tma_load_3d(d + kSlotV, &prm.tm_v, 0, row, 0, cb);
            if (tail) {  // warp-uniform; once per sequence
                const int rows = P.tail;
                const uint32_t nt = *reinterpret_cast<volatile uint32_t *>(&m->tails);
                drain_bar(a, &m->tail_full, nt & 1);  // bounded, and never left in flight
                for (int c = lane; c < (kPage - rows) * 16; c += 32) {  // both 64 x 128 B halves
                    const int r = rows + (c >> 4), half = (c >> 3) & 1;
                    *reinterpret_cast<uint4 *>(d + kSlotV + half * 8192 + r * 128 + (c & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async();  // before the slot's next bulk copy
                __syncwarp();
                if (lane == 0) {
                    m->tails = nt + 1;
                    mbar_arrive(bar);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&m->pages_empty[t % kPageSlots]);
    }
    // leave no copy in flight: wait for the last fill of every ring slot (block kb - 1 - i went to
    // slot (kb - 1 - i) % kRing, the ((kb - 1 - i) / kFillPeriod)-th fill of its group's barrier)
    if (lane == 0)
        for (int i = 0; i < kRing && i < kb; i++) {
            const int last = kb - 1 - i;
            drain_bar(a, &m->ring_full[last % kRefineGroups][last % kRing],
                      (last / kFillPeriod) & 1);
        }
}

// ------------------------------------------------------------------------------------------
// Scan warps (stage 2).
// ------------------------------------------------------------------------------------------
// Scan warp 0 computes the unit's query operands and thresholds into a unit slot.
__device__ __forceinline__ void fill_unit(const DecodeArgs &a, Misc *m, UnitOps &U, int b, int h,
                                          int lane) {
    const int g = lane >> 2, tig = lane & 3;
    ThumbOps T;
    ResidOps Rr;
    load_thumb_ops(a, b, h, lane, T);
    load_resid_ops(a, b, h, lane, Rr);
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
        float mx = -INFINITY;
        const int u = b * a.Hkv + h;
        wait_count(a, m, slot_counter(a, u), a.nf);  // every stage-1 slot of the unit is in
        for (int sl = 0; sl < a.nf; sl++)
            mx = fmaxf(mx, __ldcg(a.ws_m1 + ((size_t)u * a.nf + sl) * kMaxG + lane));
        U.mt[lane] = mx;
        U.thr[lane] = lane < a.G && !a.keep_in ? mx - a.delta : INFINITY;
    }
    if (lane == 0) U.n = len_of(a, b);
}

// Scan warp mt, every sub-chunk: provisional scores of rows 16mt .. 16mt+15 of each block into
// the score buffer, and a vote for every block where one of those rows passes m~ - delta (an OR
// into the sub-chunk's vote word, then one arrival on its decision barrier). Blocks k and k+3 are
// scanned side by side (two independent dependency chains); tiles past the sub-chunk's end are
// computed from stale buffer contents (reads stay inside the buffer) and ignored.
__device__ __forceinline__ void scanner(const DecodeArgs &a, const Smem &S, int cta, int ncta,
                                        int mt, int lane) {
    Misc *m = S.misc;
    const int g = lane >> 2, tig = lane & 3;
    const uint32_t m0 = 0x00030003u << (2 * tig);
    const int r0 = 16 * mt + g, r1 = r0 + 8;
    const float sm = a.sm_scale;
    Sched sch;
    sch.init(a, cta, ncta);
    Sub s;
    ThumbOps Q;  // the unit's thumbnail B fragments, query sums and thresholds, in registers
    float thr0 = 0.0f, thr1 = 0.0f;
    int n = 0;
    int ui = -1;
    for (int t = 0; sch.next(a, s); t++) {
        if (s.first) {
            ui++;
            const int us = ui & 1;
            if (ui >= 2) wait_bar(a, m, &m->unit_free[us], ((ui >> 1) - 1) & 1);
            if (mt == 0) fill_unit(a, m, S.unit[us], s.b, s.h, lane);
            named_barrier_sync(1, 128);
            if (mt == 0 && lane == 0) mbar_arrive(&m->unit_ready[us]);
            const UnitOps &U = S.unit[us];
            load_frags(U.bt, lane, Q.bt0, Q.bt1);
            const float4 q0 = U.qs[2 * tig], q1 = U.qs[2 * tig + 1];
            Q.qs[0][0] = q0.x; Q.qs[0][1] = q0.y; Q.qs[0][2] = q0.z; Q.qs[0][3] = q0.w;
            Q.qs[1][0] = q1.x; Q.qs[1][1] = q1.y; Q.qs[1][2] = q1.z; Q.qs[1][3] = q1.w;
            thr0 = U.thr[2 * tig];
            thr1 = U.thr[2 * tig + 1];
            n = U.n;
        }
        const int tb = t % kThumbBufs, sb = t % kShatBufs;
        wait_bar(a, m, &m->thumb_full[tb], (t / kThumbBufs) & 1);
        if (t >= kShatBufs) wait_bar(a, m, &m->shat_free[sb], ((t / kShatBufs) - 1) & 1);
        const uint8_t *tbuf = S.thumb + tb * kThumbBuf;
        float4 *shat = reinterpret_cast<float4 *>(S.shat + sb * kShatBuf);
        uint32_t votes = 0;
        // Every tile pair is computed and used unconditionally (a partial sub-chunk scores stale
        // buffer contents past its end, masked out below): a pair whose second tile is consumed
        // only under a condition gets that tile's computation moved under the condition, and the
        // two tiles then no longer overlap.
#pragma unroll 1
        for (int kA = 0; kA < kSub / 2; kA++) {
            const int kB = kA + kSub / 2;
            const float4 eA = scan_tile(tbuf + kA * kThumbBlock, r0, r1, m0, Q, sm);
            const float4 eB = scan_tile(tbuf + kB * kThumbBlock, r0, r1, m0, Q, sm);
            const bool pA = tile_passes(eA, true, true, thr0, thr1);
            const bool pB = tile_passes(eB, true, true, thr0, thr1);
            if (__any_sync(0xffffffffu, pA)) votes |= 1u << kA;
            if (__any_sync(0xffffffffu, pB)) votes |= 1u << kB;
            shat[(kA * 4 + mt) * 32 + lane] = eA;
            shat[(kB * 4 + mt) * 32 + lane] = eB;
        }
        votes &= (1u << s.cnt) - 1u;
        // a sequence's partial last block: rows past the sequence hold arbitrary bits and must not
        // vote, so its vote is taken again over the rows inside the sequence (warp-uniform, once
        // per sequence and KV head)
        const int tail_rows = n & (kPage - 1);
        if (s.j0 + s.cnt == s.nblk && tail_rows) {
            const int k = s.cnt - 1;
            const float4 e = shat[(k * 4 + mt) * 32 + lane];
            const bool p = tile_passes(e, r0 < tail_rows, r1 < tail_rows, thr0, thr1);
            votes = (votes & ~(1u << k)) | (__any_sync(0xffffffffu, p) ? 1u << k : 0u);
        }
        __syncwarp();
        if (lane == 0) {
            if (votes) atomicOr(&m->vote[t % kDepth], votes);
            mbar_arrive(&m->decision[t % kDepth]);  // releases the vote and the warp's scores
        }
    }
}

// ------------------------------------------------------------------------------------------
// Refine groups (stage 3).
// ------------------------------------------------------------------------------------------
// Fresh state for a unit: the reference starts at its pseudo-max m~ (a large negative finite
// value when m~ is -inf, so that the first finite score raises it through the rescale path).
__device__ __forceinline__ void reset_refine(RefineState &R, const UnitOps &U, int lane) {
    const float m0 = U.mt[2 * (lane & 3)], m1 = U.mt[2 * (lane & 3) + 1];
    R.m0 = m0 == -INFINITY ? kNoReference : m0;
    R.m1 = m1 == -INFINITY ? kNoReference : m1;
    R.nl0 = -R.m0 * kLog2e;
    R.nl1 = -R.m1 * kLog2e;
    R.l0 = R.l1 = 0.0f;
#pragma unroll
    for (int i = 0; i < 2; i++) R.o[i][0] = R.o[i][1] = R.o[i][2] = R.o[i][3] = 0.0f;
}


// One kept block held in a ring slot, by the 4 warps of refine group grp: warp mt's exact scores of
// rows 16mt .. 16mt+15 (provisional score from the scan + residual correction), then the group's
// softmax and P.V update.
__device__ __forceinline__ void refine_block(const DecodeArgs &a, const Smem &S, const uint8_t *slot,
                                             const ResidOps &Q, int n, const float4 est, int blk,
                                             RefineState &R, int grp, int mt, int pb, int lane) {
    const int g = lane >> 2, tig = lane & 3;
    // ---- scores of rows r0, r1 (heads 2tig, 2tig+1)
    const int r0 = 16 * mt + g, r1 = r0 + 8;
    uint2 x0[4], x1[4];
#pragma unroll
    for (int gg = 0; gg < 4; gg++) {
        const int o = 32 * gg + 8 * tig;
        x0[gg] = *reinterpret_cast<const uint2 *>(slot + resid_offset(r0, o));
        x1[gg] = *reinterpret_cast<const uint2 *>(slot + resid_offset(r1, o));
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

    softmax_pv(S.misc, S.px + (grp * 2 + pb) * kPxBuf, slot + kSlotV, s00, s01, s10, s11, R, grp,
               mt, pb, lane);
}

// End of this CTA's segment of a unit, refine group grp: its record, ticket and share of the merge.
__device__ __forceinline__ void unit_end(const DecodeArgs &a, const Smem &S, const Sub &s,
                                         const RefineState &R, int cta, int ncta, int64_t T,
                                         int grp, int mt, int lane) {
    const int u = s.b * a.Hkv + s.h;
    write_record(a, S.misc, R, unit_record(a, u, cta, grp), grp, mt, lane);
    finish_unit(a, S.misc, s, cta, ncta, T, grp, mt, lane);
}

// Wait until the copies of kept block kb have landed in its ring slot. The refine groups share the
// ring (consecutive occupants of a slot may belong to different groups) and may drift apart; each
// group therefore has its own fill barrier per slot, whose consecutive phases are the group's own
// blocks kb, kb + kFillPeriod, ..., consumed in order: the parity wait is exact however far the
// other groups lag.
__device__ __forceinline__ void wait_fill(const DecodeArgs &a, Misc *m, int slot, int kb) {
    wait_bar(a, m, &m->ring_full[kb % kRefineGroups][slot], (kb / kFillPeriod) & 1);
}

// Refine warp mt of group grp: walks the schedule, takes the kept blocks kb % kRefineGroups == grp.
__device__ __forceinline__ void refiner(const DecodeArgs &a, const Smem &S, int cta, int ncta,
                                        int grp, int mt, int lane) {
    Misc *m = S.misc;
    Sched sch;
    sch.init(a, cta, ncta);
    Sub s;
    RefineState R;
    ResidOps Q;  // the unit's residual B fragments and query sums, kept in registers
    int n = 0;
    int ui = -1, kb = 0, pb = 0;
    for (int t = 0; sch.next(a, s); t++) {
        if (s.first) {
            ui++;
            wait_bar(a, m, &m->unit_ready[ui & 1], (ui >> 1) & 1);
            const UnitOps &U = S.unit[ui & 1];
            reset_refine(R, U, lane);
            load_frags(U.br, lane, Q.br0, Q.br1);
            const int tig = lane & 3;
            const float4 q0 = U.qs[2 * tig], q1 = U.qs[2 * tig + 1];
            Q.qs[0][0] = q0.x; Q.qs[0][1] = q0.y; Q.qs[0][2] = q0.z; Q.qs[0][3] = q0.w;
            Q.qs[1][0] = q1.x; Q.qs[1][1] = q1.y; Q.qs[1][2] = q1.z; Q.qs[1][3] = q1.w;
            n = U.n;
        }
        const int ds = t % kDepth;
        wait_bar(a, m, &m->ring_seen[ds], (t / kDepth) & 1);
        // the kept blocks decide the group's barriers, so the group leaves together when a wait
        // has run out in this CTA (the mask may then never have been published)
        if (named_barrier_or(2 + grp, 128, aborted(m))) break;
        const uint32_t mask = *reinterpret_cast<volatile uint32_t *>(&m->final_mask[ds]);
        if (grp == 0 && mt == 0 && a.keep_mask && lane < s.cnt)
            a.keep_mask[((size_t)s.b * a.Hkv + s.h) * a.max_blocks + s.j0 + lane] =
                (mask >> lane) & 1u;
        const float4 *shat = reinterpret_cast<const float4 *>(S.shat + (t % kShatBufs) * kShatBuf);
        for (int k = 0; k < s.cnt; k++) {
            if (!((mask >> k) & 1u)) continue;
            if (kb % kRefineGroups == grp) {
                const int slot = kb % kRing;
                wait_fill(a, m, slot, kb);
                refine_block(a, S, S.ring + slot * kSlotBytes, Q, n, shat[(k * 4 + mt) * 32 + lane],
                             s.j0 + k, R, grp, mt, pb, lane);
                pb ^= 1;
                __syncwarp();
                if (lane == 0) mbar_arrive(&m->ring_empty[slot]);
            }
            kb++;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&m->shat_free[t % kShatBufs]);
        if (s.last) {
            unit_end(a, S, s, R, cta, ncta, sch.T, grp, mt, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(&m->unit_free[ui & 1]);
        }
    }
}

// ------------------------------------------------------------------------------------------
// Main kernel: persistent, one CTA per SM (at most one per block, so every range is non-empty).
// ------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kMainThreads, 1)
    main_kernel(const __grid_constant__ MainParams prm) {
    const DecodeArgs &a = prm.a;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = align_shared<1024>(smem_raw);
    Smem S;
    S.ring = base + kOffRing;
    S.thumb = base + kOffThumb;
    S.shat = base + kOffShat;
    S.px = base + kOffPx;
    S.unit = reinterpret_cast<UnitOps *>(base + kOffUnit);
    S.misc = reinterpret_cast<Misc *>(base + kOffMisc);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // CTAs 0 .. ncta-1 walk the blocks; every CTA of the grid takes part in stage 1 (which also
    // writes the results of empty sequences, so it runs when no CTA walks anything)
    const int64_t T = total_blocks(a);
    const int ncta = (int)(T < (int64_t)gridDim.x ? T : (int64_t)gridDim.x);
    const int cta = blockIdx.x;
    const bool walker = cta < ncta;

    if (threadIdx.x == 0) {
        Misc *m = S.misc;
        m->aborted = 0;
        for (int i = 0; i < kDepth; i++) {
            m->vote[i] = 0;
            mbar_init(&m->decision[i], 4);   // the scan warps
            mbar_init(&m->ring_seen[i], 1);  // the ring warp
        }
        for (int i = 0; i < kPageSlots; i++) {
            mbar_init(&m->pages_full[i], 1);
            mbar_init(&m->pages_empty[i], 2);  // thumbnail warp and ring warp
        }
        for (int i = 0; i < kThumbBufs; i++) mbar_init(&m->thumb_full[i], 1);
        for (int i = 0; i < kShatBufs; i++) mbar_init(&m->shat_free[i], 4 * kRefineGroups);
        for (int i = 0; i < kRing; i++) {
            for (int g = 0; g < kRefineGroups; g++) mbar_init(&m->ring_full[g][i], 1);
            mbar_init(&m->ring_empty[i], 4);  // the refine group that took the block
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(&m->unit_ready[i], 1);  // scan warp 0
            mbar_init(&m->unit_free[i], 4 * kRefineGroups);  // refine warps
        }
        mbar_init(&m->tail_full, 1);  // the ring warp
        m->tails = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (warp < 4) {
        regs_decrease<kProducerRegs>();
        if (!walker) return;
        if (warp == 0) ring_issuer(prm, S, lane);
        else if (warp == 1) pager(a, S, cta, ncta, lane);
        else if (warp == 2) thumb_issuer(a, S, lane);
    } else if (warp < 8) {
        if (kScanRegs < kLaunchRegs) regs_decrease<kScanRegs>();
        if (walker) scanner(a, S, cta, ncta, warp - 4, lane);
    } else {
        regs_increase<kRefineRegs>();
        pseudo_max_slots<kRefineGroups>(a, S.misc, cta, gridDim.x, (warp - 8) >> 2, warp & 3, lane);
        if (walker) refiner(a, S, cta, ncta, (warp - 8) >> 2, warp & 3, lane);
    }
}

// ------------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------------
cudaError_t launch_decode(const DecodeArgs &a, int main_ctas, cudaStream_t stream) {
    static int smem_set[kMaxDevicesTracked];
    const cudaError_t ea = raise_smem_limit(main_kernel, kSmemBytes, smem_set);
    if (ea != cudaSuccess) return ea;
    MainParams prm;
    memset(&prm, 0, sizeof prm);
    prm.a = a;
    const uint64_t rows = (uint64_t)a.P * a.Hkv * kPage;
    if (!make_tile_map(&prm.tm_v, const_cast<__nv_bfloat16 *>(a.v), rows))
        return cudaErrorInvalidValue;

    if (a.prof_start) cudaEventRecord(a.prof_start, stream);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(main_ctas);
    cfg.blockDim = dim3(kMainThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    // scan warps wait for stage-1 slots computed by other CTAs: all CTAs must be resident
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, main_kernel, prm);
    if (e != cudaSuccess) return e;
    if (a.prof_stop) cudaEventRecord(a.prof_stop, stream);
    return cudaGetLastError();
}

}  // namespace ffd
