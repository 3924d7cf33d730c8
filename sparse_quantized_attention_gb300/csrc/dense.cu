// dense.cu -- dense bf16 flash-decode attention, the in-library comparison for FFD.
//
// Source: the pages compare FFD with FlashAttention-2 decoding ("Faster Than Flash", Main results:
// kernel speedup and end-to-end throughput). This kernel computes plain softmax attention over
// every cached token with the original bf16 keys. It is the FFD step without stages 1 and 2: a
// persistent CTA per SM walks an equal share of all blocks (splitkv.cuh schedule), a copy warp
// streams each block's K and V tiles (two 3-D TMA copies, 32 KB) into a 6-slot ring, and two
// groups of four warps take alternate blocks: scores q.K on the tensor cores, then the same
// online-softmax and P.V update, records and by-head merge as the FFD path.
#include "splitkv.cuh"

namespace ffd {
namespace {

constexpr int kDRing = 6;          // ring slots: K tile, then V tile, of one block
constexpr int kDPageSlots = 8;     // sub-chunks whose block-table entries are resolved ahead
constexpr int kDThreads = 128 + 128 * kRefineGroups;  // copy warpgroup + refine groups
constexpr int kDFillPeriod = kDRing / gcd_c(kDRing, kRefineGroups) * kRefineGroups;
constexpr int kDSlotK = 0;
constexpr int kDSlotV = 16384;
constexpr int kDSlotBytes = 32768;
constexpr int kDOffPx = kDRing * kDSlotBytes;                   // [group][2][kPxBuf]
constexpr int kDOffMisc = kDOffPx + kRefineGroups * 2 * kPxBuf;
constexpr int kDMiscBytes = 2048;
constexpr int kDSmemBytes = kDOffMisc + kDMiscBytes + 1024;     // + slack to align to 1 KB
static_assert(kDSmemBytes <= 232448, "shared memory per CTA");

// One sub-chunk's tiles as the page warp hands them to the copy warp.
struct DensePages {
    int32_t row[kSub];  // first row of each block's tile: (page * Hkv + h) * 64
    uint32_t bad;       // entries outside [0, P), one bit per block (never loaded)
    int32_t cnt;        // blocks; 0 ends this CTA's schedule
    int32_t tail;       // rows of block cnt - 1 when it is the sequence's partial last block, else 0
};

struct DenseMisc {
    uint32_t aborted;
    uint32_t merge_flag[kRefineGroups];
    uint32_t slot_bad[kDRing];               // the block in ring slot s was not loaded
    uint32_t over[kRefineGroups][2][4];      // as in the FFD kernel (softmax_pv)
    float wmax[kRefineGroups][2][4][kMaxG];
    float lsum[kRefineGroups][4][kMaxG];
    DensePages ps[kDPageSlots];
    uint64_t pages_full[kDPageSlots];
    uint64_t pages_empty[kDPageSlots];
    uint64_t full[kRefineGroups][kDRing];    // [group of the block][slot]
    uint64_t empty[kDRing];
    uint64_t tail_full;  // the copy warp's own copies of a partial last block
    uint32_t tails;      // partial last blocks the copy warp has copied so far
};
static_assert(sizeof(DenseMisc) <= kDMiscBytes, "control block");

struct DenseParams {
    CUtensorMap tm_k, tm_v;
    DecodeArgs a;
};

// Page warp: resolves the block-table entries of every sub-chunk of the CTA's schedule (one lane
// per block) into the page ring; entries outside [0, P) raise FFD_ERRBIT_BOUNDS and are skipped.
__device__ __forceinline__ void dense_pager(const DecodeArgs &a, DenseMisc *m, int cta, int ncta,
                                            int lane) {
    Sched sch;
    sch.init(a, cta, ncta);
    Sub s;
    for (int t = 0;; t++) {
        const bool more = sch.next(a, s);
        const int ps = t % kDPageSlots;
        if (t >= kDPageSlots) wait_bar(a, m, &m->pages_empty[ps], ((t / kDPageSlots) - 1) & 1);
        if (aborted(m)) return;
        DensePages &P = m->ps[ps];
        bool bad = false;
        if (more && lane < s.cnt) {
            const int page = a.block_table[(size_t)s.b * a.max_blocks + s.j0 + lane];
            bad = page < 0 || page >= a.P;
            if (bad) raise_error(a.err, FFD_ERRBIT_BOUNDS);
            P.row[lane] = bad ? 0 : (page * a.Hkv + s.h) * kPage;
        }
        const uint32_t badm = __ballot_sync(0xffffffffu, bad);
        if (lane == 0) {
            P.bad = badm;
            P.cnt = more ? s.cnt : 0;
            P.tail = more && s.j0 + s.cnt == s.nblk ? (len_of(a, s.b) & (kPage - 1)) : 0;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&m->pages_full[ps]);
        if (!more) return;
    }
}

// Copy warp: block kb goes to ring slot kb % kDRing as soon as the slot is free; lanes 0 and 1
// issue the K and V copies side by side. Each refine group has its own fill barrier per slot
// (consecutive phases = its blocks kb, kb + kDFillPeriod, ...). A sequence's partial last block
// is copied under the warp's own barrier: the warp waits for it, zeroes the V rows past the
// sequence (a zero probability times a NaN there would poison P.V) and then completes the slot's
// fill barrier itself.
__device__ __forceinline__ void dense_ring(const DenseParams &prm, DenseMisc *m, uint8_t *ring,
                                           int lane) {
    const DecodeArgs &a = prm.a;
    if (lane == 0) {
        prefetch_tensormap(&prm.tm_k);
        prefetch_tensormap(&prm.tm_v);
    }
    int kb = 0;
    for (int t = 0;; t++) {
        const int ps = t % kDPageSlots;
        wait_bar(a, m, &m->pages_full[ps], (t / kDPageSlots) & 1);
        const DensePages &P = m->ps[ps];
        const int cnt = P.cnt;
        if (cnt == 0 || aborted(m)) break;
        const int tail_k = P.tail ? cnt - 1 : -1;  // the partial last block, if any
        for (int k = 0; k < cnt; k++, kb++) {
            const int slot = kb % kDRing, round = kb / kDRing;
            if (round > 0) wait_bar(a, m, &m->empty[slot], (round - 1) & 1);
            if (aborted(m)) break;  // a wait ran out: the slot may still be filling, arm nothing
            uint64_t *bar = &m->full[kb % kRefineGroups][slot];
            const bool bad = (P.bad >> k) & 1u;
            uint8_t *d = ring + slot * kDSlotBytes;
            const bool tail = !bad && k == tail_k;
            uint64_t *cb = tail ? &m->tail_full : bar;
            if (lane == 0) {
                m->slot_bad[slot] = bad;
                if (bad) mbar_arrive(bar);
                else mbar_arrive_expect_tx(cb, kDSlotBytes);
            }
            __syncwarp();
            if (!bad) {
                if (lane == 0) tma_load_3d(d + kDSlotK, &prm.tm_k, 0, P.row[k], 0, cb);
                else if (lane == 1) tma_load_3d(d + kDSlotV, &prm.tm_v, 0, P.row[k], 0, cb);
            }
            if (tail) {  // warp-uniform; once per sequence
                const int rows = P.tail;
                const uint32_t nt = *reinterpret_cast<volatile uint32_t *>(&m->tails);
                drain_bar(a, &m->tail_full, nt & 1);  // bounded, and never left in flight
                for (int c = lane; c < (kPage - rows) * 16; c += 32) {  // both 64 x 128 B halves
                    const int r = rows + (c >> 4), half = (c >> 3) & 1;
                    *reinterpret_cast<uint4 *>(d + kDSlotV + half * 8192 + r * 128 + (c & 7) * 16) =
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
        if (lane == 0) mbar_arrive(&m->pages_empty[ps]);
    }
    // leave no copy in flight: wait for the last fill of every ring slot
    if (lane == 0)
        for (int i = 0; i < kDRing && i < kb; i++) {
            const int last = kb - 1 - i;
            drain_bar(a, &m->full[last % kRefineGroups][last % kDRing], (last / kDFillPeriod) & 1);
        }
}

// Refine warp mt of group grp: blocks kb % kRefineGroups == grp of the CTA's schedule. Scores of
// rows r0 = 16mt + g, r1 = r0 + 8 for heads 2tig, 2tig+1: K rows by ldmatrix from the swizzled
// tile (A operand), q of head g as bf16 pairs (B operand, exact), fp32 accumulation over the 8
// k-steps of 16 channels.
__device__ __forceinline__ void dense_refiner(const DecodeArgs &a, DenseMisc *m, uint8_t *ring,
                                              uint8_t *px, int cta, int ncta, int grp, int mt,
                                              int lane) {
    const int g = lane >> 2, tig = lane & 3;
    const int mi = lane >> 3, jr = lane & 7;
    const int tok = 16 * mt + ((mi & 1) << 3) + jr;  // the row this lane addresses for ldmatrix
    Sched sch;
    sch.init(a, cta, ncta);
    Sub s;
    RefineState R;
    uint32_t qb0[8], qb1[8];
    int n = 0, kb = 0, pb = 0;
    while (sch.next(a, s)) {
        if (s.first) {
            const bool hv = g < a.G;
            const uint32_t *qw = reinterpret_cast<const uint32_t *>(
                a.q + ((size_t)s.b * a.Hq + s.h * a.G + (hv ? g : 0)) * kD);
#pragma unroll
            for (int kc = 0; kc < 8; kc++) {
                qb0[kc] = hv ? qw[8 * kc + tig] : 0u;      // channels 16kc + 2tig, +1
                qb1[kc] = hv ? qw[8 * kc + 4 + tig] : 0u;  // channels 16kc + 8 + 2tig, +1
            }
            R.m0 = R.m1 = kNoReference;  // the first block raises it through the rescale path
            R.nl0 = R.nl1 = -kNoReference * kLog2e;
            R.l0 = R.l1 = 0.0f;
#pragma unroll
            for (int i = 0; i < 2; i++) R.o[i][0] = R.o[i][1] = R.o[i][2] = R.o[i][3] = 0.0f;
            n = len_of(a, s.b);
        }
        for (int k = 0; k < s.cnt; k++, kb++) {
            if (kb % kRefineGroups != grp) continue;
            const int slot = kb % kDRing;
            wait_bar(a, m, &m->full[grp][slot], (kb / kDFillPeriod) & 1);
            // the slot's state decides the group's barriers, so the group leaves together when a
            // wait has run out in this CTA
            if (named_barrier_or(2 + grp, 128, aborted(m))) return;
            const uint8_t *d = ring + slot * kDSlotBytes;
            if (!*reinterpret_cast<volatile uint32_t *>(&m->slot_bad[slot])) {  // group-uniform
                const uint32_t kbase = smem_u32(d + kDSlotK);
                float D[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int kc = 0; kc < 8; kc++) {
                    const int c = 2 * kc + (mi >> 1);  // 16-byte chunk of the 256-byte row
                    uint32_t a0, a1, a2, a3;
                    ldmatrix_x4(a0, a1, a2, a3,
                                kbase + (c >> 3) * 8192 + tok * 128 + (((c & 7) ^ jr) << 4));
                    mma_bf16(D, a0, a1, a2, a3, qb0[kc], qb1[kc]);
                }
                const float sm = a.sm_scale;
                const int t0 = (s.j0 + k) * kPage + 16 * mt + g;
                const bool v0 = t0 < n, v1 = t0 + 8 < n;
                softmax_pv(m, px + (grp * 2 + pb) * kPxBuf, d + kDSlotV, v0 ? D[0] * sm : -INFINITY,
                           v0 ? D[1] * sm : -INFINITY, v1 ? D[2] * sm : -INFINITY,
                           v1 ? D[3] * sm : -INFINITY, R, grp, mt, pb, lane);
                pb ^= 1;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&m->empty[slot]);
        }
        if (s.last) {
            const int u = s.b * a.Hkv + s.h;
            write_record(a, m, R, unit_record(a, u, cta, grp), grp, mt, lane);
            finish_unit(a, m, s, cta, ncta, sch.T, grp, mt, lane);
        }
    }
}

// Persistent, one CTA per SM; CTAs 0 .. ncta-1 walk the blocks. Warp 2 of every CTA writes the
// zero output of empty sequences (no CTA walks them) and flags lengths past the block table.
__global__ void __launch_bounds__(kDThreads, 1) dense_kernel(const __grid_constant__ DenseParams prm) {
    const DecodeArgs &a = prm.a;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = align_shared<1024>(smem_raw);
    uint8_t *ring = base;
    uint8_t *px = base + kDOffPx;
    DenseMisc *m = reinterpret_cast<DenseMisc *>(base + kDOffMisc);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t T = total_blocks(a);
    const int ncta = (int)(T < (int64_t)gridDim.x ? T : (int64_t)gridDim.x);
    const int cta = blockIdx.x;
    const bool walker = cta < ncta;
    if (threadIdx.x == 0) {
        m->aborted = 0;
        for (int i = 0; i < kDPageSlots; i++) {
            mbar_init(&m->pages_full[i], 1);
            mbar_init(&m->pages_empty[i], 1);  // the copy warp
        }
        for (int i = 0; i < kDRing; i++) {
            for (int g = 0; g < kRefineGroups; g++) mbar_init(&m->full[g][i], 1);
            mbar_init(&m->empty[i], 4);  // the refine group that took the block
        }
        mbar_init(&m->tail_full, 1);  // the copy warp
        m->tails = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (warp == 0) {
        if (walker) dense_ring(prm, m, ring, lane);
    } else if (warp == 1) {
        if (walker) dense_pager(a, m, cta, ncta, lane);
    } else if (warp == 2) {
        for (int u = cta; u < a.B * a.Hkv; u += gridDim.x) {
            const int b = u / a.Hkv, h = u % a.Hkv;
            const int raw_n = a.seq_lens[b];
            const int n = len_of(a, b);
            if (lane == 0 && h == 0 && raw_n != n) raise_error(a.err, FFD_ERRBIT_BOUNDS);
            if (n == 0)
                for (int idx = lane; idx < a.G * kD; idx += 32)
                    a.out[((size_t)b * a.Hq + h * a.G) * kD + idx] = 0.0f;
        }
    } else if (warp >= 4 && walker) {
        dense_refiner(a, m, ring, px, cta, ncta, (warp - 4) >> 2, warp & 3, lane);
    }
}

}  // namespace

cudaError_t launch_dense(const DecodeArgs &a, int ctas, cudaStream_t stream) {
    static int smem_set[kMaxDevicesTracked];
    const cudaError_t ea = raise_smem_limit(dense_kernel, kDSmemBytes, smem_set);
    if (ea != cudaSuccess) return ea;
    DenseParams prm;
    memset(&prm, 0, sizeof prm);
    prm.a = a;
    const uint64_t rows = (uint64_t)a.P * a.Hkv * kPage;
    if (!make_tile_map(&prm.tm_k, const_cast<__nv_bfloat16 *>(a.k), rows) ||
        !make_tile_map(&prm.tm_v, const_cast<__nv_bfloat16 *>(a.v), rows))
        return cudaErrorInvalidValue;
    if (a.prof_start) cudaEventRecord(a.prof_start, stream);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(kDThreads);
    cfg.dynamicSmemBytes = kDSmemBytes;
    cfg.stream = stream;
    // the last groups of a unit wait for the unit's other CTAs: all CTAs must be resident
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, dense_kernel, prm);
    if (e != cudaSuccess) return e;
    if (a.prof_stop) cudaEventRecord(a.prof_stop, stream);
    return cudaGetLastError();
}

}  // namespace ffd
