// splitkv.cuh -- split-KV flash-decoding machinery shared by the FFD decode kernel and the dense
// comparison kernel: the persistent work schedule, bounded waits, the online-softmax state and
// its per-block update on the tensor cores, the per-(CTA, unit) records and their log-sum-exp
// merge. The decode step this serves is the one of "Faster Than Flash" (Methodology §3: exact
// attention over the selected blocks, split over the KV sequence); the dense kernel is the same
// computation over every block.
#pragma once

#include <cudaTypedefs.h>

#include "common.cuh"
#include "ptx.cuh"

namespace ffd {

constexpr int gcd_c(int x, int y) { return y == 0 ? x : gcd_c(y, x % y); }
constexpr int kSub = 6;              // blocks per sub-chunk (scan decision unit)
static_assert(kSub % 2 == 0, "the scan takes blocks k and k + kSub/2 side by side");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleMargin = 30.0f;        // lazy softmax rescaling, natural-log units
constexpr float kMarginLog2 = kRescaleMargin * kLog2e;
constexpr float kNoReference = -1.0e30f;       // softmax reference when there is none yet
constexpr int kPxBuf = 4 * 32 * 16;            // P^T fragments of one block (4 k-steps)

// ------------------------------------------------------------------------------------------
// Work schedule. The blocks of all (sequence, KV head) units, concatenated unit by unit, are cut
// into `ncta` contiguous ranges of equal length; each range is walked in sub-chunks of at most
// kSub blocks that never cross a unit. Every role of a CTA walks the same sequence.
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ int len_of(const DecodeArgs &a, int b) {
    const int n = a.seq_lens[b];
    const int cap = a.max_blocks * kPage;
    return n < 0 ? 0 : (n > cap ? cap : n);
}

__device__ __forceinline__ int nblocks_of(const DecodeArgs &a, int b) {
    return (len_of(a, b) + kPage - 1) / kPage;
}

__device__ __forceinline__ int64_t total_blocks(const DecodeArgs &a) {
    int64_t T = 0;
    for (int bb = 0; bb < a.B; bb++) T += (int64_t)a.Hkv * nblocks_of(a, bb);
    return T;
}

struct Sub {
    int b, h, j0, cnt;  // unit (b, h), first block, block count
    int nblk;           // blocks of the unit
    int64_t x0;         // global index of the sub-chunk's first block
    bool first;         // first sub-chunk of this CTA's segment of the unit
    bool last;          // last sub-chunk of this CTA's segment of the unit
};

struct Sched {
    int64_t x, x1, T;
    int b, h, j, nbb;  // current unit (b, h), next block j of its nbb blocks
    bool fresh;

    __device__ void init(const DecodeArgs &a, int cta, int ncta) {
        T = total_blocks(a);
        x = T * cta / ncta;
        x1 = T * (cta + 1) / ncta;
        int64_t pre = 0;
        b = h = j = nbb = 0;
        fresh = true;
        for (; b < a.B; b++) {
            const int nb = nblocks_of(a, b);
            const int64_t span = (int64_t)a.Hkv * nb;
            if (x < pre + span) {
                nbb = nb;
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
        s.j0 = j;
        s.nblk = nbb;
        s.cnt = cnt;
        s.x0 = x;
        s.first = fresh;
        s.last = (j + cnt == nbb) || (x + cnt == x1);
        fresh = false;
        x += cnt;
        j += cnt;
        if (j == nbb) {
            j = 0;
            fresh = true;
            if (++h == a.Hkv) {
                h = 0;
                for (b++; b < a.B; b++) {
                    nbb = nblocks_of(a, b);
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
// Bounded waits.
// ------------------------------------------------------------------------------------------
// Bounded wait: after a.wait_ns the CTA records FFD_ERRBIT_TIMEOUT, marks itself aborted and
// stops waiting (its results are then garbage, but every loop still ends).
template <class M>
__device__ __forceinline__ void wait_bar(const DecodeArgs &a, M *m, uint64_t *bar, uint32_t parity) {
    if (*reinterpret_cast<volatile uint32_t *>(&m->aborted)) return;
    if (mbar_try_wait(bar, parity)) return;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > a.wait_ns) {
            raise_error(a.err, FFD_ERRBIT_TIMEOUT);
            *reinterpret_cast<volatile uint32_t *>(&m->aborted) = 1;
            return;
        }
    }
}

// Wait for a copy this CTA issued, ignoring the abort flag (still bounded in time): no CTA exits
// with a copy into its shared memory in flight.
__device__ __forceinline__ void drain_bar(const DecodeArgs &a, uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > a.wait_ns) {
            raise_error(a.err, FFD_ERRBIT_TIMEOUT);
            return;
        }
    }
}

template <class M>
__device__ __forceinline__ bool aborted(M *m) {
    return *reinterpret_cast<volatile uint32_t *>(&m->aborted) != 0;
}

// Bounded wait until the global counter *c reaches target (written by other CTAs, which the
// cooperative launch keeps resident).
template <class M>
__device__ __forceinline__ void wait_count(const DecodeArgs &a, M *m, const int *c, int target) {
    if (ld_acquire_gpu(c) >= target) return;
    const uint64_t t0 = globaltimer_ns();
    while (ld_acquire_gpu(c) < target) {
        if (aborted(m)) return;
        if (globaltimer_ns() - t0 > a.wait_ns) {
            raise_error(a.err, FFD_ERRBIT_TIMEOUT);
            *reinterpret_cast<volatile uint32_t *>(&m->aborted) = 1;
            return;
        }
        __nanosleep(32);
    }
}

// ------------------------------------------------------------------------------------------
// Online softmax of one refine group.
// ------------------------------------------------------------------------------------------
// Softmax state of one refine warp. The reference m (heads 2tig, 2tig+1) is the same in every
// warp of a group; l holds this warp's rows only; o is O^T for channels 32mt + 16i + {g, g+8}
// and heads {2tig, 2tig+1}: o[i] = {(g, 2tig), (g, 2tig+1), (g+8, 2tig), (g+8, 2tig+1)}.
struct RefineState {
    float m0, m1, l0, l1;
    float nl0, nl1;  // -m * log2(e): p = 2^(s log2(e) - m log2(e)) is one FMA and one EX2
    float o[2][4];
};

// P^T fragments (bf16 hi and lo parts) of this warp's 16 rows for the PV k-step mt.
__device__ __forceinline__ uint4 p_fragments(float p00, float p01, float p10, float p11) {
    const uint32_t h0 = pack_bf16x2(p00, p01), h1 = pack_bf16x2(p10, p11);
    const uint32_t l0 = pack_bf16x2(p00 - __uint_as_float(h0 << 16),
                                    p01 - __uint_as_float(h0 & 0xffff0000u));
    const uint32_t l1 = pack_bf16x2(p10 - __uint_as_float(h1 << 16),
                                    p11 - __uint_as_float(h1 & 0xffff0000u));
    return make_uint4(movmatrix_trans(h0), movmatrix_trans(h1), movmatrix_trans(l0),
                      movmatrix_trans(l1));
}

// One block's probabilities and P.V for refine group grp (4 warps, named barrier 2 + grp), given
// warp mt's exact scores of rows r0 = 16mt + g and r1 = r0 + 8 for heads 2tig, 2tig+1 (-inf for
// rows past the sequence). The probabilities are taken against the group's reference m, which is
// raised (with a rescale of the state) only when a score passes m + kRescaleMargin in any warp;
// the P^T fragments (bf16 hi and lo parts) are exchanged through px_buf; then O^T for channels
// 32mt .. 32mt+31 over all 64 rows. vtile: the block's V rows as two 64 x 128 B halves (channels
// 0-63, then 64-127), 16-byte chunk c of row r stored at c ^ (r % 8). M: the kernel's shared
// control block (over[groups][2][4], wmax[groups][2][4][kMaxG]); pb selects the buffer pair.
template <class M>
__device__ __forceinline__ void softmax_pv(M *m, uint8_t *px_buf, const uint8_t *vtile, float s00,
                                           float s01, float s10, float s11, RefineState &R,
                                           int grp, int mt, int pb, int lane) {
    const int g = lane >> 2, tig = lane & 3;
    const uint32_t bar_id = 2 + grp;
    uint4 *px = reinterpret_cast<uint4 *>(px_buf);
    // ---- probabilities against the group's reference: x = (s - m) log2(e), p = 2^x
    float x00 = fmaf(s00, kLog2e, R.nl0), x01 = fmaf(s01, kLog2e, R.nl1);
    float x10 = fmaf(s10, kLog2e, R.nl0), x11 = fmaf(s11, kLog2e, R.nl1);
    const bool over = fmaxf(fmaxf(x00, x01), fmaxf(x10, x11)) > kMarginLog2;
    const uint32_t any_over = __any_sync(0xffffffffu, over);
    float p00 = ex2_approx(x00), p01 = ex2_approx(x01);
    float p10 = ex2_approx(x10), p11 = ex2_approx(x11);
    if (any_over) {  // this warp's row maxima, for the group's new reference
        float mx0 = fmaxf(s00, s10), mx1 = fmaxf(s01, s11);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
        }
        if (g == 0) {
            m->wmax[grp][pb][mt][2 * tig] = mx0;
            m->wmax[grp][pb][mt][2 * tig + 1] = mx1;
        }
    }
    if (lane == 0) m->over[grp][pb][mt] = any_over;
    px[mt * 32 + lane] = p_fragments(p00, p01, p10, p11);
    named_barrier_sync(bar_id, 128);
    const uint32_t group_over = m->over[grp][pb][0] | m->over[grp][pb][1] |
                                m->over[grp][pb][2] | m->over[grp][pb][3];
    if (group_over) {  // rare: raise the reference to the block maximum, rescale, redo P
        float mn0 = R.m0, mn1 = R.m1;
#pragma unroll
        for (int w = 0; w < 4; w++) {
            if (m->over[grp][pb][w]) {
                mn0 = fmaxf(mn0, m->wmax[grp][pb][w][2 * tig]);
                mn1 = fmaxf(mn1, m->wmax[grp][pb][w][2 * tig + 1]);
            }
        }
        const float al0 = ex2_approx((R.m0 - mn0) * kLog2e);
        const float al1 = ex2_approx((R.m1 - mn1) * kLog2e);
        R.m0 = mn0;
        R.m1 = mn1;
        R.nl0 = -mn0 * kLog2e;
        R.nl1 = -mn1 * kLog2e;
        R.l0 *= al0;
        R.l1 *= al1;
#pragma unroll
        for (int i = 0; i < 2; i++) {
            R.o[i][0] *= al0;
            R.o[i][1] *= al1;
            R.o[i][2] *= al0;
            R.o[i][3] *= al1;
        }
        p00 = ex2_approx(fmaf(s00, kLog2e, R.nl0));
        p01 = ex2_approx(fmaf(s01, kLog2e, R.nl1));
        p10 = ex2_approx(fmaf(s10, kLog2e, R.nl0));
        p11 = ex2_approx(fmaf(s11, kLog2e, R.nl1));
        px[mt * 32 + lane] = p_fragments(p00, p01, p10, p11);
        named_barrier_sync(bar_id, 128);
    }
    R.l0 += p00 + p10;
    R.l1 += p01 + p11;

    // ---- O^T(channels 32mt .. 32mt+31) += V^T P^T over the block's 64 rows. V^T fragments by
    // ldmatrix.trans from the swizzled tile (16-byte chunk c of row r is stored at c ^ (r % 8)).
    const int mi = lane >> 3, jr = lane & 7;
    const uint32_t vbase = smem_u32(vtile) + (mt >> 1) * 8192;
#pragma unroll
    for (int ks = 0; ks < 4; ks++) {
        const uint4 bp = px[ks * 32 + lane];
        const int tok = 16 * ks + ((mi >> 1) << 3) + jr;
#pragma unroll
        for (int i = 0; i < 2; i++) {
            const int md = 2 * mt + i;  // channels 16md .. 16md+15
            const int chunk = 2 * (md & 3) + (mi & 1);
            uint32_t v0r, v1r, v2r, v3r;
            ldmatrix_x4_trans(v0r, v1r, v2r, v3r, vbase + tok * 128 + ((chunk ^ jr) << 4));
            mma_bf16(R.o[i], v0r, v1r, v2r, v3r, bp.x, bp.y);
            mma_bf16(R.o[i], v0r, v1r, v2r, v3r, bp.z, bp.w);
        }
    }
}

// ------------------------------------------------------------------------------------------
// Split merge: out_i = sum_r e^(m_r - M) num_r / sum_r e^(m_r - M) den_r over a unit's records.
// Records of CTAs cf..cl, one per refine group (NG per CTA: kRefineGroups in the fused kernel),
// are contiguous from ws_part[(u + cf) * NG]; a record holds (num[128], m, den) per head. Counters in
// ws_cnt: [0, units) merge tickets, [units, 2 units) stage-1 slots, [2 units, 3 units) merge
// reports, [3 units, 4 units) merger declarations.
// ------------------------------------------------------------------------------------------
template <int NG = kRefineGroups>
__device__ __forceinline__ float *unit_record(const DecodeArgs &a, int u, int c, int grp) {
    return a.ws_part + ((size_t)(u + c) * NG + grp) * a.G * kPartStride;
}

// Merge of head i of a unit by one refine group (128 threads, thread = output channel), after
// every record of the unit is written. Records are loaded in independent batches: the maxima
// (lane r loads record r), then 16 records at a time whose weights, denominators and channel
// values are loaded together.
template <int NG = kRefineGroups>
__device__ __forceinline__ void merge_head(const DecodeArgs &a, int b, int h, int cf, int cl, int i,
                                           int mt, int lane) {
    const int u = b * a.Hkv + h;
    const int nr = NG * (cl - cf + 1);
    const size_t rstride = (size_t)a.G * kPartStride;
    const float *hb = unit_record<NG>(a, u, cf, 0) + (size_t)i * kPartStride;
    const int ch = 32 * mt + lane;
    float M = -INFINITY;
    for (int r = lane; r < nr; r += 32) M = fmaxf(M, __ldcg(hb + r * rstride + kD));
    M = warp_max(M);
    float num = 0.0f, den = 0.0f;
    if (M != -INFINITY) {
#pragma unroll 1
        for (int r0 = 0; r0 < nr; r0 += 16) {
            const int cnt = nr - r0 < 16 ? nr - r0 : 16;
            const float *own = hb + (size_t)(r0 + (lane < cnt ? lane : 0)) * rstride;
            const float mr = lane < cnt ? __ldcg(own + kD) : -INFINITY;
            const float dr = lane < cnt ? __ldcg(own + kD + 1) : 0.0f;
            float x[16];
#pragma unroll
            for (int j = 0; j < 16; j++)
                x[j] = __ldcg(hb + (size_t)(r0 + (j < cnt ? j : 0)) * rstride + ch);
            const float f = mr == -INFINITY ? 0.0f : exp2f((mr - M) * kLog2e);
            den = fmaf(f, dr, den);
#pragma unroll
            for (int j = 0; j < 16; j++) {
                const float fj = __shfl_sync(0xffffffffu, f, j);
                if (j < cnt) num = fmaf(fj, x[j], num);
            }
        }
        den = warp_sum(den);
    }
    a.out[((size_t)b * a.Hq + h * a.G + i) * kD + ch] = den > 0.0f ? num / den : 0.0f;
    if (a.m_tilde && mt == 0) {  // the reported pseudo-max, from the stage-1 slots
        float mx = -INFINITY;
        for (int sl = lane; sl < a.nf; sl += 32)
            mx = fmaxf(mx, __ldcg(a.ws_m1 + ((size_t)u * a.nf + sl) * kMaxG + i));
        mx = warp_max(mx);
        if (lane == 0) a.m_tilde[(size_t)b * a.Hq + h * a.G + i] = mx;
    }
}

__device__ __forceinline__ int *slot_counter(const DecodeArgs &a, int u) {
    return a.ws_cnt + a.B * a.Hkv + u;
}

__device__ __forceinline__ int *done_counter(const DecodeArgs &a, int u) {
    return a.ws_cnt + 2 * a.B * a.Hkv + u;
}

// Declarations of the unit's ranked mergers: bit r (rank r has taken its ticket), bit 8 + r (and
// its CTA has no work after this segment).
__device__ __forceinline__ int *declare_word(const DecodeArgs &a, int u) {
    return a.ws_cnt + 3 * a.B * a.Hkv + u;
}

// A refine group's record of softmax state R: (num[128], m, den) per head, den summed over the
// group's warps through m->lsum, each warp writing its own channels.
template <class M>
__device__ __forceinline__ void write_record(const DecodeArgs &a, M *m, const RefineState &R,
                                             float *rec, int grp, int mt, int lane) {
    const int g = lane >> 2, tig = lane & 3;
    const uint32_t bar_id = 2 + grp;
    float l0 = R.l0, l1 = R.l1;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, o);
        l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    if (g == 0) {
        m->lsum[grp][mt][2 * tig] = l0;
        m->lsum[grp][mt][2 * tig + 1] = l1;
    }
    named_barrier_sync(bar_id, 128);
    const int h0 = 2 * tig, h1 = 2 * tig + 1;
#pragma unroll
    for (int i = 0; i < 2; i++) {
        const int d = 32 * mt + 16 * i + g;
        if (h0 < a.G) {
            rec[h0 * kPartStride + d] = R.o[i][0];
            rec[h0 * kPartStride + d + 8] = R.o[i][2];
        }
        if (h1 < a.G) {
            rec[h1 * kPartStride + d] = R.o[i][1];
            rec[h1 * kPartStride + d + 8] = R.o[i][3];
        }
    }
    if (mt == 0 && g == 0) {
        const float L0 = (m->lsum[grp][0][h0] + m->lsum[grp][1][h0]) +
                         (m->lsum[grp][2][h0] + m->lsum[grp][3][h0]);
        const float L1 = (m->lsum[grp][0][h1] + m->lsum[grp][1][h1]) +
                         (m->lsum[grp][2][h1] + m->lsum[grp][3][h1]);
        if (h0 < a.G) {
            rec[h0 * kPartStride + kD] = R.m0;
            rec[h0 * kPartStride + kD + 1] = L0;
        }
        if (h1 < a.G) {
            rec[h1 * kPartStride + kD] = R.m1;
            rec[h1 * kPartStride + kD + 1] = L1;
        }
    }
}

// Bounded wait until (*word & mask) == mask (bits other groups set right after their tickets).
template <class M>
__device__ __forceinline__ unsigned int wait_bits(const DecodeArgs &a, M *m, const int *word,
                                                  unsigned int mask) {
    unsigned int v = (unsigned int)ld_acquire_gpu(word);
    const uint64_t t0 = globaltimer_ns();
    while ((v & mask) != mask) {
        if (aborted(m)) break;
        if (globaltimer_ns() - t0 > a.wait_ns) {
            raise_error(a.err, FFD_ERRBIT_TIMEOUT);
            *reinterpret_cast<volatile uint32_t *>(&m->aborted) = 1;
            break;
        }
        __nanosleep(32);
        v = (unsigned int)ld_acquire_gpu(word);
    }
    return v;
}

// After its record is written: the group's ticket for the unit of sub-chunk s. The groups that
// take the last nm = min(G, groups of the unit) tickets are ranked 0 .. nm-1 in ticket order and
// merge the unit's heads, head i by rank i % nm. A ranked group declares right after its ticket
// whether it is final (its CTA has no work after this segment). The last group finds every record
// written; it waits for the other ranks' declarations (made a moment after their tickets) and
// merges its own heads and those of every rank that is not final. A final group of lower rank
// waits for the remaining tickets (their groups are at the ends of their ranges too) and merges
// its heads. A group whose CTA still has work never waits for other groups' records: the other
// parts of the unit may be walked at the very end of other CTAs' ranges.
template <class M, int NG = kRefineGroups>
__device__ __forceinline__ void finish_unit(const DecodeArgs &a, M *m, const Sub &s, int cta,
                                            int ncta, int64_t T, int grp, int mt, int lane) {
    const uint32_t bar_id = 2 + grp;
    const int u = s.b * a.Hkv + s.h;
    __threadfence();
    named_barrier_sync(bar_id, 128);
    const int64_t first = s.x0 - s.j0;  // global index of the unit's first block
    const int cf = cta_of(first, T, ncta), cl = cta_of(first + s.nblk - 1, T, ncta);
    const int target = NG * (cl - cf + 1);
    const int nm = a.G < target ? a.G : target;
    const bool final_seg = s.x0 + s.cnt == T * (cta + 1) / ncta;
    if (mt == 0 && lane == 0) {
        const int r = atomicAdd(a.ws_cnt + u, 1) - (target - nm);
        uint32_t role = 0;  // bit 0: merges; bit 1: waits for every ticket first; bits 8..15:
                            // ranks whose heads it merges; 4: ranked, merges nothing
        if (r >= 0 && r < nm - 1) {
            atomicOr(reinterpret_cast<unsigned int *>(declare_word(a, u)),
                     (1u << r) | (final_seg ? 1u << (8 + r) : 0u));
            role = final_seg ? 3u | ((1u << r) << 8) : 4u;
        } else if (r == nm - 1) {
            const unsigned int d = wait_bits(a, m, declare_word(a, u), (1u << r) - 1u);
            uint32_t cover = 1u << r;
            for (int q = 0; q < r; q++)
                if (!((d >> (8 + q)) & 1u)) cover |= 1u << q;
            role = 1u | (cover << 8);
        }
        m->merge_flag[grp] = role;
    }
    named_barrier_sync(bar_id, 128);
    const uint32_t role = m->merge_flag[grp];
    if (role == 0) return;
    if (role & 1u) {
        if ((role & 2u) && mt == 0 && lane == 0) wait_count(a, m, a.ws_cnt + u, target);
        named_barrier_sync(bar_id, 128);
        __threadfence();
        const uint32_t cover = (role >> 8) & 0xffu;
        for (int i = 0; i < a.G; i++)
            if ((cover >> (i % nm)) & 1u) merge_head<NG>(a, s.b, s.h, cf, cl, i, mt, lane);
        named_barrier_sync(bar_id, 128);
    }
    if (mt == 0 && lane == 0) {
        // every ranked group reports once its heads are merged (or at once when it merges none);
        // the last report clears the unit's counters for the next call
        if (atomicAdd(done_counter(a, u), 1) == nm - 1) {
            a.ws_cnt[u] = 0;
            *slot_counter(a, u) = 0;
            *done_counter(a, u) = 0;
            *declare_word(a, u) = 0;
        }
    }
}

// ------------------------------------------------------------------------------------------
// Host: TMA tensor map of a bf16 [rows][128] tile array (V, or K on the dense path).
// ------------------------------------------------------------------------------------------
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// The array as a 3-D tensor {64 channels, rows, 2 channel halves} (strides 256 B per row, 128 B
// per half) with a box of {64, 64, 2}: one copy lands a block's 64 rows as two 64 x 128 B tiles
// with the 128-byte swizzle (16-byte chunk c of row r at c ^ (r % 8)), channels 0-63 first.
inline bool make_tile_map(CUtensorMap *map, void *ptr, uint64_t rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {64, rows, 2};
    const cuuint64_t strides[2] = {kD * 2, 128};
    const cuuint32_t box[3] = {64, (cuuint32_t)kPage, 2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace ffd
