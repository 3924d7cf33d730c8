// stage1.cuh -- stage 1 of the FFD decode step (the pseudo-max m~ of every (sequence, KV head)
// unit), shared by the fused kernel and the scan-then-refine kernel. M is the kernel's shared
// control block: it provides wmax[groups][2][4][kMaxG] (per-warp row maxima).
//
// Source: "Faster Than Flash", Methodology §2 (m~_i is the maximum exact score over the sink
// tokens j < S and the local tokens n - L <= j < n) and §3 (stage 1 pseudo-max estimation).
#pragma once

#include "common.cuh"
#include "ptx.cuh"
#include "scan.cuh"
#include "splitkv.cuh"

namespace ffd {

// ------------------------------------------------------------------------------------------
// Stage 1 (pseudo-max), run by the NG refine groups of every CTA at the start of a decode kernel,
// before any block reaches them. The (unit, forced-block slot) pairs are cut into equal contiguous
// runs, one per group of the grid (ncta * NG); in a group, warp mt takes rows 16mt .. 16mt+15 of the
// slot's block. Exact scores s = sm q . K^ (thumbnail + residual, on tensor cores) of the block's
// sink and local tokens; their per-head maximum goes to ws_m1 (the pseudo-max m~ of a unit is the
// maximum over its slots), then the unit's slot counter is raised. Scan warp 0 of every CTA that
// walks the unit waits for all of its slots before it sets the thresholds. Slot 0 of every unit
// also clears the keep-mask tail past the sequence and, for an empty sequence (which no CTA
// walks, so its counter stays at zero), writes the zero output and m~ = -inf.
// ------------------------------------------------------------------------------------------
template <int NG, class M>
__device__ __forceinline__ void pseudo_max_slots(const DecodeArgs &a, M *m, int cta, int nctas,
                                                 int grp, int mt, int lane) {
    const int units = a.B * a.Hkv;
    const int nz = units * a.nf;
    const int workers = nctas * NG;
    const int tid = 32 * mt + lane;
    const int g = lane >> 2, tig = lane & 3;
    // a worker takes a contiguous run of (unit, slot) pairs, so that with more pairs than workers
    // (many short sequences) it keeps one unit's query operands and length across its slots
    const int wk = cta * NG + grp;
    const int z0 = (int)((int64_t)nz * wk / workers), z1 = (int)((int64_t)nz * (wk + 1) / workers);
    int it = 0, cu = -1, raw_n = 0, n = 0;
    // block-table entries of 32 consecutive slots of the current unit, one per lane (slot
    // pg_base + lane), read together instead of one dependent read per pair
    int pg_base = -1, pg_mine = -1;
    int pending = 0;  // slots of unit cu written since its counter was last raised
    ThumbOps Q;
    ResidOps QR;
    for (int z = z0; z < z1; z++, it++) {
        const int u = z / a.nf, slot = z % a.nf;
        const int b = u / a.Hkv, h = u % a.Hkv;
        if (u != cu) {
            // the query operands do not depend on the page: their loads overlap the two dependent
            // loads (sequence length, then block table) that locate the block
            load_thumb_ops(a, b, h, lane, Q);
            load_resid_ops(a, b, h, lane, QR);
            raw_n = a.seq_lens[b];
            n = len_of(a, b);
            cu = u;
            pg_base = -1;
        }
        const int nb = (n + kPage - 1) / kPage;
        if (slot == 0) {
            if (tid == 0 && h == 0 && raw_n != n) raise_error(a.err, FFD_ERRBIT_BOUNDS);
            if (a.keep_mask)
                for (int blk = nb + tid; blk < a.max_blocks; blk += 128)
                    a.keep_mask[(size_t)u * a.max_blocks + blk] = 0;
            if (n == 0) {
                for (int idx = tid; idx < a.G * kD; idx += 128)
                    a.out[((size_t)b * a.Hq + h * a.G) * kD + idx] = 0.0f;
                if (a.m_tilde && tid < a.G)
                    a.m_tilde[(size_t)b * a.Hq + h * a.G + tid] = -INFINITY;
            }
        }
        if (n == 0) continue;  // uniform across the group; nobody waits for this unit
        const ForcedBlocks fb(n, a.S, a.L);
        float *mdst = a.ws_m1 + ((size_t)u * a.nf + slot) * kMaxG;
        int page = -1;
        const int blk = slot < fb.count ? fb.block(slot) : 0;
        if (slot < fb.count) {
            if (pg_base < 0 || slot >= pg_base + 32) {  // warp-uniform
                pg_base = slot;
                const int sl = slot + lane;
                pg_mine = sl < fb.count ? a.block_table[(size_t)b * a.max_blocks + fb.block(sl)] : -1;
            }
            page = __shfl_sync(0xffffffffu, pg_mine, slot - pg_base);
            if (page < 0 || page >= a.P) page = -1;  // flagged by the page warp
        }
        float mx0 = -INFINITY, mx1 = -INFINITY;
        if (page >= 0) {  // uniform across the group
            const size_t tile = (size_t)page * a.Hkv + h;
            const uint8_t *trec = a.thumb + tile * kThumbRec;
            const uint8_t *rrec = a.resid + tile * kResidRec;
            const int r0 = 16 * mt + g, r1 = r0 + 8;
            const float4 e = exact_tile(trec, rrec, r0, r1, tig, Q, QR, a.sm_scale);
            const int t0 = blk * kPage + r0, t1 = blk * kPage + r1;
            // pseudo-max candidates: sink and local tokens inside the sequence
            const bool v0 = t0 < n && (t0 < a.S || t0 >= n - a.L);
            const bool v1 = t1 < n && (t1 < a.S || t1 >= n - a.L);
            const float s00 = v0 ? e.x : -INFINITY;
            const float s01 = v0 ? e.y : -INFINITY;
            const float s10 = v1 ? e.z : -INFINITY;
            const float s11 = v1 ? e.w : -INFINITY;
            mx0 = fmaxf(s00, s10);
            mx1 = fmaxf(s01, s11);
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
            }
        }
        // the reduction buffers alternate between pairs: a buffer is written again two pairs
        // later, after the next pair's barrier, which every reader of this pair has passed
        float (&red)[4][kMaxG] = m->wmax[grp][it & 1];
        if (g == 0) {
            red[mt][2 * tig] = mx0;
            red[mt][2 * tig + 1] = mx1;
        }
        named_barrier_sync(2 + grp, 128);
        if (tid < kMaxG)
            mdst[tid] = tid < a.G ? fmaxf(fmaxf(red[0][tid], red[1][tid]),
                                          fmaxf(red[2][tid], red[3][tid]))
                                  : -INFINITY;
        pending++;
        // the unit's counter is raised once per run of its slots: the writers' fence, then one
        // add of the slots written
        if (z + 1 == z1 || (z + 1) / a.nf != u) {
            if (tid < kMaxG) __threadfence();
            named_barrier_sync(2 + grp, 128);
            if (tid == 0) atomicAdd(slot_counter(a, u), pending);
            pending = 0;
        }
    }
    // the reduction buffers are the refine warps' block-maxima buffers
    named_barrier_sync(2 + grp, 128);
}

// ------------------------------------------------------------------------------------------
// Stage 1 by single warps (the scan-then-refine kernel, where it runs beside the scan): worker
// wk of `workers` takes an equal contiguous run of the (unit, slot) pairs and computes all 64
// rows of each slot's block itself, four m-tiles of rows (16 mt + g, 16 mt + g + 8). Outputs as
// above; in addition the warp that fills a unit's last slot writes the unit's m~ per head to
// ws_mt[u][0 .. 8) and then raises the slot counter once more (to nf + 1), so that a reader
// needing m~ itself waits for nf + 1 and loads 8 values instead of every slot.
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void pseudo_max_warp(const DecodeArgs &a, int wk, int workers,
                                                int lane) {
    const int units = a.B * a.Hkv;
    const int nz = units * a.nf;
    const int g = lane >> 2, tig = lane & 3;
    const int z0 = (int)((int64_t)nz * wk / workers), z1 = (int)((int64_t)nz * (wk + 1) / workers);
    int cu = -1, raw_n = 0, n = 0;
    ThumbOps Q;
    ResidOps QR;
    for (int z = z0; z < z1; z++) {
        const int u = z / a.nf, slot = z % a.nf;
        const int b = u / a.Hkv, h = u % a.Hkv;
        if (u != cu) {
            load_thumb_ops(a, b, h, lane, Q);
            load_resid_ops(a, b, h, lane, QR);
            raw_n = a.seq_lens[b];
            n = len_of(a, b);
            cu = u;
        }
        const int nb = (n + kPage - 1) / kPage;
        if (slot == 0) {
            if (lane == 0 && h == 0 && raw_n != n) raise_error(a.err, FFD_ERRBIT_BOUNDS);
            if (a.keep_mask)
                for (int blk = nb + lane; blk < a.max_blocks; blk += 32)
                    a.keep_mask[(size_t)u * a.max_blocks + blk] = 0;
            if (n == 0) {
                for (int idx = lane; idx < a.G * kD; idx += 32)
                    a.out[((size_t)b * a.Hq + h * a.G) * kD + idx] = 0.0f;
                if (a.m_tilde && lane < a.G)
                    a.m_tilde[(size_t)b * a.Hq + h * a.G + lane] = -INFINITY;
            }
        }
        if (n == 0) continue;  // warp-uniform; nobody waits for this unit
        const ForcedBlocks fb(n, a.S, a.L);
        float *mdst = a.ws_m1 + ((size_t)u * a.nf + slot) * kMaxG;
        int page = -1;
        const int blk = slot < fb.count ? fb.block(slot) : 0;
        if (slot < fb.count) {
            page = a.block_table[(size_t)b * a.max_blocks + blk];
            if (page < 0 || page >= a.P) page = -1;  // flagged by the scan's producer
        }
        float mx0 = -INFINITY, mx1 = -INFINITY;
        if (page >= 0) {  // warp-uniform
            const size_t tile = (size_t)page * a.Hkv + h;
            const uint8_t *trec = a.thumb + tile * kThumbRec;
            const uint8_t *rrec = a.resid + tile * kResidRec;
#pragma unroll 1
            for (int mt = 0; mt < 4; mt++) {  // one m-tile at a time: 128 registers
                const int r0 = 16 * mt + g, r1 = r0 + 8;
                const float4 e = exact_tile(trec, rrec, r0, r1, tig, Q, QR, a.sm_scale);
                const int t0 = blk * kPage + r0, t1 = blk * kPage + r1;
                // pseudo-max candidates: sink and local tokens inside the sequence
                const bool v0 = t0 < n && (t0 < a.S || t0 >= n - a.L);
                const bool v1 = t1 < n && (t1 < a.S || t1 >= n - a.L);
                mx0 = fmaxf(mx0, fmaxf(v0 ? e.x : -INFINITY, v1 ? e.z : -INFINITY));
                mx1 = fmaxf(mx1, fmaxf(v0 ? e.y : -INFINITY, v1 ? e.w : -INFINITY));
            }
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
            }
        }
        if (g == 0) {  // lanes 0..3: heads 2 tig and 2 tig + 1
            mdst[2 * tig] = 2 * tig < a.G ? mx0 : -INFINITY;
            mdst[2 * tig + 1] = 2 * tig + 1 < a.G ? mx1 : -INFINITY;
            __threadfence();
        }
        __syncwarp();
        int prev = 0;
        if (lane == 0) {
            prev = atomicAdd(slot_counter(a, u), 1);
            __threadfence();
        }
        __syncwarp();
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev == a.nf - 1) {  // the unit's last slot: its m~ per head
            // head lane & 7 over slots lane >> 3, + 4, ...; the four partial maxima of a head are
            // then combined across the warp
            float mx = -INFINITY;
            for (int sl = lane >> 3; sl < a.nf; sl += 4)
                mx = fmaxf(mx, __ldcg(a.ws_m1 + ((size_t)u * a.nf + sl) * kMaxG + (lane & 7)));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            if (lane < kMaxG) {
                a.ws_mt[(size_t)u * kMaxG + lane] = mx;
                __threadfence();
            }
            __syncwarp();
            if (lane == 0) atomicAdd(slot_counter(a, u), 1);
        }
    }
}

}  // namespace ffd
