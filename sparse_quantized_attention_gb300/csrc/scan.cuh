// scan.cuh -- the stage-2 provisional scores on the tensor cores, shared by the FFD decode kernel
// and the comparison selectors: query operands of a (sequence, KV head) unit, and the scores
// s^ = sm * q . x^2 of 16 x 8 (token, head) tiles of a thumbnail record.
//
// Source: "Faster Than Flash", Methodology §1 (2-bit thumbnails as a fast proxy for importance)
// and §3 (stage 2 streams the 2-bit keys and computes provisional scores).
//
// Tensor-core operands (mma.sync m16n8k16, bf16 in, fp32 accumulate; 16 tokens x 8 heads):
// A = codes of 16 tokens, B = the GQA group's queries (heads as N, padded to 8). 2-bit codes enter
// as bf16 bit patterns (code << s) with s <= 6: exponent field 0, so the value is exactly
// code * 2^s * 2^-133. B holds q * 2^(kKq - s), so every product is exactly code * q * 2^(kKq-133)
// and one LOP3 turns two codes into an operand register. Channel order inside each 16-channel
// MMA step is permuted (the same permutation on A and B); a dot product does not depend on it.
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace ffd {

constexpr int kKq = 100;             // q enters the MMA scaled by 2^kKq (|q| < 2^27 required)
constexpr float kUnscale = 8589934592.0f;      // 2^(133 - kKq)
constexpr float kQMax = 134217728.0f;          // 2^27

// ------------------------------------------------------------------------------------------
// Query operands. Thread (g = lane/4, tig = lane%4) holds the B fragments of head g and, for the
// epilogue, the per-group query sums of heads 2*tig and 2*tig+1.
// ------------------------------------------------------------------------------------------
struct ThumbOps {
    uint32_t bt0[8], bt1[8];  // chunk kc = channels 16kc .. 16kc+15, head g
    float qs[2][4];           // sum of q over group gg for heads 2tig, 2tig+1
};

// Per-group query sums of heads 2tig, 2tig+1, from this thread's partial sums of head g over the
// channels c = tig (mod 4): quad reduction, then fetch from the quads of heads 2tig and 2tig+1.
__device__ __forceinline__ void group_sums(float (&part)[4], int tig, float (&qs)[2][4]) {
#pragma unroll
    for (int gg = 0; gg < 4; gg++) {
        part[gg] += __shfl_xor_sync(0xffffffffu, part[gg], 1);
        part[gg] += __shfl_xor_sync(0xffffffffu, part[gg], 2);
    }
#pragma unroll
    for (int gg = 0; gg < 4; gg++) {
        qs[0][gg] = __shfl_sync(0xffffffffu, part[gg], 8 * tig);
        qs[1][gg] = __shfl_sync(0xffffffffu, part[gg], 8 * tig + 4);
    }
}

__device__ __forceinline__ const __nv_bfloat16 *q_row(const DecodeArgs &a, int b, int h, int g) {
    return a.q + ((size_t)b * a.Hq + h * a.G + (g < a.G ? g : 0)) * kD;
}

// The operands from qrow, the query row of head g (global or shared memory; hv: g < G, else the
// head is padding and its operands are zero).
__device__ __forceinline__ void thumb_ops_from_row(const __nv_bfloat16 *qrow, bool hv, int lane,
                                                   int *err, ThumbOps &Q) {
    const int tig = lane & 3;
    float big = 0.0f;
    auto ld = [&](int c) {
        const float v = hv ? __bfloat162float(qrow[c]) : 0.0f;
        big = fmaxf(big, fabsf(v));
        return v;
    };
    const float st = __int_as_float((127 + kKq - 2 * tig) << 23);  // 2^(kKq - 2 tig)
    float part[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int kc = 0; kc < 8; kc++) {
        const float x0 = ld(16 * kc + tig), x1 = ld(16 * kc + 8 + tig);
        const float x2 = ld(16 * kc + 4 + tig), x3 = ld(16 * kc + 12 + tig);
        Q.bt0[kc] = pack_bf16x2(x0 * st, x1 * st);
        Q.bt1[kc] = pack_bf16x2(x2 * st, x3 * st);
        part[kc >> 1] += (x0 + x1) + (x2 + x3);
    }
    group_sums(part, tig, Q.qs);
    if (!(big < kQMax)) raise_error(err, FFD_ERRBIT_RANGE);
}

__device__ __forceinline__ void load_thumb_ops(const DecodeArgs &a, int b, int h, int lane,
                                               ThumbOps &Q) {
    const int g = lane >> 2;
    thumb_ops_from_row(q_row(a, b, h, g), g < a.G, lane, a.err, Q);
}

// The query rows of unit (b, h) -- G rows of kD bf16, contiguous in q -- copied to shared memory
// at sq (16-byte vectors; q is 16-byte aligned and a unit's rows start at a multiple of 256
// bytes) by threads tid = 0 .. nthr-1. One round trip, in place of every warp's scattered reads
// of the same rows; the caller synchronises before reading sq.
__device__ __forceinline__ void stage_query(const DecodeArgs &a, int b, int h, __nv_bfloat16 *sq,
                                            int tid, int nthr) {
    const uint4 *src = reinterpret_cast<const uint4 *>(a.q + ((size_t)b * a.Hq + h * a.G) * kD);
    uint4 *dst = reinterpret_cast<uint4 *>(sq);
    for (int i = tid; i < a.G * kD / 8; i += nthr) dst[i] = src[i];
}

// D[gg] = sum over group gg of q . code (scaled by 2^(kKq-133)) for rows (g, g+8) x heads.
__device__ __forceinline__ void thumb_mma(float (&D)[4][4], const uint32_t (&w0)[8],
                                          const uint32_t (&w1)[8], uint32_t m0,
                                          const ThumbOps &Q) {
#pragma unroll
    for (int gg = 0; gg < 4; gg++) D[gg][0] = D[gg][1] = D[gg][2] = D[gg][3] = 0.0f;
#pragma unroll
    for (int kc = 0; kc < 8; kc++) {
        const uint32_t a0 = w0[kc] & m0, a1 = w1[kc] & m0;
        const uint32_t a2 = (w0[kc] >> 8) & m0, a3 = (w1[kc] >> 8) & m0;
        mma_bf16(D[kc >> 1], a0, a1, a2, a3, Q.bt0[kc], Q.bt1[kc]);
    }
}

__device__ __forceinline__ void unpack4h(uint2 v, float (&f)[4]) {
    const float2 lo = __half22float2(*reinterpret_cast<const __half2 *>(&v.x));
    const float2 hi = __half22float2(*reinterpret_cast<const __half2 *>(&v.y));
    f[0] = lo.x;
    f[1] = lo.y;
    f[2] = hi.x;
    f[3] = hi.y;
}

// Provisional score s^ = sm * sum_g (scale_g q_g.c_g + zero_g sum(q_g)) of accumulator entry e.
__device__ __forceinline__ float est_score(const float (&D)[4][4], int e, const float (&sf)[4],
                                           const float (&zf)[4], const float (&qs)[4], float sm) {
    float acc = 0.0f;
#pragma unroll
    for (int gg = 0; gg < 4; gg++)
        acc = fmaf(sf[gg] * kUnscale, D[gg][e], fmaf(zf[gg], qs[gg], acc));
    return acc * sm;
}

// Provisional scores of one m-tile (rows r0 = 16 mt + g and r1 = r0 + 8 of a thumbnail block in
// shared memory), for heads 2tig, 2tig+1: {(r0,h0), (r0,h1), (r1,h0), (r1,h1)}.
__device__ __forceinline__ float4 scan_tile(const uint8_t *base, int r0, int r1, uint32_t m0,
                                            const ThumbOps &Q, float sm) {
    const uint4 *c0 = reinterpret_cast<const uint4 *>(base + r0 * kThumbRow);
    const uint4 *c1 = reinterpret_cast<const uint4 *>(base + r1 * kThumbRow);
    const uint4 p0 = c0[0], p1 = c0[1], p2 = c1[0], p3 = c1[1];
    const uint32_t w0[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
    const uint32_t w1[8] = {p2.x, p2.y, p2.z, p2.w, p3.x, p3.y, p3.z, p3.w};
    float D[4][4];
    thumb_mma(D, w0, w1, m0, Q);
    float sf0[4], sf1[4], zf0[4], zf1[4];
    const uint2 *ts = reinterpret_cast<const uint2 *>(base + kThumbScaleOff);
    const uint2 *tz = reinterpret_cast<const uint2 *>(base + kThumbZeroOff);
    unpack4h(ts[r0], sf0);
    unpack4h(ts[r1], sf1);
    unpack4h(tz[r0], zf0);
    unpack4h(tz[r1], zf1);
    float4 e;
    e.x = est_score(D, 0, sf0, zf0, Q.qs[0], sm);
    e.y = est_score(D, 1, sf0, zf0, Q.qs[1], sm);
    e.z = est_score(D, 2, sf1, zf1, Q.qs[0], sm);
    e.w = est_score(D, 3, sf1, zf1, Q.qs[1], sm);
    return e;
}

// scan_tile's scores divided by sm * 2^(133 - kKq), for a caller that needs only their maximum
// over rows: the query sums enter divided by 2^(133 - kKq) (qsr, a power-of-two scaling, exact
// for normal values), so every partial sum is the scan_tile one times 2^(kKq - 133) and no
// per-score multiply is left; the caller multiplies the maximum by sm * 2^(133 - kKq) > 0, which
// gives the maximum of scan_tile's scores bit for bit (rounding is monotonic).
__device__ __forceinline__ float raw_score(const float (&D)[4][4], int e, const float (&sf)[4],
                                           const float (&zf)[4], const float (&qsr)[4]) {
    float acc = 0.0f;
#pragma unroll
    for (int gg = 0; gg < 4; gg++) acc = fmaf(sf[gg], D[gg][e], fmaf(zf[gg], qsr[gg], acc));
    return acc;
}

__device__ __forceinline__ float4 scan_tile_raw(const uint8_t *base, int r0, int r1, uint32_t m0,
                                                const ThumbOps &Q, const float (&qsr)[2][4]) {
    const uint4 *c0 = reinterpret_cast<const uint4 *>(base + r0 * kThumbRow);
    const uint4 *c1 = reinterpret_cast<const uint4 *>(base + r1 * kThumbRow);
    const uint4 p0 = c0[0], p1 = c0[1], p2 = c1[0], p3 = c1[1];
    const uint32_t w0[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
    const uint32_t w1[8] = {p2.x, p2.y, p2.z, p2.w, p3.x, p3.y, p3.z, p3.w};
    float D[4][4];
    thumb_mma(D, w0, w1, m0, Q);
    float sf0[4], sf1[4], zf0[4], zf1[4];
    const uint2 *ts = reinterpret_cast<const uint2 *>(base + kThumbScaleOff);
    const uint2 *tz = reinterpret_cast<const uint2 *>(base + kThumbZeroOff);
    unpack4h(ts[r0], sf0);
    unpack4h(ts[r1], sf1);
    unpack4h(tz[r0], zf0);
    unpack4h(tz[r1], zf1);
    float4 e;
    e.x = raw_score(D, 0, sf0, zf0, qsr[0]);
    e.y = raw_score(D, 1, sf0, zf0, qsr[1]);
    e.z = raw_score(D, 2, sf1, zf1, qsr[0]);
    e.w = raw_score(D, 3, sf1, zf1, qsr[1]);
    return e;
}

// Query operands of the residual correction: int8 codes enter the MMA as (c8 + 128), with the
// same scaling as the thumbnail codes; the +128 is removed with the per-group query sums.
struct ResidOps {
    uint32_t br0[8], br1[8];  // chunk 2gg + half, head g
    float qs[2][4];
};

__device__ __forceinline__ void resid_ops_from_row(const __nv_bfloat16 *qrow, bool hv, int lane,
                                                   ResidOps &Q) {
    const int tig = lane & 3;
    const float sr = __int_as_float((127 + kKq) << 23);  // 2^kKq
    float part[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int gg = 0; gg < 4; gg++) {
        const int base = 32 * gg + 8 * tig;
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; e++) y[e] = hv ? __bfloat162float(qrow[base + e]) : 0.0f;
        Q.br0[2 * gg] = pack_bf16x2(y[0] * sr, y[2] * sr);
        Q.br1[2 * gg] = pack_bf16x2(y[1] * sr, y[3] * sr);
        Q.br0[2 * gg + 1] = pack_bf16x2(y[4] * sr, y[6] * sr);
        Q.br1[2 * gg + 1] = pack_bf16x2(y[5] * sr, y[7] * sr);
        part[gg] = ((y[0] + y[1]) + (y[2] + y[3])) + ((y[4] + y[5]) + (y[6] + y[7]));
    }
    group_sums(part, tig, Q.qs);
}

__device__ __forceinline__ void load_resid_ops(const DecodeArgs &a, int b, int h, int lane,
                                               ResidOps &Q) {
    const int g = lane >> 2;
    resid_ops_from_row(q_row(a, b, h, g), g < a.G, lane, Q);
}

// D[gg] = sum over group gg of q . (c8 + 128) (scaled by 2^(kKq-133)).
// x0[gg] / x1[gg]: bytes 32gg + 8tig .. +7 of rows g / g+8.
__device__ __forceinline__ void resid_mma(float (&D)[4][4], const uint2 (&x0)[4],
                                          const uint2 (&x1)[4], const ResidOps &Q) {
#pragma unroll
    for (int gg = 0; gg < 4; gg++) D[gg][0] = D[gg][1] = D[gg][2] = D[gg][3] = 0.0f;
#pragma unroll
    for (int gg = 0; gg < 4; gg++) {
#pragma unroll
        for (int half = 0; half < 2; half++) {
            const uint32_t v0 = half ? x0[gg].y : x0[gg].x;
            const uint32_t v1 = half ? x1[gg].y : x1[gg].x;
            const uint32_t a0 = (v0 & 0x00FF00FFu) ^ 0x00800080u;
            const uint32_t a1 = (v1 & 0x00FF00FFu) ^ 0x00800080u;
            const uint32_t a2 = ((v0 >> 8) & 0x00FF00FFu) ^ 0x00800080u;
            const uint32_t a3 = ((v1 >> 8) & 0x00FF00FFu) ^ 0x00800080u;
            mma_bf16(D[gg], a0, a1, a2, a3, Q.br0[2 * gg + half], Q.br1[2 * gg + half]);
        }
    }
}

// Residual correction sm * sum_g r_scale_g q_g . c8_g of accumulator entry e.
__device__ __forceinline__ float corr_score(const float (&D)[4][4], int e, const float (&sr)[4],
                                            const float (&qs)[4], float sm) {
    float acc = 0.0f;
#pragma unroll
    for (int gg = 0; gg < 4; gg++)
        acc = fmaf(sr[gg], fmaf(kUnscale, D[gg][e], -128.0f * qs[gg]), acc);
    return acc * sm;
}


// Exact scores s = sm * q . K^ (thumbnail plus residual) of rows r0 and r1 of a block whose
// thumbnail and residual records are at trec and rrec (global or shared memory), for heads 2tig,
// 2tig+1: {(r0,h0), (r0,h1), (r1,h0), (r1,h1)}.
__device__ __forceinline__ float4 exact_tile(const uint8_t *trec, const uint8_t *rrec, int r0,
                                             int r1, int tig, const ThumbOps &Q,
                                             const ResidOps &QR, float sm) {
    uint32_t w0[8], w1[8];
    {
        const uint4 *c0 = reinterpret_cast<const uint4 *>(trec + r0 * kThumbRow);
        const uint4 *c1 = reinterpret_cast<const uint4 *>(trec + r1 * kThumbRow);
        const uint4 p0 = c0[0], p1 = c0[1], p2 = c1[0], p3 = c1[1];
        w0[0] = p0.x; w0[1] = p0.y; w0[2] = p0.z; w0[3] = p0.w;
        w0[4] = p1.x; w0[5] = p1.y; w0[6] = p1.z; w0[7] = p1.w;
        w1[0] = p2.x; w1[1] = p2.y; w1[2] = p2.z; w1[3] = p2.w;
        w1[4] = p3.x; w1[5] = p3.y; w1[6] = p3.z; w1[7] = p3.w;
    }
    uint2 x0[4], x1[4];
#pragma unroll
    for (int gg = 0; gg < 4; gg++) {
        x0[gg] = *reinterpret_cast<const uint2 *>(rrec + resid_offset(r0, 32 * gg + 8 * tig));
        x1[gg] = *reinterpret_cast<const uint2 *>(rrec + resid_offset(r1, 32 * gg + 8 * tig));
    }
    float sf0[4], sf1[4], zf0[4], zf1[4], sr0[4], sr1[4];
    const uint2 *ts = reinterpret_cast<const uint2 *>(trec + kThumbScaleOff);
    const uint2 *tz = reinterpret_cast<const uint2 *>(trec + kThumbZeroOff);
    const uint2 *rs = reinterpret_cast<const uint2 *>(rrec + kResidScaleOff);
    unpack4h(ts[r0], sf0);
    unpack4h(ts[r1], sf1);
    unpack4h(tz[r0], zf0);
    unpack4h(tz[r1], zf1);
    unpack4h(rs[r0], sr0);
    unpack4h(rs[r1], sr1);
    float D[4][4], Dr[4][4];
    thumb_mma(D, w0, w1, 0x00030003u << (2 * tig), Q);
    resid_mma(Dr, x0, x1, QR);
    float4 e;
    e.x = est_score(D, 0, sf0, zf0, Q.qs[0], sm) + corr_score(Dr, 0, sr0, Q.qs[0], sm);
    e.y = est_score(D, 1, sf0, zf0, Q.qs[1], sm) + corr_score(Dr, 1, sr0, Q.qs[1], sm);
    e.z = est_score(D, 2, sf1, zf1, Q.qs[0], sm) + corr_score(Dr, 2, sr1, Q.qs[0], sm);
    e.w = est_score(D, 3, sf1, zf1, Q.qs[1], sm) + corr_score(Dr, 3, sr1, Q.qs[1], sm);
    return e;
}

}  // namespace ffd
