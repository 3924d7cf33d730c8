// quant.cuh -- the per-group quantiser shared by the whole-cache quantiser and the append kernel:
// one thread turns the 32 bf16 keys of one channel group of one token into the group's 2-bit
// thumbnail codes, fp16 scale and zero, int8 residual codes and fp16 residual scale, and stores
// them into the (page, KV head) records.
//
// Source: "Faster Than Flash", Methodology §1 (2-bit thumbnails for score estimation, 8-bit
// residuals that rebuild the keys close to fp16 precision); the format is the one include/ffd.h
// states.
//
// Every arithmetic step is a single IEEE fp32 operation with an explicit rounding intrinsic, so
// the outputs are bit-defined. The per-channel code needs round-half-even of the correctly
// rounded quotient (x - zero) / scale (and r / r_scale), without an IEEE division per channel:
// the 2-bit code counts the exact rounding boundaries (k + 1/2) scale below x - zero; the int8
// code is formed from a correctly rounded reciprocal, with the clamp folded into a saturating
// multiply, and rounded with one fused multiply-add, and where that fast quotient lies within a
// few ulps of a rounding boundary (ties are frequent: keys, zeros and scales sit on the bf16 /
// fp16 grids) the side of the boundary is decided exactly (boundary_step below). The adds and
// fused multiply-adds run two channels at a time on the packed fp32 pipe (f32x2: IEEE
// round-to-nearest in each lane, so every lane's result is the scalar operation's).
#pragma once

#include "common.cuh"

namespace ffd {
namespace quant {

// 1.5 * 2^23: adding it to |t| < 2^22 rounds t to an integer half-to-even (the sum's ulp is 1),
// and the integer is then the sum's low mantissa bits (two's complement for t < 0).
constexpr float kMagic = 12582912.0f;
// kMagic - 127, the base of the residual codes' sums (its low byte is 0x81 = -127 mod 256)
constexpr float kMagicB = 12582785.0f;
// Half-width of the window around k + 1/2 in which the fast residual quotient is not trusted: it
// evaluates r / r_scale as 254 sat(r * rcp(254 r_scale) + 1/2) - 127, with an error below
// 1.6e-5 on [-127, 127].
constexpr float kNearB = 4.0e-5f;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// x / b rounded to nearest, for x >= 0 and a divisor b with c = RN(1/b), without an IEEE division
// in the common case: q0 = RN(x c) lies within an ulp of x / b, the remainder x - q0 b is exact in
// one fused multiply-add, and one more fused multiply-add rounds the quotient correctly
// (Markstein's correction step with a precomputed reciprocal). For b = 3 and b = 127 the result
// equals the IEEE quotient for every finite non-negative fp32 x (tests/test_gpu_quant_division.py
// checks all of them); a non-finite x takes the IEEE division.
constexpr float kThird = 1.0f / 3.0f;    // RN(1/3)
constexpr float kInv127 = 1.0f / 127.0f; // RN(1/127)
__device__ __forceinline__ float div_const(float x, float b, float c) {
    if (!(x <= 3.4028234663852886e38f)) return __fdiv_rn(x, b);  // +inf or NaN
    const float q0 = __fmul_rn(x, c);
    const float r = __fmaf_rn(-q0, b, x);
    return __fmaf_rn(r, c, q0);
}

// Exact rounding near a boundary. With t the fast quotient of a / b and c = rint(t), the only
// rounding boundary within reach is k = c + 1/2 sign(t - c); k * b is exact in fp32 (k has at
// most 9 significant bits, b is an fp16 value), so e = a - k b, formed by one fused multiply-add,
// has the exact sign of a / b - k. Because a and b lie on the fp32 and fp16 grids, the IEEE
// quotient rounds onto k only when a / b == k exactly (e == 0, a tie: half to even); otherwise
// it lies on the same side of k as a / b. Returns the step (-1, 0, +1) to add to c.
__device__ __forceinline__ float boundary_step(float a, float b, float c, float d, bool c_odd) {
    const float dir = copysignf(1.0f, d);
    const float e = __fmaf_rn(-__fadd_rn(c, 0.5f * dir), b, a);
    if (e == 0.0f) return c_odd ? dir : 0.0f;
    return (e > 0.0f) == (d > 0.0f) ? dir : 0.0f;
}

// The quantised form of one group of 32 channels of one token.
struct GroupCodes {
    uint32_t codes[2];   // 2-bit codes, channel c of the group at bit 2c of the 64-bit pair
    uint32_t packed[8];  // int8 residual codes, channel c in byte c % 4 of word c / 4
    __half scale, zero, rscale;
    bool bad;            // a key outside the fp16 range, or NaN
};

__device__ __forceinline__ void load_words(const __nv_bfloat16 *src, uint32_t (&u)[16]) {
    const uint4 *p = reinterpret_cast<const uint4 *>(src);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const uint4 w = __ldg(p + i);
        u[4 * i] = w.x;
        u[4 * i + 1] = w.y;
        u[4 * i + 2] = w.z;
        u[4 * i + 3] = w.w;
    }
}

// Group scale and zero (and the range check) from the 32 keys in u (word m: channels 2m in the
// low half, 2m+1 in the high half).
__device__ __forceinline__ void group_params(const uint32_t (&u)[16], GroupCodes &o) {
    // the NaN-propagating forms let the range check see a NaN key
    __nv_bfloat162 mn2 = *reinterpret_cast<const __nv_bfloat162 *>(&u[0]);
    __nv_bfloat162 mx2 = mn2;
#pragma unroll
    for (int m = 1; m < 16; m++) {
        const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(&u[m]);
        mn2 = __hmin2_nan(mn2, v);
        mx2 = __hmax2_nan(mx2, v);
    }
    float mn = __bfloat162float(__hmin_nan(mn2.x, mn2.y));
    float mx = __bfloat162float(__hmax_nan(mx2.x, mx2.y));
    o.bad = !(fabsf(mn) < 65504.0f) || !(fabsf(mx) < 65504.0f);
    if (mn == 0.0f) mn = 0.0f;  // a signed-zero extreme counts as +0
    if (mx == 0.0f) mx = 0.0f;
    o.zero = __float2half_rn(mn);
    o.scale = __float2half_rn(div_const(__fsub_rn(mx, mn), 3.0f, kThird));
}

// 2-bit code of a = x - zero: the number of rounding boundaries (k + 1/2) scale below a (b0, b1,
// b2), exact in fp32. On these grids the IEEE quotient a / scale lies on the same side of k + 1/2
// as a lies of (k + 1/2) scale, and equals k + 1/2 only when a does (see boundary_step), so a tie
// at 1/2 or 5/2 rounds down and a tie at 3/2 rounds up (half to even). scale 0 gives code 0.
__device__ __forceinline__ float code2_of(float a, float b0, float b1, float b2) {
    return (a > b0 ? 1.0f : 0.0f) + (a >= b1 ? 1.0f : 0.0f) + (a > b2 ? 1.0f : 0.0f);
}

// The int8 codes clamp(rint(r / r_scale), -127, 127) of two residuals r, in the low byte of each
// result (two's complement), from r254 = rcp(254 r_scale) (0 when r_scale is 0): the clamp is the
// saturation of tp = r r254 + 1/2, and tp * 254 + kMagicB rounds to kMagicB + code + 127. The
// distance to the nearest rounding boundary is formed negated (e = -d, exactly, as rounding is
// symmetric), and the exact side test runs only for a lane within kNearB of a boundary.
__device__ __forceinline__ void code8_pair(float2 r, float rscale, float r254, uint32_t &b0,
                                           uint32_t &b1) {
    const float2 tp = make_float2(__saturatef(__fmaf_rn(r.x, r254, 0.5f)),
                                  __saturatef(__fmaf_rn(r.y, r254, 0.5f)));
    float2 cm = __ffma2_rn(tp, make_float2(254.0f, 254.0f), make_float2(kMagicB, kMagicB));
    const float2 q = __fadd2_rn(cm, make_float2(-kMagicB, -kMagicB));  // code + 127, exact
    const float2 e = __ffma2_rn(tp, make_float2(-254.0f, -254.0f), q);
    const bool near_x = fabsf(e.x) > 0.5f - kNearB, near_y = fabsf(e.y) > 0.5f - kNearB;
    if (near_x | near_y) {  // one branch for the pair; rarely taken
        if (near_x) {
            const float code = __fsub_rn(cm.x, kMagic);  // exact
            cm.x = __fadd_rn(cm.x, boundary_step(r.x, rscale, code, -e.x,
                                                  (__float_as_uint(cm.x) & 1u) != 0));
        }
        if (near_y) {
            const float code = __fsub_rn(cm.y, kMagic);
            cm.y = __fadd_rn(cm.y, boundary_step(r.y, rscale, code, -e.y,
                                                  (__float_as_uint(cm.y) & 1u) != 0));
        }
    }
    b0 = __float_as_uint(cm.x);
    b1 = __float_as_uint(cm.y);
}

// Quantise the group held in u (word m: channels 2m in the low half, 2m+1 in the high half).
__device__ __forceinline__ void quantize_group(const uint32_t (&u)[16], GroupCodes &o) {
    group_params(u, o);
    const float zf = __half2float(o.zero);
    const float sf = __half2float(o.scale);
    const float b0 = sf == 0.0f ? INFINITY : __fmul_rn(0.5f, sf);
    const float b1 = sf == 0.0f ? INFINITY : __fmul_rn(1.5f, sf);
    const float b2 = sf == 0.0f ? INFINITY : __fmul_rn(2.5f, sf);

    // stage A: 2-bit codes and the residual r = x - x^2, two channels (one word) at a time. The
    // codes are summed as code * 4^c in fp32 (exact: each sum stays below 2^24; even and odd
    // channels in separate lanes, added at the end), 12 + 4 channels per 32-bit word; both
    // channels of a word fall in the same part.
    float2 acc[4];
#pragma unroll
    for (int p = 0; p < 4; p++) acc[p] = make_float2(0.0f, 0.0f);
    float2 r[16];
    float amax = 0.0f;
#pragma unroll
    for (int m = 0; m < 16; m++) {
        const int c = 2 * m;
        const float2 x = make_float2(bf16_lo(u[m]), bf16_hi(u[m]));
        const float2 a = __fadd2_rn(x, make_float2(-zf, -zf));  // x - zero
        const float2 code = make_float2(code2_of(a.x, b0, b1, b2), code2_of(a.y, b0, b1, b2));
        const int part = (c >> 4) * 2 + ((c & 15) >= 12);
        const float w0 = (float)(1u << (2 * ((c & 15) % 12)));
        acc[part] = __ffma2_rn(code, make_float2(w0, 4.0f * w0), acc[part]);
        // r = x - (code * scale + zero); the negated product-sum is exact negation
        r[m] = __fadd2_rn(x, __ffma2_rn(code, make_float2(-sf, -sf), make_float2(-zf, -zf)));
        amax = fmaxf(amax, fmaxf(fabsf(r[m].x), fabsf(r[m].y)));
    }
    o.codes[0] = __float2uint_rn(__fadd_rn(acc[0].x, acc[0].y)) |
                 (__float2uint_rn(__fadd_rn(acc[1].x, acc[1].y)) << 24);
    o.codes[1] = __float2uint_rn(__fadd_rn(acc[2].x, acc[2].y)) |
                 (__float2uint_rn(__fadd_rn(acc[3].x, acc[3].y)) << 24);

    o.rscale = __float2half_rn(div_const(amax, 127.0f, kInv127));
    const float sr = __half2float(o.rscale);
    const float r254 = sr == 0.0f ? 0.0f : __frcp_rn(__fmul_rn(sr, 254.0f));  // exact product

    // stage B: symmetric int8 residual codes, four channels per word
#pragma unroll
    for (int w = 0; w < 8; w++) {
        uint32_t b[4];
        code8_pair(r[2 * w], sr, r254, b[0], b[1]);
        code8_pair(r[2 * w + 1], sr, r254, b[2], b[3]);
        o.packed[w] = __byte_perm(__byte_perm(b[0], b[1], 0x0040),
                                  __byte_perm(b[2], b[3], 0x0040), 0x5410);
    }
}

// Write group g of token `row` into the tile's thumbnail and residual records.
__device__ __forceinline__ void store_group(const GroupCodes &o, uint8_t *trec, uint8_t *rrec,
                                            int row, int g) {
    *reinterpret_cast<uint2 *>(trec + row * kThumbRow + 8 * g) = make_uint2(o.codes[0], o.codes[1]);
    // residual chunk j = 2g + s (channels 16 j .. 16 j + 15) is stored at chunk j ^ (row % 8)
#pragma unroll
    for (int s = 0; s < 2; s++) {
        const int j = 2 * g + s;
        *reinterpret_cast<uint4 *>(rrec + row * kD + 16 * (j ^ (row & 7))) = make_uint4(
            o.packed[4 * s], o.packed[4 * s + 1], o.packed[4 * s + 2], o.packed[4 * s + 3]);
    }
    reinterpret_cast<__half *>(trec + kThumbScaleOff)[row * kGroups + g] = o.scale;
    reinterpret_cast<__half *>(trec + kThumbZeroOff)[row * kGroups + g] = o.zero;
    reinterpret_cast<__half *>(rrec + kResidScaleOff)[row * kGroups + g] = o.rscale;
}

// Append one channel group g of the new token of sequence b, KV head h: the token goes to row
// p % 64 of page block_table[b][p / 64], p = positions[b] (negative: nothing to append). Its key
// group is quantised into the records; its value group (and, with k_cache, its raw key group) is
// copied into the row. A position past the block table's row or a page outside [0, P) raises
// FFD_ERRBIT_BOUNDS and writes nothing; a key outside the fp16 range raises FFD_ERRBIT_RANGE.
__device__ __forceinline__ void append_group(int b, int h, int g, int Hkv, int P, int max_blocks,
                                             const int32_t *positions, const int32_t *block_table,
                                             const __nv_bfloat16 *k_new,
                                             const __nv_bfloat16 *v_new, uint8_t *thumb,
                                             uint8_t *resid, __nv_bfloat16 *v_cache,
                                             __nv_bfloat16 *k_cache, int *err) {
    const int pos = positions[b];
    if (pos < 0) return;  // no token for this sequence in this step
    if (pos >= max_blocks * kPage) {
        if (g == 0 && h == 0) raise_error(err, FFD_ERRBIT_BOUNDS);
        return;
    }
    const int page = block_table[(int64_t)b * max_blocks + pos / kPage];
    if (page < 0 || page >= P) {
        if (g == 0 && h == 0) raise_error(err, FFD_ERRBIT_BOUNDS);
        return;
    }
    const int row = pos % kPage;
    const int64_t tile = (int64_t)page * Hkv + h;
    const int64_t src = ((int64_t)b * Hkv + h) * kD;
    const int64_t dst = (tile * kPage + row) * kD;
    uint32_t u[16];
    load_words(k_new + src + 32 * g, u);
    GroupCodes o;
    quantize_group(u, o);
    if (o.bad) raise_error(err, FFD_ERRBIT_RANGE);
    store_group(o, thumb + tile * kThumbRec, resid + tile * kResidRec, row, g);
    const uint4 *vs = reinterpret_cast<const uint4 *>(v_new + src + 32 * g);
    uint4 *vd = reinterpret_cast<uint4 *>(v_cache + dst + 32 * g);
#pragma unroll
    for (int i = 0; i < 4; i++) vd[i] = __ldg(vs + i);
    if (k_cache) {
        uint4 *kd = reinterpret_cast<uint4 *>(k_cache + dst + 32 * g);
#pragma unroll
        for (int i = 0; i < 4; i++)
            kd[i] = make_uint4(u[4 * i], u[4 * i + 1], u[4 * i + 2], u[4 * i + 3]);
    }
}

}  // namespace quant
}  // namespace ffd
