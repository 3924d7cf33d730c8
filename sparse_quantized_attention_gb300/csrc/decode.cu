// decode.cu -- FFD decode attention: stage 1 (pseudo-max), fused stage 2 + 3 (Top-delta scan and
// refinement over kept blocks, split-KV online softmax), and the log-sum-exp merge.
//
// Source: "Faster Than Flash", Methodology §2 (Top-delta rule s_ij >= m~_i - delta, pseudo-max
// from sink and local tokens) and §3 (three-stage fused kernel: pseudo-max estimation; stream the
// 2-bit keys, compute provisional scores and filter blocks; load the 8-bit residuals and V of the
// selected blocks and compute exact attention). The split-KV online softmax with a log-sum-exp
// merge is the flash-decoding scheme the method's name refers to.
#include "common.cuh"

namespace ffd {

// ------------------------------------------------------------------------------------------
// Stage 1: one CTA per (forced-block slot, sequence x KV head). Exact scores
// s = sm * q . K^ (K^ = thumbnail + residual) of the sink / local tokens of one block; writes the
// per-head maximum of the block to ws_m1. 128 threads: token t = tid/2, channel half tid%2.
// ------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(128) stage1_kernel(DecodeArgs a) {
    __shared__ float qs[kMaxG][kD + 4];
    __shared__ float red[4][kMaxG];
    const int bh = blockIdx.y;
    const int b = bh / a.Hkv, h = bh % a.Hkv;
    const int slot = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = checked_seq_len(a, b);
    const ForcedBlocks fb(n, a.S, a.L);
    float *dst = a.ws_m1 + ((size_t)bh * a.nf + slot) * kMaxG;
    int page = -1;
    if (slot < fb.count) {
        page = a.block_table[(size_t)b * a.max_blocks + fb.block(slot)];
        if (page < 0 || page >= a.P) {
            if (tid == 0) raise_error(a.err, FFD_ERRBIT_BOUNDS);
            page = -1;
        }
    }
    if (page < 0) {
        if (tid < kMaxG) dst[tid] = -INFINITY;
        return;
    }
    const int blk = fb.block(slot);
    for (int idx = tid; idx < a.G * kD; idx += blockDim.x) {
        const int i = idx / kD, c = idx % kD;
        qs[i][c] = __bfloat162float(a.q[((size_t)b * a.Hq + h * a.G + i) * kD + c]);
    }
    __syncthreads();

    const int t = tid >> 1, hf = tid & 1;
    const int j = blk * kPage + t;
    const bool valid = j < n && (j < a.S || j >= n - a.L);
    const size_t row = ((size_t)page * a.Hkv + h) * kPage + t;
    float acc[kMaxG];
#pragma unroll
    for (int i = 0; i < kMaxG; i++) acc[i] = 0.0f;
#pragma unroll
    for (int gg = 0; gg < 2; gg++) {
        const int g = 2 * hf + gg;
        const float sf = __half2float(a.t_scale[row * kGroups + g]);
        const float zf = __half2float(a.t_zero[row * kGroups + g]);
        const float sr = __half2float(a.r_scale[row * kGroups + g]);
        const uint2 cw = *reinterpret_cast<const uint2 *>(a.thumb + row * kThumbRow + g * 8);
        const int4 *rp = reinterpret_cast<const int4 *>(a.resid + row * kD + g * kGroupSize);
        int4 r8[2] = {rp[0], rp[1]};
        const int8_t *r8b = reinterpret_cast<const int8_t *>(r8);
#pragma unroll
        for (int c = 0; c < kGroupSize; c++) {
            const uint32_t word = c < 16 ? cw.x : cw.y;
            const float code = (float)((word >> (2 * (c & 15))) & 3u);
            const float x2 = __fmaf_rn(code, sf, zf);
            const float kh = __fmaf_rn((float)r8b[c], sr, x2);
#pragma unroll
            for (int i = 0; i < kMaxG; i++)
                if (i < a.G) acc[i] = fmaf(qs[i][g * kGroupSize + c], kh, acc[i]);
        }
    }
#pragma unroll
    for (int i = 0; i < kMaxG; i++) {
        acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], 1);
        float s = valid ? acc[i] * a.sm_scale : -INFINITY;
        s = warp_max(s);
        if (lane == 0) red[warp][i] = s;
    }
    __syncthreads();
    if (tid < a.G)
        dst[tid] = fmaxf(fmaxf(red[0][tid], red[1][tid]), fmaxf(red[2][tid], red[3][tid]));
    else if (tid < kMaxG)
        dst[tid] = -INFINITY;
}

// ------------------------------------------------------------------------------------------
// Stages 2 + 3, one CTA per (split, sequence x KV head); 128 threads.
//   scan:   token t = tid/2 and channel half tid%2 compute the provisional score from the 2-bit
//           thumbnail, group-factored: s^ = sm * sum_g (scale_g * (q_g . c_g) + zero_g * sum q_g).
//   filter: the block is kept when any valid token of any head reaches m~ - delta, or when it is
//           a sink / local block.
//   refine: s = s^ + sm * sum_g r_scale_g * (q_g . c8_g) (the scan result is reused); online
//           softmax per head; PV with thread = (channel pair, half of the heads).
// ------------------------------------------------------------------------------------------
template <int G>
__global__ void __launch_bounds__(128) main_kernel(DecodeArgs a) {
    __shared__ float qs[G][kD + 4];
    __shared__ float qsum[G][kGroups];
    __shared__ float thr[G];
    __shared__ float sp[kPage][G + 1];  // scores, then probabilities
    __shared__ float m_run[G], l_run[G], alpha[G];

    const int bh = blockIdx.y;
    const int split = blockIdx.x;
    const int b = bh / a.Hkv, h = bh % a.Hkv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = checked_seq_len(a, b);
    const ForcedBlocks fb(n, a.S, a.L);
    const int blk0 = split * a.blk_per_split;
    const int blk_end = min(blk0 + a.blk_per_split, a.max_blocks);
    const int blk1 = min(blk_end, fb.nb);

    for (int idx = tid; idx < G * kD; idx += blockDim.x) {
        const int i = idx / kD, c = idx % kD;
        qs[i][c] = __bfloat162float(a.q[((size_t)b * a.Hq + h * G + i) * kD + c]);
    }
    if (tid < G) {
        float m = -INFINITY;
        for (int s = 0; s < a.nf; s++) m = fmaxf(m, a.ws_m1[((size_t)bh * a.nf + s) * kMaxG + tid]);
        thr[tid] = m - a.delta;  // -inf when delta = +inf or no sink/local token exists
        m_run[tid] = -INFINITY;
        l_run[tid] = 0.0f;
        if (split == 0 && a.m_tilde) a.m_tilde[(size_t)b * a.Hq + h * G + tid] = m;
    }
    if (a.keep_mask)
        for (int blk = max(blk0, fb.nb) + tid; blk < blk_end; blk += blockDim.x)
            a.keep_mask[(size_t)bh * a.max_blocks + blk] = 0;
    __syncthreads();
    if (tid < G * kGroups) {
        const int i = tid / kGroups, g = tid % kGroups;
        float s = 0.0f;
        for (int c = 0; c < kGroupSize; c++) s += qs[i][g * kGroupSize + c];
        qsum[i][g] = s;
    }
    __syncthreads();

    const int t = tid >> 1, hf = tid & 1;
    const int dp = tid & 63, hh = tid >> 6;  // PV mapping: channel pair, head half
    float o[4][2];
#pragma unroll
    for (int k = 0; k < 4; k++) o[k][0] = o[k][1] = 0.0f;

    for (int blk = blk0; blk < blk1; blk++) {
        int page = a.block_table[(size_t)b * a.max_blocks + blk];
        if (page < 0 || page >= a.P) {  // uniform across the CTA
            if (tid == 0) {
                raise_error(a.err, FFD_ERRBIT_BOUNDS);
                if (a.keep_mask) a.keep_mask[(size_t)bh * a.max_blocks + blk] = 0;
            }
            continue;
        }
        const size_t row = ((size_t)page * a.Hkv + h) * kPage + t;
        const int j = blk * kPage + t;
        const bool valid = j < n;

        // ---- stage 2: provisional scores from the thumbnail
        float est[G];
#pragma unroll
        for (int i = 0; i < G; i++) est[i] = 0.0f;
#pragma unroll
        for (int gg = 0; gg < 2; gg++) {
            const int g = 2 * hf + gg;
            const float sf = __half2float(a.t_scale[row * kGroups + g]);
            const float zf = __half2float(a.t_zero[row * kGroups + g]);
            const uint2 cw = *reinterpret_cast<const uint2 *>(a.thumb + row * kThumbRow + g * 8);
            float acc[G];
#pragma unroll
            for (int i = 0; i < G; i++) acc[i] = 0.0f;
#pragma unroll
            for (int c = 0; c < kGroupSize; c++) {
                const uint32_t word = c < 16 ? cw.x : cw.y;
                const float code = (float)((word >> (2 * (c & 15))) & 3u);
#pragma unroll
                for (int i = 0; i < G; i++) acc[i] = fmaf(qs[i][g * kGroupSize + c], code, acc[i]);
            }
#pragma unroll
            for (int i = 0; i < G; i++) est[i] = fmaf(sf, acc[i], fmaf(zf, qsum[i][g], est[i]));
        }
        bool pass = false;
#pragma unroll
        for (int i = 0; i < G; i++) {
            est[i] += __shfl_xor_sync(0xffffffffu, est[i], 1);
            pass |= valid && (est[i] * a.sm_scale >= thr[i]);
        }
        const bool keep = __syncthreads_or(pass) || fb.forced(blk);
        if (a.keep_mask && tid == 0) a.keep_mask[(size_t)bh * a.max_blocks + blk] = keep ? 1 : 0;
        if (!keep) continue;

        // ---- stage 3: residual correction, exact scores
        float corr[G];
#pragma unroll
        for (int i = 0; i < G; i++) corr[i] = 0.0f;
#pragma unroll
        for (int gg = 0; gg < 2; gg++) {
            const int g = 2 * hf + gg;
            const float sr = __half2float(a.r_scale[row * kGroups + g]);
            const int4 *rp = reinterpret_cast<const int4 *>(a.resid + row * kD + g * kGroupSize);
            int4 r8[2] = {rp[0], rp[1]};
            const int8_t *r8b = reinterpret_cast<const int8_t *>(r8);
            float acc[G];
#pragma unroll
            for (int i = 0; i < G; i++) acc[i] = 0.0f;
#pragma unroll
            for (int c = 0; c < kGroupSize; c++) {
                const float c8 = (float)r8b[c];
#pragma unroll
                for (int i = 0; i < G; i++) acc[i] = fmaf(qs[i][g * kGroupSize + c], c8, acc[i]);
            }
#pragma unroll
            for (int i = 0; i < G; i++) corr[i] = fmaf(sr, acc[i], corr[i]);
        }
#pragma unroll
        for (int i = 0; i < G; i++) {
            corr[i] += __shfl_xor_sync(0xffffffffu, corr[i], 1);
            const float s = valid ? (est[i] + corr[i]) * a.sm_scale : -INFINITY;
            if (hf == 0) sp[t][i] = s;
        }
        __syncthreads();

        // ---- online softmax bookkeeping: warp w handles heads w, w+4
        for (int i = warp; i < G; i += 4) {
            const float v0 = sp[lane][i], v1 = sp[lane + 32][i];
            const float mb = warp_max(fmaxf(v0, v1));
            const float m_old = m_run[i];
            const float m_new = fmaxf(m_old, mb);
            const float al = m_old == -INFINITY ? 0.0f : exp2f((m_old - m_new) * 1.4426950408889634f);
            const float p0 = v0 == -INFINITY ? 0.0f : exp2f((v0 - m_new) * 1.4426950408889634f);
            const float p1 = v1 == -INFINITY ? 0.0f : exp2f((v1 - m_new) * 1.4426950408889634f);
            sp[lane][i] = p0;
            sp[lane + 32][i] = p1;
            const float ps = warp_sum(p0 + p1);
            __syncwarp();
            if (lane == 0) {
                l_run[i] = l_run[i] * al + ps;
                m_run[i] = m_new;
                alpha[i] = al;
            }
        }
        __syncthreads();

        // ---- PV
        const __nv_bfloat16 *vrow = a.v + ((size_t)page * a.Hkv + h) * kPage * kD + 2 * dp;
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const int i = hh * 4 + k;
            if (i < G) {
                o[k][0] *= alpha[i];
                o[k][1] *= alpha[i];
            }
        }
        for (int tt = 0; tt < kPage; tt++) {
            const float2 vf = __bfloat1622float2(
                *reinterpret_cast<const __nv_bfloat162 *>(vrow + (size_t)tt * kD));
#pragma unroll
            for (int k = 0; k < 4; k++) {
                const int i = hh * 4 + k;
                if (i < G) {
                    const float p = sp[tt][i];
                    o[k][0] = fmaf(p, vf.x, o[k][0]);
                    o[k][1] = fmaf(p, vf.y, o[k][1]);
                }
            }
        }
        __syncthreads();
    }

    float *part = a.ws_part + ((size_t)bh * a.splits + split) * G * kPartStride;
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const int i = hh * 4 + k;
        if (i < G) {
            part[i * kPartStride + 2 * dp] = o[k][0];
            part[i * kPartStride + 2 * dp + 1] = o[k][1];
        }
    }
    if (tid < G) {
        part[tid * kPartStride + kD] = m_run[tid];
        part[tid * kPartStride + kD + 1] = l_run[tid];
    }
}

// ------------------------------------------------------------------------------------------
// Log-sum-exp merge of the split partials: out = sum_s e^(m_s - M) o_s / sum_s e^(m_s - M) l_s.
// One CTA per (sequence, query head); thread = channel. Shared by the dense kernel.
// ------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(128) merge_kernel(DecodeArgs a) {
    const int bq = blockIdx.x;
    const int b = bq / a.Hq, qh = bq % a.Hq;
    const int h = qh / a.G, i = qh % a.G;
    const int bh = b * a.Hkv + h;
    const int c = threadIdx.x;
    const float *part = a.ws_part + (size_t)bh * a.splits * a.G * kPartStride + i * kPartStride;
    const size_t split_stride = (size_t)a.G * kPartStride;
    float M = -INFINITY;
    for (int s = 0; s < a.splits; s++) M = fmaxf(M, part[s * split_stride + kD]);
    float num = 0.0f, den = 0.0f;
    if (M != -INFINITY) {
        for (int s = 0; s < a.splits; s++) {
            const float m = part[s * split_stride + kD];
            if (m == -INFINITY) continue;
            const float w = exp2f((m - M) * 1.4426950408889634f);
            den = fmaf(w, part[s * split_stride + kD + 1], den);
            num = fmaf(w, part[s * split_stride + c], num);
        }
    }
    a.out[(size_t)bq * kD + c] = den > 0.0f ? num / den : 0.0f;
}

template <int G>
static void launch_main(const DecodeArgs &a, cudaStream_t stream) {
    main_kernel<G><<<dim3(a.splits, a.B * a.Hkv), 128, 0, stream>>>(a);
}

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream) {
    if (a.nf > 0) stage1_kernel<<<dim3(a.nf, a.B * a.Hkv), 128, 0, stream>>>(a);
    if (a.prof_start) cudaEventRecord(a.prof_start, stream);
    switch (a.G) {
        case 1: launch_main<1>(a, stream); break;
        case 2: launch_main<2>(a, stream); break;
        case 3: launch_main<3>(a, stream); break;
        case 4: launch_main<4>(a, stream); break;
        case 5: launch_main<5>(a, stream); break;
        case 6: launch_main<6>(a, stream); break;
        case 7: launch_main<7>(a, stream); break;
        case 8: launch_main<8>(a, stream); break;
        default: return cudaErrorInvalidValue;
    }
    if (a.prof_stop) cudaEventRecord(a.prof_stop, stream);
    merge_kernel<<<a.B * a.Hq, kD, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_merge(const DecodeArgs &a, cudaStream_t stream) {
    merge_kernel<<<a.B * a.Hq, kD, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace ffd
