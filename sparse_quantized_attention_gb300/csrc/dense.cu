// dense.cu -- dense bf16 flash-decode attention, the in-library comparison for FFD.
//
// Source: the pages compare FFD with FlashAttention-2 decoding ("Faster Than Flash", Main results:
// kernel speedup and end-to-end throughput). This kernel computes plain softmax attention over
// every cached token with the original bf16 keys, split over the KV sequence with the same
// partial format and log-sum-exp merge as the FFD path.
#include "common.cuh"

namespace ffd {

template <int G>
__global__ void __launch_bounds__(128) dense_kernel(DecodeArgs a) {
    __shared__ float qs[G][kD + 4];
    __shared__ float sp[kPage][G + 1];
    __shared__ float m_run[G], l_run[G], alpha[G];

    const int bh = blockIdx.y;
    const int split = blockIdx.x;
    const int b = bh / a.Hkv, h = bh % a.Hkv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = checked_seq_len(a, b);
    const int nb = (n + kPage - 1) / kPage;
    const int blk0 = split * a.blk_per_split;
    const int blk1 = min(min(blk0 + a.blk_per_split, a.max_blocks), nb);

    for (int idx = tid; idx < G * kD; idx += blockDim.x) {
        const int i = idx / kD, c = idx % kD;
        qs[i][c] = __bfloat162float(a.q[((size_t)b * a.Hq + h * G + i) * kD + c]);
    }
    if (tid < G) {
        m_run[tid] = -INFINITY;
        l_run[tid] = 0.0f;
    }
    __syncthreads();

    const int t = tid >> 1, hf = tid & 1;
    const int dp = tid & 63, hh = tid >> 6;
    float o[4][2];
#pragma unroll
    for (int k = 0; k < 4; k++) o[k][0] = o[k][1] = 0.0f;

    for (int blk = blk0; blk < blk1; blk++) {
        const int page = a.block_table[(size_t)b * a.max_blocks + blk];
        if (page < 0 || page >= a.P) {
            if (tid == 0) raise_error(a.err, FFD_ERRBIT_BOUNDS);
            continue;
        }
        const size_t tile = (size_t)page * a.Hkv + h;
        const int j = blk * kPage + t;
        const bool valid = j < n;
        const uint4 *kp = reinterpret_cast<const uint4 *>(a.k + (tile * kPage + t) * kD + hf * 64);
        float acc[G];
#pragma unroll
        for (int i = 0; i < G; i++) acc[i] = 0.0f;
#pragma unroll
        for (int w = 0; w < 8; w++) {
            const uint4 raw = kp[w];
            const uint32_t wd[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const float k0 = __uint_as_float(wd[e] << 16);
                const float k1 = __uint_as_float(wd[e] & 0xffff0000u);
                const int c = hf * 64 + w * 8 + e * 2;
#pragma unroll
                for (int i = 0; i < G; i++) {
                    acc[i] = fmaf(qs[i][c], k0, acc[i]);
                    acc[i] = fmaf(qs[i][c + 1], k1, acc[i]);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < G; i++) {
            acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], 1);
            if (hf == 0) sp[t][i] = valid ? acc[i] * a.sm_scale : -INFINITY;
        }
        __syncthreads();
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
        const __nv_bfloat16 *vrow = a.v + tile * kPage * kD + 2 * dp;
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

// Log-sum-exp merge of the split partials: out = sum_s e^(m_s - M) o_s / sum_s e^(m_s - M) l_s.
// One CTA per (sequence, query head); thread = channel.
__global__ void __launch_bounds__(128) dense_merge_kernel(DecodeArgs a) {
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
static void launch_dense_g(const DecodeArgs &a, cudaStream_t stream) {
    dense_kernel<G><<<dim3(a.splits, a.B * a.Hkv), 128, 0, stream>>>(a);
}

cudaError_t launch_dense(const DecodeArgs &a, cudaStream_t stream) {
    if (a.prof_start) cudaEventRecord(a.prof_start, stream);
    switch (a.G) {
        case 1: launch_dense_g<1>(a, stream); break;
        case 2: launch_dense_g<2>(a, stream); break;
        case 3: launch_dense_g<3>(a, stream); break;
        case 4: launch_dense_g<4>(a, stream); break;
        case 5: launch_dense_g<5>(a, stream); break;
        case 6: launch_dense_g<6>(a, stream); break;
        case 7: launch_dense_g<7>(a, stream); break;
        case 8: launch_dense_g<8>(a, stream); break;
        default: return cudaErrorInvalidValue;
    }
    if (a.prof_stop) cudaEventRecord(a.prof_stop, stream);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dense_merge_kernel<<<a.B * a.Hq, kD, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace ffd
