// Router: gate GEMM -> top-k -> renormalised weights.
// ["MoE 混合专家架构" 2.1 门控机制 (Linear without bias, topk on logits, softmax over
//  the k kept logits); adv12 4.1 steps 1-3 and Q1 (renormalise the kept weights);
//  "MoE 混合专家架构" 4.2 数值稳定性 (max-subtracted softmax).]
#pragma once
#include "common.cuh"

namespace moe {

// ---- logits = x * W_gate (+ bias), fp32 CUDA-core GEMM -------------------------------
// CTA tile 64 tokens x 64 experts, K step 16, 256 threads with a 4x4 register tile
// each. x is converted to fp32 on the way into shared memory (exact for bf16).
constexpr int RT_BM = 64, RT_BN = 64, RT_BK = 16;

template <typename XT>
__global__ void __launch_bounds__(256) router_logits_kernel(const XT* __restrict__ x,
                                                            const float* __restrict__ Wg,
                                                            const float* __restrict__ bias,
                                                            float* __restrict__ logits, int T,
                                                            int d, int E) {
    __shared__ float xs[RT_BK][RT_BM + 4];
    __shared__ float ws[RT_BK][RT_BN + 4];
    const int tid = threadIdx.x;
    const int tx = tid % 16, ty = tid / 16;
    const long long t0 = (long long)blockIdx.x * RT_BM;
    const int e0 = blockIdx.y * RT_BN;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < d; k0 += RT_BK) {
        // x tile: 64 tokens x 16 k; thread loads 4 consecutive k of one token
        {
            const int tl = tid / 4, kl = (tid % 4) * 4;
            const long long t = t0 + tl;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int kk = k0 + kl + q;
                xs[kl + q][tl] = (t < T && kk < d) ? load_act(x, t * d + kk) : 0.0f;
            }
        }
        // W tile: 16 k x 64 experts; thread loads 4 consecutive experts of one k
        {
            const int kl = tid / 16, el = (tid % 16) * 4;
            const int kk = k0 + kl;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int e = e0 + el + q;
                ws[kl][el + q] = (kk < d && e < E) ? Wg[(long long)kk * E + e] : 0.0f;
            }
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < RT_BK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = xs[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = ws[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const long long t = t0 + ty * 4 + i;
        if (t >= T) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = e0 + tx * 4 + j;
            if (e < E) logits[t * E + e] = acc[i][j] + (bias ? bias[e] : 0.0f);
        }
    }
}

// ---- top-k + renormalisation: one warp per token -----------------------------------
// Expert e lives in lane e % 32, register e / 32 (E <= 1024). Each of the k rounds
// is a warp arg-max over (logit desc, id asc) of the experts not taken yet. The
// k kept weights are exp(L_j - L_0) / sum_j' exp(L_j' - L_0), summed in slot order.
__device__ __forceinline__ bool better(float v, int e, float bv, int be) {
    return be < 0 || v > bv || (v == bv && e < be);
}

__global__ void __launch_bounds__(256) topk_renorm_kernel(const float* __restrict__ logits, int T,
                                                          int E, int k, int* __restrict__ idx,
                                                          float* __restrict__ w) {
    const int lane = threadIdx.x & 31;
    const long long t = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    const float* L = logits + t * E;
    float v[32];
    uint32_t avail = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int e = lane + 32 * i;
        v[i] = 0.0f;
        if (e < E) {
            v[i] = L[e];
            avail |= 1u << i;
        }
    }
    float my_v = 0.0f, l0 = 0.0f;
    int my_e = 0;
    for (int j = 0; j < k; ++j) {
        float bv = 0.0f;
        int be = -1;
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if ((avail >> i) & 1u)
                if (better(v[i], lane + 32 * i, bv, be)) {
                    bv = v[i];
                    be = lane + 32 * i;
                }
#pragma unroll
        for (int off = 16; off; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oe = __shfl_xor_sync(0xffffffffu, be, off);
            if (oe >= 0 && better(ov, oe, bv, be)) {
                bv = ov;
                be = oe;
            }
        }
        if ((be & 31) == lane) avail &= ~(1u << (be >> 5));
        if (lane == j) {
            my_v = bv;
            my_e = be;
        }
        if (j == 0) l0 = bv;
    }
    const float ex = (lane < k) ? expf(my_v - l0) : 0.0f;
    float s = 0.0f;
    for (int j = 0; j < k; ++j) s += __shfl_sync(0xffffffffu, ex, j);
    if (lane < k) {
        idx[t * k + lane] = my_e;
        w[t * k + lane] = ex / s;
    }
}

}  // namespace moe
