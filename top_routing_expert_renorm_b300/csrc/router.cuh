// Router: gate GEMM -> top-k -> renormalised weights.
// ["MoE 混合专家架构" 2.1 门控机制 (Linear without bias, topk on logits, softmax over
//  the k kept logits); adv12 4.1 steps 1-3 and Q1 (renormalise the kept weights);
//  "MoE 混合专家架构" 4.2 数值稳定性 (max-subtracted softmax).]
#pragma once
#include <type_traits>
#include "common.cuh"

namespace moe {

// Every router path writes raw partial sums of x * W_gate; topk_renorm_kernel adds
// the parts in a fixed order (plus the bias) to form the fp32 logits, so the
// result does not depend on scheduling.

// ---- path 1: x * W_gate, fp32 CUDA-core GEMM (fp32 activations) ------------------------
// CTA tile 64 tokens x 64 experts, K step 16, 256 threads with a 4x4 register tile
// each. x is converted to fp32 on the way into shared memory (exact for bf16).
constexpr int RT_BM = 64, RT_BN = 64, RT_BK = 16;

template <typename XT>
__global__ void __launch_bounds__(256) router_logits_kernel(const XT* __restrict__ x,
                                                            const float* __restrict__ Wg,
                                                            float* __restrict__ logits, int T,
                                                            int d, int E) {
    pdl_entry();
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
            if (e < E) logits[t * E + e] = acc[i][j];
        }
    }
}

// ---- path 2: bf16 activations, many tokens: tensor cores on an exact 3-way split ------
// Every fp32 gate weight v is split into three bf16 terms hi + mid + lo == v exactly
// (hi = bf16(v), mid = bf16(v - hi), lo = v - hi - mid, which has at most 8 significant
// bits). Products of a bf16 activation with each term are exact in fp32, so running
// x [T, d] against B = [hi; mid; lo] ([3*Ep, d], K-major) on the bf16 tensor cores with
// fp32 accumulation gives fp32-accurate logits. This kernel transposes W_gate [d, E]
// into that layout (32x32 tiles through shared memory) and writes the one-group
// row / M-tile tables of the GEMM.
constexpr int kRouterPad = 32;   // experts are padded to Ep = round_up(E, 32) per term

__global__ void __launch_bounds__(256) gate_split_kernel(const float* __restrict__ Wg, int d,
                                                         int E, int Ep,
                                                         __nv_bfloat16* __restrict__ Bg, int T,
                                                         int* __restrict__ tables,
                                                         unsigned long long* __restrict__ counter,
                                                         int* __restrict__ tile_cnt, int n_tile_cnt) {
    // tile_cnt (nullable): the arrival counters of the router GEMM's K-split M tiles,
    // zeroed here
    pdl_entry();
    const int nthreads = gridDim.x * gridDim.y * blockDim.x;
    const int tid = (blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x;
    if (tile_cnt)
        for (int i = tid; i < n_tile_cnt; i += nthreads) tile_cnt[i] = 0;
    __shared__ float tile[32][33];
    const int k0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8
    for (int r = ty; r < 32; r += 8) {
        const int k = k0 + r, e = e0 + tx;
        tile[r][tx] = (k < d && e < E) ? Wg[(long long)k * E + e] : 0.0f;
    }
    __syncthreads();
    for (int r = ty; r < 32; r += 8) {
        const int e = e0 + r, k = k0 + tx;
        if (e >= Ep || k >= d) continue;
        const float v = tile[tx][r];
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        const float r1 = v - __bfloat162float(hi);
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
        Bg[(long long)e * d + k] = hi;
        Bg[((long long)Ep + e) * d + k] = mid;
        Bg[(2ll * Ep + e) * d + k] = lo;
    }
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
        tables[0] = 0;                      // row offsets of the single group
        tables[1] = T;
        tables[2] = 0;                      // its M-tile offsets
        tables[3] = (T + 127) / 128;
        *counter = 0ull;                    // tile counter of the router GEMM
    }
}

// ---- path 3: bf16 activations, few tokens: split-K CUDA-core kernel --------------------
// CTA (256 threads) = 32 experts (lane) x a 256-long K slice (warp w takes 32 of it) x
// up to TT tokens (blockIdx.z chunk). Each thread first issues all 32 of its W_gate
// loads, then accumulates its 32 K values for every token; the 8 warps are summed
// through shared memory in a fixed order and the CTA writes one partial [slice][T][E].
// Wide grids keep all SMs streaming W_gate.
constexpr int RS_E = 32, RS_K = 256;

template <int TT>
__global__ void __launch_bounds__(256) router_splitk_kernel(const __nv_bfloat16* __restrict__ x,
                                                            const float* __restrict__ Wg,
                                                            float* __restrict__ parts, int T,
                                                            int d, int E) {
    __shared__ __nv_bfloat16 xs[TT][RS_K];
    __shared__ float red[8][8][RS_E + 1];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int e = blockIdx.x * RS_E + lane;
    const int k0 = blockIdx.y * RS_K;
    const int t0 = blockIdx.z * TT;
    const int nt = min(TT, T - t0);
    // W_gate is a layer input no kernel of the library writes: its loads may start
    // before the preceding kernel has finished; x may be that kernel's output.
    float wv[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int k = k0 + w * 32 + i;
        wv[i] = (k < d && e < E) ? __ldg(Wg + (long long)k * E + e) : 0.0f;
    }
    pdl_entry();
    for (int i = threadIdx.x; i < TT * RS_K; i += blockDim.x) {
        const int t = i / RS_K, kk = i % RS_K;
        xs[t][kk] = (t < nt && k0 + kk < d) ? x[(long long)(t0 + t) * d + k0 + kk]
                                             : __float2bfloat16_rn(0.0f);
    }
    __syncthreads();
    float acc[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) {
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) a = fmaf(__bfloat162float(xs[t][w * 32 + i]), wv[i], a);
        acc[t] = a;
    }
    float* out = parts + (long long)blockIdx.y * T * E;
#pragma unroll
    for (int c = 0; c < TT / 8; ++c) {
        __syncthreads();
#pragma unroll
        for (int t = 0; t < 8; ++t) red[w][t][lane] = acc[c * 8 + t];
        __syncthreads();
        for (int i = threadIdx.x; i < 8 * RS_E; i += blockDim.x) {
            const int t = i / RS_E, l = i % RS_E;
            const int tt = c * 8 + t, ee = blockIdx.x * RS_E + l;
            if (tt < nt && ee < E) {
                float s = 0.0f;
#pragma unroll
                for (int q = 0; q < 8; ++q) s += red[q][t][l];
                out[(long long)(t0 + tt) * E + ee] = s;
            }
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

// Logit (t, e) = sum_{p < n_parts} parts[p*part_stride + t*row_stride + e] (+ bias[e]),
// summed in part order; written to `logits` [T, E] when that is non-null.
// A CTA handles kTopkTok tokens: all 256 threads first form the CTA's logits in shared
// memory (every (token, expert) sum issues its part loads in batches of 8, so few
// round trips are exposed even with many parts), then warp w selects for token w.
// cand (nullable, re-routing): the experts ranked k .. 2k-1 by the same order and within
// the same candidate set, -1 where the set has fewer experts.
constexpr int kTopkTok = 8;

// VPL: logits per lane of the selecting warp, ceil(E / 32) rounded up to 2, 8 or 32.
template <int VPL>
__global__ void __launch_bounds__(256, 3) topk_renorm_kernel(const float* __restrict__ parts,
                                                          int n_parts, long long part_stride,
                                                          long long row_stride,
                                                          const float* __restrict__ bias,
                                                          float* __restrict__ logits, int T,
                                                          int E, int k, int n_group,
                                                          int topk_group, int* __restrict__ idx,
                                                          float* __restrict__ w,
                                                          int* __restrict__ cand) {
    pdl_entry();
    extern __shared__ float sL[];   // [kTopkTok][E]
    const int lane = threadIdx.x & 31;
    const long long t0 = (long long)blockIdx.x * kTopkTok;
    const int nt = (int)min((long long)kTopkTok, (long long)T - t0);
    // Logits: every thread issues the part loads of several sums before their adds, so one
    // memory round trip serves them. Few parts (the tensor-core router's three terms): 8
    // sums per thread, all parts in one batch of 4 (DeepSeek-V3 shape: 53 -> 39 us); many
    // parts (the split-K router's K slices, decode): 4 sums per thread, parts in batches
    // of 8 (one sum per thread with batches of 32 was slower: T = 8, 21 -> 59 us). Adds
    // run in part order.
    const int n = nt * E;
    auto form = [&](auto es_tag, auto pb_tag) {
        constexpr int ES = decltype(es_tag)::value, PB = decltype(pb_tag)::value;
        for (int i0 = threadIdx.x; i0 < n; i0 += ES * blockDim.x) {
            const float* L[ES];
            float s[ES];
#pragma unroll
            for (int u = 0; u < ES; ++u) {
                const int i = min(i0 + u * (int)blockDim.x, n - 1);
                const int tt = i / E, e = i - tt * E;
                L[u] = parts + (t0 + tt) * row_stride + e;
                s[u] = 0.0f;
            }
            for (int p = 0; p < n_parts; p += PB) {
                float v[ES][PB];
#pragma unroll
                for (int u = 0; u < ES; ++u)
#pragma unroll
                    for (int q = 0; q < PB; ++q)
                        v[u][q] = (i0 + u * (int)blockDim.x < n && p + q < n_parts)
                                      ? L[u][(long long)(p + q) * part_stride]
                                      : 0.0f;
#pragma unroll
                for (int u = 0; u < ES; ++u)
#pragma unroll
                    for (int q = 0; q < PB; ++q)
                        if (p + q < n_parts) s[u] = (p + q == 0) ? v[u][q] : s[u] + v[u][q];
            }
#pragma unroll
            for (int u = 0; u < ES; ++u) {
                const int i = i0 + u * blockDim.x;
                if (i >= n) break;
                const int tt = i / E, e = i - tt * E;
                float sv = s[u];
                if (bias) sv += bias[e];
                sL[i] = sv;
                if (logits) logits[(t0 + tt) * E + e] = sv;
            }
        }
    };
    if (n_parts <= 4) form(std::integral_constant<int, 8>{}, std::integral_constant<int, 4>{});
    else form(std::integral_constant<int, 4>{}, std::integral_constant<int, 8>{});
    __syncthreads();
    const int wt = threadIdx.x >> 5;
    if (wt >= nt) return;
    const long long t = t0 + wt;
    const float* Ls = sL + wt * E;
    float v[VPL];
    uint32_t avail = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        v[i] = 0.0f;
        if (e < E) {
            v[i] = Ls[e];
            avail |= 1u << i;
        }
    }
    if (n_group > 0) {
        // Group-limited routing: lane g < n_group scores group g by its best logit; the
        // topk_group best groups (ties to the lower group id) are kept and every expert
        // of the other groups leaves the candidate set.
        const int gsize = E / n_group;
        float gbest = 0.0f;
        if (lane < n_group) {
            gbest = Ls[lane * gsize];
            for (int e = lane * gsize + 1; e < (lane + 1) * gsize; ++e) gbest = fmaxf(gbest, Ls[e]);
        }
        uint32_t gavail = (lane < n_group) ? 1u : 0u, chosen = 0;
        for (int j = 0; j < topk_group; ++j) {
            float bv = gbest;
            int bg = gavail ? lane : -1;
#pragma unroll
            for (int off = 16; off; off >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                const int og = __shfl_xor_sync(0xffffffffu, bg, off);
                if (og >= 0 && better(ov, og, bv, bg)) {
                    bv = ov;
                    bg = og;
                }
            }
            chosen |= 1u << bg;
            if (bg == lane) gavail = 0;
        }
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !((chosen >> (e / gsize)) & 1u)) avail &= ~(1u << i);
        }
    }
    // Each lane keeps its own best remaining candidate (lb, le); a round takes the warp's
    // best of those (logit descending, id ascending), which leaves the candidate set, and
    // only the lane that owned it rescans its (E / 32) values. be = -1 when the set is empty.
    const int nv = (E + 31) / 32;   // values per lane (warp-uniform)
    float lb = 0.0f;
    int le = -1;
    auto local_best = [&]() {
        lb = 0.0f;
        le = -1;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            if (i >= nv) break;
            if (((avail >> i) & 1u) && better(v[i], lane + 32 * i, lb, le)) {
                lb = v[i];
                le = lane + 32 * i;
            }
        }
    };
    local_best();
    auto pick = [&](float& bv, int& be) {
        bv = lb;
        be = le;
#pragma unroll
        for (int off = 16; off; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oe = __shfl_xor_sync(0xffffffffu, be, off);
            if (oe >= 0 && better(ov, oe, bv, be)) {
                bv = ov;
                be = oe;
            }
        }
        if (be >= 0 && (be & 31) == lane) {
            avail &= ~(1u << (be >> 5));
            local_best();
        }
    };
    float my_v = 0.0f, l0 = 0.0f;
    int my_e = 0;
    for (int j = 0; j < k; ++j) {
        float bv;
        int be;
        pick(bv, be);
        if (lane == j) {
            my_v = bv;
            my_e = be;
        }
        if (j == 0) l0 = bv;
    }
    if (cand) {
        int my_c = -1;
        for (int j = 0; j < k; ++j) {
            float bv;
            int be;
            pick(bv, be);
            if (lane == j) my_c = be;
        }
        if (lane < k) cand[t * k + lane] = my_c;
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
