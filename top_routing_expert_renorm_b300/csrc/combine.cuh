// Linear (fp32) experts and the weighted combine.
// ["adv12 — MoE + EPLB" 4.1: experts are nn.Linear(d_model, d_model) and
//  out[mask] += weight * expert_e(x[mask]); "MOE 学习笔记" 输出聚合示例 (weighted sum of
//  the selected experts' outputs); "MoE 并行" Capacity Factor (overflow -> residual).]
#pragma once
#include "common.cuh"

namespace moe {

// ---- LINEAR experts in fp32: y[r] = scale_r * (W_g x[r] + b_g) -------------------------
// One thread per output element; row r belongs to the group g with
// row_offsets[g] <= r < row_offsets[g+1] (binary search); P = row_offsets[G].
// scale_r = topk_w[perm_token[r]*k + perm_slot[r]] when topk_w is given, else 1.
__global__ void __launch_bounds__(256) linear_expert_kernel(
    const float* __restrict__ xin, const int* __restrict__ row_offsets, int G,
    const float* __restrict__ W, const float* __restrict__ b, const float* __restrict__ topk_w,
    const int* __restrict__ perm_token, const int* __restrict__ perm_slot, int k,
    float* __restrict__ y, int d, long long max_rows) {
    pdl_entry();
    const int P = row_offsets[G];
    const long long n = (long long)P * d;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n && i < max_rows * d;
         i += stride) {
        const long long r = i / d;
        const int o = (int)(i % d);
        int lo = 0, hi = G;   // row_offsets[lo] <= r < row_offsets[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (row_offsets[mid] <= r) lo = mid;
            else hi = mid;
        }
        const float* wrow = W + ((long long)lo * d + o) * d;
        const float* xr = xin + r * d;
        float acc = 0.0f;
        for (int c = 0; c < d; ++c) acc = fmaf(wrow[c], xr[c], acc);
        if (b) acc += b[(long long)lo * d + o];
        if (topk_w) acc *= topk_w[(long long)perm_token[r] * k + perm_slot[r]];
        y[i] = acc;
    }
}

// ---- combine: out[t] = (res ? x[t] : 0) + sum_j kept y[slot_dest[t,j]] (+ y_shared[t]) ----
// The k slot rows are summed in slot order, so the result does not depend on
// scheduling.
template <typename OT>
__device__ __forceinline__ void load4(const OT* p, float4& v);
template <>
__device__ __forceinline__ void load4<float>(const float* p, float4& v) {
    v = *reinterpret_cast<const float4*>(p);
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16* p, float4& v) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
    const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
    v = make_float4(fa.x, fa.y, fb.x, fb.y);
}
template <typename OT>
__device__ __forceinline__ void store4(OT* p, const float4& v);
template <>
__device__ __forceinline__ void store4<float>(float* p, const float4& v) {
    *reinterpret_cast<float4*>(p) = v;
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p, const float4& v) {
    uint2 u;
    u.x = pack_bf16x2(v.x, v.y);
    u.y = pack_bf16x2(v.z, v.w);
    *reinterpret_cast<uint2*>(p) = u;
}

// One warp per task = (token, span of `cpt` consecutive 256-column chunks), grid-stride:
// whole tokens when there are many, single chunks when there are few, so that few
// tokens still spread over many SMs. slot_dest of the token is read once per task by
// lanes 0..k-1 and broadcast by shuffles; each lane owns two float4 column groups of a
// chunk. Additions run in slot order and skip dropped slots (adding +0 would turn a
// -0 residual into +0). The slot loop stays a plain loop: the kernel needs few
// registers, so many warps per SM keep the HBM reads in flight.
__device__ __forceinline__ void add4(float4& a, const float4& v) {
    a.x += v.x;
    a.y += v.y;
    a.z += v.z;
    a.w += v.w;
}
__device__ __forceinline__ void fma4(float4& a, float s, const float4& v) {
    a.x = fmaf(s, v.x, a.x);
    a.y = fmaf(s, v.y, a.y);
    a.z = fmaf(s, v.z, a.z);
    a.w = fmaf(s, v.w, a.w);
}

constexpr int kCombineGroup = 8;

template <typename OT>
__global__ void __launch_bounds__(256, 2) combine_kernel(const OT* __restrict__ x,
                                                      const float* __restrict__ y,
                                                      const int* __restrict__ slot_dest,
                                                      const float* __restrict__ y_shared,
                                                      const float* __restrict__ ovf_w,
                                                      OT* __restrict__ out, int T, int d, int k,
                                                      int add_residual, int cpt) {
    pdl_entry();
    const int lane = threadIdx.x & 31;
    const int chunks = (d + 255) / 256;
    const int spans = (chunks + cpt - 1) / cpt;
    const long long work = (long long)T * spans;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long wi = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); wi < work;
         wi += warps) {
        const long long t = wi / spans;
        const int sp = (int)(wi - t * spans);
        const int mydest = lane < k ? slot_dest[t * k + lane] : -1;
        // overflow to the shared expert: its weight is 1 + the dropped slots' weights,
        // summed in fp32 in slot order
        float a_sh = 1.0f;
        if (ovf_w) {
            const float wd = (lane < k && mydest < 0) ? ovf_w[t * k + lane] : 0.0f;
            for (int j = 0; j < k; ++j) a_sh += __shfl_sync(0xffffffffu, wd, j);
        }
        const int cend = min(chunks, (sp + 1) * cpt);
        for (int ch = sp * cpt; ch < cend; ++ch) {
            const int ca = ch * 256 + lane * 4, cb = ca + 128;
            const bool va = ca < d, vb = cb < d;
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
            if (add_residual) {
                if (va) load4<OT>(x + t * d + ca, a);
                if (vb) load4<OT>(x + t * d + cb, b);
            }
            // Slots in groups of kCombineGroup: the group's row loads are all issued before
            // its adds, which then run in slot order (a dropped slot adds nothing).
            for (int j0 = 0; j0 < k; j0 += kCombineGroup) {
                int r[kCombineGroup];
                float4 ya[kCombineGroup], yb[kCombineGroup];
#pragma unroll
                for (int u = 0; u < kCombineGroup; ++u) {
                    r[u] = (j0 + u < k) ? __shfl_sync(0xffffffffu, mydest, j0 + u) : -1;
                    ya[u] = yb[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (r[u] >= 0) {
                        const float* yr = y + (long long)r[u] * d;
                        if (va) ya[u] = *reinterpret_cast<const float4*>(yr + ca);
                        if (vb) yb[u] = *reinterpret_cast<const float4*>(yr + cb);
                    }
                }
#pragma unroll
                for (int u = 0; u < kCombineGroup; ++u) {
                    if (r[u] < 0) continue;
                    if (va) add4(a, ya[u]);
                    if (vb) add4(b, yb[u]);
                }
            }
            if (y_shared) {
                const float* ys = y_shared + t * d;
                if (ovf_w) {
                    if (va) fma4(a, a_sh, *reinterpret_cast<const float4*>(ys + ca));
                    if (vb) fma4(b, a_sh, *reinterpret_cast<const float4*>(ys + cb));
                } else {
                    if (va) add4(a, *reinterpret_cast<const float4*>(ys + ca));
                    if (vb) add4(b, *reinterpret_cast<const float4*>(ys + cb));
                }
            }
            if (va) store4<OT>(out + t * d + ca, a);
            if (vb) store4<OT>(out + t * d + cb, b);
        }
    }
}

}  // namespace moe
