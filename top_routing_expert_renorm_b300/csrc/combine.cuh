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

// The same combine over compact expert-output rows (bf16 layers): row r holds fp16
// values at y16 + r * d whose 32-column chunks carry a power-of-two scale 2^e, e one
// signed byte at y_exp + r * ld_e + chunk (ld_e: d / 32 rounded up to 16). Scaling by 2^e
// is exact, and the sums run in the fp32 order of combine_kernel.
//
// Each warp streams its rows through shared memory with cp.async, CH16_STAGES - 1 steps
// ahead, so the bytes in flight do not depend on registers or occupancy. A step is one
// 512-column chunk of a token and a group of up to 8 slots: each slot's row piece is
// 1 KB contiguous (a lane copies 16 bytes at lane * 8 and at 256 + lane * 8 columns),
// with the chunk's 16 exponent bytes per slot, with the first group the residual row and
// with the last group (where it is added) the shared-expert row (fp32). Row pieces of 512 bytes (256 columns) ran no faster
// than the fp32 rows' 1 KB pieces: the scattered row reads are bound by their count.
constexpr int CH16_STAGES = 3, CH16_WARPS = 6, CH16_COLS = 512;
constexpr int CH16_DATA = kCombineGroup * 2 * 32 * 16;   // slot rows
constexpr int CH16_SH = CH16_DATA;                        // + shared row (2 x 32 lanes x 32 B)
constexpr int CH16_RES = CH16_SH + 2 * 32 * 32;           // + residual row (2 x 32 lanes x 16 B)
constexpr int CH16_EXP = CH16_RES + 2 * 32 * 16;          // + exponent bytes (16 per slot)
constexpr int CH16_STAGE = CH16_EXP + kCombineGroup * 16;
constexpr int ch16_smem_bytes() { return CH16_WARPS * CH16_STAGES * CH16_STAGE; }

__device__ __forceinline__ void cp_async_cg16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit_group() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait_groups() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void add2_h16(float& a0, float& a1, uint32_t w, float sc) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
    a0 += f.x * sc;   // f * 2^e is exact
    a1 += f.y * sc;
}
__device__ __forceinline__ void add8_h16(float4& lo, float4& hi, const uint4& v, float sc) {
    add2_h16(lo.x, lo.y, v.x, sc);
    add2_h16(lo.z, lo.w, v.y, sc);
    add2_h16(hi.x, hi.y, v.z, sc);
    add2_h16(hi.z, hi.w, v.w, sc);
}
__device__ __forceinline__ float exp2_int(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

__global__ void __launch_bounds__(CH16_WARPS * 32, 1) combine_h16_kernel(
    const __nv_bfloat16* __restrict__ x, const __half* __restrict__ y16,
    const int8_t* __restrict__ y_exp, int ld_e, const int* __restrict__ slot_dest,
    const float* __restrict__ y_shared, const float* __restrict__ ovf_w,
    __nv_bfloat16* __restrict__ out, int T, int d, int k, int add_residual, int cpt) {
    // cpt: 512-column chunks per warp task
    extern __shared__ __align__(128) uint8_t ch16_smem[];
    pdl_entry();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint8_t* wsm = ch16_smem + warp * (CH16_STAGES * CH16_STAGE);
    const uint32_t wsa = smem_addr(wsm);
    const int chunks = (d + CH16_COLS - 1) / CH16_COLS;
    const int groups = (k + kCombineGroup - 1) / kCombineGroup;
    const int spans = (chunks + cpt - 1) / cpt;
    const long long work = (long long)T * spans;
    const long long warps = (long long)gridDim.x * CH16_WARPS;
    for (long long wi = (long long)blockIdx.x * CH16_WARPS + warp; wi < work; wi += warps) {
        const long long t = wi / spans;
        const int sp = (int)(wi - t * spans);
        const int mydest = lane < k ? slot_dest[t * k + lane] : -1;
        float a_sh = 1.0f;
        if (ovf_w) {
            const float wd = (lane < k && mydest < 0) ? ovf_w[t * k + lane] : 0.0f;
            for (int j = 0; j < k; ++j) a_sh += __shfl_sync(0xffffffffu, wd, j);
        }
        const int c0 = sp * cpt, c1 = min(chunks, c0 + cpt);
        const int nsteps = (c1 - c0) * groups;
        // copies of step st into its stage (an empty group when st is past the end)
        auto issue = [&](int st) {
            if (st < nsteps) {   // (warp-uniform)
                const int ch = c0 + st / groups, g = st % groups;
                const uint32_t sa = wsa + (st % CH16_STAGES) * CH16_STAGE;
                // every lane takes part in the shuffles before any lane-dependent branch
                int rr[kCombineGroup];
#pragma unroll
                for (int u = 0; u < kCombineGroup; ++u) {
                    const int j = g * kCombineGroup + u;
                    rr[u] = __shfl_sync(0xffffffffu, mydest, j & 31);
                    if (j >= k) rr[u] = -1;
                }
                const int je = g * kCombineGroup + lane;   // lanes 0..7: exponent bytes of slot je
                const int re = __shfl_sync(0xffffffffu, mydest, je & 31);
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int ca = ch * CH16_COLS + hf * 256 + lane * 8;
                    if (ca >= d) continue;   // d % 64 == 0: a lane's 8 columns are all in or out
#pragma unroll
                    for (int u = 0; u < kCombineGroup; ++u)
                        if (rr[u] >= 0)
                            cp_async_cg16(sa + ((u * 2 + hf) * 32 + lane) * 16,
                                          y16 + (long long)rr[u] * d + ca);
                    if (g == 0 && add_residual)
                        cp_async_cg16(sa + CH16_RES + (hf * 32 + lane) * 16, x + t * d + ca);
                    if (g == groups - 1 && y_shared) {   // added after the last group
                        const float* ys = y_shared + t * d + ca;
                        cp_async_cg16(sa + CH16_SH + (hf * 32 + lane) * 32, ys);
                        cp_async_cg16(sa + CH16_SH + (hf * 32 + lane) * 32 + 16, ys + 4);
                    }
                }
                // the chunk's 16 exponent bytes (a row holds 16 * chunks of them)
                if (lane < kCombineGroup && je < k && re >= 0)
                    cp_async_cg16(sa + CH16_EXP + lane * 16, y_exp + (long long)re * ld_e + ch * 16);
            }
            cp_async_commit_group();
        };
#pragma unroll
        for (int st = 0; st < CH16_STAGES - 1; ++st) issue(st);
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        float4 acc[2][2] = {{z, z}, {z, z}};
        for (int st = 0; st < nsteps; ++st) {
            issue(st + CH16_STAGES - 1);
            cp_async_wait_groups<CH16_STAGES - 1>();   // step st's copies are complete
            __syncwarp();
            const int ch = c0 + st / groups, g = st % groups;
            const uint8_t* sp8 = wsm + (st % CH16_STAGES) * CH16_STAGE;
            int rr[kCombineGroup];
#pragma unroll
            for (int u = 0; u < kCombineGroup; ++u) {
                const int j = g * kCombineGroup + u;
                rr[u] = __shfl_sync(0xffffffffu, mydest, j & 31);
                if (j >= k) rr[u] = -1;
            }
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int ca = ch * CH16_COLS + hf * 256 + lane * 8;
                if (ca >= d) continue;
                float4& a0 = acc[hf][0];
                float4& a1 = acc[hf][1];
                if (g == 0) {
                    a0 = a1 = z;
                    if (add_residual) {
                        const __nv_bfloat16* xr = reinterpret_cast<const __nv_bfloat16*>(
                            sp8 + CH16_RES + (hf * 32 + lane) * 16);
                        load4<__nv_bfloat16>(xr, a0);
                        load4<__nv_bfloat16>(xr + 4, a1);
                    }
                }
#pragma unroll
                for (int u = 0; u < kCombineGroup; ++u) {
                    if (rr[u] < 0) continue;
                    const uint4 v = *reinterpret_cast<const uint4*>(sp8 + ((u * 2 + hf) * 32 + lane) * 16);
                    const int e = reinterpret_cast<const int8_t*>(sp8 + CH16_EXP + u * 16)[hf * 8 + (lane >> 2)];
                    add8_h16(a0, a1, v, exp2_int(e));
                }
                if (g == groups - 1) {
                    if (y_shared) {
                        const uint8_t* shp = sp8 + CH16_SH + (hf * 32 + lane) * 32;
                        const float4 v0 = *reinterpret_cast<const float4*>(shp);
                        const float4 v1 = *reinterpret_cast<const float4*>(shp + 16);
                        if (ovf_w) {
                            fma4(a0, a_sh, v0);
                            fma4(a1, a_sh, v1);
                        } else {
                            add4(a0, v0);
                            add4(a1, v1);
                        }
                    }
                    store4<__nv_bfloat16>(out + t * d + ca, a0);
                    store4<__nv_bfloat16>(out + t * d + ca + 4, a1);
                }
            }
            __syncwarp();   // the stage is read before a later step's copies refill it
        }
        cp_async_wait_groups<0>();
        __syncwarp();
    }
}

}  // namespace moe
