// Persistent grouped GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// For every group g (an expert) and its contiguous rows [row_offsets[g], row_offsets[g+1])
// of A, computes rows of D = A * B_g^T with bf16 operands and fp32 accumulation in
// tensor memory, then applies a fused epilogue (bias, GELU or SwiGLU -> bf16, or
// routing-weight scale -> fp32). This is the expert stage of the MoE layer:
// "MoE 混合专家架构" 5.2 专家融合与并行 (stacked expert weights, each expert's slice
// applied to the tokens routed to it, silu on the W1 slice) run as one launch over
// all experts instead of a loop.
//
// Tiling: 128 rows x 256 accumulator columns x 64 K per stage, 4-stage TMA ring
// (48 KB per stage, 128-byte swizzle), two 256-column fp32 accumulators in TMEM so
// the epilogue of one tile overlaps the MMAs of the next.
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = MMA issuer (+ TMEM
// allocation), warps 2-5 = epilogue (warp w reads TMEM lanes 32*(w%4) .. +31).
// Tiles are ordered expert-major, then N block, then M block, so the CTAs working
// at the same time share one weight slice (read once from HBM) while the
// expert's activation rows stay in L2.
// For SwiGLU a tile's 256 B rows are 128 gate rows (n0..) and 128 up rows
// (F+n0..) of the same expert, loaded as two TMA boxes, so the epilogue can form
// silu(gate) * up for 128 output columns without repacking the weights.
#pragma once
#include "common.cuh"

namespace moe {

enum EpiKind : int { EPI_F32 = 0, EPI_GELU_BF16 = 1, EPI_SWIGLU_BF16 = 2, EPI_SCALE_F32 = 3 };

struct GemmParams {
    int G;                     // groups
    int N;                     // output columns per group (SwiGLU: F)
    int K;                     // reduction length (multiple of 64)
    int b_rows_per_group;      // rows of B per group (N, or 2F for SwiGLU)
    int up_offset;             // SwiGLU: F (first up row); otherwise 128 (second box)
    int n_tiles;               // N blocks per group
    const int* row_offsets;    // [G+1] device
    const int* mtile_offsets;  // [G+1] device: exclusive scan of ceil(rows_g / 128)
    void* out;                 // D rows, same row numbering as A
    long long ld_out;          // elements per output row
    const float* bias;         // [G][b_rows_per_group] fp32 or null
    const float* topk_w;       // EPI_SCALE_F32: row r scaled by topk_w[perm_token[r]*k + perm_slot[r]]
    const int* perm_token;
    const int* perm_slot;
    int top_k;
};

constexpr int GM_BM = 128, GM_BN = 256, GM_BK = 64, GM_STAGES = 4;
constexpr int GM_A_BYTES = GM_BM * GM_BK * 2;     // 16 KB
constexpr int GM_B_BYTES = GM_BN * GM_BK * 2;     // 32 KB
constexpr int GM_STAGE_BYTES = GM_A_BYTES + GM_B_BYTES;
constexpr int GM_THREADS = 192;
constexpr int GM_TMEM_COLS = 512;
constexpr int GM_MAX_GROUPS = 1025;

__host__ __device__ constexpr int gm_smem_bytes(int G) {
    return 1024 + GM_STAGES * GM_STAGE_BYTES + 256 + 2 * (G + 1) * 4;
}

__device__ __forceinline__ void gm_decode(long long t, int G, int n_tiles, const int* s_mt, int& g,
                                          int& mb, int& nb) {
    int lo = 0, hi = G;   // s_mt[lo]*n_tiles <= t < s_mt[hi]*n_tiles
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((long long)s_mt[mid] * n_tiles <= t) lo = mid;
        else hi = mid;
    }
    g = lo;
    const long long local = t - (long long)s_mt[g] * n_tiles;
    const int mt = s_mt[g + 1] - s_mt[g];
    nb = (int)(local / mt);
    mb = (int)(local % mt);
}

template <int EPI>
__device__ __forceinline__ void gm_epilogue_tile(const GemmParams& p, uint32_t tb, int g, int nb,
                                                 bool row_ok, long long grow) {
    const float* brow = p.bias ? p.bias + (long long)g * p.b_rows_per_group : nullptr;
    if constexpr (EPI == EPI_SWIGLU_BF16) {
        const int n0 = nb * 128;
        __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) + grow * p.ld_out;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            float gv[32], uv[32];
            __syncwarp();
            tmem_load_32cols(tb + c * 32, gv);
            tmem_load_32cols(tb + 128 + c * 32, uv);
            const int col = n0 + c * 32;
            if (row_ok && col < p.N) {
                uint32_t packed[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float g0 = gv[2 * i], g1 = gv[2 * i + 1], u0 = uv[2 * i], u1 = uv[2 * i + 1];
                    if (brow) {
                        g0 += brow[col + 2 * i];
                        g1 += brow[col + 2 * i + 1];
                        u0 += brow[p.up_offset + col + 2 * i];
                        u1 += brow[p.up_offset + col + 2 * i + 1];
                    }
                    packed[i] = pack_bf16x2(silu(g0) * u0, silu(g1) * u1);
                }
                uint4* dst = reinterpret_cast<uint4*>(orow + col);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                                        packed[4 * i + 3]);
            }
        }
    } else if constexpr (EPI == EPI_GELU_BF16) {
        const int n0 = nb * GM_BN;
        __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) + grow * p.ld_out;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
            float v[32];
            __syncwarp();
            tmem_load_32cols(tb + c * 32, v);
            const int col = n0 + c * 32;
            if (row_ok && col < p.N) {
                uint32_t packed[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float a0 = v[2 * i], a1 = v[2 * i + 1];
                    if (brow) {
                        a0 += brow[col + 2 * i];
                        a1 += brow[col + 2 * i + 1];
                    }
                    packed[i] = pack_bf16x2(gelu_erf(a0), gelu_erf(a1));
                }
                uint4* dst = reinterpret_cast<uint4*>(orow + col);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                                        packed[4 * i + 3]);
            }
        }
    } else {
        const int n0 = nb * GM_BN;
        float scale = 1.0f;
        if constexpr (EPI == EPI_SCALE_F32) {
            if (row_ok)
                scale = p.topk_w[(long long)p.perm_token[grow] * p.top_k + p.perm_slot[grow]];
        }
        float* orow = reinterpret_cast<float*>(p.out) + grow * p.ld_out;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
            float v[32];
            __syncwarp();
            tmem_load_32cols(tb + c * 32, v);
            const int col = n0 + c * 32;
            if (row_ok && col < p.N) {
                float4* dst = reinterpret_cast<float4*>(orow + col);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    float4 o;
                    o.x = v[4 * i + 0] + (brow ? brow[col + 4 * i + 0] : 0.0f);
                    o.y = v[4 * i + 1] + (brow ? brow[col + 4 * i + 1] : 0.0f);
                    o.z = v[4 * i + 2] + (brow ? brow[col + 4 * i + 2] : 0.0f);
                    o.w = v[4 * i + 3] + (brow ? brow[col + 4 * i + 3] : 0.0f);
                    if constexpr (EPI == EPI_SCALE_F32) {
                        o.x *= scale;
                        o.y *= scale;
                        o.z *= scale;
                        o.w *= scale;
                    }
                    dst[i] = o;
                }
            }
        }
    }
}

template <int EPI>
__global__ void __launch_bounds__(GM_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* tiles = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + GM_STAGES * GM_STAGE_BYTES);
    // barrier slots: full[0..3], empty[4..7], tfull[8..9], tempty[10..11], drain[12]
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 16);
    volatile int* s_abort = reinterpret_cast<volatile int*>(bars + 17);
    int* s_ro = reinterpret_cast<int*>(bars + 32);
    int* s_mt = s_ro + (p.G + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto bar = [&](int i) { return smem_addr(bars + i); };
    const int FULL = 0, EMPTY = GM_STAGES, TFULL = 2 * GM_STAGES, TEMPTY = 2 * GM_STAGES + 2,
              DRAIN = 2 * GM_STAGES + 4;

    for (int i = threadIdx.x; i <= p.G; i += blockDim.x) {
        s_ro[i] = p.row_offsets[i];
        s_mt[i] = p.mtile_offsets[i];
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < GM_STAGES; ++s) {
            mbar_init(bar(FULL + s), 1);
            mbar_init(bar(EMPTY + s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar(TFULL + a), 1);
            mbar_init(bar(TEMPTY + a), 4);
        }
        mbar_init(bar(DRAIN), 1);
        *s_abort = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(s_tmem), GM_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;
    const long long total = (long long)s_mt[p.G] * p.n_tiles;
    const int kblocks = p.K / GM_BK;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            int stage = 0;
            uint32_t ph = 0;
            int last_par[GM_STAGES];
#pragma unroll
            for (int s = 0; s < GM_STAGES; ++s) last_par[s] = -1;
            bool ok = true;
            for (long long t = blockIdx.x; t < total && ok; t += gridDim.x) {
                int g, mb, nb;
                gm_decode(t, p.G, p.n_tiles, s_mt, g, mb, nb);
                const int a_row = s_ro[g] + mb * GM_BM;
                const int n0 = (EPI == EPI_SWIGLU_BF16) ? nb * 128 : nb * GM_BN;
                const int b0 = g * p.b_rows_per_group + n0;
                const int b1 = b0 + p.up_offset;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (*s_abort || !mbar_wait(bar(EMPTY + stage), ph ^ 1)) {
                        *s_abort = 1;
                        ok = false;
                        break;
                    }
                    const uint32_t sa = smem_addr(tiles + stage * GM_STAGE_BYTES);
                    mbar_arrive_expect_tx(bar(FULL + stage), GM_STAGE_BYTES);
                    tma_load_2d(sa, &tmA, bar(FULL + stage), kb * GM_BK, a_row);
                    tma_load_2d(sa + GM_A_BYTES, &tmB, bar(FULL + stage), kb * GM_BK, b0);
                    tma_load_2d(sa + GM_A_BYTES + GM_B_BYTES / 2, &tmB, bar(FULL + stage),
                                kb * GM_BK, b1);
                    last_par[stage] = (int)ph;
                    if (++stage == GM_STAGES) {
                        stage = 0;
                        ph ^= 1;
                    }
                }
            }
            // Every copy this thread started must have landed before the CTA exits.
            for (int s = 0; s < GM_STAGES; ++s)
                if (last_par[s] >= 0) mbar_wait(bar(FULL + s), (uint32_t)last_par[s]);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            constexpr uint32_t idesc = idesc_bf16_f32(GM_BM, GM_BN);
            int stage = 0, acc = 0;
            uint32_t ph = 0, aph = 0;
            for (long long t = blockIdx.x; t < total; t += gridDim.x) {
                if (*s_abort || !mbar_wait(bar(TEMPTY + acc), aph ^ 1)) {
                    *s_abort = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t dt = tmem_base + (uint32_t)(acc * GM_BN);
                bool ok = true;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait(bar(FULL + stage), ph)) {
                        *s_abort = 1;
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_addr(tiles + stage * GM_STAGE_BYTES);
                    const uint32_t sb = sa + GM_A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < GM_BK / 16; ++kk)
                        umma_bf16(dt, sw128_kmajor_desc(sa + kk * 32), sw128_kmajor_desc(sb + kk * 32),
                                  idesc, (kb | kk) != 0 ? 1u : 0u);
                    umma_commit(bar(EMPTY + stage));
                    if (++stage == GM_STAGES) {
                        stage = 0;
                        ph ^= 1;
                    }
                }
                if (!ok) break;
                umma_commit(bar(TFULL + acc));
                acc ^= 1;
                if (acc == 0) aph ^= 1;
            }
            // All MMAs issued by this thread must be complete before TMEM is freed.
            umma_commit(bar(DRAIN));
            mbar_wait(bar(DRAIN), 0);
        }
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        const int q = warp & 3;
        int acc = 0;
        uint32_t aph = 0;
        for (long long t = blockIdx.x; t < total; t += gridDim.x) {
            int g, mb, nb;
            gm_decode(t, p.G, p.n_tiles, s_mt, g, mb, nb);
            int ok = 1;
            if (lane == 0) ok = (!*s_abort && mbar_wait(bar(TFULL + acc), aph)) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) *s_abort = 1;
                break;
            }
            tc_fence_after();
            const int r_in = q * 32 + lane;
            const int rows_g = s_ro[g + 1] - s_ro[g];
            const bool row_ok = mb * GM_BM + r_in < rows_g;
            const long long grow = (long long)s_ro[g] + (long long)mb * GM_BM + r_in;
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * GM_BN);
            gm_epilogue_tile<EPI>(p, tb, g, nb, row_ok, grow);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(TEMPTY + acc));
            acc ^= 1;
            if (acc == 0) aph ^= 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, GM_TMEM_COLS);
    }
}

}  // namespace moe
