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
// Tiling (MT = 1): 128 rows x 256 accumulator columns x 64 K per stage, 4-stage TMA
// ring (48 KB per stage, 128-byte swizzle), two 256-column fp32 accumulators in TMEM so
// the epilogue of one tile overlaps the MMAs of the next.
// Wide tiles (MT = 2, groups of >= ~200 rows): 256 rows x 256 columns per tile, two M = 128
// MMAs per K step sharing the B tile, 3-stage ring of 64 KB stages, the two 128-row
// halves filling all 512 TMEM columns (one accumulator set). Per FLOP a tile then moves
// a third fewer operand bytes from L2 and the ring covers 1.5x the load latency, at the
// cost of an epilogue that no longer overlaps the next tile's MMAs.
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = MMA issuer (+ TMEM
// allocation), warps 2-5 = epilogue (warp w reads TMEM lanes 32*(w%4) .. +31).
// Tiles are ordered expert-major, then N block, then M block, so the CTAs working
// at the same time share one weight slice (read once from HBM) while the
// expert's activation rows stay in L2. CTAs take tiles dynamically from a global
// counter: the first M tile of a weight slice streams it from HBM while its sibling
// M tiles re-read it from L2, so tiles differ in cost and a fixed round-robin would
// give some SMs most of the HBM traffic. The producer thread fetches the next tile
// id and hands it to the MMA and epilogue warps through a small ring in shared memory.
// For SwiGLU a tile's 256 B rows are 128 gate rows (n0..) and 128 up rows
// (F+n0..) of the same expert, loaded as two TMA boxes, so the epilogue can form
// silu(gate) * up for 128 output columns without repacking the weights.
// CTA pairs (GemmParams::pair): two-CTA clusters take pairs of consecutive 128-row tiles
// of one group and N block; each CTA loads half of the B tile and multicasts it to both.
// Outputs: bf16 rows (GELU / SwiGLU, top-1 combine), fp32 rows (32-byte stores, or with
// 128-row tiles one bulk tensor store per warp and 32 x 32 box staged in shared memory),
// or compact rows (EPI_SCALE_H16: fp16 with a power-of-two scale per 32 columns).
#pragma once
#include "common.cuh"

namespace moe {

enum EpiKind : int {
    EPI_F32 = 0,
    EPI_GELU_BF16 = 1,
    EPI_SWIGLU_BF16 = 2,
    EPI_SCALE_F32 = 3,
    // top-1 layers without a shared expert: the down projection is also the combine,
    // out[t] = [resid[t] +] w * (acc + b) in bf16 at t = perm_token[row]
    EPI_COMBINE1_BF16 = 4,
    // router with E <= 64: accumulator columns [p*Ep, p*Ep + E) are the three bf16-split
    // terms of x * W_gate; the epilogue forms the logits, selects the top k and writes the
    // renormalised weights (the top-k kernel is not launched)
    EPI_ROUTER_TOPK = 5,
    // EPI_SCALE_F32's values stored compactly: each 32-column chunk of a row as fp16
    // v * 2^-e, e chosen from the chunk's largest finite magnitude so that it lands in
    // [2^14, 2^15), and e as one signed byte in out_exp [rows][ld_exp]
    EPI_SCALE_H16 = 6
};

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
    const float* w_scale;      // [G][b_rows_per_group] fp32 per weight row (INT8 weights), or
                               // null: column n of the accumulator is multiplied by its row's
                               // scale before the bias and the epilogue
    const float* topk_w;       // EPI_SCALE_F32: row r scaled by topk_w[perm_token[r]*k + perm_slot[r]]
    const int* perm_token;
    const int* perm_slot;
    // Gathered A (nullable): row r of A is row a_gather[r] of a_src (a_row_bytes per row);
    // the CTA then has 128 more threads that load A with cp.async instead of TMA
    const int* a_gather;
    const uint8_t* a_src;
    long long a_row_bytes;
    int top_k;
    const __nv_bfloat16* resid;   // EPI_COMBINE1_BF16: residual x [T, ld_out], nullable
    int* r_idx;                   // EPI_ROUTER_TOPK: top-k ids [T, top_k]
    float* r_w;                   //                  renormalised weights [T, top_k]
    int r_E, r_Ep;                //                  experts, padded experts per term (32 | 64)
    long long r_rows;             //                  T (rows of r_part per part)
    int* r_hist;                  //                  nullable [ceil(T / 32)][r_E]: selected
                                  //                  experts per 32 tokens (one epilogue warp)
    float* r_part;                //                  k_splits > 1: partial logits [S][T][r_Ep]
    int* r_tile_cnt;              //                  and arrivals per M tile (zeroed before)
    // split-K: every output tile is computed as k_splits units over consecutive ranges of
    // kb_per_split K blocks; with partial != null each unit stores its raw fp32 sums at
    // partial + split * part_stride + row * ld_part + column (columns as in B's rows, so
    // a SwiGLU unit writes gate columns n and up columns F + n), and splitk_reduce_kernel
    // applies the epilogue afterwards.
    int k_splits;
    int kb_per_split;
    float* partial;
    long long part_stride;
    long long ld_part;
    // Dynamic scheduling: a CTA takes unit blockIdx.x first, then gridDim.x + the value
    // it fetched-and-incremented from this counter (zeroed by the kernel that writes
    // the launch's tables). Null: static round-robin over the units.
    unsigned long long* tile_counter;
    // An extra group (the shared expert) in the same launch: group xg1 - 1 (0 = none) reads
    // its A rows from the second A map (rows from 0; gathered: row r of the group is row r of
    // a_src) and its weights from the second B map (rows from 0), with bias xg_bias [N1]; its
    // output rows follow the others' in the row numbering of row_offsets.
    int xg1;
    const float* xg_bias;
    // 1: the output row of group-row r is r (out already points at the group's first row)
    // instead of row_offsets[g] + r (single-group launches whose rows sit at a device-side
    // offset of A)
    int out_local;
    // 1 (fp32 epilogues): whole 32-row warp slices of a tile are written through the
    // output tensor map (staged in shared memory, one bulk tensor store per 32 x 32 box)
    int tma_out;
    int8_t* out_exp;   // EPI_SCALE_H16: the chunk exponents, ld_exp bytes per row
    int ld_exp;
    // 1 (128-row tiles, unsplit, no gathered A, no extra group; launched as clusters of
    // two CTAs): a unit is a pair of consecutive M tiles of one group and N block; CTA
    // rank r of the cluster computes tile 2 * pair + r, each CTA loads one 128-row half of
    // the B tile and multicasts it to both, and a stage is refilled only after both CTAs'
    // MMAs have read it. Units are assigned to clusters round-robin.
    int pair;
};

constexpr int GM_BM = 128, GM_BN = 256, GM_BK = 64, GM_STAGES = 4;
constexpr int GM_A_BYTES = GM_BM * GM_BK * 2;     // 16 KB
constexpr int GM_B_BYTES = GM_BN * GM_BK * 2;     // 32 KB
constexpr int GM_STAGE_BYTES = GM_A_BYTES + GM_B_BYTES;
// per M-tile height MT (128-row halves per tile): ring depth and stage size
__host__ __device__ constexpr int gm_stages(int MT) { return MT == 1 ? GM_STAGES : 3; }
__host__ __device__ constexpr int gm_stage_bytes(int MT) { return MT * GM_A_BYTES + GM_B_BYTES; }
constexpr int GM_THREADS = 192;
constexpr int GM_GATHER_THREADS = 128;    // extra warps 6..9 that gather A rows
constexpr int GM_TMEM_COLS = 512;
constexpr int GM_MAX_GROUPS = 1025;
constexpr int GM_TQ = 8;            // depth of the ring of scheduled unit ids
constexpr int GM_HDR_BYTES = 512;   // barriers, TMEM address, abort flag, unit-id ring

constexpr int GM_RHIST_BYTES = 4 * 64 * 4;   // router top-k: 64 counters per epilogue warp
// fp32 epilogues: one staging box (32 rows x 32 fp32, 128-byte swizzle) per epilogue warp;
// EPI_SCALE_H16: 32 rows x 64 fp16 in the same 4 KB
__host__ __device__ constexpr bool gm_stages_out(int epi) {
    return epi == EPI_F32 || epi == EPI_SCALE_F32 || epi == EPI_SCALE_H16;
}
constexpr int GM_OUT_BOX = 32;
constexpr int GM_OUT_STAGE_BYTES = 4 * GM_OUT_BOX * GM_OUT_BOX * 4;
__host__ __device__ constexpr int gm_smem_bytes(int G, int MT = 1, int epi = -1) {
    // ring, output staging, header, row / M-tile / tile-pair tables, router counters
    return 1024 + gm_stages(MT) * gm_stage_bytes(MT) + (gm_stages_out(epi) ? GM_OUT_STAGE_BYTES : 0) +
           GM_HDR_BYTES + 3 * (G + 1) * 4 + GM_RHIST_BYTES;
}

// s_mt[0..G] = exclusive scan over the groups of ceil(rows_g / bm), from the row offsets
// s_ro[0..G] (both in shared memory); one warp, lanes take contiguous runs of groups.
__device__ __forceinline__ void gm_tile_table_warp(const int* s_ro, int* s_mt, int G, int bm,
                                                   int lane) {
    const int per = (G + 31) / 32;
    const int g0 = min(G, lane * per), g1 = min(G, g0 + per);
    int sum = 0;
    for (int g = g0; g < g1; ++g) sum += (s_ro[g + 1] - s_ro[g] + bm - 1) / bm;
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    int run = incl - sum;
    for (int g = g0; g < g1; ++g) {
        s_mt[g] = run;
        run += (s_ro[g + 1] - s_ro[g] + bm - 1) / bm;
    }
    if (lane == 31) s_mt[G] = incl;
}

// s_mp[0..G] = exclusive scan over the groups of ceil(tiles_g / 2) (tile pairs), from the
// M-tile offsets s_mt[0..G]; one warp.
__device__ __forceinline__ void gm_pair_table_warp(const int* s_mt, int* s_mp, int G, int lane) {
    const int per = (G + 31) / 32;
    const int g0 = min(G, lane * per), g1 = min(G, g0 + per);
    int sum = 0;
    for (int g = g0; g < g1; ++g) sum += (s_mt[g + 1] - s_mt[g] + 1) / 2;
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    int run = incl - sum;
    for (int g = g0; g < g1; ++g) {
        s_mp[g] = run;
        run += (s_mt[g + 1] - s_mt[g] + 1) / 2;
    }
    if (lane == 31) s_mp[G] = incl;
}

// Work unit t -> (group g, M block mb, N block nb, K split ks). Units of one group are
// ordered N block, then M block, then K split.
__device__ __forceinline__ void gm_decode(long long t, int G, int n_tiles, int S, const int* s_mt,
                                          int& g, int& mb, int& nb, int& ks) {
    const long long per = (long long)n_tiles * S;   // units per M tile
    int lo = 0, hi = G;   // s_mt[lo]*per <= t < s_mt[hi]*per
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((long long)s_mt[mid] * per <= t) lo = mid;
        else hi = mid;
    }
    g = lo;
    const long long local = t - (long long)s_mt[g] * per;
    const int mt = s_mt[g + 1] - s_mt[g];
    const long long ms = (long long)mt * S;
    nb = (int)(local / ms);
    const int rem = (int)(local - (long long)nb * ms);
    mb = rem / S;
    ks = rem - mb * S;
}

// Raw fp32 accumulator of one unit -> its split-K partial rows.
template <int EPI>
__device__ __forceinline__ void gm_epilogue_partial(const GemmParams& p, uint32_t tb, int nb, int ks,
                                                    bool row_ok, long long grow) {
    float* prow = p.partial + (long long)ks * p.part_stride + grow * p.ld_part;
    const bool v8 = ((reinterpret_cast<uintptr_t>(p.partial) |
                      (uintptr_t)((p.part_stride | p.ld_part) * 4)) & 31) == 0;
    constexpr int chunks = GM_BN / 32;
#pragma unroll 1
    for (int c = 0; c < chunks; ++c) {
        float v[32];
        __syncwarp();
        tmem_load_32cols(tb + c * 32, v);
        int col;
        if constexpr (EPI == EPI_SWIGLU_BF16)
            col = (c < chunks / 2) ? nb * 128 + c * 32 : p.N + nb * 128 + (c - chunks / 2) * 32;
        else
            col = nb * GM_BN + c * 32;
        const int lim = (EPI == EPI_SWIGLU_BF16) ? ((c < chunks / 2) ? p.N : 2 * p.N) : p.N;
        if (row_ok && col < lim) {
            if (v8) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    st_global_v8(prow + col + 8 * i,
                                 make_float4(v[8 * i], v[8 * i + 1], v[8 * i + 2], v[8 * i + 3]),
                                 make_float4(v[8 * i + 4], v[8 * i + 5], v[8 * i + 6], v[8 * i + 7]));
            } else {
                float4* dst = reinterpret_cast<float4*>(prow + col);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
            }
        }
    }
}

template <int EPI>
__device__ __forceinline__ void gm_epilogue_tile(const GemmParams& p, uint32_t tb, int g, int nb,
                                                 bool row_ok, long long grow, int mb = 0,
                                                 int ks = 0, volatile int* s_flag = nullptr,
                                                 int* s_rh = nullptr, const CUtensorMap* tm_out = nullptr,
                                                 uint32_t out_stage = 0, bool tma = false) {
    // mb, ks, s_flag: EPI_ROUTER_TOPK with K split (see there); s_rh: that epilogue
    // warp's 64 histogram counters in shared memory
    // tma (fp32 epilogues, warp-uniform: the warp's 32 rows are consecutive output rows,
    // all in the group): each 32-column box is staged at out_stage (4 KB, 1024-byte
    // aligned, the 128-byte swizzle of tm_out) and written by one bulk tensor store
    const float* brow = p.bias ? p.bias + (long long)g * p.b_rows_per_group : nullptr;
    if (g == p.xg1 - 1) brow = p.xg_bias;   // the extra group (bf16 weights: no row scales)
    const float* srow = p.w_scale ? p.w_scale + (long long)g * p.b_rows_per_group : nullptr;
    if constexpr (EPI == EPI_SWIGLU_BF16) {
        const int n0 = nb * 128;
        __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) + grow * p.ld_out;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            float gv[32], uv[32];
            __syncwarp();
            tmem_load_2x32cols(tb + c * 32, tb + 128 + c * 32, gv, uv);
            const int col = n0 + c * 32;
            if (row_ok && col < p.N) {
                if (srow) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        gv[i] *= srow[col + i];
                        uv[i] *= srow[p.up_offset + col + i];
                    }
                }
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
                    packed[i] = pack_bf16x2(silu_fast(g0) * u0, silu_fast(g1) * u1);
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
                if (srow) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] *= srow[col + i];
                }
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
    } else if constexpr (EPI == EPI_ROUTER_TOPK) {
        // Logit e = term0 + term1 + term2 (+ bias[e]), then k rounds of arg-max (logit
        // descending, lower id on ties) and w_j = exp(L_j - L_0) / sum_j' exp(L_j' - L_0)
        // summed in slot order: the same fp32 operations as topk_renorm_kernel.
        constexpr int MAXE = 64;
        const int Ep = p.r_Ep, E = p.r_E, k = p.top_k;
        float L[MAXE];
#pragma unroll
        for (int c = 0; c < MAXE / 32; ++c) {
            if (c * 32 < Ep) {
                float a[32], b[32], d3[32];
                __syncwarp();
                tmem_load_32cols(tb + c * 32, a);
                tmem_load_32cols(tb + Ep + c * 32, b);
                tmem_load_32cols(tb + 2 * Ep + c * 32, d3);
#pragma unroll
                for (int i = 0; i < 32; ++i) L[c * 32 + i] = a[i] + b[i] + d3[i];
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) L[c * 32 + i] = 0.0f;
            }
        }
        if (p.k_splits > 1) {
            // K split in two parts (few M tiles): each part stores its partial logits; the
            // CTA whose part arrives second at the M tile adds the other part (a commutative
            // fp32 add, so the result does not depend on which one that is) and selects.
            // The four epilogue warps meet at named barrier 1.
            float* mine = p.r_part + ((long long)ks * p.r_rows + grow) * Ep;
            if (row_ok) {
#pragma unroll
                for (int e = 0; e < MAXE; e += 4)
                    if (e < Ep)
                        *reinterpret_cast<float4*>(mine + e) = make_float4(L[e], L[e + 1], L[e + 2], L[e + 3]);
            }
            __threadfence();
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (threadIdx.x == 64) *s_flag = atomicAdd(p.r_tile_cnt + mb, 1);
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (*s_flag != p.k_splits - 1) return;   // another part finishes this tile
            __threadfence();
            if (row_ok) {
                const float* other = p.r_part + ((long long)(1 - ks) * p.r_rows + grow) * Ep;
#pragma unroll
                for (int e = 0; e < MAXE; e += 4) {
                    if (e < Ep) {
                        const float4 v = __ldcg(reinterpret_cast<const float4*>(other + e));
                        L[e] += v.x;
                        L[e + 1] += v.y;
                        L[e + 2] += v.z;
                        L[e + 3] += v.w;
                    }
                }
            }
        }
        int ids[32];
        if (row_ok) {
            if (p.bias) {
#pragma unroll
                for (int e = 0; e < MAXE; ++e)
                    if (e < E) L[e] += p.bias[e];
            }
            if (p.out) {
                float* lrow = reinterpret_cast<float*>(p.out) + grow * p.ld_out;
#pragma unroll
                for (int e = 0; e < MAXE; ++e)
                    if (e < E) lrow[e] = L[e];
            }
            uint64_t taken = 0;
            float vals[32];
            for (int j = 0; j < k; ++j) {
                float bv = 0.0f;
                int be = -1;
#pragma unroll
                for (int e = 0; e < MAXE; ++e)
                    if (e < E && !((taken >> e) & 1ull) && (be < 0 || L[e] > bv)) {
                        bv = L[e];
                        be = e;
                    }
                taken |= 1ull << be;
                vals[j] = bv;
                ids[j] = be;
            }
            float ex[32];
            float ssum = 0.0f;
            for (int j = 0; j < k; ++j) {
                ex[j] = expf(vals[j] - vals[0]);
                ssum += ex[j];
            }
            for (int j = 0; j < k; ++j) {
                p.r_idx[grow * k + j] = ids[j];
                p.r_w[grow * k + j] = ex[j] / ssum;
            }
        }
        // The dispatch's expert histogram, one row per warp (32 consecutive tokens): the
        // lanes holding the same id in slot j form a __match_any_sync group whose lowest
        // lane adds the group's size to the warp's counters in shared memory (no atomics),
        // then the warp stores its row. Every row of a token block that holds a token is
        // written, so the rows need no zeroing.
        if (p.r_hist) {
            const int lane = threadIdx.x & 31;
            const unsigned lt_mask = (1u << lane) - 1u;
            s_rh[lane] = 0;
            s_rh[lane + 32] = 0;
            __syncwarp();
            for (int j = 0; j < k; ++j) {
                const int e = row_ok ? ids[j] : -1;
                const unsigned peers = __match_any_sync(0xffffffffu, e);
                if (e >= 0 && (peers & lt_mask) == 0) s_rh[e] += __popc(peers);
                __syncwarp();
            }
            const long long r32 = (grow - lane) >> 5;   // the warp's 32-token row
            if (grow - lane < p.r_rows) {
                int* hrow = p.r_hist + r32 * E;
                if (lane < E) hrow[lane] = s_rh[lane];
                if (lane + 32 < E) hrow[lane + 32] = s_rh[lane + 32];
            }
            __syncwarp();
        }
    } else if constexpr (EPI == EPI_COMBINE1_BF16) {
        // Same fp32 operations, in the same order, as the scale epilogue followed by the
        // combine kernel: y = (acc + b) * w, then out = resid + y (or 0 + y), rounded once.
        const int n0 = nb * GM_BN;
        long long tok = 0;
        float scale = 0.0f;
        if (row_ok) {
            tok = p.perm_token[grow];
            scale = p.topk_w[tok * p.top_k + p.perm_slot[grow]];
        }
        __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) + tok * p.ld_out;
        const __nv_bfloat16* xrow = p.resid ? p.resid + tok * p.ld_out : nullptr;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
            float v[32];
            __syncwarp();
            tmem_load_32cols(tb + c * 32, v);
            const int col = n0 + c * 32;
            if (row_ok && col < p.N) {
                if (srow) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] *= srow[col + i];
                }
                uint32_t xin[16];
                if (xrow) {
                    const uint4* xs = reinterpret_cast<const uint4*>(xrow + col);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint4 u = xs[i];
                        xin[4 * i] = u.x;
                        xin[4 * i + 1] = u.y;
                        xin[4 * i + 2] = u.z;
                        xin[4 * i + 3] = u.w;
                    }
                }
                uint32_t packed[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float y0 = (v[2 * i] + (brow ? brow[col + 2 * i] : 0.0f)) * scale;
                    float y1 = (v[2 * i + 1] + (brow ? brow[col + 2 * i + 1] : 0.0f)) * scale;
                    float a0 = 0.0f, a1 = 0.0f;
                    if (xrow) {
                        const __nv_bfloat162 xx = *reinterpret_cast<const __nv_bfloat162*>(&xin[i]);
                        const float2 xf = __bfloat1622float2(xx);
                        a0 = xf.x;
                        a1 = xf.y;
                    }
                    packed[i] = pack_bf16x2(a0 + y0, a1 + y1);
                }
                uint4* dst = reinterpret_cast<uint4*>(orow + col);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                                        packed[4 * i + 3]);
            }
        }
    } else if constexpr (EPI == EPI_SCALE_H16) {
        const int n0 = nb * GM_BN;
        const int lane = threadIdx.x & 31;
        float scale = 1.0f;
        if (row_ok) scale = p.topk_w[(long long)p.perm_token[grow] * p.top_k + p.perm_slot[grow]];
        __half* orow = reinterpret_cast<__half*>(p.out) + grow * p.ld_out;
        int8_t* erow = p.out_exp + grow * p.ld_exp;
        const bool v8 = ((reinterpret_cast<uintptr_t>(p.out) | (uintptr_t)(p.ld_out * 2)) & 31) == 0;
        // the tile row's 8 exponents leave as one 8-byte store when all 8 chunks are in N
        const bool whole = n0 + GM_BN <= p.N;
        uint32_t ex_lo = 0, ex_hi = 0;
#pragma unroll 1
        for (int c2 = 0; c2 < 8; c2 += 2) {   // two 32-column chunks per TMEM wait
            float vv[2][32];
            __syncwarp();
            tmem_load_2x32cols(tb + c2 * 32, tb + (c2 + 1) * 32, vv[0], vv[1]);
            uint32_t hp[2][16];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float (&v)[32] = vv[h];
                const int col = n0 + (c2 + h) * 32;
                // the fp32 operations of EPI_SCALE_F32, in its order
                float m = 0.0f;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    if (srow) v[i] *= srow[col + i];
                    v[i] = (v[i] + (brow ? brow[col + i] : 0.0f)) * scale;
                    const float a = fabsf(v[i]);
                    m = (a <= 3.40282347e38f) ? fmaxf(m, a) : m;   // finite values only
                }
                // 2^ex <= m < 2^(ex+1) for normal m; the chunk is stored as v * 2^-e, e = ex - 14
                const int ex = (int)((__float_as_uint(m) >> 23) & 0xffu) - 127;
                const int e = min(126, max(-126, ex - 14));
                const float inv = __uint_as_float((uint32_t)(127 - e) << 23);   // 2^-e
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const __half2 hh = __floats2half2_rn(v[2 * i] * inv, v[2 * i + 1] * inv);
                    hp[h][i] = *reinterpret_cast<const uint32_t*>(&hh);
                }
                const int cc = c2 + h;
                const uint32_t eb = (uint32_t)(e & 0xff) << (8 * (cc & 3));
                if (cc < 4) ex_lo |= eb;
                else ex_hi |= eb;
                if (!tma && row_ok && col < p.N) {
                    if (v8) {
                        st_global_v8_b32(orow + col, hp[h]);
                        st_global_v8_b32(orow + col + 16, hp[h] + 8);
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(orow + col);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_uint4(hp[h][4 * i], hp[h][4 * i + 1], hp[h][4 * i + 2],
                                                hp[h][4 * i + 3]);
                    }
                }
                if (!whole && row_ok && col < p.N) erow[col / 32] = (int8_t)e;
            }
            const int col2 = n0 + c2 * 32;
            if (tma && col2 < p.N) {
                // 64 columns (128 bytes) of the warp's 32 rows: one box
                if (lane == 0) bulk_wait_read_all();
                __syncwarp();
                const uint32_t rb = out_stage + lane * 128;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t* w = hp[i >> 2] + 4 * (i & 3);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(rb + ((i ^ (lane & 7)) << 4)),
                                 "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                                 : "memory");
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(tm_out, out_stage, col2, (int)grow);
                    bulk_commit();
                }
            }
        }
        if (whole && row_ok)
            *reinterpret_cast<uint2*>(erow + n0 / 32) = make_uint2(ex_lo, ex_hi);
    } else {
        const int n0 = nb * GM_BN;
        const int lane = threadIdx.x & 31;
        float scale = 1.0f;
        if constexpr (EPI == EPI_SCALE_F32) {
            if (row_ok)
                scale = p.topk_w[(long long)p.perm_token[grow] * p.top_k + p.perm_slot[grow]];
        }
        float* orow = reinterpret_cast<float*>(p.out) + grow * p.ld_out;
        // 32-byte stores when every row starts on a 32-byte boundary (the caller's buffers
        // need only 16-byte alignment)
        const bool v8 = ((reinterpret_cast<uintptr_t>(p.out) | (uintptr_t)(p.ld_out * 4)) & 31) == 0;
#pragma unroll 1
        for (int c2 = 0; c2 < 8; c2 += 2) {   // two 32-column chunks per TMEM wait
            float vv[2][32];
            __syncwarp();
            tmem_load_2x32cols(tb + c2 * 32, tb + (c2 + 1) * 32, vv[0], vv[1]);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float (&v)[32] = vv[h];
                const int col = n0 + (c2 + h) * 32;
                if ((row_ok || tma) && col < p.N) {
                    if (srow) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] *= srow[col + i];
                    }
                    float4 o[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        o[i].x = v[4 * i + 0] + (brow ? brow[col + 4 * i + 0] : 0.0f);
                        o[i].y = v[4 * i + 1] + (brow ? brow[col + 4 * i + 1] : 0.0f);
                        o[i].z = v[4 * i + 2] + (brow ? brow[col + 4 * i + 2] : 0.0f);
                        o[i].w = v[4 * i + 3] + (brow ? brow[col + 4 * i + 3] : 0.0f);
                        if constexpr (EPI == EPI_SCALE_F32) {
                            o[i].x *= scale;
                            o[i].y *= scale;
                            o[i].z *= scale;
                            o[i].w *= scale;
                        }
                    }
                    if (tma) {
                        // the previous box has left the staging buffer
                        if (lane == 0) bulk_wait_read_all();
                        __syncwarp();
                        const uint32_t rb = out_stage + lane * 128;
#pragma unroll
                        for (int i = 0; i < 8; ++i) st_shared_v4(rb + ((i ^ (lane & 7)) << 4), o[i]);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(tm_out, out_stage, col, (int)grow);
                            bulk_commit();
                        }
                    } else if (v8) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) st_global_v8(orow + col + 8 * i, o[2 * i], o[2 * i + 1]);
                    } else {
                        float4* dst = reinterpret_cast<float4*>(orow + col);
#pragma unroll
                        for (int i = 0; i < 8; ++i) dst[i] = o[i];
                    }
                }
            }
        }
    }
}

// 16-byte global -> shared copy that zero-fills when src_bytes is 0 (rows past a group).
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
constexpr int GM_GATHER_DEPTH = 2;   // stages a gather thread keeps in flight before arriving

template <int EPI, int MT = 1>
__global__ void __launch_bounds__(GM_THREADS + GM_GATHER_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmA2,
                        const __grid_constant__ CUtensorMap tmB2,
                        const __grid_constant__ CUtensorMap tmD, const GemmParams p) {
    // tmA2 / tmB2: A rows and weights of the extra group p.xg1 - 1 (copies of tmA / tmB
    // when the launch has none); tmD: the fp32 output [rows, N] in 32 x 32 boxes (used
    // when p.tma_out)
    static_assert(MT == 1 || MT == 2, "tiles are 128 or 256 rows");
    static_assert(MT == 1 || EPI != EPI_ROUTER_TOPK, "the router runs 128-row tiles");
    constexpr int STAGES = gm_stages(MT);
    constexpr int STAGE_BYTES = gm_stage_bytes(MT);
    constexpr int A_BYTES = MT * GM_A_BYTES;
    constexpr int BM = MT * GM_BM;
    constexpr int NACC = MT == 1 ? 2 : 1;   // accumulator sets in TMEM (256 x 128 lanes each)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* tiles = smem;
    // fp32 epilogues: the four epilogue warps' output staging boxes follow the ring
    uint8_t* out_stage = smem + STAGES * STAGE_BYTES;
    constexpr int OUT_BYTES = gm_stages_out(EPI) ? GM_OUT_STAGE_BYTES : 0;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES + OUT_BYTES);
    // barrier slots: full[0..3], empty[4..7], tfull[8..9], tempty[10..11], drain[12],
    // unit-id ring full[16..23] / empty[24..31]
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 32);
    volatile int* s_abort = reinterpret_cast<volatile int*>(bars + 33);
    volatile int* s_flag = reinterpret_cast<volatile int*>(bars + 34);   // router K split
    volatile long long* s_unit = reinterpret_cast<volatile long long*>(bars + 40);   // [GM_TQ]
    int* s_ro = reinterpret_cast<int*>(bars + GM_HDR_BYTES / 8);
    int* s_mt = s_ro + (p.G + 1);
    int* s_rh = s_mt + (p.G + 1);   // [4][64] router histogram counters
    int* s_mp = s_rh + 4 * 64;      // [G + 1] tile-pair offsets (pair mode)
    const bool pair = MT == 1 && p.pair;
    const uint32_t crank = pair ? cluster_ctarank() : 0u;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto bar = [&](int i) { return smem_addr(bars + i); };
    const int FULL = 0, EMPTY = GM_STAGES, TFULL = 2 * GM_STAGES, TEMPTY = 2 * GM_STAGES + 2,
              DRAIN = 2 * GM_STAGES + 4, QFULL = 16, QEMPTY = 16 + GM_TQ;

    const bool gather = p.a_gather != nullptr;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar(FULL + s), gather ? 5 : 1);   // + the four gather warps
            mbar_init(bar(EMPTY + s), pair ? 2 : 1);   // pair: both CTAs' MMAs
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar(TFULL + a), 1);
            mbar_init(bar(TEMPTY + a), 4);
        }
        mbar_init(bar(DRAIN), 1);
        for (int i = 0; i < GM_TQ; ++i) {
            mbar_init(bar(QFULL + i), 1);
            mbar_init(bar(QEMPTY + i), gather ? 9 : 5);   // MMA, 4 epilogue (+ 4 gather) warps
        }
        *s_abort = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (p.xg1) {
            tma_prefetch_desc(&tmA2);
            tma_prefetch_desc(&tmB2);
        }
        if (gm_stages_out(EPI) && p.tma_out) tma_prefetch_desc(&tmD);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(s_tmem), GM_TMEM_COLS);
        tmem_relinquish();
    }
    // pair: both CTAs' barriers are initialised before either multicasts into the other
    if (pair) cluster_sync_all();
    // Everything above is local set-up that may overlap the end of the preceding kernel;
    // the tables and operands may be its outputs.
    pdl_entry();
    for (int i = threadIdx.x; i <= p.G; i += blockDim.x) {
        s_ro[i] = p.row_offsets[i];
        if (MT == 1) s_mt[i] = p.mtile_offsets[i];
    }
    if (MT > 1) {   // tiles of BM rows: the table is formed here from the row offsets
        __syncthreads();
        if (warp == 2) gm_tile_table_warp(s_ro, s_mt, p.G, BM, lane);
    }
    if (pair) {
        __syncthreads();
        if (warp == 2) gm_pair_table_warp(s_mt, s_mp, p.G, lane);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;
    const long long total = pair ? (long long)s_mp[p.G] * p.n_tiles
                                 : (long long)s_mt[p.G] * p.n_tiles * p.k_splits;
    // unit t -> group, M tile, N block, K split (pair: tile 2 * pair index + this CTA's rank)
    auto decode = [&](long long t, int& g, int& mb, int& nb, int& ks) {
        if (pair) {
            gm_decode(t, p.G, p.n_tiles, 1, s_mp, g, mb, nb, ks);
            mb = 2 * mb + (int)crank;
        } else {
            gm_decode(t, p.G, p.n_tiles, p.k_splits, s_mt, g, mb, nb, ks);
        }
    };
    const int kblocks = p.K / GM_BK;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            int stage = 0;
            uint32_t ph = 0;
            int last_par[STAGES];
#pragma unroll
            for (int s = 0; s < STAGES; ++s) last_par[s] = -1;
            bool ok = true;
            int q = 0;
            uint32_t qph = 0;
            long long t = pair ? (long long)cluster_id_x() : (long long)blockIdx.x;
            while (true) {
                // publish the next unit id (-1: no more work) to the MMA and epilogue warps
                if (*s_abort || !mbar_wait(bar(QEMPTY + q), qph ^ 1)) {
                    *s_abort = 1;
                    break;
                }
                const long long pub = (ok && t < total) ? t : -1;
                s_unit[q] = pub;
                mbar_arrive(bar(QFULL + q));
                if (++q == GM_TQ) {
                    q = 0;
                    qph ^= 1;
                }
                if (pub < 0) break;
                const long long next =
                    pair ? t + (long long)cluster_count_x()
                    : p.tile_counter ? (long long)gridDim.x + (long long)atomicAdd(p.tile_counter, 1ull)
                                     : t + gridDim.x;
                int g, mb, nb, ks;
                decode(t, g, mb, nb, ks);
                const int kb0 = ks * p.kb_per_split;
                const int kb1 = min(kblocks, kb0 + p.kb_per_split);
                const bool xg = g == p.xg1 - 1;   // the extra group: its own A and B maps
                const CUtensorMap* mA = xg ? &tmA2 : &tmA;
                const CUtensorMap* mB = xg ? &tmB2 : &tmB;
                const int a_row = (xg ? 0 : s_ro[g]) + mb * BM;
                const int n0 = (EPI == EPI_SWIGLU_BF16) ? nb * 128 : nb * GM_BN;
                const int b0 = (xg ? 0 : g * p.b_rows_per_group) + n0;
                const int b1 = b0 + p.up_offset;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (*s_abort || !mbar_wait(bar(EMPTY + stage), ph ^ 1)) {
                        *s_abort = 1;
                        ok = false;
                        break;
                    }
                    const uint32_t sa = smem_addr(tiles + stage * STAGE_BYTES);
                    mbar_arrive_expect_tx(bar(FULL + stage), gather ? GM_B_BYTES : STAGE_BYTES);
                    if (!gather) {
#pragma unroll
                        for (int h = 0; h < MT; ++h)
                            tma_load_2d(sa + h * GM_A_BYTES, mA, bar(FULL + stage), kb * GM_BK,
                                        a_row + h * GM_BM);
                    }
                    if (pair) {   // this CTA's half of B, into both CTAs' stage
                        tma_load_2d_mc(sa + A_BYTES + crank * (GM_B_BYTES / 2), mB, bar(FULL + stage),
                                       kb * GM_BK, crank ? b1 : b0, (uint16_t)3);
                    } else {
                        tma_load_2d(sa + A_BYTES, mB, bar(FULL + stage), kb * GM_BK, b0);
                        tma_load_2d(sa + A_BYTES + GM_B_BYTES / 2, mB, bar(FULL + stage),
                                    kb * GM_BK, b1);
                    }
                    last_par[stage] = (int)ph;
                    if (++stage == STAGES) {
                        stage = 0;
                        ph ^= 1;
                    }
                }
                t = next;
            }
            // Every copy this thread started must have landed before the CTA exits.
            for (int s = 0; s < STAGES; ++s)
                if (last_par[s] >= 0) mbar_wait(bar(FULL + s), (uint32_t)last_par[s]);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            constexpr uint32_t idesc = idesc_bf16_f32(GM_BM, GM_BN);
            int stage = 0, acc = 0;
            uint32_t ph = 0, aph = 0;
            int q = 0;
            uint32_t qph = 0;
            while (true) {
                if (*s_abort || !mbar_wait(bar(QFULL + q), qph)) {
                    *s_abort = 1;
                    break;
                }
                const long long t = s_unit[q];
                mbar_arrive(bar(QEMPTY + q));
                if (++q == GM_TQ) {
                    q = 0;
                    qph ^= 1;
                }
                if (t < 0) break;
                // MT = 1: accumulator set acc (columns acc*256), freed as a whole.
                // MT = 2: halves h (columns h*256) freed one after the other (TEMPTY + h).
                if (*s_abort || !mbar_wait(bar(TEMPTY + acc), aph ^ 1)) {
                    *s_abort = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t dt = tmem_base + (uint32_t)(acc * GM_BN);
                const long long within = t % p.k_splits;   // the unit's K split
                const int kb0 = (int)within * p.kb_per_split;
                const int kb1 = min(kblocks, kb0 + p.kb_per_split);
                bool ok = true;
                int kb_start = kb0;
                if constexpr (MT == 2) {
                    // While the epilogue still drains half 1 of the previous tile, run half
                    // 0's MMAs over the first J stages of this one; then half 1's over the
                    // same stages, releasing them. Each half still accumulates in K order.
                    const int J = min(STAGES, kb1 - kb0);
                    int st = stage;
                    uint32_t sph = ph;
                    for (int j = 0; j < J && ok; ++j) {
                        if (!mbar_wait(bar(FULL + st), sph)) {
                            *s_abort = 1;
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sa = smem_addr(tiles + st * STAGE_BYTES);
#pragma unroll
                        for (int kk = 0; kk < GM_BK / 16; ++kk)
                            umma_bf16(dt, sw128_kmajor_desc(sa + kk * 32),
                                      sw128_kmajor_desc(sa + A_BYTES + kk * 32), idesc,
                                      (j != 0 || kk != 0) ? 1u : 0u);
                        if (++st == STAGES) {
                            st = 0;
                            sph ^= 1;
                        }
                    }
                    if (!ok) break;
                    if (*s_abort || !mbar_wait(bar(TEMPTY + 1), aph ^ 1)) {
                        *s_abort = 1;
                        break;
                    }
                    tc_fence_after();
                    for (int j = 0; j < J; ++j) {
                        const uint32_t sa = smem_addr(tiles + stage * STAGE_BYTES);
#pragma unroll
                        for (int kk = 0; kk < GM_BK / 16; ++kk)
                            umma_bf16(dt + GM_BN, sw128_kmajor_desc(sa + GM_A_BYTES + kk * 32),
                                      sw128_kmajor_desc(sa + A_BYTES + kk * 32), idesc,
                                      (j != 0 || kk != 0) ? 1u : 0u);
                        umma_commit(bar(EMPTY + stage));
                        if (++stage == STAGES) {
                            stage = 0;
                            ph ^= 1;
                        }
                    }
                    kb_start = kb0 + J;
                }
                for (int kb = kb_start; kb < kb1; ++kb) {
                    if (!mbar_wait(bar(FULL + stage), ph)) {
                        *s_abort = 1;
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_addr(tiles + stage * STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < GM_BK / 16; ++kk)
#pragma unroll
                        for (int h = 0; h < MT; ++h)
                            umma_bf16(dt + (uint32_t)(h * GM_BN),
                                      sw128_kmajor_desc(sa + h * GM_A_BYTES + kk * 32),
                                      sw128_kmajor_desc(sb + kk * 32), idesc,
                                      (kb != kb0 || kk != 0) ? 1u : 0u);
                    // pair: the stage is free once both CTAs' MMAs have read it
                    if (pair) umma_commit_mc(bar(EMPTY + stage), (uint16_t)3);
                    else umma_commit(bar(EMPTY + stage));
                    if (++stage == STAGES) {
                        stage = 0;
                        ph ^= 1;
                    }
                }
                if (!ok) break;
                umma_commit(bar(TFULL + acc));
                if (++acc == NACC) {
                    acc = 0;
                    aph ^= 1;
                }
            }
            // All MMAs issued by this thread must be complete before TMEM is freed.
            umma_commit(bar(DRAIN));
            mbar_wait(bar(DRAIN), 0);
        }
    } else if (warp >= 6) {
        // ---------------- A rows gathered with cp.async (warps 6..9) ----------------
        // Thread a copies 16-byte chunk (a & 7) of rows (a >> 3) + 16 i, i = 0..8*MT-1, of
        // each K block into the 128-byte-swizzled A tile. A stage's copies are waited for
        // (and made visible to the tensor core) GM_GATHER_DEPTH stages later, then the warp
        // arrives on the stage's FULL barrier.
        constexpr int RPT = 8 * MT;   // rows per thread
        const int a = threadIdx.x - GM_THREADS;
        const int chunk = a & 7, r0 = a >> 3;
        int stage = 0;
        uint32_t ph = 0;
        int q = 0;
        uint32_t qph = 0;
        int pend[GM_GATHER_DEPTH + 1];   // stages issued but not yet arrived, oldest first
#pragma unroll
        for (int i = 0; i <= GM_GATHER_DEPTH; ++i) pend[i] = 0;
        int npend = 0;
        auto release_oldest = [&]() {   // the oldest pending stage has landed: FULL
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(FULL + pend[0]));
#pragma unroll
            for (int i = 0; i < GM_GATHER_DEPTH; ++i) pend[i] = pend[i + 1];
            --npend;
        };
        bool ok = true;
        while (ok) {
            long long t = -1;
            int got = 1;
            if (lane == 0) {
                if (*s_abort || !mbar_wait(bar(QFULL + q), qph)) {
                    *s_abort = 1;
                    got = 0;
                } else {
                    t = s_unit[q];
                    mbar_arrive(bar(QEMPTY + q));
                }
            }
            if (++q == GM_TQ) {
                q = 0;
                qph ^= 1;
            }
            got = __shfl_sync(0xffffffffu, got, 0);
            t = __shfl_sync(0xffffffffu, t, 0);
            if (!got || t < 0) break;
            int g, mb, nb, ks;
            decode(t, g, mb, nb, ks);
            const int kb0 = ks * p.kb_per_split;
            const int kb1 = min(kblocks, kb0 + p.kb_per_split);
            const int rows_g = s_ro[g + 1] - s_ro[g];
            const uint8_t* src[RPT];
            uint32_t nbytes[RPT];
            const bool xg = g == p.xg1 - 1;   // the extra group reads row r of a_src
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                const int r = mb * BM + r0 + 16 * i;
                const bool valid = r < rows_g;
                const long long tok = valid ? (xg ? (long long)r : (long long)p.a_gather[s_ro[g] + r]) : 0;
                src[i] = p.a_src + tok * p.a_row_bytes + chunk * 16;
                nbytes[i] = valid ? 16u : 0u;
            }
            for (int kb = kb0; kb < kb1; ++kb) {
                const bool w_ok = !*s_abort && mbar_wait(bar(EMPTY + stage), ph ^ 1);
                if (!__all_sync(0xffffffffu, w_ok)) {
                    if (lane == 0) *s_abort = 1;
                    ok = false;
                    break;
                }
                const uint32_t sa = smem_addr(tiles + stage * STAGE_BYTES);
#pragma unroll
                for (int i = 0; i < RPT; ++i) {
                    const int r = r0 + 16 * i;   // row of the BM-row tile (halves are contiguous)
                    cp_async_16(sa + r * 128 + ((chunk ^ (r & 7)) << 4), src[i] + kb * GM_BK * 2,
                                nbytes[i]);
                }
                cp_async_commit();
                pend[npend++] = stage;
                if (npend > GM_GATHER_DEPTH) {
                    cp_async_wait<GM_GATHER_DEPTH>();
                    release_oldest();
                }
                if (++stage == STAGES) {
                    stage = 0;
                    ph ^= 1;
                }
            }
        }
        cp_async_wait<0>();
        while (npend > 0) release_oldest();
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        const int q = warp & 3;
        int acc = 0;
        uint32_t aph = 0;
        int uq = 0;
        uint32_t uqph = 0;
        while (true) {
            long long t = -1;
            int got = 1;
            if (lane == 0) {
                if (*s_abort || !mbar_wait(bar(QFULL + uq), uqph)) {
                    got = 0;
                } else {
                    t = s_unit[uq];
                    mbar_arrive(bar(QEMPTY + uq));
                }
            }
            got = __shfl_sync(0xffffffffu, got, 0);
            t = __shfl_sync(0xffffffffu, t, 0);
            if (++uq == GM_TQ) {
                uq = 0;
                uqph ^= 1;
            }
            if (!got) {
                if (lane == 0) *s_abort = 1;
                break;
            }
            if (t < 0) break;
            int g, mb, nb, ks;
            decode(t, g, mb, nb, ks);
            int ok = 1;
            if (lane == 0) ok = (!*s_abort && mbar_wait(bar(TFULL + acc), aph)) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) *s_abort = 1;
                break;
            }
            tc_fence_after();
            const int rows_g = s_ro[g + 1] - s_ro[g];
#pragma unroll 1
            for (int h = 0; h < MT; ++h) {
                const int r_in = h * GM_BM + q * 32 + lane;
                const int r_tile = mb * BM + r_in;   // row within the group
                const bool row_ok = r_tile < rows_g;
                const long long grow = p.out_local ? (long long)r_tile : (long long)s_ro[g] + r_tile;
                const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) +
                                    (uint32_t)((acc + h) * GM_BN);
                if (p.partial) {
                    gm_epilogue_partial<EPI>(p, tb, nb, ks, row_ok, grow);
                } else {
                    const bool tma = gm_stages_out(EPI) && p.tma_out && __all_sync(0xffffffffu, row_ok);
                    gm_epilogue_tile<EPI>(p, tb, g, nb, row_ok, grow, mb, ks, s_flag,
                                          s_rh + (warp & 3) * 64, &tmD,
                                          smem_addr(out_stage + q * (GM_OUT_STAGE_BYTES / 4)), tma);
                }
                if (MT == 2 && h == 0) {   // half 0 is free for the next tile's MMAs
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(TEMPTY + 0));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(TEMPTY + (MT == 2 ? 1 : acc)));
            if (++acc == NACC) {
                acc = 0;
                aph ^= 1;
            }
        }
        // the warp's bulk stores are written before the kernel ends
        if (gm_stages_out(EPI) && lane == 0) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, GM_TMEM_COLS);
    }
    // pair: neither CTA leaves while the other may still multicast into it or arrive on
    // its barriers
    if (pair) cluster_sync_all();
}

// ---- split-K reduction + epilogue ---------------------------------------------------
// For rows r < rows_total[0] (the kept rows P) and output columns c (4 per thread):
// sums the k_splits partials in split order, then applies the same epilogue as the
// unsplit kernel (bias, GELU / SwiGLU -> bf16, or routing-weight scale -> fp32).
template <int EPI>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const GemmParams p,
                                                            const int* __restrict__ rows_total) {
    pdl_entry();
    const int P = *rows_total;
    const int nq = p.N / 4;
    const long long work = (long long)P * nq;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < work;
         i += (long long)gridDim.x * blockDim.x) {
        const long long r = i / nq;
        const int c = (int)(i - r * nq) * 4;
        const float* src = p.partial + r * p.ld_part + c;
        float4 a = *reinterpret_cast<const float4*>(src);
        float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
        if constexpr (EPI == EPI_SWIGLU_BF16) u = *reinterpret_cast<const float4*>(src + p.N);
        for (int s = 1; s < p.k_splits; ++s) {
            const float4 v = *reinterpret_cast<const float4*>(src + s * p.part_stride);
            a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
            if constexpr (EPI == EPI_SWIGLU_BF16) {
                const float4 w = *reinterpret_cast<const float4*>(src + s * p.part_stride + p.N);
                u.x += w.x; u.y += w.y; u.z += w.z; u.w += w.w;
            }
        }
        if (p.bias || p.w_scale) {
            int lo = 0, hi = p.G;   // row_offsets[lo] <= r < row_offsets[hi]
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (p.row_offsets[mid] <= r) lo = mid;
                else hi = mid;
            }
            if (p.w_scale) {
                const float* sc = p.w_scale + (long long)lo * p.b_rows_per_group + c;
                a.x *= sc[0]; a.y *= sc[1]; a.z *= sc[2]; a.w *= sc[3];
                if constexpr (EPI == EPI_SWIGLU_BF16) {
                    const float* su = sc + p.up_offset;
                    u.x *= su[0]; u.y *= su[1]; u.z *= su[2]; u.w *= su[3];
                }
            }
        }
        if (p.bias) {
            int lo = 0, hi = p.G;   // row_offsets[lo] <= r < row_offsets[hi]
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (p.row_offsets[mid] <= r) lo = mid;
                else hi = mid;
            }
            const float* b = p.bias + (long long)lo * p.b_rows_per_group + c;
            a.x += b[0]; a.y += b[1]; a.z += b[2]; a.w += b[3];
            if constexpr (EPI == EPI_SWIGLU_BF16) {
                const float* bu = b + p.up_offset;
                u.x += bu[0]; u.y += bu[1]; u.z += bu[2]; u.w += bu[3];
            }
        }
        if constexpr (EPI == EPI_SWIGLU_BF16 || EPI == EPI_GELU_BF16) {
            float h0, h1, h2, h3;
            if constexpr (EPI == EPI_SWIGLU_BF16) {
                h0 = silu_fast(a.x) * u.x; h1 = silu_fast(a.y) * u.y; h2 = silu_fast(a.z) * u.z;
                h3 = silu_fast(a.w) * u.w;
            } else {
                h0 = gelu_erf(a.x); h1 = gelu_erf(a.y); h2 = gelu_erf(a.z); h3 = gelu_erf(a.w);
            }
            uint2 o;
            o.x = pack_bf16x2(h0, h1);
            o.y = pack_bf16x2(h2, h3);
            *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.out) + r * p.ld_out + c) = o;
        } else {
            if constexpr (EPI == EPI_SCALE_F32) {
                const float sc = p.topk_w[(long long)p.perm_token[r] * p.top_k + p.perm_slot[r]];
                a.x *= sc; a.y *= sc; a.z *= sc; a.w *= sc;
            }
            *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + r * p.ld_out + c) = a;
        }
    }
}

}  // namespace moe
