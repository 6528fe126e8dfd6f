// Grouped GEMM with weight-only INT8 or INT4 weights for groups of few rows (decode).
//
// "MoE 混合专家架构" 5.3 量化支持: INT8 / INT4 expert weights,
// D[r][n] = s[n] * sum_k A[r][k] * q[n][k].
// With a handful of token rows per expert the layer is a stream of weight codes; widening
// the codes in shared memory (grouped_gemm_q8_kernel) costs six bytes of shared-memory
// traffic per code and caps the stream below the HBM rate. Here the roles of the operands
// are swapped: the weight tile is the MMA's A operand (M = 128 weight rows), widened from
// int8 to bf16 in registers and stored straight into TMEM, and up to QT_NT = 32 rows of
// activations form the B operand (N = 32) in shared memory. Shared memory then carries
// the codes once in (TMA) and once out (converters), plus the small activation tile.
//
// A work unit is (group g, 256 weight rows nb, 32 activation rows mb, K split ks); its two
// 128-row halves h = 0, 1 (SwiGLU: gate and up rows of the same 128 features) go to two
// TMEM accumulators of 32 columns each. K advances in blocks of QT_BK = 128 codes, so that
// each weight row is read from HBM in 128-byte pieces. TMEM columns: accumulator a, half
// h at a*64 + h*32; widened A stage c, half h at 128 + c*128 + h*64 (64 columns = 128 bf16
// of K). A K tail of 64 reads zero codes and zero activations past the end of the rows.
// INT4 codes (BITS = 4) are packed two per byte along K (even k in the low nibble), so a
// 128-byte box row holds 256 codes: each code stage then feeds two TMEM stages of 128
// codes, and K splits start on a code stage (an even number of 128-code blocks).
// bf16 weights (BITS = 16, no row scales) stream the same way for decode-sized groups:
// a 128-byte box row holds 64 weights, so two code stages feed one TMEM stage, and the
// converters copy the rows into TMEM unchanged.
//   warp 0       unit scheduler + TMA of the codes (two 128-row boxes of 128 bytes,
//                128-byte swizzle) into a QT_NQ-deep ring;
//   warps 1, 15  MMA issuers (A from TMEM, B from shared memory), warp 1 for the weight
//                rows of half 0 and warp 15 for half 1: each tcgen05.mma with A in TMEM
//                holds its issuing thread far longer than the tensor pipe needs for it,
//                so two issuers keep twice the MMAs in flight;
//   warps 2-5    epilogue: lane = weight row (output feature), column = activation row;
//   warp 6       TMA of the bf16 activation rows into a QT_NB-deep ring;
//   warps 7-14   converters: warp 7 + 4h + i widens rows 32q .. 32q+31 (q = warp % 4, the
//                TMEM lane quarter the warp may access) of half h into a QT_NC-deep
//                ring of TMEM stages.
// The tile table over 32-row activation tiles is built by each CTA from the row offsets.
#pragma once
#include "grouped_gemm_q8.cuh"

namespace moe {

constexpr int QT_NT = 32;                           // activation rows per tile (MMA N)
constexpr int QT_BK = 128;                          // codes per K block (MMA and TMEM stage)
constexpr int QT_NQ = 5, QT_NB = 4, QT_NC = 3;
constexpr int QT_Q_BYTES = GM_BN * QT_BK;           // 256 weight rows x 128 bytes = 32 KB
constexpr int QT_B_BYTES = QT_NT * QT_BK * 2;       // 32 rows x 128 bf16 = 8 KB (two boxes)
constexpr int QT_RING_BYTES = QT_NQ * QT_Q_BYTES + QT_NB * QT_B_BYTES;
constexpr int QT_HDR_BYTES = 1024;
constexpr int QT_THREADS = 512;
constexpr int QT_TMEM_COLS = 512;
constexpr int QT_ACC_COL = 0, QT_A_COL = 128;
static_assert(QT_A_COL + QT_NC * 2 * (QT_BK / 4) <= QT_TMEM_COLS, "TMEM columns overflow");

__host__ __device__ constexpr int gm_q8t_smem_bytes(int G) {
    return 1024 + QT_RING_BYTES + QT_HDR_BYTES + 2 * (G + 1) * 4;
}

// Four-bit codes -> bf16, exactly and without conversion instructions: nibble v (two's
// complement code q) xor 8 is u = q + 8 in 0..15; the bf16 pattern 0x4300 | u is 128 + u
// (bf16 keeps 7 fraction bits, enough for 4), and subtracting 136 leaves q. Word w holds
// codes k..k+7 of a row (nibble i = code k+i); the mask pairs nibbles i and i+4 in the
// two halves of a word, and a byte permute re-pairs them as (k+2j, k+2j+1).
__device__ __forceinline__ void widen8_i4(uint32_t w, uint32_t (&o)[4]) {
    constexpr uint32_t k136 = 0x43084308u;   // bf16 136.0 in both halves
    uint32_t pr[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t b = ((w >> (4 * i)) & 0x000F000Fu) ^ k136;   // 128 + u of (k+i, k+i+4)
        const __nv_bfloat162 v = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&b),
                                         *reinterpret_cast<const __nv_bfloat162*>(&k136));
        pr[i] = *reinterpret_cast<const uint32_t*>(&v);
    }
    o[0] = __byte_perm(pr[0], pr[1], 0x5410);   // (k, k+1)
    o[1] = __byte_perm(pr[2], pr[3], 0x5410);   // (k+2, k+3)
    o[2] = __byte_perm(pr[0], pr[1], 0x7632);   // (k+4, k+5)
    o[3] = __byte_perm(pr[2], pr[3], 0x7632);   // (k+6, k+7)
}

// One half of a unit's accumulator (32 activation rows of weight row / feature f) ->
// split-K partials or the epilogue's output.
template <int EPI>
__device__ __forceinline__ void qt_store_half(const GemmParams& p, const float (&v)[32], int g,
                                              int f, int ks, long long row0, int nvalid) {
    if (f >= p.N) return;
    if (p.partial) {
        float* P = p.partial + (long long)ks * p.part_stride + row0 * p.ld_part + f;
#pragma unroll
        for (int j = 0; j < QT_NT; ++j)
            if (j < nvalid) P[(long long)j * p.ld_part] = v[j];
        return;
    }
    const long long wrow = (long long)g * p.b_rows_per_group + f;
    const float s = p.w_scale ? p.w_scale[wrow] : 1.0f;
    const float b = p.bias ? p.bias[wrow] : 0.0f;
    if constexpr (EPI == EPI_GELU_BF16) {
        __nv_bfloat16* O = reinterpret_cast<__nv_bfloat16*>(p.out) + row0 * p.ld_out + f;
#pragma unroll
        for (int j = 0; j < QT_NT; ++j)
            if (j < nvalid) O[(long long)j * p.ld_out] = __float2bfloat16_rn(gelu_erf(v[j] * s + b));
    } else {
        float* O = reinterpret_cast<float*>(p.out) + row0 * p.ld_out + f;
#pragma unroll
        for (int j = 0; j < QT_NT; ++j) {
            if (j < nvalid) {
                float o = v[j] * s + b;
                if constexpr (EPI == EPI_SCALE_F32)
                    o *= p.topk_w[(long long)p.perm_token[row0 + j] * p.top_k + p.perm_slot[row0 + j]];
                O[(long long)j * p.ld_out] = o;
            }
        }
    }
}

template <int EPI, int BITS>
__global__ void __launch_bounds__(QT_THREADS, 1)
    grouped_gemm_q8t_kernel(const __grid_constant__ CUtensorMap tmA,
                            const __grid_constant__ CUtensorMap tmQ, const GemmParams p) {
    static_assert(EPI == EPI_GELU_BF16 || EPI == EPI_SWIGLU_BF16 || EPI == EPI_SCALE_F32 ||
                      EPI == EPI_F32,
                  "epilogue not supported by the swapped INT8 kernel");
    static_assert(BITS == 8 || BITS == 4 || BITS == 16, "codes are 8 or 4 bits wide, or bf16");
    constexpr int KPQ = BITS == 16 ? 1 : 8 / BITS;   // 128-code K blocks per code stage
    constexpr int QPK = BITS == 16 ? 2 : 1;          // code stages per 128-code K block
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* q_tiles = smem;                                   // NQ x 32 KB of codes
    uint8_t* b_tiles = smem + QT_NQ * QT_Q_BYTES;              // NB x 8 KB bf16 activations
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + QT_RING_BYTES);
    const int QFULL = 0, QEMPTY = QT_NQ, BFULL = 2 * QT_NQ, BEMPTY = BFULL + QT_NB,
              CFULL = BEMPTY + QT_NB, CEMPTY = CFULL + QT_NC, TFULL = CEMPTY + QT_NC,
              TEMPTY = TFULL + 2, DRAIN = TEMPTY + 2, UFULL = 48, UEMPTY = 48 + GM_TQ;
    static_assert(2 * (QT_NQ + QT_NB + QT_NC) + 5 <= 48, "barrier slots overlap");
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 64);
    volatile int* s_abort = reinterpret_cast<volatile int*>(bars + 65);
    volatile long long* s_unit = reinterpret_cast<volatile long long*>(bars + 66);   // [GM_TQ]
    static_assert((66 + GM_TQ) * 8 <= QT_HDR_BYTES && 48 + 2 * GM_TQ <= 64, "header overflow");
    int* s_ro = reinterpret_cast<int*>(bars + QT_HDR_BYTES / 8);
    int* s_mt = s_ro + (p.G + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto bar = [&](int i) { return smem_addr(bars + i); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < QT_NQ; ++s) {
            mbar_init(bar(QFULL + s), 1);
            mbar_init(bar(QEMPTY + s), 8);    // the eight converter warps
        }
        for (int s = 0; s < QT_NB; ++s) {
            mbar_init(bar(BFULL + s), 1);
            mbar_init(bar(BEMPTY + s), 2);    // the two MMA issuers' commits
        }
        for (int s = 0; s < QT_NC; ++s) {
            mbar_init(bar(CFULL + s), 8);     // the eight converter warps
            mbar_init(bar(CEMPTY + s), 2);    // the two MMA issuers' commits
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar(TFULL + a), 2);
            mbar_init(bar(TEMPTY + a), 4);
        }
        mbar_init(bar(DRAIN), 2);
        for (int i = 0; i < GM_TQ; ++i) {
            mbar_init(bar(UFULL + i), 1);
            mbar_init(bar(UEMPTY + i), 15);  // 2 MMA, B producer, 4 epilogue, 8 converter warps
        }
        *s_abort = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmQ);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(s_tmem), QT_TMEM_COLS);
        tmem_relinquish();
    }
    pdl_entry();
    for (int i = threadIdx.x; i <= p.G; i += blockDim.x) s_ro[i] = p.row_offsets[i];
    __syncthreads();
    if (warp == 0) {   // tile table: s_mt[g] = sum over g' < g of ceil(rows_g' / QT_NT)
        int carry = 0;
        for (int base = 0; base < p.G; base += 32) {
            const int g = base + lane;
            int v = g < p.G ? (max(0, s_ro[g + 1] - s_ro[g]) + QT_NT - 1) / QT_NT : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, v, off);
                if (lane >= off) v += n;
            }
            if (g < p.G) s_mt[g + 1] = carry + v;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) s_mt[0] = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;
    const long long total = (long long)s_mt[p.G] * p.n_tiles * p.k_splits;
    const int kblocks = (p.K + QT_BK - 1) / QT_BK;

    // Takes the next unit id from the ring (one thread); false when the kernel aborts.
    auto take_unit = [&](int& q, uint32_t& qph, long long& t) -> bool {
        if (*s_abort || !mbar_wait(bar(UFULL + q), qph)) {
            *s_abort = 1;
            return false;
        }
        t = s_unit[q];
        mbar_arrive(bar(UEMPTY + q));
        if (++q == GM_TQ) {
            q = 0;
            qph ^= 1;
        }
        return true;
    };
    // The same, for a whole warp (lane 0 takes the id and broadcasts it).
    auto warp_take_unit = [&](int& q, uint32_t& qph, long long& t) -> bool {
        int got = 1;
        t = -1;
        if (lane == 0) got = take_unit(q, qph, t) ? 1 : 0;
        got = __shfl_sync(0xffffffffu, got, 0);
        t = __shfl_sync(0xffffffffu, t, 0);
        return got && t >= 0;
    };

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- unit scheduler + TMA of the int8 weight codes ----------------
            int stage = 0;
            uint32_t ph = 0;
            int last_par[QT_NQ];
#pragma unroll
            for (int s = 0; s < QT_NQ; ++s) last_par[s] = -1;
            bool ok = true;
            int q = 0;
            uint32_t qph = 0;
            long long t = blockIdx.x;
            while (true) {
                if (*s_abort || !mbar_wait(bar(UEMPTY + q), qph ^ 1)) {
                    *s_abort = 1;
                    break;
                }
                const long long pub = (ok && t < total) ? t : -1;
                s_unit[q] = pub;
                mbar_arrive(bar(UFULL + q));
                if (++q == GM_TQ) {
                    q = 0;
                    qph ^= 1;
                }
                if (pub < 0) break;
                const long long next =
                    p.tile_counter ? (long long)gridDim.x + (long long)atomicAdd(p.tile_counter, 1ull)
                                   : t + gridDim.x;
                int g, mb, nb, ks;
                gm_decode(t, p.G, p.n_tiles, p.k_splits, s_mt, g, mb, nb, ks);
                const int kb0 = ks * p.kb_per_split;
                const int kb1 = min(kblocks, kb0 + p.kb_per_split);
                const int n0 = (EPI == EPI_SWIGLU_BF16) ? nb * 128 : nb * GM_BN;
                const int b0 = g * p.b_rows_per_group + n0;
                const int b1 = b0 + p.up_offset;
                // code stage kb holds 128-code blocks KPQ*kb .. KPQ*kb + KPQ-1 (x = kb * 128
                // bytes); bf16: stages 2 kb and 2 kb + 1 hold the halves of block kb
                for (int kb = kb0 * QPK / KPQ; kb < (kb1 * QPK + KPQ - 1) / KPQ; ++kb) {
                    if (*s_abort || !mbar_wait(bar(QEMPTY + stage), ph ^ 1)) {
                        *s_abort = 1;
                        ok = false;
                        break;
                    }
                    const uint32_t sq = smem_addr(q_tiles + stage * QT_Q_BYTES);
                    mbar_arrive_expect_tx(bar(QFULL + stage), QT_Q_BYTES);
                    tma_load_2d(sq, &tmQ, bar(QFULL + stage), kb * QT_BK, b0);
                    tma_load_2d(sq + QT_Q_BYTES / 2, &tmQ, bar(QFULL + stage), kb * QT_BK, b1);
                    last_par[stage] = (int)ph;
                    if (++stage == QT_NQ) {
                        stage = 0;
                        ph ^= 1;
                    }
                }
                t = next;
            }
            for (int s = 0; s < QT_NQ; ++s)
                if (last_par[s] >= 0) mbar_wait(bar(QFULL + s), (uint32_t)last_par[s]);
        }
    } else if (warp == 6) {
        if (lane == 0) {
            // ---------------- TMA of the activation rows (B operand) --------------------
            int stage = 0;
            uint32_t ph = 0;
            int last_par[QT_NB];
#pragma unroll
            for (int s = 0; s < QT_NB; ++s) last_par[s] = -1;
            int q = 0;
            uint32_t qph = 0;
            bool ok = true;
            while (ok) {
                long long t;
                if (!take_unit(q, qph, t) || t < 0) break;
                int g, mb, nb, ks;
                gm_decode(t, p.G, p.n_tiles, p.k_splits, s_mt, g, mb, nb, ks);
                const int kb0 = ks * p.kb_per_split;
                const int kb1 = min(kblocks, kb0 + p.kb_per_split);
                const int a_row = s_ro[g] + mb * QT_NT;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (*s_abort || !mbar_wait(bar(BEMPTY + stage), ph ^ 1)) {
                        *s_abort = 1;
                        ok = false;
                        break;
                    }
                    const uint32_t sb = smem_addr(b_tiles + stage * QT_B_BYTES);
                    mbar_arrive_expect_tx(bar(BFULL + stage), QT_B_BYTES);
                    tma_load_2d(sb, &tmA, bar(BFULL + stage), kb * QT_BK, a_row);
                    tma_load_2d(sb + QT_B_BYTES / 2, &tmA, bar(BFULL + stage), kb * QT_BK + 64, a_row);
                    last_par[stage] = (int)ph;
                    if (++stage == QT_NB) {
                        stage = 0;
                        ph ^= 1;
                    }
                }
            }
            for (int s = 0; s < QT_NB; ++s)
                if (last_par[s] >= 0) mbar_wait(bar(BFULL + s), (uint32_t)last_par[s]);
        }
    } else if (warp >= 7 && warp < 15) {
        // ---------------- converters: int8 / int4 codes -> bf16 A operand in TMEM ----------
        const int qd = warp & 3, h = (warp - 7) >> 2;
        const int r = h * 128 + qd * 32 + lane;          // weight row of the stage
        const int sw = r & 7;                            // 128-byte swizzle of that row
        const uint32_t t_lane = tmem_base + ((uint32_t)(qd * 32) << 16) + QT_A_COL + h * 64;
        int qs = 0, cs = 0;
        uint32_t qph = 0, cph = 0;
        int uq = 0;
        uint32_t uqph = 0;
        // 64 codes (chunks c0 .. c0+3 of the row) -> 32 bf16x2 columns
        auto widen_half = [&](const uint8_t* row, int c0, uint32_t (&v)[32]) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint4 w = *reinterpret_cast<const uint4*>(row + (((c0 + c) ^ sw) << 4));
                widen4(w.x, v[8 * c + 0], v[8 * c + 1]);
                widen4(w.y, v[8 * c + 2], v[8 * c + 3]);
                widen4(w.z, v[8 * c + 4], v[8 * c + 5]);
                widen4(w.w, v[8 * c + 6], v[8 * c + 7]);
            }
        };
        // 64 four-bit codes (chunks c0, c0+1 of the row) -> 32 bf16x2 columns
        auto widen_half4 = [&](const uint8_t* row, int c0, uint32_t (&v)[32]) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const uint4 w = *reinterpret_cast<const uint4*>(row + (((c0 + c) ^ sw) << 4));
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t o[4];
                    widen8_i4(ws[j], o);
#pragma unroll
                    for (int i = 0; i < 4; ++i) v[16 * c + 4 * j + i] = o[i];
                }
            }
        };
        bool ok = true;
        while (ok) {
            long long t;
            if (!warp_take_unit(uq, uqph, t)) break;
            int g, mb, nb, ks;
            gm_decode(t, p.G, p.n_tiles, p.k_splits, s_mt, g, mb, nb, ks);
            const int kb0 = ks * p.kb_per_split;
            const int kb1 = min(kblocks, kb0 + p.kb_per_split);
            for (int kb = kb0; kb < kb1; ++kb) {
                if constexpr (BITS == 16) {
                    // bf16: codes 0..63 of the block from code stage qs, 64..127 from the next;
                    // each stage is released once its half is copied
                    const bool w_ok = !*s_abort && mbar_wait(bar(CEMPTY + cs), cph ^ 1);
                    if (!__all_sync(0xffffffffu, w_ok)) {
                        if (lane == 0) *s_abort = 1;
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    uint32_t v[2][32];
                    bool got = true;
#pragma unroll
                    for (int hs = 0; hs < 2; ++hs) {
                        const bool q_ok = !*s_abort && mbar_wait(bar(QFULL + qs), qph);
                        if (!__all_sync(0xffffffffu, q_ok)) {
                            got = false;
                            break;
                        }
                        const uint8_t* row = q_tiles + qs * QT_Q_BYTES + r * QT_BK;
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const uint4 w = *reinterpret_cast<const uint4*>(row + ((c ^ sw) << 4));
                            v[hs][4 * c + 0] = w.x;
                            v[hs][4 * c + 1] = w.y;
                            v[hs][4 * c + 2] = w.z;
                            v[hs][4 * c + 3] = w.w;
                        }
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(QEMPTY + qs));   // codes consumed
                        if (++qs == QT_NQ) {
                            qs = 0;
                            qph ^= 1;
                        }
                    }
                    if (!got) {
                        if (lane == 0) *s_abort = 1;
                        ok = false;
                        break;
                    }
                    tmem_store_32cols(t_lane + cs * 128, v[0]);
                    tmem_store_32cols(t_lane + cs * 128 + 32, v[1]);
                    tmem_store_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(CFULL + cs));
                    if (++cs == QT_NC) {
                        cs = 0;
                        cph ^= 1;
                    }
                    continue;
                }
                // sub: the 128-code block of the code stage. The stage's first block waits
                // for the codes; its last block (or the unit's last) releases them.
                const int sub = (kb - kb0) % KPQ;
                const bool w_ok = !*s_abort && (sub != 0 || mbar_wait(bar(QFULL + qs), qph)) &&
                                  mbar_wait(bar(CEMPTY + cs), cph ^ 1);
                if (!__all_sync(0xffffffffu, w_ok)) {
                    if (lane == 0) *s_abort = 1;
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint8_t* row = q_tiles + qs * QT_Q_BYTES + r * QT_BK;
                uint32_t v0[32], v1[32];
                if constexpr (BITS == 8) {
                    widen_half(row, 0, v0);
                    widen_half(row, 4, v1);
                    tmem_store_32cols(t_lane + cs * 128, v0);
                    tmem_store_32cols(t_lane + cs * 128 + 32, v1);
                } else {
                    // 4-bit codes: the first 64 codes' TMEM store is in flight while the
                    // next 64 are widened (both register sets stay untouched until the wait);
                    // measured faster for INT4 and slower for INT8, whose loads of the second
                    // half then no longer overlap the first half's widening
                    widen_half4(row, 4 * sub, v0);
                    tmem_store_32cols(t_lane + cs * 128, v0);
                    widen_half4(row, 4 * sub + 2, v1);
                    tmem_store_32cols(t_lane + cs * 128 + 32, v1);
                }
                __syncwarp();
                const bool q_done = sub == KPQ - 1 || kb == kb1 - 1;
                if (q_done && lane == 0) mbar_arrive(bar(QEMPTY + qs));   // codes consumed
                tmem_store_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(CFULL + cs));
                if (q_done && ++qs == QT_NQ) {
                    qs = 0;
                    qph ^= 1;
                }
                if (++cs == QT_NC) {
                    cs = 0;
                    cph ^= 1;
                }
            }
        }
    } else if (warp == 1 || warp == 15) {
        if (lane == 0) {
            // ---------------- MMA issuers: warp 1 half 0, warp 15 half 1 ----------------
            const int hh = warp == 1 ? 0 : 1;
            constexpr uint32_t idesc = idesc_bf16_f32(128, QT_NT);
            int bs = 0, cs = 0, acc = 0;
            uint32_t bph = 0, cph = 0, aph = 0;
            int q = 0;
            uint32_t qph = 0;
            while (true) {
                long long t;
                if (!take_unit(q, qph, t) || t < 0) break;
                if (*s_abort || !mbar_wait(bar(TEMPTY + acc), aph ^ 1)) {
                    *s_abort = 1;
                    break;
                }
                tc_fence_after();
                const int kb0 = (int)(t % p.k_splits) * p.kb_per_split;
                const int kb1 = min(kblocks, kb0 + p.kb_per_split);
                bool ok = true;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(bar(CFULL + cs), cph) || !mbar_wait(bar(BFULL + bs), bph)) {
                        *s_abort = 1;
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sb = smem_addr(b_tiles + bs * QT_B_BYTES);
                    const uint32_t dt = tmem_base + QT_ACC_COL + acc * 64 + hh * 32;
                    const uint32_t at = tmem_base + QT_A_COL + cs * 128 + hh * 64;
#pragma unroll
                    for (int kk = 0; kk < QT_BK / 16; ++kk)   // B: two 64-wide K boxes
                        umma_bf16_tmem_a(dt, at + kk * 8,
                                         sw128_kmajor_desc(sb + (kk >> 2) * (QT_B_BYTES / 2) +
                                                           (kk & 3) * 32),
                                         idesc, (kb != kb0 || kk != 0) ? 1u : 0u);
                    umma_commit(bar(CEMPTY + cs));
                    umma_commit(bar(BEMPTY + bs));
                    if (++bs == QT_NB) {
                        bs = 0;
                        bph ^= 1;
                    }
                    if (++cs == QT_NC) {
                        cs = 0;
                        cph ^= 1;
                    }
                }
                if (!ok) break;
                umma_commit(bar(TFULL + acc));
                acc ^= 1;
                if (acc == 0) aph ^= 1;
            }
            umma_commit(bar(DRAIN));
            mbar_wait(bar(DRAIN), 0);
        }
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        const int qd = warp & 3;
        const int m = qd * 32 + lane;   // weight row within a half
        int acc = 0;
        uint32_t aph = 0;
        int uq = 0;
        uint32_t uqph = 0;
        while (true) {
            long long t;
            if (!warp_take_unit(uq, uqph, t)) break;
            int g, mb, nb, ks;
            gm_decode(t, p.G, p.n_tiles, p.k_splits, s_mt, g, mb, nb, ks);
            int ok = 1;
            if (lane == 0) ok = (!*s_abort && mbar_wait(bar(TFULL + acc), aph)) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) *s_abort = 1;
                break;
            }
            tc_fence_after();
            float a0[32], a1[32];
            const uint32_t tb = tmem_base + ((uint32_t)(qd * 32) << 16) + QT_ACC_COL + acc * 64;
            tmem_load_32cols(tb, a0);
            tmem_load_32cols(tb + 32, a1);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(TEMPTY + acc));   // accumulator free again
            acc ^= 1;
            if (acc == 0) aph ^= 1;

            const int r0 = mb * QT_NT;
            const int nvalid = min(QT_NT, s_ro[g + 1] - s_ro[g] - r0);
            const long long row0 = (long long)s_ro[g] + r0;
            if constexpr (EPI == EPI_SWIGLU_BF16) {
                const int f = nb * 128 + m;
                if (f < p.N) {
                    if (p.partial) {
                        float* P = p.partial + (long long)ks * p.part_stride + row0 * p.ld_part + f;
#pragma unroll
                        for (int j = 0; j < QT_NT; ++j) {
                            if (j < nvalid) {
                                P[(long long)j * p.ld_part] = a0[j];
                                P[(long long)j * p.ld_part + p.N] = a1[j];
                            }
                        }
                    } else {
                        const long long wg = (long long)g * p.b_rows_per_group + f;
                        const float sg = p.w_scale ? p.w_scale[wg] : 1.0f;
                        const float su = p.w_scale ? p.w_scale[wg + p.up_offset] : 1.0f;
                        const float bg = p.bias ? p.bias[wg] : 0.0f;
                        const float bu = p.bias ? p.bias[wg + p.up_offset] : 0.0f;
                        __nv_bfloat16* O = reinterpret_cast<__nv_bfloat16*>(p.out) + row0 * p.ld_out + f;
#pragma unroll
                        for (int j = 0; j < QT_NT; ++j)
                            if (j < nvalid)
                                O[(long long)j * p.ld_out] =
                                    __float2bfloat16_rn(silu_fast(a0[j] * sg + bg) * (a1[j] * su + bu));
                    }
                }
            } else {
                qt_store_half<EPI>(p, a0, g, nb * GM_BN + m, ks, row0, nvalid);
                qt_store_half<EPI>(p, a1, g, nb * GM_BN + 128 + m, ks, row0, nvalid);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, QT_TMEM_COLS);
    }
}

}  // namespace moe
