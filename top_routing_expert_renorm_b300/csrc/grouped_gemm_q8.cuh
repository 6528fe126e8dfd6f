// Grouped GEMM with weight-only INT8 B on the 5th-generation tensor cores.
//
// "MoE 混合专家架构" 5.3 量化支持: expert weights may be stored as INT8. Each weight row n
// holds codes q[n][k] (int8) and one fp32 scale s[n]; D[r][n] = s[n] * sum_k A[r][k] *
// q[n][k]. The codes are widened exactly to bf16 in shared memory (|q| <= 127 needs 8
// significant bits), the tensor cores accumulate A * q in fp32 in TMEM, and the epilogue
// multiplies column n by s[n] (GemmParams::w_scale) before the bias and the activation,
// so the epilogues of grouped_gemm_kernel apply unchanged. HBM carries one byte per
// weight instead of two.
//
// Same work units, scheduling, TMEM accumulators and epilogue as grouped_gemm_kernel
// (grouped_gemm.cuh); the operand pipeline differs:
//   warp 0      unit scheduler + TMA of the int8 B tile (two 128-row boxes of 64 bytes)
//               into a GM_Q8_NQ-deep ring;
//   warps 7-10  converters: together widen each B stage (a quarter each) into the 128-byte
//               swizzled K-major bf16 layout of a GM_Q8_NC-deep ring the MMA reads, then
//               makes the writes visible to the tensor core (fence.proxy.async);
//   warp 6      TMA of the bf16 A tile into its own GM_Q8_NA-deep ring;
//   warp 1      MMA issuer;  warps 2-5  epilogue.
#pragma once
#include "grouped_gemm.cuh"

namespace moe {

constexpr int GM_Q8_NA = 3, GM_Q8_NQ = 6, GM_Q8_NC = 2;
constexpr int GM_Q8_Q_BYTES = GM_BN * GM_BK;          // 16 KB of int8 codes per stage
constexpr int GM_Q8_RING_BYTES = GM_Q8_NA * GM_A_BYTES + GM_Q8_NC * GM_B_BYTES + GM_Q8_NQ * GM_Q8_Q_BYTES;
constexpr int GM_Q8_THREADS = 352;

__host__ __device__ constexpr int gm_q8_smem_bytes(int G) {
    return 1024 + GM_Q8_RING_BYTES + GM_HDR_BYTES + 2 * (G + 1) * 4;
}

// Four int8 codes (one 32-bit word) -> two bf16x2 words, exactly and without conversion
// instructions (those issue at a fraction of the ALU rate). Each code, offset to
// u = q + 128 by flipping its top bit, becomes the low mantissa byte of 2^23 (fp32 bit
// pattern 0x4B0000uu); subtracting 2^23 + 128 leaves q exactly. With |q| <= 128, q has at
// most 8 significant bits, so its bf16 pattern is the upper half of its fp32 pattern.
__device__ __forceinline__ void widen4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t x = w ^ 0x80808080u;
    constexpr float kBias = 8388736.0f;   // 2^23 + 128
    const float f0 = __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7650)) - kBias;
    const float f1 = __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7651)) - kBias;
    const float f2 = __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7652)) - kBias;
    const float f3 = __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7653)) - kBias;
    lo = __byte_perm(__float_as_uint(f0), __float_as_uint(f1), 0x7632);
    hi = __byte_perm(__float_as_uint(f2), __float_as_uint(f3), 0x7632);
}


template <int EPI>
__global__ void __launch_bounds__(GM_Q8_THREADS, 1)
    grouped_gemm_q8_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmQ, const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* a_tiles = smem;                                              // NA x 16 KB bf16
    uint8_t* c_tiles = smem + GM_Q8_NA * GM_A_BYTES;                      // NC x 32 KB bf16
    uint8_t* q_tiles = c_tiles + GM_Q8_NC * GM_B_BYTES;                   // NQ x 16 KB int8
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + GM_Q8_RING_BYTES);
    const int AFULL = 0, AEMPTY = GM_Q8_NA, QFULL = 2 * GM_Q8_NA, QEMPTY = QFULL + GM_Q8_NQ,
              CFULL = QEMPTY + GM_Q8_NQ, CEMPTY = CFULL + GM_Q8_NC, TFULL = CEMPTY + GM_Q8_NC,
              TEMPTY = TFULL + 2, DRAIN = TEMPTY + 2, UFULL = 32, UEMPTY = 32 + GM_TQ;
    static_assert(2 * (GM_Q8_NA + GM_Q8_NQ + GM_Q8_NC) + 5 <= 32, "barrier slots overlap");
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 48);
    volatile int* s_abort = reinterpret_cast<volatile int*>(bars + 49);
    volatile long long* s_unit = reinterpret_cast<volatile long long*>(bars + 52);   // [GM_TQ]
    static_assert((52 + GM_TQ) * 8 <= GM_HDR_BYTES, "header overflow");
    int* s_ro = reinterpret_cast<int*>(bars + GM_HDR_BYTES / 8);
    int* s_mt = s_ro + (p.G + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto bar = [&](int i) { return smem_addr(bars + i); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < GM_Q8_NA; ++s) {
            mbar_init(bar(AFULL + s), 1);
            mbar_init(bar(AEMPTY + s), 1);
        }
        for (int s = 0; s < GM_Q8_NQ; ++s) {
            mbar_init(bar(QFULL + s), 1);
            mbar_init(bar(QEMPTY + s), 4);   // the four converter warps
        }
        for (int s = 0; s < GM_Q8_NC; ++s) {
            mbar_init(bar(CFULL + s), 4);    // the four converter warps
            mbar_init(bar(CEMPTY + s), 1);   // MMA commit
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar(TFULL + a), 1);
            mbar_init(bar(TEMPTY + a), 4);
        }
        mbar_init(bar(DRAIN), 1);
        for (int i = 0; i < GM_TQ; ++i) {
            mbar_init(bar(UFULL + i), 1);
            mbar_init(bar(UEMPTY + i), 10);  // MMA, A producer, 4 epilogue, 4 converter warps
        }
        *s_abort = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmQ);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(s_tmem), GM_TMEM_COLS);
        tmem_relinquish();
    }
    pdl_entry();
    for (int i = threadIdx.x; i <= p.G; i += blockDim.x) {
        s_ro[i] = p.row_offsets[i];
        s_mt[i] = p.mtile_offsets[i];
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;
    const long long total = (long long)s_mt[p.G] * p.n_tiles * p.k_splits;
    const int kblocks = p.K / GM_BK;

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

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- unit scheduler + TMA of the int8 weight codes ----------------
            int stage = 0;
            uint32_t ph = 0;
            int last_par[GM_Q8_NQ];
#pragma unroll
            for (int s = 0; s < GM_Q8_NQ; ++s) last_par[s] = -1;
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
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (*s_abort || !mbar_wait(bar(QEMPTY + stage), ph ^ 1)) {
                        *s_abort = 1;
                        ok = false;
                        break;
                    }
                    const uint32_t sq = smem_addr(q_tiles + stage * GM_Q8_Q_BYTES);
                    mbar_arrive_expect_tx(bar(QFULL + stage), GM_Q8_Q_BYTES);
                    tma_load_2d(sq, &tmQ, bar(QFULL + stage), kb * GM_BK, b0);
                    tma_load_2d(sq + GM_Q8_Q_BYTES / 2, &tmQ, bar(QFULL + stage), kb * GM_BK, b1);
                    last_par[stage] = (int)ph;
                    if (++stage == GM_Q8_NQ) {
                        stage = 0;
                        ph ^= 1;
                    }
                }
                t = next;
            }
            for (int s = 0; s < GM_Q8_NQ; ++s)
                if (last_par[s] >= 0) mbar_wait(bar(QFULL + s), (uint32_t)last_par[s]);
        }
    } else if (warp == 6) {
        if (lane == 0) {
            // ---------------- TMA of the activation rows (A) ----------------------------
            int stage = 0;
            uint32_t ph = 0;
            int last_par[GM_Q8_NA];
#pragma unroll
            for (int s = 0; s < GM_Q8_NA; ++s) last_par[s] = -1;
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
                const int a_row = s_ro[g] + mb * GM_BM;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (*s_abort || !mbar_wait(bar(AEMPTY + stage), ph ^ 1)) {
                        *s_abort = 1;
                        ok = false;
                        break;
                    }
                    const uint32_t sa = smem_addr(a_tiles + stage * GM_A_BYTES);
                    mbar_arrive_expect_tx(bar(AFULL + stage), GM_A_BYTES);
                    tma_load_2d(sa, &tmA, bar(AFULL + stage), kb * GM_BK, a_row);
                    last_par[stage] = (int)ph;
                    if (++stage == GM_Q8_NA) {
                        stage = 0;
                        ph ^= 1;
                    }
                }
            }
            for (int s = 0; s < GM_Q8_NA; ++s)
                if (last_par[s] >= 0) mbar_wait(bar(AFULL + s), (uint32_t)last_par[s]);
        }
    } else if (warp >= 7) {
        // ---------------- converters: int8 codes -> swizzled bf16 B tiles ------------------
        const int cw = warp - 7;
        int qs = 0, cs = 0;
        uint32_t qph = 0, cph = 0;
        int uq = 0;
        uint32_t uqph = 0;
        while (true) {
            long long t = -1;
            int got = 1;
            if (lane == 0) got = take_unit(uq, uqph, t) ? 1 : 0;
            got = __shfl_sync(0xffffffffu, got, 0);
            t = __shfl_sync(0xffffffffu, t, 0);
            if (!got || t < 0) break;
            int g, mb, nb, ks;
            gm_decode(t, p.G, p.n_tiles, p.k_splits, s_mt, g, mb, nb, ks);
            const int kb0 = ks * p.kb_per_split;
            const int kb1 = min(kblocks, kb0 + p.kb_per_split);
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                // every lane waits: each one reads TMA-written codes and overwrites a stage
                // the tensor core has finished reading
                const bool w_ok = !*s_abort && mbar_wait(bar(QFULL + qs), qph) &&
                                  mbar_wait(bar(CEMPTY + cs), cph ^ 1);
                if (!__all_sync(0xffffffffu, w_ok)) {
                    if (lane == 0) *s_abort = 1;
                    ok = false;
                    break;
                }
                const uint8_t* src = q_tiles + qs * GM_Q8_Q_BYTES;
                uint8_t* dst = c_tiles + cs * GM_B_BYTES;
                // 1024 chunks of 16 codes per stage; chunk u is row u/4, codes 16(u%4)..+15.
                // Eight consecutive lanes read 128 contiguous bytes and write eight distinct
                // 16-byte bank groups (rows 2i and 2i+1 swizzle to disjoint chunk sets).
#pragma unroll
                for (int it = 0; it < GM_Q8_Q_BYTES / 16 / 128; ++it) {
                    const int u = it * 128 + cw * 32 + lane;
                    const int r = u >> 2, v = u & 3;
                    const uint4 w = *reinterpret_cast<const uint4*>(src + u * 16);
                    uint4 c0, c1;
                    widen4(w.x, c0.x, c0.y);
                    widen4(w.y, c0.z, c0.w);
                    widen4(w.z, c1.x, c1.y);
                    widen4(w.w, c1.z, c1.w);
                    *reinterpret_cast<uint4*>(dst + r * 128 + (((2 * v) ^ (r & 7)) << 4)) = c0;
                    *reinterpret_cast<uint4*>(dst + r * 128 + (((2 * v + 1) ^ (r & 7)) << 4)) = c1;
                }
                fence_proxy_async_smem();   // generic-proxy writes -> tensor core reads
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar(QEMPTY + qs));
                    mbar_arrive(bar(CFULL + cs));
                }
                if (++qs == GM_Q8_NQ) {
                    qs = 0;
                    qph ^= 1;
                }
                if (++cs == GM_Q8_NC) {
                    cs = 0;
                    cph ^= 1;
                }
            }
            if (!ok) break;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            constexpr uint32_t idesc = idesc_bf16_f32(GM_BM, GM_BN);
            int as = 0, cs = 0, acc = 0;
            uint32_t aph_s = 0, cph = 0, aph = 0;
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
                const uint32_t dt = tmem_base + (uint32_t)(acc * GM_BN);
                const int kb0 = (int)(t % p.k_splits) * p.kb_per_split;
                const int kb1 = min(kblocks, kb0 + p.kb_per_split);
                bool ok = true;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(bar(CFULL + cs), cph) || !mbar_wait(bar(AFULL + as), aph_s)) {
                        *s_abort = 1;
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_addr(a_tiles + as * GM_A_BYTES);
                    const uint32_t sb = smem_addr(c_tiles + cs * GM_B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < GM_BK / 16; ++kk)
                        umma_bf16(dt, sw128_kmajor_desc(sa + kk * 32), sw128_kmajor_desc(sb + kk * 32),
                                  idesc, (kb != kb0 || kk != 0) ? 1u : 0u);
                    umma_commit(bar(AEMPTY + as));
                    umma_commit(bar(CEMPTY + cs));
                    if (++as == GM_Q8_NA) {
                        as = 0;
                        aph_s ^= 1;
                    }
                    if (++cs == GM_Q8_NC) {
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
        int acc = 0;
        uint32_t aph = 0;
        int uq = 0;
        uint32_t uqph = 0;
        while (true) {
            long long t = -1;
            int got = 1;
            if (lane == 0) got = take_unit(uq, uqph, t) ? 1 : 0;
            got = __shfl_sync(0xffffffffu, got, 0);
            t = __shfl_sync(0xffffffffu, t, 0);
            if (!got || t < 0) break;
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
            const int r_in = qd * 32 + lane;
            const int rows_g = s_ro[g + 1] - s_ro[g];
            const int r_tile = mb * GM_BM + r_in;
            const bool row_ok = r_tile < rows_g;
            const long long grow = (long long)s_ro[g] + r_tile;
            const uint32_t tb = tmem_base + ((uint32_t)(qd * 32) << 16) + (uint32_t)(acc * GM_BN);
            if (p.partial) gm_epilogue_partial<EPI>(p, tb, nb, ks, row_ok, grow);
            else gm_epilogue_tile<EPI>(p, tb, g, nb, row_ok, grow);
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

// ---- per-row absmax INT8 quantisation of bf16 weights --------------------------------
// One warp per row: s = max|w| / 127 (fp32), q = rne(w / s) clamped to [-127, 127] (fp32
// division and rounding: the same decision the reference quantiser makes); s = 0 and
// q = 0 for an all-zero row. cols is a multiple of 8.
__global__ void __launch_bounds__(256) quantize_rows_i8_kernel(const __nv_bfloat16* __restrict__ w,
                                                               long long rows, int cols,
                                                               int8_t* __restrict__ q,
                                                               float* __restrict__ scale) {
    pdl_entry();
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows;
         r += warps) {
        const __nv_bfloat16* wr = w + r * cols;
        float m = 0.0f;
        for (int c = lane; c < cols; c += 32) m = fmaxf(m, fabsf(__bfloat162float(wr[c])));
#pragma unroll
        for (int off = 16; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        const float s = __fdiv_rn(m, 127.0f);
        if (lane == 0) scale[r] = s;
        int8_t* qr = q + r * cols;
        for (int c = lane; c < cols; c += 32) {
            int v = 0;
            if (s > 0.0f) {
                v = __float2int_rn(__fdiv_rn(__bfloat162float(wr[c]), s));
                v = max(-127, min(127, v));
            }
            qr[c] = (int8_t)v;
        }
    }
}

// ---- per-row absmax INT4 quantisation of bf16 weights --------------------------------
// One warp per row: s = max|w| / 7 (fp32), q = rne(w / s) clamped to [-7, 7]; s = 0 and
// q = 0 for an all-zero row. Two codes per byte (column 2j in the low nibble of byte j,
// 4-bit two's complement); cols is even, a row takes cols / 2 bytes.
__global__ void __launch_bounds__(256) quantize_rows_i4_kernel(const __nv_bfloat16* __restrict__ w,
                                                               long long rows, int cols,
                                                               uint8_t* __restrict__ q,
                                                               float* __restrict__ scale) {
    pdl_entry();
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows;
         r += warps) {
        const __nv_bfloat16* wr = w + r * cols;
        float m = 0.0f;
        for (int c = lane; c < cols; c += 32) m = fmaxf(m, fabsf(__bfloat162float(wr[c])));
#pragma unroll
        for (int off = 16; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        const float s = __fdiv_rn(m, 7.0f);
        if (lane == 0) scale[r] = s;
        uint8_t* qr = q + r * (cols / 2);
        for (int j = lane; j < cols / 2; j += 32) {
            int v[2] = {0, 0};
            if (s > 0.0f) {
#pragma unroll
                for (int u = 0; u < 2; ++u)
                    v[u] = max(-7, min(7, __float2int_rn(__fdiv_rn(__bfloat162float(wr[2 * j + u]), s))));
            }
            qr[j] = (uint8_t)((v[0] & 15) | ((v[1] & 15) << 4));
        }
    }
}

}  // namespace moe
