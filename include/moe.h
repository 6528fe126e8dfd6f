/*
 * moe.h — C ABI of the single-GPU Mixture-of-Experts layer forward for B300 (sm_103a).
 *
 * One MoE layer, forward only, on one GPU:
 *   route    : gate GEMM x[T,d] * W_gate[d,E] -> logits, top-k per token, and the
 *              kept weights renormalised to sum to 1;
 *   dispatch : per-expert histogram, prefix sum, optional capacity limit, and a
 *              permutation of the kept (token, slot) assignments into
 *              expert-contiguous rows (the multi-GPU all-to-all becomes a copy
 *              inside HBM);
 *   expert   : every expert's FFN on its contiguous block of rows (grouped GEMM);
 *   combine  : weighted sum of each token's expert outputs, back in token order.
 *
 * Sources (page title, section):
 *   "adv12 — Mixture of Experts (MoE) + EPLB 专家负载均衡": 3.1 Top-k routing diagram,
 *       4.1 MoELayer step table, 4.2 expert_imbalance, 4.3 eplb_rebalance, Q1, Q2.
 *   "MoE 混合专家架构：LLM稀疏化计算的关键演进": 1.2 Switch Transformer, 2.1 门控机制,
 *       4.2 数值稳定性, 5.2 专家融合与并行.
 *   "MoE 并行": 流程说明 (router -> dispatch -> experts -> gather -> weighted combine),
 *       Capacity Factor.
 *   "MOE 学习笔记": 输出聚合示例.
 *
 * Conventions for every entry point:
 *   - All tensors are dense, row-major, caller-owned DEVICE memory unless stated;
 *     the library never allocates or frees device memory. Scratch space comes
 *     from a caller-owned workspace of moe_workspace_size() bytes.
 *   - Every device pointer must be 16-byte aligned (MOE_ERR_MISALIGNED otherwise).
 *   - Arguments are validated on the host before anything is launched; on an
 *     error nothing is enqueued. Calls are asynchronous on `stream` (0 = legacy
 *     default stream) and never synchronise the host, except
 *     moe_last_device_status().
 *   - There is no CPU fallback: without a usable CUDA device the calls return
 *     MOE_ERR_CUDA.
 *   - Kernels never trap. A device-side bounded wait that runs out, or an
 *     out-of-range expert id in caller data, is recorded in a device error word
 *     and reported by moe_last_device_status().
 *   - Non-finite inputs are not checked; selection then follows IEEE float
 *     comparison.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* null pointer, bad size, k > E, ... */
    MOE_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. GELU in fp32) */
    MOE_ERR_MISALIGNED = 3,    /* a pointer is not 16-byte aligned */
    MOE_ERR_WORKSPACE = 4,     /* workspace missing or smaller than moe_workspace_size() */
    MOE_ERR_CUDA = 5,          /* a CUDA runtime/driver call or a launch failed */
    MOE_ERR_TIMEOUT = 6,       /* a device-side bounded wait expired (kernel gave up) */
    MOE_ERR_DEVICE_INDEX = 7   /* a kernel saw an expert id outside [0,E) and skipped it */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_I8 = 2, MOE_I4 = 3 } moe_dtype;

/* Expert FFN forms.
 *  LINEAR : y = W1 x + b1; W1 [E][d][d] fp32 (the tutorial's nn.Linear(d, d) experts).
 *  GELU   : y = W2 gelu(W1 x + b1) + b2, exact-erf GELU; W1 [E][F][d], W2 [E][d][F].
 *  SWIGLU : y = W2 (silu(W1[0:F] x) * W1[F:2F] x) + b2; W1 [E][2F][d], W2 [E][d][F].
 * GELU and SWIGLU run in bf16 with fp32 accumulation; the hidden activation h is
 * rounded to bf16 before the second GEMM. LINEAR runs in fp32. */
typedef enum { MOE_EXPERT_LINEAR = 0, MOE_EXPERT_GELU = 1, MOE_EXPERT_SWIGLU = 2 } moe_expert_kind;

/* What happens to an assignment (t, j) beyond its expert's capacity.
 *  DROP    : it contributes 0 ["MoE 并行" Capacity Factor: overflow takes the residual path;
 *            adv12 Q2 option 1].
 *  SHARED  : its weight w_tj moves to the shared expert, whose weight for token t becomes
 *            1 + sum of the token's dropped w ["MoE 并行" Q4, Q5; adv12 Q2 option 2].
 *            Needs has_shared.
 *  REROUTE : one re-routing round ["MoE 并行" 推理时的负载均衡, dynamic re-routing to the next
 *            expert; "MoE 混合专家架构" 4.2 capacity check]: token t's dropped slots, in slot
 *            order, propose to its experts ranked k, k+1, ... (same order and, with
 *            group-limited routing, the same groups as the top k) keeping their weights;
 *            each expert accepts proposals in token order while its round-0 rows plus the
 *            accepted ones stay below the capacity; the rest stay dropped. */
typedef enum { MOE_OVERFLOW_DROP = 0, MOE_OVERFLOW_SHARED = 1, MOE_OVERFLOW_REROUTE = 2 } moe_overflow;

typedef struct {
    int32_t T;                 /* tokens (rows of x); 0 is a valid no-op */
    int32_t d;                 /* model width; multiple of 8 (of 64 for GELU/SWIGLU) */
    int32_t E;                 /* routed experts, 1..1024 */
    int32_t top_k;             /* experts per token, 1..min(E, 32) */
    int32_t F;                 /* expert hidden width (GELU/SWIGLU), multiple of 64 */
    float capacity_factor;     /* <= 0: no limit; else cap = ceil(cf*T*k/E) clipped to [1,T] */
    int32_t act_dtype;         /* moe_dtype of x, expert weights and out:
                                  MOE_F32 for LINEAR, MOE_BF16 for GELU/SWIGLU */
    int32_t kind;              /* moe_expert_kind */
    int32_t has_shared;        /* 1: one always-on shared expert of the same kind, weight 1 */
    int32_t add_residual;      /* 1: out = x + combine (tokens whose every slot overflowed
                                  the capacity leave the layer as x, bit for bit) */
    int32_t n_group;           /* 0: plain top-k. Else group-limited routing ["MoE 并行" 通信瓶颈,
                                  Hierarchical Routing; adv12 5, device-limited routing]: the
                                  E experts form n_group groups of E/n_group consecutive ids
                                  (n_group divides E, at most 32) ... */
    int32_t topk_group;        /* ... only the topk_group groups with the highest best-expert
                                  logit (ties to the lower group id) supply the top k;
                                  1 <= topk_group <= n_group, k <= topk_group * E / n_group */
    int32_t w_dtype;           /* 0 (or act_dtype): weights in act_dtype. MOE_I8 (GELU/SWIGLU
                                  only): weight-only INT8 experts ["MoE 混合专家架构" 5.3 量化支持]:
                                  w1/w2 hold int8 codes q and s1/s2 one fp32 scale per weight
                                  row; the experts compute with s[n] * q[n][k] (see
                                  moe_quantize_i8). Routed and shared experts alike.
                                  MOE_I4: the same with 4-bit codes in [-7, 7], two per byte
                                  (w1 [E][N1][d/2], w2 [E][d][F/2] bytes; see moe_quantize_i4). */
    int32_t overflow;          /* moe_overflow; 0 = MOE_OVERFLOW_DROP */
    int32_t y_fp32;            /* Expert-output rows inside moe_forward (routed experts with
                                  bf16 weights, top_k >= 4, more than 4 rows per expert on
                                  average and an unsplit down projection; other layers
                                  always keep fp32 rows): 0 = fp16 with one
                                  power-of-two scale per 32 columns of a row (half the bytes
                                  of fp32; every element keeps fp16's 11-bit significand and
                                  no finite value overflows), 1 = fp32, as moe_expert_ffn
                                  always writes them. */
} moe_config;

/* One set of stacked expert weights (nn.Linear [out, in] layout, K contiguous).
 * Routed: w1 [E][N1][d], b1 [E][N1], w2 [E][d][F], b2 [E][d] with N1 = d, F or 2F.
 * Shared: the same with E = 1. Biases are fp32 and nullable; w2/b2 unused for LINEAR. */
typedef struct {
    const void* w1;
    const float* b1;
    const void* w2;
    const float* b2;
    const float* s1;   /* MOE_I8 / MOE_I4 weights: scales [E][N1] of the w1 rows, else ignored */
    const float* s2;   /* MOE_I8 / MOE_I4 weights: scales [E][d] of the w2 rows, else ignored */
} moe_expert_weights;

/* Bytes of scratch needed by any entry point below for this configuration
 * (one workspace serves all of them; regions do not overlap between stages).
 * Returns 0 for an invalid configuration. */
size_t moe_workspace_size(const moe_config* cfg);

/* Rows of the permuted buffers: P_max = T * top_k (the kept count P <= P_max is
 * only known on the device, in offsets[E]). Returns -1 for an invalid config. */
int64_t moe_max_rows(const moe_config* cfg);

/* Expert capacity ["MoE 并行", Capacity Factor; adv12 Q2]:
 * ceil(cf * T * k / E) computed in double, clipped to [1, T]; T when cf <= 0.
 * Host-only. Returns -1 for an invalid configuration. */
int32_t moe_capacity(const moe_config* cfg);

/* Routing ["MoE 混合专家架构" 2.1 门控机制; adv12 4.1 steps 1-3, Q1; 1.2 Switch for k = 1].
 *   x         [T, d]  act_dtype
 *   W_gate    [d, E]  fp32 (E contiguous)
 *   gate_bias [E]     fp32, nullable (added to the logits)
 *   logits    [T, E]  fp32 output, nullable
 *   topk_idx  [T, k]  int32 output: experts ordered by logit descending, ties to
 *                     the lower expert id
 *   topk_w    [T, k]  fp32 output: exp(L_j - L_0) / sum_j' exp(L_j' - L_0) over the
 *                     k kept logits = softmax then divide by the kept sum
 *   ws        workspace (required)
 * Logits are fp32 sums of exact fp32 products x_i * W_gate[i, e] (bf16 activations with
 * many tokens run on the tensor cores against W_gate split exactly into three bf16
 * terms); partial sums are added in a fixed order, so results are reproducible run to
 * run, and selection is bit-reproducible given the logits.
 * With MOE_OVERFLOW_REROUTE it also stores each token's experts ranked k .. 2k-1 in ws,
 * where moe_dispatch reads them. */
moe_status moe_route(const moe_config* cfg, const void* x, const float* W_gate,
                     const float* gate_bias, float* logits, int32_t* topk_idx, float* topk_w,
                     void* ws, cudaStream_t stream);

/* Dispatch ["MoE 并行" 流程说明 Token Dispatch and Capacity Factor; adv12 3.2 bincount, Q2].
 *   topk_idx   [T, k] int32 input (values must lie in [0, E))
 *   x          [T, d] act_dtype input; only read when x_perm is non-NULL
 *   load       [E]    int32 output: assignments per expert before capacity (sum = T*k)
 *   counts     [E]    int32 output: kept = min(load, cap)
 *   offsets    [E+1]  int32 output: exclusive prefix sum of counts; offsets[E] = P
 *   perm_token [T*k]  int32 output: rows [offsets[e], offsets[e+1]) list expert e's kept
 *                     tokens in ascending token order; entries >= P are unspecified
 *   perm_slot  [T*k]  int32 output: the slot j (0..k-1) of each listed assignment
 *   slot_dest  [T, k] int32 output: row of (t, j) in the permuted order, -1 if dropped
 *                     (assignments beyond the capacity are dropped in token order)
 *   x_perm     [T*k, d] act_dtype output, nullable: x_perm[p] = x[perm_token[p]]
 *   ws         workspace
 * Everything is deterministic (no order-dependent atomics).
 * MOE_OVERFLOW_REROUTE: ws must hold what moe_route wrote for the same tokens (the
 * next-ranked experts). counts = kept rows after re-routing; expert e's rows are its
 * round-0 rows (token order) followed by the re-routed rows it accepted (token order);
 * slot_dest points re-routed slots at their new expert's rows; load stays the top-k
 * bincount before capacity. */
moe_status moe_dispatch(const moe_config* cfg, const int32_t* topk_idx, const void* x,
                        int32_t* load, int32_t* counts, int32_t* offsets, int32_t* perm_token,
                        int32_t* perm_slot, int32_t* slot_dest, void* x_perm, void* ws,
                        cudaStream_t stream);

/* Expert FFNs on expert-contiguous rows ["MoE 混合专家架构" 5.2 (stacked weights, silu
 * on the W1 slice); adv12 4.1 step 4 (expert_e(x[mask]), weighted)].
 *   x_perm   [T*k, d] act_dtype, rows [0, P) valid (from moe_dispatch)
 *   offsets  [E+1] int32 (from moe_dispatch)
 *   routed   routed expert weights (required); shared: nullable, used iff cfg->has_shared
 *   x        [T, d] act_dtype: input of the shared expert (nullable without shared)
 *   topk_w, perm_token, perm_slot: from moe_route / moe_dispatch; row p is scaled by
 *            topk_w[perm_token[p]*k + perm_slot[p]]
 *   y        [T*k + T*has_shared, d] fp32 output: row p < P holds w * expert(x_perm[p]);
 *            row T*k + t holds the shared expert's output for token t (weight 1)
 *   ws       workspace
 * bf16 kinds run on the tensor cores (tcgen05, TMEM accumulators, TMA-fed). */
moe_status moe_expert_ffn(const moe_config* cfg, const void* x_perm, const int32_t* offsets,
                          const moe_expert_weights* routed, const moe_expert_weights* shared,
                          const void* x, const float* topk_w, const int32_t* perm_token,
                          const int32_t* perm_slot, float* y, void* ws, cudaStream_t stream);

/* Combine ["MOE 学习笔记" 输出聚合示例; "MoE 并行" Result Gather + 加权组合].
 *   out[t] = (add_residual ? x[t] : 0) + sum_{j = 0..k-1, slot kept} y[slot_dest[t,j]]
 *            + (has_shared ? a_t * y[T*k + t] : 0)
 * summed in fp32 in that order and rounded once to act_dtype; a_t = 1, or with
 * MOE_OVERFLOW_SHARED a_t = 1 + sum of topk_w[t, j] over the dropped slots (fp32, slot order).
 *   x [T, d] (read iff add_residual), y as written by moe_expert_ffn, topk_w [T, k] (read
 *   iff MOE_OVERFLOW_SHARED, else nullable), slot_dest [T, k], out [T, d] act_dtype output. */
moe_status moe_combine(const moe_config* cfg, const void* x, const float* y,
                       const float* topk_w, const int32_t* slot_dest, void* out,
                       cudaStream_t stream);

/* The whole layer: route -> dispatch -> expert FFNs -> combine, stream-ordered, no
 * host synchronisation. out [T, d] act_dtype. Optional outputs (nullable):
 * topk_idx [T, k], topk_w [T, k], load [E]. ws must hold moe_workspace_size(cfg)
 * bytes (checked against ws_bytes). Results equal the staged entry points' up to the
 * expert-output row format (moe_config.y_fp32) and floating-point summation order; with
 * y_fp32 = 1 (or fp32 rows anyway) the operations are the same. */
moe_status moe_forward(const moe_config* cfg, const void* x, const float* W_gate,
                       const float* gate_bias, const moe_expert_weights* routed,
                       const moe_expert_weights* shared, void* out, int32_t* topk_idx,
                       float* topk_w, int32_t* load, void* ws, size_t ws_bytes,
                       cudaStream_t stream);

/* Grouped GEMM building block of the expert stage, exposed for testing:
 * for every group g and row r in [row_offsets[g], row_offsets[g+1]):
 *   D[r, n] = sum_k A[r, k] * B[g, n, k]     (bf16 inputs, fp32 accumulate and output)
 *   A [a_rows, K] bf16, B [G][N][K] bf16, D [a_rows, N] fp32, row_offsets [G+1] int32
 *   (device, non-decreasing, row_offsets[G] <= a_rows). K and N multiples of 64.
 *   ws: at least moe_grouped_gemm_ws_size(G) bytes. */
size_t moe_grouped_gemm_ws_size(int32_t G);
moe_status moe_grouped_gemm(const void* A, int64_t a_rows, const void* B, int32_t G,
                            int32_t N, int32_t K, const int32_t* row_offsets, float* D,
                            void* ws, cudaStream_t stream);

/* moe_dispatch without a workspace: the pages have no counterpart to this entry
 * point; it exists for callers that cannot allocate device memory when they call
 * the layer, for example a plugin running inside a host framework that owns all
 * device memory and exposes no allocator to it, or a latency-critical loop that
 * must not take the implicit device synchronisation of cudaMalloc.
 * Arguments and outputs are those of moe_dispatch minus `ws`; the caller still
 * passes every input and output buffer. The dispatch scratch (2 * ceil(T/256) * E
 * int32) lives in a 1 MiB static device array inside the library, held on every
 * GPU that loads the library until the process exits. Problems with
 * ceil(T/256) * E > 131072 are rejected with MOE_ERR_WORKSPACE (with E = 1024 that
 * allows T <= 32768 tokens; with E = 256, T <= 131072). It calls no cudaMalloc, cudaFree or
 * other allocating routine. Its first call on a device looks up the array's
 * device address (cudaGetSymbolAddress, with that device current), so make that
 * first call before any stream capture. That address is kept for the rest of the
 * process: resetting the device (cudaDeviceReset) after the first call is not
 * supported, since the array then lives at a new address. All calls share the one array: calls that
 * overlap on the GPU (different streams, or different host threads) race on it and
 * must be ordered by the caller. MOE_OVERFLOW_REROUTE needs the workspace moe_route
 * wrote and is rejected here with MOE_ERR_UNSUPPORTED. */
moe_status moe_dispatch_noalloc(const moe_config* cfg, const int32_t* topk_idx, const void* x,
                                int32_t* load, int32_t* counts, int32_t* offsets,
                                int32_t* perm_token, int32_t* perm_slot, int32_t* slot_dest,
                                void* x_perm, cudaStream_t stream);

/* Weight-only INT8 codes of bf16 weights [the reading of "MoE 混合专家架构" 5.3 used by
 * MOE_I8 experts]: for every row r of w [rows, cols] (bf16, cols a multiple of 8):
 *   scale[r] = max_c |w[r][c]| / 127   (fp32)
 *   q[r][c]  = round-half-even(w[r][c] / scale[r]) clamped to [-127, 127]   (fp32 division)
 * and scale 0 / codes 0 for an all-zero row. q [rows, cols] int8 and scale [rows] fp32 are
 * caller-owned device buffers. Stacked expert weights [E][N][K] are E*N rows of K. */
moe_status moe_quantize_i8(const void* w, int64_t rows, int32_t cols, int8_t* q, float* scale,
                           cudaStream_t stream);

/* Weight-only INT4 codes of bf16 weights [the same reading with 4-bit codes, used by MOE_I4
 * experts]: for every row r of w [rows, cols] (bf16, cols a multiple of 32):
 *   scale[r] = max_c |w[r][c]| / 7   (fp32)
 *   code(r, c) = round-half-even(w[r][c] / scale[r]) clamped to [-7, 7]   (fp32 division)
 * and scale 0 / codes 0 for an all-zero row. q [rows, cols / 2] bytes: byte j of row r holds
 * code(r, 2j) in its low nibble and code(r, 2j+1) in its high nibble, each as a 4-bit two's
 * complement. q and scale [rows] fp32 are caller-owned device buffers. */
moe_status moe_quantize_i4(const void* w, int64_t rows, int32_t cols, uint8_t* q, float* scale,
                           cudaStream_t stream);

/* Host-only load report [adv12 3.3 EPLB, 4.2 expert_imbalance, 4.3 eplb_rebalance]:
 * imbalance = max(load) / (min(load) + 1e-6); LPT placement of the E experts on D
 * devices (heaviest first, equal loads by ascending id, each to the currently
 * least-loaded device, lowest index on ties). load_host [E], assign [E] and
 * dev_load [D] are HOST arrays. */
moe_status moe_load_report(const int32_t* load_host, int32_t E, int32_t D, int32_t* assign,
                           int64_t* dev_load, double* imbalance);

/* Synchronises `stream`, then reads and clears the device error word:
 * MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_INDEX, MOE_ERR_CUDA for an asynchronous CUDA
 * error, else MOE_OK. */
moe_status moe_last_device_status(cudaStream_t stream);

const char* moe_status_string(moe_status s);

/* ---- instrumentation ------------------------------------------------------
 * moe_profile_begin() starts recording a CUDA event pair around every kernel
 * this library launches (on the launching stream). moe_profile_end() waits for
 * the recorded events, stops recording and fills up to max_stats entries, one
 * per kernel name, with launch count and summed device time; it returns the
 * number of distinct kernels (or -1 on error). Recording adds two event
 * records per launch and allocates nothing on the device. */
typedef struct {
    const char* name;          /* static string owned by the library */
    int64_t launches;
    double total_ms;
} moe_kernel_stat;

moe_status moe_profile_begin(void);
int32_t moe_profile_end(moe_kernel_stat* stats, int32_t max_stats);

/* Kernels launched by this library since the process started. */
uint64_t moe_kernel_launch_count(void);

/* Self-test of the device-side failure path: launches one thread that waits on an
 * mbarrier phase nothing will complete, gives up after budget_cycles SM clocks
 * (0 .. 2^32) and records a timeout, so that the next moe_last_device_status()
 * returns MOE_ERR_TIMEOUT. Nothing faults, traps or hangs. */
moe_status moe_selftest_wait_timeout(int64_t budget_cycles, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
