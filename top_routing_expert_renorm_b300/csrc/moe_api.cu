// Host side of the MoE layer library: argument validation, workspace carving,
// TMA descriptor encoding, kernel launches and the exported C ABI (include/moe.h).
// Everything is stream-ordered; nothing here synchronises the host except
// moe_last_device_status() and moe_profile_end().
#include "moe.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <numeric>
#include <utility>
#include <vector>

#include "common.cuh"
#include "router.cuh"
#include "dispatch.cuh"
#include "grouped_gemm.cuh"
#include "grouped_gemm_q8.cuh"
#include "grouped_gemm_q8t.cuh"
#include "combine.cuh"

using namespace moe;

namespace {

// ---------------------------------------------------------------------------------
// launch accounting and optional per-kernel event timing
// ---------------------------------------------------------------------------------
std::atomic<uint64_t> g_launches{0};

struct ProfRec {
    const char* name;
    cudaEvent_t a, b;
};
struct Prof {
    std::mutex mu;
    bool on = false;
    std::vector<ProfRec> recs;
    std::vector<cudaEvent_t> pool;
    size_t used = 0;
} g_prof;

cudaEvent_t prof_event_locked() {
    if (g_prof.used == g_prof.pool.size()) {
        cudaEvent_t e = nullptr;
        if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
        g_prof.pool.push_back(e);
    }
    return g_prof.pool[g_prof.used++];
}

void prof_pre(const char* name, cudaStream_t s, cudaEvent_t* after) {
    *after = nullptr;
    if (!g_prof.on) return;
    std::lock_guard<std::mutex> lk(g_prof.mu);
    if (!g_prof.on) return;
    cudaEvent_t a = prof_event_locked(), b = prof_event_locked();
    if (!a || !b) return;
    cudaEventRecord(a, s);
    g_prof.recs.push_back({name, a, b});
    *after = b;
}

// Launches a kernel with programmatic stream serialization (see pdl_wait() in the
// device code) and returns the launch status.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = grid;
    lc.blockDim = block;
    lc.dynamicSmemBytes = smem;
    lc.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = at;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, kernel, std::forward<Args>(args)...);
}

// The same launch as clusters of cluster_x CTAs along x (grid.x a multiple of it).
template <typename... KArgs, typename... Args>
cudaError_t launch_k_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, int cluster_x, Args&&... args) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = grid;
    lc.blockDim = block;
    lc.dynamicSmemBytes = smem;
    lc.stream = stream;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = (unsigned)cluster_x;
    at[1].val.clusterDim.y = 1;
    at[1].val.clusterDim.z = 1;
    lc.attrs = at;
    lc.numAttrs = 2;
    return cudaLaunchKernelEx(&lc, kernel, std::forward<Args>(args)...);
}

// EXPR is a launch_k(...) call.
#define MOE_LAUNCH(NAME, STREAM, ...)                                   \
    do {                                                                \
        cudaEvent_t moe_after_;                                         \
        prof_pre(NAME, STREAM, &moe_after_);                            \
        const cudaError_t moe_err_ = (__VA_ARGS__);                     \
        if (moe_after_) cudaEventRecord(moe_after_, STREAM);            \
        g_launches.fetch_add(1, std::memory_order_relaxed);             \
        if (moe_err_ != cudaSuccess) return MOE_ERR_CUDA;               \
    } while (0)

// ---------------------------------------------------------------------------------
// device facts
// ---------------------------------------------------------------------------------
int current_device() {
    int dev = 0;
    cudaGetDevice(&dev);
    return dev;
}

int num_sms() {
    static int cache[64] = {0};
    const int dev = current_device();
    if (dev < 0 || dev >= 64) return 148;
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D bf16 tensor [rows, cols] (cols contiguous) read in boxes of 64 columns x
// box_rows rows with the 128-byte swizzle; out-of-range rows read as zero.
bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D int8 tensor [rows, cols] read in boxes of box_cols bytes x box_rows rows, unswizzled
// or swizzled (the INT8 GEMMs widen the codes themselves).
bool make_tmap_i8(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                  uint32_t box_cols = 64, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D output [rows, cols] of fp32 (or fp16) with a row stride of ld elements, written in
// boxes of 128 bytes x 32 rows with the 128-byte swizzle (the grouped GEMM's fp32 and
// compact epilogues).
bool make_tmap_out(CUtensorMap* m, void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                   bool fp16) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const uint64_t es = fp16 ? 2 : 4;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {ld * es};
    const cuuint32_t box[2] = {(cuuint32_t)(128 / es), GM_OUT_BOX};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base,
              dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Bytes per row of the chunk exponents of compact expert-output rows of d values: one per
// 32 columns, rounded up to 16 so that a row's exponents start 16-byte aligned.
int compact_exp_ld(long long d) { return (int)(((d / 32) + 15) & ~15ll); }

// ---------------------------------------------------------------------------------
// validation
// ---------------------------------------------------------------------------------
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool is_bf16_kind(const moe_config& c) {
    return c.kind == MOE_EXPERT_GELU || c.kind == MOE_EXPERT_SWIGLU;
}

int64_t n1_of(const moe_config& c) {
    return c.kind == MOE_EXPERT_LINEAR ? c.d : (c.kind == MOE_EXPERT_GELU ? c.F : 2ll * c.F);
}

moe_status check_cfg(const moe_config* c) {
    if (!c) return MOE_ERR_INVALID_ARG;
    if (c->T < 0 || c->E < 1 || c->E > 1024 || c->top_k < 1 || c->top_k > 32 || c->top_k > c->E)
        return MOE_ERR_INVALID_ARG;
    if (c->d < 8 || c->d % 8 != 0) return MOE_ERR_INVALID_ARG;
    if ((int64_t)c->T * c->top_k >= (1ll << 31)) return MOE_ERR_INVALID_ARG;
    if (!std::isfinite(c->capacity_factor)) return MOE_ERR_INVALID_ARG;
    if ((c->has_shared != 0 && c->has_shared != 1) || (c->add_residual != 0 && c->add_residual != 1))
        return MOE_ERR_INVALID_ARG;
    if (c->act_dtype != MOE_F32 && c->act_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if (c->w_dtype != 0 && c->w_dtype != c->act_dtype) {
        if (c->w_dtype != MOE_I8 && c->w_dtype != MOE_I4) return MOE_ERR_INVALID_ARG;
        if (c->kind != MOE_EXPERT_GELU && c->kind != MOE_EXPERT_SWIGLU) return MOE_ERR_UNSUPPORTED;
    }
    if (c->overflow < MOE_OVERFLOW_DROP || c->overflow > MOE_OVERFLOW_REROUTE) return MOE_ERR_INVALID_ARG;
    if (c->overflow == MOE_OVERFLOW_SHARED && !c->has_shared) return MOE_ERR_INVALID_ARG;
    if (c->n_group != 0) {
        if (c->n_group < 1 || c->n_group > 32 || c->E % c->n_group != 0) return MOE_ERR_INVALID_ARG;
        if (c->topk_group < 1 || c->topk_group > c->n_group) return MOE_ERR_INVALID_ARG;
        if ((int64_t)c->top_k > (int64_t)c->topk_group * (c->E / c->n_group)) return MOE_ERR_INVALID_ARG;
    }
    switch (c->kind) {
        case MOE_EXPERT_LINEAR:
            if (c->act_dtype != MOE_F32) return MOE_ERR_UNSUPPORTED;
            break;
        case MOE_EXPERT_GELU:
        case MOE_EXPERT_SWIGLU:
            if (c->act_dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
            if (c->d % 64 != 0 || c->F < 64 || c->F % 64 != 0) return MOE_ERR_INVALID_ARG;
            if ((int64_t)c->E * n1_of(*c) >= (1ll << 31) || (int64_t)c->E * c->d >= (1ll << 31))
                return MOE_ERR_INVALID_ARG;
            break;
        default:
            return MOE_ERR_INVALID_ARG;
    }
    return MOE_OK;
}

int32_t capacity_of(const moe_config& c) {
    if (!(c.capacity_factor > 0.0f)) return c.T;
    double v = std::ceil((double)c.capacity_factor * (double)c.T * (double)c.top_k / (double)c.E);
    if (v < 1.0) v = 1.0;
    if (v > (double)c.T) v = (double)c.T;
    return (int32_t)v;
}

// ---------------------------------------------------------------------------------
// workspace layout (256-byte aligned regions, identical for every entry point)
// ---------------------------------------------------------------------------------
// ---------------------------------------------------------------------------------
// split-K plan of one grouped-GEMM launch
// ---------------------------------------------------------------------------------
// When an upper bound on the launch's output tiles cannot fill the SMs twice, every
// tile is cut along K into S units (at least 4 K blocks each) so that the units
// spread over whole waves of SMs; S maximises the fraction of SM slots in use
// (a larger S must win by 2 %). The plan depends only on the configuration, so the
// workspace can hold its partial sums.
struct SplitPlan {
    int S = 1;
    int kbs = 0;   // K blocks per split
};

SplitPlan split_plan(long long max_mtiles, int n_tiles, int K, int sms, int bk = GM_BK) {
    // bk: K elements per block of the kernel that runs (GM_BK, or QT_BK for the
    // weight-streaming INT8 kernel)
    SplitPlan sp;
    const int KB = (K + bk - 1) / bk;
    sp.kbs = KB;
    const long long tiles = max_mtiles * n_tiles;
    if (tiles <= 0 || tiles >= 2ll * sms) return sp;
    auto eff = [&](long long units) {
        const long long waves = (units + sms - 1) / sms;
        return (double)units / (double)(waves * sms);
    };
    double best = eff(tiles);
    for (int S = 2; S <= 16; ++S) {
        const int kbs = (KB + S - 1) / S;
        if (kbs < 4) break;
        const int Se = (KB + kbs - 1) / kbs;
        const double e = eff(tiles * Se);
        if (e > best + 0.02) {
            best = e;
            sp.S = Se;
            sp.kbs = kbs;
        }
    }
    return sp;
}

// Router scratch: raw partial logits (and, on the tensor-core path, the split gate
// weights and the one-group tables). Paths: fp32 activations -> CUDA-core GEMM;
// bf16 activations with T >= kRouterTensorMinT -> exact 3-way bf16 split on the tensor
// cores; fewer bf16 tokens -> split-K CUDA-core kernel.
constexpr int kRouterTensorMinT = 256;

struct RouterPlan {
    int path;                 // 1 fp32 CUDA core, 2 tensor cores, 3 split-K
    int Ep;                   // padded experts per term (path 2)
    int n_parts;
    long long part_stride, row_stride;
    size_t bg_bytes, d_bytes, scratch_bytes;
    int ksplit = 1;           // path 2 with the fused top-k: K split of the router GEMM
    long long mtiles = 0;     // its M tiles
};

size_t al256(size_t b) { return (b + 255) & ~size_t(255); }

// The whole dispatch in one CTA (few assignments and experts, no re-routing).
bool dispatch_one_cta(const moe_config& c) {
    return (long long)c.T * c.top_k <= kOneCtaMaxAssign && c.E <= kOneCtaMaxE &&
           c.overflow != MOE_OVERFLOW_REROUTE;
}

// The tensor-core router selects the top k in its GEMM epilogue when the three terms of
// the padded experts fit one accumulator, routing is plain top-k and no re-routing
// candidates are needed.
bool router_fused_topk(const moe_config& c, int Ep) {
    return Ep <= 64 && c.n_group == 0 && c.overflow != MOE_OVERFLOW_REROUTE;
}

RouterPlan router_plan(const moe_config& c) {
    RouterPlan r{};
    const size_t T = (size_t)c.T, E = (size_t)c.E, d = (size_t)c.d;
    if (c.act_dtype == MOE_F32) {
        r.path = 1;
        r.n_parts = 1;
        r.row_stride = c.E;
        r.scratch_bytes = al256(T * E * 4);
    } else if (c.T >= kRouterTensorMinT) {
        r.path = 2;
        r.Ep = (c.E + kRouterPad - 1) / kRouterPad * kRouterPad;
        r.n_parts = 3;
        r.part_stride = r.Ep;
        r.row_stride = 3ll * r.Ep;
        r.bg_bytes = al256(3 * (size_t)r.Ep * d * 2);
        // partial logits when the three terms do not fit one accumulator (E > 64); otherwise
        // the GEMM epilogue selects the top k itself, with K split in two when there are
        // too few M tiles to fill half the SMs and K is long enough for the split to pay
        // (d >= 2048; two partial logit sets, per-tile counters)
        const bool fused = router_fused_topk(c, r.Ep);
        r.mtiles = ((long long)c.T + 127) / 128;
        r.ksplit = (fused && 2 * r.mtiles <= num_sms() && c.d / GM_BK >= 32) ? 2 : 1;
        r.d_bytes = fused ? (r.ksplit > 1 ? al256(2 * T * (size_t)r.Ep * 4) : 0)
                          : al256(T * 3 * (size_t)r.Ep * 4);
        r.scratch_bytes = r.bg_bytes + r.d_bytes + 256 +
                          (r.ksplit > 1 ? al256((size_t)r.mtiles * 4) : 0);
    } else {
        r.path = 3;
        r.n_parts = (c.d + RS_K - 1) / RS_K;
        r.part_stride = (long long)c.T * c.E;
        r.row_stride = c.E;
        r.scratch_bytes = al256((size_t)r.n_parts * T * E * 4);
    }
    return r;
}

// Weight-only quantised experts: codes plus one fp32 scale per weight row.
bool quant_w(const moe_config& c) { return c.w_dtype == MOE_I8 || c.w_dtype == MOE_I4; }
// Bits per weight code of the expert GEMMs (16: bf16 weights).
int code_bits(const moe_config& c) {
    return c.w_dtype == MOE_I4 ? 4 : c.w_dtype == MOE_I8 ? 8 : 16;
}

// INT8 experts with few rows per group run the weight-streaming kernel
// (grouped_gemm_q8t_kernel: operands swapped, 32-row activation tiles): the routed
// experts when they average at most 32 rows, the shared expert up to 64 tokens.
// INT4 experts always run it. Routed bf16 experts run its bf16 mode when they average at
// most kStreamBf16Rows rows (decode): the 128-row tiles of the bf16 kernel would carry
// a zero-filled A tile for each token row.
constexpr int kStreamBf16Rows = 4;
bool q8t_routed(const moe_config& c) {
    if (c.w_dtype == MOE_I4) return true;
    if (c.w_dtype == MOE_I8) return (long long)c.T * c.top_k <= 32ll * c.E;
    return is_bf16_kind(c) && (long long)c.T * c.top_k <= (long long)kStreamBf16Rows * c.E;
}
bool q8t_shared(const moe_config& c) {
    return c.w_dtype == MOE_I4 || (c.w_dtype == MOE_I8 && c.T <= 64);
}

// Tile heights of the bf16 expert GEMMs. 256-row tiles (two M = 128 MMAs sharing each B
// tile, one accumulator set) move a third fewer operand bytes per FLOP and their 3-stage
// ring covers 1.5x the load latency of the 128-row tiles' 4-stage ring, but their epilogue
// no longer overlaps the next tile's MMAs. Measured (per-role wait counters): they win for
// groups of >= ~200 rows when K is long enough for the mainloop to dwarf the epilogue --
// the up projections (K = d) and down projections with K = F >= 4096; for the DeepSeek-V3
// down projection (K = 2048, fp32 row stores) they lose. With 256-row tiles the A rows are
// read from a materialised x_perm by TMA: the cp.async row gather cannot keep enough of
// the 3-stage ring in flight.
constexpr double kWideTileMinRows = 192.0;
constexpr int kWideDownMinK = 4096;

struct ExpertTiles {
    int up = 1, down = 1, sh_up = 1, sh_down = 1;
};

ExpertTiles expert_tiles(const moe_config& c) {
    ExpertTiles t;
    if (c.kind == MOE_EXPERT_LINEAR || c.w_dtype == MOE_I8 || c.w_dtype == MOE_I4) return t;
    const double routed_rows = (double)c.T * c.top_k / c.E;
    const bool r = routed_rows >= kWideTileMinRows, sh = (double)c.T >= kWideTileMinRows;
    t.up = r ? 2 : 1;
    t.down = (r && c.F >= kWideDownMinK) ? 2 : 1;
    t.sh_up = sh ? 2 : 1;
    t.sh_down = (sh && c.F >= kWideDownMinK) ? 2 : 1;
    return t;
}

// Split plan of a weight-streaming launch, in 128-code K blocks. An INT4 code stage holds
// two of them and a split must start on one, so INT4 plans are made over 256-code blocks.
SplitPlan qt_split_plan(long long max_mtiles, int n_tiles, int K, int sms, int bits) {
    const int per = bits >= 8 ? 1 : 8 / bits;
    SplitPlan sp = split_plan(max_mtiles, n_tiles, K, sms, QT_BK * per);
    sp.kbs *= per;
    return sp;
}

// Upper bound on the M tiles of the routed experts: sum_e ceil(n_e / m) over the
// non-empty experts <= P / m + min(E, P), m = 128 rows (32 for the weight-streaming
// INT8 kernel).
long long routed_mtiles_bound(const moe_config& c) {
    const long long Pmax = (long long)c.T * c.top_k;
    return Pmax / (q8t_routed(c) ? QT_NT : kMTile) + std::min<long long>(c.E, Pmax);
}

struct FfnPlan {
    SplitPlan up, down, sh_up, sh_down;
    size_t partial_floats = 0;   // largest partial buffer any of the four launches needs
};

FfnPlan ffn_plan(const moe_config& c) {
    FfnPlan f;
    if (!(c.kind == MOE_EXPERT_GELU || c.kind == MOE_EXPERT_SWIGLU)) return f;
    const int sms = num_sms();
    const long long Pmax = (long long)c.T * c.top_k;
    const int up_nt = c.kind == MOE_EXPERT_SWIGLU ? (c.F + 127) / 128 : (c.F + GM_BN - 1) / GM_BN;
    const int dn_nt = (c.d + GM_BN - 1) / GM_BN;
    const long long N1 = c.kind == MOE_EXPERT_SWIGLU ? 2ll * c.F : c.F;
    const long long mt = routed_mtiles_bound(c);
    const int bits = code_bits(c);
    f.up = q8t_routed(c) ? qt_split_plan(mt, up_nt, c.d, sms, bits) : split_plan(mt, up_nt, c.d, sms);
    f.down = q8t_routed(c) ? qt_split_plan(mt, dn_nt, c.F, sms, bits) : split_plan(mt, dn_nt, c.F, sms);
    auto need = [&](const SplitPlan& sp, long long rows, long long cols) {
        if (sp.S > 1) f.partial_floats = std::max<size_t>(f.partial_floats, (size_t)(sp.S * rows * cols));
    };
    need(f.up, Pmax, N1);
    need(f.down, Pmax, c.d);
    if (c.has_shared) {
        const int sm = q8t_shared(c) ? QT_NT : kMTile;
        const long long smt = (c.T + sm - 1) / sm;
        f.sh_up = q8t_shared(c) ? qt_split_plan(smt, up_nt, c.d, sms, bits)
                                : split_plan(smt, up_nt, c.d, sms);
        f.sh_down = q8t_shared(c) ? qt_split_plan(smt, dn_nt, c.F, sms, bits)
                                  : split_plan(smt, dn_nt, c.F, sms);
        need(f.sh_up, c.T, N1);
        need(f.sh_down, c.T, c.d);
    }
    return f;
}

// Tile counters of the expert-stage grouped-GEMM launches (dynamic scheduling).
enum { kCntUp = 0, kCntDown = 1, kCntSharedUp = 2, kCntSharedDown = 3, kNumCounters = 4 };

struct WsLayout {
    size_t logits, idx, w, load, counts, offsets, blockcnt, blockoff, cand, prop, cnt0,
        perm_token, perm_slot,
        slot_dest, x_perm, mtile, shared_tab, counters, h, hs, y, partial, total;
};

WsLayout ws_layout(const moe_config& c) {
    WsLayout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += (bytes + 255) & ~size_t(255);
        return o;
    };
    const size_t T = (size_t)c.T, k = (size_t)c.top_k, E = (size_t)c.E, d = (size_t)c.d;
    const size_t F = (size_t)std::max(c.F, 0);
    const size_t Pmax = T * k;
    const size_t nb = std::max<size_t>(1, (T + kDispTok - 1) / kDispTok);
    const size_t es = c.act_dtype == MOE_BF16 ? 2 : 4;
    L.logits = take(router_plan(c).scratch_bytes);   // router scratch
    L.idx = take(Pmax * 4);
    L.w = take(Pmax * 4);
    L.load = take(E * 4);
    L.counts = take(E * 4);
    L.offsets = take((E + 2) * 4);   // + the shared expert's end (moe_forward)
    L.blockcnt = take(std::max(nb, (T + 31) / 32) * E * 4);   // per chunk, or per 32 tokens
    L.blockoff = take(nb * E * 4);
    const bool rr = c.overflow == MOE_OVERFLOW_REROUTE;
    L.cand = take(rr ? Pmax * 4 : 0);
    L.prop = take(rr ? Pmax * 4 : 0);
    L.cnt0 = take(rr ? E * 4 : 0);
    L.perm_token = take(Pmax * 4);
    L.perm_slot = take(Pmax * 4);
    L.slot_dest = take(Pmax * 4);
    L.x_perm = take(Pmax * d * es);
    L.mtile = take((E + 2) * 4);
    L.shared_tab = take(4 * 4);
    L.counters = take(kNumCounters * 8);
    // H rows: routed [0, P) and, when moe_forward runs the shared expert as an extra group of
    // the routed up projection, the shared expert's rows [P, P + T)
    L.h = take(is_bf16_kind(c) ? (Pmax + (c.has_shared ? T : 0)) * F * 2 : 0);
    L.hs = take(is_bf16_kind(c) && c.has_shared ? T * F * 2 : 0);
    L.y = take((Pmax + (c.has_shared ? T : 0)) * d * 4);
    L.partial = take(ffn_plan(c).partial_floats * 4);
    L.total = off;
    return L;
}

template <typename P>
P* at(void* ws, size_t off) {
    return reinterpret_cast<P*>(static_cast<char*>(ws) + off);
}

// ---------------------------------------------------------------------------------
// stage implementations (arguments already validated)
// ---------------------------------------------------------------------------------
moe_status dispatch_impl(const moe_config& c, const int32_t* idx, const void* x, int32_t* load,
                         int32_t* counts, int32_t* offsets, int32_t* perm_token, int32_t* perm_slot,
                         int32_t* slot_dest, void* x_perm, int32_t* blockcnt, int32_t* blockoff,
                         int32_t* mtile, unsigned long long* counters, cudaStream_t s,
                         const int32_t* cand = nullptr, int32_t* prop = nullptr,
                         int32_t* cnt0 = nullptr, DroppedRows dr = DroppedRows{},
                         bool hist_ready = false) {
    // hist_ready: blockcnt already holds the expert histogram, one row per 32 tokens
    // (filled by the router's top-k epilogue)
    // counters (nullable): the routed up/down GEMM tile counters, zeroed here
    // cand, prop, cnt0: re-routing candidates (from the router) and scratch
    // dr: top-1 layers with the combine fused into the down projection write the output
    //     rows of dropped tokens here
    const int T = c.T, E = c.E, k = c.top_k;
    const int cap = capacity_of(c);
    const int nb = (T + kDispTok - 1) / kDispTok;
    const int rsm = kDispWarps * E * sizeof(int);
    if (c.overflow == MOE_OVERFLOW_REROUTE) {
        if (!cand || !prop || !cnt0) return MOE_ERR_UNSUPPORTED;
        // round 0 (ranks only), proposals of the dropped slots, room and offsets, then
        // ranks of the proposals and the scatter of every slot
        MOE_LAUNCH("dispatch_hist", s,
                   launch_k(dispatch_hist_kernel, nb, 256, kDispWarps * E * sizeof(int), s, idx, T, k, E,
                            blockcnt));
        MOE_LAUNCH("dispatch_scan", s,
                   launch_k(dispatch_scan_kernel, 1, 1024, 0, s, blockcnt, nb, E, cap, blockoff,
                            load, counts, offsets, nullptr, nullptr, 0));
        MOE_LAUNCH("dispatch_rank_status", s,
                   launch_k(dispatch_rank_kernel<kRankStatus>, nb, 256, rsm, s, idx, T, k, E, cap,
                            blockoff, offsets, perm_token, perm_slot, slot_dest, nullptr, nullptr,
                            DroppedRows{}));
        MOE_LAUNCH("reroute_propose", s,
                   launch_k(reroute_propose_kernel, nb, 256, kDispWarps * E * sizeof(int), s, slot_dest, cand,
                            T, k, E, prop, blockcnt));
        MOE_LAUNCH("reroute_scan", s,
                   launch_k(reroute_scan_kernel, 1, 1024, 0, s, blockcnt, nb, E, cap, blockoff,
                            counts, cnt0, offsets, mtile, counters, 2));
        MOE_LAUNCH("dispatch_rank_reroute", s,
                   launch_k(dispatch_rank_kernel<kRankReroute>, nb, 256, rsm, s, prop, T, k, E,
                            cap, blockoff, offsets, perm_token, perm_slot, slot_dest, idx, cnt0, dr));
    } else if ((long long)T * k <= kTinyAssign) {
        MOE_LAUNCH("dispatch_tiny", s,
                   launch_k(dispatch_tiny_kernel, 1, 32, 2 * E * sizeof(int), s, idx, T, k, E, cap,
                            load, counts, offsets, perm_token, perm_slot, slot_dest, mtile,
                            counters, 2, dr));
    } else if (dispatch_one_cta(c)) {
        MOE_LAUNCH("dispatch_one_cta", s,
                   launch_k(dispatch_one_cta_kernel, 1, 1024, 33 * E * sizeof(int), s, idx, T, k,
                            E, cap, load, counts, offsets, perm_token, perm_slot, slot_dest,
                            mtile, counters, 2, dr, nullptr, 0, 1));
    } else {
        if (!hist_ready)
            MOE_LAUNCH("dispatch_hist", s,
                       launch_k(dispatch_hist_kernel, nb, 256, kDispWarps * E * sizeof(int), s, idx, T, k, E,
                                blockcnt));
        if (E <= kOneCtaMaxE) {
            // one CTA per chunk: scan folded into the ranking kernel
            MOE_LAUNCH("dispatch_rank", s,
                       launch_k(dispatch_one_cta_kernel, nb, 1024, 33 * E * sizeof(int), s, idx, T,
                                k, E, cap, load, counts, offsets, perm_token, perm_slot, slot_dest,
                                mtile, counters, 2, dr, blockcnt, nb,
                                hist_ready ? kDispTok / 32 : 1));
        } else {
            MOE_LAUNCH("dispatch_scan", s,
                       launch_k(dispatch_scan_kernel, 1, 1024, 0, s, blockcnt, nb, E, cap, blockoff,
                                load, counts, offsets, mtile, counters, 2));
            MOE_LAUNCH("dispatch_rank", s,
                       launch_k(dispatch_rank_kernel<kRankScatter>, nb, 256, rsm, s, idx, T, k, E,
                                cap, blockoff, offsets, perm_token, perm_slot, slot_dest, nullptr,
                                nullptr, dr));
        }
    }
    if (x_perm) {
        const int es = c.act_dtype == MOE_BF16 ? 2 : 4;
        const long long Pmax = (long long)T * k;
        if (k >= 2) {   // by token: every row of x read once
            const int blocks = (int)std::min<long long>((T + 7) / 8, (long long)num_sms() * 16);
            MOE_LAUNCH("gather_rows", s,
                       launch_k(gather_rows_by_token_kernel, std::max(blocks, 1), 256, 0, s,
                                static_cast<const uint8_t*>(x), slot_dest, T, k,
                                static_cast<uint8_t*>(x_perm), c.d * es));
        } else {
            const int blocks = (int)std::min<long long>((Pmax + 7) / 8, (long long)num_sms() * 16);
            MOE_LAUNCH("gather_rows", s,
                       launch_k(gather_rows_kernel, std::max(blocks, 1), 256, 0, s,
                           static_cast<const uint8_t*>(x), perm_token, offsets + E,
                           static_cast<uint8_t*>(x_perm), c.d * es));
        }
    }
    return MOE_OK;
}

template <int EPI>
const char* gemm_name() {
    switch (EPI) {
        case EPI_F32: return "grouped_gemm_f32";
        case EPI_GELU_BF16: return "grouped_gemm_gelu";
        case EPI_SWIGLU_BF16: return "grouped_gemm_swiglu";
        case EPI_COMBINE1_BF16: return "grouped_gemm_combine1";
        case EPI_ROUTER_TOPK: return "router_gemm_topk";
        case EPI_SCALE_H16: return "grouped_gemm_scale_h16";
        default: return "grouped_gemm_scale";
    }
}

template <int EPI>
const char* gemm_q8_name() {
    switch (EPI) {
        case EPI_F32: return "grouped_gemm_q8_f32";
        case EPI_GELU_BF16: return "grouped_gemm_q8_gelu";
        case EPI_SWIGLU_BF16: return "grouped_gemm_q8_swiglu";
        case EPI_COMBINE1_BF16: return "grouped_gemm_q8_combine1";
        default: return "grouped_gemm_q8_scale";
    }
}

template <int EPI>
const char* gemm_q8t_name(int bits) {
    const int b = bits == 4 ? 0 : bits == 8 ? 1 : 2;
    static const char* const f32[3] = {"grouped_gemm_q4t_f32", "grouped_gemm_q8t_f32",
                                       "grouped_gemm_st_f32"};
    static const char* const gelu[3] = {"grouped_gemm_q4t_gelu", "grouped_gemm_q8t_gelu",
                                        "grouped_gemm_st_gelu"};
    static const char* const swiglu[3] = {"grouped_gemm_q4t_swiglu", "grouped_gemm_q8t_swiglu",
                                          "grouped_gemm_st_swiglu"};
    static const char* const scale[3] = {"grouped_gemm_q4t_scale", "grouped_gemm_q8t_scale",
                                         "grouped_gemm_st_scale"};
    switch (EPI) {
        case EPI_F32: return f32[b];
        case EPI_GELU_BF16: return gelu[b];
        case EPI_SWIGLU_BF16: return swiglu[b];
        default: return scale[b];
    }
}

constexpr bool q8t_supports(int epi) {
    return epi == EPI_F32 || epi == EPI_GELU_BF16 || epi == EPI_SWIGLU_BF16 || epi == EPI_SCALE_F32;
}

template <int EPI>
const char* reduce_name() {
    switch (EPI) {
        case EPI_F32: return "splitk_reduce_f32";
        case EPI_GELU_BF16: return "splitk_reduce_gelu";
        case EPI_SWIGLU_BF16: return "splitk_reduce_swiglu";
        default: return "splitk_reduce_scale";
    }
}

// CTAs of a paired 128-row grouped GEMM launch: twice the number of two-CTA clusters that can
// be resident at once (at most one CTA per SM; the pair schedule is round-robin, so every
// cluster should be resident from the start), or 0 when that cannot be determined.
template <int EPI>
int gm_pair_grid(int sms) {
    static std::once_flag once[64];
    static int grid[64];
    const int dev = current_device();
    if (dev < 0 || dev >= 64) return 0;
    std::call_once(once[dev], [&] {
        grid[dev] = 0;
        if (cudaFuncSetAttribute(grouped_gemm_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 gm_smem_bytes(GM_MAX_GROUPS, 1, EPI)) != cudaSuccess)
            return;
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3((unsigned)(sms & ~1));
        lc.blockDim = dim3(GM_THREADS);
        lc.dynamicSmemBytes = gm_smem_bytes(GM_MAX_GROUPS, 1, EPI);
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = 2;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        lc.attrs = at;
        lc.numAttrs = 1;
        int nc = 0;
        if (cudaOccupancyMaxActiveClusters(&nc, grouped_gemm_kernel<EPI>, &lc) == cudaSuccess)
            grid[dev] = 2 * std::min(nc, sms / 2);
    });
    return grid[dev];
}

// One grouped-GEMM launch (plus, when sp.S > 1, the split-K reduction that applies the
// epilogue). `partial` must hold sp.S * a_rows * (SwiGLU ? 2N : N) floats when split.
template <int EPI>
moe_status launch_gemm(const void* A, int64_t a_rows, int K, const void* B, int64_t b_rows_total,
                       int b_rows_per_group, int G, int N, const int32_t* row_offsets,
                       const int32_t* mtile_offsets, void* out, long long ld_out, const float* bias,
                       const float* topk_w, const int32_t* perm_token, const int32_t* perm_slot,
                       int top_k, cudaStream_t s, const char* name = nullptr,
                       SplitPlan sp = SplitPlan(), float* partial = nullptr,
                       unsigned long long* counter = nullptr, const void* resid = nullptr,
                       int* r_idx = nullptr, float* r_w = nullptr, int r_E = 0, int r_Ep = 0,
                       const float* w_scale = nullptr, bool swap_ab = false,
                       int* r_hist = nullptr, const int32_t* a_gather = nullptr,
                       int a_row_bytes = 0, float* r_part = nullptr, int* r_tile_cnt = nullptr,
                       int w_bits = 8, int mt = 1, const void* A2 = nullptr, int64_t a2_rows = 0,
                       const void* B2 = nullptr, int64_t b2_rows = 0, const float* bias2 = nullptr,
                       int xg = -1, bool out_local = false, int64_t out_rows = -1,
                       int8_t* out_exp = nullptr, bool pair_ok = false) {
    // mt: 128-row halves per tile of the bf16 kernel (2: 256-row tiles, unsplit launches)
    // out_rows: rows of out (default a_rows: output rows are numbered like A's)
    // out_exp (EPI_SCALE_H16, bf16 kernel, unsplit): the chunk exponents of out's rows,
    // compact_exp_ld(ld_out) bytes per row
    // pair_ok: run 128-row tiles in CTA pairs sharing each B tile (GemmParams::pair) when
    // the launch allows it (unsplit, TMA-loaded A, no extra group, bf16 weights)
    // xg >= 0 (bf16 kernel, unsplit): group xg reads A rows 0.. of A2 [a2_rows, K] (gathered
    // A: rows 0.. of A itself) and weights B2 [b2_rows, K], with bias bias2
    // out_local: output row r of the (single) group is row r of out
    // r_part, r_tile_cnt (EPI_ROUTER_TOPK with sp.S == 2): the epilogue's split-K exchange
    // a_gather (bf16 kernel only): logical A row r (r < a_rows) is row a_gather[r] of A,
    // loaded by the kernel's gather warps
    // w_scale != null: B holds w_bits-wide codes (8: int8; 4: two per byte, even k in the
    // low nibble), one fp32 scale per B row (INT8 / INT4 kernels); with swap_ab the
    // weight-streaming kernel for few rows per group runs (INT4: only that kernel)
    if (a_rows <= 0 || G <= 0) return MOE_OK;
    if (G > GM_MAX_GROUPS) return MOE_ERR_UNSUPPORTED;
    if (EPI == EPI_SCALE_H16 && (w_scale || (sp.S > 1 && partial) || !out_exp || ld_out % 32 != 0))
        return MOE_ERR_UNSUPPORTED;
    // (bf16 weights stream through the swapped kernel too: w_bits 16, no row scales)
    swap_ab = swap_ab && (w_scale != nullptr || w_bits == 16);
    if (swap_ab && !q8t_supports(EPI)) return MOE_ERR_UNSUPPORTED;
    if (w_scale && w_bits != 8 && (w_bits != 4 || !swap_ab)) return MOE_ERR_UNSUPPORTED;
    if (w_bits == 4 && sp.S > 1 && sp.kbs % 2 != 0) return MOE_ERR_UNSUPPORTED;
    CUtensorMap ta, tb, ta2, tb2;
    const bool gathered = a_gather && !w_scale;
    if (xg >= 0 && (w_scale || sp.S > 1 || !B2)) return MOE_ERR_UNSUPPORTED;
    const uint64_t b_cols = (w_scale && w_bits == 4) ? (uint64_t)K / 2
                            : (swap_ab && w_bits == 16) ? 2ull * K : (uint64_t)K;   // bytes
    if (swap_ab ? !make_tmap_i8(&tb, B, (uint64_t)b_rows_total, b_cols, GM_BN / 2, QT_BK,
                                CU_TENSOR_MAP_SWIZZLE_128B)
        : w_scale ? !make_tmap_i8(&tb, B, (uint64_t)b_rows_total, (uint64_t)K, GM_BN / 2)
                  : !make_tmap_bf16(&tb, B, (uint64_t)b_rows_total, (uint64_t)K, GM_BN / 2))
        return MOE_ERR_CUDA;
    // gathered A is read with cp.async, not through a tensor map (a_rows counts the
    // logical, permuted rows)
    if (gathered) ta = tb;
    else if (!make_tmap_bf16(&ta, A, (uint64_t)a_rows, (uint64_t)K, swap_ab ? QT_NT : GM_BM))
        return MOE_ERR_CUDA;
    ta2 = ta;
    tb2 = tb;
    if (xg >= 0) {
        if (!make_tmap_bf16(&tb2, B2, (uint64_t)b2_rows, (uint64_t)K, GM_BN / 2)) return MOE_ERR_CUDA;
        if (!gathered && !make_tmap_bf16(&ta2, A2, (uint64_t)a2_rows, (uint64_t)K, GM_BM))
            return MOE_ERR_CUDA;
    }
    GemmParams p{};
    p.G = G;
    p.N = N;
    p.K = K;
    p.b_rows_per_group = b_rows_per_group;
    p.up_offset = (EPI == EPI_SWIGLU_BF16) ? N : GM_BN / 2;
    p.n_tiles = (EPI == EPI_SWIGLU_BF16) ? (N + 127) / 128 : (N + GM_BN - 1) / GM_BN;
    p.row_offsets = row_offsets;
    p.mtile_offsets = mtile_offsets;
    p.out = out;
    p.ld_out = ld_out;
    p.bias = bias;
    p.topk_w = topk_w;
    p.perm_token = perm_token;
    p.perm_slot = perm_slot;
    p.top_k = top_k;
    const bool split = sp.S > 1 && partial != nullptr;
    p.k_splits = split ? sp.S : 1;
    p.kb_per_split = split ? sp.kbs : (swap_ab ? (K + QT_BK - 1) / QT_BK : K / GM_BK);
    p.partial = split ? partial : nullptr;
    p.ld_part = (EPI == EPI_SWIGLU_BF16) ? 2ll * N : N;
    p.part_stride = (long long)a_rows * p.ld_part;
    p.tile_counter = counter;
    p.xg1 = xg + 1;
    p.xg_bias = bias2;
    p.out_local = out_local ? 1 : 0;
    p.out_exp = out_exp;
    p.ld_exp = compact_exp_ld(ld_out);
    bool pair = pair_ok && mt == 1 && !split && !gathered && xg < 0 && !w_scale &&
                EPI != EPI_ROUTER_TOPK;
    const int pair_grid = pair ? gm_pair_grid<EPI>(num_sms()) : 0;
    if (pair_grid < 2) pair = false;
    p.pair = pair ? 1 : 0;
    // fp32 (and compact fp16) outputs of the bf16 kernel leave through a tensor map when
    // its strides allow
    CUtensorMap td = ta;
    // (128-row tiles only: with 256-row tiles the epilogue frees TMEM for the next tile's
    // MMAs, and the staging buffer's reuse waits slowed it down)
    const long long out_es = EPI == EPI_SCALE_H16 ? 2 : 4;
    if (gm_stages_out(EPI) && mt == 1 && !split && !w_scale && (ld_out * out_es) % 16 == 0 &&
        aligned16(out) && N > 0 &&
        make_tmap_out(&td, out, (uint64_t)(out_rows >= 0 ? out_rows : a_rows), (uint64_t)N,
                      (uint64_t)ld_out, EPI == EPI_SCALE_H16))
        p.tma_out = 1;
    p.resid = static_cast<const __nv_bfloat16*>(resid);
    p.r_idx = r_idx;
    p.r_w = r_w;
    p.r_E = r_E;
    p.r_Ep = r_Ep;
    p.w_scale = w_scale;
    p.r_hist = r_hist;
    if constexpr (EPI == EPI_ROUTER_TOPK) {
        p.r_rows = a_rows;
        if (sp.S > 1) {   // the epilogue adds the two K parts itself (no partial buffer pass)
            if (sp.S != 2 || !r_part || !r_tile_cnt) return MOE_ERR_UNSUPPORTED;
            p.k_splits = sp.S;
            p.kb_per_split = sp.kbs;
            p.r_part = r_part;
            p.r_tile_cnt = r_tile_cnt;
        }
    }
    if (gathered) {
        p.a_gather = a_gather;
        p.a_src = static_cast<const uint8_t*>(A);
        p.a_row_bytes = a_row_bytes;
    }
    const int smem = gm_smem_bytes(G, 1, EPI);
    static std::once_flag attr_once[64];
    static cudaError_t attr_err[64];
    const int dev = current_device();
    if (dev >= 0 && dev < 64) {
        std::call_once(attr_once[dev], [&] {
            attr_err[dev] = cudaFuncSetAttribute(grouped_gemm_kernel<EPI>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 gm_smem_bytes(GM_MAX_GROUPS, 1, EPI));
        });
        if (attr_err[dev] != cudaSuccess) return MOE_ERR_CUDA;
    }
    const int grid = num_sms();
    if (swap_ab) {
        if constexpr (q8t_supports(EPI)) {
            static std::once_flag qt_once[3][64];
            static cudaError_t qt_err[3][64];
            const int b4 = w_bits == 4 ? 1 : w_bits == 16 ? 2 : 0;
            auto kern = b4 == 1 ? grouped_gemm_q8t_kernel<EPI, 4>
                        : b4 == 2 ? grouped_gemm_q8t_kernel<EPI, 16> : grouped_gemm_q8t_kernel<EPI, 8>;
            if (dev >= 0 && dev < 64) {
                std::call_once(qt_once[b4][dev], [&] {
                    qt_err[b4][dev] = cudaFuncSetAttribute(kern,
                                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                           gm_q8t_smem_bytes(GM_MAX_GROUPS));
                });
                if (qt_err[b4][dev] != cudaSuccess) return MOE_ERR_CUDA;
            }
            MOE_LAUNCH(name ? name : gemm_q8t_name<EPI>(w_bits), s,
                       launch_k(kern, grid, QT_THREADS, gm_q8t_smem_bytes(G), s, ta, tb, p));
        }
    } else if (w_scale) {
        if constexpr (EPI == EPI_SCALE_H16) {
            return MOE_ERR_UNSUPPORTED;   // (rejected above; no INT8 instance of it)
        } else {
            static std::once_flag q8_once[64];
            static cudaError_t q8_err[64];
            if (dev >= 0 && dev < 64) {
                std::call_once(q8_once[dev], [&] {
                    q8_err[dev] = cudaFuncSetAttribute(grouped_gemm_q8_kernel<EPI>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       gm_q8_smem_bytes(GM_MAX_GROUPS));
                });
                if (q8_err[dev] != cudaSuccess) return MOE_ERR_CUDA;
            }
            MOE_LAUNCH(name ? name : gemm_q8_name<EPI>(), s,
                       launch_k(grouped_gemm_q8_kernel<EPI>, grid, GM_Q8_THREADS,
                                gm_q8_smem_bytes(G), s, ta, tb, p));
        }
    } else if (mt == 2 && !split) {
        if constexpr (EPI != EPI_ROUTER_TOPK) {
            static std::once_flag wide_once[64];
            static cudaError_t wide_err[64];
            if (dev >= 0 && dev < 64) {
                std::call_once(wide_once[dev], [&] {
                    wide_err[dev] = cudaFuncSetAttribute(grouped_gemm_kernel<EPI, 2>,
                                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                         gm_smem_bytes(GM_MAX_GROUPS, 2, EPI));
                });
                if (wide_err[dev] != cudaSuccess) return MOE_ERR_CUDA;
            }
            MOE_LAUNCH(name ? name : gemm_name<EPI>(), s,
                       launch_k(grouped_gemm_kernel<EPI, 2>, grid,
                                GM_THREADS + (p.a_gather ? GM_GATHER_THREADS : 0),
                                gm_smem_bytes(G, 2, EPI), s, ta, tb, ta2, tb2, td, p));
        } else {
            return MOE_ERR_UNSUPPORTED;
        }
    } else if (pair) {
        MOE_LAUNCH(name ? name : gemm_name<EPI>(), s,
                   launch_k_cluster(grouped_gemm_kernel<EPI>, pair_grid, GM_THREADS, smem, s, 2, ta,
                                    tb, ta2, tb2, td, p));
    } else {
        MOE_LAUNCH(name ? name : gemm_name<EPI>(), s,
                   launch_k(grouped_gemm_kernel<EPI>, grid,
                            GM_THREADS + (p.a_gather ? GM_GATHER_THREADS : 0), smem, s, ta, tb, ta2,
                            tb2, td, p));
    }
    if constexpr (EPI != EPI_SCALE_H16) {   // (compact rows come from unsplit launches only)
        if (split) {
            const long long work = a_rows * (long long)(N / 4);
            const int blocks = (int)std::max<long long>(
                1, std::min<long long>((work + 255) / 256, (long long)num_sms() * 8));
            MOE_LAUNCH(reduce_name<EPI>(), s,
                       launch_k(splitk_reduce_kernel<EPI>, blocks, 256, 0, s, p, row_offsets + G));
        }
    }
    return MOE_OK;
}

#define MOE_TRY(...)                        \
    do {                                    \
        const moe_status st_ = (__VA_ARGS__); \
        if (st_ != MOE_OK) return st_;      \
    } while (0)

moe_status route_impl(const moe_config& c, const void* x, const float* Wg, const float* bias,
                      float* logits, int32_t* idx, float* w, void* scratch, int32_t* cand,
                      cudaStream_t s, int32_t* hist = nullptr) {
    // cand: the re-routing candidates [T, k] (written iff overflow == REROUTE)
    // hist: the dispatch's expert histogram, one row per 32 tokens [ceil(T / 32)][E], written
    //       by the fused top-k epilogue when non-null (the caller checks that it is fused)
    if (c.overflow != MOE_OVERFLOW_REROUTE) cand = nullptr;
    const int T = c.T, E = c.E, d = c.d, k = c.top_k;
    const RouterPlan rp = router_plan(c);
    float* parts = static_cast<float*>(scratch);
    if (rp.path == 1) {
        const dim3 grid((T + RT_BM - 1) / RT_BM, (E + RT_BN - 1) / RT_BN);
        MOE_LAUNCH("router_logits_f32", s,
                   launch_k(router_logits_kernel<float>, grid, 256, 0, s, static_cast<const float*>(x),
                                                                    Wg, parts, T, d, E));
    } else if (rp.path == 2) {
        __nv_bfloat16* Bg = static_cast<__nv_bfloat16*>(scratch);
        parts = reinterpret_cast<float*>(static_cast<char*>(scratch) + rp.bg_bytes);
        int32_t* tables =
            reinterpret_cast<int32_t*>(static_cast<char*>(scratch) + rp.bg_bytes + rp.d_bytes);
        int32_t* tile_cnt = rp.ksplit > 1
                                ? reinterpret_cast<int32_t*>(static_cast<char*>(scratch) +
                                                             rp.bg_bytes + rp.d_bytes + 256)
                                : nullptr;
        const dim3 grid((d + 31) / 32, rp.Ep / 32);
        MOE_LAUNCH("gate_split", s,
                   launch_k(gate_split_kernel, grid, 256, 0, s,
                       Wg, d, E, rp.Ep, Bg, T, tables,
                       reinterpret_cast<unsigned long long*>(tables + 4), tile_cnt,
                       (int)rp.mtiles));
        if (router_fused_topk(c, rp.Ep)) {   // the three terms fit one accumulator: fused top-k
            SplitPlan sp;
            sp.S = rp.ksplit;
            sp.kbs = (d / GM_BK + sp.S - 1) / sp.S;
            MOE_TRY(launch_gemm<EPI_ROUTER_TOPK>(
                x, T, d, Bg, 3ll * rp.Ep, 3 * rp.Ep, 1, 3 * rp.Ep, tables, tables + 2, logits, E,
                bias, nullptr, nullptr, nullptr, k, s, nullptr, sp, nullptr,
                reinterpret_cast<unsigned long long*>(tables + 4), nullptr, idx, w, E, rp.Ep,
                nullptr, false, hist, nullptr, 0, parts, tile_cnt));
            return MOE_OK;
        }
        MOE_TRY(launch_gemm<EPI_F32>(x, T, d, Bg, 3ll * rp.Ep, 3 * rp.Ep, 1, 3 * rp.Ep, tables,
                                     tables + 2, parts, 3ll * rp.Ep, nullptr, nullptr, nullptr,
                                     nullptr, 1, s, "router_gemm_tc", SplitPlan(), nullptr,
                                     reinterpret_cast<unsigned long long*>(tables + 4)));
    } else {
        const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
        if (T <= 8) {
            const dim3 grid((E + RS_E - 1) / RS_E, rp.n_parts, 1);
            MOE_LAUNCH("router_splitk", s,
                       launch_k(router_splitk_kernel<8>, grid, 256, 0, s, xb, Wg, parts, T, d, E));
        } else {
            const dim3 grid((E + RS_E - 1) / RS_E, rp.n_parts, (T + 63) / 64);
            MOE_LAUNCH("router_splitk", s,
                       launch_k(router_splitk_kernel<64>, grid, 256, 0, s, xb, Wg, parts, T, d, E));
        }
    }
    const int tk_blocks = (T + kTopkTok - 1) / kTopkTok;
    const size_t tk_smem = kTopkTok * E * sizeof(float);
#define MOE_TOPK(VPL)                                                                           \
    MOE_LAUNCH("topk_renorm", s,                                                                \
               launch_k(topk_renorm_kernel<VPL>, tk_blocks, 256, tk_smem, s, parts, rp.n_parts, \
                        rp.part_stride, rp.row_stride, bias, logits, T, E, k, c.n_group,        \
                        c.topk_group, idx, w, cand))
    if (E <= 64) MOE_TOPK(2);
    else if (E <= 256) MOE_TOPK(8);
    else MOE_TOPK(32);
#undef MOE_TOPK
    return MOE_OK;
}

moe_status ffn_impl(const moe_config& c, const void* x_perm, const int32_t* offsets,
                    const moe_expert_weights& R, const moe_expert_weights* S, const void* x,
                    const float* topk_w, const int32_t* perm_token, const int32_t* perm_slot,
                    float* y, int32_t* mtile, bool mtile_ready, int32_t* shared_tab,
                    __nv_bfloat16* h, __nv_bfloat16* hs, float* partial,
                    unsigned long long* counters, cudaStream_t s, void* fused_out = nullptr,
                    bool gather_a = false, bool merge_shared = false, int8_t* y_exp = nullptr) {
    // y_exp (moe_forward; bf16 weights, unsplit routed down projection): the routed rows
    // of y are written compactly (EPI_SCALE_H16: fp16 values at y, chunk exponents at
    // y_exp); the shared expert's rows stay fp32
    // merge_shared (moe_forward; bf16 weights, a shared expert, unsplit up projections,
    // offsets and mtile with E + 2 entries): the shared expert runs as group E of the
    // routed up projection (its H rows follow the routed ones), and its down projection
    // reads those rows through offsets[E .. E+1]
    // gather_a: x_perm is not materialised; the routed up projection reads row p of its A
    // from x[perm_token[p]] (bf16 weights only)
    // fused_out (top-1, no shared expert, unsplit down projection): the down projection
    // writes the layer output [T, d] directly (combine fused); y is not written
    // counters: kNumCounters tile counters; [kCntUp], [kCntDown] are already zero when
    // mtile_ready (the dispatch kernel that wrote the M-tile table zeroed them)
    const int T = c.T, E = c.E, d = c.d, k = c.top_k, F = c.F;
    const FfnPlan fp = ffn_plan(c);
    const long long Pmax = (long long)T * k;
    float* y_shared = y + Pmax * d;
    if (c.kind == MOE_EXPERT_LINEAR) {
        const long long n = Pmax * d;
        const int blocks = (int)std::max<long long>(1, std::min<long long>((n + 255) / 256, 65535));
        MOE_LAUNCH("linear_expert", s,
                   launch_k(linear_expert_kernel, blocks, 256, 0, s,
                       static_cast<const float*>(x_perm), offsets, E,
                       static_cast<const float*>(R.w1), R.b1, topk_w, perm_token, perm_slot, k, y,
                       d, Pmax));
        if (c.has_shared) {
            MOE_LAUNCH("single_group_table", s,
                       launch_k(single_group_table_kernel, 1, 32, 0, s, T, shared_tab, shared_tab + 2,
                                                                  nullptr, 0));
            const long long ns = (long long)T * d;
            const int sb = (int)std::max<long long>(1, std::min<long long>((ns + 255) / 256, 65535));
            MOE_LAUNCH("linear_expert", s,
                       launch_k(linear_expert_kernel, sb, 256, 0, s,
                           static_cast<const float*>(x), shared_tab, 1,
                           static_cast<const float*>(S->w1), S->b1, nullptr, nullptr, nullptr, k,
                           y_shared, d, T));
        }
        return MOE_OK;
    }
    if (!mtile_ready)
        MOE_LAUNCH("mtile_table", s,
                   launch_k(mtile_table_kernel, 1, 1024, 0, s, offsets, E, mtile, counters + kCntUp, 2));
    const int64_t N1 = n1_of(c);
    // INT8 / INT4 weights: per-row scales select the quantised-weight kernels
    const bool q8 = quant_w(c);
    const int wb = code_bits(c);
    const float* rs1 = q8 ? R.s1 : nullptr;
    const float* rs2 = q8 ? R.s2 : nullptr;
    const bool swap_r = q8t_routed(c), swap_s = q8t_shared(c);
    const bool ga = gather_a && !q8;
    const void* a_up = ga ? x : x_perm;
    const int32_t* a_idx = ga ? perm_token : nullptr;
    const ExpertTiles et = expert_tiles(c);
    // 128-row down projections run as CTA pairs sharing each B tile (GemmParams::pair)
    // when their groups' tile counts are mostly even: a group with an odd count leaves one
    // CTA of its last pair idle (DeepSeek-V3 shape at capacity 320, where many experts have
    // three tiles: 7.63 -> 7.9 ms; at capacity 256: 6.27 -> 6.13 ms). Even enough: at most
    // two tiles per expert (capacity <= 256 rows, two tiles expected), or six or more.
    const double rows_e = (double)T * k / E;
    const int32_t cap = capacity_of(c);
    const bool pair_down = et.down == 1 && rows_e >= kWideTileMinRows &&
                           ((cap > 0 && cap <= 2 * kMTile) || rows_e >= 6.0 * kMTile);
    const int sh_tiles = (T + kMTile - 1) / kMTile;
    const bool pair_sh = et.sh_down == 1 && sh_tiles >= 2 && (sh_tiles % 2 == 0 || sh_tiles >= 6);
    auto down_routed = [&](const float* row_scale, bool swap) -> moe_status {
        if (y_exp)
            return launch_gemm<EPI_SCALE_H16>(
                h, Pmax, F, R.w2, (int64_t)E * d, d, E, d, offsets, mtile, y, d, R.b2, topk_w,
                perm_token, perm_slot, k, s, nullptr, SplitPlan(), nullptr, counters + kCntDown,
                nullptr, nullptr, nullptr, 0, 0, nullptr, false, nullptr, nullptr, 0, nullptr,
                nullptr, wb, et.down, nullptr, 0, nullptr, 0, nullptr, -1, false, -1, y_exp,
                pair_down);
        return launch_gemm<EPI_SCALE_F32>(h, Pmax, F, R.w2, (int64_t)E * d, d, E, d, offsets,
                                          mtile, y, d, R.b2, topk_w, perm_token, perm_slot, k, s,
                                          nullptr, fp.down, partial, counters + kCntDown, nullptr,
                                          nullptr, nullptr, 0, 0, row_scale, swap, nullptr,
                                          nullptr, 0, nullptr, nullptr, wb, et.down, nullptr, 0,
                                          nullptr, 0, nullptr, -1, false, -1, nullptr, pair_down);
    };
    if (y_exp && (q8 || fp.down.S > 1 || fused_out)) return MOE_ERR_UNSUPPORTED;
    if (merge_shared) {
        if (!(c.has_shared && !q8 && fp.up.S == 1 && fp.sh_up.S == 1 && fp.sh_down.S == 1))
            return MOE_ERR_UNSUPPORTED;
        MOE_LAUNCH("append_group", s, launch_k(append_group_kernel, 1, 32, 0, s,
                                                const_cast<int32_t*>(offsets), mtile, E, T));
        const int mt = ga ? 1 : et.up;
        const char* nm = c.kind == MOE_EXPERT_SWIGLU ? "grouped_gemm_swiglu" : "grouped_gemm_gelu";
        if (c.kind == MOE_EXPERT_SWIGLU)
            MOE_TRY(launch_gemm<EPI_SWIGLU_BF16>(
                a_up, Pmax, d, R.w1, (int64_t)E * N1, (int)N1, E + 1, F, offsets, mtile, h, F, R.b1,
                nullptr, nullptr, nullptr, k, s, nm, SplitPlan(), nullptr, counters + kCntUp,
                nullptr, nullptr, nullptr, 0, 0, nullptr, false, nullptr, a_idx, d * 2, nullptr,
                nullptr, wb, mt, x, T, S->w1, N1, S->b1, E));
        else
            MOE_TRY(launch_gemm<EPI_GELU_BF16>(
                a_up, Pmax, d, R.w1, (int64_t)E * N1, (int)N1, E + 1, F, offsets, mtile, h, F, R.b1,
                nullptr, nullptr, nullptr, k, s, nm, SplitPlan(), nullptr, counters + kCntUp,
                nullptr, nullptr, nullptr, 0, 0, nullptr, false, nullptr, a_idx, d * 2, nullptr,
                nullptr, wb, mt, x, T, S->w1, N1, S->b1, E));
        MOE_TRY(down_routed(nullptr, false));
        MOE_LAUNCH("single_group_table", s,
                   launch_k(single_group_table_kernel, 1, 32, 0, s, T, shared_tab, shared_tab + 2,
                            counters + kCntSharedUp, 2));
        // rows [P, P + T) of H (offsets[E .. E+1]), written to the shared rows of y
        return launch_gemm<EPI_F32>(h, Pmax + T, F, S->w2, d, d, 1, d, offsets + E, shared_tab + 2,
                                    y_shared, d, S->b2, nullptr, nullptr, nullptr, k, s, nullptr,
                                    SplitPlan(), nullptr, counters + kCntSharedDown, nullptr,
                                    nullptr, nullptr, 0, 0, nullptr, false, nullptr, nullptr, 0,
                                    nullptr, nullptr, wb, et.sh_down, nullptr, 0, nullptr, 0,
                                    nullptr, -1, true, T, nullptr, pair_sh);
    }
    if (c.kind == MOE_EXPERT_SWIGLU)
        MOE_TRY(launch_gemm<EPI_SWIGLU_BF16>(a_up, Pmax, d, R.w1, (int64_t)E * N1, (int)N1, E, F,
                                             offsets, mtile, h, F, R.b1, nullptr, nullptr, nullptr,
                                             k, s, nullptr, fp.up, partial, counters + kCntUp,
                                             nullptr, nullptr, nullptr, 0, 0, rs1, swap_r, nullptr,
                                             a_idx, d * 2, nullptr, nullptr, wb, ga ? 1 : et.up));
    else
        MOE_TRY(launch_gemm<EPI_GELU_BF16>(a_up, Pmax, d, R.w1, (int64_t)E * N1, (int)N1, E, F,
                                           offsets, mtile, h, F, R.b1, nullptr, nullptr, nullptr, k,
                                           s, nullptr, fp.up, partial, counters + kCntUp, nullptr,
                                           nullptr, nullptr, 0, 0, rs1, swap_r, nullptr, a_idx,
                                           d * 2, nullptr, nullptr, wb, ga ? 1 : et.up));
    if (fused_out)
        MOE_TRY(launch_gemm<EPI_COMBINE1_BF16>(h, Pmax, F, R.w2, (int64_t)E * d, d, E, d, offsets,
                                               mtile, fused_out, d, R.b2, topk_w, perm_token,
                                               perm_slot, k, s, nullptr, SplitPlan(), nullptr,
                                               counters + kCntDown, c.add_residual ? x : nullptr,
                                               nullptr, nullptr, 0, 0, rs2));
    else
        MOE_TRY(down_routed(rs2, swap_r));
    if (c.has_shared) {
        MOE_LAUNCH("single_group_table", s,
                   launch_k(single_group_table_kernel, 1, 32, 0, s, T, shared_tab, shared_tab + 2,
                                                              counters + kCntSharedUp, 2));
        if (c.kind == MOE_EXPERT_SWIGLU)
            MOE_TRY(launch_gemm<EPI_SWIGLU_BF16>(x, T, d, S->w1, N1, (int)N1, 1, F, shared_tab,
                                                 shared_tab + 2, hs, F, S->b1, nullptr, nullptr,
                                                 nullptr, k, s, nullptr, fp.sh_up, partial,
                                                 counters + kCntSharedUp, nullptr, nullptr,
                                                 nullptr, 0, 0, q8 ? S->s1 : nullptr, swap_s,
                                           nullptr, nullptr, 0, nullptr, nullptr, wb, et.sh_up));
        else
            MOE_TRY(launch_gemm<EPI_GELU_BF16>(x, T, d, S->w1, N1, (int)N1, 1, F, shared_tab,
                                               shared_tab + 2, hs, F, S->b1, nullptr, nullptr,
                                               nullptr, k, s, nullptr, fp.sh_up, partial,
                                               counters + kCntSharedUp, nullptr, nullptr, nullptr,
                                               0, 0, q8 ? S->s1 : nullptr, swap_s,
                                           nullptr, nullptr, 0, nullptr, nullptr, wb, et.sh_up));
        MOE_TRY(launch_gemm<EPI_F32>(hs, T, F, S->w2, d, d, 1, d, shared_tab, shared_tab + 2,
                                     y_shared, d, S->b2, nullptr, nullptr, nullptr, k, s, nullptr,
                                     fp.sh_down, partial, counters + kCntSharedDown, nullptr,
                                     nullptr, nullptr, 0, 0, q8 ? S->s2 : nullptr, swap_s,
                                     nullptr, nullptr, 0, nullptr, nullptr, wb, et.sh_down, nullptr,
                                     0, nullptr, 0, nullptr, -1, false, -1, nullptr, pair_sh));
    }
    return MOE_OK;
}

moe_status combine_impl(const moe_config& c, const void* x, const float* y,
                        const int32_t* slot_dest, const float* topk_w, void* out, cudaStream_t s,
                        const int8_t* y_exp = nullptr) {
    // topk_w: read iff overflow == SHARED (the dropped slots' weights join the shared expert)
    // y_exp (bf16 layers): the routed rows of y are compact (see ffn_impl)
    const float* ovf_w = (c.overflow == MOE_OVERFLOW_SHARED && c.has_shared) ? topk_w : nullptr;
    const int T = c.T, d = c.d, k = c.top_k;
    const long long Pmax = (long long)T * k;
    const float* ysh = c.has_shared ? y + Pmax * d : nullptr;
    // tasks of cpt 256-column chunks: whole tokens unless that leaves fewer than ~4096 tasks
    const int chunks = (d + 255) / 256;
    const int cpt = (int)std::max<long long>(
        1, std::min<long long>(chunks, (long long)chunks * T / 4096));
    const long long work = (long long)T * ((chunks + cpt - 1) / cpt);
    const int blocks = (int)std::max<long long>(1, std::min<long long>((work + 7) / 8,
                                                                       (long long)num_sms() * 8));
    if (y_exp && c.act_dtype == MOE_F32) return MOE_ERR_UNSUPPORTED;
    if (c.act_dtype == MOE_F32)
        MOE_LAUNCH("combine_f32", s,
                   launch_k(combine_kernel<float>, blocks, 256, 0, s,
                       static_cast<const float*>(x), y, slot_dest, ysh, ovf_w,
                       static_cast<float*>(out), T, d, k, c.add_residual, cpt));
    else if (y_exp) {
        // one block of CH16_WARPS warps per SM, tasks of 512-column chunks (see
        // combine_h16_kernel): whole tokens unless that leaves fewer than ~4096 tasks
        const int ch16 = (d + CH16_COLS - 1) / CH16_COLS;
        const int cpt16 = (int)std::max<long long>(
            1, std::min<long long>(ch16, (long long)ch16 * T / 4096));
        static std::once_flag c16_once[64];
        static cudaError_t c16_err[64];
        const int dev = current_device();
        if (dev >= 0 && dev < 64) {
            std::call_once(c16_once[dev], [&] {
                c16_err[dev] = cudaFuncSetAttribute(combine_h16_kernel,
                                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                    ch16_smem_bytes());
            });
            if (c16_err[dev] != cudaSuccess) return MOE_ERR_CUDA;
        }
        MOE_LAUNCH("combine_h16", s,
                   launch_k(combine_h16_kernel, num_sms(), CH16_WARPS * 32, ch16_smem_bytes(), s,
                       static_cast<const __nv_bfloat16*>(x), reinterpret_cast<const __half*>(y),
                       y_exp, compact_exp_ld(d), slot_dest, ysh, ovf_w,
                       static_cast<__nv_bfloat16*>(out), T, d, k, c.add_residual, cpt16));
    } else
        MOE_LAUNCH("combine_bf16", s,
                   launch_k(combine_kernel<__nv_bfloat16>, blocks, 256, 0, s,
                       static_cast<const __nv_bfloat16*>(x), y, slot_dest, ysh, ovf_w,
                       static_cast<__nv_bfloat16*>(out), T, d, k, c.add_residual, cpt));
    return MOE_OK;
}

moe_status check_weights(const moe_config& c, const moe_expert_weights* W) {
    if (!W || !W->w1) return MOE_ERR_INVALID_ARG;
    if (c.kind != MOE_EXPERT_LINEAR && !W->w2) return MOE_ERR_INVALID_ARG;
    if (quant_w(c) && (!W->s1 || !W->s2)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(W->w1) || !aligned16(W->w2) || !aligned16(W->b1) || !aligned16(W->b2) ||
        !aligned16(W->s1) || !aligned16(W->s2))
        return MOE_ERR_MISALIGNED;
    return MOE_OK;
}

}  // namespace

// =====================================================================================
// exported C ABI
// =====================================================================================
extern "C" {

size_t moe_workspace_size(const moe_config* cfg) {
    if (check_cfg(cfg) != MOE_OK) return 0;
    return ws_layout(*cfg).total;
}

int64_t moe_max_rows(const moe_config* cfg) {
    if (check_cfg(cfg) != MOE_OK) return -1;
    return (int64_t)cfg->T * cfg->top_k;
}

int32_t moe_capacity(const moe_config* cfg) {
    if (check_cfg(cfg) != MOE_OK) return -1;
    return capacity_of(*cfg);
}

moe_status moe_route(const moe_config* cfg, const void* x, const float* W_gate,
                     const float* gate_bias, float* logits, int32_t* topk_idx, float* topk_w,
                     void* ws, cudaStream_t stream) {
    MOE_TRY(check_cfg(cfg));
    const moe_config& c = *cfg;
    if (c.T == 0) return MOE_OK;
    if (!x || !W_gate || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
    if (!ws) return MOE_ERR_WORKSPACE;
    if (!aligned16(x) || !aligned16(W_gate) || !aligned16(gate_bias) || !aligned16(logits) ||
        !aligned16(topk_idx) || !aligned16(topk_w) || !aligned16(ws))
        return MOE_ERR_MISALIGNED;
    const WsLayout L = ws_layout(c);
    return route_impl(c, x, W_gate, gate_bias, logits, topk_idx, topk_w, at<void>(ws, L.logits),
                      at<int32_t>(ws, L.cand), stream);
}

moe_status moe_dispatch(const moe_config* cfg, const int32_t* topk_idx, const void* x,
                        int32_t* load, int32_t* counts, int32_t* offsets, int32_t* perm_token,
                        int32_t* perm_slot, int32_t* slot_dest, void* x_perm, void* ws,
                        cudaStream_t stream) {
    MOE_TRY(check_cfg(cfg));
    const moe_config& c = *cfg;
    if (c.T == 0) return MOE_OK;
    if (!topk_idx || !load || !counts || !offsets || !perm_token || !perm_slot || !slot_dest)
        return MOE_ERR_INVALID_ARG;
    if (x_perm && !x) return MOE_ERR_INVALID_ARG;
    if (!ws) return MOE_ERR_WORKSPACE;
    const void* ptrs[] = {topk_idx, x, load, counts, offsets, perm_token, perm_slot, slot_dest,
                          x_perm, ws};
    for (const void* p : ptrs)
        if (!aligned16(p)) return MOE_ERR_MISALIGNED;
    const WsLayout L = ws_layout(c);
    return dispatch_impl(c, topk_idx, x, load, counts, offsets, perm_token, perm_slot, slot_dest,
                         x_perm, at<int32_t>(ws, L.blockcnt), at<int32_t>(ws, L.blockoff), nullptr,
                         nullptr, stream, at<int32_t>(ws, L.cand), at<int32_t>(ws, L.prop),
                         at<int32_t>(ws, L.cnt0));
}

moe_status moe_expert_ffn(const moe_config* cfg, const void* x_perm, const int32_t* offsets,
                          const moe_expert_weights* routed, const moe_expert_weights* shared,
                          const void* x, const float* topk_w, const int32_t* perm_token,
                          const int32_t* perm_slot, float* y, void* ws, cudaStream_t stream) {
    MOE_TRY(check_cfg(cfg));
    const moe_config& c = *cfg;
    if (c.T == 0) return MOE_OK;
    if (!x_perm || !offsets || !topk_w || !perm_token || !perm_slot || !y) return MOE_ERR_INVALID_ARG;
    MOE_TRY(check_weights(c, routed));
    if (c.has_shared) {
        if (!x) return MOE_ERR_INVALID_ARG;
        MOE_TRY(check_weights(c, shared));
    }
    if (!ws) return MOE_ERR_WORKSPACE;
    const void* ptrs[] = {x_perm, offsets, x, topk_w, perm_token, perm_slot, y, ws};
    for (const void* p : ptrs)
        if (!aligned16(p)) return MOE_ERR_MISALIGNED;
    const WsLayout L = ws_layout(c);
    return ffn_impl(c, x_perm, offsets, *routed, shared, x, topk_w, perm_token, perm_slot, y,
                    at<int32_t>(ws, L.mtile), false, at<int32_t>(ws, L.shared_tab),
                    at<__nv_bfloat16>(ws, L.h), at<__nv_bfloat16>(ws, L.hs),
                    at<float>(ws, L.partial), at<unsigned long long>(ws, L.counters), stream);
}

moe_status moe_combine(const moe_config* cfg, const void* x, const float* y,
                       const float* topk_w, const int32_t* slot_dest, void* out,
                       cudaStream_t stream) {
    MOE_TRY(check_cfg(cfg));
    const moe_config& c = *cfg;
    if (c.T == 0) return MOE_OK;
    if (!y || !slot_dest || !out || (c.add_residual && !x)) return MOE_ERR_INVALID_ARG;
    if (c.overflow == MOE_OVERFLOW_SHARED && !topk_w) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y) || !aligned16(slot_dest) || !aligned16(topk_w) ||
        !aligned16(out))
        return MOE_ERR_MISALIGNED;
    return combine_impl(c, x, y, slot_dest, topk_w, out, stream);
}

moe_status moe_forward(const moe_config* cfg, const void* x, const float* W_gate,
                       const float* gate_bias, const moe_expert_weights* routed,
                       const moe_expert_weights* shared, void* out, int32_t* topk_idx,
                       float* topk_w, int32_t* load, void* ws, size_t ws_bytes,
                       cudaStream_t stream) {
    MOE_TRY(check_cfg(cfg));
    const moe_config& c = *cfg;
    if (c.T == 0) return MOE_OK;
    if (!x || !W_gate || !out) return MOE_ERR_INVALID_ARG;
    MOE_TRY(check_weights(c, routed));
    if (c.has_shared) MOE_TRY(check_weights(c, shared));
    const WsLayout L = ws_layout(c);
    if (!ws || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    const void* ptrs[] = {x, W_gate, gate_bias, out, topk_idx, topk_w, load, ws};
    for (const void* p : ptrs)
        if (!aligned16(p)) return MOE_ERR_MISALIGNED;
    int32_t* idx = topk_idx ? topk_idx : at<int32_t>(ws, L.idx);
    float* w = topk_w ? topk_w : at<float>(ws, L.w);
    int32_t* ld = load ? load : at<int32_t>(ws, L.load);
    int32_t* offsets = at<int32_t>(ws, L.offsets);
    int32_t* perm_token = at<int32_t>(ws, L.perm_token);
    int32_t* perm_slot = at<int32_t>(ws, L.perm_slot);
    int32_t* slot_dest = at<int32_t>(ws, L.slot_dest);
    void* x_perm = at<void>(ws, L.x_perm);
    // bf16 experts with k >= 4 and 128-row tiles: the up projection gathers its rows of x
    // itself (no x_perm copy, which is k times the size of x). With fewer slots per token
    // the copy is cheaper than the slower A loads of the gathering kernel (16-byte cp.async
    // instead of TMA), and 256-row tiles read a materialised x_perm (see expert_tiles).
    const bool gather_a = is_bf16_kind(c) && !quant_w(c) && !q8t_routed(c) && c.top_k >= 4 &&
                          expert_tiles(c).up == 1;
    float* y = at<float>(ws, L.y);
    int32_t* mtile = at<int32_t>(ws, L.mtile);
    // Top-1 layers without a shared expert write the output from the down projection.
    const bool fuse1 = is_bf16_kind(c) && c.top_k == 1 && !c.has_shared && !q8t_routed(c) &&
                       ffn_plan(c).down.S == 1;
    // The fused router top-k also counts the dispatch histogram when the dispatch runs as
    // separate kernels (one kernel fewer).
    const RouterPlan rp = router_plan(c);
    const bool hist_by_router = rp.path == 2 && router_fused_topk(c, rp.Ep) && !dispatch_one_cta(c);
    MOE_TRY(route_impl(c, x, W_gate, gate_bias, nullptr, idx, w, at<void>(ws, L.logits),
                       at<int32_t>(ws, L.cand), stream,
                       hist_by_router ? at<int32_t>(ws, L.blockcnt) : nullptr));
    MOE_TRY(dispatch_impl(c, idx, x, ld, at<int32_t>(ws, L.counts), offsets, perm_token, perm_slot,
                          slot_dest, gather_a ? nullptr : x_perm, at<int32_t>(ws, L.blockcnt),
                          at<int32_t>(ws, L.blockoff), mtile,
                          at<unsigned long long>(ws, L.counters), stream, at<int32_t>(ws, L.cand),
                          at<int32_t>(ws, L.prop), at<int32_t>(ws, L.cnt0),
                          fuse1 ? DroppedRows{static_cast<const uint8_t*>(x),
                                              static_cast<uint8_t*>(out), c.d * 2, c.add_residual}
                                : DroppedRows{},
                          hist_by_router));
    // The shared expert as group E of the routed up projection (one launch, one tail).
    const FfnPlan fpl = ffn_plan(c);
    const bool merge_shared = c.has_shared && is_bf16_kind(c) && !quant_w(c) && !q8t_routed(c) &&
                              fpl.up.S == 1 && fpl.sh_up.S == 1 && fpl.sh_down.S == 1;
    // Compact routed rows of y (fp16 + a power-of-two scale per 32 columns, inside the fp32
    // region: values in its first Pmax * d * 2 bytes, then Pmax rows of compact_exp_ld(d)
    // exponent bytes; the shared rows keep their fp32 place after the routed ones).
    // k >= 4 only: with fewer slots per token the compact combine's copy pipeline holds
    // too few rows per step to beat the fp32 combine (Mixtral-shaped top-2 layer: 0.061 ms
    // against 0.045 ms), and the bytes saved are small.
    const bool compact_y = !c.y_fp32 && is_bf16_kind(c) && !quant_w(c) && !q8t_routed(c) &&
                           !fuse1 && fpl.down.S == 1 && c.top_k >= 4;
    int8_t* y_exp = compact_y ? reinterpret_cast<int8_t*>(y) + (long long)c.T * c.top_k * c.d * 2
                              : nullptr;
    MOE_TRY(ffn_impl(c, x_perm, offsets, *routed, shared, x, w, perm_token, perm_slot, y, mtile,
                     true, at<int32_t>(ws, L.shared_tab), at<__nv_bfloat16>(ws, L.h),
                     at<__nv_bfloat16>(ws, L.hs), at<float>(ws, L.partial),
                     at<unsigned long long>(ws, L.counters), stream, fuse1 ? out : nullptr,
                     gather_a, merge_shared, y_exp));
    if (fuse1) return MOE_OK;   // dropped tokens were written by the dispatch
    return combine_impl(c, x, y, slot_dest, w, out, stream, y_exp);
}

// M-tile table ((G+1) int32), then the tile counter (8-byte aligned).
size_t gg_counter_offset(int32_t G) { return ((size_t)(G + 1) * 4 + 7) & ~size_t(7); }

size_t moe_grouped_gemm_ws_size(int32_t G) {
    if (G < 1 || G > 1024) return 0;
    return gg_counter_offset(G) + 8;
}

moe_status moe_grouped_gemm(const void* A, int64_t a_rows, const void* B, int32_t G, int32_t N,
                            int32_t K, const int32_t* row_offsets, float* D, void* ws,
                            cudaStream_t stream) {
    if (!A || !B || !row_offsets || !D) return MOE_ERR_INVALID_ARG;
    if (G < 1 || G > 1024 || N < 64 || N % 64 != 0 || K < 64 || K % 64 != 0 || a_rows < 0 ||
        a_rows >= (1ll << 31) || (int64_t)G * N >= (1ll << 31))
        return MOE_ERR_INVALID_ARG;
    if (!ws) return MOE_ERR_WORKSPACE;
    if (!aligned16(A) || !aligned16(B) || !aligned16(row_offsets) || !aligned16(D) || !aligned16(ws))
        return MOE_ERR_MISALIGNED;
    if (a_rows == 0) return MOE_OK;
    int32_t* mtile = static_cast<int32_t*>(ws);
    unsigned long long* counter =
        reinterpret_cast<unsigned long long*>(static_cast<char*>(ws) + gg_counter_offset(G));
    MOE_LAUNCH("mtile_table", stream,
               launch_k(mtile_table_kernel, 1, 1024, 0, stream, row_offsets, G, mtile, counter, 1));
    return launch_gemm<EPI_F32>(A, a_rows, K, B, (int64_t)G * N, N, G, N, row_offsets, mtile, D, N,
                                nullptr, nullptr, nullptr, nullptr, 1, stream, nullptr,
                                SplitPlan(), nullptr, counter);
}

moe_status moe_quantize_i8(const void* w, int64_t rows, int32_t cols, int8_t* q, float* scale,
                           cudaStream_t stream) {
    if (!w || !q || !scale || rows < 0 || cols < 8 || cols % 8 != 0) return MOE_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(q) || !aligned16(scale)) return MOE_ERR_MISALIGNED;
    if (rows == 0) return MOE_OK;
    const int blocks = (int)std::max<long long>(
        1, std::min<long long>((rows + 7) / 8, (long long)num_sms() * 16));
    MOE_LAUNCH("quantize_i8", stream,
               launch_k(quantize_rows_i8_kernel, blocks, 256, 0, stream,
                        static_cast<const __nv_bfloat16*>(w), (long long)rows, (int)cols, q, scale));
    return MOE_OK;
}

moe_status moe_quantize_i4(const void* w, int64_t rows, int32_t cols, uint8_t* q, float* scale,
                           cudaStream_t stream) {
    if (!w || !q || !scale || rows < 0 || cols < 32 || cols % 32 != 0) return MOE_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(q) || !aligned16(scale)) return MOE_ERR_MISALIGNED;
    if (rows == 0) return MOE_OK;
    const int blocks = (int)std::max<long long>(
        1, std::min<long long>((rows + 7) / 8, (long long)num_sms() * 16));
    MOE_LAUNCH("quantize_i4", stream,
               launch_k(quantize_rows_i4_kernel, blocks, 256, 0, stream,
                        static_cast<const __nv_bfloat16*>(w), (long long)rows, (int)cols, q, scale));
    return MOE_OK;
}

moe_status moe_load_report(const int32_t* load_host, int32_t E, int32_t D, int32_t* assign,
                           int64_t* dev_load, double* imbalance) {
    if (!load_host || !assign || !dev_load || !imbalance || E < 1 || D < 1)
        return MOE_ERR_INVALID_ARG;
    int32_t mx = load_host[0], mn = load_host[0];
    for (int e = 1; e < E; ++e) {
        mx = std::max(mx, load_host[e]);
        mn = std::min(mn, load_host[e]);
    }
    *imbalance = (double)mx / ((double)mn + 1e-6);
    std::vector<int> order(E);
    std::iota(order.begin(), order.end(), 0);
    std::stable_sort(order.begin(), order.end(),
                     [&](int a, int b) { return load_host[a] > load_host[b]; });
    std::fill(dev_load, dev_load + D, 0);
    for (int e : order) {
        const int dv = (int)(std::min_element(dev_load, dev_load + D) - dev_load);
        assign[e] = dv;
        dev_load[dv] += load_host[e];
    }
    return MOE_OK;
}

moe_status moe_last_device_status(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_dev_error, sizeof(v)) != cudaSuccess) return MOE_ERR_CUDA;
    if (v) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_dev_error, &zero, sizeof(zero)) != cudaSuccess) return MOE_ERR_CUDA;
    }
    if (v & DEVERR_TIMEOUT) return MOE_ERR_TIMEOUT;
    if (v & DEVERR_INDEX) return MOE_ERR_DEVICE_INDEX;
    return MOE_OK;
}

const char* moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
        case MOE_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case MOE_ERR_WORKSPACE: return "workspace missing or too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_TIMEOUT: return "device-side wait timed out";
        case MOE_ERR_DEVICE_INDEX: return "expert id out of range in device data";
    }
    return "unknown status";
}

moe_status moe_profile_begin(void) {
    std::lock_guard<std::mutex> lk(g_prof.mu);
    g_prof.recs.clear();
    g_prof.used = 0;
    g_prof.on = true;
    return MOE_OK;
}

int32_t moe_profile_end(moe_kernel_stat* stats, int32_t max_stats) {
    std::lock_guard<std::mutex> lk(g_prof.mu);
    g_prof.on = false;
    std::vector<moe_kernel_stat> agg;
    for (const ProfRec& r : g_prof.recs) {
        if (cudaEventSynchronize(r.b) != cudaSuccess) return -1;
        float ms = 0.0f;
        if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) return -1;
        auto it = std::find_if(agg.begin(), agg.end(),
                               [&](const moe_kernel_stat& s) { return std::strcmp(s.name, r.name) == 0; });
        if (it == agg.end()) agg.push_back({r.name, 1, (double)ms});
        else {
            it->launches += 1;
            it->total_ms += ms;
        }
    }
    g_prof.recs.clear();
    g_prof.used = 0;
    if (stats)
        for (int i = 0; i < (int)agg.size() && i < max_stats; ++i) stats[i] = agg[i];
    return (int32_t)agg.size();
}

uint64_t moe_kernel_launch_count(void) { return g_launches.load(); }

moe_status moe_selftest_wait_timeout(int64_t budget_cycles, cudaStream_t stream) {
    if (budget_cycles < 0 || budget_cycles > kWaitBudgetCycles) return MOE_ERR_INVALID_ARG;
    MOE_LAUNCH("selftest_wait", stream, launch_k(selftest_wait_kernel, 1, 32, 0, stream, budget_cycles));
    return MOE_OK;
}

}  // extern "C"

// =====================================================================================
// moe_dispatch_noalloc: moe_dispatch with its scratch in a fixed static device array
// =====================================================================================
// The dispatch kernels need two tables of ceil(T/256) x E ints (per-chunk counts and
// per-chunk rank bases). Here they live in this file-scope array instead of a caller
// workspace. Every GPU that loads the library holds the array until the process
// exits. Every word the kernels read is written earlier in the same call, so nothing
// has to be cleared between calls.
namespace {
constexpr long long kNoallocScratchInts = 1ll << 18;   // 1 MiB
}
static __device__ __align__(256) int32_t g_noalloc_scratch[kNoallocScratchInts];

namespace {
std::mutex g_noalloc_mu;
int32_t* g_noalloc_ptr[64] = {};

// Device address of g_noalloc_scratch on the current device, looked up once per
// device with that device current (host code cannot use the symbol itself as a
// device pointer).
moe_status noalloc_scratch(int32_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
        g_noalloc_ptr[dev] = static_cast<int32_t*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return MOE_OK;
}
}  // namespace

extern "C" moe_status moe_dispatch_noalloc(const moe_config* cfg, const int32_t* topk_idx,
                                           const void* x, int32_t* load, int32_t* counts,
                                           int32_t* offsets, int32_t* perm_token,
                                           int32_t* perm_slot, int32_t* slot_dest, void* x_perm,
                                           cudaStream_t stream) {
    MOE_TRY(check_cfg(cfg));
    const moe_config& c = *cfg;
    if (c.overflow == MOE_OVERFLOW_REROUTE) return MOE_ERR_UNSUPPORTED;   // needs moe_route's ws
    if (c.T == 0) return MOE_OK;
    if (!topk_idx || !load || !counts || !offsets || !perm_token || !perm_slot || !slot_dest)
        return MOE_ERR_INVALID_ARG;
    if (x_perm && !x) return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {topk_idx, x, load, counts, offsets, perm_token, perm_slot, slot_dest,
                          x_perm};
    for (const void* p : ptrs)
        if (!aligned16(p)) return MOE_ERR_MISALIGNED;
    const long long nb = ((long long)c.T + kDispTok - 1) / kDispTok;
    if (2 * nb * (long long)c.E > kNoallocScratchInts) return MOE_ERR_WORKSPACE;
    int32_t* scratch = nullptr;
    MOE_TRY(noalloc_scratch(&scratch));
    return dispatch_impl(c, topk_idx, x, load, counts, offsets, perm_token, perm_slot, slot_dest,
                         x_perm, scratch, scratch + nb * c.E, nullptr, nullptr, stream);
}
