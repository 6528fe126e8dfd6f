// Dispatch: per-expert histogram -> prefix sums with capacity -> stable ranks ->
// permutation into expert-contiguous rows -> row gather.
// ["MoE 并行" 流程说明 (Token Dispatch groups tokens by expert) and Capacity Factor
//  (overflow tokens take the residual path); adv12 3.2 (bincount of the routing)
//  and Q2 (capacity 20: load 38 keeps 20, overflows 18).]
//
// The flattened assignment list s = t*k + j is cut into chunks of kDispTok tokens,
// one CTA each. Ranks are stable in token order: inside a CTA every warp owns a
// contiguous run of assignments, ranks inside a warp come from __match_any_sync
// groups, and per-(warp, expert) running counters are prefix-summed across warps
// and across CTAs. Nothing depends on the order in which atomics land, so every
// output is deterministic.
#pragma once
#include "common.cuh"

namespace moe {

constexpr int kDispTok = 256;    // tokens per dispatch chunk (one CTA)

// Top-1 layers whose combine runs in the down projection's epilogue: the dispatch writes
// the output row of every dropped token itself, as x (with the residual) or 0, bit for bit
// what the combine writes for a token without kept slots ["MoE 并行" Capacity Factor:
// overflow takes the residual path]. out == nullptr: nothing to write.
struct DroppedRows {
    const uint8_t* x;
    uint8_t* out;
    int row_bytes;   // multiple of 16
    int add_residual;
};

// Slots i = base + lane (k = 1: slot i is token i) whose bit is set in `dropped`: the
// warp copies each row in 16-byte vectors.
__device__ __forceinline__ void write_dropped_rows(const DroppedRows& dr, unsigned dropped,
                                                   long long base, int lane) {
    const int nvec = dr.row_bytes / 16;
    while (dropped) {
        const int l = __ffs(dropped) - 1;
        dropped &= dropped - 1;
        const long long t = base + l;
        uint4* dst = reinterpret_cast<uint4*>(dr.out + t * dr.row_bytes);
        const uint4* src = reinterpret_cast<const uint4*>(dr.x + t * dr.row_bytes);
        for (int c = lane; c < nvec; c += 32)
            dst[c] = dr.add_residual ? src[c] : make_uint4(0u, 0u, 0u, 0u);
    }
}
constexpr int kDispWarps = 8;
constexpr int kMTile = 128;      // rows per tensor-core M tile

// ---- warp-private counts of a run of expert ids (no atomics) --------------------------
// The warp's lanes read 32 ids at a time; lanes holding the same id form one
// __match_any_sync group, whose lowest lane adds the group's size to the warp's own
// counter row `my` [E] in shared memory. Only one lane of a warp writes a counter at a
// time, so no update can be lost and the result does not depend on any ordering.
// Ids outside [0, E) are skipped (and reported when `report`; re-routing proposals use
// -1 for "none" and are counted with report = false).
__device__ __forceinline__ void warp_count_ids(const int* __restrict__ idx, long long wbeg,
                                               long long wend, int E, int* my, bool report) {
    const int lane = threadIdx.x & 31;
    const unsigned lt_mask = (1u << lane) - 1u;
    for (long long base = wbeg; base < wend; base += 32) {
        const long long i = base + lane;
        int e = (i < wend) ? idx[i] : -1;
        if (i < wend && (e < 0 || e >= E)) {
            if (report) raise_error(DEVERR_INDEX);
            e = -1;
        }
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && (peers & lt_mask) == 0) my[e] += __popc(peers);
        __syncwarp();
    }
}

// ---- histogram: blockcnt[b][e] = assignments of chunk b routed to e ------------------
// Warp w counts a contiguous run of the chunk's assignments into its own row of
// shared memory (warp_count_ids); the rows are then summed per expert. No atomics.
__global__ void __launch_bounds__(256) dispatch_hist_kernel(const int* __restrict__ idx, int T,
                                                            int k, int E,
                                                            int* __restrict__ blockcnt) {
    pdl_entry();
    extern __shared__ int wcnt[];   // [kDispWarps][E]
    const int wid = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kDispWarps * E; i += blockDim.x) wcnt[i] = 0;
    __syncthreads();
    const long long beg = (long long)blockIdx.x * kDispTok * k;
    const long long end = min((long long)(blockIdx.x + 1) * kDispTok, (long long)T) * k;
    const long long seg = ((end - beg + kDispWarps - 1) / kDispWarps + 31) / 32 * 32;
    const long long wbeg = beg + wid * seg;
    warp_count_ids(idx, wbeg, min(wbeg + seg, end), E, wcnt + wid * E, true);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int c = 0;
        for (int w = 0; w < kDispWarps; ++w) c += wcnt[w * E + e];
        blockcnt[(long long)blockIdx.x * E + e] = c;
    }
}

// ---- block-wide exclusive scan of one int per thread (blockDim.x == 1024) -------------
__device__ __forceinline__ int block_excl_scan_1024(int v, int* s_warp /*[32]*/, int& total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) s_warp[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int s = s_warp[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, off);
            if (lane >= off) s += y;
        }
        s_warp[lane] = s;   // inclusive over warps
    }
    __syncthreads();
    total = s_warp[31];
    const int warp_base = wid ? s_warp[wid - 1] : 0;
    const int r = warp_base + x - v;
    __syncthreads();
    return r;
}

// M-tile table from the per-group row counts (one group per thread of a 1024-thread
// CTA): tables[0..G] = exclusive scan of ceil(rows/128). Every thread must call it (it
// contains barriers); tables may be null.
__device__ __forceinline__ void write_tile_tables(int rows, int g, int G, int* s_warp,
                                                  int* __restrict__ tables) {
    int tot;
    const int off = block_excl_scan_1024((rows + kMTile - 1) / kMTile, s_warp, tot);
    if (tables) {
        if (g < G) tables[g] = off;
        if (g == 0) tables[G] = tot;
    }
}

// ---- one CTA: load, capacity, offsets, per-chunk rank bases, M-tile table ----------
// blockoff[b][e] = assignments of e in chunks before b (rank base of chunk b).
// mtile_offsets[e] = exclusive prefix sum over experts of ceil(counts/128).
__global__ void __launch_bounds__(1024) dispatch_scan_kernel(
    const int* __restrict__ blockcnt, int nb, int E, int cap, int* __restrict__ blockoff,
    int* __restrict__ load, int* __restrict__ counts, int* __restrict__ offsets,
    int* __restrict__ mtile_offsets, unsigned long long* __restrict__ counters, int n_counters) {
    pdl_entry();
    __shared__ int s_warp[32];
    const int e = threadIdx.x;
    if (counters && e < n_counters) counters[e] = 0ull;
    int kept = 0;
    if (e < E) {
        int run = 0;
        for (int b = 0; b < nb; ++b) {
            const long long i = (long long)b * E + e;
            const int c = blockcnt[i];
            blockoff[i] = run;
            run += c;
        }
        load[e] = run;
        kept = min(run, cap);
        counts[e] = kept;
    }
    int total;
    const int off = block_excl_scan_1024(kept, s_warp, total);
    if (e < E) offsets[e] = off;
    if (e == 0) offsets[E] = total;
    write_tile_tables(kept, e, E, s_warp, mtile_offsets);
}

// ---- stable rank + scatter of the kept assignments ------------------------------------
// MODE kRankScatter: rank the ids of `idx` and scatter the kept ones (rank < cap).
// Re-routing ["MoE 并行" 推理时的负载均衡: an over-limit token goes to the next expert]:
// MODE kRankStatus ranks the original ids and only records slot_dest[i] = round-0 rank
// (kept), -1 (dropped) or -2 (invalid id, skipped as in the plain dispatch); MODE kRankReroute ranks the proposals `idx` = prop (the
// dropped slots' next-ranked experts, -1 for none) and scatters every slot: a round-0
// row of expert e at offsets[e] + its round-0 rank, an accepted proposal (rank <
// cap - cnt0[e]) after the cnt0[e] round-0 rows of its new expert.
enum { kRankScatter = 0, kRankStatus = 1, kRankReroute = 2 };

template <int MODE>
__global__ void __launch_bounds__(256) dispatch_rank_kernel(
    const int* __restrict__ idx, int T, int k, int E, int cap, const int* __restrict__ blockoff,
    const int* __restrict__ offsets, int* __restrict__ perm_token, int* __restrict__ perm_slot,
    int* __restrict__ slot_dest, const int* __restrict__ orig_idx, const int* __restrict__ cnt0,
    DroppedRows dr) {
    pdl_entry();
    extern __shared__ int wcnt[];   // [kDispWarps][E] running counters
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kDispWarps * E; i += blockDim.x) wcnt[i] = 0;
    __syncthreads();
    const long long beg = (long long)blockIdx.x * kDispTok * k;
    const long long end = min((long long)(blockIdx.x + 1) * kDispTok, (long long)T) * k;
    const long long n = end - beg;
    const long long seg = ((n + kDispWarps - 1) / kDispWarps + 31) / 32 * 32;
    const long long wbeg = beg + wid * seg;
    const long long wend = min(wbeg + seg, end);
    int* my = wcnt + wid * E;
    const unsigned lt_mask = (1u << lane) - 1u;
    // pass 1: per-warp totals
    for (long long base = wbeg; base < wend; base += 32) {
        const long long i = base + lane;
        int e = (i < wend) ? idx[i] : -1;
        if (e >= E) e = -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && (peers & lt_mask) == 0) my[e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    // pass 2: exclusive scan over warps, seeded with the chunk's rank base
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = blockoff[(long long)blockIdx.x * E + e];
        for (int w = 0; w < kDispWarps; ++w) {
            const int c = wcnt[w * E + e];
            wcnt[w * E + e] = run;
            run += c;
        }
    }
    __syncthreads();
    // pass 3: ranks and scatter
    for (long long base = wbeg; base < wend; base += 32) {
        const long long i = base + lane;
        bool dropped = false;
        int e = (i < wend) ? idx[i] : -1;
        if (e >= E) e = -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        int rank = 0;
        if (e >= 0) rank = my[e] + __popc(peers & lt_mask);
        __syncwarp();
        if (e >= 0 && (peers & lt_mask) == 0) my[e] += __popc(peers);
        __syncwarp();
        if (i < wend) {
            if constexpr (MODE == kRankStatus) {
                slot_dest[i] = (e >= 0) ? (rank < cap ? rank : -1) : -2;   // -2: invalid id
            } else {
                int pos = -1;
                if constexpr (MODE == kRankScatter) {
                    if (e >= 0 && rank < cap) pos = offsets[e] + rank;
                } else {
                    const int r0 = slot_dest[i];
                    if (r0 >= 0) pos = offsets[orig_idx[i]] + r0;
                    else if (e >= 0 && rank < cap - cnt0[e]) pos = offsets[e] + cnt0[e] + rank;
                }
                if (pos >= 0) {
                    perm_token[pos] = (int)(i / k);
                    perm_slot[pos] = (int)(i % k);
                }
                slot_dest[i] = pos;
                if (dr.out) dropped = pos < 0;
            }
        }
        if constexpr (MODE != kRankStatus) {
            if (dr.out) write_dropped_rows(dr, __ballot_sync(0xffffffffu, dropped), base, lane);
        }
    }
}

// ---- re-routing: proposals of the dropped slots and their per-chunk histogram ----------
// slot_dest holds the round-0 status (rank, -1 dropped, -2 invalid). Token t's dropped
// slots, in slot
// order, take cand[t][0], cand[t][1], ... (its experts ranked k, k+1, ...; -1 = none):
// prop[t*k + j] = that expert, -1 for kept slots. blockcnt[b][e] = proposals of chunk b
// to expert e.
__global__ void __launch_bounds__(256) reroute_propose_kernel(const int* __restrict__ slot_dest,
                                                              const int* __restrict__ cand, int T,
                                                              int k, int E, int* __restrict__ prop,
                                                              int* __restrict__ blockcnt) {
    pdl_entry();
    extern __shared__ int wcnt[];   // [kDispWarps][E]
    const int wid = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kDispWarps * E; i += blockDim.x) wcnt[i] = 0;
    // pass 1: one thread per token hands its dropped slots their proposals
    const int t_end = min((blockIdx.x + 1) * kDispTok, T);
    for (int t = blockIdx.x * kDispTok + threadIdx.x; t < t_end; t += blockDim.x) {
        int m = 0;
        for (int j = 0; j < k; ++j) {
            const long long i = (long long)t * k + j;
            int e = -1;
            if (slot_dest[i] == -1) {
                e = cand[(long long)t * k + m];
                ++m;
                if (e >= E) {
                    raise_error(DEVERR_INDEX);
                    e = -1;
                }
            }
            prop[i] = e < 0 ? -1 : e;
        }
    }
    __syncthreads();   // the chunk's proposals are written (and visible to this CTA)
    // pass 2: warp-private counts of the chunk's proposals, summed per expert
    const long long beg = (long long)blockIdx.x * kDispTok * k;
    const long long end = (long long)t_end * k;
    const long long seg = ((end - beg + kDispWarps - 1) / kDispWarps + 31) / 32 * 32;
    const long long wbeg = beg + wid * seg;
    warp_count_ids(prop, wbeg, min(wbeg + seg, end), E, wcnt + wid * E, false);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int c = 0;
        for (int w = 0; w < kDispWarps; ++w) c += wcnt[w * E + e];
        blockcnt[(long long)blockIdx.x * E + e] = c;
    }
}

// ---- the whole dispatch in one CTA of 1024 threads -------------------------------------
// For n = T*k <= kOneCtaMaxAssign and E <= kOneCtaMaxE (one launch instead of three).
// Warp w owns the contiguous run of assignments [w*seg, (w+1)*seg) (seg a multiple of 32)
// and reads its ids in batches of kOneCtaBatch rounds (all loads of a batch in flight
// together). Pass 1 counts each warp's run per expert (__match_any_sync groups); the
// warp counters then become rank bases in warp order, while all threads form load,
// counts, offsets and the M-tile table; pass 2 ranks and scatters. Ranks are stable in
// token order, as in the three-kernel path, and no scratch memory is used. Needs
// (32 + 1) * E ints of dynamic shared memory.
constexpr int kOneCtaBatch = 16;
// One CTA ranks about 8k assignments in the time the three-kernel path takes; beyond
// a few thousand the parallel path wins.
constexpr int kOneCtaMaxAssign = 4096;
constexpr int kOneCtaMaxE = 320;

//
// With blockcnt (the per-chunk histogram of dispatch_hist_kernel or of the router's
// epilogue) the same kernel runs one CTA per chunk of kDispTok tokens instead: each CTA
// takes its rank bases from the chunks before it and the totals from all of them, so the
// scan needs no kernel of its own; CTA 0 writes load, counts, offsets and the M-tile table.
__global__ void __launch_bounds__(1024) dispatch_one_cta_kernel(
    const int* __restrict__ idx, int T, int k, int E, int cap, int* __restrict__ load,
    int* __restrict__ counts, int* __restrict__ offsets, int* __restrict__ perm_token,
    int* __restrict__ perm_slot, int* __restrict__ slot_dest, int* __restrict__ mtile_offsets,
    unsigned long long* __restrict__ counters, int n_counters, DroppedRows dr,
    const int* __restrict__ blockcnt, int nb, int hist_sub) {
    // hist_sub: rows of blockcnt per chunk (1: per-chunk counts of dispatch_hist_kernel;
    // kDispTok / 32: per-warp counts of 32 tokens each from the router's top-k epilogue),
    // summed here
    pdl_entry();
    extern __shared__ int dsm[];
    const bool first = blockIdx.x == 0;
    if (first && counters && (int)threadIdx.x < n_counters) counters[threadIdx.x] = 0ull;
    __shared__ int s_warp[32];
    int* wcnt = dsm;            // [32][E] running counters
    int* s_off = dsm + 32 * E;  // [E] offsets
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) wcnt[i] = 0;
    const long long cbeg = blockcnt ? (long long)blockIdx.x * kDispTok * k : 0;
    const long long cend =
        blockcnt ? min((long long)(blockIdx.x + 1) * kDispTok, (long long)T) * k : (long long)T * k;
    const long long n = cend - cbeg;
    const int seg = (int)(((n + 31) / 32 + 31) / 32 * 32);   // assignments per warp
    const int rounds = seg / 32;
    const long long wbeg = cbeg + (long long)wid * seg;
    const long long wend = min(wbeg + seg, cend);
    int* my = wcnt + wid * E;
    const unsigned lt_mask = (1u << lane) - 1u;
    // ids of rounds r0 .. r0+kOneCtaBatch-1 of this lane (-1 past the run or out of range)
    auto load_batch = [&](int r0, int (&ids)[kOneCtaBatch], bool report) {
#pragma unroll
        for (int j = 0; j < kOneCtaBatch; ++j) {
            const long long i = wbeg + (long long)(r0 + j) * 32 + lane;
            int e = -1;
            if (r0 + j < rounds && i < wend) {
                e = idx[i];
                if (e < 0 || e >= E) {
                    if (report) raise_error(DEVERR_INDEX);
                    e = -1;
                }
            }
            ids[j] = e;
        }
    };
    __syncthreads();
    // pass 1: per-warp totals (out-of-range ids are reported once, here, and skipped)
    for (int r0 = 0; r0 < rounds; r0 += kOneCtaBatch) {
        int ids[kOneCtaBatch];
        load_batch(r0, ids, true);
#pragma unroll
        for (int j = 0; j < kOneCtaBatch; ++j) {
            const int e = ids[j];
            const unsigned peers = __match_any_sync(0xffffffffu, e);
            if (e >= 0 && (peers & lt_mask) == 0) my[e] += __popc(peers);
            __syncwarp();
        }
    }
    __syncthreads();
    // Histogram rows of all chunks (chunked mode): thread (g, e) of G = 1024 / E groups sums
    // rows g, g + G, ... of expert e, both over all rows and over the rows of the chunks
    // before this one; the G partial sums are then added in group order.
    __shared__ int s_hsum[2][1024];
    if (blockcnt) {
        const int G = (int)blockDim.x / E;
        const int g = threadIdx.x / E, ee = threadIdx.x - g * E;
        if (g < G) {
            const int sub_tok = kDispTok / hist_sub;   // tokens per row
            const int rows = (int)(((long long)T + sub_tok - 1) / sub_tok);
            const int before = (int)blockIdx.x * hist_sub;
            int run_p = 0, all_p = 0;
            int b = g;
            for (; b + 3 * G < rows; b += 4 * G) {   // four loads in flight
                int c[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) c[u] = blockcnt[(long long)(b + u * G) * E + ee];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    all_p += c[u];
                    if (b + u * G < before) run_p += c[u];
                }
            }
            for (; b < rows; b += G) {
                const int c = blockcnt[(long long)b * E + ee];
                all_p += c;
                if (b < before) run_p += c;
            }
            s_hsum[0][threadIdx.x] = run_p;
            s_hsum[1][threadIdx.x] = all_p;
        }
    }
    __syncthreads();
    // load, capacity, offsets; warp counters become rank bases (after the earlier chunks)
    const int e = threadIdx.x;
    int kept = 0;
    if (e < E) {
        int run = 0, all = 0;
        if (blockcnt) {
            const int G = (int)blockDim.x / E;
            for (int g = 0; g < G; ++g) {
                run += s_hsum[0][g * E + e];
                all += s_hsum[1][g * E + e];
            }
        }
        for (int w = 0; w < 32; ++w) {
            const int c = wcnt[w * E + e];
            wcnt[w * E + e] = run;
            run += c;
        }
        if (!blockcnt) all = run;
        kept = min(all, cap);
        if (first) {
            load[e] = all;
            counts[e] = kept;
        }
    }
    int total;
    const int off = block_excl_scan_1024(kept, s_warp, total);
    if (e < E) {
        s_off[e] = off;
        if (first) offsets[e] = off;
    }
    if (first && e == 0) offsets[E] = total;
    const int tiles = (kept + kMTile - 1) / kMTile;
    int ttot;
    const int toff = block_excl_scan_1024(tiles, s_warp, ttot);
    if (first && mtile_offsets) {
        if (e < E) mtile_offsets[e] = toff;
        if (e == 0) mtile_offsets[E] = ttot;
    }
    __syncthreads();
    // pass 2: stable ranks and scatter
    for (int r0 = 0; r0 < rounds; r0 += kOneCtaBatch) {
        int ids[kOneCtaBatch];
        load_batch(r0, ids, false);
#pragma unroll
        for (int j = 0; j < kOneCtaBatch; ++j) {
            const long long i = wbeg + (long long)(r0 + j) * 32 + lane;
            const int ex = ids[j];
            const unsigned peers = __match_any_sync(0xffffffffu, ex);
            int rank = 0;
            if (ex >= 0) rank = my[ex] + __popc(peers & lt_mask);
            __syncwarp();
            if (ex >= 0 && (peers & lt_mask) == 0) my[ex] += __popc(peers);
            __syncwarp();
            bool dropped = false;
            if (r0 + j < rounds && i < wend) {
                if (ex >= 0 && rank < cap) {
                    const int pos = s_off[ex] + rank;
                    perm_token[pos] = (int)(i / k);
                    perm_slot[pos] = (int)(i % k);
                    slot_dest[i] = pos;
                } else {
                    slot_dest[i] = -1;
                    dropped = true;
                }
            }
            if (dr.out)
                write_dropped_rows(dr, __ballot_sync(0xffffffffu, dropped),
                                   wbeg + (long long)(r0 + j) * 32, lane);
        }
    }
}

// ---- the whole dispatch for n = T * k <= 32 assignments: one warp ---------------------
// Lane i holds assignment i (token i / k, slot i % k). Its rank among the assignments of
// its expert in token order is the number of lower lanes in its __match_any_sync group;
// each group's lowest lane writes the group's size as the expert's load. Each lane then
// scans a contiguous run of experts (counts min(load, cap), their offsets and 128-row
// tile counts), a warp scan joins the runs, and the kept assignments are scattered.
// Same outputs as dispatch_one_cta_kernel, without its block-wide phases.
constexpr int kTinyAssign = 32;
__global__ void __launch_bounds__(32) dispatch_tiny_kernel(
    const int* __restrict__ idx, int T, int k, int E, int cap, int* __restrict__ load,
    int* __restrict__ counts, int* __restrict__ offsets, int* __restrict__ perm_token,
    int* __restrict__ perm_slot, int* __restrict__ slot_dest, int* __restrict__ mtile_offsets,
    unsigned long long* __restrict__ counters, int n_counters, DroppedRows dr) {
    pdl_entry();
    extern __shared__ int tsm[];
    int* s_load = tsm;       // [E]
    int* s_off = tsm + E;    // [E]
    const int lane = threadIdx.x;
    if (counters && lane < n_counters) counters[lane] = 0ull;
    const int n = T * k;
    for (int e = lane; e < E; e += 32) s_load[e] = 0;
    int ex = -1;
    if (lane < n) {
        ex = idx[lane];
        if (ex < 0 || ex >= E) {
            raise_error(DEVERR_INDEX);
            ex = -1;
        }
    }
    const unsigned peers = __match_any_sync(0xffffffffu, ex);
    const unsigned lower = peers & ((1u << lane) - 1u);
    const int rank = __popc(lower);
    __syncwarp();
    if (ex >= 0 && lower == 0) s_load[ex] = __popc(peers);
    __syncwarp();
    // lane l scans experts [l * per, (l + 1) * per)
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    int kept_run = 0, tiles_run = 0;
    for (int e = e0; e < e1; ++e) {
        const int kept = min(s_load[e], cap);
        kept_run += kept;
        tiles_run += (kept + kMTile - 1) / kMTile;
    }
    int kept_incl = kept_run, tiles_incl = tiles_run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, kept_incl, off);
        const int b = __shfl_up_sync(0xffffffffu, tiles_incl, off);
        if (lane >= off) {
            kept_incl += a;
            tiles_incl += b;
        }
    }
    int koff = kept_incl - kept_run, toff = tiles_incl - tiles_run;
    for (int e = e0; e < e1; ++e) {
        const int l = s_load[e], kept = min(l, cap);
        load[e] = l;
        counts[e] = kept;
        offsets[e] = koff;
        s_off[e] = koff;
        if (mtile_offsets) mtile_offsets[e] = toff;
        koff += kept;
        toff += (kept + kMTile - 1) / kMTile;
    }
    if (lane == 31) {
        offsets[E] = kept_incl;
        if (mtile_offsets) mtile_offsets[E] = tiles_incl;
    }
    __syncwarp();
    bool dropped = false;
    if (lane < n) {
        if (ex >= 0 && rank < cap) {
            const int pos = s_off[ex] + rank;
            perm_token[pos] = lane / k;
            perm_slot[pos] = lane % k;
            slot_dest[lane] = pos;
        } else {
            slot_dest[lane] = -1;
            dropped = true;
        }
    }
    if (dr.out) write_dropped_rows(dr, __ballot_sync(0xffffffffu, dropped), 0, lane);
}

// ---- the same copy organised by token (k >= 2): one warp per token reads its row of x once
// and writes it to each of its kept slots' rows (slot_dest[t*k + j] >= 0), so x is read
// once instead of k times. 16-byte vectors, four per lane in flight; row_bytes is a
// multiple of 16.
__global__ void __launch_bounds__(256) gather_rows_by_token_kernel(
    const uint8_t* __restrict__ x, const int* __restrict__ slot_dest, int T, int k,
    uint8_t* __restrict__ x_perm, int row_bytes) {
    pdl_entry();
    const int lane = threadIdx.x & 31;
    const int nvec = row_bytes / 16;
    const int warps = gridDim.x * (blockDim.x >> 5);
    for (int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += warps) {
        const int mydest = lane < k ? slot_dest[(long long)t * k + lane] : -1;
        const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * row_bytes);
        for (int c0 = 0; c0 < nvec; c0 += 128) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c = c0 + u * 32 + lane;
                if (c < nvec) v[u] = __ldg(src + c);
            }
            for (int j = 0; j < k; ++j) {
                const int pos = __shfl_sync(0xffffffffu, mydest, j);
                if (pos < 0) continue;
                uint4* dst = reinterpret_cast<uint4*>(x_perm + (size_t)pos * row_bytes);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int c = c0 + u * 32 + lane;
                    if (c < nvec) dst[c] = v[u];
                }
            }
        }
    }
}

// ---- x_perm[p] = x[perm_token[p]] for p < P = offsets[E]; one warp per row -----------
// 16-byte vector copies, four loads in flight per lane before their stores;
// row_bytes is a multiple of 16.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint8_t* __restrict__ x,
                                                          const int* __restrict__ perm_token,
                                                          const int* __restrict__ total_rows,
                                                          uint8_t* __restrict__ x_perm,
                                                          int row_bytes) {
    pdl_entry();
    const int P = *total_rows;
    const int lane = threadIdx.x & 31;
    const int nvec = row_bytes / 16;
    const int warps = gridDim.x * (blockDim.x >> 5);
    for (int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < P; r += warps) {
        const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)perm_token[r] * row_bytes);
        uint4* dst = reinterpret_cast<uint4*>(x_perm + (size_t)r * row_bytes);
        int c = lane;
        for (; c + 96 < nvec; c += 128) {
            const uint4 a = __ldg(src + c), b = __ldg(src + c + 32), d = __ldg(src + c + 64),
                        e = __ldg(src + c + 96);
            dst[c] = a;
            dst[c + 32] = b;
            dst[c + 64] = d;
            dst[c + 96] = e;
        }
        for (; c < nvec; c += 32) dst[c] = __ldg(src + c);
    }
}

// ---- re-routing: room, final counts, offsets, M-tile table (one CTA, expert/thread) ----
// counts[e] holds the round-0 counts on entry (saved to cnt0); expert e accepts
// min(proposals, cap - cnt0[e]) proposals; blockoff[b][e] becomes the rank base of chunk
// b's proposals. Also zeroes the expert GEMMs' tile counters.
__global__ void __launch_bounds__(1024) reroute_scan_kernel(
    const int* __restrict__ blockcnt, int nb, int E, int cap, int* __restrict__ blockoff,
    int* __restrict__ counts, int* __restrict__ cnt0, int* __restrict__ offsets,
    int* __restrict__ mtile_offsets, unsigned long long* __restrict__ counters, int n_counters) {
    pdl_entry();
    __shared__ int s_warp[32];
    const int e = threadIdx.x;
    if (counters && e < n_counters) counters[e] = 0ull;
    int kept = 0;
    if (e < E) {
        int run = 0;
        for (int b = 0; b < nb; ++b) {
            const long long i = (long long)b * E + e;
            const int c = blockcnt[i];
            blockoff[i] = run;
            run += c;
        }
        const int c0 = counts[e];
        cnt0[e] = c0;
        kept = c0 + min(run, max(0, cap - c0));
        counts[e] = kept;
    }
    int total;
    const int off = block_excl_scan_1024(kept, s_warp, total);
    if (e < E) offsets[e] = off;
    if (e == 0) offsets[E] = total;
    write_tile_tables(kept, e, E, s_warp, mtile_offsets);
}

// ---- M-tile table from offsets (expert stage entry): single CTA of 1024 threads ----
// The table kernels also zero the tile counters of the grouped-GEMM launches that
// follow them (counters may be null).
__global__ void __launch_bounds__(1024) mtile_table_kernel(const int* __restrict__ offsets, int G,
                                                           int* __restrict__ mtile_offsets,
                                                           unsigned long long* __restrict__ counters,
                                                           int n_counters) {
    pdl_entry();
    __shared__ int s_warp[32];
    const int g = threadIdx.x;
    if (counters && g < n_counters) counters[g] = 0ull;
    const int rows = (g < G) ? offsets[g + 1] - offsets[g] : 0;
    write_tile_tables(rows, g, G, s_warp, mtile_offsets);
}

// Row and M-tile offsets of one more group of `rows` rows after the E groups of a
// dispatch (the shared expert as group E of the routed up projection): offsets[E + 1] and
// mtile_offsets[E + 1].
__global__ void append_group_kernel(int* __restrict__ offsets, int* __restrict__ mtile_offsets,
                                    int E, int rows) {
    pdl_entry();
    if (threadIdx.x == 0) {
        offsets[E + 1] = offsets[E] + rows;
        if (mtile_offsets) mtile_offsets[E + 1] = mtile_offsets[E] + (rows + kMTile - 1) / kMTile;
    }
}

// Row and M-tile tables of a single group of `rows` rows (the shared expert).
__global__ void single_group_table_kernel(int rows, int* __restrict__ row_offsets,
                                          int* __restrict__ mtile_offsets,
                                          unsigned long long* __restrict__ counters,
                                          int n_counters) {
    pdl_entry();
    if (counters && (int)threadIdx.x < n_counters) counters[threadIdx.x] = 0ull;
    if (threadIdx.x == 0) {
        row_offsets[0] = 0;
        row_offsets[1] = rows;
        mtile_offsets[0] = 0;
        mtile_offsets[1] = (rows + kMTile - 1) / kMTile;
    }
}

}  // namespace moe
