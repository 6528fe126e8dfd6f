// Oracle for the single-GPU MoE layer forward: plain, slow, single-threaded C++.
//
// TEST INFRASTRUCTURE ONLY. Nothing in the product path (the CUDA library and its
// Python binding) includes, links or calls this file. Only the test suite, the
// package smoke check and the benchmark's CPU-baseline leg load liboracle.so.
// It shares no header, helper, table or constant with the CUDA code.
//
// Every quantity is accumulated in double and rounded once at the end to the
// storage type. Loops run in the order the pages describe the method; nothing is
// blocked, fused or reordered.
//
// Sources (page title, section):
//   [Gate]     "MoE 混合专家架构：LLM稀疏化计算的关键演进", section 2.1 门控机制 (TopKGating:
//              Linear without bias -> topk on logits -> softmax over the k logits).
//   [Steps]    "adv12 — Mixture of Experts (MoE) + EPLB", section 4.1 MoELayer step table
//              (softmax(gate(x)) -> topk -> topk_val/sum -> mask + weighted sum -> bincount).
//   [Renorm]   same page, Q1 (why topk_val is renormalised; 0.4/0.3 -> 0.571/0.429).
//   [Capacity] "MoE 并行", section Capacity Factor; adv12 Q2 (capacity 20, load 38 -> 18 overflow).
//   [Agg]      "MOE 学习笔记", 输出聚合示例 (0.7*[0.2,0.4] + 0.3*[0.5,0.3] = [0.29,0.37]).
//   [Switch]   "MoE 混合专家架构", section 1.2 Switch Transformer (k = 1, argmax, weight 1).
//   [SafeSM]   "MoE 混合专家架构", section 4.2 数值稳定性 (max-subtracted softmax).
//   [Merged]   "MoE 混合专家架构", section 5.2 专家融合与并行 (stacked W1, silu on the W1 slice).
//   [LPT]      adv12 sections 3.3 EPLB and 4.3 eplb_rebalance; 4.2 expert_imbalance; Q3.
//   [Quant]    "MoE 混合专家架构", section 5.3 量化支持 (expert weights may be stored as INT8 /
//              INT4 with an acceptable accuracy loss).
//   [Hier]     "MoE 并行", 通信瓶颈 table, row Hierarchical Routing (pick groups first, then
//              experts); adv12 section 5 (DeepSeek-V3: device-limited routing, each token's
//              experts lie on at most M devices).
//   [Reroute]  "MoE 并行", 推理时的负载均衡 (dynamic re-routing: a token whose expert is over
//              its limit goes to the next expert); "MoE 混合专家架构" section 4.2 (capacity
//              check that redistributes the excess tokens of a full expert).
//   [OvfShared] "MoE 并行" Q4 (inference: capacity limit, overflow tokens go to the shared
//              expert) and Q5; adv12 Q2 option 2 (overflow routed to the shared expert).
//
// Readings where the pages are silent or disagree (each one is listed in the design notes):
//   * selection is done on logits with ties broken toward the lower expert id;
//   * kept weights are renormalised over the k selected experts, before capacity;
//   * capacity = ceil(cf * T * k / E) clipped to [1, T]; cf <= 0 means no limit;
//   * over-capacity assignments are dropped in ascending token order and add 0;
//   * GELU is the exact-erf form; SwiGLU gate rows are [0,F) of W1, up rows [F,2F);
//   * the hidden activation h is rounded to bf16 when the weights are bf16;
//   * the shared expert has weight 1 for every token;
//   * group-limited routing scores a group by its best expert logit (the pages name the
//     two steps but not the score);
//   * INT8 experts are weight-only, symmetric, one absmax scale per weight row (the pages
//     name INT8 / INT4 but no scheme);
//   * overflow to the shared expert: a dropped slot's weight is added to the (always-on)
//     shared expert's weight of that token;
//   * re-routing: one round; a token's dropped slots, in slot order, go to its next-ranked
//     experts (ranks k, k+1, ...) and keep their weights; each expert accepts them in token
//     order while it has room under the capacity; rejected slots stay dropped.
//
// Parity status: every exported function is pinned by the CPU test suite against
// values printed on the pages, closed forms, or brute force on tiny inputs,
// except the seed-42 toy histogram printed on the adv12 page (section 6), which
// cannot be regenerated because the page's run.py is not given: parity unpinned
// for that histogram; it is used only as an input to the load-report pins.

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <vector>
#include <algorithm>

namespace {

enum { ORC_F32 = 0, ORC_BF16 = 1 };
enum { ORC_LINEAR = 0, ORC_GELU = 1, ORC_SWIGLU = 2 };

// bf16 storage -> value: a bf16 is the top 16 bits of an IEEE binary32.
double bf16_bits_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return (double)f;
}

double load_elem(const void* p, int dtype, long long i) {
    if (dtype == ORC_F32) return (double)((const float*)p)[i];
    return bf16_bits_to_double(((const uint16_t*)p)[i]);
}

// Round a real (held in double) to the nearest bf16, ties to even, in one step.
// bf16 keeps 8 significant bits and float's exponent range; below 2^-126 the
// quantum stays 2^-133 (subnormals).
uint16_t double_to_bf16_rne(double v) {
    if (std::isnan(v)) return 0x7FC0;
    if (v == 0.0) return std::signbit(v) ? 0x8000 : 0x0000;
    int e;
    std::frexp(v, &e);                 // |v| = m * 2^e, m in [0.5, 1)
    int qexp = e - 8;                  // quantum for 8 significant bits
    if (qexp < -133) qexp = -133;
    double q = std::ldexp(1.0, qexp);
    double r = std::nearbyint(v / q) * q;   // default rounding mode: nearest-even
    // r is now exactly a bf16 value (or overflows past the largest finite one).
    float f = (float)r;                // exact when representable; inf on overflow
    if (std::fabs(r) > 3.3895313892515355e38) f = std::signbit(r) ? -INFINITY : INFINITY;
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

double gelu_exact(double a) { return 0.5 * a * (1.0 + std::erf(a / std::sqrt(2.0))); }
double silu(double a) { return a / (1.0 + std::exp(-a)); }

void store_out(void* out, int dtype, long long i, double v) {
    if (dtype == ORC_F32) ((float*)out)[i] = (float)v;
    else ((uint16_t*)out)[i] = double_to_bf16_rne(v);
}

}  // namespace

extern "C" {

// ---- small exported helpers (pinned individually) ---------------------------
uint16_t oracle_bf16_round(double v) { return double_to_bf16_rne(v); }
double oracle_gelu(double a) { return gelu_exact(a); }
double oracle_silu(double a) { return silu(a); }

// O1 gate logits [Gate], [Steps] step 1: L[t,e] = sum_i x[t,i] * Wg[i,e] (+ b[e]).
// Wg is stored [d, E] (E contiguous). rows == NULL computes all T rows into
// logits[T, E]; otherwise only rows[0..nrows) into logits[nrows, E].
void oracle_gate_logits(const void* x, int x_dtype, const float* Wg, const float* bias,
                        int T, int d, int E, const int32_t* rows, int nrows, float* logits) {
    int n = rows ? nrows : T;
    for (int r = 0; r < n; ++r) {
        long long t = rows ? rows[r] : r;
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i)
                acc += load_elem(x, x_dtype, t * d + i) * (double)Wg[(long long)i * E + e];
            if (bias) acc += (double)bias[e];
            logits[(long long)r * E + e] = (float)acc;
        }
    }
}

// O2 + O3 top-k and renormalisation [Gate], [Steps] steps 2-3, [Renorm], [SafeSM].
// Experts are ordered by (logit descending, id ascending); the first k are kept.
// The kept weights are softmax over the k kept logits, computed max-subtracted:
// w_j = exp(L_j - L_0) / sum_{j'<k} exp(L_j' - L_0). This equals taking the full
// softmax, keeping the k largest probabilities and dividing by their sum.
void oracle_topk_renorm(const float* logits, int T, int E, int k, int32_t* idx, float* w) {
    for (int t = 0; t < T; ++t) {
        const float* L = logits + (long long)t * E;
        // Selection by repeated scan for the best remaining expert (plain, O(k*E)).
        std::vector<char> taken(E, 0);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || L[e] > L[best]) best = e;   // strict '>' keeps the lower id on ties
            }
            taken[best] = 1;
            idx[(long long)t * k + j] = best;
        }
        double l0 = (double)L[idx[(long long)t * k]];
        double s = 0.0;
        for (int j = 0; j < k; ++j) s += std::exp((double)L[idx[(long long)t * k + j]] - l0);
        for (int j = 0; j < k; ++j)
            w[(long long)t * k + j] = (float)(std::exp((double)L[idx[(long long)t * k + j]] - l0) / s);
    }
}

// Group-limited routing [Hier]: experts are split into n_group groups of E / n_group
// consecutive ids. First the topk_group groups whose best expert logit is highest are
// chosen (ties to the lower group id); then the k experts with the highest logits among
// the chosen groups' experts (ties to the lower id); the kept weights are renormalised
// as in oracle_topk_renorm.
void oracle_topk_renorm_grouped(const float* logits, int T, int E, int k, int n_group,
                                int topk_group, int32_t* idx, float* w) {
    const int gsize = E / n_group;
    for (int t = 0; t < T; ++t) {
        const float* L = logits + (long long)t * E;
        // step 1: score of each group = its best expert logit
        std::vector<float> gscore(n_group);
        for (int g = 0; g < n_group; ++g) {
            float m = L[g * gsize];
            for (int e = g * gsize + 1; e < (g + 1) * gsize; ++e)
                if (L[e] > m) m = L[e];
            gscore[g] = m;
        }
        // step 2: the topk_group best groups
        std::vector<char> chosen(n_group, 0);
        for (int j = 0; j < topk_group; ++j) {
            int best = -1;
            for (int g = 0; g < n_group; ++g) {
                if (chosen[g]) continue;
                if (best < 0 || gscore[g] > gscore[best]) best = g;
            }
            chosen[best] = 1;
        }
        // step 3: the k best experts of the chosen groups
        std::vector<char> taken(E, 0);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e] || !chosen[e / gsize]) continue;
                if (best < 0 || L[e] > L[best]) best = e;
            }
            taken[best] = 1;
            idx[(long long)t * k + j] = best;
        }
        // step 4: renormalised weights of the kept experts
        double l0 = (double)L[idx[(long long)t * k]];
        double s = 0.0;
        for (int j = 0; j < k; ++j) s += std::exp((double)L[idx[(long long)t * k + j]] - l0);
        for (int j = 0; j < k; ++j)
            w[(long long)t * k + j] = (float)(std::exp((double)L[idx[(long long)t * k + j]] - l0) / s);
    }
}

// O4 expert load [Steps] step 5 (bincount of the selected expert ids, before capacity).
void oracle_load(const int32_t* idx, int T, int k, int E, int32_t* load) {
    for (int e = 0; e < E; ++e) load[e] = 0;
    for (long long i = 0; i < (long long)T * k; ++i) load[idx[i]] += 1;
}

// O5 capacity [Capacity]: tokens an expert may take. cf <= 0 means unlimited (T).
int32_t oracle_capacity(double cf, int T, int k, int E) {
    if (!(cf > 0.0)) return T;
    double c = std::ceil(cf * (double)T * (double)k / (double)E);
    if (c < 1.0) c = 1.0;
    if (c > (double)T) c = (double)T;
    return (int32_t)c;
}

// O6 + O7 dispatch: group the kept (token, slot) assignments by expert.
// For each expert the assignments are taken in ascending token order; the r-th
// one (r = 0, 1, ...) is kept iff r < cap [Capacity] (overflow falls through).
// counts[e] = kept count, offsets = exclusive prefix sum of counts (offsets[E] = P),
// perm_token / perm_slot list the kept assignments expert by expert, and
// slot_dest[t*k + j] is the row of (t, j) in that list, or -1 if dropped.
void oracle_dispatch(const int32_t* idx, int T, int k, int E, int cap,
                     int32_t* counts, int32_t* offsets, int32_t* perm_token,
                     int32_t* perm_slot, int32_t* slot_dest) {
    std::vector<long long> rank(E, 0);
    for (int e = 0; e < E; ++e) counts[e] = 0;
    // First pass: how many are kept per expert.
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int e = idx[(long long)t * k + j];
            if (rank[e] < cap) counts[e] += 1;
            rank[e] += 1;
        }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    // Second pass: place each kept assignment.
    for (int e = 0; e < E; ++e) rank[e] = 0;
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            long long s = (long long)t * k + j;
            int e = idx[s];
            if (rank[e] < cap) {
                int pos = offsets[e] + (int)rank[e];
                perm_token[pos] = t;
                perm_slot[pos] = j;
                slot_dest[s] = pos;
            } else {
                slot_dest[s] = -1;
            }
            rank[e] += 1;
        }
}

// Next-ranked experts for re-routing [Reroute]: cand[t][0..m) are the experts at
// positions k .. k+m-1 of token t's ranking (logit descending, id ascending), or -1 where
// the ranking has fewer experts. With n_group > 0 the ranking covers only the experts of
// the topk_group chosen groups (chosen as in oracle_topk_renorm_grouped).
void oracle_rank_candidates(const float* logits, int T, int E, int k, int n_group, int topk_group,
                            int m, int32_t* cand) {
    for (int t = 0; t < T; ++t) {
        const float* L = logits + (long long)t * E;
        std::vector<char> allowed(E, 1);
        if (n_group > 0) {
            const int gsize = E / n_group;
            std::vector<float> gscore(n_group);
            for (int g = 0; g < n_group; ++g) {
                float mx = L[g * gsize];
                for (int e = g * gsize + 1; e < (g + 1) * gsize; ++e)
                    if (L[e] > mx) mx = L[e];
                gscore[g] = mx;
            }
            std::vector<char> chosen(n_group, 0);
            for (int j = 0; j < topk_group; ++j) {
                int best = -1;
                for (int g = 0; g < n_group; ++g) {
                    if (chosen[g]) continue;
                    if (best < 0 || gscore[g] > gscore[best]) best = g;
                }
                chosen[best] = 1;
            }
            for (int e = 0; e < E; ++e) allowed[e] = chosen[e / gsize];
        }
        std::vector<char> taken(E, 0);
        for (int pos = 0; pos < k + m; ++pos) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e] || !allowed[e]) continue;
                if (best < 0 || L[e] > L[best]) best = e;
            }
            if (best >= 0) taken[best] = 1;
            if (pos >= k) cand[(long long)t * m + (pos - k)] = best;
        }
    }
}

// Dispatch with one round of re-routing [Reroute], [Capacity].
// Round 0 is oracle_dispatch's rule: per expert, assignments in ascending token order,
// the r-th kept iff r < cap. Round 1: the dropped slots of token t, in slot order, propose
// to cand[t][0], cand[t][1], ... (k candidates per token; -1 = none); each expert takes its
// proposals in ascending (token, slot) order while its round-0 rows plus the proposals it
// has taken stay below cap. Expert e's rows are its round-0 rows (token order) followed by
// its round-1 rows (token order). route_idx[t][j] is the expert that processes slot
// (t, j) (the original one unless re-routed); slot_dest as in oracle_dispatch.
void oracle_dispatch_reroute(const int32_t* idx, const int32_t* cand, int T, int k, int E, int cap,
                             int32_t* counts, int32_t* offsets, int32_t* perm_token,
                             int32_t* perm_slot, int32_t* slot_dest, int32_t* route_idx) {
    const long long n = (long long)T * k;
    // round 0: ranks in token order
    std::vector<int> r0(n, -1);
    std::vector<int> kept0(E, 0), seen(E, 0);
    for (long long s = 0; s < n; ++s) {
        const int e = idx[s];
        if (seen[e] < cap) {
            r0[s] = seen[e];
            kept0[e] += 1;
        }
        seen[e] += 1;
    }
    // round 1: proposals of the dropped slots, accepted in token order while there is room
    std::vector<int> prop(n, -1), r1(n, -1), acc1(E, 0);
    for (int t = 0; t < T; ++t) {
        int m = 0;
        for (int j = 0; j < k; ++j) {
            const long long s = (long long)t * k + j;
            if (r0[s] >= 0) continue;
            prop[s] = cand[(long long)t * k + m];
            m += 1;
        }
    }
    for (long long s = 0; s < n; ++s) {
        const int e = prop[s];
        if (e < 0) continue;
        if (kept0[e] + acc1[e] < cap) {
            r1[s] = acc1[e];
            acc1[e] += 1;
        }
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) {
        counts[e] = kept0[e] + acc1[e];
        offsets[e + 1] = offsets[e] + counts[e];
    }
    for (long long s = 0; s < n; ++s) {
        const int t = (int)(s / k), j = (int)(s % k);
        int pos = -1;
        route_idx[s] = idx[s];
        if (r0[s] >= 0) {
            pos = offsets[idx[s]] + r0[s];
        } else if (r1[s] >= 0) {
            pos = offsets[prop[s]] + kept0[prop[s]] + r1[s];
            route_idx[s] = prop[s];
        }
        slot_dest[s] = pos;
        if (pos >= 0) {
            perm_token[pos] = t;
            perm_slot[pos] = j;
        }
    }
}

// O8 one token through one expert [Steps] (expert_e(x)), [Merged] (stacked W1 slice).
//   LINEAR: y = W1 x + b1                (W1 [d][d]; the tiny tutorial expert)
//   GELU:   h = gelu(W1 x + b1), y = W2 h + b2         (W1 [F][d], W2 [d][F])
//   SWIGLU: h = silu(W1[0:F] x) * (W1[F:2F] x), y = W2 h + b2   (W1 [2F][d])
// h is rounded to bf16 when w_dtype is bf16. y is returned unrounded (double).
void oracle_expert_row(int kind, const void* x_row, int x_dtype,
                       const void* w1, const float* b1, const void* w2, const float* b2,
                       int w_dtype, int d, int F, double* y) {
    if (kind == ORC_LINEAR) {
        for (int o = 0; o < d; ++o) {
            double acc = 0.0;
            for (int c = 0; c < d; ++c)
                acc += load_elem(w1, w_dtype, (long long)o * d + c) * load_elem(x_row, x_dtype, c);
            if (b1) acc += (double)b1[o];
            y[o] = acc;
        }
        return;
    }
    std::vector<double> h(F);
    for (int f = 0; f < F; ++f) {
        double a = 0.0;
        for (int c = 0; c < d; ++c)
            a += load_elem(w1, w_dtype, (long long)f * d + c) * load_elem(x_row, x_dtype, c);
        if (b1) a += (double)b1[f];
        double hv;
        if (kind == ORC_GELU) {
            hv = gelu_exact(a);
        } else {
            double u = 0.0;
            for (int c = 0; c < d; ++c)
                u += load_elem(w1, w_dtype, (long long)(F + f) * d + c) * load_elem(x_row, x_dtype, c);
            if (b1) u += (double)b1[F + f];
            hv = silu(a) * u;
        }
        h[f] = (w_dtype == ORC_BF16) ? bf16_bits_to_double(double_to_bf16_rne(hv)) : hv;
    }
    for (int o = 0; o < d; ++o) {
        double acc = 0.0;
        for (int f = 0; f < F; ++f) acc += load_elem(w2, w_dtype, (long long)o * F + f) * h[f];
        if (b2) acc += (double)b2[o];
        y[o] = acc;
    }
}

// Weight-only INT8 experts [Quant]: every weight row n (an output channel of W1 or W2)
// is stored as int8 codes q[n][k] and one fp32 scale s[n]; the expert computes with the
// dequantised weights s[n] * q[n][k] (formed exactly in double).
//   quantize: s = max_k |w[n][k]| / 127, q = round-half-even(w / s) clamped to [-127, 127],
//   both in fp32 arithmetic (a floating-point decision that yields an integer code is made
//   in the precision the kernel uses); an all-zero row has s = 0 and q = 0.
void oracle_quantize_rows_i8(const uint16_t* w_bf16, long long rows, int cols, int8_t* q,
                             float* scale) {
    for (long long r = 0; r < rows; ++r) {
        float m = 0.0f;
        for (int c = 0; c < cols; ++c) {
            const float v = std::fabs((float)bf16_bits_to_double(w_bf16[r * cols + c]));
            if (v > m) m = v;
        }
        const float sc = m / 127.0f;
        scale[r] = sc;
        for (int c = 0; c < cols; ++c) {
            float qv = 0.0f;
            if (sc > 0.0f) {
                const float v = (float)bf16_bits_to_double(w_bf16[r * cols + c]);
                qv = std::nearbyint(v / sc);   // default rounding mode: nearest, ties to even
                if (qv > 127.0f) qv = 127.0f;
                if (qv < -127.0f) qv = -127.0f;
            }
            q[r * cols + c] = (int8_t)qv;
        }
    }
}

// Weight-only INT4 experts [Quant]: the INT8 form with codes in [-7, 7] (the symmetric
// range of a 4-bit two's complement code; -8 is never produced):
//   s = max_k |w[n][k]| / 7, q = round-half-even(w / s) clamped to [-7, 7], in fp32.
// Storage, two codes per byte along the row: byte j of a row holds column 2j in its low
// nibble and column 2j+1 in its high nibble, each as the 4-bit two's complement of the code;
// a row of `cols` codes (cols even) takes cols / 2 bytes.
void oracle_quantize_rows_i4(const uint16_t* w_bf16, long long rows, int cols, uint8_t* packed,
                             float* scale) {
    for (long long r = 0; r < rows; ++r) {
        float m = 0.0f;
        for (int c = 0; c < cols; ++c) {
            const float v = std::fabs((float)bf16_bits_to_double(w_bf16[r * cols + c]));
            if (v > m) m = v;
        }
        const float sc = m / 7.0f;
        scale[r] = sc;
        for (int c = 0; c < cols; c += 2) {
            int code[2] = {0, 0};
            for (int u = 0; u < 2; ++u) {
                if (sc > 0.0f) {
                    const float v = (float)bf16_bits_to_double(w_bf16[r * cols + c + u]);
                    float qv = std::nearbyint(v / sc);   // nearest, ties to even
                    if (qv > 7.0f) qv = 7.0f;
                    if (qv < -7.0f) qv = -7.0f;
                    code[u] = (int)qv;
                }
            }
            packed[r * (cols / 2) + c / 2] = (uint8_t)((code[0] & 15) | ((code[1] & 15) << 4));
        }
    }
}

// The codes of a packed INT4 matrix [rows, cols / 2] as int8 [rows, cols]: the nibble's
// value v in 0..15 is the code v for v < 8 and v - 16 otherwise.
void oracle_unpack_i4(const uint8_t* packed, long long rows, int cols, int8_t* q) {
    for (long long r = 0; r < rows; ++r)
        for (int c = 0; c < cols; ++c) {
            const uint8_t b = packed[r * (cols / 2) + c / 2];
            const int v = (c % 2 == 0) ? (b & 15) : (b >> 4);
            q[r * cols + c] = (int8_t)(v < 8 ? v : v - 16);
        }
}

// O8 with INT8 weights: as oracle_expert_row for GELU / SWIGLU, the weight of row n,
// column c being s[n] * q[n][c]. h is rounded to bf16 (the activations are bf16).
void oracle_expert_row_q8(int kind, const void* x_row, int x_dtype, const int8_t* q1,
                          const float* s1, const float* b1, const int8_t* q2, const float* s2,
                          const float* b2, int d, int F, double* y) {
    auto w1 = [&](long long r, int c) { return (double)s1[r] * (double)q1[r * d + c]; };
    auto w2 = [&](long long r, int c) { return (double)s2[r] * (double)q2[r * F + c]; };
    std::vector<double> h(F);
    for (int f = 0; f < F; ++f) {
        double a = 0.0;
        for (int c = 0; c < d; ++c) a += w1(f, c) * load_elem(x_row, x_dtype, c);
        if (b1) a += (double)b1[f];
        double hv;
        if (kind == ORC_GELU) {
            hv = gelu_exact(a);
        } else {
            double u = 0.0;
            for (int c = 0; c < d; ++c) u += w1(F + f, c) * load_elem(x_row, x_dtype, c);
            if (b1) u += (double)b1[F + f];
            hv = silu(a) * u;
        }
        h[f] = bf16_bits_to_double(double_to_bf16_rne(hv));
    }
    for (int o = 0; o < d; ++o) {
        double acc = 0.0;
        for (int f = 0; f < F; ++f) acc += w2(o, f) * h[f];
        if (b2) acc += (double)b2[o];
        y[o] = acc;
    }
}

// O9 combine for one token [Agg], [Steps] step 4, [Capacity] (overflow -> residual):
// out = (add_residual ? x : 0) + sum_{j kept, ascending} w_j * y_j + (shared ? a * ys : 0),
// accumulated in double, rounded once to out_dtype. ys may be NULL.
// ys_k holds k rows of d values; kept[j] == 0 marks a dropped slot.
// a = 1, or with overflow_to_shared [OvfShared] a = 1 + sum_{j dropped} w_j.
void oracle_combine_row_ovf(const void* x_row, int x_dtype, int add_residual, int d, int k,
                            const float* w, const int32_t* kept, const double* ys_k,
                            const double* ys_shared, int overflow_to_shared, void* out_row,
                            int out_dtype) {
    double a = 1.0;
    if (overflow_to_shared)
        for (int j = 0; j < k; ++j)
            if (!kept[j]) a += (double)w[j];
    for (int c = 0; c < d; ++c) {
        double acc = add_residual ? load_elem(x_row, x_dtype, c) : 0.0;
        for (int j = 0; j < k; ++j)
            if (kept[j]) acc += (double)w[j] * ys_k[(long long)j * d + c];
        if (ys_shared) acc += a * ys_shared[c];
        store_out(out_row, out_dtype, c, acc);
    }
}
void oracle_combine_row(const void* x_row, int x_dtype, int add_residual, int d, int k,
                        const float* w, const int32_t* kept, const double* ys_k,
                        const double* ys_shared, void* out_row, int out_dtype) {
    oracle_combine_row_ovf(x_row, x_dtype, add_residual, d, k, w, kept, ys_k, ys_shared, 0,
                           out_row, out_dtype);
}

// Whole forward for inputs held entirely in host memory (small problems).
// kind/w_dtype as in oracle_expert_row; x and out share act dtype x_dtype.
// Weights: w1 [E][N1][d], b1 [E][N1] (nullable), w2 [E][d][F], b2 [E][d] (nullable),
// N1 = d (LINEAR), F (GELU), 2F (SWIGLU). Shared expert (nullable): one such expert.
// Outputs: out [T][d]; idx, w [T][k]; logits [T][E]; load [E]; counts [E];
// offsets [E+1]; perm_token, perm_slot [T*k]; slot_dest [T*k].
// overflow: 0 = dropped slots add 0; 1 = their weight goes to the shared expert
// [OvfShared]; 2 = one re-routing round to the next-ranked experts [Reroute] (idx then
// holds the expert that processes each slot). load is always the raw top-k bincount.
void oracle_forward(int kind, int T, int d, int E, int k, int F, double cf, int add_residual,
                    const void* x, int x_dtype, const float* Wg, const float* gate_bias,
                    const void* w1, const float* b1, const void* w2, const float* b2,
                    const void* sw1, const float* sb1, const void* sw2, const float* sb2,
                    int w_dtype, void* out, float* logits, int32_t* idx, float* w,
                    int32_t* load, int32_t* counts, int32_t* offsets, int32_t* perm_token,
                    int32_t* perm_slot, int32_t* slot_dest, int overflow) {
    oracle_gate_logits(x, x_dtype, Wg, gate_bias, T, d, E, nullptr, 0, logits);
    oracle_topk_renorm(logits, T, E, k, idx, w);
    oracle_load(idx, T, k, E, load);
    int cap = oracle_capacity(cf, T, k, E);
    if (overflow == 2) {
        std::vector<int32_t> cand((size_t)T * k), orig(idx, idx + (size_t)T * k);
        oracle_rank_candidates(logits, T, E, k, 0, 0, k, cand.data());
        oracle_dispatch_reroute(orig.data(), cand.data(), T, k, E, cap, counts, offsets,
                                perm_token, perm_slot, slot_dest, idx);
    } else {
        oracle_dispatch(idx, T, k, E, cap, counts, offsets, perm_token, perm_slot, slot_dest);
    }
    long long N1 = (kind == ORC_LINEAR) ? d : (kind == ORC_GELU ? F : 2LL * F);
    long long w1_per = N1 * d, w2_per = (kind == ORC_LINEAR) ? 0 : (long long)d * F;
    long long esz = (w_dtype == ORC_F32) ? 4 : 2;
    long long xsz = (x_dtype == ORC_F32) ? 4 : 2;
    std::vector<double> ys((size_t)k * d), ysh(d);
    std::vector<int32_t> kept(k);
    for (int t = 0; t < T; ++t) {
        const char* xr = (const char*)x + (long long)t * d * xsz;
        for (int j = 0; j < k; ++j) {
            long long s = (long long)t * k + j;
            kept[j] = slot_dest[s] >= 0;
            if (!kept[j]) continue;
            int e = idx[s];
            oracle_expert_row(kind, xr, x_dtype,
                              (const char*)w1 + e * w1_per * esz, b1 ? b1 + e * N1 : nullptr,
                              w2 ? (const char*)w2 + e * w2_per * esz : nullptr,
                              b2 ? b2 + (long long)e * d : nullptr, w_dtype, d, F, &ys[(size_t)j * d]);
        }
        if (sw1) oracle_expert_row(kind, xr, x_dtype, sw1, sb1, sw2, sb2, w_dtype, d, F, ysh.data());
        oracle_combine_row_ovf(xr, x_dtype, add_residual, d, k, w + (long long)t * k, kept.data(),
                               ys.data(), sw1 ? ysh.data() : nullptr, overflow == 1,
                               (char*)out + (long long)t * d * xsz, x_dtype);
    }
}

// O10 load report [LPT]. imbalance = max(load) / (min(load) + 1e-6).
// LPT: experts taken by load descending (stable: equal loads keep ascending id),
// each placed on the currently least-loaded device (lowest index on ties).
// naive_load: experts split into D contiguous blocks of ceil(E/D).
// Variances are the unbiased (n-1) sample variance of the D device loads.
void oracle_load_report(const int32_t* load, int E, int D, int32_t* assign, int64_t* dev_load,
                        int64_t* naive_load, double* imbalance, double* var_lpt, double* var_naive) {
    int32_t mx = load[0], mn = load[0];
    for (int e = 1; e < E; ++e) { mx = std::max(mx, load[e]); mn = std::min(mn, load[e]); }
    *imbalance = (double)mx / ((double)mn + 1e-6);
    std::vector<int> order(E);
    for (int e = 0; e < E; ++e) order[e] = e;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return load[a] > load[b]; });
    for (int d = 0; d < D; ++d) dev_load[d] = 0;
    for (int i = 0; i < E; ++i) {
        int e = order[i];
        int best = 0;
        for (int d = 1; d < D; ++d) if (dev_load[d] < dev_load[best]) best = d;
        assign[e] = best;
        dev_load[best] += load[e];
    }
    int per = (E + D - 1) / D;
    for (int d = 0; d < D; ++d) naive_load[d] = 0;
    for (int e = 0; e < E; ++e) naive_load[e / per] += load[e];
    auto var = [&](const int64_t* v) {
        if (D < 2) return 0.0;
        double m = 0.0;
        for (int d = 0; d < D; ++d) m += (double)v[d];
        m /= D;
        double s = 0.0;
        for (int d = 0; d < D; ++d) s += ((double)v[d] - m) * ((double)v[d] - m);
        return s / (D - 1);
    };
    *var_lpt = var(dev_load);
    *var_naive = var(naive_load);
}

}  // extern "C"
