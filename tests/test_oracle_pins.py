"""Pins for the CPU oracle: values printed on the pages, closed forms, brute force.

Each test checks the oracle against something other than itself, so that a
plausible slip in it (a dropped term, a wrong index or sign, a swapped operand,
a wrong tie-break) fails at least one of them.
"""

import itertools
import math

import numpy as np
import pytest

import oracle as orc
from synth import host_fill, normal_K, NORMAL


# --------------------------------------------------------------------------
# helpers: an independent dense formulation, written the way the adv12 page's
# step table orders the forward (softmax over all experts, top-k on the
# probabilities, divide by their sum, mask-weighted sum over every expert).
# --------------------------------------------------------------------------

def bf16_bits_to_f64(a):
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16_value(v):
    """float64 -> float32 (RNE) -> bf16 (RNE via the carry trick), returned as float64."""
    f = np.asarray(v, np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return bf16_bits_to_f64(u.astype(np.uint16))


def as_f64(a):
    return bf16_bits_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def dense_expert(kind, X, w1, b1, w2, b2, F):
    """All tokens through one expert (float64), textbook formulas."""
    W1 = as_f64(w1)
    A = X @ W1.T + (0 if b1 is None else b1.astype(np.float64))
    if kind == orc.LINEAR:
        return A
    if kind == orc.GELU:
        from scipy.special import erf
        H = 0.5 * A * (1 + erf(A / math.sqrt(2)))
    else:
        g, u = A[:, :F], A[:, F:]
        H = g / (1 + np.exp(-g)) * u
    if w1.dtype == np.uint16:
        H = f64_to_bf16_value(H)
    Y = H @ as_f64(w2).T + (0 if b2 is None else b2.astype(np.float64))
    return Y


def dense_forward(kind, x, Wg, gb, W, k, F, add_residual=False):
    X = as_f64(x)
    T, d = X.shape
    E = Wg.shape[1]
    L = X @ Wg.astype(np.float64) + (0 if gb is None else gb.astype(np.float64))
    L = L.astype(np.float32).astype(np.float64)     # the layer's logits are fp32
    P = np.exp(L - L.max(axis=1, keepdims=True))
    P /= P.sum(axis=1, keepdims=True)
    M = np.zeros((T, E))
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-P[t, e], e))[:k]
        s = sum(P[t, e] for e in order)
        for e in order:
            M[t, e] = P[t, e] / s
    out = X.copy() if add_residual else np.zeros((T, d))
    for e in range(E):
        Ye = dense_expert(kind, X, W["w1"][e], None if W["b1"] is None else W["b1"][e],
                          None if W["w2"] is None else W["w2"][e],
                          None if W["b2"] is None else W["b2"][e], F)
        out += M[:, [e]] * Ye
    if W.get("shared") is not None:
        sw1, sb1, sw2, sb2 = W["shared"]
        out += dense_expert(kind, X, sw1, sb1, sw2, sb2, F)
    return out, M


def rand(shape, seed, tid, std=1.0, bf16=False):
    n = int(np.prod(shape))
    return host_fill(seed, tid, 0, n, NORMAL, normal_K(std), bf16).reshape(shape)


def small_problem(kind, T, d, E, k, F, seed, bf16, biases=False, shared=False):
    x = rand((T, d), seed, 1, 1.0, bf16)
    Wg = rand((d, E), seed, 2, 1 / math.sqrt(d))
    N1 = d if kind == orc.LINEAR else (F if kind == orc.GELU else 2 * F)
    W = dict(w1=rand((E, N1, d), seed, 4, 1 / math.sqrt(d), bf16),
             b1=rand((E, N1), seed, 5, 1 / math.sqrt(d)) if biases else None,
             w2=None if kind == orc.LINEAR else rand((E, d, F), seed, 6, 1 / math.sqrt(F), bf16),
             b2=rand((E, d), seed, 7, 0.1) if (biases and kind != orc.LINEAR) else None)
    W["shared"] = None
    if shared:
        W["shared"] = (rand((N1, d), seed, 8, 1 / math.sqrt(d), bf16), None,
                       rand((d, F), seed, 10, 1 / math.sqrt(F), bf16), None)
    return x, Wg, W


def run_oracle(kind, x, Wg, gb, W, k, F, cf=0.0, add_residual=False):
    return orc.forward(kind, x, Wg, gb, W["w1"], W["b1"], W["w2"], W["b2"], k, F, cf=cf,
                       add_residual=add_residual, shared=W.get("shared"))


# --------------------------------------------------------------------------
# values printed on the pages
# --------------------------------------------------------------------------

def test_renorm_printed_example(golden):
    g = golden("renorm_adv12_q1.json")
    logits = np.log(np.array([g["probs"]], np.float64)).astype(np.float32)
    idx, w = orc.topk_renorm(logits, g["k"])
    assert idx[0].tolist() == g["expected_idx"]
    assert np.round(w[0].astype(np.float64), g["printed_decimals"]).tolist() == g["expected_w"]
    # the exact values are 4/7 and 3/7
    assert abs(w[0, 0] - 4 / 7) < 2e-7 and abs(w[0, 1] - 3 / 7) < 2e-7
    assert abs(sum(g["probs"][:2]) - g["unnormalised_sum"]) < 1e-12


def test_aggregation_printed_example(golden):
    g = golden("aggregation_moe_notes.json")
    ys = np.array(g["expert_outputs"], np.float64)
    x_row = np.zeros(2, np.float32)
    out = orc.combine_row(x_row, False, g["weights"], [1, 1], ys, None, orc.F32)
    assert np.allclose(out, g["expected"], atol=1e-7)


def test_aggregation_through_whole_forward(golden):
    """Same example driven through the full oracle forward: two LINEAR experts with
    zero weight matrices and biases equal to the printed outputs; the gate bias
    makes the renormalised routing weights 0.7 and 0.3."""
    g = golden("aggregation_moe_notes.json")
    T, d, E, k = 1, 2, 2, 2
    x = np.zeros((T, d), np.float32)
    Wg = np.zeros((d, E), np.float32)
    gb = np.log(np.array(g["weights"], np.float64)).astype(np.float32)
    w1 = np.zeros((E, d, d), np.float32)
    b1 = np.array(g["expert_outputs"], np.float32)
    r = orc.forward(orc.LINEAR, x, Wg, gb, w1, b1, None, None, k, d)
    assert r["idx"][0].tolist() == [0, 1]
    assert np.allclose(r["w"][0], g["weights"], atol=1e-7)
    assert np.allclose(r["out"][0], g["expected"], atol=1e-6)


def test_capacity_printed_example(golden):
    g = golden("capacity_adv12_q2.json")
    T, k, E = g["T"], g["k"], g["E"]
    # a routing table with the page's loads: each token picks two different experts
    idx = np.zeros((T, k), np.int32)
    remaining = list(g["loads"])
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-remaining[e], e))[:k]
        idx[t] = order
        for e in order:
            remaining[e] -= 1
    assert remaining == [0] * E
    ld = orc.load(idx, E)
    assert ld.tolist() == g["loads"] and int(ld.sum()) == g["total_routings"] == T * k
    counts, offsets, pt, ps, sd = orc.dispatch(idx, E, g["capacity"])
    assert counts[0] == g["expert0_kept"]
    assert int((sd[idx == 0] < 0).sum()) == g["expert0_overflow"]
    assert counts.tolist() == [min(l, g["capacity"]) for l in g["loads"]]
    # the kept ones are the earliest tokens of each expert
    for e in range(E):
        toks = [t for t in range(T) if e in idx[t]]
        assert pt[offsets[e]:offsets[e + 1]].tolist() == toks[:g["capacity"]]


def test_capacity_factor_definition():
    # capacity = ceil(cf * T * k / E), clipped to [1, T]; cf <= 0 means no limit
    assert orc.capacity(1.25, 8192, 1, 64) == 160           # Switch-shaped workload
    assert orc.capacity(1.0, 8192, 8, 256) == 256            # DeepSeek-shaped, cf 1.0
    assert orc.capacity(1.25, 8192, 8, 256) == 320           # DeepSeek-shaped, cf 1.25
    assert orc.capacity(0.625, 64, 2, 4) == 20               # the adv12 Q2 capacity
    assert orc.capacity(0.0, 100, 2, 4) == 100
    assert orc.capacity(-1.0, 100, 2, 4) == 100
    assert orc.capacity(1.0, 10, 1, 3) == 4                  # ceil(3.33)
    assert orc.capacity(1e-9, 10, 1, 3) == 1                 # clipped below
    assert orc.capacity(100.0, 10, 2, 4) == 10               # clipped above


def test_load_report_printed_example(golden):
    g = golden("eplb_adv12.json")
    r = orc.load_report(np.array(g["loads"], np.int32), g["devices"])
    assert r["assign"].tolist() == g["lpt_assignment"]
    assert r["dev_load"].tolist() == g["lpt_device_load"]
    assert r["naive_load"].tolist() == g["naive_device_load"]
    assert r["var_naive"] == g["naive_variance"]
    assert r["var_lpt"] == g["lpt_variance"]
    assert round(r["imbalance"], 3) == g["imbalance_3dp"]
    assert max(r["dev_load"]) == g["optimum_makespan"]


@pytest.mark.parametrize("seed", range(12))
def test_lpt_four_thirds_bound(seed):
    """LPT makespan <= (4/3 - 1/(3D)) * optimum (Graham), optimum by brute force."""
    rng = np.random.default_rng(seed)
    E = int(rng.integers(2, 9))
    D = int(rng.integers(2, 4))
    loads = rng.integers(0, 50, E).astype(np.int32)
    r = orc.load_report(loads, D)
    opt = min(max(sum(int(loads[e]) for e in range(E) if a[e] == dv) for dv in range(D))
              for a in itertools.product(range(D), repeat=E))
    assert max(r["dev_load"]) <= (4 / 3 - 1 / (3 * D)) * opt + 1e-9
    assert int(r["dev_load"].sum()) == int(loads.sum())
    # greedy rule: each expert went to a least-loaded device at its turn
    order = sorted(range(E), key=lambda e: (-loads[e], e))
    dl = [0] * D
    for e in order:
        dv = dl.index(min(dl))
        assert r["assign"][e] == dv
        dl[dv] += int(loads[e])


# --------------------------------------------------------------------------
# closed forms and special cases
# --------------------------------------------------------------------------

def test_gelu_and_silu_closed_forms(golden):
    g = golden("normal_cdf_table.json")
    for xs, phi in g["phi"].items():
        x = float(xs)
        assert abs(orc.gelu(x) - x * phi) < 1e-15 * max(1, abs(x)) + 1e-16
    lg = g["logistic"]
    for xs, s in lg.items():
        if xs == "source":
            continue
        x = float(xs)
        assert abs(orc.silu(x) - x * s) < 1e-15
    assert orc.silu(40.0) == pytest.approx(40.0, rel=1e-15)
    assert abs(orc.silu(-40.0)) < 1e-15


def test_bf16_rounding_cases():
    assert orc.bf16_round(1.0) == 0x3F80
    assert orc.bf16_round(-2.0) == 0xC000
    assert orc.bf16_round(1 + 2 ** -8) == 0x3F80            # tie -> even (down)
    assert orc.bf16_round(1 + 3 * 2 ** -8) == 0x3F82        # tie -> even (up)
    assert orc.bf16_round(1 + 2 ** -8 + 2 ** -30) == 0x3F81  # just above the tie
    assert orc.bf16_round(0.0) == 0x0000
    assert orc.bf16_round(-0.0) == 0x8000
    assert orc.bf16_round(3.0e38) == 0x7F62                   # 3.0e38 -> 0x7F62 (2.997e38..)
    assert orc.bf16_round(1e39) == 0x7F80                     # overflow -> inf
    assert orc.bf16_round(2.0 ** -133) == 0x0001              # smallest subnormal


def test_k1_weight_is_exactly_one():
    """Switch routing (k = 1): the renormalised weight is exactly 1."""
    rng = np.random.default_rng(3)
    logits = rng.normal(size=(50, 16)).astype(np.float32)
    idx, w = orc.topk_renorm(logits, 1)
    assert (w == 1.0).all()
    assert (idx[:, 0] == logits.argmax(axis=1)).all()


def test_zero_gate_ties_to_lower_ids():
    logits = np.zeros((5, 8), np.float32)
    idx, w = orc.topk_renorm(logits, 3)
    assert (idx == np.array([0, 1, 2])).all()
    assert np.allclose(w, 1 / 3, atol=1e-7)
    # -0.0 and +0.0 compare equal: still ties toward the lower id
    logits[:, 0] = -0.0
    idx, _ = orc.topk_renorm(logits, 2)
    assert (idx == np.array([0, 1])).all()


def test_ties_mixed_with_larger_values():
    logits = np.array([[1.0, 3.0, 3.0, 2.0, 3.0]], np.float32)
    idx, w = orc.topk_renorm(logits, 4)
    assert idx[0].tolist() == [1, 2, 4, 3]
    assert w[0, 0] == w[0, 1] == w[0, 2]


def test_weights_sum_to_one_and_order():
    rng = np.random.default_rng(4)
    logits = (rng.normal(size=(200, 32)) * 3).astype(np.float32)
    idx, w = orc.topk_renorm(logits, 8)
    assert np.allclose(w.astype(np.float64).sum(axis=1), 1.0, atol=2e-6)
    assert (np.diff(w, axis=1) <= 0).all()            # slot order = descending logit
    for t in range(200):
        ref = sorted(range(32), key=lambda e: (-logits[t, e], e))[:8]
        assert idx[t].tolist() == ref


def test_textbook_ffn_single_token():
    """1 token, 1 expert, no capacity: the layer is that expert's FFN."""
    for kind in (orc.GELU, orc.SWIGLU):
        x, Wg, W = small_problem(kind, 1, 16, 1, 1, 8, seed=5, bf16=True)
        r = run_oracle(kind, x, Wg, None, W, 1, 8)
        ref = dense_expert(kind, as_f64(x), W["w1"][0], None, W["w2"][0], None, 8)
        assert np.allclose(bf16_bits_to_f64(r["out"]), f64_to_bf16_value(ref), rtol=0, atol=0)


def test_swiglu_gate_rows_come_first():
    """W1 rows [0,F) are the gate (inside silu), rows [F,2F) the up projection."""
    d, F = 1, 1
    x = np.array([1.0], np.float32)
    w1 = np.array([[1.0], [2.0]], np.float32)     # gate -> 1, up -> 2
    w2 = np.array([[1.0]], np.float32)
    y = orc.expert_row(orc.SWIGLU, x, w1, None, w2, None, d, F)
    s1 = 1 / (1 + math.exp(-1.0))
    assert abs(y[0] - 1.0 * s1 * 2.0) < 1e-15     # silu(1)*2, not silu(2)*1


def test_expert_biases_enter_where_stated():
    d, F = 2, 2
    x = np.array([0.0, 0.0], np.float32)
    w1 = np.zeros((F, d), np.float32)
    b1 = np.array([1.0, -1.0], np.float32)
    w2 = np.eye(2, dtype=np.float32)
    b2 = np.array([0.5, 0.25], np.float32)
    y = orc.expert_row(orc.GELU, x, w1, b1, w2, b2, d, F)
    assert np.allclose(y, [orc.gelu(1.0) + 0.5, orc.gelu(-1.0) + 0.25], atol=1e-15)
    y = orc.expert_row(orc.LINEAR, x, np.eye(2, dtype=np.float32), b1, None, None, d, F)
    assert np.allclose(y, b1, atol=0)


def test_gate_logits_bruteforce():
    x = rand((7, 24), 9, 1, 1.0, True)
    Wg = rand((24, 5), 9, 2, 0.2)
    gb = rand((5,), 9, 3, 1.0)
    L = orc.gate_logits(x, Wg, gb)
    ref = bf16_bits_to_f64(x) @ Wg.astype(np.float64) + gb
    assert np.array_equal(L, ref.astype(np.float32))
    Lr = orc.gate_logits(x, Wg, gb, rows=[6, 2])
    assert np.array_equal(Lr, L[[6, 2]])


# --------------------------------------------------------------------------
# brute force on tiny inputs
# --------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(6))
def test_dispatch_bruteforce(seed):
    rng = np.random.default_rng(100 + seed)
    T, E = int(rng.integers(1, 40)), int(rng.integers(1, 9))
    k = int(rng.integers(1, E + 1))
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    cap = int(rng.integers(1, T + 1))
    counts, offsets, pt, ps, sd = orc.dispatch(idx, E, cap)
    pos = 0
    for e in range(E):
        assert offsets[e] == pos
        hits = [(t, j) for t in range(T) for j in range(k) if idx[t, j] == e]
        kept, dropped = hits[:cap], hits[cap:]
        assert counts[e] == len(kept)
        for r, (t, j) in enumerate(kept):
            assert pt[pos + r] == t and ps[pos + r] == j and sd[t, j] == pos + r
        for (t, j) in dropped:
            assert sd[t, j] == -1
        pos += len(kept)
    assert offsets[E] == pos == counts.sum()
    assert counts.sum() == np.minimum(orc.load(idx, E), cap).sum()


@pytest.mark.parametrize("kind", [orc.LINEAR, orc.GELU, orc.SWIGLU])
@pytest.mark.parametrize("k", [1, 2, 3])
def test_dense_bruteforce_equals_sparse(kind, k):
    """Dense sum over all experts masked by the renormalised routing weights
    equals the oracle's sparse top-k path (no capacity limit)."""
    T, d, E, F = 9, 16, 4, 8
    bf16 = kind != orc.LINEAR
    x, Wg, W = small_problem(kind, T, d, E, k, F, seed=20 + k + 3 * kind, bf16=bf16,
                             biases=True)
    gb = rand((E,), 21, 3, 0.5)
    r = run_oracle(kind, x, Wg, gb, W, k, F)
    ref, M = dense_forward(kind, x, Wg, gb, W, k, F)
    w_dense = np.take_along_axis(M, r["idx"].astype(np.int64), axis=1)
    assert np.allclose(r["w"], w_dense, atol=2e-7)
    got = as_f64(r["out"])
    if bf16:
        assert np.abs(got - ref).max() <= 2 ** -7 * np.abs(ref).max()
    else:
        assert np.allclose(got, ref, rtol=1e-6, atol=1e-6)


def test_k_equals_E_is_dense_softmax_mixture():
    T, d, E, F = 6, 8, 4, 8
    x, Wg, W = small_problem(orc.LINEAR, T, d, E, E, F, seed=31, bf16=False, biases=True)
    r = run_oracle(orc.LINEAR, x, Wg, None, W, E, F)
    X = x.astype(np.float64)
    L = (X @ Wg.astype(np.float64)).astype(np.float32).astype(np.float64)
    P = np.exp(L - L.max(1, keepdims=True))
    P /= P.sum(1, keepdims=True)
    ref = sum(P[:, [e]] * (X @ W["w1"][e].astype(np.float64).T + W["b1"][e]) for e in range(E))
    assert np.allclose(r["out"], ref, rtol=1e-6, atol=1e-6)
    assert all(sorted(row) == list(range(E)) for row in r["idx"].tolist())


def test_shared_expert_weight_one_and_residual():
    T, d, E, k, F = 5, 16, 3, 2, 8
    x, Wg, W = small_problem(orc.SWIGLU, T, d, E, k, F, seed=41, bf16=True, shared=True)
    r = run_oracle(orc.SWIGLU, x, Wg, None, W, k, F, add_residual=True)
    ref, _ = dense_forward(orc.SWIGLU, x, Wg, None, W, k, F, add_residual=True)
    assert np.abs(as_f64(r["out"]) - ref).max() <= 2 ** -7 * np.abs(ref).max()


def test_dropped_tokens_pass_through_unchanged():
    """With the residual on, a token whose every slot overflowed outputs x bit-exactly."""
    T, d, E, k, F = 40, 64, 2, 1, 64
    x, Wg, W = small_problem(orc.GELU, T, d, E, k, F, seed=51, bf16=True)
    gb = np.array([5.0, -5.0], np.float32)                # everyone wants expert 0
    r = run_oracle(orc.GELU, x, Wg, gb, W, k, F, cf=0.25, add_residual=True)
    cap = orc.capacity(0.25, T, k, E)
    assert cap == 5
    dropped = (r["slot_dest"] < 0).all(axis=1)
    assert dropped.sum() >= T - 2 * cap
    assert np.array_equal(r["out"][dropped], x[dropped])
    assert not np.array_equal(r["out"][~dropped], x[~dropped])


def test_load_sums_to_T_times_k():
    rng = np.random.default_rng(8)
    for _ in range(5):
        T, E = int(rng.integers(1, 300)), int(rng.integers(1, 40))
        k = int(rng.integers(1, E + 1))
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        assert orc.load(idx, E).sum() == T * k


# --------------------------------------------------------------------------
# group-limited routing ["MoE 并行" 通信瓶颈 table, Hierarchical Routing: groups
# first, then experts; adv12 section 5: each token's experts on at most M devices]
# --------------------------------------------------------------------------

def _brute_grouped(L, k, n_group, topk_group):
    """Enumerate every choice of topk_group groups and every k-subset of their experts.
    The chosen groups are the subset whose (group best logit, -group id) pairs, sorted
    descending, are lexicographically largest; the experts are the k-subset of those
    groups' experts whose (logit, -id) pairs, sorted descending, are largest."""
    E = L.shape[0]
    gs = E // n_group
    gkey = [(float(L[g * gs:(g + 1) * gs].max()), -g) for g in range(n_group)]
    best_groups = max(itertools.combinations(range(n_group), topk_group),
                      key=lambda c: sorted((gkey[g] for g in c), reverse=True))
    cand = [e for e in range(E) if e // gs in best_groups]
    best = max(itertools.combinations(cand, k),
               key=lambda c: sorted(((float(L[e]), -e) for e in c), reverse=True))
    return sorted(best, key=lambda e: (-float(L[e]), e))


@pytest.mark.parametrize("seed", range(6))
def test_grouped_topk_equals_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    for E, n_group, topk_group, k in ((8, 4, 2, 3), (12, 3, 1, 2), (8, 2, 1, 4), (12, 4, 3, 5)):
        # a coarse grid of values makes ties (within and across groups) common
        L = (rng.integers(-4, 5, size=(6, E)) / 4.0).astype(np.float32)
        idx, w = orc.topk_renorm(L, k, n_group, topk_group)
        for t in range(L.shape[0]):
            assert list(idx[t]) == _brute_grouped(L[t], k, n_group, topk_group)
            ex = np.exp(L[t, idx[t]].astype(np.float64) - L[t, idx[t][0]])
            assert np.allclose(w[t], ex / ex.sum(), rtol=1e-6, atol=0)


@pytest.mark.parametrize("E,k,n_group,topk_group", [
    (16, 3, 1, 1),     # one group holds every expert
    (16, 3, 4, 4),     # every group kept
    (16, 3, 16, 3),    # groups of one expert, as many groups kept as experts needed
    (32, 8, 32, 12),
])
def test_grouped_topk_reduces_to_plain_topk(E, k, n_group, topk_group):
    rng = np.random.default_rng(E + k)
    L = rng.standard_normal((50, E)).astype(np.float32)
    a = orc.topk_renorm(L, k, n_group, topk_group)
    b = orc.topk_renorm(L, k)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_grouped_topk_worked_example():
    # Four groups of two experts, keep two groups, top 3. Group best logits are
    # 0.9 (g0), 0.85 (g1), 0.86 (g2), 0.2 (g3), so groups 0 and 2 are kept and the
    # third expert is 1 (0.1, lower id than expert 5 at 0.1) - not expert 2 (0.85),
    # which plain top-3 would take. (Derived by hand from the two steps above.)
    L = np.array([[0.9, 0.1, 0.85, 0.84, 0.86, 0.1, 0.2, 0.1]], np.float32)
    idx, _ = orc.topk_renorm(L, 3, 4, 2)
    assert idx[0].tolist() == [0, 4, 1]
    assert orc.topk_renorm(L, 3)[0][0].tolist() == [0, 4, 2]


def test_grouped_topk_keeps_experts_within_the_chosen_groups():
    rng = np.random.default_rng(7)
    E, k, n_group, topk_group = 256, 8, 8, 4
    L = rng.standard_normal((200, E)).astype(np.float32)
    idx, _ = orc.topk_renorm(L, k, n_group, topk_group)
    gs = E // n_group
    for t in range(200):
        groups = set(int(e) // gs for e in idx[t])
        assert len(groups) <= topk_group
        gbest = L[t].reshape(n_group, gs).max(axis=1)
        chosen_min = min(gbest[g] for g in groups)
        # every group with a better best logit than the weakest chosen group is used
        # or was out-competed inside the chosen groups: its best expert is not above the
        # k-th kept logit
        kth = L[t, idx[t][-1]]
        for g in range(n_group):
            if g not in groups and gbest[g] > chosen_min:
                assert gbest[g] <= kth


# --------------------------------------------------------------------------
# weight-only INT8 experts ["MoE 混合专家架构" 5.3 量化支持: expert weights in INT8 / INT4]
# reading: one symmetric absmax scale per weight row, s = max|w| / 127, q = rne(w / s)
# --------------------------------------------------------------------------

def _bf16_bits(values):
    f = np.asarray(values, np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def test_quantize_rows_on_the_grid_are_exact():
    # rows whose entries are integers m times a power of two, with max |m| = 127: the
    # scale is that power of two and the codes are the integers themselves
    rng = np.random.default_rng(1)
    m = rng.integers(-127, 128, size=(6, 40))
    m[:, 3] = 127 * np.array([1, -1, 1, -1, 1, -1])
    scales = 2.0 ** np.array([-7, -3, 0, 2, -12, -1])
    w = _bf16_bits(m * scales[:, None])
    q, s = orc.quantize_rows_i8(w)
    assert np.array_equal(s, scales.astype(np.float32))
    assert np.array_equal(q.astype(np.int64), m)


def test_quantize_rows_bound_max_and_zero_row():
    rng = np.random.default_rng(2)
    vals = rng.standard_normal((50, 64)).astype(np.float32) * rng.uniform(0.01, 10, (50, 1))
    vals[7] = 0.0
    w = _bf16_bits(vals)
    wf = bf16_bits_to_f64(w)
    q, s = orc.quantize_rows_i8(w)
    assert s[7] == 0.0 and not q[7].any()
    for r in range(50):
        if r == 7:
            continue
        amax = np.abs(wf[r]).max()
        assert s[r] == np.float32(np.float32(amax) / np.float32(127.0))
        assert np.abs(q[r]).max() == 127                 # the largest entry maps to +-127
        err = np.abs(wf[r] - s[r].astype(np.float64) * q[r])
        # nearest code, up to the fp32 rounding of w / s (half an ulp of a value below 128)
        assert (err <= s[r] * (0.5 + 2.0 ** -17)).all()


def test_quantize_rows_ties_go_to_even():
    # scale 2^-6 (the row holds 127 * 2^-6); 2.5 * 2^-6 and 3.5 * 2^-6 lie halfway between codes
    w = _bf16_bits([[127 * 2.0 ** -6, 2.5 * 2.0 ** -6, 3.5 * 2.0 ** -6, -2.5 * 2.0 ** -6]])
    q, s = orc.quantize_rows_i8(w)
    assert s[0] == 2.0 ** -6
    assert q[0].tolist() == [127, 2, 4, -2]


@pytest.mark.parametrize("kind,F", [(orc.GELU, 48), (orc.SWIGLU, 32)])
def test_int8_expert_equals_bf16_expert_on_exactly_representable_weights(kind, F):
    # power-of-two scales: every s * q is a bf16 value, so the INT8 expert must agree
    # bit for bit with the (pinned) bf16 expert given those weights
    rng = np.random.default_rng(kind + F)
    d = 24
    N1 = F if kind == orc.GELU else 2 * F
    q1 = rng.integers(-127, 128, (N1, d)).astype(np.int8)
    q2 = rng.integers(-127, 128, (d, F)).astype(np.int8)
    s1 = (2.0 ** rng.integers(-12, -4, N1)).astype(np.float32)
    s2 = (2.0 ** rng.integers(-12, -4, d)).astype(np.float32)
    b1 = rng.standard_normal(N1).astype(np.float32)
    b2 = rng.standard_normal(d).astype(np.float32)
    w1 = _bf16_bits(s1[:, None] * q1.astype(np.float32))
    w2 = _bf16_bits(s2[:, None] * q2.astype(np.float32))
    assert np.array_equal(bf16_bits_to_f64(w1), s1[:, None].astype(np.float64) * q1)
    for t in range(4):
        x = _bf16_bits(rng.standard_normal(d))
        a = orc.expert_row_q8(kind, x, q1, s1, b1, q2, s2, b2, d, F)
        b = orc.expert_row(kind, x, w1, b1, w2, b2, d, F)
        assert np.array_equal(a, b)


# --------------------------------------------------------------------------
# weight-only INT4 experts (same page and section): s = max|w| / 7, q = rne(w / s) in
# [-7, 7], two codes per byte (even column in the low nibble, 4-bit two's complement)
# --------------------------------------------------------------------------

def test_int4_packing_worked_example():
    # max 7 -> s = 1; 3.5 and 2.5 are ties (to 4 and 2), -2.5 and -3.5 too (to -2 and -4)
    w = _bf16_bits([[7.0, -7.0, 1.0, -2.0, 3.5, 2.5, 0.0, 6.0, -2.5, -3.5]])
    packed, s = orc.quantize_rows_i4(w)
    assert s[0] == 1.0
    # codes 7,-7 | 1,-2 | 4,2 | 0,6 | -2,-4 as (low, high) nibbles
    assert packed[0].tolist() == [0x97, 0xE1, 0x24, 0x60, 0xCE]
    assert orc.unpack_i4(packed)[0].tolist() == [7, -7, 1, -2, 4, 2, 0, 6, -2, -4]


def test_int4_unpack_covers_every_nibble():
    # nibble v means v for v < 8 and v - 16 otherwise, low nibble first
    packed = np.arange(256, dtype=np.uint8).reshape(1, 256)
    q = orc.unpack_i4(packed)[0].astype(np.int64)
    v = np.arange(256)
    signed = lambda n: np.where(n < 8, n, n - 16)
    assert np.array_equal(q[0::2], signed(v & 15))
    assert np.array_equal(q[1::2], signed(v >> 4))


def test_int4_quantize_on_the_grid_is_exact():
    rng = np.random.default_rng(11)
    m = rng.integers(-7, 8, size=(6, 40))
    m[:, 5] = 7 * np.array([1, -1, 1, -1, 1, -1])
    scales = 2.0 ** np.array([-9, -3, 0, 3, -14, -1])
    w = _bf16_bits(m * scales[:, None])
    packed, s = orc.quantize_rows_i4(w)
    assert packed.shape == (6, 20)
    assert np.array_equal(s, scales.astype(np.float32) * np.float32(1.0))
    assert np.array_equal(orc.unpack_i4(packed).astype(np.int64), m)


def test_int4_quantize_bound_max_and_zero_row():
    rng = np.random.default_rng(12)
    vals = rng.standard_normal((50, 64)).astype(np.float32) * rng.uniform(0.01, 10, (50, 1))
    vals[9] = 0.0
    w = _bf16_bits(vals)
    wf = bf16_bits_to_f64(w)
    packed, s = orc.quantize_rows_i4(w)
    q = orc.unpack_i4(packed)
    assert s[9] == 0.0 and not packed[9].any()
    assert q.min() >= -7 and q.max() <= 7             # -8 is never produced
    for r in range(50):
        if r == 9:
            continue
        amax = np.abs(wf[r]).max()
        assert s[r] == np.float32(np.float32(amax) / np.float32(7.0))
        assert np.abs(q[r]).max() == 7
        err = np.abs(wf[r] - s[r].astype(np.float64) * q[r])
        # nearest code in [-7, 7], up to the fp32 rounding of w / s (|w / s| < 8)
        assert (err <= s[r] * (0.5 + 2.0 ** -20)).all()


@pytest.mark.parametrize("kind,F", [(orc.GELU, 48), (orc.SWIGLU, 32)])
def test_int4_expert_equals_bf16_expert_on_exactly_representable_weights(kind, F):
    # the INT4 expert is the INT8 expert on the unpacked codes; with power-of-two scales
    # every s * q is a bf16 value and the result equals the bf16 expert's bit for bit
    rng = np.random.default_rng(100 + kind + F)
    d = 24
    N1 = F if kind == orc.GELU else 2 * F
    m1 = rng.integers(-7, 8, (N1, d))
    m2 = rng.integers(-7, 8, (d, F))
    m1[:, 0] = 7 * rng.choice([-1, 1], N1)     # every row reaches 7: the scale is s itself
    m2[:, 0] = 7 * rng.choice([-1, 1], d)
    s1 = (2.0 ** rng.integers(-9, -2, N1)).astype(np.float32)
    s2 = (2.0 ** rng.integers(-9, -2, d)).astype(np.float32)
    w1 = _bf16_bits(s1[:, None] * m1)
    w2 = _bf16_bits(s2[:, None] * m2)
    p1, t1 = orc.quantize_rows_i4(w1)
    p2, t2 = orc.quantize_rows_i4(w2)
    q1, q2 = orc.unpack_i4(p1), orc.unpack_i4(p2)
    assert np.array_equal(t1[:, None].astype(np.float64) * q1, s1[:, None].astype(np.float64) * m1)
    assert np.array_equal(t2[:, None].astype(np.float64) * q2, s2[:, None].astype(np.float64) * m2)
    b1 = rng.standard_normal(N1).astype(np.float32)
    b2 = rng.standard_normal(d).astype(np.float32)
    for t in range(4):
        x = _bf16_bits(rng.standard_normal(d))
        a = orc.expert_row_q8(kind, x, q1, t1, b1, q2, t2, b2, d, F)
        b = orc.expert_row(kind, x, w1, b1, w2, b2, d, F)
        assert np.array_equal(a, b)


# --------------------------------------------------------------------------
# overflow variants: re-routing to the next-ranked expert, overflow weight to the
# shared expert ("MoE 并行" 推理时的负载均衡 and Q4; adv12 Q2)
# --------------------------------------------------------------------------

def _random_logits(T, E, seed, hot=()):
    L = rand((T, E), seed, 3, 1.0)
    for e in hot:
        L[:, e] += 2.0          # a few popular experts, so that capacity bites
    return np.ascontiguousarray(L, np.float32)


def test_rank_candidates_match_a_sort():
    L = _random_logits(40, 12, 5)
    L[3, 4] = L[3, 7]           # a tie: the lower id ranks first
    for k, m in ((1, 1), (2, 2), (3, 3), (5, 7)):
        cand = orc.rank_candidates(L, k, m)
        for t in range(40):
            order = sorted(range(12), key=lambda e: (-float(L[t, e]), e))
            want = (order[k:k + m] + [-1] * m)[:m]
            assert cand[t].tolist() == want
    # group-limited: only the chosen groups' experts are ranked
    n_group, topk_group, k = 4, 2, 2
    cand = orc.rank_candidates(L, k, 4, n_group, topk_group)
    gs = 12 // n_group
    for t in range(40):
        gscore = [max(float(L[t, e]) for e in range(g * gs, (g + 1) * gs)) for g in range(n_group)]
        groups = sorted(range(n_group), key=lambda g: (-gscore[g], g))[:topk_group]
        pool = [e for e in range(12) if e // gs in groups]
        order = sorted(pool, key=lambda e: (-float(L[t, e]), e))
        assert cand[t].tolist() == order[k:k + 4]           # 6 experts in the pool, 4 asked
        idx, _ = orc.topk_renorm(L[t:t + 1], k, n_group, topk_group)
        assert idx[0].tolist() == order[:k]                 # consistent with the top-k


def test_reroute_hand_example_top1():
    # four tokens all prefer expert 0 (capacity 1); their second choices are 1, 1, 2, 1.
    # Round 0 keeps token 0 on expert 0. Round 1: tokens 1 and 3 ask expert 1 (token 1
    # first in token order takes its only row), token 2 asks expert 2 (accepted).
    L = np.array([[3, 2, 1], [3, 2, 1], [3, 1, 2], [3, 2, 1]], np.float32)
    idx, _ = orc.topk_renorm(L, 1)
    cand = orc.rank_candidates(L, 1, 1)
    assert cand[:, 0].tolist() == [1, 1, 2, 1]
    counts, offsets, pt, ps, sd, ri = orc.dispatch_reroute(idx, cand, 3, 1)
    assert counts.tolist() == [1, 1, 1] and offsets.tolist() == [0, 1, 2, 3]
    assert pt.tolist() == [0, 1, 2] and ps.tolist() == [0, 0, 0]
    assert sd[:, 0].tolist() == [0, 1, 2, -1]
    assert ri[:, 0].tolist() == [0, 1, 2, 0]


def test_reroute_hand_example_two_dropped_slots():
    # E=4, k=2, capacity 1, every token ranks experts 0 > 1 > 2 > 3. Token 0 keeps 0 and
    # 1; tokens 1 and 2 drop both slots. Round 1: slot 0 of a token asks its third-ranked
    # expert (2), slot 1 its fourth (3); token 1 gets both rows, token 2 is rejected.
    L = np.tile(np.array([[4, 3, 2, 1]], np.float32), (3, 1))
    idx, _ = orc.topk_renorm(L, 2)
    cand = orc.rank_candidates(L, 2, 2)
    assert cand.tolist() == [[2, 3]] * 3
    counts, offsets, pt, ps, sd, ri = orc.dispatch_reroute(idx, cand, 4, 1)
    assert counts.tolist() == [1, 1, 1, 1]
    assert pt.tolist() == [0, 0, 1, 1] and ps.tolist() == [0, 1, 0, 1]
    assert sd.tolist() == [[0, 1], [2, 3], [-1, -1]]
    assert ri.tolist() == [[0, 1], [2, 3], [0, 1]]


def test_reroute_cannot_create_capacity_printed_loads():
    # adv12 Q2 / section 3.2: loads [38, 34, 29, 27] at capacity 20. Every expert is over
    # capacity, so no re-routed slot finds room: 80 rows kept, 18 + 14 + 9 + 7 = 48 dropped.
    loads = [38, 34, 29, 27]
    idx = np.concatenate([np.full(n, e, np.int32) for e, n in enumerate(loads)])
    rng = np.random.default_rng(0)
    idx = rng.permutation(idx).reshape(-1, 1)
    T = idx.shape[0]
    L = np.zeros((T, 4), np.float32)
    L[np.arange(T), idx[:, 0]] = 1.0
    cand = orc.rank_candidates(L, 1, 1)
    counts, offsets, pt, ps, sd, ri = orc.dispatch_reroute(idx, cand, 4, 20)
    assert counts.tolist() == [20, 20, 20, 20]
    assert int((sd < 0).sum()) == 48
    c0, o0, pt0, ps0, sd0 = orc.dispatch(idx, 4, 20)
    assert np.array_equal(sd, sd0) and np.array_equal(pt, pt0)


def test_reroute_without_capacity_is_plain_dispatch():
    L = _random_logits(60, 8, 7, hot=(1, 2))
    for k in (1, 2, 3):
        idx, _ = orc.topk_renorm(L, k)
        cand = orc.rank_candidates(L, k, k)
        r = orc.dispatch_reroute(idx, cand, 8, 60)
        p = orc.dispatch(idx, 8, 60)
        for a, b in zip(r[:5], p):
            assert np.array_equal(a, b)
        assert np.array_equal(r[5], idx)


@pytest.mark.parametrize("T,E,k,cap,seed", [(200, 16, 4, 40, 1), (300, 8, 1, 30, 2),
                                            (150, 32, 8, 30, 3), (64, 6, 3, 20, 4)])
def test_reroute_invariants(T, E, k, cap, seed):
    L = _random_logits(T, E, seed, hot=(0, 3 % E))
    idx, _ = orc.topk_renorm(L, k)
    cand = orc.rank_candidates(L, k, k)
    counts, offsets, pt, ps, sd, ri = orc.dispatch_reroute(idx, cand, E, cap)
    c0, o0, pt0, ps0, sd0 = orc.dispatch(idx, E, cap)
    P = int(offsets[E])
    assert (counts <= cap).all() and P == int(counts.sum())
    assert P >= int(c0.sum())                                # never fewer rows than dropping
    kept0 = sd0 >= 0
    assert ((sd >= 0) | ~kept0).all()                       # round-0 rows stay
    assert np.array_equal(ri[kept0], idx[kept0])
    proposals = {}
    for t in range(T):
        m = 0
        for j in range(k):
            if kept0[t, j]:
                continue
            want = int(cand[t, m])
            m += 1
            if sd[t, j] >= 0:
                assert ri[t, j] == want                     # re-routed to its next candidate
            else:
                assert ri[t, j] == idx[t, j]
            if want >= 0:
                proposals.setdefault(want, []).append((t, j, sd[t, j] >= 0))
        kept_e = [int(ri[t, j]) for j in range(k) if sd[t, j] >= 0]
        assert len(kept_e) == len(set(kept_e))              # a token meets an expert once
    for e, props in proposals.items():
        accepted = [a for (_, _, a) in props]
        # accepted in token order while there is room: a prefix, as long as the room
        n_acc = sum(accepted)
        assert accepted == [True] * n_acc + [False] * (len(props) - n_acc)
        assert n_acc == min(len(props), cap - int(c0[e]))
    # rows of each expert: round-0 rows in token order, then round-1 rows in token order
    for e in range(E):
        rows = list(zip(pt[offsets[e]:offsets[e + 1]], ps[offsets[e]:offsets[e + 1]]))
        r0 = [(t, j) for (t, j) in rows if kept0[t, j]]
        r1 = [(t, j) for (t, j) in rows if not kept0[t, j]]
        assert rows == r0 + r1 and r0 == sorted(r0) and r1 == sorted(r1)
    for t in range(T):
        for j in range(k):
            if sd[t, j] >= 0:
                assert pt[sd[t, j]] == t and ps[sd[t, j]] == j


def test_overflow_to_shared_expert():
    kind, T, d, E, k, F = orc.LINEAR, 24, 8, 4, 2, 8
    x, Wg, W = small_problem(kind, T, d, E, k, F, seed=9, bf16=False, shared=True)
    gb = np.array([3.0, 0, 0, 0], np.float32)        # expert 0 is every token's first choice
    sh = W["shared"]
    W["shared"] = (sh[0], rand((d,), 9, 9, 0.1), None, None)
    common = dict(cf=0.5, add_residual=True, shared=W["shared"])
    r0 = orc.forward(kind, x, Wg, gb, W["w1"], W["b1"], None, None, k, F, overflow=0, **common)
    r1 = orc.forward(kind, x, Wg, gb, W["w1"], W["b1"], None, None, k, F, overflow=1, **common)
    assert np.array_equal(r0["slot_dest"], r1["slot_dest"])
    dropped = r0["slot_dest"] < 0
    assert dropped.any() and dropped.all(axis=1).any()
    X = x.astype(np.float64)
    S = X @ W["shared"][0].astype(np.float64).T + W["shared"][1].astype(np.float64)
    a = (r0["w"].astype(np.float64) * dropped).sum(axis=1, keepdims=True)
    # the dropped weight multiplies the shared expert: out1 - out0 = a * S
    diff = r1["out"].astype(np.float64) - r0["out"].astype(np.float64)
    tol = 4e-7 * (np.abs(r0["out"]).astype(np.float64) + np.abs(a * S) + 1e-6)
    assert (np.abs(diff - a * S) <= tol).all()
    # a fully dropped token: its weights sum to 1, so it leaves as x + 2 * S(x)
    full = dropped.all(axis=1)
    want = X[full] + 2.0 * S[full]
    assert np.allclose(r1["out"][full], want, rtol=2e-6, atol=1e-6)
    # without capacity nothing is dropped and the variants agree bit for bit
    r0n = orc.forward(kind, x, Wg, gb, W["w1"], W["b1"], None, None, k, F, overflow=0,
                      add_residual=True, shared=W["shared"])
    r1n = orc.forward(kind, x, Wg, gb, W["w1"], W["b1"], None, None, k, F, overflow=1,
                      add_residual=True, shared=W["shared"])
    assert np.array_equal(r0n["out"], r1n["out"])


def test_reroute_forward_matches_dense_mixture_of_processing_experts():
    # the forward with re-routing equals a dense sum over experts where each kept slot's
    # weight sits on the expert that processes it (route_idx)
    kind, T, d, E, k, F = orc.LINEAR, 40, 8, 6, 2, 8
    x, Wg, W = small_problem(kind, T, d, E, k, F, seed=13, bf16=False, biases=True)
    gb = np.array([2.0, 1.5, 0, 0, 0, 0], np.float32)
    r = orc.forward(kind, x, Wg, gb, W["w1"], W["b1"], None, None, k, F, cf=0.75, overflow=2)
    base = orc.forward(kind, x, Wg, gb, W["w1"], W["b1"], None, None, k, F, cf=0.75)
    assert int((r["slot_dest"] >= 0).sum()) > int((base["slot_dest"] >= 0).sum())
    X = x.astype(np.float64)
    M = np.zeros((T, E))
    for t in range(T):
        for j in range(k):
            if r["slot_dest"][t, j] >= 0:
                M[t, r["idx"][t, j]] += float(r["w"][t, j])
    out = np.zeros((T, d))
    for e in range(E):
        out += M[:, [e]] * (X @ W["w1"][e].astype(np.float64).T + W["b1"][e].astype(np.float64))
    assert np.allclose(r["out"], out, rtol=2e-6, atol=1e-6)
    assert np.array_equal(r["load"], base["load"])          # load is the raw top-k bincount
