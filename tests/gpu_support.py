"""Helpers for the GPU parity tests: run the CUDA path through the C ABI, run the
oracle on the same seeded inputs, and compare under the stated criteria.

Criteria (the layer's parity contract):
  * logits: |gpu - oracle| <= 1e-5 * (sum_i |x_i * Wg_ie| + |b_e|)
  * top-k ids, load, counts, offsets, permutation and drop masks: bit-exact, with
    the oracle fed the GPU's own fp32 logits
  * kept weights: |gpu - oracle| <= 2e-6
  * bf16 expert outputs: max|gpu - oracle| <= 2e-2 * max|oracle| and
    mean(|gpu - oracle| / (|oracle| + 1e-3 * max|oracle|)) <= 5e-3
  * fp32 (Linear experts) outputs: max|gpu - oracle| <= 1e-5 * max|oracle|
"""

import numpy as np
import torch

import oracle as orc
import top_routing_expert_renorm_b300 as moe


def bf16_to_f64(a):
    a = np.asarray(a)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_np(t):
    """torch tensor (any device) -> numpy; bf16 becomes uint16 bit patterns."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def as_f64(a):
    return bf16_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


class DeviceRun:
    """Inputs of a workload on the device and on the host, and the CUDA path's
    stage outputs (route, dispatch, expert FFN, combine) plus moe_forward."""

    def __init__(self, wl, device="cuda"):
        self.wl = wl
        self.dev = device
        self.inp = wl.device_inputs(device)
        self.cfg = moe.config_for(wl)

    def run(self, fp32_y=False):
        """fp32_y: also run moe_forward with fp32 expert-output rows (out_f32y), the
        format of the staged path (moe_forward's default rows are fp16 with a
        power-of-two scale per 32 columns)."""
        wl, inp, cfg = self.wl, self.inp, self.cfg
        T, E, k, d = wl.T, wl.E, wl.k, wl.d
        i32 = dict(dtype=torch.int32, device=self.dev)
        f32 = dict(dtype=torch.float32, device=self.dev)
        ws = torch.empty(moe.workspace_size(cfg), dtype=torch.uint8, device=self.dev)
        Pmax = T * k
        self.logits = torch.empty(T, E, **f32)
        self.idx = torch.empty(T, k, **i32)
        self.w = torch.empty(T, k, **f32)
        moe.route(cfg, inp["x"], inp["wg"], inp["gate_bias"], self.logits, self.idx, self.w, ws)
        self.load = torch.empty(E, **i32)
        self.counts = torch.empty(E, **i32)
        self.offsets = torch.empty(E + 1, **i32)
        self.perm_token = torch.full((Pmax,), -7, **i32)
        self.perm_slot = torch.full((Pmax,), -7, **i32)
        self.slot_dest = torch.empty(T, k, **i32)
        self.x_perm = torch.empty(Pmax, d, dtype=inp["x"].dtype, device=self.dev)
        moe.dispatch(cfg, self.idx, inp["x"], self.load, self.counts, self.offsets,
                     self.perm_token, self.perm_slot, self.slot_dest, self.x_perm, ws)
        if wl.int8 or wl.int4:
            # INT8 / INT4 experts: codes and row scales from the library's quantiser
            bits = 8 if wl.int8 else 4
            self.q = moe.quantize_weights(inp["w1"], inp["w2"], bits=bits)
            routed = moe.weights(self.q[0], inp["b1"], self.q[2], inp["b2"], self.q[1], self.q[3])
            shared = None
            if inp["shared"] is not None:
                sw1, sb1, sw2, sb2 = inp["shared"]
                self.sq = moe.quantize_weights(sw1, sw2, bits=bits)
                shared = moe.weights(self.sq[0], sb1, self.sq[2], sb2, self.sq[1], self.sq[3])
        else:
            routed = moe.weights(inp["w1"], inp["b1"], inp["w2"], inp["b2"])
            shared = moe.weights(*inp["shared"]) if inp["shared"] is not None else None
        self.y = torch.empty(Pmax + (T if wl.has_shared else 0), d, **f32)
        moe.expert_ffn(cfg, self.x_perm, self.offsets, routed, shared, inp["x"], self.w,
                       self.perm_token, self.perm_slot, self.y, ws)
        self.out_stages = torch.empty_like(inp["x"])
        moe.combine(cfg, inp["x"], self.y, self.slot_dest, self.out_stages, topk_w=self.w)
        # the fused entry point on a fresh workspace
        ws2 = torch.empty_like(ws)
        self.out = torch.empty_like(inp["x"])
        self.idx_f = torch.empty(T, k, **i32)
        self.w_f = torch.empty(T, k, **f32)
        self.load_f = torch.empty(E, **i32)
        moe.forward(cfg, inp["x"], inp["wg"], inp["gate_bias"], routed, shared, self.out, ws2,
                    topk_idx=self.idx_f, topk_w=self.w_f, load=self.load_f)
        if fp32_y:
            cfg32 = moe.config_for(wl)
            cfg32.y_fp32 = 1
            self.out_f32y = torch.empty_like(inp["x"])
            moe.forward(cfg32, inp["x"], inp["wg"], inp["gate_bias"], routed, shared,
                        self.out_f32y, torch.empty_like(ws))
        st = moe.last_device_status()
        assert st == 0, f"device status {moe.status_string(st)}"
        torch.cuda.synchronize()
        return self


# ---- comparisons --------------------------------------------------------------------

def check_logits(wl, x_host, rows, L_gpu_rows):
    Wg = wl.wg_host()
    gb = wl.gate_bias_host()
    L_ref = orc.gate_logits(x_host, Wg, gb, rows=rows)
    X = as_f64(x_host[rows])
    scale = np.abs(X) @ np.abs(Wg.astype(np.float64))
    if gb is not None:
        scale += np.abs(gb.astype(np.float64))
    err = np.abs(L_gpu_rows.astype(np.float64) - L_ref.astype(np.float64))
    worst = float((err / (scale + 1e-30)).max())
    assert (err <= 1e-5 * scale + 1e-30).all(), f"logit error {worst:.3e} of scale"
    return worst


def check_routing(r):
    """idx bit-exact and w within 2e-6 against the oracle fed the GPU logits."""
    L = to_np(r.logits)
    idx_ref, w_ref = orc.topk_renorm(L, r.wl.k, r.wl.n_group, r.wl.topk_group)
    idx = to_np(r.idx)
    assert np.array_equal(idx, idx_ref), f"{(idx != idx_ref).sum()} top-k ids differ"
    w = to_np(r.w)
    assert np.abs(w - w_ref).max() <= 2e-6
    assert np.array_equal(to_np(r.idx_f), idx_ref)
    assert np.abs(to_np(r.w_f) - w_ref).max() <= 2e-6
    return idx_ref, w_ref


def check_dispatch(r, idx_ref):
    """Dispatch outputs bit-exact against the oracle fed the GPU's routing. Returns the
    capacity, slot_dest, P and the expert that processes each slot (re-routing moves
    dropped slots to the token's next-ranked experts)."""
    wl = r.wl
    cap = orc.capacity(np.float32(wl.cf), wl.T, wl.k, wl.E)
    assert moe.capacity(r.cfg) == cap
    if wl.overflow == "reroute":
        cand = orc.rank_candidates(to_np(r.logits), wl.k, wl.k, wl.n_group, wl.topk_group)
        counts, offsets, pt, ps, sd, route_idx = orc.dispatch_reroute(idx_ref, cand, wl.E, cap)
    else:
        counts, offsets, pt, ps, sd = orc.dispatch(idx_ref, wl.E, cap)
        route_idx = idx_ref
    ld = orc.load(idx_ref, wl.E)
    assert np.array_equal(to_np(r.load), ld)
    assert np.array_equal(to_np(r.load_f), ld)
    assert np.array_equal(to_np(r.counts), counts)
    assert np.array_equal(to_np(r.offsets), offsets)
    P = int(offsets[-1])
    assert np.array_equal(to_np(r.perm_token)[:P], pt)
    assert np.array_equal(to_np(r.perm_slot)[:P], ps)
    assert np.array_equal(to_np(r.slot_dest), sd)
    return cap, sd, P, route_idx


def _expert_fn(wl, e, shared=False):
    """Oracle expert of the workload: bf16 weights, or their INT8 / INT4 codes for quantised
    layers (INT4 codes unpacked from the oracle's own packing)."""
    w1, b1, w2, b2 = (wl.w1_host(e, shared), wl.b1_host(e, shared), wl.w2_host(e, shared),
                      wl.b2_host(e, shared))
    if wl.int8 or wl.int4:
        q1, s1 = (orc.quantize_rows_i8 if wl.int8 else orc.quantize_rows_i4)(w1)
        q2, s2 = (orc.quantize_rows_i8 if wl.int8 else orc.quantize_rows_i4)(w2)
        if wl.int4:
            q1, q2 = orc.unpack_i4(q1), orc.unpack_i4(q2)
        return lambda xr: orc.expert_row_q8(wl.kind_code, xr, q1, s1, b1, q2, s2, b2, wl.d, wl.F)
    return lambda xr: orc.expert_row(wl.kind_code, xr, w1, b1, w2, b2, wl.d, wl.F)


def check_quantized_weights(r, experts):
    """The library's INT8 / INT4 codes and scales equal the oracle's, bit for bit."""
    wl = r.wl
    q1, s1, q2, s2 = r.q
    quant = orc.quantize_rows_i8 if wl.int8 else orc.quantize_rows_i4
    for e in experts:
        oq1, os1 = quant(wl.w1_host(e))
        oq2, os2 = quant(wl.w2_host(e))
        assert np.array_equal(to_np(q1[e]), oq1) and np.array_equal(to_np(s1[e]), os1)
        assert np.array_equal(to_np(q2[e]), oq2) and np.array_equal(to_np(s2[e]), os2)


def expert_outputs(wl, requests, x_all):
    """Oracle expert outputs for requests {expert id or "shared": tokens}, one expert's
    weights in memory at a time. Returns {(expert, token): y[d] float64}."""
    out = {}
    for e in sorted(requests, key=str):
        fn = _expert_fn(wl, 0, True) if e == "shared" else _expert_fn(wl, e)
        for t in sorted(requests[e]):
            out[(e, t)] = fn(np.ascontiguousarray(x_all[t]))
        del fn
    return out


def oracle_rows(wl, x_all, rows, idx_ref, w_ref, sd, ys=None):
    """Oracle outputs for the given tokens, with routing fed from the GPU logits; idx_ref
    names the expert that processes each kept slot. ys: expert outputs computed already."""
    req = {}
    for t in rows:
        for j in range(wl.k):
            if sd[t, j] >= 0:
                req.setdefault(int(idx_ref[t, j]), set()).add(int(t))
        if wl.has_shared:
            req.setdefault("shared", set()).add(int(t))
    ys = dict(ys or {})
    missing = {e: {t for t in ts if (e, t) not in ys} for e, ts in req.items()}
    ys.update(expert_outputs(wl, {e: ts for e, ts in missing.items() if ts}, x_all))
    out = []
    for t in rows:
        xr = np.ascontiguousarray(x_all[t])
        yk = np.zeros((wl.k, wl.d))
        kept = (sd[t] >= 0).astype(np.int32)
        for j in range(wl.k):
            if kept[j]:
                yk[j] = ys[(int(idx_ref[t, j]), int(t))]
        ysh = ys[("shared", int(t))] if wl.has_shared else None
        out.append(orc.combine_row(xr, wl.add_residual, w_ref[t], kept, yk, ysh,
                                   orc.BF16 if wl.bf16 else orc.F32,
                                   overflow_to_shared=wl.overflow == "shared"))
    return np.stack(out)


def check_outputs(wl, got, ref):
    g, o = as_f64(got), as_f64(ref)
    mx = np.abs(o).max()
    err = np.abs(g - o)
    if wl.bf16:
        eps = 1e-3 * mx
        mean_rel = float((err / (np.abs(o) + eps)).mean())
        assert err.max() <= 2e-2 * mx, f"max err {err.max():.3e} vs {2e-2 * mx:.3e}"
        assert mean_rel <= 5e-3, f"mean relative error {mean_rel:.3e}"
        return float(err.max() / mx), mean_rel
    assert err.max() <= 1e-5 * mx, f"max err {err.max():.3e} vs {1e-5 * mx:.3e}"
    return float(err.max() / mx), 0.0


def targeted_tokens(r, idx_ref, route_idx, sd, n_total, seed):
    """Tokens where a tiled kernel is most likely to break, plus seeded random ones up to
    n_total: the tokens at rows 0, 127, 128, 255, 256 and the last row of a few experts'
    row blocks (first and last touched expert, the most loaded one, a middle one, and the
    first and last with more than one 128-row M tile), rows 0, 127, 128 and T-1 of the
    shared expert, capacity-dropped tokens and re-routed tokens. Also returns the
    targeted positions p of the permuted rows."""
    wl = r.wl
    offsets = to_np(r.offsets).astype(np.int64)
    pt = to_np(r.perm_token)
    counts = np.diff(offsets)
    touched = np.nonzero(counts)[0]
    picks = {int(touched[0]), int(touched[-1]), int(touched[np.argmax(counts[touched])]),
             int(touched[len(touched) // 2])}
    big = touched[counts[touched] > 128]
    if len(big):
        picks.update({int(big[0]), int(big[-1])})
    positions = []
    for e in sorted(picks):
        n = int(counts[e])
        for q in sorted({0, 127, 128, 255, 256, n - 1}):
            if 0 <= q < n:
                positions.append(int(offsets[e]) + q)
    tokens = {int(pt[p]) for p in positions}
    if wl.has_shared:
        tokens.update(t for t in (0, 127, 128, wl.T - 1) if 0 <= t < wl.T)
    rng = np.random.default_rng(seed)
    dropped = np.nonzero((sd < 0).any(axis=1))[0]
    if len(dropped):
        tokens.update(int(t) for t in rng.choice(dropped, size=min(2, len(dropped)), replace=False))
    full = np.nonzero((sd < 0).all(axis=1))[0]
    if len(full):
        tokens.add(int(full[0]))
    moved = np.nonzero(((route_idx != idx_ref) & (sd >= 0)).any(axis=1))[0]
    if len(moved):
        tokens.update(int(t) for t in rng.choice(moved, size=min(2, len(moved)), replace=False))
    rest = np.setdiff1d(np.arange(wl.T), np.fromiter(tokens, np.int64, len(tokens)))
    need = max(0, n_total - len(tokens))
    if need and len(rest):
        tokens.update(int(t) for t in rng.choice(rest, size=min(need, len(rest)), replace=False))
    return np.array(sorted(tokens), dtype=np.int64), np.array(positions, dtype=np.int64)


def check_expert_rows(r, positions, route_idx, w_ref, x_all, rows):
    """Rows of the staged expert output y (fp32, routing weight applied) at the given
    permuted positions, against the oracle expert times the slot's weight; and the shared
    expert's rows of the checked tokens. Returns the expert outputs it computed, plus those
    of every slot of `rows` (for the token-level check)."""
    wl = r.wl
    pt, ps = to_np(r.perm_token), to_np(r.perm_slot)
    sd = to_np(r.slot_dest)
    y = r.y.cpu().numpy()
    req = {}
    for p in positions:
        t, j = int(pt[p]), int(ps[p])
        req.setdefault(int(route_idx[t, j]), set()).add(t)
    for t in rows:
        for j in range(wl.k):
            if sd[t, j] >= 0:
                req.setdefault(int(route_idx[t, j]), set()).add(int(t))
    shared_rows = sorted({int(t) for t in rows})
    if wl.has_shared:
        req["shared"] = set(shared_rows)
    ys = expert_outputs(wl, req, x_all)
    got, ref = [], []
    for p in positions:
        t, j = int(pt[p]), int(ps[p])
        ref.append(ys[(int(route_idx[t, j]), t)] * float(w_ref[t, j]))
        got.append(y[p])
    if wl.has_shared:
        Pmax = wl.T * wl.k
        for t in shared_rows:
            ref.append(ys[("shared", t)])
            got.append(y[Pmax + t])
    check_outputs(wl, np.stack(got), np.stack(ref))
    return ys


def full_check(wl, sample=None, seed=0, targeted=False):
    """Run the CUDA path on `wl` and check it against the oracle.
    sample=None: every token; otherwise that many tokens (routing and dispatch are still
    checked in full): seeded random ones, or with targeted=True the tile-boundary,
    dropped and re-routed tokens of targeted_tokens() topped up with random ones, plus the
    staged expert-output rows at the targeted positions."""
    r = DeviceRun(wl).run()
    x_all = wl.x_host()
    idx_ref, w_ref = check_routing(r)
    cap, sd, P, route_idx = check_dispatch(r, idx_ref)
    positions = np.empty(0, np.int64)
    if sample is None or sample >= wl.T:
        rows = np.arange(wl.T)
    elif targeted:
        rows, positions = targeted_tokens(r, idx_ref, route_idx, sd, sample, seed)
    else:
        rng = np.random.default_rng(seed)
        rows = np.sort(rng.choice(wl.T, size=sample, replace=False))
    check_logits(wl, x_all, rows, to_np(r.logits)[rows])
    # gathered rows are exact copies
    xp = to_np(r.x_perm)[:P]
    pt = to_np(r.perm_token)[:P]
    chk = np.arange(0, P, max(1, P // 512))
    assert np.array_equal(xp[chk], x_all[pt[chk]])
    if wl.int8 or wl.int4:
        used = sorted({int(e) for e in idx_ref[rows].ravel()})
        check_quantized_weights(r, used[:8])
    ys = None
    if len(positions) and wl.kind != "linear":
        ys = check_expert_rows(r, positions, route_idx, w_ref, x_all, rows)
    ref = oracle_rows(wl, x_all, rows, route_idx, w_ref, sd, ys)
    stats = check_outputs(wl, to_np(r.out)[rows], ref)
    check_outputs(wl, to_np(r.out_stages)[rows], ref)
    r.checked_rows = rows
    return r, stats
