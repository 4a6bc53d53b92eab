"""Shared helpers of the parity tests: tolerance metrics and torch <-> oracle conversions.

Tolerances (stated for the layer): bf16 outputs within 2e-2 max-abs-relative and 1e-3
mean-relative of the oracle; outputs that read an FP8-e4m3 KV cache within 5e-2
max-abs-relative (mean-relative 2e-3, derived: the two sides quantise with the same rule and
differ only where an FP32 rounding difference flips an e4m3 code); router logits within 1e-5
relative, with the row's RMS as the floor of the denominator; selected expert indices
bit-exact (as sets; the order is by score).
"""
import numpy as np
import torch

import oracle as O

BF16_MAX_REL, BF16_MEAN_REL = 2e-2, 1e-3
FP8_MAX_REL, FP8_MEAN_REL = 5e-2, 2e-3
LOGIT_REL = 1e-5

# Every comparison made in the session: (test id, what, max-abs-rel, mean-rel, stated max bar,
# stated mean bar, kind) with kind "stated" (held to the stated bars) or "chained" (held to
# the widened bar of chained steps). conftest.py prints a summary at the end of the run.
LEDGER = []
CURRENT_TEST = [""]


def _record(what, mx, mn, lim_mx, lim_mn, kind):
    LEDGER.append((CURRENT_TEST[0], what, float(mx), float(mn), lim_mx, lim_mn, kind))


def np64(t):
    return t.detach().float().cpu().double().numpy()


def max_abs_rel(a, r):
    a, r = np.asarray(a, np.float64), np.asarray(r, np.float64)
    return float(np.max(np.abs(a - r)) / max(np.max(np.abs(r)), 1e-30))


def mean_rel(a, r):
    a, r = np.asarray(a, np.float64), np.asarray(r, np.float64)
    return float(np.mean(np.abs(a - r)) / max(np.mean(np.abs(r)), 1e-30))


def assert_close(a, r, what, fp8=False):
    mx, mn = max_abs_rel(a, r), mean_rel(a, r)
    lim_mx, lim_mn = (FP8_MAX_REL, FP8_MEAN_REL) if fp8 else (BF16_MAX_REL, BF16_MEAN_REL)
    print(f"{what}: max-abs-rel {mx:.3e} mean-rel {mn:.3e} (bars {lim_mx} / {lim_mn})")
    _record(what, mx, mn, lim_mx, lim_mn, "stated")
    assert np.all(np.isfinite(a)), f"{what}: non-finite output"
    assert mx <= lim_mx and mn <= lim_mn, \
        f"{what}: max-abs-rel {mx:.3e} (<= {lim_mx}), mean-rel {mn:.3e} (<= {lim_mn})"
    return mx, mn


def assert_logits_close(a, r, what="router logits"):
    a, r = np.asarray(a, np.float64), np.asarray(r, np.float64)
    rms = np.sqrt(np.mean(r * r, axis=-1, keepdims=True))
    den = np.maximum(np.abs(r), rms)
    worst = float(np.max(np.abs(a - r) / den))
    assert worst <= LOGIT_REL, f"{what}: relative error {worst:.3e} > {LOGIT_REL}"
    return worst


def oracle_cache(kc):
    """Oracle copy of a binding KVCache (values for bf16, codes for fp8)."""
    if kc.fp8:
        k, v = kc.k.cpu().numpy(), kc.v.cpu().numpy()
        return O.KVCache(k, v, "fp8", kc.k_scale, kc.v_scale, window=kc.window)
    # bf16 values are exact in float32, which halves the host copy of a long cache
    return O.KVCache(kc.k.float().cpu().numpy(), kc.v.float().cpu().numpy(), "bf16",
                     window=kc.window)


def route_margins_per_token(cfg, b):
    """Per token: the kept/dropped group-score gap and the k-th/(k+1)-th expert gap inside
    the kept groups, from biased scores b [T][E]."""
    per = cfg.n_experts // cfg.n_groups
    T = b.shape[0]
    gg, eg = np.zeros(T), np.zeros(T)
    for t in range(T):
        bt = b[t].astype(np.float64)
        gsc = np.sort(bt.reshape(cfg.n_groups, per), axis=1)[:, -2:].sum(axis=1)
        order = np.lexsort((np.arange(cfg.n_groups), -gsc))
        gg[t] = gsc[order[cfg.topk_groups - 1]] - gsc[order[cfg.topk_groups]]
        cand = np.sort(np.concatenate([bt[g * per:(g + 1) * per]
                                       for g in order[: cfg.topk_groups]]))[::-1]
        eg[t] = cand[cfg.topk - 1] - cand[cfg.topk]
    return gg, eg


def routing_stable(cfg, logits_ref, logits_alts, corr_bias, factor=3.0):
    """True when every token's routing is decided by more than the perturbation moves its
    scores: expert gap >= max(1e-6, factor * shift_t) and group gap >= max(1e-6,
    2 * factor * shift_t), shift_t = the token's largest sigmoid-score change."""
    sig = lambda z: 1.0 / (1.0 + np.exp(-np.asarray(z, np.float64)))   # noqa: E731
    s0 = sig(logits_ref)
    shift = np.zeros(s0.shape[0])
    for la in logits_alts:
        shift = np.maximum(shift, np.max(np.abs(sig(la) - s0), axis=1))
    b = s0 + np.asarray(corr_bias, np.float64)
    gg, eg = route_margins_per_token(cfg, b)
    return bool(np.all(gg >= np.maximum(1e-6, 2 * factor * shift)) and
                np.all(eg >= np.maximum(1e-6, factor * shift)))


def routing_tolerance(cfg, logits_ref, logits_alts, corr_bias, factor=3.0):
    """Per token: (stable, tol). tol = factor x the token's largest sigmoid-score change under
    FP32-level perturbation; stable when its expert gap >= max(1e-6, tol) and its group gap
    >= max(1e-6, 2 tol)."""
    sig = lambda z: 1.0 / (1.0 + np.exp(-np.asarray(z, np.float64)))   # noqa: E731
    s0 = sig(logits_ref)
    shift = np.zeros(s0.shape[0])
    for la in logits_alts:
        shift = np.maximum(shift, np.max(np.abs(sig(la) - s0), axis=1))
    tol = factor * shift
    gg, eg = route_margins_per_token(cfg, s0 + np.asarray(corr_bias, np.float64))
    stable = (gg >= np.maximum(1e-6, 2 * tol)) & (eg >= np.maximum(1e-6, tol))
    return stable, tol


def routing_choice_valid(cfg, logits_ref, corr_bias, sel, tol):
    """Whether expert set `sel` of one token is a correct top-k choice within `tol` of the
    oracle's biased scores: its groups are among the best up to tol (group scores up to 2 tol)
    and each selected expert is within tol of the k-th best score of the kept groups."""
    per = cfg.n_experts // cfg.n_groups
    b = 1.0 / (1.0 + np.exp(-np.asarray(logits_ref, np.float64))) + np.asarray(corr_bias, np.float64)
    gsc = np.sort(b.reshape(cfg.n_groups, per), axis=1)[:, -2:].sum(axis=1)
    kth_group = np.sort(gsc)[::-1][cfg.topk_groups - 1]
    groups = sorted(set(int(e) // per for e in sel))
    if len(groups) > cfg.topk_groups or any(gsc[g] < kth_group - 2 * tol for g in groups):
        return False
    cand = np.concatenate([b[g * per:(g + 1) * per] for g in groups])
    kth = np.sort(cand)[::-1][min(cfg.topk, len(cand)) - 1]
    return len(set(int(e) for e in sel)) == cfg.topk and all(b[int(e)] >= kth - tol for e in sel)


def route_margins(cfg, u, w_router, corr_bias):
    """Smallest gap, over tokens, between the kept/dropped group scores and between the k-th
    and (k+1)-th expert scores inside the kept groups (oracle FP32 scores)."""
    _, _, b = O.route_scores(cfg, u, w_router, corr_bias)
    per = cfg.n_experts // cfg.n_groups
    gmin = emin = np.inf
    for t in range(b.shape[0]):
        bt = b[t].astype(np.float64)
        gsc = np.sort(bt.reshape(cfg.n_groups, per), axis=1)[:, -2:].sum(axis=1)
        order = np.lexsort((np.arange(cfg.n_groups), -gsc))
        gs = gsc[order]
        gmin = min(gmin, gs[cfg.topk_groups - 1] - gs[cfg.topk_groups])
        keep = order[: cfg.topk_groups]
        cand = np.sort(np.concatenate([bt[g * per:(g + 1) * per] for g in keep]))[::-1]
        emin = min(emin, cand[cfg.topk - 1] - cand[cfg.topk])
    return gmin, emin


def device_tensor(x, device="cuda"):
    return x.to(device) if isinstance(x, torch.Tensor) else torch.as_tensor(x, device=device)


# ---------------------------------------------------------------------------------------
# Chained steps: bars scaled by the oracle's own rounding-order sensitivity
# ---------------------------------------------------------------------------------------

def flatten_trace(trace, h_final=None, prefix=""):
    """Oracle or GPU layer trace -> {name: float64 array}; router logits under 'L{i}.logits'."""
    out = {}
    for i, tr in enumerate(trace):
        for k in ("q", "attn", "mlp"):
            v = tr[k]
            out[f"{prefix}L{i}.{k}"] = v if isinstance(v, np.ndarray) else np64(v)
        r = tr.get("route")
        if r is not None:
            lg = r[0]
            out[f"{prefix}L{i}.logits"] = lg.astype(np.float64) if isinstance(lg, np.ndarray) \
                else lg.cpu().double().numpy()
    if h_final is not None:
        out[prefix + "h"] = h_final if isinstance(h_final, np.ndarray) else np64(h_final)
    return out


def noise_floor(run, n=2, alts_out=None):
    """run() -> flattened oracle outputs of a chained computation, computed from scratch.
    Returns (reference, floors) where floors[name] = (max-abs-rel, mean-rel, max |delta|)
    of n reruns under FP32-level perturbation of every rounding point, against the reference.
    The perturbed outputs are appended to alts_out when given."""
    from oracle.noise import perturbed_rounding
    ref = run()
    floors = {k: (0.0, 0.0, 0.0) for k in ref}
    for s in range(n):
        with perturbed_rounding(seed=s + 1):
            alt = run()
        if alts_out is not None:
            alts_out.append(alt)
        for k in ref:
            a, r = alt[k], ref[k]
            floors[k] = (max(floors[k][0], max_abs_rel(a, r)), max(floors[k][1], mean_rel(a, r)),
                         max(floors[k][2], float(np.max(np.abs(a - r)))))
    return ref, floors


def floors_on_rows(ref, alts, keys, rows):
    """Perturbation floors of `keys` recomputed over the token rows in `rows` only."""
    out = {}
    for k in keys:
        vals = [(max_abs_rel(a[k][rows], ref[k][rows]), mean_rel(a[k][rows], ref[k][rows]),
                 float(np.max(np.abs(a[k][rows] - ref[k][rows])))) for a in alts]
        out[k] = tuple(max(v[i] for v in vals) for i in range(3))
    return out


def assert_chained_close(got, ref, floors, fp8=False, factor=3.0, rows=None, row_keys=()):
    """Stated bars, or factor x the oracle's own perturbation divergence where that is larger.
    For the keys in row_keys only the token rows in `rows` (a boolean mask) are compared."""
    report = {}
    for k in ref:
        if k.endswith((".logits", ".idx")):
            continue
        lim_mx = max(FP8_MAX_REL if fp8 else BF16_MAX_REL, factor * floors[k][0])
        lim_mn = max(FP8_MEAN_REL if fp8 else BF16_MEAN_REL, factor * floors[k][1])
        a, r = got[k], ref[k]
        if rows is not None and k in row_keys:
            a, r = a[rows], r[rows]
        mx, mn = max_abs_rel(a, r), mean_rel(a, r)
        stated = mx <= (FP8_MAX_REL if fp8 else BF16_MAX_REL) and \
            mn <= (FP8_MEAN_REL if fp8 else BF16_MEAN_REL)
        _record(k, mx, mn, FP8_MAX_REL if fp8 else BF16_MAX_REL,
                FP8_MEAN_REL if fp8 else BF16_MEAN_REL, "chained")
        print(f"{k}: max-abs-rel {mx:.3e} mean-rel {mn:.3e} (stated bar "
              f"{'met' if stated else 'NOT met'}; oracle noise floor {floors[k][0]:.2e} / "
              f"{floors[k][1]:.2e})")
        assert np.all(np.isfinite(a)), f"{k}: non-finite"
        assert mx <= lim_mx and mn <= lim_mn, \
            f"{k}: max-abs-rel {mx:.3e} (<= {lim_mx:.3e}), mean-rel {mn:.3e} (<= {lim_mn:.3e})"
        report[k] = (mx, mn, lim_mx, lim_mn)
    return report


ROUTE_MARGIN_FACTOR = 4.0


def route_margin_ok(shape, trace, weights, floors):
    """Every MoE layer's routing must be decided by more than the perturbation moves the
    scores: margins (oracle FP32 scores) >= max(1e-6, 4 x the largest score shift)."""
    for i, tr in enumerate(trace):
        if tr.get("route") is None:
            continue
        shift = 0.25 * floors[f"L{i}.logits"][2]      # sigmoid slope <= 1/4
        g, e = route_margins(shape, tr["mlp_in"], weights[i]["router"], weights[i]["corr_bias"])
        if min(g, e) < max(1e-6, ROUTE_MARGIN_FACTOR * shift):
            return False
    return True


def codes_close(got_codes, ref_codes, scale, max_frac=0.02):
    """FP8 cache codes. The two sides quantise FP32 values that differ by rounding: a bf16
    flip in the projection output moves a rotated element by up to ~2^-8 of its largest
    partner, so elements near zero may move several fine (subnormal) steps. Bound: every
    decoded value within one e4m3 step (1/8 relative) of the oracle's plus 2^-6 of the
    head's largest magnitude; at most max_frac of the codes differ; mean-rel <= 2e-3."""
    import oracle.codecs as C
    gv = C.e4m3_decode(got_codes).astype(np.float64) * scale
    rv = C.e4m3_decode(ref_codes).astype(np.float64) * scale
    bound = 0.125 * np.abs(rv) + 2.0 ** -6 * np.max(np.abs(rv), axis=-1, keepdims=True)
    assert np.all(np.abs(gv - rv) <= bound), "fp8 values differ beyond one step"
    assert np.mean(got_codes != ref_codes) <= max_frac, \
        f"{np.mean(got_codes != ref_codes):.3%} of fp8 codes differ"
    assert mean_rel(gv, rv) <= FP8_MEAN_REL


# ---------------------------------------------------------------------------------------
# Whole stacks end to end on tie-free routing draws
# ---------------------------------------------------------------------------------------

def min_route_gap(cfg, u, router, corr_bias):
    """Smallest group or expert gap (oracle.route_gaps) over the tokens u [T][H]."""
    _, _, b = O.route_scores(cfg, u, router, corr_bias)
    gg, eg = O.route_gaps(cfg, b)
    return float(min(gg.min(), eg.min()))


def oracle_stack_phases(shape, Wo, caches, phases, choose_router=None, layers=None):
    """The oracle's stack run layer by layer over consecutive phases of tokens.

    phases: list of (e [T][H] embeddings or residual stream, seq_id [T], pos [T]); phase i+1
    comes after phase i (e.g. a prefill then a decode token). caches: one oracle KVCache per
    layer, filled in place. At layer l every phase runs oracle.layer_forward in order; when
    choose_router(l, u) returns a router dict for the MoE layer's inputs u (all phases'
    tokens stacked), the layer is rerun with it. Rerunning is exact: a phase writes its own
    tokens' cache slots and, attention being causal, reads none written by a later phase (the
    caller keeps ring capacities above the positions written).
    Returns (h per phase, per-phase traces: one dict per layer with q, g, attn, mlp_in, mlp,
    route and the layer's output h)."""
    L = shape.n_layers
    layers = list(range(L)) if layers is None else layers
    st = [O.boundary_norm(None, e, None, Wo[layers[0]]["attn_pre"], 1, shape.eps)
          for e, _, _ in phases]
    traces = [[] for _ in phases]
    for i, l in enumerate(layers):
        nxt = Wo[layers[i + 1]]["attn_pre"] if i + 1 < len(layers) else None

        def run(Wl, l=l, nxt=nxt):
            outs, trs = [], []
            for (h, u), (_, seq, pos) in zip(st, phases):
                tr = []
                outs.append(O.layer_forward(shape, l, Wl, h, u, caches[l], seq, pos, nxt, tr))
                tr[0]["h"] = outs[-1][0]
                trs.append(tr[0])
            return outs, trs

        outs, trs = run(Wo[l])
        if choose_router is not None and trs[0]["route"] is not None:
            R = choose_router(l, np.concatenate([t["mlp_in"] for t in trs]))
            if R is not None:
                Wo[l] = dict(Wo[l], **R)
                outs, trs = run(Wo[l])
        st = outs
        for tr, t in zip(traces, trs):
            tr.append(t)
    return [h for h, _ in st], traces


def tie_free_router_chooser(shape, seed, min_gap, device, chosen, max_tries=20000):
    """choose_router for oracle_stack_phases: keeps a layer's router when every token's routing
    gaps are >= min_gap, else walks synth's router redraws (attempt 1, 2, ...) to the first
    that clears them. chosen[l] = (attempt, device tensors) records what the GPU must use."""
    import synth

    def choose(l, u):
        def draw(a):
            R = synth.router_weights(shape, l, seed, device=device, attempt=a)
            return R, {k: np64(v) for k, v in R.items()}

        attempt, (Rd, Rh) = synth.first_accepted(
            draw, lambda r: min_route_gap(shape, u, r[1]["router"], r[1]["corr_bias"]) >= min_gap,
            max_tries)
        chosen[l] = (attempt, Rd)
        return None if attempt == 0 else Rh

    return choose


def trace_dict(traces, phase_names, layers):
    """{'<phase>.L<l>.<q|attn|mlp|h>': float64 array, '<phase>.L<l>.idx': sorted indices}
    from per-phase traces (oracle arrays or GPU tensors)."""
    out = {}
    for name, tr in zip(phase_names, traces):
        for l, t in zip(layers, tr):
            for k in ("q", "attn", "mlp", "h"):
                v = t[k]
                out[f"{name}.L{l}.{k}"] = v.astype(np.float64) if isinstance(v, np.ndarray) \
                    else np64(v)
            if t.get("route") is not None:
                idx = t["route"][1]
                idx = idx if isinstance(idx, np.ndarray) else idx.cpu().numpy()
                out[f"{name}.L{l}.idx"] = np.sort(np.asarray(idx), 1)
    return out


def compare_chained(got, ref, fp8=False, floors=None, widened=(), factor=3.0, label=""):
    """Element-by-element comparison of chained outputs, printed for every key.

    Routing ('.idx' keys) must be identical. Every other key is held to the stated bars
    (2e-2 max-abs-rel, 1e-3 mean-rel; FP8-KV 5e-2 / 2e-3), except the keys listed in `widened`:
    those are held to max(stated, factor x the oracle's own divergence under FP32-level
    perturbation) from `floors`, the documented exception for chained steps whose oracle
    noise floor is itself above the stated bar. Returns the printed rows."""
    lim_mx0, lim_mn0 = (FP8_MAX_REL, FP8_MEAN_REL) if fp8 else (BF16_MAX_REL, BF16_MEAN_REL)
    rows, bad = [], []
    for k in ref:
        if k.endswith(".idx"):
            same = np.array_equal(got[k], ref[k])
            rows.append(f"{label}{k}: routing {'identical' if same else 'DIFFERS'}")
            if not same:
                diff = np.nonzero(np.any(got[k] != ref[k], axis=1))[0]
                bad.append(f"{k}: routing differs on tokens {diff.tolist()[:10]}")
            continue
        a, r = got[k], ref[k]
        mx, mn = max_abs_rel(a, r), mean_rel(a, r)
        fl = floors.get(k) if floors else None
        lim_mx, lim_mn = lim_mx0, lim_mn0
        if k in widened and fl is not None:
            lim_mx, lim_mn = max(lim_mx, factor * fl[0]), max(lim_mn, factor * fl[1])
        stated_ok = mx <= lim_mx0 and mn <= lim_mn0
        _record(f"{label}{k}", mx, mn, lim_mx0, lim_mn0, "chained" if k in widened else "stated")
        rows.append(f"{label}{k}: max-abs-rel {mx:.3e} mean-rel {mn:.3e} "
                    f"(stated bar {'met' if stated_ok else 'NOT met'}"
                    + (f"; oracle noise floor {fl[0]:.2e} / {fl[1]:.2e}" if fl else "")
                    + (f"; widened bar {lim_mx:.2e} / {lim_mn:.2e}" if k in widened else "") + ")")
        if not np.all(np.isfinite(a)):
            bad.append(f"{k}: non-finite")
        elif mx > lim_mx or mn > lim_mn:
            bad.append(f"{k}: max-abs-rel {mx:.3e} (<= {lim_mx:.2e}), mean-rel {mn:.3e} "
                       f"(<= {lim_mn:.2e})")
    print("\n".join(rows))
    assert not bad, "; ".join(bad)
    return rows
