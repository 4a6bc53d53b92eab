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
