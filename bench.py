"""Benchmark of the Beam decoder-layer forward on GB300 (one JSON line on rank 0).

Default: the 6-layer truncated stack (layers 0-2 dense SwiGLU, 3-5 256-expert MoE; layers 0-4
sliding-window, layer 5 NoPE with SSMax) decoding one token of one sequence over 100,000
cached tokens per layer with a BF16 cache: the line's value is µs per token per layer, with
the HBM roofline of the step and of its dominant call. The same line carries a "prefill"
object: the same stack and weights prefilling 8 sequences x 2048 new tokens appended to
100,000 cached ones (tokens/s, tensor rooflines of the dominant GEMM call and of the NoPE
attention call, the GEMM calls' share of the BF16 peak).

Other workloads (seeded synthetic inputs, random-init weights; shapes of the Beam layer):
  stack_decode  --batch/--context/--kv (the 8-K / batch-128 / FP8 case is
                --batch 128 --context 8192 --kv fp8)
  stack_prefill --seqs x --chunk new tokens after --context
  stack_verify  --batch sequences x --chunk (1-16) new tokens each after --context: the
                multi-token verification step of speculative decoding
  swa_decode    one full-width sliding-window MoE layer, batch-1 decode, context 4096
  nope_decode   one full-width NoPE MoE layer, decode at context 100,000 (--batch, --kv)

A step is one pass of the whole layer (or stack) over one batch of new tokens; the residual
stream h it updates in place carries over to the next step. Inputs are resident in HBM when
the timed region starts; each step streams far more than the 129 MB L2 (the layer's weights),
so no flush is needed. The K timed steps are captured as one CUDA graph and replayed once
between two events; each call's time comes from a second replay of the same K steps with a
timing event (an external event node) before every call.

--experts nvfp4 / fp8 gives the MoE layers NVFP4 or block-scaled FP8 expert weights
(beam_moe_nvfp4 / beam_moe_fp8; decode workloads).

--impl reference times the CPU oracle on the same workload instead (a bounded sample per step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from synth import BEAM  # noqa: E402

METRIC = "Beam-layer decode µs/token & HBM GB/s % of peak; prefill tokens/s"
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------- helpers ----

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], "measured"
    return FALLBACK_HBM_GBS, "fallback"


def max_over_ranks(x, world, device):
    """The largest of the ranks' values of x, on every rank (x itself for one rank): a step
    time taken on each rank becomes the slowest rank's."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job(ms_step, tokens_per_rank, world, n_layers, prefill):
    """(value, unit) over all ranks: prefill tokens/s = every rank's tokens over the slowest
    rank's step; decode µs/token/layer = that step over every rank's tokens and the layers."""
    if prefill:
        return tokens_per_rank * world / (ms_step * 1e-3), "tokens/s"
    return ms_step * 1000.0 / (tokens_per_rank * world) / n_layers, "us/token/layer"


def emit(res, rank):
    """Rank 0 prints the JSON line; the other ranks print nothing. Returns whether it printed."""
    if rank != 0 or res is None:
        return False
    print(json.dumps(res), flush=True)
    return True


def is_nope(l, L):
    return (l + 1) % 6 == 0 or l == L - 1


def expert_bytes(shape, fmt="bf16"):
    """Weight bytes of one expert: BF16; NVFP4 (half a byte per element, one e4m3 scale per
    16 elements, two FP32 matrix scales); or FP8 (a byte per element, one FP32 scale per
    128 x 128 block of each matrix)."""
    H, F = shape.hidden, shape.d_ff_expert
    n = 3 * H * F
    if fmt == "nvfp4":
        return n // 2 + n // 16 + 8
    if fmt == "fp8":
        blocks = lambda r, c: -(-r // 128) * -(-c // 128)  # noqa: E731
        return n + 4 * (blocks(2 * F, H) + blocks(H, F))
    return 2 * n


def layer_bytes(shape, dense, n_experts_touched, kv_bytes, fmt="bf16"):
    """Algorithmic HBM bytes of one layer step: every weight byte the step must read once,
    the KV bytes it must read, the gains; activations are negligible (<0.1%)."""
    H, D = shape.hidden, shape.head_dim
    b = shape.qkvg_rows * H * 2 + H * shape.q_rows * 2           # packed QKVG, o_proj
    b += 4 * H * 2 + 2 * D * 2 + shape.n_q * 2                   # gains, gate bias
    if dense:
        b += 3 * H * shape.d_ff_dense * 2
    else:
        b += shape.n_experts * H * 4 + shape.n_experts * 4       # FP32 router
        b += n_experts_touched * expert_bytes(shape, fmt)
    return b + kv_bytes


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None
        time.sleep(0.25)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.p is not None:
            time.sleep(0.15)
            self.p.terminate()
            try:
                self.out, _ = self.p.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()
                self.out = ""

    def summary(self):
        rows = []
        for line in self.out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            try:
                rows.append((float(f[0]), float(f[1]), float(f[2]), f[3:7]))
            except (ValueError, IndexError):
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v == "Active"})
        loaded = [r[0] for r in rows if r[2] > 200.0] or [r[0] for r in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def source_hash(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key):
    """Per-launch DRAM bytes of a kernel from a committed ncu summary, if it was taken on the
    current source of that kernel (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel_key)
    if not d:
        return None
    if d.get("source_hash") != source_hash(d["sources"]):
        return None
    return d["bytes_per_launch"]


# --------------------------------------------------------------------------- workloads ----

def stack_weights(args, layers, device):
    """Device weights of the held layers (one dict per layer, synth.layer_weights), with NVFP4
    or FP8 expert weights on the MoE layers under --experts nvfp4 / fp8."""
    W = []
    for l in layers:
        quant = args.experts != "bf16" and l not in BEAM.dense_layers
        W.append(synth.layer_weights(BEAM, l, args.seed, device=device, with_experts=not quant))
        if quant and args.experts == "nvfp4":
            W[-1]["nvfp4"] = synth.expert_weights_nvfp4(BEAM, l, args.seed, device=device)
        elif quant:
            W[-1]["fp8"] = synth.expert_weights_fp8(BEAM, l, args.seed, device=device)
    return W


def workload_shape(kind, args):
    """(layers, context, sequences, new tokens per sequence) of a workload."""
    if kind == "swa_decode":
        return [3], 4096, 1, 1
    if kind == "nope_decode":
        return [5], 100_000, args.batch, 1
    if kind == "stack_prefill":
        return list(range(6)), args.context, args.seqs, args.chunk
    if kind == "stack_verify":
        return list(range(6)), args.context, args.batch, args.chunk
    return list(range(6)), args.context, args.batch, 1      # stack_decode


class Workload:
    """Weights, caches and inputs of one benchmark case on the device. W: weights to share
    with another workload over the same layers (else drawn here)."""

    def __init__(self, args, device, kind, W=None):
        from hybrid_attention_moe_gb300 import beam as B
        from hybrid_attention_moe_gb300.stack import BeamStack
        self.B = B
        self.args = args
        self.device = device
        self.kind = kind
        shape = BEAM
        layers, ctx, batch, chunk = workload_shape(kind, args)
        fp8 = args.kv == "fp8"
        self.layers, self.ctx, self.batch, self.fp8 = layers, ctx, batch, fp8
        self.chunk = chunk
        self.prefill = kind == "stack_prefill"
        self.tokens = batch * chunk
        # the bound on tokens per sequence that beam_attn is given, which picks its form:
        # split-K decode up to 4 (up to 16 when there are few sequences), query tiles above;
        # --attn-form forces one or the other (a bound of 1, or one above 16)
        form = getattr(args, "attn_form", "natural")
        self.attn_form = form
        self.q_bound = chunk if form == "natural" else (1 if form == "decode" else max(chunk, 17))
        scale = 1.0
        self.experts = args.experts
        W = stack_weights(args, layers, device) if W is None else W
        caches = []
        for l in layers:
            nope = is_nope(l, shape.n_layers)
            # a sliding-window ring holds window + chunk - 1 keys, rounded up to whole 128-key
            # tiles (the tensor-core prefill walks the ring in tile-aligned slots)
            cap, win = ((ctx + chunk + 8, 0) if nope else
                        (-(-(shape.window + chunk - 1) // 128) * 128, shape.window))
            c = synth.kv_cache(shape, batch, cap, args.seed, l, fp8=fp8, k_scale=scale,
                               v_scale=scale, device=device)
            caches.append(B.KVCache(c["k"], c["v"], win, scale, scale))
        self.shape = shape
        self.stack = BeamStack(shape, W, caches, first_layer=layers[0], device=device)
        self.seq, self.pos = synth.prefill_positions([ctx] * batch, chunk, device)
        self.max_pos = ctx + chunk
        self.e = synth.activations(self.tokens, shape.hidden, args.seed, "h", device)
        self.W = W
        self.caches = caches

    def config(self):
        return {
            "workload": self.kind, "layers": self.layers, "batch": self.batch,
            "new_tokens_per_seq": self.chunk, "context": self.ctx,
            "kv_cache": "fp8_e4m3" if self.fp8 else "bf16",
            "expert_weights": self.experts,
            "attn_form": self.attn_form,
            "hidden": BEAM.hidden, "heads": f"{BEAM.n_q}q/{BEAM.n_kv}kv x {BEAM.head_dim}",
            "experts": f"{BEAM.n_experts} (8 groups, top-4 groups, top-8), d_ff {BEAM.d_ff_expert}",
        }

    def step_calls(self):
        """The library calls of one step as (name, fn) closures over fixed buffers."""
        B, st = self.B, self.stack
        T = self.tokens
        b = st.buffers(T)
        ws = st.ws.get(B.workspace_bytes(st.cfgs[0], T, self.max_pos))
        b["h"].copy_(self.e)
        calls = [("pre_norm", lambda: B.beam_boundary_norm(None, b["h"], b["u"], None,
                                                           st.W[0]["attn_pre"], 1,
                                                           st.cfgs[0].eps))]
        for i in range(st.L):
            W, cfg, kc, l = st.W[i], st.cfgs[i], st.caches[i], st.ids[i]
            nxt = st.W[i + 1]["attn_pre"] if i + 1 < st.L else None
            calls += [
                (f"L{l}.qkv_gate", lambda W=W, cfg=cfg, kc=kc: B.beam_qkv_gate(
                    cfg, b["u"], W["w_qkvg"], W["q_norm"], W["k_norm"], self.seq, self.pos,
                    b["q"], b["g"], kc, ws)),
                (f"L{l}.attn", lambda W=W, cfg=cfg, kc=kc: B.beam_attn(
                    cfg, b["q"], b["g"], W["gate_bias"], kc, self.seq, self.pos, self.max_pos,
                    W["w_o"], b["a"], ws, max_q_per_seq=self.q_bound)),
                (f"L{l}.norm_attn", lambda W=W, cfg=cfg, l=l: B.beam_boundary_norm(
                    b["a"], b["h"], b["u"], W["attn_post"], W["mlp_pre"], 2 * l + 2, cfg.eps)),
            ]
            if st.dense[i]:
                calls.append((f"L{l}.dense_mlp", lambda W=W, cfg=cfg: B.beam_dense_mlp(
                    cfg, b["u"], W["w_gate_up"], W["w_down"], b["m"], ws)))
            else:
                calls += [
                    (f"L{l}.route", lambda W=W, cfg=cfg: B.beam_route(
                        cfg, b["u"], W["router"], W["corr_bias"], b["logits"], b["idx"], b["w"],
                        ws)),
                    (f"L{l}.moe", (lambda W=W, cfg=cfg: B.beam_moe_nvfp4(
                        cfg, b["u"], b["idx"], b["w"], W["nvfp4"], b["m"], ws)) if "nvfp4" in W
                     else (lambda W=W, cfg=cfg: B.beam_moe_fp8(
                         cfg, b["u"], b["idx"], b["w"], W["fp8"], b["m"], ws)) if "fp8" in W
                     else (lambda W=W, cfg=cfg: B.beam_moe(
                         cfg, b["u"], b["idx"], b["w"], W["w_gate_up"], W["w_down"], b["m"], ws))),
                ]
            calls.append((f"L{l}.norm_mlp", lambda W=W, cfg=cfg, l=l, nxt=nxt:
                          B.beam_boundary_norm(b["m"], b["h"], b["u"] if nxt is not None else None,
                                               W["mlp_post"], nxt, 2 * l + 3, cfg.eps)))
        return calls, b

    def flops(self):
        """Algorithmic FLOPs of one step per call kind (tensor-core contractions) and the
        router's FP32 FLOPs."""
        s = self.shape
        T, H = self.tokens, s.hidden
        out = {}
        for i, l in enumerate(self.layers):
            nope = is_nope(l, s.n_layers)
            keys = 0
            for t in range(self.chunk):
                p = self.ctx + 1 + t
                keys += p if nope else min(s.window, p)
            keys *= self.batch
            out[f"L{l}.qkv_gate"] = 2.0 * T * s.qkvg_rows * H
            out[f"L{l}.attn"] = 4.0 * s.head_dim * s.n_q * keys + 2.0 * T * H * s.q_rows
            if l in s.dense_layers:
                out[f"L{l}.dense_mlp"] = 2.0 * T * 3 * H * s.d_ff_dense
            else:
                out[f"L{l}.moe"] = 2.0 * T * s.topk * 3 * H * s.d_ff_expert
                out[f"L{l}.route"] = 2.0 * T * s.n_experts * H
        return out

    def touched_experts(self, b):
        """Distinct experts each MoE layer's routing selected in the last step."""
        return len(set(b["idx"].cpu().numpy().ravel().tolist()))

    def algorithmic_bytes(self, touched):
        shape = self.shape
        tot = 0
        per = {}
        for i, l in enumerate(self.layers):
            nope = is_nope(l, shape.n_layers)
            keys = self.ctx + 1 if nope else min(shape.window, self.ctx + 1)
            elem = 1 if self.fp8 else 2
            kv = self.batch * (keys + self.chunk - 1) * shape.n_kv * shape.head_dim * 2 * elem
            dense = l in shape.dense_layers
            per[l] = layer_bytes(shape, dense, touched.get(l, shape.topk), kv, self.experts)
            tot += per[l]
        return tot, per


# --------------------------------------------------------------------------- our arm ----

def measure(wl, args, world, device):
    """Times one workload: K steps captured as one CUDA graph and replayed between two events
    on the launching stream (after W warm-up replays), the per-call breakdown from a second
    replay with an event before every call, the end-to-end variant through host buffers, and
    the roofline of the dominant call. Returns the fields of a bench line."""
    B_mod = wl.B
    calls, b = wl.step_calls()
    names = [n for n, _ in calls]
    stream = torch.cuda.Stream(device)
    torch.cuda.synchronize()
    # eager warm-up: sets kernel attributes and sizes the workspace before any capture
    with torch.cuda.stream(stream):
        for _ in range(2):
            for _, fn in calls:
                fn()
    torch.cuda.synchronize()
    c0 = B_mod.beam_launch_count()
    with torch.cuda.stream(stream):
        for _, fn in calls:
            fn()
    torch.cuda.synchronize()
    launches_step = B_mod.beam_launch_count() - c0

    step_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(step_graph, stream=stream):
        for _, fn in calls:
            fn()
    # the timed region: K steps in one graph (no nodes between the calls, so consecutive
    # kernels keep their programmatic-launch overlap)
    timed = torch.cuda.CUDAGraph()
    with torch.cuda.graph(timed, stream=stream):
        for _ in range(args.steps):
            for _, fn in calls:
                fn()
    # the per-call breakdown: the same K steps with a timing event (an external event node)
    # before every call, replayed right after the timed region
    try:
        events = [[torch.cuda.Event(enable_timing=True, external=True)
                   for _ in range(len(calls) + 1)] for _ in range(args.steps)]
        evg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(evg, stream=stream):
            for s in range(args.steps):
                for i, (_, fn) in enumerate(calls):
                    events[s][i].record(stream)
                    fn()
                events[s][-1].record(stream)
        mode = ("one graph of all timed steps; per-call times from a second replay with "
                "external timing events between the calls")
    except (TypeError, RuntimeError):
        evg, events = None, None
        mode = "one graph of all timed steps; no per-call breakdown (no external events)"
    torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step_graph.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with Clocks(torch.cuda.current_device()) as clk, torch.cuda.stream(stream):
        t0.record(stream)
        timed.replay()
        t1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms_step = t0.elapsed_time(t1) / args.steps
    per_call_us = {}
    evented_ms = None
    if evg is not None:
        with torch.cuda.stream(stream):
            evg.replay()
        torch.cuda.synchronize()
        evented_ms = events[0][0].elapsed_time(events[-1][-1]) / args.steps
        for i, name in enumerate(names):
            per_call_us[name] = 1000.0 * float(np.mean(
                [events[s][i].elapsed_time(events[s][i + 1]) for s in range(args.steps)]))
    ms_step = max_over_ranks(ms_step, world, device)

    # experts touched by the routing of the last step (the idx buffer holds the last MoE
    # layer's selection; the others are taken to touch as many)
    touched = {}
    moe_layers = [l for i, l in enumerate(wl.layers) if not wl.stack.dense[i]]
    if moe_layers:
        n = wl.touched_experts(b)
        for l in moe_layers:
            touched[l] = n
    algo_bytes, _ = wl.algorithmic_bytes(touched)
    value, unit = whole_job(ms_step, wl.tokens, world, len(wl.layers), wl.prefill)
    hbm, hbm_kind = peaks()
    layer_gbs = algo_bytes / (ms_step * 1e-3) / 1e9

    res = {"value": round(value, 1 if wl.prefill else 3), "unit": unit,
           "ms_per_step": round(ms_step, 4), "higher_is_better": bool(wl.prefill)}
    if not wl.prefill:
        res["layer_hbm"] = {"algorithmic_bytes_per_step": algo_bytes,
                            "achieved_gbs": round(layer_gbs, 1), "peak_gbs": hbm,
                            "frac": round(layer_gbs / hbm, 4), "peak_kind": hbm_kind}
    if per_call_us and not wl.prefill:
        dom = max(per_call_us, key=per_call_us.get)
        dom_bytes, dom_key = dominant_bytes(wl, dom, touched)
        dom_gbs = dom_bytes / (per_call_us[dom] * 1e-6) / 1e9
        res["roofline"] = {
            "bound": "hbm", "kernel": dom, "achieved": round(dom_gbs, 1), "peak": hbm,
            "unit": "GB/s", "frac": round(dom_gbs / hbm, 4), "traffic": ncu_traffic(dom_key),
            "bytes_per_launch": dom_bytes, "duration_us": round(per_call_us[dom], 2),
            "peak_kind": hbm_kind}
    elif per_call_us:
        tf_peak, tf_kind = tensor_peak()
        fl = wl.flops()

        def tensor_roof(key):
            ach = fl[key] / (per_call_us[key] * 1e-6) / 1e12
            return {"bound": "tensor", "kernel": key, "achieved": round(ach, 1),
                    "peak": tf_peak, "unit": "TFLOP/s", "frac": round(ach / tf_peak, 4),
                    "traffic": ncu_traffic(key.split(".")[1] + "_prefill"),
                    "flops_per_launch": fl[key], "duration_us": round(per_call_us[key], 2),
                    "peak_kind": tf_kind}

        gemm_keys = [k for k in fl if k.endswith((".qkv_gate", ".dense_mlp", ".moe"))]
        attn_keys = [k for k in fl if k.endswith(".attn")]
        res["roofline"] = tensor_roof(max(gemm_keys, key=per_call_us.get))
        res["attention_roofline"] = tensor_roof(max(attn_keys, key=per_call_us.get))
        tc_flops = sum(v for k, v in fl.items() if not k.endswith(".route"))
        gemm_us = sum(per_call_us[k] for k in gemm_keys)
        gemm_fl = sum(fl[k] for k in gemm_keys)
        res["tensor"] = {
            "step_tflops": round(tc_flops / (ms_step * 1e-3) / 1e12, 1),
            "step_flops": tc_flops,
            "gemm_calls_tflops": round(gemm_fl / (gemm_us * 1e-6) / 1e12, 1),
            "gemm_calls_frac": round(gemm_fl / (gemm_us * 1e-6) / 1e12 / tf_peak, 4),
            "peak": tf_peak, "peak_kind": tf_kind}
    res["per_call_us"] = {k: round(v, 2) for k, v in per_call_us.items()}
    res["per_call_replay_ms_per_step"] = None if evented_ms is None else round(evented_ms, 4)
    res["timing"] = mode
    res["e2e"] = run_e2e(args, wl, step_graph, stream, world, device)
    res["gpu_launches"] = launches_step * args.steps
    res["clocks"] = clk.summary()
    res["_stream"], res["_b"] = stream, b
    return res


def run_ours(args, rank, world, device):
    import __graft_entry__ as ge
    ge.build()
    wl = Workload(args, device, args.workload)
    m = measure(wl, args, world, device)
    stream, b = m.pop("_stream"), m.pop("_b")
    head = time_lm_head(args, wl, b, stream) if args.lm_head_vocab > 0 else None
    res = {
        "metric": METRIC,
        "value": m["value"],
        "unit": m["unit"],
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": m["ms_per_step"],
        "higher_is_better": m["higher_is_better"],
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) activations and KV cache, random-init N(0,0.02) weights",
        "config": dict(wl.config(), **{
            "parallelism": "replicas" if world > 1 else "single",
            "l2": "no flush: each step streams "
                  f"{wl.algorithmic_bytes({})[0] / 1e6:.0f} MB of weights and cache (> 129 MB L2)",
            "timing": m["timing"]}),
    }
    for k in ("layer_hbm", "roofline", "attention_roofline", "tensor", "per_call_us",
              "per_call_replay_ms_per_step", "e2e", "gpu_launches"):
        if k in m:
            res[k] = m[k]
    if head is not None:
        res["lm_head"] = head
    res["clocks"] = m["clocks"]
    if world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(args, wl, budget_s=args.cpu_budget)
    if args.workload == "stack_decode" and not args.no_prefill:
        # the same stack, same weights: prefill of args.seqs x args.chunk new tokens after
        # args.context cached ones, as its own object of the line
        del wl.stack, wl.caches
        torch.cuda.empty_cache()
        pw = Workload(args, device, "stack_prefill", W=wl.W)
        p = measure(pw, args, world, device)
        p.pop("_stream"), p.pop("_b")
        p["config"] = dict(pw.config(), timing=p.pop("timing"),
                           l2="no flush: each step streams the stack's weights "
                              f"({sum(t.numel() * t.element_size() for w in pw.W for t in w.values() if torch.is_tensor(t)) / 1e9:.1f} GB)")
        if world == 1 and not args.no_cpu_baseline:
            p["cpu_baseline"] = cpu_baseline(args, pw, budget_s=args.cpu_budget)
        res["prefill"] = p
    return res


def time_lm_head(args, wl, b, stream):
    """The LM head after the stack, timed beside the step (its own graph of K calls, CUDA
    events on the launching stream): the final norm of the last residual stream h, then
    beam_lm_head over a vocabulary of args.lm_head_vocab rows with the 30*tanh(z/30) cap.
    Algorithmic bytes per call: the vocabulary rows (V x H bf16), the tokens' u and h, and one
    write of the FP32 logits."""
    B = wl.B
    V, H, T = args.lm_head_vocab, wl.shape.hidden, wl.tokens
    head = synth.lm_head_weights(wl.shape, V, args.seed, device=wl.device)
    u = torch.empty((T, H), dtype=torch.bfloat16, device=wl.device)
    logits = torch.empty((T, V), dtype=torch.float32, device=wl.device)
    eps = wl.stack.cfgs[0].eps

    def call():
        B.beam_boundary_norm(None, b["h"], u, None, head["final_norm"], 1, eps)
        B.beam_lm_head(u, head["w_lm"], logits, softcap=30.0)

    with torch.cuda.stream(stream):
        for _ in range(2):
            call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(args.steps):
            call()
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        g.replay()
        t1.record(stream)
    torch.cuda.synchronize()
    us = t0.elapsed_time(t1) * 1000.0 / args.steps
    nbytes = V * H * 2 + T * H * 2 * 2 + T * V * 4
    hbm, hbm_kind = peaks()
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"vocab": V, "tokens": T, "softcap": 30.0, "us_per_call": round(us, 2),
            "bytes_per_call": nbytes, "achieved_gbs": round(gbs, 1), "peak_gbs": hbm,
            "frac": round(gbs / hbm, 4), "peak_kind": hbm_kind,
            "calls": "final norm + beam_lm_head (projection, then the softcap pass)"}


def tensor_peak():
    """Dense BF16 tensor peak for a kernel timed inside a long step: the sustained figure."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("bf16_tflops_sustained", d["bf16_tflops"]), "measured (sustained)"
    return 1700.0, "fallback (sustained)"


def dominant_bytes(wl, name, touched):
    """Algorithmic bytes of one call of the step (weights and cache it must read once)."""
    l = int(name.split(".")[0][1:])
    if name.endswith(".moe"):
        key = "moe_decode" + ("" if wl.experts == "bf16" else "_" + wl.experts) + f"_t{wl.tokens}"
        return touched[l] * expert_bytes(BEAM, wl.experts), key
    if name.endswith(".attn"):
        nope = is_nope(l, BEAM.n_layers)
        keys = wl.ctx + 1 if nope else min(BEAM.window, wl.ctx + 1)
        elem = 1 if wl.fp8 else 2
        kv = wl.batch * keys * BEAM.n_kv * BEAM.head_dim * 2 * elem
        return kv + BEAM.hidden * BEAM.q_rows * 2, ("attn_nope_decode" if nope else
                                                     "attn_swa_decode") + f"_t{wl.tokens}"
    if name.endswith(".dense_mlp"):
        return 3 * BEAM.hidden * BEAM.d_ff_dense * 2, f"dense_decode_t{wl.tokens}"
    if name.endswith(".route"):
        return BEAM.n_experts * BEAM.hidden * 4, f"route_decode_t{wl.tokens}"
    if name.endswith(".qkv_gate"):
        return BEAM.qkvg_rows * BEAM.hidden * 2, f"qkv_decode_t{wl.tokens}"
    return 2 * wl.batch * BEAM.hidden * 2, "norm"


def run_e2e(args, wl, step_graph, stream, world, device):
    """Same step with the tokens' hidden state copied in from pinned host memory and the
    output h copied back, both inside the timed region."""
    b = wl.stack.buffers(wl.tokens)
    h_host = wl.e.cpu().pin_memory()
    out_host = torch.empty_like(h_host).pin_memory()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        t0.record(stream)
        for _ in range(args.steps):
            b["h"].copy_(h_host, non_blocking=True)
            step_graph.replay()
            out_host.copy_(b["h"], non_blocking=True)
        t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = max_over_ranks(t0.elapsed_time(t1) / args.steps, world, device)
    nbytes = h_host.numel() * h_host.element_size()
    value, unit = whole_job(ms, wl.tokens, world, len(wl.layers), wl.prefill)
    return {"value": round(value, 1 if wl.prefill else 3), "unit": unit,
            "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes}


# ------------------------------------------------------------------------ oracle arm ----

def oracle_layers(wl):
    """Host views of the workload's weights and first-sequence caches for the oracle: float32
    copies (bf16 values are exact; the oracle widens them) and experts fetched on first use."""
    import oracle as O

    def host(t):
        return t.float().cpu().numpy()

    class Lazy:
        def __init__(self, t):
            self.t, self.c = t, {}

        def __getitem__(self, e):
            if e not in self.c:
                self.c[e] = host(self.t[e])
            return self.c[e]

    class LazyNvfp4:
        """expert -> the six NVFP4 arrays of oracle.moe_nvfp4, copied to the host on first use"""
        def __init__(self, d):
            self.d, self.c = d, {}

        def __getitem__(self, e):
            if e not in self.c:
                h = {k: v[e].cpu().numpy() for k, v in self.d.items()}
                self.c[e] = (h["gate_up"], h["gate_up_scale"], float(h["gate_up_global"]),
                             h["down"], h["down_scale"], float(h["down_global"]))
            return self.c[e]

    class LazyFp8:
        """expert -> the four FP8 arrays of oracle.moe_fp8, copied to the host on first use"""
        def __init__(self, d):
            self.d, self.c = d, {}

        def __getitem__(self, e):
            if e not in self.c:
                h = {k: v[e].cpu().numpy() for k, v in self.d.items()}
                self.c[e] = (h["gate_up"], h["gate_up_scale"], h["down"], h["down_scale"])
            return self.c[e]

    Wo = []
    for W in wl.W:
        d = {}
        for k, v in W.items():
            if k == "nvfp4":
                d["nvfp4_experts"] = LazyNvfp4(v)
            elif k == "fp8":
                d["fp8_experts"] = LazyFp8(v)
            else:
                d[k] = Lazy(v) if (k in ("w_gate_up", "w_down") and v.dim() == 3) else host(v)
        Wo.append(d)
    caches = []
    for kc in wl.caches:
        if kc.fp8:
            caches.append(O.KVCache(kc.k[:1].cpu().numpy(), kc.v[:1].cpu().numpy(), "fp8",
                                    kc.k_scale, kc.v_scale, window=kc.window))
        else:
            caches.append(O.KVCache(host(kc.k[:1]), host(kc.v[:1]), "bf16", window=kc.window))
    return Wo, caches


def oracle_sample(args, wl, layers=None, n_tokens=1):
    """A bounded oracle workload: the first n_tokens new tokens of sequence 0 (a decode token,
    or the head of its prefill chunk) through the held layers (or the given subset)."""
    import oracle as O
    shape = wl.shape
    Wo, caches = oracle_layers(wl)
    idx = list(range(len(wl.layers))) if layers is None else \
        [wl.layers.index(l) for l in layers]
    h0 = wl.e[:n_tokens].float().cpu().numpy().astype(np.float64)
    pos = [wl.ctx + 1 + t for t in range(n_tokens)]
    seq = [0] * n_tokens

    def run():
        h, u = O.boundary_norm(None, h0, None, Wo[idx[0]]["attn_pre"], 1, shape.eps)
        for j, i in enumerate(idx):
            nxt = Wo[idx[j + 1]]["attn_pre"] if j + 1 < len(idx) else None
            h, u = O.layer_forward(shape, wl.layers[i], Wo[i], h, u, caches[i], seq, pos, nxt)
        return h

    run()   # untimed: fetches the experts the oracle's own routing picks
    return run


def cpu_baseline(args, wl, budget_s=15.0):
    """The oracle, as it stands, on the host cores: a bounded sample of the workload, repeated
    until budget_s of CPU time. Decode: the first sequence's new token through every held
    layer (µs per token per layer). Prefill: the first PREFILL_SAMPLE tokens of sequence 0's
    chunk through every layer (tokens/s; the oracle's cost per token is the same for every
    token of the chunk up to the 2% growth of the NoPE keys across it)."""
    n_tok = PREFILL_SAMPLE if wl.prefill else 1
    run = oracle_sample(args, wl, n_tokens=n_tok)
    n, t_total = 0, 0.0
    while t_total < budget_s and n < 50:
        t = time.perf_counter()
        run()
        t_total += time.perf_counter() - t
        n += 1
    if wl.prefill:
        val, unit = round(n * n_tok / t_total, 3), "tokens/s"
        sample = (f"{n} x the first {n_tok} tokens of sequence 0's {wl.chunk}-token chunk "
                  f"(positions {wl.ctx + 1}-{wl.ctx + n_tok}) through layers {wl.layers}; "
                  f"rate extrapolated to the {wl.batch} x {wl.chunk}-token step; float64 "
                  f"NumPy oracle, {t_total:.1f} s")
    else:
        val, unit = round(t_total / n * 1e6 / len(wl.layers), 1), "us/token/layer"
        sample = (f"{n} x the first new token of sequence 0 through layers {wl.layers} "
                  f"(context {wl.ctx}); float64 NumPy oracle, {t_total:.1f} s")
    return {"value": val, "unit": unit, "cores": os.cpu_count(), "kind": "oracle",
            "sample": sample}


PREFILL_SAMPLE = 2


def run_reference(args, rank, world, device):
    """The oracle arm: rank 0 times the oracle on the host cores, each step one layer of the
    workload for the first sequence's first new token (the held layers in turn), so that the
    whole run stays within minutes; the value is µs per token per layer (tokens/s for
    prefill, from the first PREFILL_SAMPLE tokens of the chunk per step)."""
    if rank != 0:
        return None
    wl = Workload(args, device, args.workload)
    n_tok = PREFILL_SAMPLE if wl.prefill else 1
    runs = [oracle_sample(args, wl, layers=[l], n_tokens=n_tok) for l in wl.layers]
    for i in range(args.warmup):
        runs[i % len(runs)]()
    t = time.perf_counter()
    for i in range(args.steps):
        runs[i % len(runs)]()
    dt = (time.perf_counter() - t) / args.steps
    val, unit = (round(n_tok / dt, 3), "tokens/s") if wl.prefill else \
        (round(dt * 1e6, 1), "us/token/layer")
    sample = (f"per step one layer of {wl.layers} in turn for the first "
              f"{'new token' if n_tok == 1 else f'{n_tok} tokens of the chunk'} of sequence 0")
    return {
        "impl": "reference", "metric": METRIC, "value": val, "unit": unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1000, 2), "higher_is_better": bool(wl.prefill),
        "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same inputs as the CUDA arm)",
        "config": dict(wl.config(), sample=sample),
        "cpu_baseline": {"value": val, "unit": unit, "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": val, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------------------------ main ----

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="stack_decode",
                    choices=["stack_decode", "stack_prefill", "stack_verify", "swa_decode",
                             "nope_decode"])
    ap.add_argument("--seqs", type=int, default=8, help="prefill: sequences per step")
    ap.add_argument("--chunk", type=int, default=2048,
                    help="prefill: new tokens per sequence; stack_verify: tokens per sequence")
    ap.add_argument("--attn-form", default="natural", choices=["natural", "decode", "prefill"],
                    help="stack_verify: force beam_attn's split-K decode form or its query-tile "
                         "prefill form (natural: the library's own choice)")
    ap.add_argument("--no-prefill", action="store_true",
                    help="stack_decode: skip the prefill object (same stack, same weights)")
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--context", type=int, default=100_000)
    ap.add_argument("--kv", default="bf16", choices=["bf16", "fp8"])
    ap.add_argument("--experts", default="bf16", choices=["bf16", "nvfp4", "fp8"],
                    help="expert weight format of the MoE layers (decode only for nvfp4, fp8)")
    ap.add_argument("--lm-head-vocab", type=int, default=0,
                    help="also time the LM head after the stack over this many vocabulary rows "
                         "(beside the step; 0: off)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.lm_head_vocab and args.workload == "stack_prefill":
        ap.error("--lm-head-vocab is timed for decode workloads")
    if args.experts != "bf16":
        args.no_prefill = True   # the stack_decode line's prefill object stays BF16
    if args.workload == "stack_verify" and not 1 <= args.chunk <= 16:
        ap.error("stack_verify takes 1-16 new tokens per sequence (--chunk)")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.warmup < 3:
        args.warmup = 3
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device(device))
    if args.impl == "reference":
        res = run_reference(args, rank, world, device)
    else:
        res = run_ours(args, rank, world, device)
    emit(res, rank)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
