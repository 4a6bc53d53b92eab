"""Seeded synthetic inputs for the Beam decoder layer.

Shapes follow the Beam architecture as described on the vLLM "Reflection Beam 1.0" page
(section "Beam model architecture": hidden 5120, 48 query / 8 KV heads of dim 128, a 512-token
sliding window, 256 experts in 8 groups with top-4 groups / top-8 experts and d_ff 2560, dense
SwiGLU d_ff 20480 on layers 0-2) plus a tiny shape of the same structure for CPU-speed tests.

Value distributions (stated choices, the pages give none):
  projection weights          N(0, 0.02), stored BF16
  RMSNorm gains, Q/K gains    1 + N(0, 0.1), stored BF16 (so a kernel that drops a gain fails)
  per-head gate bias          N(0, 1), stored BF16
  router weights              N(0, 0.02), FP32
  router correction bias      N(0, 0.01), FP32
  activations / embeddings    N(0, 1), stored BF16
  prior KV-cache contents     N(0, 1); BF16, or FP8-e4m3 codes of N(0,1)/scale

Every tensor gets its own seed, derived from (seed, layer, tensor name[, expert]) with CRC32,
so any tensor can be regenerated alone.  Tensors are drawn with torch's generator on the
device they are made on; the CPU and CUDA streams differ, so a parity test draws once and
hands the same tensor (copied to the host) to the oracle.

Nothing here computes any part of the layer.
"""
from __future__ import annotations

import dataclasses
import zlib

import torch


@dataclasses.dataclass(frozen=True)
class BeamShape:
    hidden: int
    n_q: int
    n_kv: int
    head_dim: int
    window: int
    n_experts: int
    n_groups: int
    topk_groups: int
    topk: int
    d_ff_expert: int
    d_ff_dense: int
    n_layers: int = 6
    dense_layers: tuple = (0,)
    route_scale: float = 2.5
    rope_theta: float = 10000.0
    ssmax_base: float = 2048.0
    ssmax_exp: float = 0.1
    eps: float = 1e-6

    @property
    def q_rows(self) -> int:
        return self.n_q * self.head_dim

    @property
    def kv_rows(self) -> int:
        return self.n_kv * self.head_dim

    @property
    def qkvg_rows(self) -> int:
        return 2 * self.q_rows + 2 * self.kv_rows


# Tiny Beam-shaped stack: 6 layers, layer 0 dense, layers 1-5 MoE, layer 5 full attention.
TINY = BeamShape(hidden=256, n_q=4, n_kv=2, head_dim=64, window=16, n_experts=16, n_groups=4,
                 topk_groups=2, topk=4, d_ff_expert=128, d_ff_dense=512, n_layers=6,
                 dense_layers=(0,))

# Full-width Beam layer; the truncated stack has layers 0-2 dense and 3-5 MoE.
BEAM = BeamShape(hidden=5120, n_q=48, n_kv=8, head_dim=128, window=512, n_experts=256,
                 n_groups=8, topk_groups=4, topk=8, d_ff_expert=2560, d_ff_dense=20480,
                 n_layers=6, dense_layers=(0, 1, 2))


def derived_seed(seed: int, *names) -> int:
    key = "/".join(str(x) for x in (seed,) + names).encode()
    return zlib.crc32(key) & 0x7FFFFFFF


def normal(shape, std, mean, seed, names, device="cpu", dtype=torch.bfloat16):
    """N(mean, std) drawn in FP32 with a seed derived from `names`, then cast to `dtype`."""
    g = torch.Generator(device=device)
    g.manual_seed(derived_seed(seed, *names))
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x.to(dtype)


def expert_weights(shape: BeamShape, layer: int, seed: int, device="cpu", experts=None):
    """gate/up [E, 2F, H] and down [E, H, F] BF16 weights, drawn one expert at a time."""
    E, F, H = shape.n_experts, shape.d_ff_expert, shape.hidden
    ids = range(E) if experts is None else experts
    n = len(ids)
    w_gu = torch.empty((n, 2 * F, H), dtype=torch.bfloat16, device=device)
    w_dn = torch.empty((n, H, F), dtype=torch.bfloat16, device=device)
    for i, e in enumerate(ids):
        w_gu[i] = normal((2 * F, H), 0.02, 0.0, seed, (layer, "w_gate_up", e), device)
        w_dn[i] = normal((H, F), 0.02, 0.0, seed, (layer, "w_down", e), device)
    return w_gu, w_dn


def uniform_codes(shape, low, high, seed, names, device="cpu"):
    """Integers uniform in [low, high) as uint8, with a seed derived from `names`."""
    g = torch.Generator(device=device)
    g.manual_seed(derived_seed(seed, *names))
    return torch.randint(low, high, shape, generator=g, device=device, dtype=torch.int32).to(torch.uint8)


# NVFP4 expert weights: every byte of e2m1 code pairs uniform (all 16 codes are numbers),
# block scales uniform over the e4m3 codes of [0.5, 2) (exponent fields 6 and 7), and one matrix
# scale of 0.004 per expert matrix, so that weights are of the size of the N(0, 0.02) BF16 ones.
NVFP4_SCALE_CODES = (0x30, 0x40)
NVFP4_MATRIX_SCALE = 0.004


def expert_weights_nvfp4(shape: BeamShape, layer: int, seed: int, device="cpu", experts=None):
    """NVFP4 gate/up and down weights of the experts (a dict of tensors): codes [E][2F][H/2]
    and [E][H][F/2] (uint8, even element in the low nibble), e4m3 block scales [E][2F][H/16]
    and [E][H][F/16] (uint8), FP32 matrix scales [E]."""
    E, F, H = shape.n_experts, shape.d_ff_expert, shape.hidden
    ids = list(range(E) if experts is None else experts)
    n = len(ids)
    out = {
        "gate_up": torch.empty((n, 2 * F, H // 2), dtype=torch.uint8, device=device),
        "gate_up_scale": torch.empty((n, 2 * F, H // 16), dtype=torch.uint8, device=device),
        "gate_up_global": torch.full((n,), NVFP4_MATRIX_SCALE, dtype=torch.float32, device=device),
        "down": torch.empty((n, H, F // 2), dtype=torch.uint8, device=device),
        "down_scale": torch.empty((n, H, F // 16), dtype=torch.uint8, device=device),
        "down_global": torch.full((n,), NVFP4_MATRIX_SCALE, dtype=torch.float32, device=device),
    }
    lo, hi = NVFP4_SCALE_CODES
    for i, e in enumerate(ids):
        out["gate_up"][i] = uniform_codes((2 * F, H // 2), 0, 256, seed, (layer, "nvfp4_gu", e), device)
        out["gate_up_scale"][i] = uniform_codes((2 * F, H // 16), lo, hi, seed, (layer, "nvfp4_gu_s", e), device)
        out["down"][i] = uniform_codes((H, F // 2), 0, 256, seed, (layer, "nvfp4_dn", e), device)
        out["down_scale"][i] = uniform_codes((H, F // 16), lo, hi, seed, (layer, "nvfp4_dn_s", e), device)
    return out


# Block-scaled FP8 expert weights: e4m3 magnitude codes uniform over [0x20, 0x50) (0.125 to
# 7.5, every code a finite number) with a uniform sign bit, and FP32 scales uniform in
# [0.004, 0.012) per 128 x 128 block, so that weights are of the size of the N(0, 0.02) BF16 ones.
FP8_CODES = (0x20, 0x50)
FP8_SCALE_RANGE = (0.004, 0.012)


def fp8_codes(shape, seed, names, device="cpu"):
    mag = uniform_codes(shape, FP8_CODES[0], FP8_CODES[1], seed, (*names, "mag"), device)
    sign = uniform_codes(shape, 0, 2, seed, (*names, "sign"), device)
    return mag | (sign << 7)


def fp8_scales(shape, seed, names, device="cpu"):
    g = torch.Generator(device=device)
    g.manual_seed(derived_seed(seed, *names))
    lo, hi = FP8_SCALE_RANGE
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32) * (hi - lo) + lo


def expert_weights_fp8(shape: BeamShape, layer: int, seed: int, device="cpu", experts=None):
    """Block-scaled FP8 gate/up and down weights of the experts (a dict of tensors): e4m3
    codes [E][2F][H] and [E][H][F] (uint8), FP32 scales [E][2F/128][H/128] and
    [E][H/128][F/128] (blocks rounded up)."""
    E, F, H = shape.n_experts, shape.d_ff_expert, shape.hidden
    ids = list(range(E) if experts is None else experts)
    n = len(ids)

    def blocks(x):
        return -(-x // 128)

    out = {
        "gate_up": torch.empty((n, 2 * F, H), dtype=torch.uint8, device=device),
        "gate_up_scale": torch.empty((n, blocks(2 * F), blocks(H)), dtype=torch.float32, device=device),
        "down": torch.empty((n, H, F), dtype=torch.uint8, device=device),
        "down_scale": torch.empty((n, blocks(H), blocks(F)), dtype=torch.float32, device=device),
    }
    for i, e in enumerate(ids):
        out["gate_up"][i] = fp8_codes((2 * F, H), seed, (layer, "fp8_gu", e), device)
        out["gate_up_scale"][i] = fp8_scales((blocks(2 * F), blocks(H)), seed, (layer, "fp8_gu_s", e), device)
        out["down"][i] = fp8_codes((H, F), seed, (layer, "fp8_dn", e), device)
        out["down_scale"][i] = fp8_scales((blocks(H), blocks(F)), seed, (layer, "fp8_dn_s", e), device)
    return out


def attention_weights(shape: BeamShape, layer: int, seed: int = 0, device="cpu"):
    """Norm gains and the attention sublayer's weights of one layer."""
    H, D = shape.hidden, shape.head_dim
    return {
        "attn_pre": normal((H,), 0.1, 1.0, seed, (layer, "attn_pre"), device),
        "attn_post": normal((H,), 0.1, 1.0, seed, (layer, "attn_post"), device),
        "mlp_pre": normal((H,), 0.1, 1.0, seed, (layer, "mlp_pre"), device),
        "mlp_post": normal((H,), 0.1, 1.0, seed, (layer, "mlp_post"), device),
        "w_qkvg": normal((shape.qkvg_rows, H), 0.02, 0.0, seed, (layer, "w_qkvg"), device),
        "q_norm": normal((D,), 0.1, 1.0, seed, (layer, "q_norm"), device),
        "k_norm": normal((D,), 0.1, 1.0, seed, (layer, "k_norm"), device),
        "gate_bias": normal((shape.n_q,), 1.0, 0.0, seed, (layer, "gate_bias"), device),
        "w_o": normal((H, shape.q_rows), 0.02, 0.0, seed, (layer, "w_o"), device),
    }


def router_weights(shape: BeamShape, layer: int, seed: int = 0, device="cpu", attempt: int = 0):
    """FP32 router rows [E][H] and correction bias [E]. attempt > 0 gives an independent
    redraw (synth.tie_free walks the attempts); attempt 0 is the layer's first draw."""
    E, H = shape.n_experts, shape.hidden
    tag = () if attempt == 0 else (attempt,)
    return {
        "router": normal((E, H), 0.02, 0.0, seed, (layer, "router", *tag), device, torch.float32),
        "corr_bias": normal((E,), 0.01, 0.0, seed, (layer, "corr_bias", *tag), device,
                            torch.float32),
    }


def dense_weights(shape: BeamShape, layer: int, seed: int = 0, device="cpu"):
    H, Fd = shape.hidden, shape.d_ff_dense
    return {
        "w_gate_up": normal((2 * Fd, H), 0.02, 0.0, seed, (layer, "dense_gate_up"), device),
        "w_down": normal((H, Fd), 0.02, 0.0, seed, (layer, "dense_down"), device),
    }


def lm_head_weights(shape: BeamShape, vocab: int, seed: int = 0, device="cpu", std=0.02):
    """Final norm gains [H] (N(1, 0.1), like the other norms) and vocabulary rows [V][H]."""
    H = shape.hidden
    return {
        "final_norm": normal((H,), 0.1, 1.0, seed, ("final_norm",), device),
        "w_lm": normal((vocab, H), std, 0.0, seed, ("lm_head",), device),
    }


def layer_weights(shape: BeamShape, layer: int, seed: int = 0, device="cpu",
                  dense: bool | None = None, with_experts: bool = True):
    """All weights of one layer as a dict of tensors (row-major [out][in])."""
    if dense is None:
        dense = layer in shape.dense_layers
    w = attention_weights(shape, layer, seed, device)
    if dense:
        w.update(dense_weights(shape, layer, seed, device))
    else:
        w.update(router_weights(shape, layer, seed, device))
        if with_experts:
            w["w_gate_up"], w["w_down"] = expert_weights(shape, layer, seed, device)
    return w


def activations(T: int, H: int, seed: int, name: str = "x", device="cpu"):
    return normal((T, H), 1.0, 0.0, seed, ("act", name), device)


def kv_cache(shape: BeamShape, n_seqs: int, capacity: int, seed: int, layer: int = 0,
             fp8: bool = False, k_scale: float = 1.0, v_scale: float = 1.0, device="cpu"):
    """Prior cache contents [S][Hkv][capacity][D]: N(0,1) values (BF16), or for an FP8
    cache the e4m3 codes (as uint8) of N(0,1)/scale, cast by torch."""
    dims = (n_seqs, shape.n_kv, capacity, shape.head_dim)
    out = {}
    for name, sc in (("k", k_scale), ("v", v_scale)):
        x = normal(dims, 1.0, 0.0, seed, (layer, "cache", name), device, torch.float32)
        if fp8:
            out[name] = (x / sc).to(torch.float8_e4m3fn).view(torch.uint8)
        else:
            out[name] = x.to(torch.bfloat16)
    return out


def decode_positions(contexts, device="cpu"):
    """One new token per sequence: seq_id s, 1-based position context_s + 1."""
    seq = torch.arange(len(contexts), dtype=torch.int32, device=device)
    pos = torch.tensor([c + 1 for c in contexts], dtype=torch.int32, device=device)
    return seq, pos


def prefill_positions(contexts, chunk, device="cpu"):
    """`chunk` new tokens per sequence after `context_s` cached ones, sequence-major."""
    seq, pos = [], []
    for s, c in enumerate(contexts):
        seq += [s] * chunk
        pos += list(range(c + 1, c + chunk + 1))
    return (torch.tensor(seq, dtype=torch.int32, device=device),
            torch.tensor(pos, dtype=torch.int32, device=device))
