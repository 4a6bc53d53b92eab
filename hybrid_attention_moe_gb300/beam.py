"""Python binding of libbeam.so (ctypes). Argument marshalling only: every step runs in the
library's CUDA kernels; torch supplies device memory and streams.

The functions carry the C names (beam_boundary_norm, beam_qkv_gate, beam_attn, beam_route,
beam_moe, beam_dense_mlp, ...) and take torch tensors. There is no fallback: if the library
is not built, or a call returns an error status, a BeamError is raised.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libbeam.so")

BEAM_KV_BF16, BEAM_KV_FP8_E4M3 = 0, 1
BEAM_ATTN_SWA_ROPE, BEAM_ATTN_NOPE_SSMAX = 0, 1
DEV_BAD_POSITION, DEV_BAD_SEQ, DEV_BAD_EXPERT, DEV_TIMEOUT = 0x1, 0x2, 0x4, 0x8


class BeamError(RuntimeError):
    pass


class KVCacheC(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("dtype", ctypes.c_int32),
                ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float),
                ("num_seqs", ctypes.c_int32), ("capacity", ctypes.c_int32),
                ("window", ctypes.c_int32)]


class LayerCfgC(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_q", ctypes.c_int32), ("n_kv", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("kind", ctypes.c_int32),
                ("rope_theta", ctypes.c_float), ("ssmax_base", ctypes.c_float),
                ("ssmax_exp", ctypes.c_float), ("eps", ctypes.c_float),
                ("n_experts", ctypes.c_int32), ("n_groups", ctypes.c_int32),
                ("topk_groups", ctypes.c_int32), ("topk", ctypes.c_int32),
                ("d_ff_expert", ctypes.c_int32), ("d_ff_dense", ctypes.c_int32),
                ("route_scale", ctypes.c_float)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_Z = ctypes.c_size_t
_SIGS = {
    "beam_boundary_norm": [_P, _P, _P, _P, _P, _I, _I, _I, _F, _P],
    "beam_qkv_gate": [_P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P, _Z, _P],
    "beam_attn": [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _Z, _P],
    "beam_route": [_P, _P, _P, _P, _I, _P, _P, _P, _P, _Z, _P],
    "beam_moe": [_P, _P, _P, _P, _P, _P, _I, _P, _P, _Z, _P],
    "beam_moe_nvfp4": [_P, _P, _P, _P, _P, _I, _P, _P, _Z, _P],
    "beam_moe_fp8": [_P, _P, _P, _P, _P, _I, _P, _P, _Z, _P],
    "beam_dense_mlp": [_P, _P, _P, _P, _I, _P, _P, _Z, _P],
    "beam_workspace_bytes": [_P, _I, _I],
    "beam_kv_cache_bytes": [_I, _I, _I, _I, _I],
    "beam_get_device_status": [_P, ctypes.POINTER(ctypes.c_uint32)],
    "beam_status_string": [_I],
    "beam_launch_count": [],
    "beam_last_cuda_error": [],
    "beam_gemm_bf16": [_P, _I, _I, _I, _P, _I, _I, _P, _I, _I, _P],
    "beam_route_noalloc": [_P, _P, _P, _P, _I, _P, _P, _P],
    "beam_lm_head": [_P, _P, _I, _I, _I, _F, _P, _P],
    "beam_selftest_wait_timeout": [_P],
}
_RES = {"beam_workspace_bytes": _Z, "beam_kv_cache_bytes": _Z,
        "beam_status_string": ctypes.c_char_p, "beam_launch_count": ctypes.c_uint64,
        "beam_last_cuda_error": ctypes.c_char_p}

_lib = None


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise BeamError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() or "
                            "hybrid_attention_moe_gb300/build.py")
        L = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = _RES.get(name, ctypes.c_int)
        _lib = L
    return _lib


def _check(status, what):
    if status != 0:
        msg = lib().beam_status_string(status).decode()
        if status == 3:
            msg += " [" + lib().beam_last_cuda_error().decode() + "]"
        raise BeamError(f"{what} failed: {msg} ({status})")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


@dataclasses.dataclass
class LayerCfg:
    hidden: int
    n_q: int
    n_kv: int
    head_dim: int
    kind: int
    n_experts: int
    n_groups: int
    topk_groups: int
    topk: int
    d_ff_expert: int
    d_ff_dense: int
    rope_theta: float = 10000.0
    ssmax_base: float = 2048.0
    ssmax_exp: float = 0.1
    eps: float = 1e-6
    route_scale: float = 2.5

    @classmethod
    def from_shape(cls, shape, kind):
        return cls(hidden=shape.hidden, n_q=shape.n_q, n_kv=shape.n_kv,
                   head_dim=shape.head_dim, kind=kind, n_experts=shape.n_experts,
                   n_groups=shape.n_groups, topk_groups=shape.topk_groups, topk=shape.topk,
                   d_ff_expert=shape.d_ff_expert, d_ff_dense=shape.d_ff_dense,
                   rope_theta=shape.rope_theta, ssmax_base=shape.ssmax_base,
                   ssmax_exp=shape.ssmax_exp, eps=shape.eps, route_scale=shape.route_scale)

    def c(self):
        return LayerCfgC(self.hidden, self.n_q, self.n_kv, self.head_dim, self.kind,
                         self.rope_theta, self.ssmax_base, self.ssmax_exp, self.eps,
                         self.n_experts, self.n_groups, self.topk_groups, self.topk,
                         self.d_ff_expert, self.d_ff_dense, self.route_scale)


@dataclasses.dataclass
class KVCache:
    """One layer's cache: k, v tensors [S][Hkv][capacity][D] (bf16, or uint8 e4m3 codes)."""
    k: torch.Tensor
    v: torch.Tensor
    window: int = 0
    k_scale: float = 1.0
    v_scale: float = 1.0

    @property
    def fp8(self):
        return self.k.dtype == torch.uint8

    def c(self):
        return KVCacheC(self.k.data_ptr(), self.v.data_ptr(),
                        BEAM_KV_FP8_E4M3 if self.fp8 else BEAM_KV_BF16, self.k_scale,
                        self.v_scale, self.k.shape[0], self.k.shape[2], self.window)


class Workspace:
    """Device scratch for the library calls, grown on demand (256-byte aligned)."""

    def __init__(self, device="cuda"):
        self.device = device
        self.buf = None

    def get(self, nbytes):
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.device)
        return self.buf


def workspace_bytes(cfg: LayerCfg, T: int, max_pos: int) -> int:
    c = cfg.c()
    return lib().beam_workspace_bytes(ctypes.byref(c), T, max_pos)


def kv_cache_bytes(num_seqs, n_kv, capacity, head_dim, fp8=False) -> int:
    return lib().beam_kv_cache_bytes(num_seqs, n_kv, capacity, head_dim,
                                     BEAM_KV_FP8_E4M3 if fp8 else BEAM_KV_BF16)


def beam_boundary_norm(x, h, u_out, w_post, w_pre, n, eps, stream=None):
    T, H = h.shape
    _check(lib().beam_boundary_norm(_ptr(x), _ptr(h), _ptr(u_out), _ptr(w_post), _ptr(w_pre),
                                    T, H, n, eps, _stream(stream)), "beam_boundary_norm")


def beam_qkv_gate(cfg: LayerCfg, u, w_qkvg, q_norm_w, k_norm_w, seq_id, pos, q_out, g_out,
                  cache: KVCache, ws: torch.Tensor, stream=None):
    c, kc = cfg.c(), cache.c()
    _check(lib().beam_qkv_gate(ctypes.byref(c), _ptr(u), _ptr(w_qkvg), _ptr(q_norm_w),
                               _ptr(k_norm_w), _ptr(seq_id), _ptr(pos), u.shape[0], _ptr(q_out),
                               _ptr(g_out), ctypes.byref(kc), _ptr(ws), ws.numel(),
                               _stream(stream)), "beam_qkv_gate")


def beam_attn(cfg: LayerCfg, q, g, gate_bias, cache: KVCache, seq_id, pos, max_pos, w_o, out,
              ws: torch.Tensor, stream=None, max_q_per_seq=None):
    """max_q_per_seq: most tokens of one sequence in the call (1 for decode); None = T."""
    c, kc = cfg.c(), cache.c()
    mq = q.shape[0] if max_q_per_seq is None else int(max_q_per_seq)
    _check(lib().beam_attn(ctypes.byref(c), _ptr(q), _ptr(g), _ptr(gate_bias), ctypes.byref(kc),
                           _ptr(seq_id), _ptr(pos), q.shape[0], int(max_pos), max(1, mq),
                           _ptr(w_o), _ptr(out), _ptr(ws), ws.numel(), _stream(stream)),
           "beam_attn")


def beam_route(cfg: LayerCfg, u, w_router, corr_bias, logits, topk_idx, topk_w,
               ws: torch.Tensor, stream=None):
    c = cfg.c()
    _check(lib().beam_route(ctypes.byref(c), _ptr(u), _ptr(w_router), _ptr(corr_bias),
                            u.shape[0], _ptr(logits), _ptr(topk_idx), _ptr(topk_w), _ptr(ws),
                            ws.numel(), _stream(stream)), "beam_route")


def beam_moe(cfg: LayerCfg, u, topk_idx, topk_w, w_gate_up, w_down, out, ws: torch.Tensor,
             stream=None):
    c = cfg.c()
    _check(lib().beam_moe(ctypes.byref(c), _ptr(u), _ptr(topk_idx), _ptr(topk_w),
                          _ptr(w_gate_up), _ptr(w_down), u.shape[0], _ptr(out), _ptr(ws),
                          ws.numel(), _stream(stream)), "beam_moe")


class NvFp4ExpertsC(ctypes.Structure):
    _fields_ = [("gate_up", ctypes.c_void_p), ("gate_up_scale", ctypes.c_void_p),
                ("gate_up_global", ctypes.c_void_p), ("down", ctypes.c_void_p),
                ("down_scale", ctypes.c_void_p), ("down_global", ctypes.c_void_p)]


def beam_moe_nvfp4(cfg: LayerCfg, u, topk_idx, topk_w, experts: dict, out, ws: torch.Tensor,
                   stream=None):
    """experts: the tensors of synth.expert_weights_nvfp4 (gate_up, gate_up_scale,
    gate_up_global, down, down_scale, down_global)."""
    c = cfg.c()
    w = NvFp4ExpertsC(*[_ptr(experts[k]) for k in ("gate_up", "gate_up_scale", "gate_up_global",
                                                    "down", "down_scale", "down_global")])
    _check(lib().beam_moe_nvfp4(ctypes.byref(c), _ptr(u), _ptr(topk_idx), _ptr(topk_w),
                                ctypes.byref(w), u.shape[0], _ptr(out), _ptr(ws), ws.numel(),
                                _stream(stream)), "beam_moe_nvfp4")


class Fp8ExpertsC(ctypes.Structure):
    _fields_ = [("gate_up", ctypes.c_void_p), ("gate_up_scale", ctypes.c_void_p),
                ("down", ctypes.c_void_p), ("down_scale", ctypes.c_void_p)]


def beam_moe_fp8(cfg: LayerCfg, u, topk_idx, topk_w, experts: dict, out, ws: torch.Tensor,
                 stream=None):
    """experts: the tensors of synth.expert_weights_fp8 (gate_up, gate_up_scale, down,
    down_scale)."""
    c = cfg.c()
    w = Fp8ExpertsC(*[_ptr(experts[k]) for k in ("gate_up", "gate_up_scale", "down",
                                                  "down_scale")])
    _check(lib().beam_moe_fp8(ctypes.byref(c), _ptr(u), _ptr(topk_idx), _ptr(topk_w),
                              ctypes.byref(w), u.shape[0], _ptr(out), _ptr(ws), ws.numel(),
                              _stream(stream)), "beam_moe_fp8")


def beam_dense_mlp(cfg: LayerCfg, u, w_gate_up, w_down, out, ws: torch.Tensor, stream=None):
    c = cfg.c()
    _check(lib().beam_dense_mlp(ctypes.byref(c), _ptr(u), _ptr(w_gate_up), _ptr(w_down),
                                u.shape[0], _ptr(out), _ptr(ws), ws.numel(), _stream(stream)),
           "beam_dense_mlp")


def beam_get_device_status(stream=None) -> int:
    bits = ctypes.c_uint32(0)
    _check(lib().beam_get_device_status(_stream(stream), ctypes.byref(bits)),
           "beam_get_device_status")
    return bits.value


def beam_launch_count() -> int:
    """Kernels the library has launched in this process."""
    return int(lib().beam_launch_count())


def beam_gemm_bf16(a, b, c, stream=None):
    """c = a @ b.T with a [M][K], b [N][K] bf16 and c [M][N] float32 or bfloat16."""
    M, K = a.shape
    N = b.shape[0]
    _check(lib().beam_gemm_bf16(_ptr(a), M, K, a.stride(0), _ptr(b), N, b.stride(0), _ptr(c),
                                c.stride(0), int(c.dtype == torch.bfloat16), _stream(stream)),
           "beam_gemm_bf16")


def beam_lm_head(u, w_lm, logits, softcap=30.0, stream=None):
    """logits [T][V] fp32 = softcap * tanh((u w_lm^T) / softcap); u [T][H] bf16 (final-normed),
    w_lm [V][H] bf16; softcap <= 0: no cap."""
    T, H = u.shape
    V = w_lm.shape[0]
    _check(lib().beam_lm_head(_ptr(u), _ptr(w_lm), T, H, V, float(softcap), _ptr(logits),
                              _stream(stream)), "beam_lm_head")


def beam_route_noalloc(cfg: LayerCfg, u, w_router, corr_bias, topk_idx, topk_w, stream=None):
    """beam_route without caller scratch (the logits live in the library's static array)."""
    c = cfg.c()
    _check(lib().beam_route_noalloc(ctypes.byref(c), _ptr(u), _ptr(w_router), _ptr(corr_bias),
                                    u.shape[0], _ptr(topk_idx), _ptr(topk_w), _stream(stream)),
           "beam_route_noalloc")


def beam_selftest_wait_timeout(stream=None):
    """Runs the library's bounded on-device wait against a barrier nothing completes (see
    include/beam.h); the status word then holds DEV_TIMEOUT."""
    _check(lib().beam_selftest_wait_timeout(_stream(stream)), "beam_selftest_wait_timeout")
