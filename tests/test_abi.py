"""The C-ABI library builds for sm_103a, loads without a GPU and exports every entry point
that include/beam.h declares; host-only entry points answer without a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "beam.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(beam_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from hybrid_attention_moe_gb300 import build as b
    try:
        b.nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    b.build()
    from hybrid_attention_moe_gb300 import beam as B
    return B.lib()


def test_header_declares_the_layer_calls():
    names = declared_functions()
    for n in ("beam_boundary_norm", "beam_qkv_gate", "beam_attn", "beam_route", "beam_moe",
              "beam_dense_mlp", "beam_workspace_bytes"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_host_only_entry_points(lib):
    from hybrid_attention_moe_gb300 import beam as B
    assert lib.beam_status_string(0) == b"ok"
    assert lib.beam_status_string(1) == b"invalid argument"
    # KV arithmetic of the Beam page: 9 full layers x 2 x 8 heads x 128 = 36 KiB per token BF16
    assert 9 * B.kv_cache_bytes(1, 8, 1, 128) == 36 * 1024
    assert 9 * B.kv_cache_bytes(1, 8, 1, 128, fp8=True) == 18 * 1024
    assert 9 * B.kv_cache_bytes(1, 8, 1 << 20, 128, fp8=True) == 18 << 30
    import synth
    cfg = B.LayerCfg.from_shape(synth.BEAM, B.BEAM_ATTN_NOPE_SSMAX)
    small = B.workspace_bytes(cfg, 1, 4097)
    big = B.workspace_bytes(cfg, 16384, 102_048)
    assert small % 256 == 0 and big > small
    # QKV scratch alone: 16384 tokens x 14336 rows x fp32
    assert big >= 16384 * 14336 * 4


def test_library_is_built_for_sm_103a(lib):
    from hybrid_attention_moe_gb300 import build as b
    assert "arch=compute_103a,code=sm_103a" in " ".join(b.ARCH)


def test_argument_checks_answer_before_any_launch(lib):
    """beam_lm_head and beam_moe_nvfp4 reject bad arguments (and return at once for T = 0)
    before touching the device: every call below returns from the host-side checks, so the
    16-byte-aligned placeholder addresses are never dereferenced."""
    import ctypes
    import synth
    from hybrid_attention_moe_gb300 import beam as B
    P = ctypes.c_void_p
    a, b, c = P(0x10000), P(0x20000), P(0x30000)
    # LM head: u, w_lm, T, H, V, softcap, logits, stream
    assert lib.beam_lm_head(None, b, 1, 256, 100, 30.0, c, None) == 1
    assert lib.beam_lm_head(a, b, 1, 260, 100, 30.0, c, None) == 1          # H % 8 != 0
    assert lib.beam_lm_head(a, b, 1, 256, 100, float("nan"), c, None) == 1
    assert lib.beam_lm_head(P(0x10008), b, 1, 256, 100, 30.0, c, None) == 1  # misaligned u
    assert lib.beam_lm_head(a, b, 0, 256, 100, 30.0, c, None) == 0          # T = 0: nothing
    # NVFP4 experts: H and d_ff multiples of 128
    cfg = B.LayerCfg.from_shape(synth.BEAM, B.BEAM_ATTN_SWA_ROPE).c()
    ex = B.NvFp4ExpertsC(a, a, a, a, a, a)

    def moe(T, cfg=cfg, ex=ex):
        return lib.beam_moe_nvfp4(ctypes.byref(cfg), a, b, c, ctypes.byref(ex), T, a, a, 1 << 20,
                                  None)
    # from 32 tokens the grouped path: its workspace (BF16 weights of 16 experts among it)
    # does not fit the 1 MB given, BEAM_ERR_INVALID_ARG before any launch
    assert moe(32) == 1 and moe(100) == 1
    assert moe(0) == 0
    odd = B.LayerCfg.from_shape(synth.BEAM, B.BEAM_ATTN_SWA_ROPE).c()
    odd.hidden = 5120 + 64
    assert moe(1, cfg=odd) == 2
    bad = B.NvFp4ExpertsC(a, None, a, a, a, a)
    assert moe(1, ex=bad) == 1


def test_fp8_expert_argument_checks(lib):
    """beam_moe_fp8: H and d_ff multiples of 128, every weight pointer given, a workspace
    large enough; all answered on the host before any launch."""
    import ctypes
    import synth
    from hybrid_attention_moe_gb300 import beam as B
    P = ctypes.c_void_p
    a, b, c = P(0x10000), P(0x20000), P(0x30000)
    cfg = B.LayerCfg.from_shape(synth.BEAM, B.BEAM_ATTN_SWA_ROPE).c()
    ex = B.Fp8ExpertsC(a, a, a, a)

    def moe(T, cfg=cfg, ex=ex):
        return lib.beam_moe_fp8(ctypes.byref(cfg), a, b, c, ctypes.byref(ex), T, a, a, 1 << 20,
                                None)
    # from 32 tokens the grouped path, whose workspace does not fit the 1 MB given
    assert moe(32) == 1 and moe(100) == 1
    assert moe(0) == 0
    odd = B.LayerCfg.from_shape(synth.BEAM, B.BEAM_ATTN_SWA_ROPE).c()
    odd.d_ff_expert = 2560 + 64
    assert moe(1, cfg=odd) == 2
    assert moe(1, ex=B.Fp8ExpertsC(a, None, a, a)) == 1
    assert moe(1, ex=B.Fp8ExpertsC(P(0x10008), a, a, a)) == 1     # misaligned codes
