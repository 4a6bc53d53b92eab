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
