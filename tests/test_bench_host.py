"""bench.py's algorithmic-byte accounting (the numerator of every HBM roofline fraction) against
the per-unit figures worked out from the Beam shapes: a sliding-window MoE layer at batch 1
reads 846.24 MB (QKV+gate 146.80, o_proj 62.91, FP32 router 5.24, 8 experts 629.15, a
512-key BF16 window 2.10), the NoPE layer over 100,000 cached keys 1.254 GB, a dense layer
838.90 MB and an MoE layer without KV 844.15 MB; one BF16 expert 78.64 MB, one NVFP4 expert
22.12 MB (codes, e4m3 block scales, two FP32 matrix scales)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from synth import BEAM  # noqa: E402

KV_PER_KEY_BF16 = BEAM.n_kv * BEAM.head_dim * 2 * 2     # K and V of 8 heads x 128, bf16


def test_layer_bytes_per_unit():
    assert bench.expert_bytes(BEAM) == 3 * 5120 * 2560 * 2
    assert bench.expert_bytes(BEAM, "nvfp4") == 3 * 5120 * 2560 // 2 + 3 * 5120 * 2560 // 16 + 8
    # FP8: a byte per element plus one FP32 scale per 128 x 128 block (40 x 40 + 40 x 20)
    assert bench.expert_bytes(BEAM, "fp8") == 3 * 5120 * 2560 + 4 * (40 * 40 + 40 * 20)
    swa = bench.layer_bytes(BEAM, False, 8, 512 * KV_PER_KEY_BF16)
    assert abs(swa / 1e6 - 846.24) < 0.005
    nope = bench.layer_bytes(BEAM, False, 8, 100_001 * KV_PER_KEY_BF16)
    assert abs(nope / 1e9 - 1.2538) < 5e-4
    assert abs(bench.layer_bytes(BEAM, True, 0, 0) / 1e6 - 838.90) < 0.005
    assert abs(bench.layer_bytes(BEAM, False, 8, 0) / 1e6 - 844.15) < 0.005
    # NVFP4 experts change only the experts' share
    d = bench.layer_bytes(BEAM, False, 8, 0) - bench.layer_bytes(BEAM, False, 8, 0, "nvfp4")
    assert d == 8 * (bench.expert_bytes(BEAM) - bench.expert_bytes(BEAM, "nvfp4"))


def test_traffic_entries_are_per_call():
    """profiles/traffic.json holds DRAM bytes per call of the one-token dense-MLP and expert
    calls (BF16, FP8, NVFP4): each lies within a few percent above its algorithmic bytes (no
    re-reads) and is the sum of its kernels' read and write bytes; entries whose sources
    changed since the capture report None."""
    import json
    d = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for key, fmt in (("moe_decode_t1", "bf16"), ("moe_decode_nvfp4_t1", "nvfp4"),
                     ("moe_decode_fp8_t1", "fp8")):
        assert algo_ok(d[key]["bytes_per_launch"], 8 * bench.expert_bytes(BEAM, fmt)), key
        t = bench.ncu_traffic(key)
        assert t is None or t == d[key]["bytes_per_launch"]
    dense = 3 * BEAM.hidden * BEAM.d_ff_dense * 2
    assert algo_ok(d["dense_decode_t1"]["bytes_per_launch"], dense)
    for key in ("dense_decode_t1", "moe_decode_t1", "moe_decode_fp8_t1", "moe_decode_nvfp4_t1"):
        e = d[key]
        assert e["bytes_per_launch"] == sum(r + w for r, w in e["kernels"].values()), key
    assert bench.ncu_traffic("moe_decode_t8") is None


def algo_ok(traffic, algo):
    return algo <= traffic < 1.05 * algo
