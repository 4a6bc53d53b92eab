import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


@pytest.fixture(autouse=True)
def _parity_test_id(request):
    """Names the running test in the parity ledger (tests/parity.py)."""
    mod = sys.modules.get("parity")
    if mod is not None:
        mod.CURRENT_TEST[0] = request.node.nodeid
    yield


def pytest_terminal_summary(terminalreporter):
    """A short account of every oracle comparison of the run, printed even under -q: how many
    met the stated bars, how many relied on the widened bar of chained steps, and the closest
    calls against the stated bars."""
    mod = sys.modules.get("parity")
    if mod is None or not mod.LEDGER:
        return
    led = mod.LEDGER
    within = [r for r in led if r[2] <= r[4] and r[3] <= r[5]]
    outside = [r for r in led if not (r[2] <= r[4] and r[3] <= r[5])]
    tests = {r[0] for r in led}
    w = terminalreporter.write_line
    w(f"parity: {len(led)} element-wise comparisons with the oracle in {len(tests)} tests; "
      f"{len(within)} within the stated bars (bf16 2e-2 / 1e-3, fp8 KV 5e-2 / 2e-3)")
    if outside:
        chained = [r for r in outside if r[6] == "chained"]
        worst = max(outside, key=lambda r: r[3] / r[5])
        w(f"parity: {len(outside)} outside them, {len(chained)} of these chained outputs held "
          f"to the widened bar (oracle self-divergence x3); largest mean-rel {worst[3]:.2e} "
          f"({worst[1]}, {worst[0].split('::')[-1]})")
        by_test = {}
        for r in outside:
            by_test.setdefault(r[0].split("::")[-1], []).append(r)
        for name, rs in sorted(by_test.items()):
            wr = max(rs, key=lambda r: r[3] / r[5])
            w(f"parity:   outside in {name}: {len(rs)} outputs, largest mean-rel {wr[3]:.2e} "
              f"max-abs-rel {wr[2]:.2e} ({wr[1]}, {wr[6]})")
    closest = sorted(within, key=lambda r: -max(r[2] / r[4], r[3] / r[5]))[:3]
    for r in closest:
        w(f"parity: closest within: {r[1]} max-abs-rel {r[2]:.2e} mean-rel {r[3]:.2e} "
          f"({r[0].split('::')[-1]})")
