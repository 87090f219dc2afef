import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: large CPU work")


@pytest.fixture(scope="session", autouse=True)
def native_library():
    """Build libtt_denoise.so in-tree if it is missing or older than its sources."""
    from block_wise_diffusion_denoise_b300 import build
    return build.build()


def pytest_terminal_summary(terminalreporter):
    """What the unmasking parity tests compared, per test: sequences checked against the
    float64 oracle, how many of them matched its decisions bit for bit, how many differed
    inside the near-tau or fallback-tie bands, and the positions compared."""
    support = sys.modules.get("tests.support")
    if support is None or not support.REPORT:
        return
    tr = terminalreporter
    tr.section("unmasking parity coverage")
    tr.write_line(f"{'test':60s} {'seqs':>6s} {'exact':>6s} {'near-tau':>8s} {'fb-tie':>6s} "
                  f"{'positions':>9s} {'near-tau pos':>12s} {'rule-only':>9s}")
    for name, st in support.REPORT.items():
        tr.write_line(f"{name[:60]:60s} {st.sequences:6d} {st.exact:6d} {st.near_tau_seqs:8d} "
                      f"{st.fallback_tie_seqs:6d} {st.positions:9d} {st.near_tau_positions:12d} {st.rule_only:9d}")
