import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print every GPU parity comparison's measured agreement (also on a green run)."""
    try:
        import parity
    except Exception:
        return
    if not parity.RECORDS:
        return
    terminalreporter.write_sep("-", "measured parity (CUDA path vs oracle)")
    for r in parity.RECORDS:
        terminalreporter.write_line(
            f"{r['label']}: fp8 within 1 step {r['fp8_within_1']:.6f} ({r['fp8_misses']}/{r['codes']}), "
            f"exact {r['fp8_exact']:.6f}, scale mismatches {r['sf_mismatch_blocks']}/{r['blocks']} "
            f"(band {r['sf_band_blocks']}), max abs {r['max_abs']:.2e}, rel L2 {r['rel_l2']:.2e}")
