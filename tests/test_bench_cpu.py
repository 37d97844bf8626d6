"""bench.py on the CPU: the reference arm's JSON line and the roofline's byte count.

The reference arm times the float64 oracle on a bounded sample of the headline workload.
It needs no GPU, so its output contract is checked here.
"""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] >= 3   # the contract's minimum warm-up
    assert d["config"]["workload"] == "decode_sq1024_h64_topk640_ragged"
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] == d["value"] and cpu["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_launch_count_per_call():
    # queue path (no split, at most DSA_ORDER_MAX_TOKENS tokens): order kernel + fused
    # kernel; split path and longer batches: a memset + the fused kernel
    import bench
    from top_sparse_mla_gb300 import native
    native.library()
    cases = [((1024, 64, 640, 128), 2), ((2123, 64, 640, 128), 2), ((1, 64, 640, 128), 1),
             ((64, 64, 640, 128), 2), ((32, 64, 640, 128), 1), ((4, 64, 128, 64), 2),
             ((native.DSA_ORDER_MAX_TOKENS + 1, 64, 640, 128), 1)]
    for (s_q, h_q, topk, n_swa), want in cases:
        p = native.dsa_params_init(s_q, h_q, topk, n_swa, 1 << 20, 1 << 20)
        assert bench.kernels_per_call(p, 152) == want, (s_q, topk)


def test_algorithmic_bytes_of_the_headline_workload():
    # the valid gathered rows (656 B each) plus, per token, q (64 heads x 576 bf16), the
    # codes and scales of the output, the index row, the length and the position
    import bench
    from top_sparse_mla_gb300 import workloads as W
    w = W.make("decode1024")
    n_valid = int(W.n_valid_rows(w).sum())
    assert n_valid == 360224
    assert bench.algorithmic_bytes(w) == 349037056
