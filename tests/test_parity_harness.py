"""The GPU parity comparator (tests/parity.py) on the CPU: it accepts the oracle's own
output, and each kind of error it exists to catch makes it fail."""

import numpy as np
import pytest

import oracle
import parity
from top_sparse_mla_gb300 import workloads as W


@pytest.fixture(scope="module")
def ref():
    w = W.random_case(601, s_q=4, h_q=16, n_swa_cols=64, n_cmp_cols=192, n_swa_rows=512, n_cmp_rows=2048,
                      n_sentinels=9)
    w.indices[3] = -1                     # one token without a valid column: LSE -inf
    return parity.run_oracle(w)


def _as_gpu(out, lse):
    """A result as the GPU path returns it: fp32 pre-cast output and LSE, and the codes
    its own cast produces from that output."""
    out = out.astype(np.float32).astype(np.float64)
    codes, sf = oracle.mxfp8_cast(out)
    return {"out": out, "lse": lse.astype(np.float32).astype(np.float64), "out_fp8": codes, "out_sf": sf}


def test_accepts_the_oracle_and_small_noise(ref):
    parity.compare(_as_gpu(ref["out"], ref["lse"]), ref, label="self")
    rng = np.random.default_rng(1)
    noisy = ref["out"] + rng.normal(scale=1e-6, size=ref["out"].shape)
    noisy[3] = 0.0                        # the empty token's output is exactly zero on both sides
    parity.compare(_as_gpu(noisy, ref["lse"] + 1e-3), ref, label="noise")


def test_rejects_a_pre_cast_error(ref):
    out = ref["out"].copy()
    out[0, 0, 5] += 3e-2
    with pytest.raises(AssertionError, match="max abs"):
        parity.compare(_as_gpu(out, ref["lse"]), ref)


def test_rejects_a_wrong_lse_and_a_wrong_empty_pattern(ref):
    lse = ref["lse"].copy()
    lse[1, 2] += 3e-2
    with pytest.raises(AssertionError, match="LSE error"):
        parity.compare(_as_gpu(ref["out"], lse), ref)
    lse = ref["lse"].copy()
    lse[3, 0] = 0.0                       # the empty token's -inf replaced
    with pytest.raises(AssertionError, match="-inf"):
        parity.compare(_as_gpu(ref["out"], lse), ref)


def test_rejects_wrong_codes(ref):
    g = _as_gpu(ref["out"], ref["lse"])
    sf = g["out_sf"].copy()
    i = np.argwhere(sf > 0)[0]
    sf[tuple(i)] += 1                     # one scale code off, outside any exemption
    with pytest.raises(AssertionError, match="UE8M0"):
        parity.compare(dict(g, out_sf=sf), ref)
    fp8 = g["out_fp8"].copy()
    flat = fp8.reshape(-1)
    idx = np.arange(0, flat.size, 20)    # 5 % of the codes, two steps up
    flat[idx] = np.where((flat[idx] & 0x7F) < 0x7C, flat[idx] + 2, flat[idx] - 2)
    with pytest.raises(AssertionError, match="E4M3 codes"):
        parity.compare(dict(g, out_fp8=fp8), ref)


def test_rejects_non_finite_output_and_codes_that_do_not_follow_from_it(ref):
    g = _as_gpu(ref["out"], ref["lse"])
    out = g["out"].copy()
    out[2, 1, 7] = np.nan
    with pytest.raises(AssertionError, match="non-finite"):
        parity.compare(dict(g, out=out), ref)
    # codes that are close to the oracle's but are not the cast of the returned output
    fp8 = g["out_fp8"].copy()
    j = np.argwhere((fp8 & 0x7F) > 8)[0]
    fp8[tuple(j)] += 1
    with pytest.raises(AssertionError, match="oracle cast of the kernel"):
        parity.compare(dict(g, out_fp8=fp8), ref)
