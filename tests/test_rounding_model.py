"""The operand-rounding model (tests/rounding_model.py) against the float64 oracle: the
fused kernel's split design (hi + lo fp16 parts for q~ and P_b, unscaled E4M3 codes with
the fp32 block scales applied outside the MMAs) meets the parity bar with a wide margin,
and the plain single-fp16 design does not.  This pins, on the CPU, the reason for the
kernel's operand layout: the bar asks for UE8M0 codes that match bit for bit outside a
1e-6 band and E4M3 codes within one step on 99.9 % of elements, which needs the pre-cast
output to about 1e-6 relative; a single fp16 rounding of each operand (2^-11) misses it,
and an E4M3 q~ (the FP8 x FP8 QK^T variant) misses even the 1e-2 relative L2 bound."""

import numpy as np
import pytest

import oracle
from oracle import codecs
from top_sparse_mla_gb300 import workloads as W

import parity
from rounding_model import token_output


def _metrics(w, tokens, design):
    p = oracle.OracleParams(n_swa_cols=w.n_swa_cols)
    sub = parity.subset(w, tokens)
    ref = parity.run_oracle(sub)
    out = np.stack([token_output(design, sub.q[t], sub.norm_w, sub.indices[t], int(sub.topk_length[t]),
                                 int(sub.positions[t]), sub.kv_swa, sub.kv_cmp, p) for t in range(sub.s_q)])
    out = out.astype(np.float32).astype(np.float64)        # the kernel's pre-cast is fp32
    codes, sf = oracle.mxfp8_cast(out)
    same_sf = sf == ref["out_sf"]
    amax = np.max(np.abs(ref["out"].reshape(*sf.shape, 32)), axis=-1)
    outside = (~same_sf) & ~parity.near_power_of_two(amax)
    d = codecs.e4m3_ulp_distance(codes, ref["out_fp8"])
    eq = np.repeat(same_sf[..., None], 32, axis=-1).reshape(codes.shape)
    err = np.abs(out - ref["out"])
    return {"within1": float(np.mean(d[eq] <= 1)), "sf_outside_band": int(outside.sum()),
            "max_abs": float(err.max()), "rel_l2": float(np.linalg.norm(out - ref["out"]) / np.linalg.norm(ref["out"]))}


@pytest.mark.parametrize("name,tokens", [("decode64", range(0, 64, 8)), ("decode1024", range(3, 1024, 128))])
def test_split_design_meets_the_bar_and_single_fp16_and_fp8_q_do_not(name, tokens):
    w = W.make(name)
    split = _metrics(w, list(tokens), "split")
    single = _metrics(w, list(tokens), "single")
    # the kernel's design: the bar with margin (its own GPU parity tests check the kernel)
    assert split["within1"] >= parity.FP8_ULP_FRACTION and split["sf_outside_band"] == 0
    assert split["max_abs"] <= 1e-5 and split["rel_l2"] <= 1e-5
    # one fp16 rounding per operand: the tolerances on the pre-cast values still hold,
    # the code-level bar does not
    assert single["max_abs"] <= parity.OUT_MAX_ABS and single["rel_l2"] <= 1e-2
    assert single["within1"] < parity.FP8_ULP_FRACTION or single["sf_outside_band"] > 0
    assert single["rel_l2"] > 20 * split["rel_l2"]
    # an FP8 q~ (the operand of an FP8 x FP8 QK^T) misses even the pre-cast bounds
    fp8q = _metrics(w, list(tokens), "fp8q")
    assert fp8q["rel_l2"] > 1e-2 and fp8q["within1"] < parity.FP8_ULP_FRACTION and fp8q["sf_outside_band"] > 0
