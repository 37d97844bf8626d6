"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI, run the
oracle on the same seeded inputs, compare.

Tolerances: the workload specification's matching rule for this path, as written:
  * pre-cast output (after inverse RoPE): max |err| <= 2e-2 and relative L2 <= 1e-2;
  * UE8M0 scale codes bit-exact, except blocks whose oracle amax lies within 1e-6
    relative of a power of two;
  * E4M3 codes within one step of the E4M3 lattice on at least 99.9 % of the elements
    of the blocks whose scale code matched;
  * LSE: |err| <= 2e-2 (the output's absolute bound; -inf exactly where no column is
    valid).
Where floating point decides an integer (the block exponent, the E4M3 code) the
decision is also re-taken by the oracle's cast on the kernel's own fp32 pre-cast
output, which must reproduce the kernel's codes bit for bit.
Every comparison is recorded in RECORDS (label, measured errors and fractions); the
test session prints them at its end, so a green run keeps the numbers.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
from oracle import codecs
from top_sparse_mla_gb300 import api, native
from top_sparse_mla_gb300.workloads import Workload

OUT_MAX_ABS = 2e-2
OUT_REL_L2 = 1e-2
LSE_ABS = 2e-2
FP8_ULP_FRACTION = 0.999   # E4M3 codes within one step, fraction of elements
SF_BAND_REL = 1e-6          # scale codes may differ only within this of a power of two
RECORDS: list = []


def run_gpu(w: Workload, flags: int = 0, debug: bool = True, device="cuda:0"):
    inp = api.upload(w, device, flags=flags)
    out = api.allocate_outputs(inp, debug=debug)
    api.forward(inp, out)
    torch.cuda.synchronize()
    res = {
        "out_fp8": out.out_fp8.cpu().numpy(),
        "out_sf": out.out_sf.cpu().numpy(),
        "status": native.dsa_sparse_attn_read_status(out.workspace),
    }
    if debug:
        res["out"] = out.out_precast.cpu().numpy().astype(np.float64)
        res["lse"] = out.lse.cpu().numpy().astype(np.float64)
    return res


def subset(w: Workload, tokens) -> Workload:
    tokens = np.asarray(tokens)
    return Workload(name=w.name + "_subset", q=w.q[tokens], norm_w=w.norm_w, kv_swa=w.kv_swa, kv_cmp=w.kv_cmp,
                    indices=w.indices[tokens], topk_length=w.topk_length[tokens], positions=w.positions[tokens],
                    n_swa_cols=w.n_swa_cols, seed=w.seed, kv_format=w.kv_format, cmp_scale=w.cmp_scale,
                    softmax_scale=w.softmax_scale, fp8_q=w.fp8_q)


def run_oracle(w: Workload):
    if w.kv_format == 1:   # nvfp4_ds_mla: the softmax scale as the kernel receives it (fp32)
        p = oracle.OracleParams(n_swa_cols=w.n_swa_cols, softmax_scale=float(np.float32(w.softmax_scale)))
        return oracle.nvfp4.sparse_mla_forward(w.q, w.kv_swa, w.kv_cmp, w.indices, w.topk_length, w.positions,
                                               w.norm_w, p, cmp_scale=w.cmp_scale)
    return oracle.sparse_mla_forward(w.q, w.kv_swa, w.kv_cmp, w.indices, w.topk_length, w.positions, w.norm_w,
                                     oracle.OracleParams(n_swa_cols=w.n_swa_cols, fp8_q=w.fp8_q))


def near_power_of_two(amax: np.ndarray, rel: float = SF_BAND_REL) -> np.ndarray:
    a = np.where(amax > 0, amax, 1.0)
    k = np.round(np.log2(a))
    return (amax > 0) & (np.abs(a / np.exp2(k) - 1.0) <= rel)


def compare(gpu: dict, ref: dict, tokens=None, label: str = "", out_scale: float = 1.0) -> dict:
    """Assert the matching rules; return (and record) the measured errors.

    out_scale: the factor by which the case scales the outputs relative to the
    specification's value distributions (a power of two for the range cases): the
    absolute pre-cast bound is stated for those distributions and scales with the data;
    the relative and code-level rules do not change."""
    g_out, g_lse = gpu["out"], gpu["lse"]
    g_fp8, g_sf = gpu["out_fp8"], gpu["out_sf"]
    if tokens is not None:
        g_out, g_lse, g_fp8, g_sf = g_out[tokens], g_lse[tokens], g_fp8[tokens], g_sf[tokens]
    r_out, r_lse = ref["out"], ref["lse"]
    assert np.all(np.isfinite(g_out)), f"{label}: non-finite pre-cast output"
    err = np.abs(g_out - r_out)
    max_abs = float(err.max()) if err.size else 0.0
    denom = float(np.linalg.norm(r_out))
    rel_l2 = float(np.linalg.norm(g_out - r_out) / denom) if denom > 0 else float(np.linalg.norm(g_out))
    # LSE
    inf_r, inf_g = np.isneginf(r_lse), np.isneginf(g_lse)
    lse_err = float(np.max(np.abs(g_lse[~inf_r] - r_lse[~inf_r]))) if (~inf_r).any() else 0.0
    # scales: bit-exact outside the power-of-two band
    amax = np.max(np.abs(r_out.reshape(r_out.shape[:-1] + (16, 32))), axis=-1)
    band = near_power_of_two(amax)
    sf_diff = g_sf != ref["out_sf"]
    sf_bad = int((sf_diff & ~band).sum())
    # codes: within one E4M3 step on >= 99.9 % of the elements of blocks whose scale matched
    same_blk = np.repeat((~sf_diff)[..., None], 32, axis=-1).reshape(g_fp8.shape)
    ulp = codecs.e4m3_ulp_distance(g_fp8, ref["out_fp8"])
    n = int(same_blk.sum())
    misses = int((ulp[same_blk] > 1).sum())
    frac = 1.0 - misses / n if n else 1.0
    exact = float((ulp[same_blk] == 0).mean()) if n else 1.0
    rec = {"label": label, "max_abs": max_abs, "rel_l2": rel_l2, "lse_abs": lse_err, "fp8_within_1": frac,
           "fp8_exact": exact, "fp8_misses": misses, "codes": n, "sf_mismatch_blocks": int(sf_diff.sum()),
           "sf_band_blocks": int(band.sum()), "blocks": int(g_sf.size)}
    RECORDS.append(rec)
    summary = (f"{label}: fp8 within 1 step {frac:.6f} ({misses} of {n} misses), exact {exact:.6f}, "
               f"scale mismatches {int(sf_diff.sum())} ({sf_bad} outside the 1e-6 band), "
               f"max abs {max_abs:.3e}, rel L2 {rel_l2:.3e}, LSE {lse_err:.3e}")
    assert max_abs <= OUT_MAX_ABS * out_scale, f"pre-cast max abs error too large; {summary}"
    assert rel_l2 <= OUT_REL_L2, f"pre-cast relative L2 error too large; {summary}"
    assert np.array_equal(inf_r, inf_g), f"-inf LSE pattern differs; {summary}"
    assert lse_err <= LSE_ABS, f"LSE error too large; {summary}"
    assert sf_bad == 0, f"UE8M0 codes differ outside the power-of-two band; {summary}"
    assert frac >= FP8_ULP_FRACTION, f"E4M3 codes more than one step away on too many elements; {summary}"
    # the kernel's own integer decisions, re-taken by the oracle cast on its fp32 output
    codes, sf = oracle.mxfp8_cast(g_out)
    assert np.array_equal(sf, g_sf), f"scale codes differ from the oracle cast of the kernel's pre-cast output; {summary}"
    assert np.array_equal(codes, g_fp8), f"E4M3 codes differ from the oracle cast of the kernel's output; {summary}"
    return rec
