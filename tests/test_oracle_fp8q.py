"""Pins of the oracle's E4M3-q reading (OracleParams.fp8_q, quantize_q_latent) on the CPU.

Hand-worked codes, a case where the quantisation is lossless (the oracle must then equal
the unquantised one), invariance under scaling q by powers of two (the RMS factor
cancels), and the E4M3 error bound."""

import numpy as np

import oracle
from oracle import codecs
from oracle.sparse_mla import OracleParams, quantize_q_latent
from top_sparse_mla_gb300 import workloads as W


def _bits(x):
    return W._bf16_bits(np.asarray(x, dtype=np.float32))


def test_hand_worked_codes():
    x = np.zeros((1, 576), dtype=np.float32)
    x[0, :5] = [3.5, 1.0, -0.5, 0.109375, 2.0]     # amax 3.5 -> factor 448 / 3.5 = 128 exactly
    x[0, 530] = 100.0                                # a rope dim: not part of the latent amax
    w = np.ones(576, dtype=np.float32)
    codes, amax = quantize_q_latent(_bits(x), _bits(w))
    assert amax[0] == np.float32(3.5)
    # 3.5 * 128 = 448 (0x7E); 1 * 128 = 128 (0x70); -0.5 * 128 = -64 (0xE8);
    # 0.109375 * 128 = 14 (0x56: 1.75 * 2^3); 2 * 128 = 256 (0x78)
    assert list(codes[0, :5]) == [0x7E, 0x70, 0xE8, 0x56, 0x78]
    assert np.all(codes[0, 5:] == 0)


def test_rounding_in_binary32_ties_to_even():
    # amax 3.0 -> factor fl(448 / 3) = 149.33333...; 1.0 -> 149.333 rounds to 144 (E4M3
    # steps of 16 above 128: 144 and 160), 0.75 -> 112 exactly (0x6C)
    x = np.zeros((1, 576), dtype=np.float32)
    x[0, :3] = [3.0, 1.0, 0.75]
    codes, _ = quantize_q_latent(_bits(x), _bits(np.ones(576, dtype=np.float32)))
    assert codecs.e4m3_decode(codes[0, :3]).tolist() == [448.0, 144.0, 112.0]


def test_the_factor_is_rounded_to_binary32_first():
    # amax 1.625 = 13/8: the exact factor 448 / 1.625 = 3584/13 = 275.6923076..., whose
    # binary32 value is 9034022 * 2^-15 = 275.69232177734375 (above it).  For
    # x = 39/512 the exact product is 21, a tie between the E4M3 values 20 and 22 that
    # goes to the even 20 (0x5A); with the binary32 factor the product is 21 + 2^-19
    # (one binary32 step above 21), which rounds to 22 (0x5B).  The reading decides in
    # binary32, so the code is 0x5B.
    x = np.zeros((1, 576), dtype=np.float32)
    x[0, :2] = [1.625, 39.0 / 512.0]
    codes, _ = quantize_q_latent(_bits(x), _bits(np.ones(576, dtype=np.float32)))
    assert codes[0, 0] == 0x7E and codes[0, 1] == 0x5B


def _case(seed, lossless=False):
    w = W.random_case(seed, s_q=3, h_q=8, n_swa_cols=24, n_cmp_cols=40, n_swa_rows=300, n_cmp_rows=500,
                      n_sentinels=4)
    if lossless:
        # every |q * w| equal to amax * 2^-j: each value times 448 / amax is an E4M3 value
        rng = np.random.default_rng(seed)
        mag = np.exp2(-rng.integers(0, 6, size=w.q.shape)).astype(np.float32) * 1.5
        sign = np.where(rng.random(w.q.shape) < 0.5, -1.0, 1.0).astype(np.float32)
        w.q = _bits(mag * sign)
        w.norm_w = _bits(np.ones(576, dtype=np.float32))
    return w


def _run(w, fp8_q, eps=1e-6):
    p = OracleParams(n_swa_cols=w.n_swa_cols, fp8_q=fp8_q, rms_eps=eps)
    return oracle.sparse_mla_forward(w.q, w.kv_swa, w.kv_cmp, w.indices, w.topk_length, w.positions, w.norm_w, p)


def test_lossless_case_equals_the_unquantised_oracle():
    w = _case(5, lossless=True)
    a, b = _run(w, True), _run(w, False)
    assert np.max(np.abs(a["out"] - b["out"])) < 1e-12
    assert np.max(np.abs(a["lse"] - b["lse"])) < 1e-12


def test_codes_and_output_invariant_under_powers_of_two_of_q():
    # (eps 0, so that the RMSNorm itself is scale-invariant too)
    w = _case(6)
    base = _run(w, True, eps=0.0)
    c0, _ = quantize_q_latent(w.q, w.norm_w)
    for s in (-6, 3):
        w2 = _case(6)
        w2.q = _bits(codecs.bf16_decode(w.q).astype(np.float32) * np.float32(2.0 ** s))
        c1, _ = quantize_q_latent(w2.q, w2.norm_w)
        assert np.array_equal(c0, c1)
        assert np.max(np.abs(_run(w2, True, eps=0.0)["out"] - base["out"])) < 1e-12


def test_quantised_latent_within_half_a_step():
    w = _case(7)
    p1, p0 = OracleParams(n_swa_cols=w.n_swa_cols, fp8_q=True), OracleParams(n_swa_cols=w.n_swa_cols)
    for t in range(w.s_q):
        a = oracle.q_prologue(w.q[t], w.norm_w, int(w.positions[t]), p1)
        b = oracle.q_prologue(w.q[t], w.norm_w, int(w.positions[t]), p0)
        amax = np.max(np.abs(b[:, :512]), axis=1, keepdims=True)
        assert np.all(np.abs(a[:, :512] - b[:, :512]) <= np.maximum(np.abs(b[:, :512]) * 2 ** -4, amax / 448 * 2 ** -9))
        assert np.array_equal(a[:, 512:], b[:, 512:])        # the rope part is not quantised
