"""Pins of the nvfp4_ds_mla (V4.1 cache) oracle (CPU).

Each pin checks the oracle against something other than itself: the E2M1 format's value
table, rows built by hand, float64 SDPA from torch when the indices cover a small cache,
and special cases with a closed-form output."""

import numpy as np
import torch

from oracle import codecs
from oracle import nvfp4 as N
from oracle.sparse_mla import OracleParams, rope_interleaved
from top_sparse_mla_gb300 import workloads as W


def test_e2m1_value_table():
    # OCP MX FP4 (E2M1): codes 0..7 are 0, 0.5, 1, 1.5, 2, 3, 4, 6; bit 3 is the sign
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    got = N.e2m1_decode(np.arange(16))
    assert np.array_equal(got[:8], table)
    assert np.array_equal(got[8:], [-v for v in table])
    assert np.signbit(got[8])                      # code 8 is -0


def test_compressed_row_by_hand():
    row = np.zeros((1, 288), dtype=np.uint8)
    row[0, 0] = 0x21          # dim 0: code 1 (0.5, low nibble), dim 1: code 2 (1.0)
    row[0, 1] = 0xF7          # dim 2: code 7 (6.0), dim 3: code 15 (-6.0)
    row[0, 8] = 0x0B          # dim 16: code 11 (-1.5), dim 17: 0
    row[0, 255] = 0x60        # dim 510: 0, dim 511: code 6 (4.0)
    row[0, 256] = 0x38        # scale of dims 0..15: E4M3 0x38 = 1.0
    row[0, 257] = 0x40        # scale of dims 16..31: 2.0
    row[0, 287] = 0x30        # scale of dims 496..511: 0.5
    k = N.decode_cmp_rows(row, 0.75)[0]
    expect = np.zeros(512)
    expect[[0, 1, 2, 3]] = np.array([0.5, 1.0, 6.0, -6.0]) * 1.0 * 0.75
    expect[16] = -1.5 * 2.0 * 0.75
    expect[511] = 4.0 * 0.5 * 0.75
    assert np.array_equal(k, expect)


def test_window_row_by_hand():
    row = np.zeros((1, 528), dtype=np.uint8)
    row[0, 0] = 0x38           # E4M3 1.0
    row[0, 130] = 0xC0         # E4M3 -2.0 at dim 130 (second scale block)
    row[0, 511] = 0x01         # smallest subnormal 2^-9 at dim 511
    row[0, 512:528] = np.array([0.5, 3.0, 1.0, 1024.0], dtype="<f4").view(np.uint8)
    k = N.decode_swa_rows(row)[0]
    expect = np.zeros(512)
    expect[0], expect[130], expect[511] = 0.5, -6.0, 2.0 ** -9 * 1024.0
    assert np.array_equal(k, expect)


def test_generator_round_trip_is_close():
    # the generator's encoding decodes back to the drawn keys within the formats' steps
    rng = np.random.default_rng(3)
    x = rng.standard_normal((6, 512))
    k = N.decode_cmp_rows(W.encode_rows_nvfp4_cmp(x, 0.75), 0.75)
    grp = np.repeat(np.max(np.abs(x.reshape(6, 32, 16)), axis=2), 16, axis=1)
    assert np.all(np.abs(k - x) <= grp * (0.5 / 6 * 2 + 2 ** -3))       # half an E2M1 step + scale rounding
    k8 = N.decode_swa_rows(W.encode_rows_nvfp4_swa(x))
    assert np.all(np.abs(k8 - x) <= np.abs(x) * 2 ** -4 + 2 ** -9)


def _cover_all(seed=21, h=8, n_swa=24, n_cmp=40):
    w = W.random_case(seed, s_q=3, h_q=h, n_swa_cols=n_swa, n_cmp_cols=n_cmp, n_swa_rows=n_swa, n_cmp_rows=n_cmp,
                      kv_format=1, cmp_scale=0.75)
    for t in range(3):
        w.indices[t, :n_swa] = np.random.default_rng(t).permutation(n_swa)
        w.indices[t, n_swa:] = np.random.default_rng(100 + t).permutation(n_cmp)
    w.kv_swa = W.encode_rows_nvfp4_swa(np.random.default_rng(1).standard_normal((n_swa, 512)))
    w.kv_cmp = W.encode_rows_nvfp4_cmp(np.random.default_rng(3).standard_normal((n_cmp, 512)), 0.75)
    return w


def _run(w):
    p = OracleParams(n_swa_cols=w.n_swa_cols, softmax_scale=1 / np.sqrt(512))
    return N.sparse_mla_forward(w.q, w.kv_swa, w.kv_cmp, w.indices, w.topk_length, w.positions, w.norm_w, p,
                                cmp_scale=w.cmp_scale), p


def test_attention_equals_dense_sdpa_when_indices_cover_the_cache():
    w = _cover_all()
    r, p = _run(w)
    k_all = np.concatenate([N.decode_swa_rows(w.kv_swa), N.decode_cmp_rows(w.kv_cmp, 0.75)])
    for t in range(w.s_q):
        qt = torch.from_numpy(N.q_prologue(w.q[t], w.norm_w, int(w.positions[t]), p))
        k = torch.from_numpy(k_all)          # every row of both caches; order does not matter
        o = torch.nn.functional.scaled_dot_product_attention(qt[None], k[None], k[None], scale=p.softmax_scale)[0].numpy()
        o[:, 448:] = rope_interleaved(o[:, 448:], int(w.positions[t]), 1e4, inverse=True)
        assert np.max(np.abs(r["out"][t] - o)) < 1e-12


def test_q_prologue_rotates_dims_448_to_511_only():
    w = _cover_all()
    p = OracleParams(n_swa_cols=w.n_swa_cols)
    x = codecs.bf16_decode(w.q[0]).astype(np.float64)
    wt = codecs.bf16_decode(w.norm_w).astype(np.float64)
    qt = N.q_prologue(w.q[0], w.norm_w, int(w.positions[0]), p)
    xn = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + 1e-6) * wt        # 512-dim RMS
    assert np.allclose(qt[:, :448], xn[:, :448], rtol=0, atol=1e-12)
    # the rotation keeps each pair's length and moves dims 448..511 only
    a, b = qt[:, 448::2], qt[:, 449::2]
    assert np.allclose(a * a + b * b, xn[:, 448::2] ** 2 + xn[:, 449::2] ** 2, rtol=1e-12)


def test_single_valid_column_returns_its_row():
    w = W.random_case(41, s_q=2, h_q=4, n_swa_cols=8, n_cmp_cols=8, n_swa_rows=64, n_cmp_rows=64, kv_format=1,
                      cmp_scale=0.75)
    swa_row, cmp_row = int(w.indices[0, 3]), int(w.indices[1, 12])
    w.indices[:] = -1
    w.indices[0, 3] = swa_row
    w.indices[1, 12] = cmp_row
    r, _ = _run(w)
    for t, v in ((0, N.decode_swa_rows(w.kv_swa[swa_row:swa_row + 1])[0]),
                 (1, N.decode_cmp_rows(w.kv_cmp[cmp_row:cmp_row + 1], 0.75)[0])):
        v = np.concatenate([v[:448], rope_interleaved(v[448:], int(w.positions[t]), 1e4, inverse=True)])
        assert np.max(np.abs(r["out"][t] - v[None, :])) < 1e-12


def test_sentinel_rows_are_never_read():
    # every unreferenced row is NaN in the generated pools; the output stays finite
    w = W.make("tiny_nvfp4")
    r, _ = _run(w)
    assert np.all(np.isfinite(r["out"]))
