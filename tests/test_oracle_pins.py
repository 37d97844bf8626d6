"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each test ties one oracle function to a library routine, a closed form, an invariant or
an independent restatement, chosen so that a plausible mistake (a dropped scale, a
swapped RoPE pair layout, a wrong sign, a transposed operand, a mis-rounded tie) fails
at least one of them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute, codecs
from oracle.sparse_mla import D_LATENT, OracleParams, decode_kv_rows, rope_interleaved, rmsnorm
from top_sparse_mla_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- formats
def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = codecs.e4m3_decode(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    fin = ~np.isnan(ref)
    assert np.array_equal(ref[fin], got[fin])
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF]) and got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_e4m3_encode_roundtrips_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(codecs.e4m3_encode(codecs.e4m3_decode(codes)), codes)


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.uniform(-448, 448, 20000),
        rng.standard_normal(20000) * 0.01,            # subnormal region
        rng.standard_normal(20000),
        np.ldexp(rng.integers(-64, 64, 5000) + 0.5, -9),  # exact subnormal ties
        np.ldexp(rng.integers(8, 16, 5000) + 0.5, rng.integers(-6, 6, 5000) - 3),  # exact normal ties
    ])
    x = np.clip(x, -448, 448)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = codecs.e4m3_encode(x.astype(np.float32).astype(np.float64))
    # torch keeps the sign of values that round to zero as well
    assert np.array_equal(got, ref)


def test_e4m3_encode_ties_saturation_nan():
    enc = lambda v: int(codecs.e4m3_encode(np.array([v]))[0])
    assert enc(1.0625) == 0x38          # tie between 1.0 (even) and 1.125 -> 1.0
    assert enc(1.1875) == 0x3A          # tie between 1.125 and 1.25 (even) -> 1.25
    assert enc(1.5 * 2 ** -9) == 0x02   # subnormal tie -> even (2 * 2^-9)
    assert enc(0.5 * 2 ** -9) == 0x00   # tie between 0 and 2^-9 -> 0
    assert enc(-0.5 * 2 ** -9) == 0x80
    assert enc(448.0) == 0x7E and enc(460.0) == 0x7E and enc(464.0) == 0x7E
    assert enc(1e6) == 0x7E and enc(-1e6) == 0xFE and enc(np.inf) == 0x7E
    assert enc(np.nan) == 0x7F
    assert enc(2.0 ** -6) == 0x08 and enc(240.0) == 0x77


def test_bf16_decode_matches_torch():
    bits = np.arange(0, 65536, 7, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = codecs.bf16_decode(bits)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    assert np.array_equal(ref[~np.isnan(ref)], got[~np.isnan(got)])


def test_ue8m0_shared_exponent_closed_forms():
    e = lambda a: int(codecs.mx_shared_exponent(np.array([a]))[0])
    assert e(1.0) == -8
    assert e(448.0) == 0
    assert e(0.75) == -9
    for k in range(-60, 60, 7):
        assert e(2.0 ** k) == k - 8
        assert e(2.0 ** k * (1 - 2 ** -40)) == k - 9
        assert e(2.0 ** k * (1 + 2 ** -40)) == k - 8
    assert e(0.0) == -127
    assert e(1e-300) == -127
    assert e(3e38) == 127 - 8
    assert np.array_equal(codecs.ue8m0_decode(np.array([0, 127, 254], dtype=np.uint8)), [2.0 ** -127, 1.0, 2.0 ** 127])


def test_mxfp8_block_invariants():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((500, 64)) * np.exp(rng.uniform(-20, 20, (500, 1)))
    codes, sf = codecs.mxfp8_quantize(x)
    e = sf.astype(np.int64) - 127
    xb = x.reshape(500, 2, 32)
    scaled = np.ldexp(np.abs(xb), -e[..., None])
    mx = scaled.max(axis=-1)
    assert np.all((mx >= 256) & (mx < 512))
    dec = codecs.e4m3_decode(codes).reshape(500, 2, 32) * np.ldexp(1.0, e)[..., None]
    sat = scaled >= 448
    err = np.abs(dec - xb)
    # unsaturated elements: within half a step of the E4M3 lattice at their magnitude
    lg = np.floor(np.log2(np.maximum(scaled, 1e-300))).astype(np.int64)
    step = np.ldexp(1.0, np.maximum(lg, -6) - 3 + e[..., None])
    assert np.all(err[~sat] <= 0.5 * step[~sat])
    top = np.broadcast_to(np.ldexp(448.0, e)[..., None], dec.shape)
    assert np.array_equal(np.abs(dec[sat]), top[sat])
    assert np.array_equal(np.sign(dec[sat]), np.sign(xb[sat]))


# ---------------------------------------------------------------- q prologue
def test_rope_inverse_is_identity_and_preserves_norm():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((16, 64))
    for pos in (0, 1, 77, 4095, 32767, 1 << 20):
        y = rope_interleaved(x, pos, 10000.0)
        assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=0, atol=1e-12)
        z = rope_interleaved(y, pos, 10000.0, inverse=True)
        assert np.max(np.abs(z - x)) < 1e-12


def test_rope_pair_layout_and_frequencies():
    # a unit vector on dim 2i stays inside the pair (2i, 2i+1); its angle after one
    # position step is theta_i = 10000^(-2i/64) = 10^(-i/8)
    for i in (0, 1, 5, 16, 31):
        x = np.zeros(64)
        x[2 * i] = 1.0
        y = rope_interleaved(x, 1, 10000.0)
        others = np.delete(y, [2 * i, 2 * i + 1])
        assert np.all(others == 0)
        ang = math.atan2(y[2 * i + 1], y[2 * i])
        assert abs(ang - 10.0 ** (-i / 8.0)) < 1e-12
    # composition: rotating by a then b equals rotating by a + b
    x = np.random.default_rng(2).standard_normal(64)
    assert np.max(np.abs(rope_interleaved(rope_interleaved(x, 300, 1e4), 25, 1e4) - rope_interleaved(x, 325, 1e4))) < 1e-11


def test_rmsnorm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((8, 576)) * 3.7
    y = rmsnorm(x, np.ones(576), 0.0)
    assert np.allclose(np.mean(y * y, axis=-1), 1.0, atol=1e-13)
    assert np.max(np.abs(rmsnorm(5.0 * x, np.ones(576), 0.0) - y)) < 1e-13
    w = rng.standard_normal(576)
    assert np.max(np.abs(rmsnorm(x, w, 0.0) - y * w)) < 1e-13


def test_q_prologue_only_rotates_rope_dims():
    w = W.make("tiny")
    p = OracleParams(n_swa_cols=w.n_swa_cols)
    a = oracle.q_prologue(w.q[0], w.norm_w, 0, p)
    b = oracle.q_prologue(w.q[0], w.norm_w, 1234, p)
    assert np.array_equal(a[:, :D_LATENT], b[:, :D_LATENT])
    assert not np.allclose(a[:, D_LATENT:], b[:, D_LATENT:])


# ---------------------------------------------------------------- cache rows
def test_decode_kv_rows_against_source_values():
    rng = np.random.default_rng(5)
    lat = rng.standard_normal((10, 512)).astype(np.float32) * 3
    rope = rng.standard_normal((10, 64)).astype(np.float32)
    rows = W.encode_rows(lat, rope)
    k = decode_kv_rows(rows)
    # latent: E4M3 with a per-128 scale -> relative error <= 2^-4 of the block max
    blk = np.abs(lat).reshape(10, 4, 128).max(-1)
    tol = np.repeat(blk, 128, axis=1) / 448 * 2 ** -9 * 448 / 2 ** -3   # half an E4M3 step at the block top, generous
    assert np.all(np.abs(k[:, :512] - lat) <= np.maximum(np.abs(lat) * 2 ** -4, tol))
    # rope: bf16 rounding
    assert np.all(np.abs(k[:, 512:] - rope) <= np.abs(rope) * 2 ** -8)


# ---------------------------------------------------------------- attention core
def _cover_all_case(seed=11, h=8, n_swa=24, n_cmp=40):
    w = W.random_case(seed, s_q=3, h_q=h, n_swa_cols=n_swa, n_cmp_cols=n_cmp, n_swa_rows=n_swa, n_cmp_rows=n_cmp)
    for t in range(3):  # every row of both (small) caches, in a seeded order
        w.indices[t, :n_swa] = np.random.default_rng(t).permutation(n_swa)
        w.indices[t, n_swa:] = np.random.default_rng(100 + t).permutation(n_cmp)
    w.kv_swa = W.encode_rows(np.random.default_rng(1).standard_normal((n_swa, 512)), np.random.default_rng(2).standard_normal((n_swa, 64)))
    w.kv_cmp = W.encode_rows(np.random.default_rng(3).standard_normal((n_cmp, 512)), np.random.default_rng(4).standard_normal((n_cmp, 64)))
    return w


def _run(w, **kw):
    p = OracleParams(n_swa_cols=w.n_swa_cols, **kw)
    return oracle.sparse_mla_forward(w.q, w.kv_swa, w.kv_cmp, w.indices, w.topk_length, w.positions, w.norm_w, p)


def test_attention_equals_dense_sdpa_when_indices_cover_the_cache():
    w = _cover_all_case()
    r = _run(w)
    p = OracleParams(n_swa_cols=w.n_swa_cols)
    for t in range(w.s_q):
        qt = torch.from_numpy(oracle.q_prologue(w.q[t], w.norm_w, int(w.positions[t]), p))
        rows = np.concatenate([w.kv_swa[w.indices[t, :w.n_swa_cols]], w.kv_cmp[w.indices[t, w.n_swa_cols:]]])
        k = torch.from_numpy(decode_kv_rows(rows))
        o = torch.nn.functional.scaled_dot_product_attention(qt[None], k[None], k[None, :, :512], scale=p.softmax_scale)[0].numpy()
        o[:, 448:] = rope_interleaved(o[:, 448:], int(w.positions[t]), 10000.0, inverse=True)
        assert np.max(np.abs(o - r["out"][t])) < 1e-12
        lse = torch.logsumexp(p.softmax_scale * qt @ k.T, dim=-1).numpy()
        assert np.max(np.abs(lse - r["lse"][t])) < 1e-12


def test_permuting_valid_columns_changes_nothing():
    w = W.random_case(21, s_q=4, h_q=8, n_swa_cols=16, n_cmp_cols=48, n_swa_rows=200, n_cmp_rows=300, n_sentinels=9)
    base = _run(w)
    rng = np.random.default_rng(0)
    for t in range(w.s_q):   # permute inside each pool's column range (the range decides the pool)
        w.indices[t, :16] = w.indices[t, rng.permutation(16)]
        w.indices[t, 16:] = w.indices[t, 16 + rng.permutation(48)]
    again = _run(w)
    assert np.max(np.abs(base["out"] - again["out"])) < 1e-12
    assert np.max(np.abs(base["lse"] - again["lse"])) < 1e-12


def test_sentinels_stale_rows_and_out_of_length_columns_are_never_read():
    w = W.random_case(31, s_q=5, h_q=4, n_swa_cols=16, n_cmp_cols=32, n_swa_rows=128, n_cmp_rows=256, n_sentinels=7, lengths="ragged")
    base = _run(w)
    rng = np.random.default_rng(9)
    # rows referenced by a live column
    cols = np.arange(w.topk)[None, :]
    live = (cols < w.topk_length[:, None]) & (w.indices >= 0)
    used_swa = np.unique(w.indices[:, :16][live[:, :16]])
    used_cmp = np.unique(w.indices[:, 16:][live[:, 16:]])
    for fill in ("random", "nan"):
        w2 = W.random_case(31, s_q=5, h_q=4, n_swa_cols=16, n_cmp_cols=32, n_swa_rows=128, n_cmp_rows=256, n_sentinels=7, lengths="ragged")
        for pool, used in ((w2.kv_swa, used_swa), (w2.kv_cmp, used_cmp)):
            stale = np.setdiff1d(np.arange(pool.shape[0]), used)
            if fill == "random":
                pool[stale] = rng.integers(0, 256, size=(len(stale), 656), dtype=np.uint8)
            else:
                pool[stale] = W._nan_rows(len(stale))
        # beyond-length columns point at arbitrary rows
        for t in range(w2.s_q):
            L = int(w2.topk_length[t])
            w2.indices[t, L:] = rng.integers(0, 128, size=w2.topk - L)
        again = _run(w2)
        assert np.array_equal(base["out"], again["out"])
        assert np.array_equal(base["out_fp8"], again["out_fp8"]) and np.array_equal(base["out_sf"], again["out_sf"])


def test_single_valid_column_returns_that_row():
    w = W.random_case(41, s_q=2, h_q=4, n_swa_cols=8, n_cmp_cols=8, n_swa_rows=64, n_cmp_rows=64)
    swa_row, cmp_row = int(w.indices[0, 3]), int(w.indices[1, 12])   # rows the generator filled
    w.indices[:] = -1
    w.indices[0, 3] = swa_row
    w.indices[1, 12] = cmp_row
    r = _run(w)
    for t, (pool, row) in enumerate(((w.kv_swa, swa_row), (w.kv_cmp, cmp_row))):
        v = decode_kv_rows(pool[row:row + 1])[0, :512]
        v = np.concatenate([v[:448], rope_interleaved(v[448:], int(w.positions[t]), 1e4, inverse=True)])
        assert np.max(np.abs(r["out"][t] - v[None, :])) < 1e-12


def test_empty_rows_give_zero_output_and_minus_inf_lse():
    w = W.random_case(51, s_q=3, h_q=4, n_swa_cols=8, n_cmp_cols=8, n_swa_rows=64, n_cmp_rows=64)
    w.indices[0] = -1               # every column a sentinel
    w.topk_length[1] = 0            # nothing in length
    w.topk_length[2] = -3           # negative length reads nothing
    r = _run(w)
    assert np.all(r["out"] == 0) and np.all(np.isneginf(r["lse"]))
    assert np.all(r["out_sf"] == 0) and np.all(r["out_fp8"] == 0)


def test_duplicate_columns_count_separately():
    w = _cover_all_case(seed=61, h=4, n_swa=8, n_cmp=8)
    w.indices[0, 9] = w.indices[0, 8]      # column 9 repeats column 8's compressed row
    r = _run(w)
    p = OracleParams(n_swa_cols=8)
    qt = torch.from_numpy(oracle.q_prologue(w.q[0], w.norm_w, int(w.positions[0]), p))
    rows = np.concatenate([w.kv_swa[w.indices[0, :8]], w.kv_cmp[w.indices[0, 8:]]])
    k = torch.from_numpy(decode_kv_rows(rows))       # the repeated row appears twice
    o = torch.nn.functional.scaled_dot_product_attention(qt[None], k[None], k[None, :, :512], scale=p.softmax_scale)[0].numpy()
    o[:, 448:] = rope_interleaved(o[:, 448:], int(w.positions[0]), 1e4, inverse=True)
    assert np.max(np.abs(o - r["out"][0])) < 1e-12


def test_brute_force_agrees_on_tiny_workload():
    w = W.make("tiny")
    r = _run(w)
    bo, bl = brute.forward(w.q.tolist(), w.kv_swa, w.kv_cmp, w.indices.tolist(), w.topk_length.tolist(),
                           w.positions.tolist(), w.norm_w.tolist(), w.n_swa_cols)
    assert np.max(np.abs(np.array(bo) - r["out"])) < 1e-12
    assert np.max(np.abs(np.array(bl) - r["lse"])) < 1e-12


def test_handworked_golden_example():
    fx = json.load(open(os.path.join(GOLDEN, "handworked_two_rows.json")))
    one = 0x3F80
    q = np.empty((1, 2, 576), dtype=np.uint16)
    q[0, 0] = one
    q[0, 1] = np.where(np.arange(576) % 2 == 0, one, 0xBF80)
    norm_w = np.full(576, one, dtype=np.uint16)
    zero_rope = np.zeros((1, 64), dtype=np.float32)
    def row(code):
        r = np.zeros((1, 656), dtype=np.uint8)
        r[0, :512] = code
        r[0, 512:528] = np.frombuffer(np.ones(4, dtype="<f4").tobytes(), dtype=np.uint8)
        return r
    kv_swa, kv_cmp = row(0x38), row(0x30)
    res = oracle.sparse_mla_forward(q, kv_swa, kv_cmp, np.array([[0, 0]], dtype=np.int32), np.array([2], dtype=np.int32),
                                    np.array([0], dtype=np.int32), norm_w, OracleParams(n_swa_cols=1))
    ex = fx["expected"]
    assert np.max(np.abs(res["out"][0, 0] - ex["out_head0_every_dim"])) < 1e-14
    assert np.max(np.abs(res["out"][0, 1] - ex["out_head1_every_dim"])) < 1e-14
    assert abs(res["lse"][0, 0] - ex["lse_head0"]) < 1e-12 and abs(res["lse"][0, 1] - ex["lse_head1"]) < 1e-14
    assert np.array_equal(res["out_sf"][0], np.array(ex["out_sf"], dtype=np.uint8))
    assert np.all(res["out_fp8"][0, 0] == ex["out_fp8_head0_every_dim"])
    assert np.all(res["out_fp8"][0, 1] == ex["out_fp8_head1_every_dim"])


def test_index_out_of_range_is_an_error():
    w = W.random_case(71, s_q=1, h_q=2, n_swa_cols=4, n_cmp_cols=4, n_swa_rows=16, n_cmp_rows=16)
    w.indices[0, 5] = 16
    with pytest.raises(IndexError):
        _run(w)


def test_bf16_encode_matches_torch_rounding():
    # round to nearest even on the binary32 value, as torch's float32 -> bfloat16 cast
    import torch
    from oracle import codecs as C
    rng = np.random.default_rng(31)
    x = (rng.standard_normal(50000) * np.exp2(rng.integers(-60, 60, 50000))).astype(np.float32).astype(np.float64)
    x = np.concatenate([x, [0.0, -0.0, np.inf, -np.inf, 3.3895313892515355e38, 3.4e38, 1e-40, -1e-45, 1.00390625,
                            1.01171875, -1.00390625]])
    ref = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    assert np.array_equal(C.bf16_encode(x), ref)
    assert C.bf16_encode(np.array([np.nan]))[0] == 0x7FC0
    # ties: 1 + 2^-8 is halfway between 1 and 1 + 2^-7 and goes to the even 1
    assert C.bf16_encode(np.array([1.00390625]))[0] == 0x3F80


def test_sf_swizzle_128x4_hand_worked_offsets():
    # A 130 x 8 scale matrix: two tile rows (the second one padded) of two 128 x 4 tiles.
    # Offsets worked by hand from the layout's description: tiles of 512 bytes in
    # row-major tile order; inside a tile, row r and column c at (r % 32) * 16 +
    # (r // 32) * 4 + c.
    from oracle import codecs as C
    M, K = 130, 8
    sf = np.zeros((M, K), dtype=np.uint8)
    marks = {  # (m, k): expected byte offset
        (0, 0): 0, (0, 3): 3, (0, 4): 512, (1, 0): 16, (31, 0): 496, (32, 0): 4, (33, 1): 16 + 4 + 1,
        (64, 2): 8 + 2, (96, 0): 12, (127, 3): 496 + 12 + 3, (127, 7): 512 + 511, (128, 0): 1024,
        (129, 7): 1536 + 16 + 3,
    }
    for i, (m, k) in enumerate(marks):
        sf[m, k] = 10 + i
    out = C.sf_swizzle_128x4(sf)
    assert out.shape == (256 * K,)          # rows padded to a multiple of 128
    for i, ((m, k), off) in enumerate(marks.items()):
        assert out[off] == 10 + i, (m, k, off)
    assert int(np.count_nonzero(out)) == len(marks)


def test_sf_swizzle_128x4_is_a_permutation():
    # with M a multiple of 128 every byte is written exactly once
    from oracle import codecs as C
    rng = np.random.default_rng(5)
    for M, K in ((128, 4), (256, 16), (384, 64)):
        sf = rng.integers(0, 256, size=(M, K)).astype(np.uint8)
        out = C.sf_swizzle_128x4(sf)
        assert out.size == sf.size
        assert np.array_equal(np.sort(out), np.sort(sf.ravel()))
        # each 512-byte tile holds exactly the codes of its 128 x 4 block
        for mt in range(M // 128):
            for kt in range(K // 4):
                tile = out[(mt * (K // 4) + kt) * 512:(mt * (K // 4) + kt + 1) * 512]
                block = sf[128 * mt:128 * (mt + 1), 4 * kt:4 * (kt + 1)]
                assert np.array_equal(np.sort(tile), np.sort(block.ravel()))
