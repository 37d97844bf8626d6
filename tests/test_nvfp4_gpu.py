"""Parity of the CUDA path on the nvfp4_ds_mla (V4.1) cache with the float64 oracle
(oracle.nvfp4) on GB300: 528-byte fp8 window rows, 288-byte fp4 compressed rows,
512-dim keys with the rotary dims inside."""

import numpy as np
import pytest

from top_sparse_mla_gb300 import native
from top_sparse_mla_gb300 import workloads as W

import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from top_sparse_mla_gb300.build import build
    build()
    native.library()


def _full(w, **kw):
    g = parity.run_gpu(w, **kw)
    assert g["status"] == 0 or kw.get("flags", 0), f"{w.name}: kernel status {g['status']:#x}"
    r = parity.run_oracle(w)
    return g, r, parity.compare(g, r, label=w.name)


@pytest.mark.parametrize("name", ["tiny_nvfp4", "decode1_nvfp4", "decode64_nvfp4"])
def test_named_workloads_all_elements(name):
    w = W.make(name)
    g, r, e = _full(w)
    print(name, e)


def test_split_path_is_taken_for_a_single_token():
    w = W.make("decode1_nvfp4")
    p = native.dsa_params_init(w.s_q, w.h_q, w.topk, w.n_swa_cols, w.kv_swa.shape[0], w.kv_cmp.shape[0])
    assert native.dsa_sparse_attn_num_splits(p) > 1


def test_decode1024_sampled_tokens():
    w = W.make("decode1024_nvfp4")
    g = parity.run_gpu(w)
    assert g["status"] == 0
    rng = np.random.default_rng(7)
    tok = np.unique(np.concatenate([[0, 1, w.s_q - 1], rng.choice(w.s_q, size=40, replace=False)]))
    r = parity.run_oracle(parity.subset(w, tok))
    e = parity.compare(g, r, tokens=tok, label="decode1024_nvfp4")
    print(e)


@pytest.mark.parametrize("h_q", [16, 40, 64])
def test_random_cases_ragged_with_sentinels_and_empty_rows(h_q):
    w = W.random_case(500 + h_q, s_q=37, h_q=h_q, n_swa_cols=64, n_cmp_cols=300, n_swa_rows=700, n_cmp_rows=2000,
                      n_sentinels=9, lengths="ragged", kv_format=1, cmp_scale=0.3)
    w.topk_length[[0, 17]] = 0
    w.indices[5] = -1
    _full(w)


def test_compressed_scale_and_only_one_pool():
    # all columns compressed (n_swa_cols 0), a large pool scale; then all window columns
    w = W.random_case(601, s_q=9, h_q=64, n_swa_cols=0, n_cmp_cols=400, n_swa_rows=1, n_cmp_rows=3000,
                      n_sentinels=5, kv_format=1, cmp_scale=37.5)
    _full(w)
    w = W.random_case(602, s_q=9, h_q=64, n_swa_cols=300, n_cmp_cols=0, n_swa_rows=3000, n_cmp_rows=1,
                      n_sentinels=5, kv_format=1)
    _full(w)


def test_index_bounds_check_on_both_pools():
    w = W.random_case(603, s_q=4, h_q=32, n_swa_cols=16, n_cmp_cols=48, n_swa_rows=100, n_cmp_rows=200,
                      kv_format=1, cmp_scale=0.75)
    bad = w.indices.copy()
    bad[1, 3] = 100          # one past the window pool
    bad[2, 40] = 200         # one past the compressed pool
    wb = W.Workload(name="oob_nvfp4", q=w.q, norm_w=w.norm_w, kv_swa=w.kv_swa, kv_cmp=w.kv_cmp, indices=bad,
                    topk_length=w.topk_length, positions=w.positions, n_swa_cols=w.n_swa_cols, seed=w.seed,
                    kv_format=1, cmp_scale=0.75, softmax_scale=w.softmax_scale)
    g = parity.run_gpu(wb, flags=native.DSA_FLAG_CHECK_INDICES)
    assert g["status"] == native.DSA_STATUS_INDEX_OUT_OF_RANGE
    ref = bad.copy()
    ref[1, 3] = -1
    ref[2, 40] = -1
    wr = W.Workload(name="oob_nvfp4_ref", q=w.q, norm_w=w.norm_w, kv_swa=w.kv_swa, kv_cmp=w.kv_cmp, indices=ref,
                    topk_length=w.topk_length, positions=w.positions, n_swa_cols=w.n_swa_cols, seed=w.seed,
                    kv_format=1, cmp_scale=0.75, softmax_scale=w.softmax_scale)
    parity.compare(g, parity.run_oracle(wr), label="oob_nvfp4")


def test_swizzled_scales_with_the_nvfp4_cache():
    from oracle.codecs import sf_swizzle_128x4
    w = W.make("decode64_nvfp4")
    plain = parity.run_gpu(w)
    swz = parity.run_gpu(w, flags=native.DSA_FLAG_SF_SWIZZLED)
    assert np.array_equal(plain["out_fp8"], swz["out_fp8"])
    written = sf_swizzle_128x4(np.ones((w.s_q, 16 * w.h_q), dtype=np.uint8)) == 1
    expect = sf_swizzle_128x4(plain["out_sf"].reshape(w.s_q, 16 * w.h_q))
    assert np.array_equal(swz["out_sf"][written], expect[written])
