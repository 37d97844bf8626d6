"""Parity of the CUDA path (through the C ABI) with the float64 oracle on GB300."""

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


def _full(w, out_scale=1.0, **kw):
    g = parity.run_gpu(w, **kw)
    # a bounded wait that ran out (or an index the kernel rejected) is reported as such,
    # before any value comparison
    assert g["status"] == 0 or kw.get("flags", 0), f"{w.name}: kernel status {g['status']:#x}"
    r = parity.run_oracle(w)
    return g, r, parity.compare(g, r, label=w.name, out_scale=out_scale)


def test_tiny_workload_all_elements():
    w = W.make("tiny")
    g, r, e = _full(w)
    assert g["status"] == 0
    print("tiny", e)


def test_single_token_decode_split_path():
    w = W.make("decode1")
    p = native.dsa_params_init(w.s_q, w.h_q, w.topk, w.n_swa_cols, w.kv_swa.shape[0], w.kv_cmp.shape[0])
    assert native.dsa_sparse_attn_num_splits(p) > 1          # exercises the split combine
    g, r, e = _full(w)
    print("decode1", e)


def test_batched_decode_64():
    w = W.make("decode64")
    g, r, e = _full(w)
    print("decode64", e)


@pytest.mark.parametrize("name", ["decode1024", "prefill2123"])
def test_full_size_workloads_sampled_tokens(name):
    w = W.make(name)
    g = parity.run_gpu(w)
    assert g["status"] == 0, f"{name}: kernel status {g['status']:#x}"
    rng = np.random.default_rng(123)
    tok = np.unique(np.concatenate([[0, 1, 2, w.s_q - 1], rng.choice(w.s_q, size=40, replace=False)]))
    r = parity.run_oracle(parity.subset(w, tok))
    e = parity.compare(g, r, tokens=tok, label=name)
    assert np.all(np.isfinite(g["out"])) and g["status"] == 0
    print(name, e)


@pytest.mark.parametrize("h_q", [1, 16, 40, 64])
def test_head_counts(h_q):
    w = W.random_case(200 + h_q, s_q=3, h_q=h_q, n_swa_cols=64, n_cmp_cols=200, n_swa_rows=300, n_cmp_rows=900,
                      n_sentinels=11)
    _full(w)


def test_many_tiles_ragged_tail_and_long_rows():
    # 2048 columns -> up to 16 tiles per token, ragged lengths, split combine with many splits
    w = W.random_case(301, s_q=2, h_q=64, n_swa_cols=512, n_cmp_cols=1536, n_swa_rows=4096, n_cmp_rows=8192,
                      n_sentinels=100, lengths="ragged")
    _full(w)


def test_more_tokens_than_sms_no_split():
    w = W.random_case(302, s_q=300, h_q=64, n_swa_cols=128, n_cmp_cols=173, n_swa_rows=2000, n_cmp_rows=5000,
                      n_sentinels=3, lengths="ragged")
    _full(w)


def test_empty_rows_and_degenerate_lengths():
    w = W.random_case(303, s_q=6, h_q=64, n_swa_cols=128, n_cmp_cols=512, n_swa_rows=1024, n_cmp_rows=4096)
    w.indices[0] = -1                 # all sentinels
    w.topk_length[1] = 0              # nothing in length
    w.topk_length[2] = -5             # negative length
    w.topk_length[3] = 1              # exactly one column
    w.topk_length[4] = 100000         # beyond topk: capped
    w.indices[5, 1:] = -1             # one valid column
    g, r, e = _full(w)
    assert np.all(g["out"][[0, 1, 2]] == 0) and np.all(g["out_sf"][[0, 1, 2]] == 0)
    assert np.all(g["out_fp8"][[0, 1, 2]] == 0) and np.all(np.isneginf(g["lse"][[0, 1, 2]]))


def test_duplicate_indices_and_last_pool_row():
    w = W.random_case(304, s_q=4, h_q=64, n_swa_cols=32, n_cmp_cols=96, n_swa_rows=64, n_cmp_rows=128)
    w.indices[0, 40] = w.indices[0, 41]           # duplicate column
    w.indices[1, 0] = 63                          # last SWA row
    w.indices[1, 50] = 127                        # last compressed row
    # make sure those rows hold data
    w.kv_swa[63] = W.encode_rows(np.ones((1, 512), np.float32), np.zeros((1, 64), np.float32))[0]
    w.kv_cmp[127] = W.encode_rows(np.full((1, 512), -0.5, np.float32), np.ones((1, 64), np.float32))[0]
    _full(w)


def test_index_check_flag_skips_out_of_range_and_reports():
    w = W.random_case(305, s_q=2, h_q=16, n_swa_cols=16, n_cmp_cols=48, n_swa_rows=64, n_cmp_rows=128)
    bad = w.indices.copy()
    bad[0, 3] = 64          # == pool size: out of range
    bad[1, 20] = 10 ** 6
    wb = W.Workload(name="oob", q=w.q, norm_w=w.norm_w, kv_swa=w.kv_swa, kv_cmp=w.kv_cmp, indices=bad,
                    topk_length=w.topk_length, positions=w.positions, n_swa_cols=w.n_swa_cols, seed=0)
    g = parity.run_gpu(wb, flags=native.DSA_FLAG_CHECK_INDICES)
    assert g["status"] & native.DSA_STATUS_INDEX_OUT_OF_RANGE
    ref_idx = bad.copy()
    ref_idx[0, 3] = -1
    ref_idx[1, 20] = -1
    wr = W.Workload(name="oob_ref", q=w.q, norm_w=w.norm_w, kv_swa=w.kv_swa, kv_cmp=w.kv_cmp, indices=ref_idx,
                    topk_length=w.topk_length, positions=w.positions, n_swa_cols=w.n_swa_cols, seed=0)
    parity.compare(g, parity.run_oracle(wr), label="oob")
    # a clean call on the same workspace clears the status
    g2 = parity.run_gpu(wr, flags=native.DSA_FLAG_CHECK_INDICES)
    assert g2["status"] == 0


def test_deterministic_and_production_entry_matches_debug_entry():
    w = W.make("decode64")
    a = parity.run_gpu(w, debug=True)
    b = parity.run_gpu(w, debug=False)
    c = parity.run_gpu(w, debug=True)
    assert np.array_equal(a["out_fp8"], b["out_fp8"]) and np.array_equal(a["out_sf"], b["out_sf"])
    assert np.array_equal(a["out"], c["out"])


def _scale_bf16(bits: np.ndarray, k: int) -> np.ndarray:
    """bf16 bit patterns times 2^k (exact: the exponent field moves; zeros stay zero)."""
    b = bits.astype(np.int32)
    nz = (b & 0x7F80) != 0
    return np.where(nz, b + (k << 7), b).astype(np.uint16)


def _scale_latent(kv: np.ndarray, k: int) -> np.ndarray:
    """fp8_ds_mla rows whose latent values are all times 2^k: the E4M3 codes stay, the four
    fp32 block scales move (every 128-block amax moves with them)."""
    out = kv.copy()
    sc = np.ascontiguousarray(out[:, 512:528]).view("<f4").astype(np.float64)
    out[:, 512:528] = np.ldexp(sc, k).astype("<f4").view(np.uint8)
    return out


@pytest.mark.parametrize("what,k", [("q", -12), ("q", 10), ("w", 4), ("latent", -8), ("latent", 8)])
def test_input_range_scalings(what, k):
    # The fp16 operands carry q * w with a per-head power-of-two prescale, and the cache's
    # fp32 block scales stay in fp32: scaling q, the norm weight or a row's latent values
    # by a power of two keeps the matching rule.
    w = W.random_case(310 + k + 50 * len(what), s_q=5, h_q=64, n_swa_cols=128, n_cmp_cols=512, n_swa_rows=1024,
                      n_cmp_rows=4096, n_sentinels=7, lengths="ragged")
    if what == "q":
        w.q = _scale_bf16(w.q, k)
    elif what == "w":
        w.norm_w = _scale_bf16(w.norm_w, k)
    else:
        w.kv_swa = _scale_latent(w.kv_swa, k)
        w.kv_cmp = _scale_latent(w.kv_cmp, k)
    w.name = f"range {what} x2^{k}"
    # o is a weighted mean of the latent rows: it scales with them (q and w only sharpen
    # or flatten the softmax)
    _full(w, out_scale=2.0 ** k if what == "latent" and k > 0 else 1.0)
