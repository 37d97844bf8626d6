"""The failure path on GB300, without a GPU fault: an on-chip wait that runs out.

DSA_FLAG_TEST_WAIT_TIMEOUT makes CTA 0 wait on a barrier that nothing completes. That
wait gives up after its bound (about 2 s). The CTA then reports DSA_STATUS_WAIT_TIMEOUT
in the status word, and all its roles stop. A split token whose first split never
arrives makes its other splits give up their bounded wait too. Each case checks three
things:
  * the status the host reads;
  * that the outputs the flag leaves computable are bit-identical to a clean call's;
  * that the context is still usable: the next clean call has status 0 and the same
    output.
"""

import time

import numpy as np
import pytest

from top_sparse_mla_gb300 import native
from top_sparse_mla_gb300 import workloads as W

import parity

pytestmark = pytest.mark.gpu

KEYS = ("out_fp8", "out_sf", "out", "lse")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from top_sparse_mla_gb300.build import build
    build()
    native.library()


def _splits(w):
    p = native.dsa_params_init(w.s_q, w.h_q, w.topk, w.n_swa_cols, w.kv_swa.shape[0], w.kv_cmp.shape[0])
    return native.dsa_sparse_attn_num_splits(p, 0)


def _same(a, b, tokens=slice(None)):
    for k in KEYS:
        assert np.array_equal(a[k][tokens], b[k][tokens], equal_nan=True), k


def _timed_out_run(w):
    t0 = time.perf_counter()
    g = parity.run_gpu(w, flags=native.DSA_FLAG_TEST_WAIT_TIMEOUT)
    dt = time.perf_counter() - t0
    assert g["status"] & native.DSA_STATUS_WAIT_TIMEOUT, f"status {g['status']:#x}"
    assert not g["status"] & native.DSA_STATUS_INDEX_OUT_OF_RANGE
    # the wait ran to its bound (about 2 s at the SM clock) and no further
    assert 0.5 < dt < 30.0, dt
    return g


@pytest.mark.parametrize("variant", ["fp8_ds_mla", "nvfp4_ds_mla", "fp8_q"])
def test_wait_timeout_without_splits_reports_and_recovers(variant):
    # 128 index columns: one tile, so no token is split; CTA 0 takes no item and the
    # other seven CTAs compute all eight tokens (on each of the kernel's instantiations)
    w = W.random_case(411, s_q=8, h_q=64, n_swa_cols=32, n_cmp_cols=96, n_swa_rows=256, n_cmp_rows=512,
                      n_sentinels=5, kv_format=1 if variant == "nvfp4_ds_mla" else 0,
                      cmp_scale=0.75 if variant == "nvfp4_ds_mla" else 1.0)
    w.fp8_q = variant == "fp8_q"
    assert _splits(w) == 1
    clean = parity.run_gpu(w)
    assert clean["status"] == 0
    g = _timed_out_run(w)
    _same(g, clean)
    again = parity.run_gpu(w)
    assert again["status"] == 0
    _same(again, clean)
    parity.compare(again, parity.run_oracle(w), label="after timeout")


def test_wait_timeout_with_splits_reports_and_recovers():
    # 1024 index columns over 4 tokens: every token is split over several CTAs (a
    # cooperative launch).  Token 0's first split is never computed, so its other
    # splits give up their wait for it; tokens 1..3 are complete.
    w = W.random_case(412, s_q=4, h_q=64, n_swa_cols=128, n_cmp_cols=896, n_swa_rows=512, n_cmp_rows=4096,
                      n_sentinels=17, lengths="ragged")
    assert _splits(w) > 1
    clean = parity.run_gpu(w)
    assert clean["status"] == 0
    g = _timed_out_run(w)
    _same(g, clean, tokens=slice(1, None))
    again = parity.run_gpu(w)
    assert again["status"] == 0
    _same(again, clean)
    parity.compare(again, parity.run_oracle(w), label="after timeout (split)")
