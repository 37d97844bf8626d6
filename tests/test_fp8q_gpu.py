"""Parity of the CUDA path with an E4M3 q (DSA_FLAG_FP8_Q) against the oracle's reading
of the in-kernel q quantisation (OracleParams.fp8_q) on GB300."""

import numpy as np
import pytest

from oracle import codecs
from top_sparse_mla_gb300 import native
from top_sparse_mla_gb300 import workloads as W

import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from top_sparse_mla_gb300.build import build
    build()
    native.library()


def _full(w, out_scale=1.0):
    g = parity.run_gpu(w)
    assert g["status"] == 0, f"{w.name}: kernel status {g['status']:#x}"
    return parity.compare(g, parity.run_oracle(w), label=w.name, out_scale=out_scale)


@pytest.mark.parametrize("name", ["tiny_fp8q", "decode1_fp8q", "decode64_fp8q"])
def test_named_workloads_all_elements(name):
    print(name, _full(W.make(name)))


def test_decode1024_sampled_tokens():
    w = W.make("decode1024_fp8q")
    g = parity.run_gpu(w)
    assert g["status"] == 0
    rng = np.random.default_rng(9)
    tok = np.unique(np.concatenate([[0, 1, w.s_q - 1], rng.choice(w.s_q, size=40, replace=False)]))
    print(parity.compare(g, parity.run_oracle(parity.subset(w, tok)), tokens=tok, label="decode1024_fp8q"))


@pytest.mark.parametrize("h_q", [16, 40, 64])
def test_random_cases(h_q):
    w = W.random_case(700 + h_q, s_q=29, h_q=h_q, n_swa_cols=64, n_cmp_cols=300, n_swa_rows=700, n_cmp_rows=2000,
                      n_sentinels=9, lengths="ragged")
    w.fp8_q = True
    w.topk_length[3] = 0
    _full(w)


@pytest.mark.parametrize("q_scale", [2.0 ** -12, 2.0 ** 10])
def test_q_scalings(q_scale):
    # the codes do not depend on a power-of-two scale of q (the RMS factor cancels), and
    # the output only through eps
    w = W.make("decode64_fp8q")
    w.q = W._bf16_bits(codecs.bf16_decode(w.q).astype(np.float32) * np.float32(q_scale))
    _full(w)


def test_zero_latent_head():
    # a head whose latent part is all zero: codes 0, its scores come from the rope part
    w = W.make("tiny_fp8q")
    w.q[0, 3, :512] = 0
    _full(w)
