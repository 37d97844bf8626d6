"""The queue path's token order on GB300.

When no token is split, a small kernel runs before the fused kernel. It sorts the
tokens by their number of 128-row tiles (from topk_length, clipped to [0, topk]), most
tiles first, and keeps token order among equal counts. The fused kernel's CTAs then
take tokens from one queue in that order. The order sits in the workspace right after
its 256-byte header, in the region the split path uses for its arrival counters. Above
65536 tokens the queue takes tokens in index order and no order is written.

The order decides only which CTA computes a token, never the token's result. These
tests check:
  * the order itself: a permutation, longest first and stable;
  * that every token is computed exactly once, on both sides of the 65536-token bound;
  * that a token and its twin, given the same inputs, get bit-identical outputs;
  * that tokens without a valid column, placed among long ones, are written by the
    queue path without stalling it.
"""

import numpy as np
import pytest
import torch

from top_sparse_mla_gb300 import api, native
from top_sparse_mla_gb300 import workloads as W

import parity

pytestmark = pytest.mark.gpu

HEADER_BYTES = 256
ORDER_MAX_TOKENS = native.DSA_ORDER_MAX_TOKENS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from top_sparse_mla_gb300.build import build
    build()
    native.library()


def _tiles(w):
    return (np.clip(w.topk_length.astype(np.int64), 0, w.topk) + 127) // 128


def _run(w, debug=False):
    inp = api.upload(w, "cuda:0")
    assert native.dsa_sparse_attn_num_splits(inp.params, 0) == 1
    out = api.allocate_outputs(inp, debug=debug)
    api.forward(inp, out)
    torch.cuda.synchronize()
    assert native.dsa_sparse_attn_read_status(out.workspace) == 0
    order = out.workspace[HEADER_BYTES:HEADER_BYTES + 4 * w.s_q].view(torch.int32).cpu().numpy()
    return out, order


def _ragged(seed, s_q):
    w = W.random_case(seed, s_q=s_q, h_q=8, n_swa_cols=64, n_cmp_cols=1000, n_swa_rows=2048, n_cmp_rows=8192,
                      n_sentinels=9, lengths="ragged")
    w.topk_length[::17] = -3                 # negative: no tile
    w.topk_length[5::29] = 10 ** 6           # beyond topk: capped at topk
    return w


@pytest.mark.parametrize("case", ["ragged300", "ragged2500", "equal400", "decode1024"])
def test_order_is_a_stable_longest_first_permutation(case):
    if case == "ragged300":
        w = _ragged(501, 300)
    elif case == "ragged2500":
        w = _ragged(502, 2500)                # several 1024-token chunks of the sort
    elif case == "equal400":
        w = W.random_case(503, s_q=400, h_q=8, n_swa_cols=128, n_cmp_cols=512, n_swa_rows=1024,
                          n_cmp_rows=4096)    # every token 5 tiles: the order is the identity
    else:
        w = W.make("decode1024")
    _, order = _run(w)
    assert np.array_equal(np.sort(order), np.arange(w.s_q))
    assert np.array_equal(order, np.argsort(-_tiles(w), kind="stable"))


def _repeated(s_q, seed):
    """s_q tokens: a 64-token random case repeated, so that token t equals token t % 64."""
    base = W.random_case(seed, s_q=64, h_q=2, n_swa_cols=16, n_cmp_cols=240, n_swa_rows=512, n_cmp_rows=4096,
                         n_sentinels=5, lengths="ragged")
    reps = -(-s_q // 64)

    def rep(a):
        return np.ascontiguousarray(np.concatenate([a] * reps, axis=0)[:s_q])

    w = W.Workload(name=f"repeated{s_q}", q=rep(base.q), norm_w=base.norm_w, kv_swa=base.kv_swa,
                   kv_cmp=base.kv_cmp, indices=rep(base.indices), topk_length=rep(base.topk_length),
                   positions=rep(base.positions), n_swa_cols=base.n_swa_cols, seed=seed)
    return base, w


@pytest.mark.parametrize("s_q", [ORDER_MAX_TOKENS, ORDER_MAX_TOKENS + 1])
def test_every_token_once_at_the_order_bound(s_q):
    base, w = _repeated(s_q, 504)
    out, order = _run(w, debug=True)
    if s_q <= ORDER_MAX_TOKENS:
        assert np.array_equal(order, np.argsort(-_tiles(w), kind="stable"))
    g = {"out_fp8": out.out_fp8.cpu().numpy(), "out_sf": out.out_sf.cpu().numpy(),
         "out": out.out_precast.cpu().numpy().astype(np.float64), "lse": out.lse.cpu().numpy().astype(np.float64)}
    # each token equals its twin among the first 64, bit for bit
    twin = np.arange(s_q) % 64
    for k in ("out_fp8", "out_sf", "out", "lse"):
        assert np.array_equal(g[k], g[k][twin], equal_nan=True), k
    # and the first 64 match the oracle
    parity.compare(g, parity.run_oracle(base), tokens=np.arange(64), label=f"repeated {s_q}")


def test_tokens_without_rows_among_long_ones():
    # Queue path. Two of every five tokens have only sentinels but a full topk_length:
    # they have no tile, yet the order puts them among the longest tokens. Each CTA
    # therefore meets items without tiles right after items with tiles, twice in a
    # row. The epilogue share of the item before must not wait for items the queue has
    # not handed out yet.
    w = W.random_case(505, s_q=2000, h_q=8, n_swa_cols=64, n_cmp_cols=192, n_swa_rows=2048, n_cmp_rows=8192,
                      n_sentinels=3)
    t = np.arange(w.s_q)
    w.indices[(t % 5 == 1) | (t % 5 == 2)] = -1
    _, order = _run(w)
    assert np.array_equal(order, np.argsort(-_tiles(w), kind="stable"))
    g = parity.run_gpu(w)
    assert g["status"] == 0
    parity.compare(g, parity.run_oracle(w), label="empty tokens in the queue")
