"""The top-k column selection's CUDA path (include/dsa_topk.h) against the oracle's
selection (oracle/topk.py), bit for bit: the same columns in the same order, the same
-1 padding and the same topk_length."""

import numpy as np
import pytest
import torch

from oracle.topk import topk_select
from top_sparse_mla_gb300 import native

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from top_sparse_mla_gb300.build import build
    build()
    native.library()


def _check(x: torch.Tensor, k: int, lengths=None, pad: int = 0):
    """x: bf16 [s_q, n] on the host. Runs the CUDA path with rows `pad` elements longer
    than n and compares with the oracle."""
    s_q, n = x.shape
    buf = torch.zeros((s_q, n + pad), dtype=torch.bfloat16, device="cuda")
    buf[:, :n] = x.to("cuda")
    logits = buf[:, :n]
    idx = torch.full((s_q, k), 123456, dtype=torch.int32, device="cuda")
    tl = torch.full((s_q,), 777, dtype=torch.int32, device="cuda")
    ln = None if lengths is None else torch.tensor(lengths, dtype=torch.int32, device="cuda")
    native.dsa_topk_select(logits, k, idx, tl, ln)
    torch.cuda.synchronize()
    exp_idx, exp_len = topk_select(x.float().numpy(), k, None if lengths is None else np.asarray(lengths))
    assert np.array_equal(tl.cpu().numpy(), exp_len)
    assert np.array_equal(idx.cpu().numpy(), exp_idx)


def _tied(rng, s_q, n, step=0.125):
    return torch.tensor(np.round(rng.normal(size=(s_q, n)) / step) * step, dtype=torch.bfloat16)


@pytest.mark.parametrize("n,k", [(1, 1), (7, 3), (100, 64), (1000, 640), (4097, 2048), (8192, 512), (8193, 512),
                                 (20000, 512), (65536, 2048)])
def test_random_rows_with_ties(n, k):
    rng = np.random.default_rng(n + k)
    _check(_tied(rng, 5, n), k)


def test_ragged_lengths_and_padded_rows():
    rng = np.random.default_rng(21)
    n = 3000
    x = _tied(rng, 8, n, step=0.5)
    _check(x, 700, lengths=[3000, 700, 699, 0, -3, 5000, 1, 1500], pad=40)
    # an odd row pitch: rows start off the 16-byte grid (element loads instead of vectors)
    _check(x, 700, lengths=[3000, 701, 2999, 33, 64, 5000, 31, 1500], pad=3)
    # rows of the register path's boundary length, and one past it (the shared-memory path)
    for n2 in (8192, 8193):
        y = _tied(rng, 4, n2, step=0.25)
        _check(y, 512, lengths=[n2, 4000, 513, n2 - 1], pad=5)


def test_special_values():
    vals = [float("nan"), -float("nan"), float("inf"), -float("inf"), 0.0, -0.0, 1.0, -1.0, 3.5]
    rng = np.random.default_rng(22)
    x = torch.tensor(rng.choice(vals, size=(6, 777)), dtype=torch.bfloat16)
    # NaNs with other payloads
    xb = x.view(torch.int16)
    xb[0, ::5] = 0x7FC1
    xb[1, ::7] = -0x3F                      # 0xFFC1: a negative NaN
    for k in (1, 10, 100, 400, 776, 777, 2048):
        _check(xb.view(torch.bfloat16), k)


def test_ties_across_column_chunks_and_all_equal_rows():
    # two values only: the k-th value is tied over thousands of columns, across the
    # kernel's 1024-column chunks
    rng = np.random.default_rng(23)
    x = torch.tensor(rng.integers(0, 2, size=(4, 5000)).astype(np.float32), dtype=torch.bfloat16)
    for k in (1, 1023, 1024, 1025, 2048):
        _check(x, k)
    _check(torch.zeros((3, 4096), dtype=torch.bfloat16), 2048)
    _check(torch.full((2, 10), -7.0, dtype=torch.bfloat16), 0)


def test_output_feeds_the_attention_indices():
    # the selection's form is the attention's: ascending columns, then -1
    rng = np.random.default_rng(24)
    x = _tied(rng, 3, 640)
    idx = torch.empty((3, 128), dtype=torch.int32, device="cuda")
    tl = torch.empty((3,), dtype=torch.int32, device="cuda")
    native.dsa_topk_select(x.to("cuda"), 128, idx, tl, torch.tensor([640, 100, 0], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    i, l = idx.cpu().numpy(), tl.cpu().numpy()
    assert list(l) == [128, 100, 0]
    for t in range(3):
        assert np.all(np.diff(i[t, :l[t]]) > 0) and np.all(i[t, l[t]:] == -1)


def test_many_rows_ragged():
    # more rows than the GPU holds CTAs at once: ragged lengths, rows with at most k
    # candidates and empty rows mixed in, and a row pitch of n + 8
    rng = np.random.default_rng(25)
    s_q, n, k = 1500, 2048, 256
    x = _tied(rng, s_q, n, step=0.25)
    lengths = rng.integers(-5, n + 100, size=s_q)
    lengths[::7] = rng.integers(0, k + 1, size=len(lengths[::7]))
    _check(x, k, lengths=list(lengths), pad=8)
    _check(x, k)
