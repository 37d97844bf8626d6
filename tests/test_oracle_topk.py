"""Pins of the oracle's top-k column selection (oracle/topk.py), CPU only.

The rule (vLLM PR #64364, Claims and Validation): the threshold is torch.topk's k-th
value, every column above it is selected, among the columns equal to it the
lowest-numbered ones fill the row, and the selected columns are listed in ascending
order. The pins below do not restate the oracle's sort:
  * brute force: every k-subset of a tiny row, keeping the valid ones (no unselected
    column ranks above a selected one), then the lexicographically smallest;
  * torch.topk itself, as the library routine the rule names: the threshold and the
    multiset of selected values;
  * hand-worked rows with ties, -inf and NaN;
  * the output's form: ascending, distinct, in range, padded with -1.
"""

import itertools
import math

import numpy as np
import pytest
import torch

from oracle.topk import topk_select

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _above(a: float, b: float) -> bool:
    """a ranks above b: NaN above everything (torch.topk's order), else a > b."""
    if math.isnan(a):
        return not math.isnan(b)
    if math.isnan(b):
        return False
    return a > b


def _brute(row, k, L):
    m = min(k, L)
    best = None
    for s in itertools.combinations(range(L), m):
        chosen = set(s)
        if any(_above(row[j], row[i]) for i in chosen for j in range(L) if j not in chosen):
            continue
        if best is None or s < best:
            best = s
    return list(best)


def test_brute_force_on_tiny_rows_with_heavy_ties():
    rng = np.random.default_rng(11)
    pool = np.array([-np.inf, -1.0, 0.0, 0.5, 1.0, np.inf, np.nan])
    for trial in range(300):
        n = int(rng.integers(1, 8))
        row = rng.choice(pool[:6] if trial % 3 else pool, size=n)
        for k in range(0, n + 2):
            for L in range(0, n + 1):
                idx, cnt = topk_select(row[None, :], k, np.array([L]))
                exp = _brute(list(row), k, L)
                assert cnt[0] == len(exp)
                assert list(idx[0, :cnt[0]]) == exp, (row, k, L)
                assert np.all(idx[0, cnt[0]:] == -1)


def test_threshold_and_selected_values_match_torch_topk():
    rng = np.random.default_rng(12)
    for _ in range(50):
        n = int(rng.integers(1, 300))
        k = int(rng.integers(1, n + 1))
        # bf16 values with many ties: a few hundred distinct values, rounded to bf16
        row = torch.tensor(np.round(rng.normal(size=n) * 8) / 8, dtype=torch.bfloat16)
        idx, cnt = topk_select(row.float().numpy()[None, :], k)
        assert cnt[0] == k
        sel = row.float().numpy()[idx[0]]
        vals = torch.topk(row, k).values.float().numpy()
        assert np.array_equal(np.sort(sel), np.sort(vals))
        assert sel.min() == vals[-1]                       # the k-th value is the threshold


def test_nan_ranks_first_as_in_torch_topk():
    row = np.array([0.5, np.nan, 2.0, np.inf, -np.inf, np.nan, 1.0])
    t_idx = torch.topk(torch.tensor(row), 3).indices.numpy()
    assert set(t_idx[:2]) == {1, 5}                        # torch puts both NaNs first
    idx, cnt = topk_select(row[None, :], 3)
    assert list(idx[0]) == [1, 3, 5]                       # the NaNs, then +inf


def test_hand_worked_rows():
    row = np.array([[0.5, 1.0, 0.5, 2.0, 0.5, -np.inf, 1.0]])
    # 2.0 (column 3) > 1.0 (columns 1, 6) > 0.5 (columns 0, 2, 4) > -inf (column 5)
    cases = {1: [3], 2: [1, 3], 3: [1, 3, 6], 4: [0, 1, 3, 6], 5: [0, 1, 2, 3, 6],
             6: [0, 1, 2, 3, 4, 6], 7: [0, 1, 2, 3, 4, 5, 6]}
    for k, exp in cases.items():
        idx, cnt = topk_select(row, k)
        assert cnt[0] == len(exp) and list(idx[0]) == exp
    # all equal: the lowest columns
    idx, _ = topk_select(np.zeros((1, 6)), 3)
    assert list(idx[0]) == [0, 1, 2]


def test_lengths_padding_and_shapes():
    rng = np.random.default_rng(13)
    x = rng.normal(size=(5, 40))
    lengths = np.array([40, 10, 0, -4, 99])
    idx, cnt = topk_select(x, 16, lengths)
    assert idx.shape == (5, 16) and idx.dtype == np.int32 and cnt.dtype == np.int32
    assert list(cnt) == [16, 10, 0, 0, 16]
    for t in range(5):
        c = cnt[t]
        L = min(max(lengths[t], 0), 40)
        sel = idx[t, :c]
        assert np.all(np.diff(sel) > 0) and np.all((sel >= 0) & (sel < max(L, 1)))
        assert np.all(idx[t, c:] == -1)
        if c:
            # nothing left out ranks above anything selected
            rest = np.setdiff1d(np.arange(L), sel)
            assert rest.size == 0 or x[t, rest].max() <= x[t, sel].min()
    # a row shorter than k selects every candidate
    assert list(idx[1, :10]) == list(range(10))
    idx0, cnt0 = topk_select(x, 0)
    assert idx0.shape == (5, 0) and not cnt0.any()
