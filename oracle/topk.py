"""Top-k column selection of the index producer that feeds the sparse attention (test
infrastructure only: the import rules of this package apply).

Source: vLLM PR #64364 (DeepSeek-V4.1-Flash latency_specialized decode at TP4 on
GB300), its Claims and Validation sections.  For each token, the producer
(``topk_bf16_small``) selects k columns of the indexer's bf16 logits, and its output is
specified as follows:
  * the threshold is the row's k-th largest value, the one ``torch.topk`` returns last;
  * every column above the threshold is selected;
  * among the columns equal to the threshold, the lowest-numbered ones are selected,
    as many as are needed to make k;
  * the selected columns are listed in ascending order.
The same page says the attention reads each token's top-k directly, with no index-table
build in between.  This function's output therefore has the shape of the attention's
``indices`` / ``topk_length`` inputs.

Readings where the page is silent:
  * A row may have fewer candidate columns than the logits' width. Columns at or past
    ``lengths[t]`` are not candidates, which covers causal and ragged rows. With fewer
    than k candidates, all of them are selected.
  * The row is padded to k with -1, the attention's sentinel, and ``topk_length[t]``
    is the number selected.
  * NaN orders above +inf, as ``torch.topk`` orders it; -inf is an ordinary value.
  * The page's "remap" of the selected columns is not defined there and is not part
    of this function.

Parity: pinned against a brute-force enumeration and against torch.topk in the CPU
tests. The CUDA path (dsa_topk_select) is compared with it bit for bit on the GPU.
"""

from __future__ import annotations

import numpy as np


def topk_select(logits, k: int, lengths=None):
    """logits: float array [s_q, n] (bf16 values, held exactly in float32/float64);
    k >= 0; lengths: int array [s_q] of candidate columns per row (None: all n).
    Returns (indices int32 [s_q, k], topk_length int32 [s_q])."""
    x = np.asarray(logits, dtype=np.float64)
    if x.ndim != 2:
        raise ValueError("logits must be [s_q, n]")
    if k < 0:
        raise ValueError("k must be >= 0")
    s_q, n = x.shape
    indices = np.full((s_q, k), -1, dtype=np.int32)
    count = np.zeros(s_q, dtype=np.int32)
    for t in range(s_q):
        L = n if lengths is None else min(max(int(lengths[t]), 0), n)
        m = min(k, L)
        if m == 0:
            continue
        row = x[t, :L]
        nan = np.isnan(row)
        # rank the candidates: NaN first, then by value from the largest, then by column
        # from the lowest (np.lexsort sorts by its last key first)
        rank = np.lexsort((np.arange(L), -np.where(nan, 0.0, row), ~nan))
        indices[t, :m] = np.sort(rank[:m])
        count[t] = m
    return indices, count
