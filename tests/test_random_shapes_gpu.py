"""Seeded random shapes through the C ABI against the oracle.

Each case draws s_q (around the SM count, so both the split path and the queue path
are hit), h_q, the SWA / compressed column counts, sentinels and full or ragged
lengths; sampled tokens are compared element by element with the oracle, and the
status word must stay clean.
"""

import numpy as np
import pytest

import parity
from top_sparse_mla_gb300 import workloads as W

S_Q = [1, 2, 3, 5, 17, 64, 100, 151, 152, 153, 300]
H_Q = [1, 16, 40, 64]
SWA = [0, 16, 64, 128]
CMP = [32, 96, 200, 512, 896]


def _case(i: int):
    rng = np.random.default_rng(1000 + i)
    s_q, h_q = int(rng.choice(S_Q)), int(rng.choice(H_Q))
    sw, cm = int(rng.choice(SWA)), int(rng.choice(CMP))
    w = W.random_case(2000 + i, s_q=s_q, h_q=h_q, n_swa_cols=sw, n_cmp_cols=cm, n_swa_rows=max(sw, 1) * 4,
                      n_cmp_rows=cm * 3, n_sentinels=int(rng.integers(0, 20)),
                      lengths=str(rng.choice(["full", "ragged"])))
    tok = np.unique(np.concatenate([[0, s_q - 1], rng.choice(s_q, size=min(s_q, 6), replace=False)]))
    return w, tok


@pytest.mark.gpu
@pytest.mark.parametrize("i", range(40))
def test_random_shape(i):
    w, tok = _case(i)
    g = parity.run_gpu(w)
    assert g["status"] == 0, f"case {i}: kernel status {g['status']:#x}"
    r = parity.run_oracle(parity.subset(w, tok))
    parity.compare(g, r, tokens=tok, label=f"case {i} (s_q={w.s_q}, h_q={w.h_q})")
