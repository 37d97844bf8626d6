"""The attention launched right after a producer kernel (DSA_FLAG_AFTER_PRODUCER): the
KV-cache insert rewrites the compressed-pool rows a decode batch reads, and the attention
follows on the same stream as the insert's programmatic dependent.  Each round writes
different rows, so an attention that read the pool before the insert had finished would
see the previous round's rows and miss the oracle."""

import numpy as np
import pytest
import torch

import parity
from oracle import codecs
from oracle.kv_insert import kv_insert
from top_sparse_mla_gb300 import api, native
from top_sparse_mla_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from top_sparse_mla_gb300.build import build
    build()
    native.library()


def test_attention_follows_the_kv_insert_as_a_programmatic_dependent():
    w = W.make("decode64")
    inp = api.upload(w, "cuda", flags=native.DSA_FLAG_AFTER_PRODUCER)
    assert native.dsa_sparse_attn_num_splits(inp.params) == 1           # the queue path
    out = api.allocate_outputs(inp, debug=True)
    # every compressed-pool row the batch reads
    cols = np.arange(w.topk)[None, :]
    live = (cols < w.topk_length[:, None]) & (w.indices >= 0) & (cols >= w.n_swa_cols)
    rows = np.unique(w.indices[live]).astype(np.int64)
    rng = np.random.default_rng(40)
    wn = codecs.bf16_encode(1.0 + 0.1 * rng.standard_normal(512))
    pos = rng.integers(0, 32768, size=rows.size).astype(np.int32)
    slots_d = torch.from_numpy(rows).cuda()
    pos_d = torch.from_numpy(pos).cuda()
    wn_d = torch.from_numpy(wn.view(np.int16)).cuda().view(torch.bfloat16)
    for rnd in range(3):
        kv = codecs.bf16_encode(rng.standard_normal((rows.size, 576)) * (1.0 + rnd))
        kv_d = torch.from_numpy(kv.view(np.int16)).cuda().view(torch.bfloat16)
        native.dsa_kv_insert(kv_d, pos_d, slots_d, wn_d, inp.kv_cmp)
        api.forward(inp, out)                                           # no sync in between
        torch.cuda.synchronize()
        # the oracle reads the pool bytes the kernel wrote (their codes are the oracle
        # insert's, bit for bit; scales and rotary values may differ in the last bit)
        pool = inp.kv_cmp.cpu().numpy()
        assert np.array_equal(pool[rows, :512], kv_insert(w.kv_cmp[rows], kv, pos, np.arange(rows.size), wn)[:, :512])
        got = {"out_fp8": out.out_fp8.cpu().numpy(), "out_sf": out.out_sf.cpu().numpy(),
               "out": out.out_precast.cpu().numpy().astype(np.float64), "lse": out.lse.cpu().numpy().astype(np.float64),
               "status": native.dsa_sparse_attn_read_status(out.workspace)}
        w_now = W.Workload(name=f"decode64_round{rnd}", q=w.q, norm_w=w.norm_w, kv_swa=w.kv_swa, kv_cmp=pool,
                           indices=w.indices, topk_length=w.topk_length, positions=w.positions,
                           n_swa_cols=w.n_swa_cols, seed=w.seed)
        assert got["status"] == 0
        parity.compare(got, parity.run_oracle(w_now), label=f"attention after the insert, round {rnd}")
