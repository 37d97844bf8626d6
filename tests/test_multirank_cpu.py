"""World-size-2 checks of the multi-rank path on CPU (gloo): token sharding covers the
batch exactly once; each rank takes bench.py's slice of the batch and prepares the
library call for it (parameters, split count, workspace size, launches) through the C
ABI's host entry points; sharded results reassemble to the unsharded ones; and the
max-over-ranks timing reduction bench.py uses returns the slowest rank."""

import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    import bench
    from top_sparse_mla_gb300 import native, sharding, workloads as W
    w = W.random_case(77, s_q=7, h_q=4, n_swa_cols=16, n_cmp_cols=48, n_swa_rows=128, n_cmp_rows=256,
                      n_sentinels=4, lengths="ragged")
    part = bench.rank_workload(w, rank, world)
    assert bench.rank_workload(w, rank, world, replicas=True) is w
    # the library call this rank would make for its slice (host entry points only)
    native.library()
    p = native.dsa_params_init(part.s_q, part.h_q, part.topk, part.n_swa_cols, part.kv_swa.shape[0],
                               part.kv_cmp.shape[0])
    ns = native.dsa_sparse_attn_num_splits(p, 152)
    ws = native.dsa_sparse_attn_workspace_size(p, 152)
    assert ns >= 1 and ws >= 256 and ws % 256 == 0
    assert bench.kernels_per_call(p, 152) == (2 if ns == 1 else 1)
    dist.all_gather_object(info := [None] * world, (part.s_q, ns, ws))
    r = oracle.sparse_mla_forward(part.q, part.kv_swa, part.kv_cmp, part.indices, part.topk_length,
                                  part.positions, part.norm_w, oracle.OracleParams(n_swa_cols=w.n_swa_cols))
    # variable-size shards: pad to the largest, gather, trim
    a, b = sharding.token_range(w.s_q, rank, world)
    n_max = -(-w.s_q // world)
    buf = torch.zeros((n_max, w.h_q, 512), dtype=torch.float64)
    buf[: b - a] = torch.from_numpy(r["out"])
    gathered = [torch.zeros_like(buf) for _ in range(world)]
    dist.all_gather(gathered, buf)
    slowest = bench.max_over_ranks(dist, float(rank + 1) * 0.25)
    assert sum(x[0] for x in info) == w.s_q
    if rank == 0:
        pieces = []
        for k in range(world):
            ka, kb = sharding.token_range(w.s_q, k, world)
            pieces.append(gathered[k][: kb - ka].numpy())
        np.save(os.path.join(out_dir, "sharded.npy"), np.concatenate(pieces))
        full = oracle.sparse_mla_forward(w.q, w.kv_swa, w.kv_cmp, w.indices, w.topk_length, w.positions,
                                         w.norm_w, oracle.OracleParams(n_swa_cols=w.n_swa_cols))
        np.save(os.path.join(out_dir, "full.npy"), full["out"])
        np.save(os.path.join(out_dir, "slowest.npy"), np.array([slowest]))
    dist.barrier()
    dist.destroy_process_group()


def test_token_ranges_partition_the_batch():
    from top_sparse_mla_gb300 import sharding
    for s_q in (0, 1, 5, 64, 1024, 2123):
        for world in (1, 2, 3, 8):
            seen = []
            for r in range(world):
                a, b = sharding.token_range(s_q, r, world)
                assert 0 <= a <= b <= s_q
                seen.extend(range(a, b))
            assert seen == list(range(s_q))
    with pytest.raises(ValueError):
        sharding.token_range(4, 2, 2)


def test_two_gloo_ranks_reassemble_the_unsharded_result(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    sharded = np.load(tmp_path / "sharded.npy")
    full = np.load(tmp_path / "full.npy")
    assert sharded.shape == full.shape
    assert np.array_equal(sharded, full)
    assert float(np.load(tmp_path / "slowest.npy")[0]) == 0.5
