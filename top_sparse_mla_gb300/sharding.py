"""Token sharding across ranks.

Query tokens are independent problems (each token carries its own positions, index row
and top-k length), so N ranks split a batch into N contiguous token ranges and run the
fused kernel on their own range with no collective on the data path.
"""

from __future__ import annotations

import numpy as np

from .workloads import Workload


def token_range(s_q: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous, balanced [start, stop) token range of `rank` out of `world`."""
    if world < 1 or not (0 <= rank < world):
        raise ValueError(f"bad rank {rank} of {world}")
    base, rem = divmod(s_q, world)
    start = rank * base + min(rank, rem)
    stop = start + base + (1 if rank < rem else 0)
    return start, stop


def shard(w: Workload, rank: int, world: int) -> Workload:
    """The rank's token slice of a workload (the caches are shared, not split)."""
    a, b = token_range(w.s_q, rank, world)
    sel = np.arange(a, b)
    return Workload(name=f"{w.name}_r{rank}of{world}", q=w.q[sel], norm_w=w.norm_w, kv_swa=w.kv_swa,
                    kv_cmp=w.kv_cmp, indices=w.indices[sel], topk_length=w.topk_length[sel],
                    positions=w.positions[sel], n_swa_cols=w.n_swa_cols, seed=w.seed, kv_format=w.kv_format,
                    cmp_scale=w.cmp_scale, softmax_scale=w.softmax_scale, fp8_q=w.fp8_q)
