"""Seeded synthetic inputs for the sparse-attention path (shared by the tests, the bench
and the oracle checks).

This module only draws random numbers and stores them in the input formats the kernel
consumes; it holds none of the attention arithmetic.  Input encodings use PyTorch's
dtype casts: q and the rope part in bfloat16 (round to nearest even), the cache latent
in FP8 E4M3 with one fp32 scale per 128 values (scale = block amax / 448, the value
divided by the scale and cast to E4M3).

KV row layout (fp8_ds_mla, 656 bytes, 16-byte aligned):
  bytes [0, 512)    512 E4M3 latent values
  bytes [512, 528)  4 little-endian fp32 scales, scale g covers latent [128g, 128g+128)
  bytes [528, 656)  64 bfloat16 rope values
Rows that no token references are filled with NaN (latent code 0x7F, NaN scales, NaN
rope) so that a kernel reading a stale or sentinel row shows up as NaN in its output.

The five named workloads follow the shapes and distributions of the DeepSeek-V4.1
fused-attention benchmark (h_q = 64, top-k = 128 sliding-window + 512 compressed
columns): a tiny correctness case, single-token decode, batched decode (64 tokens),
large decode (1024 tokens, ragged top-k lengths) and a 2123-token prefill chunk.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

D_LATENT = 512
D_ROPE = 64
D_QK = 576
D_V = 512
ROW_BYTES = 656
NAN_BF16 = 0x7FC0


@dataclass
class Workload:
    name: str
    q: np.ndarray            # uint16 bf16 bits [s_q, h_q, 576]
    norm_w: np.ndarray       # uint16 bf16 bits [576]
    kv_swa: np.ndarray       # uint8 [n_swa_rows, 656]
    kv_cmp: np.ndarray       # uint8 [n_cmp_rows, 656]
    indices: np.ndarray      # int32 [s_q, topk]
    topk_length: np.ndarray  # int32 [s_q]
    positions: np.ndarray    # int32 [s_q]
    n_swa_cols: int
    seed: int
    notes: dict = field(default_factory=dict)

    @property
    def s_q(self) -> int:
        return int(self.q.shape[0])

    @property
    def h_q(self) -> int:
        return int(self.q.shape[1])

    @property
    def topk(self) -> int:
        return int(self.indices.shape[1])


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _nan_rows(n: int) -> np.ndarray:
    rows = np.empty((n, ROW_BYTES), dtype=np.uint8)
    rows[:, :D_LATENT] = 0x7F
    rows[:, D_LATENT:D_LATENT + 16] = np.frombuffer(np.full(4, np.nan, dtype="<f4").tobytes(), dtype=np.uint8)
    rope = np.full(D_ROPE, NAN_BF16, dtype="<u2")
    rows[:, D_LATENT + 16:] = np.frombuffer(rope.tobytes(), dtype=np.uint8)
    return rows


def encode_rows(latent: np.ndarray, rope: np.ndarray) -> np.ndarray:
    """Store float latent [n, 512] and rope [n, 64] as fp8_ds_mla rows [n, 656]."""
    n = latent.shape[0]
    lat = torch.from_numpy(np.ascontiguousarray(latent, dtype=np.float32)).view(n, 4, 128)
    amax = lat.abs().amax(dim=2, keepdim=True)
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    codes = (lat / scale).to(torch.float8_e4m3fn).view(torch.uint8).reshape(n, D_LATENT)
    out = np.empty((n, ROW_BYTES), dtype=np.uint8)
    out[:, :D_LATENT] = codes.numpy()
    out[:, D_LATENT:D_LATENT + 16] = scale.reshape(n, 4).numpy().astype("<f4").view(np.uint8)
    out[:, D_LATENT + 16:] = _bf16_bits(rope).view(np.uint8).reshape(n, 2 * D_ROPE)
    return out


def _fill_referenced(pool: np.ndarray, rows: np.ndarray, rng: np.random.Generator, chunk: int = 65536) -> None:
    rows = np.unique(rows[rows >= 0])
    for s in range(0, len(rows), chunk):
        r = rows[s:s + chunk]
        lat = rng.standard_normal((len(r), D_LATENT), dtype=np.float32)
        rope = rng.standard_normal((len(r), D_ROPE), dtype=np.float32)
        pool[r] = encode_rows(lat, rope)


def _q_and_w(rng, s_q, h_q):
    q = _bf16_bits(rng.standard_normal((s_q, h_q, D_QK), dtype=np.float32))
    w = _bf16_bits(1.0 + 0.1 * rng.standard_normal(D_QK, dtype=np.float32))
    return q, w


def _finish(name, rng, seed, q, w, n_swa_rows, n_cmp_rows, indices, topk_length, positions, n_swa_cols, notes=None):
    kv_swa = _nan_rows(n_swa_rows)
    kv_cmp = _nan_rows(n_cmp_rows)
    cols = np.arange(indices.shape[1])[None, :]
    live = cols < topk_length[:, None]
    _fill_referenced(kv_swa, np.where(live[:, :n_swa_cols], indices[:, :n_swa_cols], -1).ravel(), rng)
    _fill_referenced(kv_cmp, np.where(live[:, n_swa_cols:], indices[:, n_swa_cols:], -1).ravel(), rng)
    return Workload(name=name, q=q, norm_w=w, kv_swa=kv_swa, kv_cmp=kv_cmp,
                    indices=np.ascontiguousarray(indices, dtype=np.int32),
                    topk_length=np.ascontiguousarray(topk_length, dtype=np.int32),
                    positions=np.ascontiguousarray(positions, dtype=np.int32),
                    n_swa_cols=int(n_swa_cols), seed=int(seed), notes=notes or {})


def random_case(seed: int, s_q: int, h_q: int, n_swa_cols: int, n_cmp_cols: int,
                n_swa_rows: int, n_cmp_rows: int, n_sentinels: int = 0,
                lengths: str = "full", max_pos: int = 4096, name: str = "random") -> Workload:
    """Generic case: each token draws distinct rows from each pool, then
    ``n_sentinels`` of its columns (seeded, any position) become -1.
    ``lengths``: "full" -> topk_length = topk; "ragged" -> uniform in [0, topk]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    topk = n_swa_cols + n_cmp_cols
    q, w = _q_and_w(rng, s_q, h_q)
    positions = rng.integers(0, max_pos, size=s_q)
    idx = np.empty((s_q, topk), dtype=np.int64)
    for t in range(s_q):
        idx[t, :n_swa_cols] = rng.choice(n_swa_rows, size=n_swa_cols, replace=False)
        idx[t, n_swa_cols:] = rng.choice(n_cmp_rows, size=n_cmp_cols, replace=False)
        if n_sentinels:
            idx[t, rng.choice(topk, size=n_sentinels, replace=False)] = -1
    if lengths == "full":
        tl = np.full(s_q, topk)
    else:
        tl = rng.integers(0, topk + 1, size=s_q)
    return _finish(name, rng, seed, q, w, n_swa_rows, n_cmp_rows, idx, tl, positions, n_swa_cols)


def _swa_ring_cols(pos: int, ring_base: int, ring: int, window: int = 128) -> np.ndarray:
    p = pos - (window - 1) + np.arange(window)
    return np.where(p >= 0, ring_base + np.mod(p, ring), -1)


def config_tiny() -> Workload:
    """s_q=2, h_q=16, 16 SWA + 32 compressed columns with 5 -1 sentinels per token,
    a 256-row SWA cache and a 512-row compressed cache (seed 0)."""
    w = random_case(0, s_q=2, h_q=16, n_swa_cols=16, n_cmp_cols=32, n_swa_rows=256, n_cmp_rows=512,
                    n_sentinels=5, name="tiny_sq2_h16_topk48")
    return w


def config_decode1() -> Workload:
    """Single-token decode: h_q=64, 128 SWA columns (the ring positions pos-127..pos of
    an 8192-row ring) + 512 compressed columns distinct from 65536 rows (seed 1)."""
    seed = 1
    rng = np.random.Generator(np.random.PCG64(seed))
    q, w = _q_and_w(rng, 1, 64)
    pos = int(rng.integers(0, 4096))
    idx = np.empty((1, 640), dtype=np.int64)
    idx[0, :128] = _swa_ring_cols(pos, 0, 8192)
    idx[0, 128:] = rng.choice(65536, size=512, replace=False)
    return _finish("decode_sq1_h64_topk640", rng, seed, q, w, 8192, 65536, idx, np.array([640]), np.array([pos]), 128)


def config_decode64() -> Workload:
    """Batched decode: 64 tokens, positions in [0, 32768), each with its own 128-row
    SWA ring in a 64x128-row pool and 512 compressed rows distinct from 262144 (seed 2)."""
    seed = 2
    rng = np.random.Generator(np.random.PCG64(seed))
    s_q = 64
    q, w = _q_and_w(rng, s_q, 64)
    pos = rng.integers(0, 32768, size=s_q)
    idx = np.empty((s_q, 640), dtype=np.int64)
    for t in range(s_q):
        idx[t, :128] = _swa_ring_cols(int(pos[t]), t * 128, 128)
        idx[t, 128:] = rng.choice(262144, size=512, replace=False)
    return _finish("decode_sq64_h64_topk640", rng, seed, q, w, s_q * 128, 262144, idx, np.full(s_q, 640), pos, 128)


def config_decode1024() -> Workload:
    """Large decode: 1024 tokens, topk_length uniform in [64, 640] with the row tail
    set to -1, each token's 128 SWA columns a random order of its own 128-row ring
    (pool 1024x128 rows), 512 compressed rows distinct from 1,048,576 (seed 3).
    Positions (not fixed by the workload description) are uniform in [0, 32768)."""
    seed = 3
    rng = np.random.Generator(np.random.PCG64(seed))
    s_q = 1024
    q, w = _q_and_w(rng, s_q, 64)
    pos = rng.integers(0, 32768, size=s_q)
    tl = rng.integers(64, 641, size=s_q)
    idx = np.empty((s_q, 640), dtype=np.int64)
    for t in range(s_q):
        idx[t, :128] = t * 128 + rng.permutation(128)
        idx[t, 128:] = rng.choice(1 << 20, size=512, replace=False)
        idx[t, tl[t]:] = -1
    return _finish("decode_sq1024_h64_topk640_ragged", rng, seed, q, w, s_q * 128, 1 << 20, idx, tl, pos, 128)


def config_prefill2123() -> Workload:
    """Prefill chunk: positions 0..2122 of one sequence; SWA columns are the causal
    window p-127..p (-1 before the sequence start) into a position-indexed pool;
    compressed columns are min(p+1, 512) distinct rows r <= p of a 2048-row pool,
    the remaining columns -1; topk_length = 640 (seed 4)."""
    seed = 4
    rng = np.random.Generator(np.random.PCG64(seed))
    s_q = 2123
    q, w = _q_and_w(rng, s_q, 64)
    pos = np.arange(s_q)
    idx = np.full((s_q, 640), -1, dtype=np.int64)
    for t in range(s_q):
        p = int(pos[t])
        idx[t, :128] = _swa_ring_cols(p, 0, 1 << 30)   # no wrap: pool rows are positions
        n = min(p + 1, 512)
        idx[t, 128:128 + n] = rng.choice(min(p + 1, 2048), size=n, replace=False)
    return _finish("prefill_sq2123_h64_topk640", rng, seed, q, w, s_q, 2048, idx, np.full(s_q, 640), pos, 128)


CONFIGS = {
    "tiny": config_tiny,
    "decode1": config_decode1,
    "decode64": config_decode64,
    "decode1024": config_decode1024,
    "prefill2123": config_prefill2123,
}


def make(name: str) -> Workload:
    return CONFIGS[name]()


def n_valid_rows(w: Workload) -> np.ndarray:
    """Valid (in-length, non-negative) index columns per token."""
    cols = np.arange(w.topk)[None, :]
    live = (cols < w.topk_length[:, None]) & (w.indices >= 0)
    return live.sum(axis=1)
