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

The nvfp4_ds_mla variants (kv_format 1, the V4.1 cache; byte layout in
include/dsa_sparse_attn.h) hold 512-dim keys with the rotary dims inside: q and norm_w
have 512 dims, kv_swa rows are 528 bytes (512 E4M3 values, 4 fp32 scales as above) and
kv_cmp rows 288 bytes (512 E2M1 values, low nibble first, then 32 E4M3 scales, one per
16 values; the values are divided by the pool's cmp_scale first, each 16-value scale is
amax / 6 cast to E4M3, and each value the nearest E2M1 value of value / scale, ties to
the even code).  Unreferenced fp4 rows carry NaN scales (E4M3 code 0x7F).

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
NVFP4_SWA_ROW_BYTES = 528
NVFP4_CMP_ROW_BYTES = 288
E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
NVFP4_CMP_SCALE = 0.75   # the named nvfp4_ds_mla workloads' kv_cmp scale


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
    kv_format: int = 0              # 0: fp8_ds_mla (656-byte rows), 1: nvfp4_ds_mla (528 / 288)
    cmp_scale: float = 1.0          # nvfp4_ds_mla: fp32 scale of every kv_cmp value
    softmax_scale: float = 1.0 / 24.0   # 1/sqrt(576); 1/sqrt(512) for nvfp4_ds_mla
    fp8_q: bool = False             # q's latent quantised to E4M3 in the kernel (DSA_FLAG_FP8_Q)

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


def encode_rows_nvfp4_swa(x: np.ndarray) -> np.ndarray:
    """Store float keys [n, 512] as nvfp4_ds_mla sliding-window rows [n, 528]: 512 E4M3
    values and 4 fp32 scales (block amax / 448)."""
    n = x.shape[0]
    lat = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).view(n, 4, 128)
    amax = lat.abs().amax(dim=2, keepdim=True)
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    out = np.empty((n, NVFP4_SWA_ROW_BYTES), dtype=np.uint8)
    out[:, :D_LATENT] = (lat / scale).to(torch.float8_e4m3fn).view(torch.uint8).reshape(n, D_LATENT).numpy()
    out[:, D_LATENT:] = scale.reshape(n, 4).numpy().astype("<f4").view(np.uint8)
    return out


def _e2m1_codes(v: np.ndarray) -> np.ndarray:
    """Nearest E2M1 code of each value (ties to the even code, saturating at 6)."""
    mag = np.minimum(np.abs(v), 6.0)
    d = np.abs(mag[..., None] - E2M1_MAGNITUDES)
    d = d + (np.arange(8) & 1) * 1e-9          # an exact tie goes to the even code
    code = np.argmin(d, axis=-1).astype(np.uint8)
    return np.where((v < 0) & (code > 0), code | 8, code).astype(np.uint8)


def encode_rows_nvfp4_cmp(x: np.ndarray, cmp_scale: float) -> np.ndarray:
    """Store float keys [n, 512] as nvfp4_ds_mla compressed rows [n, 288] (layout in the
    module docstring)."""
    n = x.shape[0]
    y = (np.asarray(x, dtype=np.float64) / cmp_scale).reshape(n, 32, 16)
    amax = np.max(np.abs(y), axis=2)
    sc_codes = torch.from_numpy((amax / 6.0).astype(np.float32)).to(torch.float8_e4m3fn)
    sc = sc_codes.to(torch.float32).numpy().astype(np.float64)
    vals = np.where(sc[..., None] > 0, y / np.where(sc > 0, sc, 1.0)[..., None], 0.0)
    nib = _e2m1_codes(vals).reshape(n, D_LATENT)
    out = np.empty((n, NVFP4_CMP_ROW_BYTES), dtype=np.uint8)
    out[:, :256] = nib[:, 0::2] | (nib[:, 1::2] << 4)
    out[:, 256:] = sc_codes.view(torch.uint8).numpy()
    return out


def _nan_rows_nvfp4(n: int, cmp: bool) -> np.ndarray:
    if cmp:
        rows = np.full((n, NVFP4_CMP_ROW_BYTES), 0x77, dtype=np.uint8)
        rows[:, 256:] = 0x7F                    # E4M3 NaN scales
        return rows
    rows = np.empty((n, NVFP4_SWA_ROW_BYTES), dtype=np.uint8)
    rows[:, :D_LATENT] = 0x7F
    rows[:, D_LATENT:] = np.frombuffer(np.full(4, np.nan, dtype="<f4").tobytes(), dtype=np.uint8)
    return rows


def _fill_referenced(pool: np.ndarray, rows: np.ndarray, rng: np.random.Generator, chunk: int = 65536,
                     kv_format: int = 0, cmp: bool = False, cmp_scale: float = 1.0) -> None:
    rows = np.unique(rows[rows >= 0])
    for s in range(0, len(rows), chunk):
        r = rows[s:s + chunk]
        lat = rng.standard_normal((len(r), D_LATENT), dtype=np.float32)
        if kv_format == 0:
            rope = rng.standard_normal((len(r), D_ROPE), dtype=np.float32)
            pool[r] = encode_rows(lat, rope)
        elif cmp:
            pool[r] = encode_rows_nvfp4_cmp(lat, cmp_scale)
        else:
            pool[r] = encode_rows_nvfp4_swa(lat)


def _q_and_w(rng, s_q, h_q, d=D_QK):
    q = _bf16_bits(rng.standard_normal((s_q, h_q, d), dtype=np.float32))
    w = _bf16_bits(1.0 + 0.1 * rng.standard_normal(d, dtype=np.float32))
    return q, w


def _finish(name, rng, seed, q, w, n_swa_rows, n_cmp_rows, indices, topk_length, positions, n_swa_cols, notes=None,
            kv_format=0, cmp_scale=1.0):
    if kv_format == 0:
        kv_swa, kv_cmp = _nan_rows(n_swa_rows), _nan_rows(n_cmp_rows)
    else:
        kv_swa, kv_cmp = _nan_rows_nvfp4(n_swa_rows, False), _nan_rows_nvfp4(n_cmp_rows, True)
    cols = np.arange(indices.shape[1])[None, :]
    live = cols < topk_length[:, None]
    _fill_referenced(kv_swa, np.where(live[:, :n_swa_cols], indices[:, :n_swa_cols], -1).ravel(), rng,
                     kv_format=kv_format)
    _fill_referenced(kv_cmp, np.where(live[:, n_swa_cols:], indices[:, n_swa_cols:], -1).ravel(), rng,
                     kv_format=kv_format, cmp=True, cmp_scale=cmp_scale)
    return Workload(name=name, q=q, norm_w=w, kv_swa=kv_swa, kv_cmp=kv_cmp,
                    indices=np.ascontiguousarray(indices, dtype=np.int32),
                    topk_length=np.ascontiguousarray(topk_length, dtype=np.int32),
                    positions=np.ascontiguousarray(positions, dtype=np.int32),
                    n_swa_cols=int(n_swa_cols), seed=int(seed), notes=notes or {},
                    kv_format=int(kv_format), cmp_scale=float(cmp_scale),
                    softmax_scale=1.0 / 24.0 if kv_format == 0 else float(1.0 / np.sqrt(512.0)))


def random_case(seed: int, s_q: int, h_q: int, n_swa_cols: int, n_cmp_cols: int,
                n_swa_rows: int, n_cmp_rows: int, n_sentinels: int = 0,
                lengths: str = "full", max_pos: int = 4096, name: str = "random", kv_format: int = 0,
                cmp_scale: float = 1.0) -> Workload:
    """Generic case: each token draws distinct rows from each pool, then
    ``n_sentinels`` of its columns (seeded, any position) become -1.
    ``lengths``: "full" -> topk_length = topk; "ragged" -> uniform in [0, topk]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    topk = n_swa_cols + n_cmp_cols
    q, w = _q_and_w(rng, s_q, h_q, D_QK if kv_format == 0 else D_LATENT)
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
    return _finish(name, rng, seed, q, w, n_swa_rows, n_cmp_rows, idx, tl, positions, n_swa_cols,
                   kv_format=kv_format, cmp_scale=cmp_scale)


def _swa_ring_cols(pos: int, ring_base: int, ring: int, window: int = 128) -> np.ndarray:
    p = pos - (window - 1) + np.arange(window)
    return np.where(p >= 0, ring_base + np.mod(p, ring), -1)


def config_tiny(kv_format: int = 0) -> Workload:
    """s_q=2, h_q=16, 16 SWA + 32 compressed columns with 5 -1 sentinels per token,
    a 256-row SWA cache and a 512-row compressed cache (seed 0)."""
    w = random_case(0, s_q=2, h_q=16, n_swa_cols=16, n_cmp_cols=32, n_swa_rows=256, n_cmp_rows=512,
                    n_sentinels=5, name="tiny_sq2_h16_topk48" + ("_nvfp4" if kv_format else ""),
                    kv_format=kv_format, cmp_scale=NVFP4_CMP_SCALE if kv_format else 1.0)
    return w


def config_decode1(kv_format: int = 0) -> Workload:
    """Single-token decode: h_q=64, 128 SWA columns (the ring positions pos-127..pos of
    an 8192-row ring) + 512 compressed columns distinct from 65536 rows (seed 1)."""
    seed = 1
    rng = np.random.Generator(np.random.PCG64(seed))
    q, w = _q_and_w(rng, 1, 64, D_QK if kv_format == 0 else D_LATENT)
    pos = int(rng.integers(0, 4096))
    idx = np.empty((1, 640), dtype=np.int64)
    idx[0, :128] = _swa_ring_cols(pos, 0, 8192)
    idx[0, 128:] = rng.choice(65536, size=512, replace=False)
    return _finish("decode_sq1_h64_topk640" + ("_nvfp4" if kv_format else ""), rng, seed, q, w, 8192, 65536, idx,
                   np.array([640]), np.array([pos]), 128, kv_format=kv_format, cmp_scale=NVFP4_CMP_SCALE if kv_format else 1.0)


def config_decode64(kv_format: int = 0) -> Workload:
    """Batched decode: 64 tokens, positions in [0, 32768), each with its own 128-row
    SWA ring in a 64x128-row pool and 512 compressed rows distinct from 262144 (seed 2)."""
    seed = 2
    rng = np.random.Generator(np.random.PCG64(seed))
    s_q = 64
    q, w = _q_and_w(rng, s_q, 64, D_QK if kv_format == 0 else D_LATENT)
    pos = rng.integers(0, 32768, size=s_q)
    idx = np.empty((s_q, 640), dtype=np.int64)
    for t in range(s_q):
        idx[t, :128] = _swa_ring_cols(int(pos[t]), t * 128, 128)
        idx[t, 128:] = rng.choice(262144, size=512, replace=False)
    return _finish("decode_sq64_h64_topk640" + ("_nvfp4" if kv_format else ""), rng, seed, q, w, s_q * 128, 262144,
                   idx, np.full(s_q, 640), pos, 128, kv_format=kv_format, cmp_scale=NVFP4_CMP_SCALE if kv_format else 1.0)


def config_decode1024(kv_format: int = 0) -> Workload:
    """Large decode: 1024 tokens, topk_length uniform in [64, 640] with the row tail
    set to -1, each token's 128 SWA columns a random order of its own 128-row ring
    (pool 1024x128 rows), 512 compressed rows distinct from 1,048,576 (seed 3).
    Positions (not fixed by the workload description) are uniform in [0, 32768)."""
    seed = 3
    rng = np.random.Generator(np.random.PCG64(seed))
    s_q = 1024
    q, w = _q_and_w(rng, s_q, 64, D_QK if kv_format == 0 else D_LATENT)
    pos = rng.integers(0, 32768, size=s_q)
    tl = rng.integers(64, 641, size=s_q)
    idx = np.empty((s_q, 640), dtype=np.int64)
    for t in range(s_q):
        idx[t, :128] = t * 128 + rng.permutation(128)
        idx[t, 128:] = rng.choice(1 << 20, size=512, replace=False)
        idx[t, tl[t]:] = -1
    return _finish("decode_sq1024_h64_topk640_ragged" + ("_nvfp4" if kv_format else ""), rng, seed, q, w, s_q * 128,
                   1 << 20, idx, tl, pos, 128, kv_format=kv_format, cmp_scale=NVFP4_CMP_SCALE if kv_format else 1.0)


def config_prefill2123(kv_format: int = 0) -> Workload:
    """Prefill chunk: positions 0..2122 of one sequence; SWA columns are the causal
    window p-127..p (-1 before the sequence start) into a position-indexed pool;
    compressed columns are min(p+1, 512) distinct rows r <= p of a 2048-row pool,
    the remaining columns -1; topk_length = 640 (seed 4)."""
    seed = 4
    rng = np.random.Generator(np.random.PCG64(seed))
    s_q = 2123
    q, w = _q_and_w(rng, s_q, 64, D_QK if kv_format == 0 else D_LATENT)
    pos = np.arange(s_q)
    idx = np.full((s_q, 640), -1, dtype=np.int64)
    for t in range(s_q):
        p = int(pos[t])
        idx[t, :128] = _swa_ring_cols(p, 0, 1 << 30)   # no wrap: pool rows are positions
        n = min(p + 1, 512)
        idx[t, 128:128 + n] = rng.choice(min(p + 1, 2048), size=n, replace=False)
    return _finish("prefill_sq2123_h64_topk640" + ("_nvfp4" if kv_format else ""), rng, seed, q, w, s_q, 2048, idx,
                   np.full(s_q, 640), pos, 128, kv_format=kv_format, cmp_scale=NVFP4_CMP_SCALE if kv_format else 1.0)


CONFIGS = {
    "tiny": config_tiny,
    "decode1": config_decode1,
    "decode64": config_decode64,
    "decode1024": config_decode1024,
    "prefill2123": config_prefill2123,
}
# the same shapes, index patterns and seeds on the nvfp4_ds_mla (V4.1) cache, and with
# an E4M3 q (the same inputs; only the kernel's flag and the oracle's reading differ)
_BASE = dict(CONFIGS)
CONFIGS.update({k + "_nvfp4": (lambda f: (lambda: f(kv_format=1)))(f) for k, f in _BASE.items()})


def _with_fp8_q(f):
    def make_it():
        w = f()
        w.fp8_q = True
        w.name += "_fp8q"
        return w
    return make_it


CONFIGS.update({k + "_fp8q": _with_fp8_q(f) for k, f in _BASE.items()})


def make(name: str) -> Workload:
    return CONFIGS[name]()


def n_valid_rows(w: Workload) -> np.ndarray:
    """Valid (in-length, non-negative) index columns per token."""
    cols = np.arange(w.topk)[None, :]
    live = (cols < w.topk_length[:, None]) & (w.indices >= 0)
    return live.sum(axis=1)
