"""KV-cache insert: new tokens' KV rows normalised, roped and quantised into fp8_ds_mla
rows of a cache pool (oracle; test infrastructure only).

The pages: "[Perf] DeepSeek-V4.1-Flash latency_specialized decode at TP4" (vLLM PR
#64364), the table "The changes and what each bought", Attention row: the KV cache write
moves into the Q/KV norm-quant kernel; its Limitations section names the norm's KV write
(test_fused_q_kv_rmsnorm).  The pages give no formula.  The reading taken (each point is
one an MLA KV projection fixes, written out here):

1. The new token's KV vector is 576 bf16 values: 512 latent dims, then 64 rotary dims.
2. The latent part is RMS-normalised over its 512 dims with its own 512-long weight:
   y = x / sqrt(mean(x^2) + eps) * w (the rotary part is not normalised).
3. The rotary part is rotated by the token's position, interleaved pairs, the same
   convention as the query's (oracle.sparse_mla.rope_interleaved): the cache stores
   keys already rotated, which is what the attention reads.
4. The latent part is quantised per 128-dim block as the cache format stores it: fp32
   scale = max|y| / 448 (1 for an all-zero block), E4M3 codes of y / scale (round to
   nearest even).  The code is an integer decided by floating point, so it is decided in
   the precision the kernel uses: y / scale equals (x*w) * (448 / max|x*w|) exactly (the
   RMS factor cancels), taken in binary32 as one rounded quotient 448 / max|x*w| per block
   and one rounded product per value (x*w is exact: two 8-bit significands), then rounded
   to E4M3.
5. The rotary part is stored as bf16 (round to nearest even); the row is 512 codes, 4
   little-endian fp32 scales and 64 bf16 values (656 bytes).
6. slots[i] < 0 skips token i (a padding token); every other row of the pool is left as
   it was.
"""

from __future__ import annotations

import numpy as np

from . import codecs
from .sparse_mla import D_LATENT, D_ROPE, ROW_BYTES, SCALE_GROUP, rope_interleaved

E4M3_MAX = 448.0


def normalised_latent(x_bits: np.ndarray, w_bits: np.ndarray, eps: float) -> np.ndarray:
    """Step 2 in float64: bf16 latent [n, 512], bf16 weight [512] -> y [n, 512]."""
    x = codecs.bf16_decode(x_bits)
    w = codecs.bf16_decode(w_bits)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * w


def quantise_latent(x_bits: np.ndarray, w_bits: np.ndarray, eps: float):
    """Step 4: (codes uint8 [n, 512], scales float64 [n, 4]) of the normalised latent.

    The scales are float64 values of max|y| / 448; the codes follow point 4 of the module
    docstring ((x*w) * (448 / max|x*w|), one binary32 quotient per block, one binary32
    product per value).
    """
    y = normalised_latent(x_bits, w_bits, eps)
    n = y.shape[0]
    xw = (codecs.bf16_decode(x_bits) * codecs.bf16_decode(w_bits)).astype(np.float32)   # exact
    codes = np.zeros((n, D_LATENT), dtype=np.uint8)
    scales = np.ones((n, D_LATENT // SCALE_GROUP), dtype=np.float64)
    for b in range(D_LATENT // SCALE_GROUP):
        blk = slice(SCALE_GROUP * b, SCALE_GROUP * (b + 1))
        m = np.max(np.abs(xw[:, blk]), axis=1, keepdims=True)                             # binary32, exact
        amax_y = np.max(np.abs(y[:, blk]), axis=1)
        nz = m[:, 0] > 0
        scales[nz, b] = amax_y[nz] / E4M3_MAX
        with np.errstate(invalid="ignore", divide="ignore"):
            r = np.float32(E4M3_MAX) / np.where(m > 0, m, np.float32(1))                      # binary32 quotient
        ratio = xw[:, blk] * r                                                                # binary32 product
        ratio = np.where(m > 0, ratio, np.float32(0)).astype(np.float64)
        codes[:, blk] = codecs.e4m3_encode(ratio)
    return codes, scales


def rotated_rope(r_bits: np.ndarray, positions: np.ndarray, base: float) -> np.ndarray:
    """Step 3 in float64 and step 5's bf16 rounding: bf16 bits [n, 64] -> bf16 bits [n, 64]."""
    r = codecs.bf16_decode(r_bits)
    out = np.empty_like(r)
    for i in range(r.shape[0]):
        out[i] = rope_interleaved(r[i], float(positions[i]), base)
    return codecs.bf16_encode(out)


def kv_insert(pool: np.ndarray, kv_bits: np.ndarray, positions: np.ndarray, slots: np.ndarray,
              kv_norm_w_bits: np.ndarray, eps: float = 1e-6, base: float = 10000.0) -> np.ndarray:
    """Steps 1-6: a copy of `pool` (uint8 [n_rows, 656]) with the new tokens' rows written.

    kv_bits uint16 [n, 576] (bf16: 512 latent, 64 rotary), positions int [n], slots int
    [n] (row of the pool, < 0 = skip), kv_norm_w_bits uint16 [512].  A slot at or past the
    pool's end raises (the kernel's unchecked case is undefined).
    """
    kv_bits = np.asarray(kv_bits, dtype=np.uint16)
    pool = np.array(pool, dtype=np.uint8, copy=True)
    assert pool.ndim == 2 and pool.shape[1] == ROW_BYTES
    codes, scales = quantise_latent(kv_bits[:, :D_LATENT], np.asarray(kv_norm_w_bits, dtype=np.uint16), eps)
    rope = rotated_rope(kv_bits[:, D_LATENT:D_LATENT + D_ROPE], positions, base)
    for i, s in enumerate(np.asarray(slots, dtype=np.int64)):
        if s < 0:
            continue
        if s >= pool.shape[0]:
            raise IndexError(f"slot {s} out of range for a pool of {pool.shape[0]} rows (token {i})")
        row = np.empty(ROW_BYTES, dtype=np.uint8)
        row[:D_LATENT] = codes[i]
        row[D_LATENT:D_LATENT + 16] = scales[i].astype("<f4").view(np.uint8)
        row[D_LATENT + 16:] = rope[i].astype("<u2").view(np.uint8)
        pool[s] = row
    return pool
