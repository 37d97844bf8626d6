"""Float64 definition of the sparse attention on the nvfp4_ds_mla (V4.1) cache (oracle;
test infrastructure only).

"Deepseek V41 Attention MegaKernel" (vLLM PR #56344), Purpose, adds the nvfp4_ds_mla KV
cache, "V4.1 fp8 528 B SWA + V4.1 fp4 288 B compressed", and gives no byte layout.
The reading taken here:

* The sizes only fit 512-dim keys whose 64 rotary dims are part of the 512 (528 =
  512 one-byte values + four fp32 scales; 288 = 512 four-bit values + 32 one-byte
  scales), and then v = k.  The fused kernel's inverse RoPE on output dims 448..511
  (same Purpose section) fits this: the output's last 64 dims are the keys' rotary
  dims.  So the rotary dims are 448..511, stored already rotated.
* Sliding-window row, 528 bytes: 512 E4M3 values | 4 little-endian fp32 scales, scale
  g for dims [128g, 128g + 128) (the fp8_ds_mla scale rule on 512 dims).
* Compressed row, 288 bytes, NVFP4: 512 E2M1 values, two per byte with dim 2i in the
  low nibble of byte i | 32 E4M3 scales, scale i for dims [16i, 16i + 16); every value
  also times one fp32 scale of the pool (cmp_scale).
* E2M1 (OCP MX FP4): 1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit;
  exponent 0 is subnormal (m * 0.5); magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.

What is computed per token t and head h, the fp8_ds_mla path's steps with d = 512:
q~ = RMSNorm over the 512 dims of q times norm_w (512); RoPE on q~ dims 448..511;
valid columns and pool choice as there; s_j = softmax_scale * q~ . k_j; o = softmax
weighted sum of v_j = k_j; inverse RoPE on o dims 448..511; MXFP8 cast.
"""

from __future__ import annotations

import numpy as np

from . import codecs
from .sparse_mla import OracleParams, mxfp8_cast, rmsnorm, rope_interleaved, valid_columns

D = 512
ROPE_START = 448
SWA_ROW_BYTES = 528
CMP_ROW_BYTES = 288
FP4_GROUP = 16
FP8_GROUP = 128


def e2m1_decode(nibbles) -> np.ndarray:
    """E2M1 codes (0..15) to float64, from the format's fields."""
    n = np.asarray(nibbles, dtype=np.int64) & 0xF
    sign = np.where(n & 8, -1.0, 1.0)
    e = (n >> 1) & 3
    m = n & 1
    mag = np.where(e == 0, 0.5 * m, np.ldexp(1.0 + 0.5 * m, e - 1))
    return sign * mag


def decode_swa_rows(rows: np.ndarray) -> np.ndarray:
    """nvfp4_ds_mla sliding-window rows uint8 [n, 528] -> float64 keys [n, 512]."""
    rows = np.asarray(rows, dtype=np.uint8)
    assert rows.ndim == 2 and rows.shape[1] == SWA_ROW_BYTES
    n = rows.shape[0]
    vals = codecs.e4m3_decode(rows[:, :D])
    scales = codecs.fp32_decode_le(rows[:, D:D + 16]).reshape(n, D // FP8_GROUP)
    return vals * np.repeat(scales, FP8_GROUP, axis=1)


def decode_cmp_rows(rows: np.ndarray, cmp_scale: float) -> np.ndarray:
    """nvfp4_ds_mla compressed rows uint8 [n, 288] -> float64 keys [n, 512]."""
    rows = np.asarray(rows, dtype=np.uint8)
    assert rows.ndim == 2 and rows.shape[1] == CMP_ROW_BYTES
    packed = rows[:, :D // 2].astype(np.int64)
    nib = np.empty((rows.shape[0], D), dtype=np.int64)
    nib[:, 0::2] = packed & 0xF        # dim 2i: low nibble of byte i
    nib[:, 1::2] = packed >> 4
    scales = codecs.e4m3_decode(rows[:, D // 2:])
    return e2m1_decode(nib) * np.repeat(scales, FP4_GROUP, axis=1) * float(cmp_scale)


def q_prologue(q_bits: np.ndarray, norm_w_bits: np.ndarray, pos: int, p: OracleParams) -> np.ndarray:
    """bf16 q [h, 512] -> normalised q~ with RoPE on dims 448..511."""
    xn = rmsnorm(codecs.bf16_decode(q_bits), codecs.bf16_decode(norm_w_bits), p.rms_eps)
    xn[..., ROPE_START:] = rope_interleaved(xn[..., ROPE_START:], pos, p.rope_base)
    return xn


def gather_keys(index_row, cols, kv_swa, kv_cmp, n_swa_cols, cmp_scale) -> np.ndarray:
    """The decoded key of every valid column, the pool chosen by column."""
    out = np.empty((len(cols), D), dtype=np.float64)
    for k, j in enumerate(cols):
        idx = int(index_row[j])
        swa = j < n_swa_cols
        pool = kv_swa if swa else kv_cmp
        if idx >= pool.shape[0]:
            raise IndexError(f"index {idx} out of range for a pool of {pool.shape[0]} rows (column {j})")
        row = pool[idx:idx + 1]
        out[k] = decode_swa_rows(row)[0] if swa else decode_cmp_rows(row, cmp_scale)[0]
    return out


def sparse_mla_forward(q, kv_swa, kv_cmp, indices, topk_length, positions, norm_w, p: OracleParams,
                       cmp_scale: float = 1.0):
    """The whole path on the nvfp4_ds_mla cache; q uint16 bf16 bits [s_q, h_q, 512],
    norm_w [512], kv_swa uint8 [n, 528], kv_cmp uint8 [n, 288].  Returns the dict of
    oracle.sparse_mla.sparse_mla_forward."""
    q = np.asarray(q)
    s_q, h_q, dq = q.shape
    assert dq == D
    out = np.zeros((s_q, h_q, D), dtype=np.float64)
    lse = np.full((s_q, h_q), -np.inf, dtype=np.float64)
    n_valid = np.zeros(s_q, dtype=np.int64)
    for t in range(s_q):
        qt = q_prologue(q[t], norm_w, int(positions[t]), p)
        cols = valid_columns(indices[t], int(topk_length[t]))
        n_valid[t] = len(cols)
        if len(cols) == 0:
            continue
        k = gather_keys(indices[t], cols, kv_swa, kv_cmp, p.n_swa_cols, cmp_scale)
        s = p.softmax_scale * (qt @ k.T)                    # [h, n]
        m = np.max(s, axis=1, keepdims=True)
        e = np.exp(s - m)
        l = np.sum(e, axis=1, keepdims=True)
        o = (e @ k) / l                                     # v = k
        lse[t] = (m + np.log(l))[:, 0]
        o[:, ROPE_START:] = rope_interleaved(o[:, ROPE_START:], int(positions[t]), p.rope_base, inverse=True)
        out[t] = o
    out_fp8, out_sf = mxfp8_cast(out)
    return {"out": out, "lse": lse, "out_fp8": out_fp8, "out_sf": out_sf, "n_valid": n_valid}
