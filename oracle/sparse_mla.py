"""Float64 definition of fused top-k sparse latent attention (oracle; test infrastructure only).

What is computed, per query token t and head h.  The stages are the ones the Purpose
section of "Deepseek V41 Attention MegaKernel" (vLLM PR #56344) lists as fused: the
query norm, RoPE, sparse attention, inverse RoPE and an FP8 cast of the output.

1. q RMSNorm over all 576 dims of the head, times a shared 576-long weight.
2. q RoPE on the last 64 dims (interleaved pairs, theta_i = base^(-2i/64), angle
   positions[t] * theta_i).  The pages give only the base (10000); the pair layout is
   a reading.
3. Valid columns: j < topk_length[t] with indices[t, j] >= 0 (the page's sentinel fix:
   sparse reads are capped at topk_length and -1 entries are never read).  Columns
   [0, n_swa_cols) index the sliding-window cache, the rest the compressed cache
   (one combined index row per token, as combine_topk_swa_indices produces).
4. Each referenced cache row is an fp8_ds_mla row: 512 E4M3 latent values, four
   fp32 scales (one per 128 latent values), 64 bf16 rope values.  k = dequantised
   latent ++ rope (576); v = dequantised latent (512).
5. s_j = softmax_scale * q~ . k_j; p = softmax over the valid columns; o = sum p_j v_j;
   lse = log sum exp s_j.  No valid column: o = 0, lse = -inf.
6. Inverse RoPE (angle -positions[t] * theta_i) on the last 64 output dims (448..511).
7. MXFP8 cast of o along the 512 dims: 32-element blocks, UE8M0 scales (see codecs).

The math is exact up to rounding, so the oracle is that definition written out: a loop
over tokens with one dense softmax per token in float64.  No blocking, no online
softmax, no split.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import codecs

D_LATENT = 512
D_ROPE = 64
D_QK = D_LATENT + D_ROPE          # 576
D_V = D_LATENT                     # 512
SCALE_GROUP = 128                  # latent values per fp32 scale
ROW_BYTES = D_LATENT + 4 * (D_LATENT // SCALE_GROUP) + 2 * D_ROPE   # 656
OUT_ROPE_START = D_V - D_ROPE      # 448: inverse RoPE acts on output dims 448..511
MX_BLOCK = 32


@dataclass(frozen=True)
class OracleParams:
    n_swa_cols: int
    softmax_scale: float = 1.0 / np.sqrt(D_QK)
    rope_base: float = 10000.0
    rms_eps: float = 1e-6
    fp8_q: bool = False       # E4M3 latent q (quantize_q_latent)


def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * w along the last axis (float64).

    Step 1, the query norm of "Deepseek V41 Attention MegaKernel" (vLLM PR #56344), Purpose;
    its span (all 576 dims) and eps are a reading, the pages fix neither.
    """
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(w, dtype=np.float64)


def rope_interleaved(x: np.ndarray, pos: float, base: float, inverse: bool = False) -> np.ndarray:
    """Rotate consecutive pairs (2i, 2i+1) of the last axis by pos * base^(-2i/n).

    Steps 2 and 6, RoPE and inverse RoPE of "Deepseek V41 Attention MegaKernel" (vLLM PR
    #56344), Purpose; the pair layout is a reading, the pages give only the base.
    """
    x = np.asarray(x, dtype=np.float64)
    n = x.shape[-1]
    i = np.arange(n // 2, dtype=np.float64)
    theta = np.power(float(base), -2.0 * i / n)
    ang = float(pos) * theta
    if inverse:
        ang = -ang
    c, s = np.cos(ang), np.sin(ang)
    x0 = x[..., 0::2]
    x1 = x[..., 1::2]
    y = np.empty_like(x)
    y[..., 0::2] = x0 * c - x1 * s
    y[..., 1::2] = x0 * s + x1 * c
    return y


def quantize_q_latent(q_bits: np.ndarray, norm_w_bits: np.ndarray):
    """E4M3 codes of q's latent part, per head: (codes uint8 [h, 512], amax float32 [h]).

    The query FP8 quantisation named on "DSV4.1 latency_specialized decode at TP4 on
    GB300" (vLLM PR #64364, "The changes and what each bought", Attention row); the page
    gives no rule, the reading taken: per token and head, amax = max |q * w| over the 512
    latent dims and code = E4M3(fl(q * w) * fl(448 / amax)), ties to even, saturating,
    each step in binary32.  The RMSNorm'd latent is then code * amax * rms_inv / 448
    (the RMS factor cancels in the code).  An all-zero latent gives codes 0.
    """
    x = codecs.bf16_decode(q_bits[..., :D_LATENT]).astype(np.float32)
    w = codecs.bf16_decode(norm_w_bits[:D_LATENT]).astype(np.float32)
    xw = x * w                                          # exact in binary32
    amax = np.max(np.abs(xw), axis=-1)
    safe = np.where(amax > 0, amax, np.float32(1.0))
    rq = np.where(amax > 0, np.float32(448.0) / safe, np.float32(0.0)).astype(np.float32)
    y = (xw * rq[..., None]).astype(np.float32)
    return codecs.e4m3_encode(y.astype(np.float64)), amax


def q_prologue(q_bits: np.ndarray, norm_w_bits: np.ndarray, pos: int, p: OracleParams) -> np.ndarray:
    """Steps 1-2 for one token: bf16 q [h, 576] -> normalised, rotated q~ [h, 576].  With
    p.fp8_q the latent dims are replaced by their E4M3 values (quantize_q_latent) times
    the head's scale amax * rms_inv / 448.

    Steps 1-2 of "Deepseek V41 Attention MegaKernel" (vLLM PR #56344), Purpose.
    """
    x = codecs.bf16_decode(q_bits)
    w = codecs.bf16_decode(norm_w_bits)
    xn = rmsnorm(x, w, p.rms_eps)
    if p.fp8_q:
        codes, amax = quantize_q_latent(q_bits, norm_w_bits)
        rms_inv = 1.0 / np.sqrt(np.mean(x * x, axis=-1) + p.rms_eps)
        xn[..., :D_LATENT] = codecs.e4m3_decode(codes) * (amax.astype(np.float64) * rms_inv / 448.0)[..., None]
    xn[..., D_LATENT:] = rope_interleaved(xn[..., D_LATENT:], pos, p.rope_base)
    return xn


def decode_kv_rows(rows: np.ndarray) -> np.ndarray:
    """fp8_ds_mla rows uint8 [n, 656] -> float64 k [n, 576] (v is k[:, :512]).

    Step 4: the fp8_ds_mla cache that "Deepseek V41 Attention MegaKernel" (vLLM PR #56344),
    Purpose and its Performance section name; the byte layout is a reading, the pages give
    none.
    """
    rows = np.asarray(rows, dtype=np.uint8)
    assert rows.ndim == 2 and rows.shape[1] == ROW_BYTES
    n = rows.shape[0]
    lat = codecs.e4m3_decode(rows[:, :D_LATENT])
    scales = codecs.fp32_decode_le(rows[:, D_LATENT:D_LATENT + 16]).reshape(n, D_LATENT // SCALE_GROUP)
    lat = lat * np.repeat(scales, SCALE_GROUP, axis=1)
    rope_bits = np.ascontiguousarray(rows[:, D_LATENT + 16:]).view("<u2")
    rope = codecs.bf16_decode(rope_bits)
    return np.concatenate([lat, rope], axis=1)


def valid_columns(index_row: np.ndarray, topk_length: int) -> np.ndarray:
    """Columns j < topk_length with a non-negative index (step 3).

    Step 3: the sentinel and topk_length rule of the bug-fix bullet of "Deepseek V41
    Attention MegaKernel" (vLLM PR #56344), Purpose.
    """
    topk = index_row.shape[0]
    n = max(0, min(int(topk_length), topk))
    cols = np.arange(n)
    return cols[np.asarray(index_row[:n]) >= 0]


def gather_rows(index_row, cols, kv_swa, kv_cmp, n_swa_cols):
    """Fetch the cache row of every valid column, choosing the cache by column.

    Step 3: one combined index row per token (SWA columns first), as the
    combine_topk_swa_indices bullet of "Deepseek V41 Attention MegaKernel" (vLLM PR #56344),
    Purpose describes.
    """
    out = np.empty((len(cols), ROW_BYTES), dtype=np.uint8)
    for k, j in enumerate(cols):
        idx = int(index_row[j])
        pool = kv_swa if j < n_swa_cols else kv_cmp
        if idx >= pool.shape[0]:
            raise IndexError(f"index {idx} out of range for a pool of {pool.shape[0]} rows (column {j})")
        out[k] = pool[idx]
    return out


def mxfp8_cast(o: np.ndarray):
    """Step 7: (E4M3 codes, UE8M0 codes) along the last axis in 32-element blocks.

    Step 7: the FP8 cast of "Deepseek V41 Attention MegaKernel" (vLLM PR #56344), Purpose,
    in the MXFP8 form of "[DSV4.1] Combine DSpark decode and prefill kernel optimizations"
    (SGLang PR #39370), first description block (the UE8M0 rule is the OCP MX one, a
    reading).
    """
    return codecs.mxfp8_quantize(o, MX_BLOCK)


def sparse_mla_forward(q, kv_swa, kv_cmp, indices, topk_length, positions, norm_w, p: OracleParams):
    """The whole path for every token.

    Arguments (numpy):
      q            uint16 bf16 bits [s_q, h_q, 576]
      kv_swa       uint8 [n_swa_rows, 656]
      kv_cmp       uint8 [n_cmp_rows, 656]
      indices      int32 [s_q, topk]
      topk_length  int32 [s_q]
      positions    int32 [s_q]
      norm_w       uint16 bf16 bits [576]
    Returns dict with
      out          float64 [s_q, h_q, 512]   pre-cast output (after inverse RoPE)
      lse          float64 [s_q, h_q]
      out_fp8      uint8 [s_q, h_q, 512]     E4M3 codes
      out_sf       uint8 [s_q, h_q, 16]      UE8M0 codes
      n_valid      int64 [s_q]

    Steps 1-7 of "Deepseek V41 Attention MegaKernel" (vLLM PR #56344), Purpose.
    """
    q = np.asarray(q)
    s_q, h_q, dq = q.shape
    assert dq == D_QK
    out = np.zeros((s_q, h_q, D_V), dtype=np.float64)
    lse = np.full((s_q, h_q), -np.inf, dtype=np.float64)
    n_valid = np.zeros(s_q, dtype=np.int64)
    for t in range(s_q):
        qt = q_prologue(q[t], norm_w, int(positions[t]), p)
        cols = valid_columns(indices[t], int(topk_length[t]))
        n_valid[t] = len(cols)
        if len(cols) == 0:
            continue
        k = decode_kv_rows(gather_rows(indices[t], cols, kv_swa, kv_cmp, p.n_swa_cols))
        v = k[:, :D_V]
        s = p.softmax_scale * (qt @ k.T)                    # [h, n]
        m = np.max(s, axis=1, keepdims=True)
        e = np.exp(s - m)
        l = np.sum(e, axis=1, keepdims=True)
        o = (e @ v) / l
        lse[t] = (m + np.log(l))[:, 0]
        o[:, OUT_ROPE_START:] = rope_interleaved(o[:, OUT_ROPE_START:], int(positions[t]), p.rope_base, inverse=True)
        out[t] = o
    out_fp8, out_sf = mxfp8_cast(out)
    return {"out": out, "lse": lse, "out_fp8": out_fp8, "out_sf": out_sf, "n_valid": n_valid}
