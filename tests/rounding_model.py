"""A numpy model of the operand roundings of the fused kernel's two contractions, used to
check on the CPU that the chosen operand precision can meet the parity bar and that a
single-fp16 design cannot (test infrastructure: it models roundings, it is not the CUDA
path and shares nothing with it).

Two designs are modelled per (token, head), both with exact float64 sums (the tensor
core's fp32 accumulation is not modelled; its error is far below the operand roundings
compared here):

- "single": q~ = fp16 of q * w (roped), each latent value fp16(fp16(code) * fp16(scale)),
  P = fp16 of the softmax numerators, and the row sum over the fp16 P.  This is the
  plain fp16 tensor-core design.
- "fp8q": the split design with the latent part of q~ quantised to E4M3 (one scale per
  head, its largest magnitude mapped to 448), the operand an FP8 x FP8 QK^T would take.
- "split": the fused kernel's design.  q~ = hi + lo (two fp16 parts of the fp32 value,
  after a per-head power-of-two prescale); the E4M3 codes enter unscaled (exact in fp16)
  and each 128-dim block's fp32 scale multiplies that block's partial score; PV takes,
  per output block b, P_b = P * scale_b / ref_b as hi + lo fp16 (ref_b a power of two,
  the largest scale of the block over the rows) and multiplies the block by ref_b; the
  row sum is over the unrounded P.

The definition each design approximates is the oracle's (oracle/sparse_mla.py): the
query norm, RoPE, softmax and PV of "Deepseek V41 Attention MegaKernel" (vLLM PR #56344),
Purpose.
"""

from __future__ import annotations

import numpy as np

from oracle import codecs
from oracle.sparse_mla import (D_LATENT, OUT_ROPE_START, SCALE_GROUP, gather_rows, q_prologue, rope_interleaved,
                               valid_columns)


def f16(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


def hi_lo(x) -> np.ndarray:
    """x as the sum of two fp16 parts (the part lost is below 2^-22 of x)."""
    hi = f16(x)
    return hi + f16(np.asarray(x, dtype=np.float64) - hi)


def _rows(rows: np.ndarray):
    n = rows.shape[0]
    codes = codecs.e4m3_decode(rows[:, :D_LATENT])
    scales = codecs.fp32_decode_le(rows[:, D_LATENT:D_LATENT + 16]).reshape(n, D_LATENT // SCALE_GROUP)
    rope = codecs.bf16_decode(np.ascontiguousarray(rows[:, D_LATENT + 16:]).view("<u2"))
    return codes, scales, rope


def token_output(design: str, q_bits, norm_w_bits, index_row, topk_length, pos, kv_swa, kv_cmp, p) -> np.ndarray:
    """Pre-cast output [h, 512] of one token under `design` ("single", "split" or "fp8q")."""
    x = codecs.bf16_decode(q_bits)
    h = x.shape[0]
    cols = valid_columns(index_row, topk_length)
    if len(cols) == 0:
        return np.zeros((h, D_LATENT))
    codes, scales, rope = _rows(gather_rows(index_row, cols, kv_swa, kv_cmp, p.n_swa_cols))
    # q~ without the RMS factor (the factor multiplies the scores), roped
    inv_rms = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + p.rms_eps)
    qt = q_prologue(q_bits, norm_w_bits, pos, p) / inv_rms
    if design == "single":
        k_lat = f16(codes * np.repeat(f16(scales), SCALE_GROUP, axis=1))
        s = f16(qt[:, :D_LATENT]) @ k_lat.T + f16(qt[:, D_LATENT:]) @ f16(rope).T
    else:
        # the prescale puts the head's largest |q * w| (before RoPE) into [2^13, 2^14)
        amax = np.max(np.abs(x * codecs.bf16_decode(norm_w_bits)), axis=1, keepdims=True)
        k2 = np.where(amax > 0, 13.0 - np.floor(np.log2(np.where(amax > 0, amax, 1.0))), 0.0)
        qs = hi_lo(qt * np.exp2(k2)) * np.exp2(-k2)
        if design == "fp8q":
            # the latent part of q~ as E4M3 with a per-head scale (max |q~| maps to 448)
            lat = qt[:, :D_LATENT]
            qsc = np.max(np.abs(lat), axis=1, keepdims=True) / 448.0
            qsc = np.where(qsc > 0, qsc, 1.0)
            qs = qs.copy()
            qs[:, :D_LATENT] = codecs.e4m3_decode(codecs.e4m3_encode(lat / qsc)) * qsc
        s = qs[:, D_LATENT:] @ f16(rope).T
        for b in range(D_LATENT // SCALE_GROUP):
            blk = slice(SCALE_GROUP * b, SCALE_GROUP * (b + 1))
            s = s + (qs[:, blk] @ codes[:, blk].T) * scales[None, :, b]
    s = s * inv_rms * p.softmax_scale
    e = np.exp(s - s.max(axis=1, keepdims=True))
    if design == "single":
        pe = f16(e)
        o = (pe @ f16(codes * np.repeat(f16(scales), SCALE_GROUP, axis=1))) / pe.sum(axis=1, keepdims=True)
    else:
        o = np.empty((h, D_LATENT))
        for b in range(D_LATENT // SCALE_GROUP):
            blk = slice(SCALE_GROUP * b, SCALE_GROUP * (b + 1))
            ref = np.exp2(np.floor(np.log2(np.max(np.abs(scales[:, b])))))
            pb = hi_lo(e * (scales[None, :, b] / ref))
            o[:, blk] = (pb @ codes[:, blk]) * ref
        o = o / e.sum(axis=1, keepdims=True)
    o[:, OUT_ROPE_START:] = rope_interleaved(o[:, OUT_ROPE_START:], pos, p.rope_base, inverse=True)
    return o
