"""Scalar pure-Python restatement of the path, for tiny inputs (oracle cross-check).

It re-derives every step with Python floats and loops -- its own format decoders
(struct / math.ldexp), its own RMSNorm, RoPE, softmax and accumulation -- so that a
mistake in the vectorised oracle (a transposed operand, a wrong pair layout, a dropped
scale) shows up as a disagreement.  It covers the float output and the LSE; the MXFP8
cast is pinned separately against closed forms.
"""

from __future__ import annotations

import math
import struct

D_LATENT, D_ROPE, ROW_BYTES = 512, 64, 656


def _e4m3(byte: int) -> float:
    sign = -1.0 if byte & 0x80 else 1.0
    e = (byte >> 3) & 15
    m = byte & 7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return sign * math.ldexp(m, -9)          # m/8 * 2^-6
    return sign * math.ldexp(8 + m, e - 10)      # (1 + m/8) * 2^(e-7)


def _bf16(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (bits & 0xFFFF) << 16))[0]


def _row_to_k(row: bytes) -> list:
    scales = struct.unpack("<4f", bytes(row[512:528]))
    k = [_e4m3(row[i]) * scales[i // 128] for i in range(512)]
    for i in range(64):
        lo, hi = row[528 + 2 * i], row[529 + 2 * i]
        k.append(_bf16(lo | (hi << 8)))
    return k


def _rotate(vec: list, start: int, pos: int, base: float, sign: float) -> None:
    for i in range(32):
        theta = base ** (-(2.0 * i) / 64.0)
        a = sign * pos * theta
        c, s = math.cos(a), math.sin(a)
        x0, x1 = vec[start + 2 * i], vec[start + 2 * i + 1]
        vec[start + 2 * i] = x0 * c - x1 * s
        vec[start + 2 * i + 1] = x0 * s + x1 * c


def forward(q, kv_swa, kv_cmp, indices, topk_length, positions, norm_w, n_swa_cols,
            softmax_scale=1.0 / 24.0, rope_base=10000.0, rms_eps=1e-6):
    """Nested lists in, nested lists out: (out [s][h][512], lse [s][h])."""
    s_q, h_q = len(q), len(q[0])
    w = [_bf16(int(b)) for b in norm_w]
    outs, lses = [], []
    for t in range(s_q):
        ks = []
        L = min(max(int(topk_length[t]), 0), len(indices[t]))
        for j in range(L):
            idx = int(indices[t][j])
            if idx < 0:
                continue
            pool = kv_swa if j < n_swa_cols else kv_cmp
            ks.append(_row_to_k(bytes(bytearray(int(b) for b in pool[idx]))))
        out_t, lse_t = [], []
        for h in range(h_q):
            x = [_bf16(int(b)) for b in q[t][h]]
            ms = sum(v * v for v in x) / len(x)
            r = 1.0 / math.sqrt(ms + rms_eps)
            x = [x[i] * r * w[i] for i in range(len(x))]
            _rotate(x, 512, int(positions[t]), rope_base, +1.0)
            if not ks:
                out_t.append([0.0] * 512)
                lse_t.append(float("-inf"))
                continue
            sc = [softmax_scale * sum(x[i] * k[i] for i in range(576)) for k in ks]
            mx = max(sc)
            ex = [math.exp(v - mx) for v in sc]
            tot = sum(ex)
            o = [sum(ex[j] * ks[j][d] for j in range(len(ks))) / tot for d in range(512)]
            _rotate(o, 448, int(positions[t]), rope_base, -1.0)
            out_t.append(o)
            lse_t.append(mx + math.log(tot))
        outs.append(out_t)
        lses.append(lse_t)
    return outs, lses
