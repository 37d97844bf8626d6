"""Pins of the KV-insert oracle (oracle/kv_insert.py): a hand-worked row, closed forms of
the quantiser, invariances, and the byte layout the attention's reader decodes."""

import numpy as np
import pytest

from oracle import codecs
from oracle.kv_insert import kv_insert, quantise_latent
from oracle.sparse_mla import ROW_BYTES, decode_kv_rows, rope_interleaved

EPS = 1e-6


def _bits(x):
    return codecs.bf16_encode(np.asarray(x, dtype=np.float64))


def _rand_kv(rng, n, scale=1.0):
    return _bits(rng.standard_normal((n, 576)) * scale)


def _w(rng):
    return _bits(1.0 + 0.1 * rng.standard_normal(512))


def test_hand_worked_row():
    # latent block 0 = (2, -1, 0.5, 0, ...), every other latent value 0, weight 1, rope
    # (1, 0) pairs at position 0.  mean(x^2) = 5.25 / 512, so y = x / sqrt(5.25/512 + 1e-6):
    # the block's scale is 2 / sqrt(5.25/512 + 1e-6) / 448 and its codes are those of
    # 448 * (2, -1, 0.5) / 2 = (448, -224, 112): 0x7E, 0xF6 (1.75 * 2^7, negative), 0x6E
    # (1.75 * 2^6).  The zero blocks keep code 0 and scale 1.  Rotation by angle 0 is the
    # identity, so the rope bits come back unchanged.
    x = np.zeros((1, 576))
    x[0, :3] = [2.0, -1.0, 0.5]
    x[0, 512::2] = 1.0
    kv = _bits(x)
    w = _bits(np.ones(512))
    pool = kv_insert(np.zeros((2, ROW_BYTES), np.uint8), kv, np.array([0]), np.array([1]), w, EPS)
    row = pool[1]
    assert list(row[:4]) == [0x7E, 0xF6, 0x6E, 0x00] and not row[4:512].any()
    sc = row[512:528].view("<f4")
    expect = np.float32(2.0 / np.sqrt(5.25 / 512 + 1e-6) / 448.0)
    assert abs(float(sc[0]) - float(expect)) <= 2 ** -22 * float(expect)
    assert list(sc[1:]) == [1.0, 1.0, 1.0]
    assert np.array_equal(row[528:].view("<u2"), kv[0, 512:])
    assert not pool[0].any()


def test_block_max_is_448_and_dequantised_values_track_the_normalised_latent():
    rng = np.random.default_rng(1)
    kv = _rand_kv(rng, 64)
    w = _w(rng)
    codes, scales = quantise_latent(kv[:, :512], w, EPS)
    vals = codecs.e4m3_decode(codes)
    for b in range(4):
        blk = vals[:, 128 * b:128 * (b + 1)]
        assert np.all(np.max(np.abs(blk), axis=1) == 448.0)   # the block max maps to +-448 exactly
    x = codecs.bf16_decode(kv[:, :512])
    y = x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + EPS) * codecs.bf16_decode(w)
    deq = vals * np.repeat(scales, 128, axis=1)
    # E4M3 keeps 3 mantissa bits: half a step is 2^-4 of the value (normals) or 2^-10 of
    # the scale (subnormals)
    bound = np.maximum(2.0 ** -4 * np.abs(y), 2.0 ** -10 * np.repeat(scales, 128, axis=1)) * (1 + 1e-6)
    assert np.all(np.abs(deq - y) <= bound)


def test_scaling_the_latent_by_a_power_of_two_changes_nothing():
    # RMSNorm is invariant to the input's scale (eps aside), and so is the quantiser
    rng = np.random.default_rng(2)
    kv = _rand_kv(rng, 16)
    w = _w(rng)
    c0, s0 = quantise_latent(kv[:, :512], w, EPS)
    big = _bits(codecs.bf16_decode(kv[:, :512]) * 2.0 ** 12)
    c1, s1 = quantise_latent(big, w, EPS)
    assert np.array_equal(c0, c1)
    assert np.allclose(s0, s1, rtol=1e-9)


def test_zero_block_and_weight_zero():
    rng = np.random.default_rng(3)
    kv = _rand_kv(rng, 4)
    x = codecs.bf16_decode(kv)
    x[:, 128:256] = 0.0
    w = codecs.bf16_decode(_w(rng))
    w[384:] = 0.0
    codes, scales = quantise_latent(_bits(x[:, :512]), _bits(w), EPS)
    assert not codes[:, 128:256].any() and np.all(scales[:, 1] == 1.0)
    assert not codes[:, 384:].any() and np.all(scales[:, 3] == 1.0)
    assert np.all(scales[:, [0, 2]] < 1.0)


def test_rope_is_rotated_by_the_position_and_rotates_back():
    rng = np.random.default_rng(4)
    kv = _rand_kv(rng, 8)
    pos = rng.integers(0, 32768, size=8)
    pool = kv_insert(np.zeros((8, ROW_BYTES), np.uint8), kv, pos, np.arange(8), _w(rng), EPS)
    stored = codecs.bf16_decode(pool[:, 528:].copy().view("<u2"))
    r = codecs.bf16_decode(kv[:, 512:])
    for i in range(8):
        back = rope_interleaved(stored[i], float(pos[i]), 10000.0, inverse=True)
        assert np.allclose(back, r[i], rtol=0, atol=2 ** -7 * np.max(np.abs(r[i])))
        # the rotation keeps each pair's length (up to the bf16 rounding)
        n0 = np.hypot(r[i, 0::2], r[i, 1::2])
        n1 = np.hypot(stored[i, 0::2], stored[i, 1::2])
        assert np.allclose(n0, n1, rtol=2 ** -7, atol=1e-30)
    assert not np.array_equal(stored, r)


def test_rows_decode_with_the_attentions_reader_and_skips_leave_the_pool_alone():
    rng = np.random.default_rng(5)
    kv = _rand_kv(rng, 6)
    w = _w(rng)
    pos = rng.integers(0, 4096, size=6)
    before = rng.integers(0, 256, size=(10, ROW_BYTES)).astype(np.uint8)
    slots = np.array([7, -1, 2, -5, 9, 0])
    pool = kv_insert(before, kv, pos, slots, w, EPS)
    untouched = [r for r in range(10) if r not in (7, 2, 9, 0)]
    assert np.array_equal(pool[untouched], before[untouched])
    k = decode_kv_rows(pool[[7, 2, 9, 0]])
    sel = [0, 2, 4, 5]
    x = codecs.bf16_decode(kv[sel, :512])
    y = x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + EPS) * codecs.bf16_decode(w)
    scale = np.repeat(np.max(np.abs(y.reshape(4, 4, 128)), axis=2) / 448.0, 128, axis=1)
    assert np.all(np.abs(k[:, :512] - y) <= np.maximum(2 ** -4 * np.abs(y), 2 ** -10 * scale) * (1 + 1e-6))
    for j, i in enumerate(sel):
        assert np.allclose(k[j, 512:], rope_interleaved(codecs.bf16_decode(kv[i, 512:]), float(pos[i]), 10000.0),
                           rtol=2 ** -8, atol=1e-30)


def test_out_of_range_slot_raises():
    rng = np.random.default_rng(6)
    with pytest.raises(IndexError):
        kv_insert(np.zeros((4, ROW_BYTES), np.uint8), _rand_kv(rng, 1), np.array([0]), np.array([4]), _w(rng), EPS)
