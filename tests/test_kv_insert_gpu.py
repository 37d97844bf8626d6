"""The KV-cache insert's CUDA path (include/dsa_kv_insert.h) against the oracle
(oracle/kv_insert.py), on seeded inputs.

What must agree, and why:
- E4M3 codes bit for bit: both sides take each code in binary32 as (x*w) times one
  rounded quotient 448 / max|x*w| per block (x*w and the max are exact), rounded to
  nearest even;
- the fp32 block scales within 2^-20 relative: the kernel's fp32 RMS statistics
  (a sum of 512 squares and a square root) against the oracle's float64;
- the rotated bf16 rope values within one bf16 step plus 2^-20 of the pair's length (the
  kernel rotates in fp32, the angle's fraction of a turn taken to 24 bits; a value near
  zero is a cancellation, so that error is absolute), identical on >= 99.9 %;
- every byte outside the written rows unchanged.
The last test writes rows with the kernel and runs the attention on them."""

import numpy as np
import pytest
import torch

import oracle
from oracle import codecs
from oracle.kv_insert import kv_insert
from oracle.sparse_mla import ROW_BYTES
from top_sparse_mla_gb300 import native

pytestmark = pytest.mark.gpu

SCALE_REL = 2.0 ** -20
ROPE_IDENTICAL = 0.999


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from top_sparse_mla_gb300.build import build
    build()
    native.library()


def _bits(x):
    return codecs.bf16_encode(np.asarray(x, dtype=np.float64))


def _inputs(seed, n, n_rows, scale=1.0, skip_every=0):
    rng = np.random.default_rng(seed)
    kv = _bits(rng.standard_normal((n, 576)) * scale)
    w = _bits(1.0 + 0.1 * rng.standard_normal(512))
    pos = rng.integers(0, 32768, size=n).astype(np.int32)
    slots = rng.permutation(n_rows)[:n].astype(np.int64)
    if skip_every:
        slots[::skip_every] = -1
    pool = rng.integers(0, 256, size=(n_rows, ROW_BYTES)).astype(np.uint8)
    return kv, w, pos, slots, pool


def _run(kv, w, pos, slots, pool, pad=0, check=False, eps=1e-6, base=10000.0):
    n = kv.shape[0]
    buf = torch.zeros((n, 576 + pad), dtype=torch.int16, device="cuda")
    buf[:, :576] = torch.from_numpy(kv.view(np.int16)).cuda()
    kv_d = buf.view(torch.bfloat16)
    pool_d = torch.from_numpy(pool.copy()).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    native.dsa_kv_insert(kv_d, torch.from_numpy(pos).cuda(), torch.from_numpy(slots).cuda(),
                         torch.from_numpy(w.view(np.int16)).cuda().view(torch.bfloat16), pool_d, eps, base,
                         check_slots=check, status=status)
    torch.cuda.synchronize()
    return pool_d.cpu().numpy(), int(status.cpu().item())


def _compare(got, ref, before, slots):
    written = sorted(int(s) for s in slots if 0 <= s < before.shape[0])
    others = np.setdiff1d(np.arange(before.shape[0]), written)
    assert np.array_equal(got[others], before[others]), "bytes outside the written rows changed"
    g, r = got[written], ref[written]
    assert np.array_equal(g[:, :512], r[:, :512]), f"{int((g[:, :512] != r[:, :512]).sum())} E4M3 codes differ"
    gs = g[:, 512:528].copy().view("<f4").astype(np.float64)
    rs = r[:, 512:528].copy().view("<f4").astype(np.float64)
    assert np.all(np.abs(gs - rs) <= SCALE_REL * np.abs(rs)), float(np.max(np.abs(gs - rs) / np.abs(rs)))
    gr = g[:, 528:].copy().view("<u2")
    rr = r[:, 528:].copy().view("<u2")
    gv, rv = codecs.bf16_decode(gr), codecs.bf16_decode(rr)
    # one bf16 step of the value, plus the fp32 rotation's error, which is absolute in the
    # pair's length (a rotated value near zero comes from cancellation)
    mag = np.repeat(np.hypot(rv[:, 0::2], rv[:, 1::2]), 2, axis=1)
    step = np.exp2(np.floor(np.log2(np.where(rv != 0, np.abs(rv), 1.0))) - 7)
    assert np.all(np.abs(gv - rv) <= step + 2.0 ** -20 * mag), "rope values differ beyond the rotation's error"
    # otherwise a value lands on the other side of a bf16 rounding tie about 3e-4 of the time
    assert (gr != rr).sum() <= max(2, (1 - ROPE_IDENTICAL) * gr.size), int((gr != rr).sum())
    return len(written)


@pytest.mark.parametrize("n,n_rows,skip", [(1, 4, 0), (7, 50, 3), (1000, 4096, 0), (4096, 8192, 5)])
def test_random_rows(n, n_rows, skip):
    kv, w, pos, slots, pool = _inputs(100 + n, n, n_rows, skip_every=skip)
    got, st = _run(kv, w, pos, slots, pool)
    ref = kv_insert(pool, kv, pos, slots, w)
    assert st == 0
    assert _compare(got, ref, pool, slots) == int((slots >= 0).sum())


def test_value_ranges_zero_blocks_and_an_odd_pitch():
    for seed, scale in ((1, 2.0 ** 40), (2, 2.0 ** -40), (3, 1.0)):
        kv, w, pos, slots, pool = _inputs(seed, 64, 256)
        x = codecs.bf16_decode(kv) * scale
        x[::4, 128:256] = 0.0                  # all-zero blocks: code 0, scale 1
        x[1::4, :512] = 0.0                    # an all-zero latent
        x[2::4, 3] = 1e4 * scale               # one dominant value per block 0
        kv = _bits(x)
        pos[:4] = [0, 1, 32767, 1 << 20]
        got, _ = _run(kv, w, pos, slots, pool, pad=8)
        _compare(got, kv_insert(pool, kv, pos, slots, w), pool, slots)


def test_checked_slots_report_and_skip_out_of_range_rows():
    kv, w, pos, slots, pool = _inputs(9, 16, 64)
    slots[3] = 64
    slots[7] = 1 << 40
    got, st = _run(kv, w, pos, slots, pool, check=True)
    assert st == native.DSA_STATUS_SLOT_OUT_OF_RANGE
    keep = slots.copy()
    keep[[3, 7]] = -1
    _compare(got, kv_insert(pool, kv, pos, keep, w), pool, keep)


def test_inserted_rows_feed_the_attention():
    # the kernel writes the compressed pool's rows of a small decode batch, then the
    # attention reads them; compared with the oracle attention on the same pool bytes
    import parity
    from top_sparse_mla_gb300 import workloads as W
    w0 = W.make("tiny")
    n_cmp = w0.kv_cmp.shape[0]
    kv, wn, pos, _, _ = _inputs(12, n_cmp, n_cmp)
    slots = np.arange(n_cmp, dtype=np.int64)
    got, st = _run(kv, wn, pos, slots, w0.kv_cmp)
    assert st == 0
    _compare(got, kv_insert(w0.kv_cmp, kv, pos, slots, wn), w0.kv_cmp, slots)
    w1 = W.Workload(name="tiny_inserted", q=w0.q, norm_w=w0.norm_w, kv_swa=w0.kv_swa, kv_cmp=got,
                    indices=w0.indices, topk_length=w0.topk_length, positions=w0.positions,
                    n_swa_cols=w0.n_swa_cols, seed=w0.seed)
    parity.compare(parity.run_gpu(w1), parity.run_oracle(w1), label="attention on kernel-inserted rows")
