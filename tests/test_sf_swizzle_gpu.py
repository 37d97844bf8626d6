"""The 128x4-swizzled scale-factor layout (DSA_FLAG_SF_SWIZZLED) on GB300.

With the flag the kernel writes the same scale codes as without it, each at the byte
the oracle's layout definition (oracle.codecs.sf_swizzle_128x4) gives it, and leaves the
padding of the last tile row untouched; every other output is unchanged.  The codes
themselves are checked against the float64 oracle as in the parity tests."""

import numpy as np
import pytest
import torch

from oracle.codecs import sf_swizzle_128x4
from top_sparse_mla_gb300 import api, native
from top_sparse_mla_gb300 import workloads as W

import parity

pytestmark = pytest.mark.gpu

PAD = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from top_sparse_mla_gb300.build import build
    build()
    native.library()


def _run(w, flags):
    inp = api.upload(w, "cuda:0", flags=flags)
    out = api.allocate_outputs(inp, debug=True)
    out.out_sf.fill_(PAD)
    api.forward(inp, out)
    torch.cuda.synchronize()
    return {"out_fp8": out.out_fp8.cpu().numpy(), "out_sf": out.out_sf.cpu().numpy(),
            "out": out.out_precast.cpu().numpy().astype(np.float64), "lse": out.lse.cpu().numpy().astype(np.float64),
            "status": native.dsa_sparse_attn_read_status(out.workspace)}


def _case(name):
    if name == "ragged_empty_rows":
        # queue path, 200 tokens (two tile rows of the scale matrix, the second padded),
        # five tokens without any valid column
        w = W.random_case(411, s_q=200, h_q=64, n_swa_cols=64, n_cmp_cols=150, n_swa_rows=1000, n_cmp_rows=3000,
                          n_sentinels=7, lengths="ragged")
        w.topk_length[[0, 3, 127, 128, 199]] = 0
        return w
    if name == "odd_heads":
        return W.random_case(412, s_q=129, h_q=40, n_swa_cols=32, n_cmp_cols=96, n_swa_rows=500, n_cmp_rows=900,
                             n_sentinels=3)
    return W.make(name)


@pytest.mark.parametrize("name", ["tiny", "decode1", "decode64", "ragged_empty_rows", "odd_heads"])
def test_swizzled_scale_layout(name):
    w = _case(name)
    plain = _run(w, 0)
    swz = _run(w, native.DSA_FLAG_SF_SWIZZLED)
    assert plain["status"] == 0 and swz["status"] == 0
    # every other output is that of the row-major layout, bit for bit
    assert np.array_equal(plain["out_fp8"], swz["out_fp8"])
    assert np.array_equal(plain["out"], swz["out"])
    s_q, h_q = w.s_q, w.h_q
    assert swz["out_sf"].size == native.sf_swizzled_bytes(s_q, h_q)
    written = sf_swizzle_128x4(np.ones((s_q, 16 * h_q), dtype=np.uint8)) == 1
    expect = sf_swizzle_128x4(plain["out_sf"].reshape(s_q, 16 * h_q))
    assert np.array_equal(swz["out_sf"][written], expect[written])
    assert np.all(swz["out_sf"][~written] == PAD)        # the padding rows are not written
    # the row-major codes against the oracle (the usual parity bar)
    r = parity.run_oracle(w)
    e = parity.compare(plain, r, label=name + "_sf_swizzled")
    print(name, e)
