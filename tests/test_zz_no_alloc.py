"""The allocation-free entry point (dsa_sparse_attn_fwd_noalloc) against the workspace
entry point (dsa_sparse_attn_fwd), both through the C ABI.

The two share the split choice and the kernel; the no-alloc call keeps its workspace in
a scratch array built into the library.  The kernel is deterministic (every output is
computed by one fixed sequence of operations, whichever CTA takes it), so both calls of
two in a row must reproduce the workspace entry point's codes and scales bit for bit:
that shows the second call starts from a cleared scratch header and clean combine
counters, which a looser comparison could hide.  This file is named so that pytest
collects it last: it must pass on a process that has already run every other test, and
on its own.
"""

import ctypes

import numpy as np
import pytest
import torch

from top_sparse_mla_gb300 import api, native
from top_sparse_mla_gb300 import workloads as W

def _assert_match(ref_fp8, ref_sf, fp8, sf, label):
    assert np.array_equal(sf, ref_sf), f"{label}: UE8M0 scale codes differ"
    diff = int((fp8 != ref_fp8).sum())
    assert diff == 0, f"{label}: {diff} E4M3 codes differ from the workspace entry point's"


def _outputs(inp):
    s_q, h_q = inp.params.s_q, inp.params.h_q
    fp8 = torch.empty((s_q, h_q, 512), dtype=torch.uint8, device=inp.q.device)
    sf = torch.empty((s_q, h_q, 16), dtype=torch.uint8, device=inp.q.device)
    return fp8, sf


def _noalloc(inp, fp8, sf, status):
    native.dsa_sparse_attn_fwd_noalloc(inp.q, inp.kv_swa, inp.kv_cmp, inp.indices, inp.topk_length,
                                       inp.positions, inp.norm_w, fp8, sf, inp.params, status_out=status)


def _check_case(w, flags=0):
    inp = api.upload(w, "cuda:0", flags=flags)
    # the workspace entry point
    ref = api.allocate_outputs(inp, debug=False)
    api.forward(inp, ref)
    torch.cuda.synchronize()
    ref_fp8, ref_sf = ref.out_fp8.cpu().numpy(), ref.out_sf.cpu().numpy()
    ref_status = native.dsa_sparse_attn_read_status(ref.workspace)
    # two allocation-free calls in a row on the same stream, into separate buffers
    outs = [_outputs(inp) for _ in range(2)]
    status = torch.full((2,), 0x7FFFFFFF, dtype=torch.int32, device="cuda:0")
    for k, (fp8, sf) in enumerate(outs):
        _noalloc(inp, fp8, sf, status[k:k + 1])
    torch.cuda.synchronize()
    for k, (fp8, sf) in enumerate(outs):
        _assert_match(ref_fp8, ref_sf, fp8.cpu().numpy(), sf.cpu().numpy(), f"{w.name} call {k + 1}")
    assert [int(x) for x in status.cpu()] == [ref_status, ref_status]
    return ref_status


@pytest.mark.gpu
def test_split_path_two_calls_in_a_row():
    # one token over five 128-row tiles: five CTAs combine through the scratch
    assert _check_case(W.make("decode1")) == 0


@pytest.mark.gpu
def test_batched_split_path_two_calls_in_a_row():
    assert _check_case(W.make("decode64")) == 0


@pytest.mark.gpu
def test_unsplit_path_two_calls_in_a_row():
    w = W.random_case(402, s_q=300, h_q=64, n_swa_cols=128, n_cmp_cols=173, n_swa_rows=2000, n_cmp_rows=5000,
                      n_sentinels=9, lengths="ragged")
    assert _check_case(w) == 0


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["decode1_nvfp4", "decode64_nvfp4", "decode1_fp8q", "decode64_fp8q"])
def test_other_kernel_instantiations_two_calls_in_a_row(name):
    # the nvfp4_ds_mla cache and the E4M3-q option (the kernel's other two instantiations)
    assert _check_case(W.make(name)) == 0


@pytest.mark.gpu
def test_status_word_reaches_status_out():
    w = W.random_case(405, s_q=2, h_q=16, n_swa_cols=16, n_cmp_cols=48, n_swa_rows=64, n_cmp_rows=128)
    w.indices[1, 20] = w.kv_cmp.shape[0] + 7       # out of range for its pool
    st = _check_case(w, flags=native.DSA_FLAG_CHECK_INDICES)
    assert st & native.DSA_STATUS_INDEX_OUT_OF_RANGE


@pytest.mark.gpu
def test_no_device_memory_is_allocated_by_the_calls():
    w = W.random_case(406, s_q=3, h_q=64, n_swa_cols=64, n_cmp_cols=448, n_swa_rows=512, n_cmp_rows=2048)
    inp = api.upload(w, "cuda:0")
    fp8, sf = _outputs(inp)
    _noalloc(inp, fp8, sf, None)      # first call on this device: scratch address lookup
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        _noalloc(inp, fp8, sf, None)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


@pytest.mark.gpu
def test_shapes_beyond_the_scratch_are_rejected_before_any_work():
    lib = native.library()
    p = native.dsa_params_init(6_000_000, 64, 0, 0, 1, 1)
    rc = lib.dsa_sparse_attn_fwd_noalloc(16, 16, 16, 16, 16, 16, 16, 16, 16, ctypes.byref(p), None, None)
    assert rc == native.DSA_ERR_SCRATCH_LIMIT
    assert "scratch" in native.dsa_error_string(rc)
    # the same shape is fine through the workspace entry point's size query
    assert native.dsa_sparse_attn_workspace_size(p) > native.DSA_NOALLOC_SCRATCH_BYTES
