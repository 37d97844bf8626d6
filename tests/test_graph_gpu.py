"""The forward call captured in a CUDA graph and replayed, against the same call made
directly (C ABI through the binding).

The single-token case takes the split path: an asynchronous memset of the workspace
header and counters, then the fused kernel's cooperative launch. The tiny case takes
the queue path: the one-CTA order kernel, then the fused kernel as its programmatic
dependent. Both sequences are captured on the caller's stream.
"""

import numpy as np
import pytest
import torch

from top_sparse_mla_gb300 import api, native
from top_sparse_mla_gb300 import workloads as W


def _direct(inp):
    out = api.allocate_outputs(inp, debug=False)
    api.forward(inp, out)
    torch.cuda.synchronize()
    return out.out_fp8.cpu().numpy(), out.out_sf.cpu().numpy()


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["tiny", "decode1", "tiny_nvfp4", "decode1_nvfp4", "tiny_fp8q"])
def test_forward_replays_from_a_cuda_graph(name):
    w = W.make(name)
    inp = api.upload(w, "cuda:0")
    if name.startswith("decode1"):
        p = native.dsa_params_init(w.s_q, w.h_q, w.topk, w.n_swa_cols, w.kv_swa.shape[0], w.kv_cmp.shape[0])
        assert native.dsa_sparse_attn_num_splits(p) > 1
    ref_fp8, ref_sf = _direct(inp)
    out = api.allocate_outputs(inp, debug=False)
    # one call outside the capture (first-use setup on the host), on a side stream
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        api.forward(inp, out)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        api.forward(inp, out)
    for _ in range(2):
        out.out_fp8.zero_()
        out.out_sf.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(out.out_fp8.cpu().numpy(), ref_fp8)
        assert np.array_equal(out.out_sf.cpu().numpy(), ref_sf)
    assert native.dsa_sparse_attn_read_status(out.workspace) == 0
