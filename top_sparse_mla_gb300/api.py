"""Convenience layer over the C ABI: device buffers for a workload and one forward call.

PyTorch only allocates device memory and supplies the stream here; the forward pass is
the CUDA library's.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import native
from .workloads import Workload


@dataclass
class DeviceInputs:
    q: torch.Tensor            # uint16 view of bf16 [s_q, h_q, 576] (512: nvfp4_ds_mla)
    kv_swa: torch.Tensor       # uint8 [n_swa_rows, 656] (528: nvfp4_ds_mla)
    kv_cmp: torch.Tensor       # uint8 [n_cmp_rows, 656] (288: nvfp4_ds_mla)
    indices: torch.Tensor      # int32 [s_q, topk]
    topk_length: torch.Tensor  # int32 [s_q]
    positions: torch.Tensor    # int32 [s_q]
    norm_w: torch.Tensor       # uint16 view of bf16 [576] (512: nvfp4_ds_mla)
    params: native.DsaParams


@dataclass
class DeviceOutputs:
    out_fp8: torch.Tensor      # uint8 [s_q, h_q, 512]
    out_sf: torch.Tensor       # uint8 [s_q, h_q, 16] (flat 128x4 tiles with DSA_FLAG_SF_SWIZZLED)
    out_precast: torch.Tensor | None
    lse: torch.Tensor | None
    workspace: torch.Tensor


def _dev(a: np.ndarray, device, dtype):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(device)


def upload(w: Workload, device="cuda", flags: int = 0) -> DeviceInputs:
    # uint16 bit patterns travel as int16 (torch has no general uint16 ops)
    p = native.dsa_params_init(w.s_q, w.h_q, w.topk, w.n_swa_cols, w.kv_swa.shape[0], w.kv_cmp.shape[0])
    p.flags = flags | (native.DSA_FLAG_FP8_Q if w.fp8_q else 0)
    p.kv_format = w.kv_format
    p.cmp_scale = w.cmp_scale
    p.softmax_scale = w.softmax_scale
    return DeviceInputs(
        q=_dev(w.q.view(np.int16), device, None),
        kv_swa=_dev(w.kv_swa, device, None),
        kv_cmp=_dev(w.kv_cmp, device, None),
        indices=_dev(w.indices, device, None),
        topk_length=_dev(w.topk_length, device, None),
        positions=_dev(w.positions, device, None),
        norm_w=_dev(w.norm_w.view(np.int16), device, None),
        params=p,
    )


def allocate_outputs(inp: DeviceInputs, debug: bool = False) -> DeviceOutputs:
    p = inp.params
    dev = inp.q.device
    ws_bytes = native.dsa_sparse_attn_workspace_size(p)
    if ws_bytes == 0:
        raise native.DsaError(native.DSA_ERR_INVALID_ARG, "dsa_sparse_attn_workspace_size")
    return DeviceOutputs(
        out_fp8=torch.empty((p.s_q, p.h_q, 512), dtype=torch.uint8, device=dev),
        # row-major [s_q, h_q, 16], or the flat 128x4-tile layout (DSA_FLAG_SF_SWIZZLED)
        out_sf=(torch.empty(native.sf_swizzled_bytes(p.s_q, p.h_q), dtype=torch.uint8, device=dev)
                if p.flags & native.DSA_FLAG_SF_SWIZZLED else
                torch.empty((p.s_q, p.h_q, 16), dtype=torch.uint8, device=dev)),
        out_precast=torch.empty((p.s_q, p.h_q, 512), dtype=torch.float32, device=dev) if debug else None,
        lse=torch.empty((p.s_q, p.h_q), dtype=torch.float32, device=dev) if debug else None,
        workspace=torch.empty(((ws_bytes + 255) // 256) * 256, dtype=torch.uint8, device=dev),
    )


def forward(inp: DeviceInputs, out: DeviceOutputs, stream=None) -> None:
    """One fused forward call on the current (or given) stream."""
    if out.out_precast is not None or out.lse is not None:
        native.dsa_sparse_attn_fwd_debug(inp.q, inp.kv_swa, inp.kv_cmp, inp.indices, inp.topk_length, inp.positions,
                                         inp.norm_w, out.out_fp8, out.out_sf, out.out_precast, out.lse, inp.params,
                                         out.workspace, stream=stream)
    else:
        native.dsa_sparse_attn_fwd(inp.q, inp.kv_swa, inp.kv_cmp, inp.indices, inp.topk_length, inp.positions,
                                   inp.norm_w, out.out_fp8, out.out_sf, inp.params, out.workspace, stream=stream)
