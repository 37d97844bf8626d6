"""ctypes binding of the C ABI in include/dsa_sparse_attn.h (argument marshalling only).

Every entry point keeps the C name.  Tensors are passed as raw device pointers
(``tensor.data_ptr()``); the stream is the caller's current CUDA stream.  All of the
computation happens in the CUDA library; when the library is missing this module raises
instead of falling back to anything else.
"""

from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

DSA_OK = 0
DSA_ERR_INVALID_ARG = -1
DSA_ERR_UNSUPPORTED_SHAPE = -2
DSA_ERR_WORKSPACE_TOO_SMALL = -3
DSA_ERR_CUDA = -4
DSA_ERR_UNSUPPORTED_DEVICE = -5
DSA_ERR_SCRATCH_LIMIT = -6
DSA_FLAG_CHECK_INDICES = 1
DSA_FLAG_TEST_WAIT_TIMEOUT = 2
DSA_STATUS_INDEX_OUT_OF_RANGE = 1
DSA_STATUS_WAIT_TIMEOUT = 2
DSA_MAX_HEADS = 64
DSA_MAX_DEVICES = 64
DSA_MAX_TOPK = 2048
DSA_ORDER_MAX_TOKENS = 65536
DSA_TOPK_MAX_COLS = 65536
DSA_TOPK_MAX_K = 2048
DSA_ROW_BYTES = 656
DSA_NOALLOC_SCRATCH_BYTES = 24 << 20
DSA_KV_FLAG_CHECK_SLOTS = 1
DSA_FLAG_AFTER_PRODUCER = 4
DSA_FLAG_SF_SWIZZLED = 8
DSA_FLAG_FP8_Q = 16
DSA_KV_FP8_DS_MLA = 0
DSA_KV_NVFP4_DS_MLA = 1
DSA_NVFP4_QK_DIMS = 512
DSA_NVFP4_SWA_ROW_BYTES = 528
DSA_NVFP4_CMP_ROW_BYTES = 288
DSA_STATUS_SLOT_OUT_OF_RANGE = 4

EXPORTED = (
    "dsa_params_init",
    "dsa_sparse_attn_workspace_size",
    "dsa_sparse_attn_fwd",
    "dsa_sparse_attn_fwd_debug",
    "dsa_sparse_attn_fwd_noalloc",
    "dsa_sparse_attn_read_status",
    "dsa_sparse_attn_num_splits",
    "dsa_error_string",
    "dsa_topk_select",
    "dsa_kv_insert",
)


class DsaParams(ctypes.Structure):
    _fields_ = [
        ("s_q", ctypes.c_int32),
        ("h_q", ctypes.c_int32),
        ("topk", ctypes.c_int32),
        ("n_swa_cols", ctypes.c_int32),
        ("n_swa_rows", ctypes.c_int64),
        ("n_cmp_rows", ctypes.c_int64),
        ("softmax_scale", ctypes.c_float),
        ("rope_base", ctypes.c_float),
        ("rms_eps", ctypes.c_float),
        ("flags", ctypes.c_uint32),
        ("kv_format", ctypes.c_int32),
        ("cmp_scale", ctypes.c_float),
    ]


class DsaError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {dsa_error_string(code)} (code {code})")
        self.code = code


_lib = None


def library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library once; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with top_sparse_mla_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    pp = ctypes.POINTER(DsaParams)
    lib.dsa_params_init.argtypes = [pp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                    ctypes.c_int64, ctypes.c_int64]
    lib.dsa_params_init.restype = ctypes.c_int
    lib.dsa_sparse_attn_workspace_size.argtypes = [pp, ctypes.c_int]
    lib.dsa_sparse_attn_workspace_size.restype = sz
    lib.dsa_sparse_attn_num_splits.argtypes = [pp, ctypes.c_int]
    lib.dsa_sparse_attn_num_splits.restype = ctypes.c_int
    lib.dsa_sparse_attn_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, pp, vp, sz, vp]
    lib.dsa_sparse_attn_fwd.restype = ctypes.c_int
    lib.dsa_sparse_attn_fwd_debug.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, pp, vp, sz, vp]
    lib.dsa_sparse_attn_fwd_debug.restype = ctypes.c_int
    lib.dsa_sparse_attn_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, pp, vp, vp]
    lib.dsa_sparse_attn_fwd_noalloc.restype = ctypes.c_int
    lib.dsa_sparse_attn_read_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
    lib.dsa_sparse_attn_read_status.restype = ctypes.c_int
    lib.dsa_error_string.argtypes = [ctypes.c_int]
    lib.dsa_error_string.restype = ctypes.c_char_p
    lib.dsa_topk_select.argtypes = [vp, ctypes.c_int64, vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, vp, vp, vp]
    lib.dsa_topk_select.restype = ctypes.c_int
    lib.dsa_kv_insert.argtypes = [vp, ctypes.c_int64, vp, vp, ctypes.c_int32, vp, ctypes.c_float, ctypes.c_float, vp,
                                  ctypes.c_int64, ctypes.c_uint32, vp, vp]
    lib.dsa_kv_insert.restype = ctypes.c_int
    _lib = lib
    return lib


def sf_swizzled_bytes(s_q: int, h_q: int) -> int:
    """Size of out_sf with DSA_FLAG_SF_SWIZZLED (DSA_SF_SWIZZLED_BYTES in the header)."""
    return ((int(s_q) + 127) // 128) * 128 * 16 * int(h_q)


def dsa_error_string(code: int) -> str:
    return library().dsa_error_string(int(code)).decode()


def dsa_params_init(s_q, h_q, topk, n_swa_cols, n_swa_rows, n_cmp_rows, **overrides) -> DsaParams:
    p = DsaParams()
    rc = library().dsa_params_init(ctypes.byref(p), s_q, h_q, topk, n_swa_cols, n_swa_rows, n_cmp_rows)
    if rc != DSA_OK:
        raise DsaError(rc, "dsa_params_init")
    for k, v in overrides.items():
        setattr(p, k, v)
    return p


def dsa_sparse_attn_workspace_size(p: DsaParams, num_sms: int = 0) -> int:
    return int(library().dsa_sparse_attn_workspace_size(ctypes.byref(p), int(num_sms)))


def dsa_sparse_attn_num_splits(p: DsaParams, num_sms: int = 0) -> int:
    return int(library().dsa_sparse_attn_num_splits(ctypes.byref(p), int(num_sms)))


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def dsa_sparse_attn_fwd(q, kv_swa, kv_cmp, indices, topk_length, positions, norm_w, out_fp8, out_sf,
                        p: DsaParams, workspace, workspace_bytes=None, stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = library().dsa_sparse_attn_fwd(_ptr(q), _ptr(kv_swa), _ptr(kv_cmp), _ptr(indices), _ptr(topk_length),
                                       _ptr(positions), _ptr(norm_w), _ptr(out_fp8), _ptr(out_sf), ctypes.byref(p),
                                       _ptr(workspace), int(workspace_bytes), _stream(stream))
    if rc != DSA_OK:
        raise DsaError(rc, "dsa_sparse_attn_fwd")


def dsa_sparse_attn_fwd_debug(q, kv_swa, kv_cmp, indices, topk_length, positions, norm_w, out_fp8, out_sf,
                              out_precast, lse, p: DsaParams, workspace, workspace_bytes=None, stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = library().dsa_sparse_attn_fwd_debug(_ptr(q), _ptr(kv_swa), _ptr(kv_cmp), _ptr(indices), _ptr(topk_length),
                                             _ptr(positions), _ptr(norm_w), _ptr(out_fp8), _ptr(out_sf),
                                             _ptr(out_precast), _ptr(lse), ctypes.byref(p), _ptr(workspace),
                                             int(workspace_bytes), _stream(stream))
    if rc != DSA_OK:
        raise DsaError(rc, "dsa_sparse_attn_fwd_debug")


def dsa_sparse_attn_fwd_noalloc(q, kv_swa, kv_cmp, indices, topk_length, positions, norm_w, out_fp8, out_sf,
                                p: DsaParams, status_out=None, stream=None) -> None:
    rc = library().dsa_sparse_attn_fwd_noalloc(_ptr(q), _ptr(kv_swa), _ptr(kv_cmp), _ptr(indices),
                                               _ptr(topk_length), _ptr(positions), _ptr(norm_w), _ptr(out_fp8),
                                               _ptr(out_sf), ctypes.byref(p), _ptr(status_out), _stream(stream))
    if rc != DSA_OK:
        raise DsaError(rc, "dsa_sparse_attn_fwd_noalloc")


def dsa_topk_select(logits, k: int, indices, topk_length, lengths=None, stream=None) -> None:
    """Top-k column selection (include/dsa_topk.h). logits: bf16 [s_q, ld] device tensor
    whose first n = logits.shape[1] columns are the candidates; indices: int32 [s_q, k];
    topk_length: int32 [s_q]; lengths: int32 [s_q] or None."""
    s_q, n = int(logits.shape[0]), int(logits.shape[1])
    if s_q > 0 and int(logits.stride(1)) != 1:
        raise DsaError(DSA_ERR_INVALID_ARG, "dsa_topk_select: logits rows must be contiguous")
    ld = int(logits.stride(0)) if s_q > 0 else n
    rc = library().dsa_topk_select(_ptr(logits), ld, _ptr(lengths), s_q, n, int(k), _ptr(indices),
                                   _ptr(topk_length), _stream(stream))
    if rc != DSA_OK:
        raise DsaError(rc, "dsa_topk_select")


def dsa_kv_insert(kv, positions, slots, kv_norm_w, pool, rms_eps: float = 1e-6, rope_base: float = 10000.0,
                  check_slots: bool = False, status=None, stream=None) -> None:
    """KV-cache insert (include/dsa_kv_insert.h). kv: bf16 [s_new, ld >= 576] device tensor
    (512 latent then 64 rotary values per row); positions: int32 [s_new]; slots: int64
    [s_new] (< 0 = skip); kv_norm_w: bf16 [512]; pool: uint8 [n_rows, 656]; status: uint32
    [1] device tensor or None."""
    s_new = int(kv.shape[0])
    if s_new > 0 and int(kv.stride(1)) != 1:
        raise DsaError(DSA_ERR_INVALID_ARG, "dsa_kv_insert: kv rows must be contiguous")
    ld = int(kv.stride(0)) if s_new > 0 else 576
    rc = library().dsa_kv_insert(_ptr(kv), ld, _ptr(positions), _ptr(slots), s_new, _ptr(kv_norm_w),
                                 float(rms_eps), float(rope_base), _ptr(pool), int(pool.shape[0]),
                                 DSA_KV_FLAG_CHECK_SLOTS if check_slots else 0, _ptr(status), _stream(stream))
    if rc != DSA_OK:
        raise DsaError(rc, "dsa_kv_insert")


def dsa_sparse_attn_read_status(workspace, stream=None) -> int:
    st = ctypes.c_uint32(0)
    rc = library().dsa_sparse_attn_read_status(_ptr(workspace), ctypes.byref(st), _stream(stream))
    if rc != DSA_OK:
        raise DsaError(rc, "dsa_sparse_attn_read_status")
    return int(st.value)
