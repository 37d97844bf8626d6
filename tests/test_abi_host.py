"""Host-side checks of the C ABI (no GPU): the library builds, loads and exports every
function the header declares; argument validation fails before anything touches a GPU."""

import ctypes
import os
import re

import pytest

from top_sparse_mla_gb300 import native
from top_sparse_mla_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa_sparse_attn.h")
HEADERS = sorted(os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h"))


@pytest.fixture(scope="module")
def lib():
    build()
    return native.library()


def declared_functions():
    text = "\n".join(open(h).read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(dsa_[a-z_0-9]+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in native.EXPORTED:
        assert n in names, n
    assert set(names) == set(native.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"missing export {name}"


def test_header_constants_match_the_binding():
    # "#define NAME 2u", "#define NAME (-1)" and "#define NAME (24u << 20)"
    pattern = re.compile(r"^#define (DSA_[A-Z0-9_]+) \(?(-?[0-9]+)u?(?: << ([0-9]+))?", re.M)
    defines = {name: int(v) << int(shift or 0) for h in HEADERS for name, v, shift in pattern.findall(open(h).read())}
    assert "DSA_FLAG_TEST_WAIT_TIMEOUT" in defines and "DSA_TOPK_MAX_COLS" in defines
    for name, value in defines.items():
        assert getattr(native, name) == value, name


def test_order_bound_matches_the_kernel_source():
    # the kernel keeps its own copy of the bound above which the queue is not ordered
    src = open(os.path.join(ROOT, "top_sparse_mla_gb300", "csrc", "dsa_sparse_attn.cu")).read()
    m = re.search(r"constexpr int ORDER_MAX_TOKENS = ([0-9]+);", src)
    assert m and int(m.group(1)) == native.DSA_ORDER_MAX_TOKENS


def test_flag_mask(lib):
    # the defined flags pass the argument check (num_splits returns 0 on a bad argument)
    p = native.dsa_params_init(4, 64, 1024, 128, 512, 4096,
                               flags=native.DSA_FLAG_CHECK_INDICES | native.DSA_FLAG_TEST_WAIT_TIMEOUT
                               | native.DSA_FLAG_AFTER_PRODUCER | native.DSA_FLAG_SF_SWIZZLED | native.DSA_FLAG_FP8_Q)
    assert native.dsa_sparse_attn_num_splits(p, 152) == 8
    for bad in (32, 64, 1 << 31):
        p.flags = bad
        assert native.dsa_sparse_attn_num_splits(p, 152) == 0


def test_topk_select_checks_arguments_before_the_device(lib):
    ok = native.DSA_OK
    fake = 1 << 20   # a 16-byte aligned address that is never dereferenced on the host
    f = lib.dsa_topk_select
    bad = native.DSA_ERR_INVALID_ARG
    assert f(fake, 100, None, -1, 100, 8, fake, fake, None) == bad          # s_q < 0
    assert f(fake, 100, None, 4, 0, 8, fake, fake, None) == bad             # n < 1
    assert f(fake, 70000, None, 4, native.DSA_TOPK_MAX_COLS + 1, 8, fake, fake, None) == bad
    assert f(fake, 100, None, 4, 100, native.DSA_TOPK_MAX_K + 1, fake, fake, None) == bad
    assert f(fake, 99, None, 4, 100, 8, fake, fake, None) == bad            # ld < n
    assert f(None, 100, None, 4, 100, 8, fake, fake, None) == bad           # no logits
    assert f(fake, 100, None, 4, 100, 8, None, fake, None) == bad           # no indices with k > 0
    assert f(fake + 1, 100, None, 4, 100, 8, fake, fake, None) == bad       # misaligned logits
    assert f(fake, 100, None, 0, 100, 8, None, None, None) == ok            # an empty batch is a no-op
    # valid arguments reach the device check, which fails without a GPU
    assert f(fake, 100, None, 4, 100, 8, fake, fake, None) in (native.DSA_ERR_CUDA, native.DSA_ERR_UNSUPPORTED_DEVICE)


def test_kv_insert_checks_arguments_before_the_device(lib):
    ok, bad = native.DSA_OK, native.DSA_ERR_INVALID_ARG
    fake = 1 << 20   # a 16-byte aligned address that is never dereferenced on the host
    f = lib.dsa_kv_insert
    args = dict(kv=fake, ld=576, pos=fake, slots=fake, n=4, w=fake, eps=1e-6, base=10000.0, pool=fake, rows=100,
                flags=0, status=None)

    def call(**kw):
        a = dict(args, **kw)
        return f(a["kv"], a["ld"], a["pos"], a["slots"], a["n"], a["w"], a["eps"], a["base"], a["pool"], a["rows"],
                 a["flags"], a["status"], None)

    assert call(n=-1) == bad
    assert call(ld=575) == bad and call(ld=580) == bad          # ld >= 576 and a multiple of 8
    assert call(eps=-1.0) == bad and call(eps=float("nan")) == bad
    assert call(base=0.0) == bad and call(base=float("inf")) == bad
    assert call(flags=2) == bad                                 # only DSA_KV_FLAG_CHECK_SLOTS is defined
    assert call(rows=-1) == bad
    assert call(kv=None) == bad and call(slots=None) == bad and call(w=None) == bad and call(pos=None) == bad
    assert call(pool=None) == bad                              # rows > 0 needs a pool
    assert call(kv=fake + 8) == bad and call(w=fake + 2) == bad and call(pool=fake + 4) == bad
    assert call(slots=fake + 4) == bad and call(status=fake + 2) == bad
    assert call(n=0, kv=None) == ok                             # an empty batch is a no-op
    # valid arguments reach the device check, which fails without a GPU
    assert call() in (native.DSA_ERR_CUDA, native.DSA_ERR_UNSUPPORTED_DEVICE)
    assert call(flags=native.DSA_KV_FLAG_CHECK_SLOTS, status=fake) in (native.DSA_ERR_CUDA,
                                                                         native.DSA_ERR_UNSUPPORTED_DEVICE)


def test_params_init_defaults(lib):
    p = native.dsa_params_init(4, 64, 640, 128, 1000, 2000)
    assert (p.s_q, p.h_q, p.topk, p.n_swa_cols, p.n_swa_rows, p.n_cmp_rows) == (4, 64, 640, 128, 1000, 2000)
    assert abs(p.softmax_scale - 1 / 24) < 1e-8 and p.rope_base == 10000.0 and abs(p.rms_eps - 1e-6) < 1e-12
    assert p.flags == 0
    assert lib.dsa_params_init(None, 1, 1, 1, 1, 1, 1) == native.DSA_ERR_INVALID_ARG


def test_error_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -99):
        assert len(native.dsa_error_string(code)) > 0


def test_split_heuristic_and_workspace_size(lib):
    p = native.dsa_params_init(1, 64, 640, 128, 8192, 65536)
    assert native.dsa_sparse_attn_num_splits(p, 152) == 5          # one 128-row tile per split
    # a work item is (token, half of the 64 heads): 64 tokens are 128 items on 152 SMs
    p = native.dsa_params_init(64, 64, 640, 128, 8192, 262144)
    assert native.dsa_sparse_attn_num_splits(p, 152) == 1
    p = native.dsa_params_init(64, 16, 640, 128, 8192, 262144)          # one half per token
    assert native.dsa_sparse_attn_num_splits(p, 152) == 2
    p = native.dsa_params_init(1024, 64, 640, 128, 131072, 1 << 20)
    assert native.dsa_sparse_attn_num_splits(p, 152) == 1
    ws1 = native.dsa_sparse_attn_workspace_size(p, 152)
    assert ws1 >= 256 + 4 * 1024 and ws1 % 256 == 0
    p = native.dsa_params_init(32, 64, 640, 128, 8192, 262144)
    assert native.dsa_sparse_attn_num_splits(p, 152) == 2
    ws2 = native.dsa_sparse_attn_workspace_size(p, 152)
    assert ws2 >= 32 * 2 * 64 * 512 * 4                              # per-split partial outputs
    bad = native.dsa_params_init(1, 65, 640, 128, 1, 1)
    assert native.dsa_sparse_attn_workspace_size(bad, 152) == 0


def test_every_split_path_shape_fits_the_no_alloc_scratch_on_152_sms(lib):
    # The split path holds (s_q x splits) fp32 partial outputs; its item count, and so
    # s_q x splits, is bounded by the SM count.  The largest such workspace on a 152-SM
    # GB300 (76 tokens of at most 32 heads, 2048 columns, 2 splits) must fit the built-in
    # scratch of the allocation-free entry point.
    worst = 0
    for h in (1, 16, 32, 33, 64):
        for topk in (129, 640, 2048):
            for s_q in range(1, 160):
                p = native.dsa_params_init(s_q, h, topk, 0, 1, 1)
                if native.dsa_sparse_attn_num_splits(p, 152) > 1:
                    worst = max(worst, native.dsa_sparse_attn_workspace_size(p, 152))
    assert 20 << 20 < worst <= native.DSA_NOALLOC_SCRATCH_BYTES


def _call(lib, p, **over):
    args = dict(q=16, kv_swa=16, kv_cmp=16, indices=16, topk_length=16, positions=16, norm_w=16, out_fp8=16,
                out_sf=16, ws=256, ws_bytes=1 << 30)
    args.update(over)
    return lib.dsa_sparse_attn_fwd(args["q"], args["kv_swa"], args["kv_cmp"], args["indices"], args["topk_length"],
                                   args["positions"], args["norm_w"], args["out_fp8"], args["out_sf"],
                                   ctypes.byref(p) if p is not None else None, args["ws"], args["ws_bytes"], None)


def test_argument_validation_happens_before_any_gpu_work(lib):
    ok = native.dsa_params_init(2, 64, 640, 128, 1000, 2000)
    assert _call(lib, None) == native.DSA_ERR_INVALID_ARG
    for field in ("q", "topk_length", "positions", "norm_w", "out_fp8", "out_sf", "ws", "indices", "kv_swa", "kv_cmp"):
        assert _call(lib, ok, **{field: None}) == native.DSA_ERR_INVALID_ARG, field
    assert _call(lib, ok, q=8) == native.DSA_ERR_INVALID_ARG          # q not 16-byte aligned
    assert _call(lib, ok, kv_cmp=24) == native.DSA_ERR_INVALID_ARG    # pool not 16-byte aligned
    assert _call(lib, ok, ws=128) == native.DSA_ERR_INVALID_ARG       # workspace not 256-byte aligned
    assert _call(lib, ok, out_fp8=2) == native.DSA_ERR_INVALID_ARG
    for h in (0, 65):
        p = native.dsa_params_init(2, h, 640, 128, 1000, 2000)
        assert _call(lib, p) == native.DSA_ERR_UNSUPPORTED_SHAPE
    p = native.dsa_params_init(2, 64, 4096, 128, 1000, 2000)
    assert _call(lib, p) == native.DSA_ERR_UNSUPPORTED_SHAPE
    p = native.dsa_params_init(2, 64, 640, 700, 1000, 2000)
    assert _call(lib, p) == native.DSA_ERR_INVALID_ARG                 # n_swa_cols > topk
    p = native.dsa_params_init(-1, 64, 640, 128, 1000, 2000)
    assert _call(lib, p) == native.DSA_ERR_INVALID_ARG
    p = native.dsa_params_init(2, 64, 640, 128, 1 << 31, 2000)
    assert _call(lib, p) == native.DSA_ERR_UNSUPPORTED_SHAPE
    p = native.dsa_params_init(2, 64, 640, 128, 1000, 2000, flags=32)
    assert _call(lib, p) == native.DSA_ERR_INVALID_ARG
    p = native.dsa_params_init(2, 64, 640, 128, 1000, 2000, softmax_scale=float("nan"))
    assert _call(lib, p) == native.DSA_ERR_INVALID_ARG
    # an empty batch is a no-op
    p = native.dsa_params_init(0, 64, 640, 128, 1000, 2000)
    assert _call(lib, p) == native.DSA_OK
    # swa-only / cmp-only shapes do not need the other pool
    p = native.dsa_params_init(2, 64, 640, 640, 1000, 0)
    assert _call(lib, p, kv_cmp=None, q=8) == native.DSA_ERR_INVALID_ARG   # fails on q, not on the missing pool


def test_cache_format_arguments(lib):
    # the two formats pass the argument check; an unknown format or a non-finite
    # compressed-pool scale does not (num_splits returns 0 on a bad argument)
    p = native.dsa_params_init(4, 64, 1024, 128, 512, 4096)
    assert p.kv_format == native.DSA_KV_FP8_DS_MLA and p.cmp_scale == 1.0
    p.kv_format = native.DSA_KV_NVFP4_DS_MLA
    assert native.dsa_sparse_attn_num_splits(p, 152) == 8
    for fmt in (2, -1):
        p.kv_format = fmt
        assert native.dsa_sparse_attn_num_splits(p, 152) == 0
    p.kv_format = native.DSA_KV_NVFP4_DS_MLA
    for bad in (float("nan"), float("inf"), float("-inf")):
        p.cmp_scale = bad
        assert native.dsa_sparse_attn_num_splits(p, 152) == 0
    p.cmp_scale = 0.0
    assert native.dsa_sparse_attn_num_splits(p, 152) == 8


def test_fp8_q_needs_the_fp8_ds_mla_cache(lib):
    p = native.dsa_params_init(4, 64, 1024, 128, 512, 4096, flags=native.DSA_FLAG_FP8_Q)
    assert native.dsa_sparse_attn_num_splits(p, 152) == 8
    p.kv_format = native.DSA_KV_NVFP4_DS_MLA
    assert native.dsa_sparse_attn_num_splits(p, 152) == 0
