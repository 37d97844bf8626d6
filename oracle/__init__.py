"""CPU oracle for fused top-k sparse latent attention (test infrastructure only).

This package is the slow, plain, float64 definition that the CUDA path is checked
against.  It is test infrastructure: only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg may import it.  The product path
(``top_sparse_mla_gb300``) never imports, links or calls anything here, and nothing
here imports the product path.  The two share only the seeded input generator
(``top_sparse_mla_gb300.workloads``), which holds none of the method's arithmetic.

Sources ("Deepseek V41 Attention MegaKernel", vLLM PR #56344, Purpose and
Performance sections): the fused kernel applies q norm, q RoPE, sparse attention over
the indexed sliding-window and compressed-cache rows (``-1`` sentinels skipped, reads
capped at ``topk_length``), inverse RoPE and an FP8 (MXFP8) cast, on the
``fp8_ds_mla`` cache format.

Modules:
  codecs      -- e4m3 / bf16 / fp32 / UE8M0 encodings written from their definitions
  sparse_mla  -- the forward pass, one token at a time, in float64
  brute       -- a scalar pure-Python restatement for tiny inputs (cross-check)
  topk        -- the index producer's top-k column selection (vLLM PR #64364, Claims
                 and Validation)
  kv_insert   -- the KV-cache insert: norm, RoPE and fp8_ds_mla quantisation of new rows
                 (vLLM PR #64364, "The changes and what each bought", Attention)
  nvfp4       -- the same attention on the nvfp4_ds_mla (V4.1) cache: 512-dim keys with
                 the rotary dims inside, fp8 and fp4 rows (vLLM PR #56344, Purpose)
"""

from . import codecs, sparse_mla, brute, topk, kv_insert, nvfp4  # noqa: F401
from .sparse_mla import (  # noqa: F401
    OracleParams,
    decode_kv_rows,
    mxfp8_cast,
    q_prologue,
    rmsnorm,
    rope_interleaved,
    sparse_mla_forward,
    valid_columns,
)
