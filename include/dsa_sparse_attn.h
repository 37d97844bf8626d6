/*
 * dsa_sparse_attn.h -- C ABI of the fused top-k sparse latent-attention kernel for
 * NVIDIA GB300 (sm_103a).
 *
 * Operation: the stages that the Purpose section of "Deepseek V41 Attention MegaKernel"
 * (vLLM PR #56344) lists as fused, namely the query norm, RoPE, sparse attention,
 * inverse RoPE and an FP8 cast of the output.  For every query token t and head h:
 *   1. q~ = RMSNorm(q[t,h,:576]) * norm_w   (fp32 statistics, eps = rms_eps)
 *   2. RoPE on q~ dims 512..575: pairs (512+2i, 513+2i) rotated by
 *      positions[t] * rope_base^(-2i/64)
 *   3. valid columns j: j < topk_length[t] and indices[t,j] >= 0 (the page's sentinel
 *      fix: reads are capped at topk_length and -1 entries are never read); columns
 *      j < n_swa_cols read kv_swa[indices[t,j]], the others kv_cmp[indices[t,j]]
 *   4. k = dequantised 512 latent values ++ 64 rope values of the row, v = latent
 *   5. o = softmax_j(softmax_scale * q~.k_j) weighted sum of v_j  (o = 0 when no column
 *      is valid)
 *   6. inverse RoPE on o dims 448..511 (angle -positions[t] * theta_i)
 *   7. MXFP8 cast of o: per 32-value block along the 512 dims, UE8M0 scale code
 *      E + 127 with E = floor(log2(block amax)) - 8 clamped to [-127, 127] (0 for an
 *      all-zero block), values o / 2^E rounded to E4M3 (ties to even, saturating).
 *
 * Data layouts (all row-major, all pointers are DEVICE pointers owned by the caller;
 * the library never allocates, frees or retains them):
 *   q           bf16  [s_q, h_q, 576]                  16-byte aligned
 *   kv_swa      uint8 [n_swa_rows, 656] fp8_ds_mla rows 16-byte aligned
 *   kv_cmp      uint8 [n_cmp_rows, 656] fp8_ds_mla rows 16-byte aligned
 *               row = 512 E4M3 latent | 4 little-endian fp32 scales (one per 128
 *               latent values) | 64 bf16 rope values
 *   indices     int32 [s_q, topk]   (-1 or any negative value = skip)
 *   topk_length int32 [s_q]         (values <= 0 read nothing; values > topk read topk)
 *   positions   int32 [s_q]
 *   norm_w      bf16  [576]                              16-byte aligned
 *   out_fp8     uint8 [s_q, h_q, 512] E4M3 codes          16-byte aligned
 *   out_sf      uint8 [s_q, h_q, 16]  UE8M0 codes (or, with DSA_FLAG_SF_SWIZZLED, the
 *               same codes in the 128x4-tile layout described at that flag)
 *   out_precast fp32  [s_q, h_q, 512] (debug entry only; may be NULL) 16-byte aligned
 *   lse         fp32  [s_q, h_q] natural-log sum-exp of the scaled scores, -inf for
 *               a token with no valid column (debug entry only; may be NULL)
 *
 * Numerics: the contractions run on fp16 tensor-core MMAs with fp32 accumulation, and
 * every operand is exact in fp16 or split into an exact-enough fp16 hi + lo pair: the
 * E4M3 codes are exact in fp16 and the rows' fp32 block scales are applied in fp32 per
 * 128-value block; q * norm_w (exact in fp32) goes in as hi + lo with a per-head
 * power-of-two prescale; the softmax weights times each block's scales go in as hi + lo.
 * The pre-cast output then agrees with a float64 evaluation to about 1e-6 relative, for
 * any scaling of q, norm_w or a row's block scales.  Ranges: a rope key (bf16) must be
 * below 65504 in magnitude (it is converted to fp16); the E4M3 NaN code is not expected
 * in a referenced row.
 *
 * Calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy default stream),
 * allocate nothing, and enqueue two operations: a small memset or a one-CTA ordering
 * kernel, then the fused kernel (see dsa_sparse_attn_fwd).
 * Arguments are checked on the host before anything is enqueued; a non-zero
 * return means nothing was enqueued (DSA_ERR_CUDA: the launch itself failed).
 * An index >= its pool's row count is undefined behaviour unless
 * DSA_FLAG_CHECK_INDICES is set; then that column is skipped and the device status
 * word gets DSA_STATUS_INDEX_OUT_OF_RANGE (read it with dsa_sparse_attn_read_status).
 * Calls that share a workspace must not overlap on the GPU.
 */
#ifndef DSA_SPARSE_ATTN_H_
#define DSA_SPARSE_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSA_OK 0
#define DSA_ERR_INVALID_ARG (-1)         /* null/misaligned pointer, bad parameter */
#define DSA_ERR_UNSUPPORTED_SHAPE (-2)   /* h_q outside [1,64], topk > DSA_MAX_TOPK, ... */
#define DSA_ERR_WORKSPACE_TOO_SMALL (-3)
#define DSA_ERR_CUDA (-4)                /* CUDA runtime error (launch, attribute, memset) */
#define DSA_ERR_UNSUPPORTED_DEVICE (-5)  /* current device is not compute capability 10.3 */
#define DSA_ERR_SCRATCH_LIMIT (-6)       /* shape needs more than DSA_NOALLOC_SCRATCH_BYTES */

#define DSA_FLAG_CHECK_INDICES 1u        /* bounds-check every index against its pool */
/* For tests of the failure path only: in CTA 0 the warp that publishes items first waits
 * on an on-chip barrier that nothing completes.  That wait runs out after its bound
 * (about 2 s), the CTA sets DSA_STATUS_WAIT_TIMEOUT, and every role of the CTA stops,
 * drains the tensor core and frees its tensor memory, so the context stays usable.
 * Without splits CTA 0 takes no item, and the other CTAs compute every output.  With
 * splits (dsa_sparse_attn_num_splits > 1) token 0's first split is never computed:
 * its other splits give up their bounded wait for it (also DSA_STATUS_WAIT_TIMEOUT),
 * so token 0's output is left unwritten, and the other tokens are complete. */
#define DSA_FLAG_TEST_WAIT_TIMEOUT 2u
/* Launch after a producer kernel without a gap: the call's first kernel (the queue
 * order kernel; the queue path is taken without splits and up to DSA_ORDER_MAX_TOKENS
 * tokens) is launched as a programmatic dependent of the kernel enqueued just before
 * it on `stream`, for example dsa_kv_insert or dsa_topk_select, which let their
 * dependents launch early.  It starts while that kernel is still running and waits for
 * its completion (griddepcontrol.wait) before it reads anything, so every input the
 * producer writes (pool rows, indices, lengths) is complete before it is read.  On the
 * split path, and in dsa_sparse_attn_fwd_noalloc, the workspace is cleared by a memset
 * first, which orders the call after the producer as usual; the flag then changes
 * nothing. */
#define DSA_FLAG_AFTER_PRODUCER 4u
/* Write out_sf in FlashInfer's 128x4 swizzled scale-factor layout, the one an MXFP8
 * GEMM reading the output as an [s_q, 512 h_q] matrix takes ("[DSV4.1] Combine DSpark
 * decode and prefill kernel optimizations", SGLang PR #39370, the mHC MXFP8 epilogue
 * paragraph, names the layout; the byte order below is this library's reading of it).
 * The scale matrix has M = s_q rows (tokens) and K = 16 h_q columns (column
 * k = 16 h + b for head h and 32-dim block b).  It is stored as 128 x 4 tiles of 512
 * bytes, tiles in row-major order (ceil(s_q / 128) tile rows of 4 h_q tiles); inside a
 * tile, entry (m, k) is at byte (m % 32) * 16 + ((m / 32) % 4) * 4 + (k % 4).  So the
 * byte offset of (m, k) is
 *     ((m / 128) * 4 h_q + k / 4) * 512 + (m % 32) * 16 + ((m / 32) % 4) * 4 + k % 4,
 * and out_sf must hold DSA_SF_SWIZZLED_BYTES(s_q, h_q) bytes.  The bytes of rows
 * m >= s_q (the last tile row's padding) are not written.  The codes themselves, and
 * every other output, are those of the row-major layout. */
#define DSA_FLAG_SF_SWIZZLED 8u
/* Quantise q's latent part to E4M3 inside the kernel before QK^T, the "query FP8
 * quantization inside the sparse-MLA kernel" of "DSV4.1 latency_specialized decode at
 * TP4 on GB300" (vLLM PR #64364, "The changes and what each bought", Attention row);
 * the rule is this library's reading.  Per token and head, over the 512 latent dims:
 * amax = max |q * norm_w| and code = E4M3(fl(q * norm_w) * fl(448 / amax)), round to
 * nearest even, saturating, every step in binary32 (q * norm_w is exact).  This is the
 * RMSNorm'd latent divided by its scale s = amax * rms_inv / 448 (the RMS factor
 * cancels), and the latent part of q~ is then code * s.  The rope dims stay as without
 * the flag (the keys' rope part is bf16).  Everything else is unchanged, so the result is
 * step 5 on that q~.  Only with DSA_KV_FP8_DS_MLA (DSA_ERR_INVALID_ARG otherwise). */
#define DSA_FLAG_FP8_Q 16u
#define DSA_SF_SWIZZLED_BYTES(s_q, h_q) ((((size_t)(s_q) + 127) / 128) * 128 * 16 * (size_t)(h_q))

#define DSA_STATUS_INDEX_OUT_OF_RANGE 1u /* an index was >= its pool size (with the flag) */
#define DSA_STATUS_WAIT_TIMEOUT 2u       /* an on-chip pipeline wait gave up; output invalid */

#define DSA_MAX_HEADS 64
#define DSA_MAX_DEVICES 64 /* device ordinals >= this return DSA_ERR_UNSUPPORTED_DEVICE */
#define DSA_MAX_TOPK 2048
#define DSA_ORDER_MAX_TOKENS 65536 /* above this the queue takes tokens in index order */
#define DSA_ROW_BYTES 656

/* Cache formats (dsa_params.kv_format).
 *
 * DSA_KV_FP8_DS_MLA: the layout described at the top of this file (576-dim keys, q and
 * norm_w of 576, 656-byte rows in both pools).
 *
 * DSA_KV_NVFP4_DS_MLA: the V4.1 cache that "Deepseek V41 Attention MegaKernel" (vLLM PR
 * #56344, Purpose) adds as nvfp4_ds_mla, "V4.1 fp8 528 B SWA + V4.1 fp4 288 B
 * compressed".  The page gives the two row sizes only; the byte layout below is this
 * library's reading.  Keys are 512 dims with the 64 rotary dims inside (dims 448..511,
 * stored already rotated), and v = k: the 512 output dims are the keys' dims, which is
 * why the output's dims 448..511 get the inverse RoPE.  So q and norm_w have 512 dims
 * (q RMSNorm over the 512, RoPE on q dims 448..511 with the same pair convention),
 * s_j = softmax_scale * q~ . k_j (softmax_scale is still the caller's, e.g.
 * 1/sqrt(512)), and steps 5-7 are unchanged.
 *   kv_swa row, 528 bytes: 512 E4M3 values | 4 little-endian fp32 scales, scale g
 *     for dims [128g, 128g + 128).
 *   kv_cmp row, 288 bytes (NVFP4): 512 E2M1 values, two per byte (dim 2i in the low
 *     nibble of byte i) | 32 E4M3 scales, scale i for dims [16i, 16i + 16).  The value
 *     of dim d is e2m1 * e4m3 scale * cmp_scale.
 * Rows are 16-byte aligned (528 = 33 * 16, 288 = 18 * 16). */
#define DSA_KV_FP8_DS_MLA 0
#define DSA_KV_NVFP4_DS_MLA 1
#define DSA_NVFP4_QK_DIMS 512
#define DSA_NVFP4_SWA_ROW_BYTES 528
#define DSA_NVFP4_CMP_ROW_BYTES 288
#define DSA_NOALLOC_SCRATCH_BYTES (24u << 20) /* built-in scratch of the no-alloc entry */

typedef struct dsa_params {
  int32_t s_q;          /* query tokens (>= 0) */
  int32_t h_q;          /* query heads, 1..64, sharing one latent KV head */
  int32_t topk;         /* index columns per token, 0..DSA_MAX_TOPK */
  int32_t n_swa_cols;   /* columns [0, n_swa_cols) index kv_swa, [n_swa_cols, topk) kv_cmp */
  int64_t n_swa_rows;   /* rows in kv_swa (< 2^31) */
  int64_t n_cmp_rows;   /* rows in kv_cmp (< 2^31) */
  float softmax_scale;  /* e.g. 1/sqrt(576) */
  float rope_base;      /* e.g. 10000 */
  float rms_eps;        /* e.g. 1e-6 */
  uint32_t flags;       /* DSA_FLAG_* */
  int32_t kv_format;    /* DSA_KV_FP8_DS_MLA or DSA_KV_NVFP4_DS_MLA (see below) */
  float cmp_scale;      /* DSA_KV_NVFP4_DS_MLA: fp32 scale of every kv_cmp value, finite */
} dsa_params;

/* Fill `p` with the defaults above for the given shape (softmax_scale 1/sqrt(576),
 * rope_base 10000, rms_eps 1e-6, flags 0, kv_format DSA_KV_FP8_DS_MLA, cmp_scale 1).
 * Returns DSA_OK or DSA_ERR_INVALID_ARG. */
int dsa_params_init(dsa_params* p, int32_t s_q, int32_t h_q, int32_t topk, int32_t n_swa_cols,
                    int64_t n_swa_rows, int64_t n_cmp_rows);

/* Bytes of device workspace the forward call needs for `p` on a GPU with `num_sms`
 * SMs (num_sms <= 0: the current device).  The workspace holds a status word and a
 * queue head, one int32 per token (a combine counter on the split path, the queue's
 * token order otherwise), the compacted row lists of every CTA and, when a token's rows
 * are split across several CTAs, the per-split partial outputs.  0 is returned for
 * invalid parameters. */
size_t dsa_sparse_attn_workspace_size(const dsa_params* p, int num_sms);

/* The fused forward pass (steps 1-7), enqueued on `stream`; everything it enqueues can
 * be captured in a CUDA graph.  A work item is one token's heads 0..31 or 32..63 (one
 * item per token when h_q <= 32), or a KV split of that.
 * - When the tokens are few (dsa_sparse_attn_num_splits > 1), each CTA takes one
 *   (token, heads, split) item. The call clears the workspace header and the combine counters
 *   with an async memset. The fused kernel's launch is then cooperative, so that the
 *   splits of a token can wait for one another before each combines its share of the
 *   partial outputs; the grid is at most one CTA per SM.
 * - Otherwise the CTAs (at most one per SM) take tokens from one queue. With at most
 *   DSA_ORDER_MAX_TOKENS tokens, a one-CTA kernel first clears the header and orders
 *   the queue: tokens with the most 128-row tiles (from topk_length) come first, equal
 *   counts in token order. The fused kernel is launched as its programmatic dependent.
 *   With more tokens, a memset clears the header and tokens go in index order.
 * The order decides which CTA computes a token, never the token's result. */
int dsa_sparse_attn_fwd(const void* q, const void* kv_swa, const void* kv_cmp,
                        const int32_t* indices, const int32_t* topk_length,
                        const int32_t* positions, const void* norm_w,
                        void* out_fp8, uint8_t* out_sf, const dsa_params* p,
                        void* workspace, size_t workspace_bytes, void* stream);

/* Same computation; additionally writes the pre-cast fp32 output (after inverse
 * RoPE) and the LSE when the pointers are non-NULL. */
int dsa_sparse_attn_fwd_debug(const void* q, const void* kv_swa, const void* kv_cmp,
                              const int32_t* indices, const int32_t* topk_length,
                              const int32_t* positions, const void* norm_w,
                              void* out_fp8, uint8_t* out_sf, float* out_precast, float* lse,
                              const dsa_params* p, void* workspace, size_t workspace_bytes,
                              void* stream);

/* Waits for `stream`, then copies the device status word (DSA_STATUS_* bits of the
 * last call that used `workspace`) into *status.  Returns DSA_OK or an error code. */
int dsa_sparse_attn_read_status(const void* workspace, uint32_t* status, void* stream);

/* Allocation-free variant of dsa_sparse_attn_fwd (the pages describe no such entry
 * point; it exists for the library's callers).  Some callers cannot hand the kernel a
 * workspace: serving engines that reserve almost all HBM for the KV pools at start-up
 * and run on a fixed memory plan, plug-in hosts that pass a kernel its tensors and
 * nothing else, and per-step code that must not call cudaMalloc or cudaFree because
 * those synchronise the device.  This entry point uses instead a scratch array of
 * DSA_NOALLOC_SCRATCH_BYTES (24 MiB) compiled into the library as a __device__
 * variable: it calls no allocator of any kind.
 *   - Same arguments and results as dsa_sparse_attn_fwd, without workspace and
 *     workspace_bytes.  The split count and the kernel are the same.
 *   - The first call on each device (that device current) looks up the scratch
 *     address with cudaGetSymbolAddress; make that first call before any stream
 *     capture.
 *   - Loading the library reserves the scratch on every device where the module is
 *     loaded, whichever entry point the caller uses.
 *   - The scratch covers every shape whose workspace (dsa_sparse_attn_workspace_size)
 *     is at most DSA_NOALLOC_SCRATCH_BYTES: on a 152-SM GB300 any shape with
 *     s_q <= 2500000 (5000000 with h_q <= 32).  The workspace holds 4 bytes per token
 *     and head half, 32 KB of row lists per SM
 *     and, on the split path, 128 KB of fp32 partial output per (token, split); the
 *     split path runs at most one item per SM, so its partials stay below
 *     SMs x 128 KB (about 24.9 MB in all on 152 SMs, inside the scratch; a part with
 *     more SMs could exceed it).  Larger shapes return DSA_ERR_SCRATCH_LIMIT with
 *     nothing enqueued.
 *   - The scratch header is cleared on `stream` before each launch.
 *   - All calls on one device share the one scratch array: calls that overlap on the
 *     GPU (different streams, not ordered by events) race and give undefined results.
 *   - status_out (device pointer, 4-byte aligned, may be NULL) receives the call's
 *     DSA_STATUS_* word, copied on `stream` after the kernel. */
int dsa_sparse_attn_fwd_noalloc(const void* q, const void* kv_swa, const void* kv_cmp,
                                const int32_t* indices, const int32_t* topk_length,
                                const int32_t* positions, const void* norm_w,
                                void* out_fp8, uint8_t* out_sf, const dsa_params* p,
                                uint32_t* status_out, void* stream);

/* Split count the forward call uses for a shape (exposed for tests and tooling). */
int dsa_sparse_attn_num_splits(const dsa_params* p, int num_sms);

/* Static description of an error code. */
const char* dsa_error_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* DSA_SPARSE_ATTN_H_ */
