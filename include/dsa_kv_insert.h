/* KV-cache insert: the new tokens' KV vectors, RMS-normalised, roped and quantised into
 * fp8_ds_mla rows of a cache pool, in one kernel.
 *
 * Defined by vLLM PR #64364 (DeepSeek-V4.1-Flash latency_specialized decode at TP4),
 * the table "The changes and what each bought", Attention row: the KV cache write is done
 * inside the Q/KV norm-quant kernel (its Limitations section names it the norm's KV
 * write).  The page gives no formula; the reading (a KV projection's standard form, in
 * the row format dsa_sparse_attn_fwd reads):
 *
 * For each new token i with slots[i] >= 0, with x = kv[i][0..512) (latent) and
 * r = kv[i][512..576) (rotary), both bf16:
 *   - y = x / sqrt(mean(x^2) + rms_eps) * kv_norm_w, over the 512 latent dims, with
 *     fp32 statistics (the rotary dims are not normalised);
 *   - per 128-dim block b: s_b = max|y_b| / 448 in fp32 (1 for an all-zero block), and
 *     the E4M3 code of each value is round-to-nearest-even of (x*w) * (448 / m_b),
 *     m_b = max_b|x*w|, in binary32: one rounded quotient per block and one rounded
 *     product per value (x*w and m_b are exact in binary32; in exact arithmetic this is
 *     y / s_b, here without the rounding of the RMS factor);
 *   - r rotated by positions[i] * rope_base^(-2j/64) on the interleaved pairs
 *     (2j, 2j + 1), as the attention rotates q, then rounded to bf16 (nearest even);
 *   - row slots[i] of `pool` := the 512 codes, the 4 scales s_b (fp32, little-endian),
 *     the 64 rotated bf16 values (DSA_ROW_BYTES = 656 bytes).
 * A token with slots[i] < 0 is skipped (padding); no other byte of the pool is written.
 * Inputs are finite bf16 values; non-finite ones give unspecified rows.  Two tokens
 * with the same slot leave one of their rows, unspecified which.
 *
 * Arguments (device pointers, owned by the caller):
 *   kv          bf16  [s_new][ld], ld >= 576, ld % 8 == 0, 16-byte aligned
 *   positions   int32 [s_new]
 *   slots       int64 [s_new]: the pool row of each token, < 0 = skip
 *   kv_norm_w   bf16  [512], 16-byte aligned
 *   pool        uint8 [n_rows][656], 16-byte aligned
 *   status      uint32 (device, 4-byte aligned) or NULL: with DSA_KV_FLAG_CHECK_SLOTS a
 *               slot >= n_rows is skipped and DSA_STATUS_SLOT_OUT_OF_RANGE is OR-ed
 *               into *status (the caller clears it); without the flag such a slot is
 *               undefined behaviour
 *   s_new >= 0, n_rows >= 0, rms_eps >= 0, rope_base > 0.
 * The call is asynchronous on `stream` (a cudaStream_t, NULL = legacy default stream),
 * allocates nothing, launches one kernel (one warp per token), and can be captured in a
 * CUDA graph.  It returns DSA_OK, or one of the following with nothing enqueued:
 *   - DSA_ERR_INVALID_ARG: a bad size or parameter, a null or misaligned pointer;
 *   - DSA_ERR_UNSUPPORTED_DEVICE: not compute capability 10.3;
 *   - DSA_ERR_CUDA.
 */
#ifndef DSA_KV_INSERT_H_
#define DSA_KV_INSERT_H_

#include <stdint.h>

#include "dsa_sparse_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

#define DSA_KV_FLAG_CHECK_SLOTS 1u         /* bounds-check every slot against n_rows */
#define DSA_STATUS_SLOT_OUT_OF_RANGE 4u    /* a slot was >= n_rows (with the flag) */

int dsa_kv_insert(const void* kv, int64_t ld, const int32_t* positions, const int64_t* slots, int32_t s_new,
                  const void* kv_norm_w, float rms_eps, float rope_base, void* pool, int64_t n_rows,
                  uint32_t flags, uint32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_KV_INSERT_H_ */
