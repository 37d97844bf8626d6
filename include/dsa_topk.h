/* Top-k column selection of the sparse indexer's logits, producing the sparse
 * attention's index rows directly.
 *
 * Defined by vLLM PR #64364 (DeepSeek-V4.1-Flash latency_specialized decode at TP4 on
 * GB300), Claims and Validation, for the `topk_bf16_small` producer. Per row t:
 *   - the candidates are the columns j < lengths[t] (all n columns when lengths is
 *     NULL; negative lengths count as 0, lengths above n as n);
 *   - the threshold is the k-th largest candidate value, the one torch.topk returns
 *     last; NaN (any sign or payload) ranks above +inf, and -0 equals +0;
 *   - every candidate above the threshold is selected, and among the candidates equal
 *     to it the lowest-numbered ones, until k are selected (all candidates if there
 *     are at most k);
 *   - the selected columns are written to indices[t][0..m) in ascending order, with
 *     m = min(k, candidates), and the rest of the row holds -1;
 *   - topk_length[t] = m.
 * This is the `indices` / `topk_length` form that dsa_sparse_attn_fwd reads.
 *
 * Arguments (device pointers, owned by the caller):
 *   logits      bf16  [s_q][ld], ld >= n, 2-byte aligned
 *   lengths     int32 [s_q], or NULL
 *   indices     int32 [s_q][k] (may be NULL when k == 0)
 *   topk_length int32 [s_q]
 *   1 <= n <= DSA_TOPK_MAX_COLS, 0 <= k <= DSA_TOPK_MAX_K, s_q >= 0.
 * The call is asynchronous on `stream` (a cudaStream_t, NULL = legacy default stream).
 * It allocates nothing, launches one kernel with one CTA per row, and can be captured
 * in a CUDA graph. It returns DSA_OK, or one of the following with nothing enqueued:
 *   - DSA_ERR_INVALID_ARG: a bad size, a null or misaligned pointer;
 *   - DSA_ERR_UNSUPPORTED_DEVICE: not compute capability 10.3, or a device ordinal >= DSA_MAX_DEVICES;
 *   - DSA_ERR_CUDA.
 */
#ifndef DSA_TOPK_H_
#define DSA_TOPK_H_

#include <stdint.h>

#include "dsa_sparse_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

#define DSA_TOPK_MAX_COLS 65536 /* a row's keys are held in shared memory, 2 bytes each */
#define DSA_TOPK_MAX_K 2048     /* the attention's DSA_MAX_TOPK */

int dsa_topk_select(const void* logits, int64_t ld, const int32_t* lengths, int32_t s_q, int32_t n, int32_t k,
                    int32_t* indices, int32_t* topk_length, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_TOPK_H_ */
