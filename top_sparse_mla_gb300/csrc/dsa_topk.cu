// Top-k column selection of the indexer logits, feeding the sparse attention's index
// rows directly (vLLM PR #64364, DeepSeek-V4.1-Flash latency_specialized decode at TP4,
// Claims and Validation: the threshold is torch.topk's k-th value, every column above
// it is selected, ties at it go to the lowest-numbered columns, and the selected columns
// are listed in ascending order).
//
// One CTA per row.  The row's bf16 logits become 16-bit keys in shared memory whose
// unsigned order is the value order: every NaN maps to the largest key (torch.topk
// ranks NaN above +inf), and -0 maps to +0's key (equal values, equal keys).  Two 8-bit
// radix-select passes find the k-th largest key T and the number of keys above it.  An
// ordered compaction over the columns then writes every column above T and the first
// `need` columns equal to T, in ascending order.

#include <cuda_runtime.h>
#include <stdint.h>

#include "dsa_topk.h"

namespace dsa_topk {

constexpr int THREADS = 1024;
constexpr int WARPS = THREADS / 32;

__device__ __forceinline__ uint32_t order_key(uint32_t b) {
  if ((b & 0x7F80u) == 0x7F80u && (b & 0x007Fu) != 0u) return 0xFFFFu;   // NaN, any sign or payload
  if (b == 0x8000u) b = 0u;                                              // -0 -> +0
  return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
}

// Exclusive block-wide count of `v` over the threads in order; `total` gets the sum.
// Every thread of the block calls it (it holds two barriers).
__device__ __forceinline__ int block_excl_count(bool v, int* s_warp, int& total) {
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const unsigned bal = __ballot_sync(0xFFFFFFFFu, v);
  const int in_warp = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) s_warp[w] = __popc(bal);
  __syncthreads();
  if (w == 0) {
    const int x = s_warp[lane];   // WARPS == 32: one entry per lane
    int incl = x;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
      if (lane >= d) incl += y;
    }
    s_warp[32 + lane] = incl - x;
    if (lane == 31) s_warp[64] = incl;
  }
  __syncthreads();
  total = s_warp[64];
  const int r = s_warp[32 + w] + in_warp;
  __syncthreads();   // s_warp is reused by the next call
  return r;
}

__global__ void __launch_bounds__(THREADS, 1) topk_kernel(const uint16_t* __restrict__ logits, long long ld,
                                                          const int32_t* __restrict__ lengths, int n, int k,
                                                          int32_t* __restrict__ indices,
                                                          int32_t* __restrict__ topk_length) {
  extern __shared__ uint16_t s_key[];   // [n]
  __shared__ int s_hist[256];
  __shared__ int s_warp[65];
  __shared__ int s_sel[2];
  static_assert(WARPS == 32, "one warp total per lane of warp 0");
  const int tid = threadIdx.x;
  const long long t = blockIdx.x;
  int L = n;
  if (lengths) {
    const int l = lengths[t];
    L = l < 0 ? 0 : (l > n ? n : l);
  }
  int32_t* out = indices + t * (long long)k;
  if (L <= k) {
    // every candidate column is selected: 0..L-1, then the -1 sentinel
    for (int j = tid; j < k; j += THREADS) out[j] = j < L ? j : -1;
    if (tid == 0) topk_length[t] = L;
    return;
  }
  // k < L from here (so k >= 0 and L >= 1)
  if (k == 0) {
    if (tid == 0) topk_length[t] = 0;
    return;
  }
  const uint16_t* row = logits + t * ld;
  for (int j = tid; j < L; j += THREADS) s_key[j] = (uint16_t)order_key(row[j]);
  // pass 1: high byte of the k-th largest key
  for (int i = tid; i < 256; i += THREADS) s_hist[i] = 0;
  __syncthreads();
  for (int j = tid; j < L; j += THREADS) atomicAdd(&s_hist[s_key[j] >> 8], 1);
  __syncthreads();
  if (tid == 0) {
    int above = 0, b = 255;
    for (; b > 0; --b) {
      if (above + s_hist[b] >= k) break;
      above += s_hist[b];
    }
    s_sel[0] = b;
    s_sel[1] = above;
  }
  __syncthreads();
  const int hi = s_sel[0];
  const int above_hi = s_sel[1];
  __syncthreads();
  // pass 2: low byte, among the keys with that high byte
  for (int i = tid; i < 256; i += THREADS) s_hist[i] = 0;
  __syncthreads();
  for (int j = tid; j < L; j += THREADS) {
    const int key = s_key[j];
    if ((key >> 8) == hi) atomicAdd(&s_hist[key & 255], 1);
  }
  __syncthreads();
  if (tid == 0) {
    int above = above_hi, b = 255;
    for (; b > 0; --b) {
      if (above + s_hist[b] >= k) break;
      above += s_hist[b];
    }
    s_sel[0] = b;
    s_sel[1] = above;
  }
  __syncthreads();
  const int T = (hi << 8) | s_sel[0];
  const int need = k - s_sel[1];   // columns equal to T to take, lowest first
  // ordered compaction: columns above T, and the first `need` columns equal to T
  int written = 0, eq_seen = 0;
  for (int c0 = 0; c0 < L; c0 += THREADS) {
    const int j = c0 + tid;
    const int key = j < L ? (int)s_key[j] : -1;
    const bool eq = key == T;
    int eq_total;
    const int eq_rank = eq_seen + block_excl_count(eq, s_warp, eq_total);
    const bool sel = key > T || (eq && eq_rank < need);
    int sel_total;
    const int pos = written + block_excl_count(sel, s_warp, sel_total);
    if (sel && pos < k) out[pos] = j;
    written += sel_total;
    eq_seen += eq_total;
  }
  if (tid == 0) topk_length[t] = k;
}

static bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace dsa_topk

extern "C" int dsa_topk_select(const void* logits, int64_t ld, const int32_t* lengths, int32_t s_q, int32_t n,
                               int32_t k, int32_t* indices, int32_t* topk_length, void* stream) {
  using namespace dsa_topk;
  if (s_q < 0 || n < 1 || n > DSA_TOPK_MAX_COLS || k < 0 || k > DSA_TOPK_MAX_K || ld < n)
    return DSA_ERR_INVALID_ARG;
  if (s_q == 0) return DSA_OK;
  if (!logits || !topk_length || (k > 0 && !indices)) return DSA_ERR_INVALID_ARG;
  if (!aligned(logits, 2) || !aligned(topk_length, 4) || (indices && !aligned(indices, 4)) ||
      (lengths && !aligned(lengths, 4)))
    return DSA_ERR_INVALID_ARG;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) return DSA_ERR_UNSUPPORTED_DEVICE;
  static int attr_done[64] = {0};
  if (dev < 64 && !attr_done[dev]) {
    if (cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(DSA_TOPK_MAX_COLS * sizeof(uint16_t))) != cudaSuccess)
      return DSA_ERR_CUDA;
    attr_done[dev] = 1;
  }
  const size_t smem = (size_t)n * sizeof(uint16_t);
  topk_kernel<<<(unsigned)s_q, THREADS, smem, (cudaStream_t)stream>>>(
      (const uint16_t*)logits, (long long)ld, lengths, n, k, indices, topk_length);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
