// Top-k column selection of the indexer logits, feeding the sparse attention's index
// rows directly (vLLM PR #64364, DeepSeek-V4.1-Flash latency_specialized decode at TP4,
// Claims and Validation: the threshold is torch.topk's k-th value, every column above
// it is selected, ties at it go to the lowest-numbered columns, and the selected columns
// are listed in ascending order).
//
// One CTA per row.  The row's bf16 logits become 16-bit keys in shared memory whose
// unsigned order is the value order: every NaN maps to the largest key (torch.topk
// ranks NaN above +inf), and -0 maps to +0's key (equal values, equal keys).  Two 8-bit
// radix-select passes find the k-th largest key T and the number of keys above it.  The
// row is then cut into 32 contiguous segments, one per warp.  Each warp counts its keys
// above T and equal to T (ballots, no block barrier).  One prefix over the warps gives
// each warp the number of columns selected before its segment: those above T, plus the
// equal ones up to `need`.  Each warp then writes its selected columns in order, so the
// output is ascending and the first `need` columns equal to T are the lowest-numbered.

#include <cuda_runtime.h>
#include <mutex>
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

__global__ void __launch_bounds__(THREADS, 1) topk_kernel(const uint16_t* __restrict__ logits, long long ld,
                                                          const int32_t* __restrict__ lengths, int n, int k,
                                                          int32_t* __restrict__ indices,
                                                          int32_t* __restrict__ topk_length) {
  extern __shared__ uint16_t s_key[];   // [n]
  __shared__ int s_hist[256];
  __shared__ int s_gt[WARPS], s_eq[WARPS];
  __shared__ int s_sel[2];
  static_assert(WARPS == 32, "one warp count per lane");
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const unsigned lt = (1u << lane) - 1u;
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
  // segment of warp w: columns [c_begin, c_end), a multiple of 32 long
  const int seg = ((L + THREADS - 1) / THREADS) * 32;
  const int c_begin = w * seg;
  const int c_end = min(c_begin + seg, L);
  int gt = 0, eq = 0;
  for (int c = c_begin; c < c_end; c += 32) {
    const int j = c + lane;
    const int key = j < c_end ? (int)s_key[j] : -1;
    gt += __popc(__ballot_sync(0xFFFFFFFFu, key > T));
    eq += __popc(__ballot_sync(0xFFFFFFFFu, key == T));
  }
  if (lane == 0) {
    s_gt[w] = gt;
    s_eq[w] = eq;
  }
  __syncthreads();
  // columns before this segment: above T, and equal to T
  const int gt_before = __reduce_add_sync(0xFFFFFFFFu, lane < w ? s_gt[lane] : 0);
  const int eq_before = __reduce_add_sync(0xFFFFFFFFu, lane < w ? s_eq[lane] : 0);
  int eq_run = eq_before;
  int sel_run = gt_before + min(eq_before, need);
  for (int c = c_begin; c < c_end; c += 32) {
    const int j = c + lane;
    const int key = j < c_end ? (int)s_key[j] : -1;
    const bool e = key == T;
    const unsigned be = __ballot_sync(0xFFFFFFFFu, e);
    const bool sel = key > T || (e && eq_run + __popc(be & lt) < need);
    const unsigned bs = __ballot_sync(0xFFFFFFFFu, sel);
    const int pos = sel_run + __popc(bs & lt);
    if (sel && pos < k) out[pos] = j;
    eq_run += __popc(be);
    sel_run += __popc(bs);
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
  if (dev < 0 || dev >= DSA_MAX_DEVICES) return DSA_ERR_UNSUPPORTED_DEVICE;
  {
    // the kernel's dynamic shared-memory limit, raised once per device (any host thread
    // may make the first call)
    static std::mutex attr_mutex;
    static bool attr_done[DSA_MAX_DEVICES];
    std::lock_guard<std::mutex> lock(attr_mutex);
    if (!attr_done[dev]) {
      if (cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)(DSA_TOPK_MAX_COLS * sizeof(uint16_t))) != cudaSuccess)
        return DSA_ERR_CUDA;
      attr_done[dev] = true;
    }
  }
  const size_t smem = (size_t)n * sizeof(uint16_t);
  topk_kernel<<<(unsigned)s_q, THREADS, smem, (cudaStream_t)stream>>>(
      (const uint16_t*)logits, (long long)ld, lengths, n, k, indices, topk_length);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
