// Top-k column selection of the indexer logits, feeding the sparse attention's index
// rows directly (vLLM PR #64364, DeepSeek-V4.1-Flash latency_specialized decode at TP4,
// Claims and Validation: the threshold is torch.topk's k-th value, every column above
// it is selected, ties at it go to the lowest-numbered columns, and the selected columns
// are listed in ascending order).
//
// One CTA of 512 threads per row.  The row's bf16 logits become 16-bit keys in shared
// memory whose unsigned order is the value order: every NaN maps to the largest key
// (torch.topk ranks NaN above +inf), and -0 maps to +0's key (equal values, equal keys).
// Two 8-bit radix-select passes find the k-th largest key T and the number of keys
// above it: a shared histogram (the first pass while the keys are written), then one
// warp's suffix scan over the 256 digits.  The
// row is then read as chunks of eight columns, one chunk per thread and round; a
// block-wide prefix of the chunks' counts above T and equal to T gives each chunk the
// number of columns selected before it: those above T, plus the equal ones up to
// `need`.  Each thread then writes its chunk's selected columns in order, so the output
// is ascending and the first `need` columns equal to T are the lowest-numbered.

#include <cuda_runtime.h>
#include <mutex>
#include <stdint.h>

#include "dsa_topk.h"

namespace dsa_topk {

constexpr int THREADS = 512;
constexpr int WARPS = THREADS / 32;

__device__ __forceinline__ uint32_t order_key(uint32_t b) {
  if ((b & 0x7F80u) == 0x7F80u && (b & 0x007Fu) != 0u) return 0xFFFFu;   // NaN, any sign or payload
  if (b == 0x8000u) b = 0u;                                              // -0 -> +0
  return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
}

// One warp: the digit b with above(b) < kk <= above(b) + hist[b], above(b) being the
// count of larger digits (1 <= kk <= the histogram's total).  Lane l holds digits
// 8l .. 8l + 7; a suffix sum over the lanes finds the one lane where the count crosses
// kk, and that lane scans its eight digits.
__device__ __forceinline__ void find_digit(const int* hist, int kk, int lane, int* out) {
  int h[8], tot = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    h[i] = hist[8 * lane + i];
    tot += h[i];
  }
  int suf = tot;   // count of digits >= 8 lane
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_down_sync(0xFFFFFFFFu, suf, o);
    if (lane + o < 32) suf += v;
  }
  int above = suf - tot;
  if (above < kk && kk <= suf) {
#pragma unroll
    for (int i = 7; i >= 0; --i) {
      if (above + h[i] >= kk) {
        out[0] = 8 * lane + i;
        out[1] = above;
        break;
      }
      above += h[i];
    }
  }
}

// Two 16-bit keys of one 32-bit word.
__device__ __forceinline__ uint32_t key_lo(uint32_t w2) { return w2 & 0xFFFFu; }
__device__ __forceinline__ uint32_t key_hi(uint32_t w2) { return w2 >> 16; }

__global__ void __launch_bounds__(THREADS, 4) topk_kernel(const uint16_t* __restrict__ logits, long long ld,
                                                       const int32_t* __restrict__ lengths, int n, int k,
                                                       int32_t* __restrict__ indices,
                                                       int32_t* __restrict__ topk_length) {
  extern __shared__ __align__(16) uint16_t s_key[];   // [n rounded up to 8]
  __shared__ int s_hist[256];
  __shared__ int s_wsum[WARPS];
  __shared__ int s_sel[2];
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
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
  for (int i = tid; i < 256; i += THREADS) s_hist[i] = 0;
  __syncthreads();
  // keys into shared memory, with the histogram of their high bytes (pass 1)
  const uint16_t* row = logits + t * ld;
  int j_vec = 0;
  if (((uintptr_t)row & 15) == 0) {
    // eight logits per 16-byte load, eight keys per 16-byte store
    j_vec = L & ~7;
    for (int j8 = tid; j8 < (L >> 3); j8 += THREADS) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(row) + j8);
      const uint32_t x[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t a = order_key(x[e] & 0xFFFFu), b = order_key(x[e] >> 16);
        o[e] = a | (b << 16);
        atomicAdd(&s_hist[a >> 8], 1);
        atomicAdd(&s_hist[b >> 8], 1);
      }
      reinterpret_cast<uint4*>(s_key)[j8] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
  for (int j = j_vec + tid; j < L; j += THREADS) {
    const uint32_t a = order_key(__ldg(row + j));
    s_key[j] = (uint16_t)a;
    atomicAdd(&s_hist[a >> 8], 1);
  }
  __syncthreads();
  if (w == 0) find_digit(s_hist, k, lane, s_sel);
  __syncthreads();
  const int hi = s_sel[0];
  const int above_hi = s_sel[1];
  __syncthreads();
  // pass 2: low byte, among the keys with that high byte (eight keys per 16-byte read)
  for (int i = tid; i < 256; i += THREADS) s_hist[i] = 0;
  __syncthreads();
  const int L8 = (L + 7) >> 3;
  for (int ci = tid; ci < L8; ci += THREADS) {
    const uint4 kv = reinterpret_cast<const uint4*>(s_key)[ci];
    const uint32_t x[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t key = (e & 1) ? key_hi(x[e >> 1]) : key_lo(x[e >> 1]);
      if (8 * ci + e < L && (int)(key >> 8) == hi) atomicAdd(&s_hist[key & 255], 1);
    }
  }
  __syncthreads();
  if (w == 0) find_digit(s_hist, k - above_hi, lane, s_sel);
  __syncthreads();
  const uint32_t T = (uint32_t)((hi << 8) | s_sel[0]);
  const int need = k - above_hi - s_sel[1];   // columns equal to T to take, lowest first
  // Output in column order.  Chunk ci (eight columns) belongs to thread ci % THREADS in
  // round ci / THREADS; per round a block-wide exclusive prefix of the chunks' counts
  // above T and equal to T (packed in one int: at most 8 x THREADS each) places them.
  int gt_base = 0, eq_base = 0;   // counts of earlier rounds
  for (int c0 = 0; c0 < L8; c0 += THREADS) {
    const int ci = c0 + tid;
    uint32_t x[4] = {0u, 0u, 0u, 0u};
    if (ci < L8) {
      const uint4 kv = reinterpret_cast<const uint4*>(s_key)[ci];
      x[0] = kv.x; x[1] = kv.y; x[2] = kv.z; x[3] = kv.w;
    }
    int gt = 0, eq = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t key = (e & 1) ? key_hi(x[e >> 1]) : key_lo(x[e >> 1]);
      const bool in = ci < L8 && 8 * ci + e < L;
      gt += (in && key > T) ? 1 : 0;
      eq += (in && key == T) ? 1 : 0;
    }
    const int packed = (gt << 16) | eq;
    int incl = packed;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) s_wsum[w] = incl;
    __syncthreads();
    int wbefore = 0, total = 0;
#pragma unroll
    for (int u = 0; u < WARPS; ++u) {
      const int sv = s_wsum[u];
      wbefore += u < w ? sv : 0;
      total += sv;
    }
    __syncthreads();   // s_wsum is rewritten by the next round
    const int excl = wbefore + incl - packed;
    int gtb = gt_base + (excl >> 16), eqb = eq_base + (excl & 0xFFFF);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t key = (e & 1) ? key_hi(x[e >> 1]) : key_lo(x[e >> 1]);
      const int col = 8 * ci + e;
      if (ci < L8 && col < L) {
        if (key > T) {
          const int pos = gtb + min(eqb, need);
          if (pos < k) out[pos] = col;
          ++gtb;
        } else if (key == T) {
          if (eqb < need && gtb + eqb < k) out[gtb + eqb] = col;
          ++eqb;
        }
      }
    }
    gt_base += total >> 16;
    eq_base += total & 0xFFFF;
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
  const size_t smem = (size_t)((n + 7) & ~7) * sizeof(uint16_t);
  topk_kernel<<<(unsigned)s_q, THREADS, smem, (cudaStream_t)stream>>>(
      (const uint16_t*)logits, (long long)ld, lengths, n, k, indices, topk_length);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
