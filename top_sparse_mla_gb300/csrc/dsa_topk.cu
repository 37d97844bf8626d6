// Top-k column selection of the indexer logits, feeding the sparse attention's index
// rows directly (vLLM PR #64364, DeepSeek-V4.1-Flash latency_specialized decode at TP4,
// Claims and Validation: the threshold is torch.topk's k-th value, every column above
// it is selected, ties at it go to the lowest-numbered columns, and the selected columns
// are listed in ascending order).
//
// One CTA per row.  The row's bf16 logits become 16-bit keys whose unsigned order is the
// value order: every NaN maps to the largest key (torch.topk ranks NaN above +inf), and
// -0 maps to +0's key (equal values, equal keys).  Two 8-bit radix-select passes find the
// k-th largest key T and the number of keys above it: a shared histogram of the high
// bytes, one warp's suffix scan over the 256 digits, then the same over the low bytes of
// the keys in the chosen high-byte bin.
//
// Rows of up to 8192 columns (the register path): 256 threads, each holding the keys of
// 32 consecutive columns in registers.  After the passes each thread has one bit mask of
// its columns above T and one of those equal to T; a block-wide exclusive prefix of the
// packed counts gives each thread the number of columns selected before its own (those
// above T, plus the equal ones up to `need`), and it writes its selected columns in
// order, so the output is ascending and the first `need` columns equal to T are the
// lowest-numbered.
//
// Longer rows (up to 65536 columns): 512 threads, the keys in shared memory, the same two
// passes, and the placement taken in rounds of 512 chunks of eight columns.

#include <cuda_runtime.h>
#include <mutex>
#include <stdint.h>

#include "dsa_topk.h"

namespace dsa_topk {

constexpr int THREADS = 512;
constexpr int WARPS = THREADS / 32;
// the register path: RT threads of RK columns each, RB CTAs per SM
constexpr int RT = 256, RK = 32, RB = 4;

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
  // a dependent launched with programmatic serialization (the attention with
  // DSA_FLAG_AFTER_PRODUCER) may start now; it waits for this kernel before reading
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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

// Keys of the two bf16 values of one 32-bit word at once (the same map as order_key):
// the sign selects XOR 0xFFFF or 0x8000 per half; -0 then reads 0x7FFF and is moved to
// +0's 0x8000; a NaN half (magnitude bits above 0x7F80) becomes 0xFFFF.
__device__ __forceinline__ uint32_t order_key2(uint32_t x) {
  const uint32_t s = (x >> 15) & 0x00010001u;
  uint32_t kk = x ^ (s * 0x7FFFu | 0x80008000u);
  // -0 came out as 0x7FFF (no other value does): +0's key
  if ((kk & 0xFFFFu) == 0x7FFFu) kk += 1u;
  if ((kk >> 16) == 0x7FFFu) kk += 0x10000u;
  // NaN (|bits| above 0x7F80) -> 0xFFFF
  const uint32_t nan = ((x & 0x7FFF7FFFu) + 0x007F007Fu) & 0x80008000u;
  return kk | ((nan >> 15) * 0xFFFFu);
}

// Register path (n <= NT * KPT): thread i owns columns KPT i .. KPT i + KPT - 1 and keeps
// their keys in registers, one per register.
template <int NT, int KPT, int MINB>
__global__ void __launch_bounds__(NT, MINB) topk_reg_kernel(const uint16_t* __restrict__ logits, long long ld,
                                                          const int32_t* __restrict__ lengths, int n, int k,
                                                          int32_t* __restrict__ indices,
                                                          int32_t* __restrict__ topk_length) {
  static_assert(KPT <= 32 && KPT % 8 == 0, "one 32-bit mask per thread; whole 16-byte loads");
  static_assert(NT >= 256 && NT <= 1024 && NT % 32 == 0, "one thread per histogram bin when clearing");
  constexpr int NWARP = NT / 32;
  __shared__ int s_hist[2][256];
  __shared__ int s_wsum[NWARP];
  __shared__ int s_sel[4];
  // a dependent launched with programmatic serialization (the attention with
  // DSA_FLAG_AFTER_PRODUCER) may start now; it waits for this kernel before reading
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const long long t = blockIdx.x;
  int L = n;
  if (lengths) {
    const int l = lengths[t];
    L = l < 0 ? 0 : (l > n ? n : l);
  }
  int32_t* out = indices + t * (long long)k;
  if (L <= k) {
    for (int j = tid; j < k; j += NT) out[j] = j < L ? j : -1;
    if (tid == 0) topk_length[t] = L;
    return;
  }
  if (k == 0) {
    if (tid == 0) topk_length[t] = 0;
    return;
  }
  for (int i = tid; i < 512; i += NT) (&s_hist[0][0])[i] = 0;
  const int c0 = KPT * tid;
  const int nv = L - c0 < 0 ? 0 : (L - c0 > KPT ? KPT : L - c0);   // valid columns of this thread
  const bool full = nv == KPT;
  const uint16_t* row = logits + t * ld;
  uint32_t key[KPT];   // one key per register; invalid slots hold 0, below every valid key
  if (full && ((uintptr_t)(row + c0) & 15) == 0) {
#pragma unroll
    for (int v = 0; v < KPT / 8; ++v) {
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(row + c0) + v);
      const uint32_t x[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t kk = order_key2(x[e]);
        key[8 * v + 2 * e] = kk & 0xFFFFu;
        key[8 * v + 2 * e + 1] = kk >> 16;
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < KPT / 2; ++i) {
      const uint32_t a = 2 * i < nv ? (uint32_t)__ldg(row + c0 + 2 * i) : 0u;
      const uint32_t b = 2 * i + 1 < nv ? (uint32_t)__ldg(row + c0 + 2 * i + 1) : 0u;
      const uint32_t kk = order_key2(a | (b << 16));
      key[2 * i] = 2 * i < nv ? (kk & 0xFFFFu) : 0u;
      key[2 * i + 1] = 2 * i + 1 < nv ? (kk >> 16) : 0u;
    }
  }
  __syncthreads();
  // pass 1: high bytes of the valid keys
  if (full) {
#pragma unroll
    for (int e = 0; e < KPT; ++e) atomicAdd(&s_hist[0][key[e] >> 8], 1);
  } else {
#pragma unroll
    for (int e = 0; e < KPT; ++e)
      if (e < nv) atomicAdd(&s_hist[0][key[e] >> 8], 1);
  }
  __syncthreads();
  if (w == 0) find_digit(s_hist[0], k, lane, s_sel);
  __syncthreads();
  const uint32_t hi = (uint32_t)s_sel[0];
  const int above_hi = s_sel[1];
  // pass 2: low bytes of the keys with that high byte (an invalid slot's key 0 can
  // match only if hi is 0; then it is skipped by its column)
  if (full || hi != 0u) {
#pragma unroll
    for (int e = 0; e < KPT; ++e)
      if ((key[e] >> 8) == hi) atomicAdd(&s_hist[1][key[e] & 255u], 1);
  } else {
#pragma unroll
    for (int e = 0; e < KPT; ++e)
      if (e < nv && (key[e] >> 8) == hi) atomicAdd(&s_hist[1][key[e] & 255u], 1);
  }
  __syncthreads();
  if (w == 0) find_digit(s_hist[1], k - above_hi, lane, s_sel + 2);
  __syncthreads();
  const uint32_t T = (hi << 8) | (uint32_t)s_sel[2];
  const int need = k - above_hi - s_sel[3];
  // T >= 1 (the k-th largest valid key is a valid key), so an invalid slot's 0 is in
  // neither mask
  uint32_t gtm = 0u, eqm = 0u;
#pragma unroll
  for (int e = 0; e < KPT; ++e) {
    gtm |= (key[e] > T) ? (1u << e) : 0u;
    eqm |= (key[e] == T) ? (1u << e) : 0u;
  }
  // block-wide exclusive prefix of (above T) << 16 | (equal to T), in column order
  const int packed = (__popc(gtm) << 16) | __popc(eqm);
  int incl = packed;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_wsum[w] = incl;
  __syncthreads();
  int ws = lane < NWARP ? s_wsum[lane] : 0;
#pragma unroll
  for (int o = 1; o < NWARP; o <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, ws, o);
    if (lane >= o) ws += v;
  }
  const int wbefore = __shfl_sync(0xFFFFFFFFu, ws, (w + 31) & 31);
  const int excl = (w > 0 ? wbefore : 0) + incl - packed;
  int gtb = excl >> 16, eqb = excl & 0xFFFF;
  uint32_t m = gtm | eqm;
  while (m) {
    const int e = __ffs(m) - 1;
    m &= m - 1u;
    const int col = c0 + e;
    if ((gtm >> e) & 1u) {
      const int pos = gtb + min(eqb, need);
      if (pos < k) out[pos] = col;
      ++gtb;
    } else {
      if (eqb < need && gtb + eqb < k) out[gtb + eqb] = col;
      ++eqb;
    }
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
  if (n <= RT * RK) {
    topk_reg_kernel<RT, RK, RB><<<(unsigned)s_q, RT, 0, (cudaStream_t)stream>>>(
        (const uint16_t*)logits, (long long)ld, lengths, n, k, indices, topk_length);
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
  }
  const size_t smem = (size_t)((n + 7) & ~7) * sizeof(uint16_t);
  topk_kernel<<<(unsigned)s_q, THREADS, smem, (cudaStream_t)stream>>>(
      (const uint16_t*)logits, (long long)ld, lengths, n, k, indices, topk_length);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
