// KV-cache insert for the fp8_ds_mla cache: RMSNorm of the new tokens' latent KV, RoPE
// of their rotary part, per-128 FP8 quantisation, and the 656-byte row write, in one
// kernel (the KV write done inside the norm kernel: vLLM PR #64364, "The changes and what
// each bought", Attention row).  The exact arithmetic is stated in include/dsa_kv_insert.h.
//
// One warp per token, eight tokens per CTA.  Lane l holds latent dims 16 l .. 16 l + 15
// (so lanes 8 b .. 8 b + 7 hold 128-dim block b) and rotary pair l.  The sum of squares
// is a warp all-reduce, each block's max |x * w| a reduce over its eight lanes.  Every
// load and store of a row is one contiguous 16- or 4-byte access per lane.

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "dsa_kv_insert.h"
#include "ptx_sm103.cuh"

namespace dsa_kv {

constexpr int D_LAT = 512;
constexpr int ROW_BYTES = 656;
constexpr int WARPS = 8;

struct Params {
  const uint16_t* kv;
  long long ld;
  const int32_t* positions;
  const int64_t* slots;
  const uint16_t* w;
  uint8_t* pool;
  long long n_rows;
  uint32_t* status;
  int s_new;
  uint32_t flags;
  float eps;
  // rotary frequency of pair j as a 64-bit fixed-point fraction of a turn:
  // frac(base^(-2j/64) / 2 pi) * 2^64, so that position * entry (mod 2^64) is the angle's
  // fraction of a turn without the rounding of a large fp32 angle
  unsigned long long turns[32];
};

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__global__ void __launch_bounds__(32 * WARPS) kv_insert_kernel(const __grid_constant__ Params P) {
  // a dependent launched with programmatic serialization may start now; it waits for
  // this kernel's completion before it reads the pool (DSA_FLAG_AFTER_PRODUCER)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const long long i = (long long)blockIdx.x * WARPS + (threadIdx.x >> 5);
  if (i >= P.s_new) return;
  const long long slot = P.slots[i];
  if (slot < 0) return;
  if (slot >= P.n_rows && (P.flags & DSA_KV_FLAG_CHECK_SLOTS)) {
    if (lane == 0 && P.status) atomicOr(P.status, DSA_STATUS_SLOT_OUT_OF_RANGE);
    return;
  }
  const uint16_t* row = P.kv + i * P.ld;
  const uint4 xa = __ldg(reinterpret_cast<const uint4*>(row) + 2 * lane);
  const uint4 xb = __ldg(reinterpret_cast<const uint4*>(row) + 2 * lane + 1);
  const uint4 wa = __ldg(reinterpret_cast<const uint4*>(P.w) + 2 * lane);
  const uint4 wb = __ldg(reinterpret_cast<const uint4*>(P.w) + 2 * lane + 1);
  const uint32_t rp = __ldg(reinterpret_cast<const uint32_t*>(row + D_LAT) + lane);
  const int pos = __ldg(P.positions + i);

  const uint32_t xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
  const uint32_t wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
  float xw[16];
  float ss = 0.f, m = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float x0 = bf16_lo(xv[k]), x1 = bf16_hi(xv[k]);
    ss = fmaf(x0, x0, fmaf(x1, x1, ss));
    xw[2 * k] = x0 * bf16_lo(wv[k]);       // exact: two 8-bit significands
    xw[2 * k + 1] = x1 * bf16_hi(wv[k]);
    m = fmaxf(m, fmaxf(fabsf(xw[2 * k]), fabsf(xw[2 * k + 1])));
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
#pragma unroll
  for (int o = 4; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  const float inv = 1.0f / sqrtf(ss * (1.0f / D_LAT) + P.eps);

  // codes: round-to-nearest-even E4M3 of (x * w) * (448 / m): one rounded quotient per
  // block, one rounded product per value (no contraction into anything else)
  const float rq = m > 0.f ? __fdiv_rn(448.0f, m) : 0.f;
  uint32_t cw[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float q[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) q[e] = __fmul_rn(xw[4 * k + e], rq);
    cw[k] = dsa::f32x2_to_e4m3x2(q[0], q[1]) | (dsa::f32x2_to_e4m3x2(q[2], q[3]) << 16);
  }
  // the block's scale: max|y| / 448 = m * inv / 448
  const float scale = m > 0.f ? __fdiv_rn(__fmul_rn(m, inv), 448.0f) : 1.0f;

  // rotary pair `lane`, angle positions[i] * theta_lane from its exact count of turns
  const unsigned long long turns = (unsigned long long)(long long)pos * P.turns[lane];
  const float frac = (float)(turns >> 40) * 5.9604644775390625e-08f;   // top 24 bits / 2^24
  float sn, cs;
  sincospif(2.0f * frac, &sn, &cs);
  const float r0 = bf16_lo(rp), r1 = bf16_hi(rp);
  const __nv_bfloat162 rr = __floats2bfloat162_rn(r0 * cs - r1 * sn, r0 * sn + r1 * cs);

  uint8_t* dst = P.pool + slot * ROW_BYTES;
  reinterpret_cast<uint4*>(dst)[lane] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
  if ((lane & 7) == 0) reinterpret_cast<float*>(dst + D_LAT)[lane >> 3] = scale;
  reinterpret_cast<__nv_bfloat162*>(dst + D_LAT + 16)[lane] = rr;
}

static bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

static void turn_table(float base, unsigned long long* out) {
  const long double two_pi = 6.283185307179586476925286766559L;
  for (int j = 0; j < 32; ++j) {
    const long double theta = powl((long double)base, -2.0L * j / 64.0L);
    const long double f = theta / two_pi - floorl(theta / two_pi);
    out[j] = (unsigned long long)(f * 18446744073709551616.0L);
  }
}

}  // namespace dsa_kv

extern "C" int dsa_kv_insert(const void* kv, int64_t ld, const int32_t* positions, const int64_t* slots,
                             int32_t s_new, const void* kv_norm_w, float rms_eps, float rope_base, void* pool,
                             int64_t n_rows, uint32_t flags, uint32_t* status, void* stream) {
  using namespace dsa_kv;
  if (s_new < 0 || n_rows < 0 || ld < 576 || ld % 8 != 0 || !(rms_eps >= 0.f) || !(rope_base > 0.f) ||
      !isfinite(rms_eps) || !isfinite(rope_base) || (flags & ~DSA_KV_FLAG_CHECK_SLOTS) != 0)
    return DSA_ERR_INVALID_ARG;
  if (s_new == 0) return DSA_OK;
  if (!kv || !positions || !slots || !kv_norm_w || (!pool && n_rows > 0) || !aligned(kv, 16) ||
      !aligned(kv_norm_w, 16) || !aligned(positions, 4) || !aligned(slots, 8) || !aligned(pool, 16) ||
      (status && !aligned(status, 4)))
    return DSA_ERR_INVALID_ARG;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) return DSA_ERR_UNSUPPORTED_DEVICE;
  Params P;
  P.kv = static_cast<const uint16_t*>(kv);
  P.ld = (long long)ld;
  P.positions = positions;
  P.slots = slots;
  P.w = static_cast<const uint16_t*>(kv_norm_w);
  P.pool = static_cast<uint8_t*>(pool);
  P.n_rows = (long long)n_rows;
  P.status = status;
  P.s_new = s_new;
  P.flags = flags;
  P.eps = rms_eps;
  turn_table(rope_base, P.turns);
  const unsigned grid = (unsigned)((s_new + WARPS - 1) / WARPS);
  kv_insert_kernel<<<grid, 32 * WARPS, 0, (cudaStream_t)stream>>>(P);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
