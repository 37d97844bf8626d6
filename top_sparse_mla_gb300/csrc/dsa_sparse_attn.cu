// Fused top-k sparse latent attention for GB300 (sm_103a): q RMSNorm + q RoPE +
// gather of fp8_ds_mla rows by index + QK^T + online softmax + PV + inverse RoPE +
// MXFP8 cast, in one persistent kernel (stages as named on "Deepseek V41 Attention
// MegaKernel", vLLM PR #56344, Purpose).
//
// Work item = (query token, KV split).  One CTA of 384 threads per SM walks items.
// Per item the CTA compacts the token's valid index columns, builds q~ (normalised,
// rotated, fp16) in shared memory, then streams the gathered rows in tiles of 128:
//
//   KD warps (4)   rows -> fp16 K~ (scale folded)  -> TMEM ring   (A of QK^T)
//   VD warps (2)   rows -> fp16 V~ (scale folded)  -> SMEM ring   (A of PV, MN-major)
//   MMA thread     S^T[128 rows x 64 heads]  = K~ . q~^T   (tcgen05, A from TMEM)
//                  O^T[512 dims x 64 heads] += V~^T . P^T  (tcgen05, A,B from SMEM)
//   SM warps (4)   S^T -> exp2 -> P (fp16, SMEM), running max / sum per head,
//                  lazy O rescale, then the epilogue: O / l, inverse RoPE, MXFP8 cast.
//
// Both contractions run with M = 128 (the row tile for QK^T, a 128-dim slice of the
// latent for PV) and N = 64 heads, so the tensor core runs full-width M even though a
// token has only 64 heads.  Accumulators live in TMEM: O^T takes columns 0..255, S^T
// 256..319, the K~ ring 320..511.
//
// Every wait on an mbarrier is bounded; on timeout the CTA raises
// DSA_STATUS_WAIT_TIMEOUT, drains its tensor-core work and frees TMEM before exiting.

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "dsa_sparse_attn.h"

namespace dsa {

constexpr int D_LAT = 512;
constexpr int D_QK = 576;
constexpr int ROW_BYTES = 656;
constexpr int TILE = 128;            // gathered rows per tile
constexpr int HP = 64;               // heads as seen by the MMAs (padded)
constexpr int NTHREADS = 384;      // 12 warps: VD 0-1, MMA 2, scan 3, KD 4-7, SM 8-11
constexpr int MMA_WARP = 2;
constexpr int SCAN_WARP = 3;
constexpr int K_SLOTS = 6;           // TMEM ring of 32-column slots (64 K~ dims each)
constexpr int V_SLOTS = 2;           // SMEM ring of [128 dims x 128 rows] fp16 blocks
constexpr int HC_PER_TILE = 9;       // 8 latent half-chunks (64 dims) + 1 rope chunk

// TMEM columns
constexpr uint32_t TM_O = 0;         // O^T: d-tile j at columns [64j, 64j+64)
constexpr uint32_t TM_S = 256;       // S^T
constexpr uint32_t TM_K = 320;       // K~ ring
constexpr uint32_t TM_COLS = 512;

// shared memory map (offsets from a 1024-aligned base)
constexpr uint32_t SM_Q = 0;                         // q~: 9 K-atoms x 8 KB (K-major, SW128)
constexpr uint32_t SM_V = SM_Q + 9 * 8192;           // V~ ring: 2 x 32 KB (MN-major, SW128)
constexpr uint32_t SM_P = SM_V + V_SLOTS * 32768;    // P: 16 KB (MN-major, SW128)
constexpr uint32_t SM_BAR = SM_P + 16384;            // mbarriers (32 x 8 B)
constexpr uint32_t SM_LIST = SM_BAR + 256;           // compacted rows (DSA_MAX_TOPK x 4 B)
constexpr uint32_t SM_NORMW = SM_LIST + DSA_MAX_TOPK * 4;   // 576 fp32
constexpr uint32_t SM_ROPE = SM_NORMW + D_QK * 4;    // 32 x (cos, sin) fp32
constexpr uint32_t SM_MREF = SM_ROPE + 256;          // 64 fp32 running max (log2 units)
constexpr uint32_t SM_LACC = SM_MREF + 256;          // 64 fp32 running sum
constexpr uint32_t SM_ALPHA = SM_LACC + 256;         // 64 fp32 rescale factors
constexpr uint32_t SM_RED = SM_ALPHA + 256;          // 4 warps x 64 fp32 exchange
constexpr uint32_t SM_LPART = SM_RED + 1024;         // 2 (tile parity) x 4 warps x 64 fp32 row sums
constexpr uint32_t SM_FLAG = SM_LPART + 2048;        // 2 x 4 fp32 per-warp flags (tile parity)
constexpr uint32_t SM_INFO = SM_FLAG + 32;           // item info (ints)
constexpr uint32_t SM_END = SM_INFO + 64;
constexpr uint32_t SMEM_BYTES = SM_END + 1024;       // + alignment slack

// mbarrier slots
enum {
  B_KFULL = 0, B_KEMPTY = B_KFULL + K_SLOTS, B_VFULL = B_KEMPTY + K_SLOTS, B_VEMPTY = B_VFULL + V_SLOTS,
  B_SFULL = B_VEMPTY + V_SLOTS, B_SEMPTY, B_PFULL, B_PEMPTY, B_ODONE, B_GRP, B_DRAIN, B_COUNT
};
static_assert(B_COUNT <= 32, "barrier area");

// item info slots
enum { I_TMEM = 0, I_ABORT, I_T, I_ROW0, I_NROWS, I_LAST, I_COUNT };

struct KParams {
  const uint16_t* q;
  const uint8_t* kv_swa;
  const uint8_t* kv_cmp;
  const int32_t* indices;
  const int32_t* topk_length;
  const int32_t* positions;
  const uint16_t* norm_w;
  uint8_t* out_fp8;
  uint8_t* out_sf;
  float* out_precast;
  float* out_lse;
  float* part_o;       // [s_q][n_splits][64][512]
  float* part_lse;     // [s_q][n_splits][64]  (log2 units)
  uint32_t* counters;  // [s_q]
  uint32_t* status;
  int s_q, h_q, topk, n_swa_cols;
  long long n_swa_rows, n_cmp_rows;
  float score_scale_log2;   // softmax_scale * log2(e)
  float rope_base;
  float rms_eps;
  uint32_t flags;
  int n_splits;
  int n_items;
};

// ------------------------------------------------------------------ PTX helpers
#define DEV __device__ __forceinline__

DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

DEV void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
DEV void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
DEV bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
DEV void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
DEV void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
DEV void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

DEV void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// D[tmem] (+)= A[tmem] . B[smem]^T
DEV void mma_ts(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}
// D[tmem] (+)= A[smem] . B[smem]^T
DEV void mma_ss(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}

// shared-memory matrix descriptor, 128-byte swizzle
DEV uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// instruction descriptor: fp16 A/B, fp32 accumulate, M=128, N=64
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t a_mn, uint32_t b_mn) {
  return (1u << 4) | (a_mn << 15) | (b_mn << 16) | ((uint32_t)(HP >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

DEV void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
DEV void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

DEV uint4 ldg_nc(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
DEV void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
DEV void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// two E4M3 codes (low byte = first) -> f16x2, times an f16x2 scale
DEV uint32_t e4m3x2_scaled(uint32_t two_codes, __half2 s2) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((unsigned short)two_codes));
  __half2 v = *reinterpret_cast<__half2*>(&h);
  v = __hmul2(v, s2);
  return *reinterpret_cast<uint32_t*>(&v);
}
// 16 E4M3 codes -> 8 f16x2 words
DEV void dequant16(uint4 c, __half2 s2, uint32_t* o) {
  o[0] = e4m3x2_scaled(c.x & 0xFFFF, s2);
  o[1] = e4m3x2_scaled(c.x >> 16, s2);
  o[2] = e4m3x2_scaled(c.y & 0xFFFF, s2);
  o[3] = e4m3x2_scaled(c.y >> 16, s2);
  o[4] = e4m3x2_scaled(c.z & 0xFFFF, s2);
  o[5] = e4m3x2_scaled(c.z >> 16, s2);
  o[6] = e4m3x2_scaled(c.w & 0xFFFF, s2);
  o[7] = e4m3x2_scaled(c.w >> 16, s2);
}
// two bf16 (low = first) -> f16x2
DEV uint32_t bf16x2_to_f16x2(uint32_t w) {
  __half2 v = __floats2half2_rn(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  return *reinterpret_cast<uint32_t*>(&v);
}
DEV uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
DEV float f16lo(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFF))); }
DEV float f16hi(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); }

// e4m3 pair: first value in the low byte
DEV uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Row pointer from a compacted list entry (bit 31 selects the compressed pool).
DEV const uint8_t* row_ptr(const KParams& P, uint32_t e) {
  const uint8_t* base = (e & 0x80000000u) ? P.kv_cmp : P.kv_swa;
  return base + (size_t)(e & 0x7FFFFFFFu) * ROW_BYTES;
}

// Reduce 16 per-lane values across the warp, one result per value: afterwards lanes
// 2m and 2m+1 both hold the reduction of value m in v[0].
template <bool IS_MAX>
DEV void reduce16(float (&v)[16], int lane) {
#pragma unroll
  for (int k = 16, n = 16; k >= 2; k >>= 1, n >>= 1) {
    const bool upper = (lane & k) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      const float recv = __shfl_xor_sync(0xFFFFFFFFu, send, k);
      v[i] = IS_MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
  const float o = __shfl_xor_sync(0xFFFFFFFFu, v[0], 1);
  v[0] = IS_MAX ? fmaxf(v[0], o) : v[0] + o;
}

// ------------------------------------------------------------------ the kernel
struct Ctx {
  uint8_t* sm;
  uint32_t sb;              // shared address of sm
  volatile int* info;
  uint32_t* status;
  unsigned long long t0;    // clock at kernel start (for wait limits)
};

constexpr unsigned long long WAIT_LIMIT_CYCLES = 4000000000ull;   // ~2 s at 2 GHz

DEV uint32_t bar_addr(const Ctx& c, int i) { return c.sb + SM_BAR + 8u * (uint32_t)i; }

// Bounded wait: returns false (and raises the abort flag) when the limit passes or
// another thread of the CTA has already aborted.
DEV bool wait_bar(const Ctx& c, int b, uint32_t parity) {
  const uint32_t addr = bar_addr(c, b);
  if (mbar_try(addr, parity)) return true;
  const unsigned long long start = clock64();
  while (true) {
    if (mbar_try(addr, parity)) return true;
    if (c.info[I_ABORT]) return false;
    if (clock64() - start > WAIT_LIMIT_CYCLES) {
      atomicOr(c.status, DSA_STATUS_WAIT_TIMEOUT);
      c.info[I_ABORT] = 1;
      return false;
    }
  }
}

// Warp-collective form: every lane polls, and the warp agrees on the outcome so that
// it never splits before a full-warp shuffle or TMEM access.
DEV bool wait_bar_w(const Ctx& c, int b, uint32_t parity) {
  const bool ok = wait_bar(c, b, parity);
  return __all_sync(0xFFFFFFFFu, ok);
}

__global__ void __launch_bounds__(NTHREADS, 1) dsa_fwd_kernel(const KParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Ctx c;
  {
    const uint32_t raw = smem_u32(smem_raw);
    c.sm = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  }
  c.sb = smem_u32(c.sm);
  c.info = reinterpret_cast<volatile int*>(c.sm + SM_INFO);
  c.status = P.status;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float* s_normw = reinterpret_cast<float*>(c.sm + SM_NORMW);
  float2* s_rope = reinterpret_cast<float2*>(c.sm + SM_ROPE);
  float* s_mref = reinterpret_cast<float*>(c.sm + SM_MREF);
  float* s_lacc = reinterpret_cast<float*>(c.sm + SM_LACC);
  float* s_alpha = reinterpret_cast<float*>(c.sm + SM_ALPHA);
  float* s_red = reinterpret_cast<float*>(c.sm + SM_RED);
  float* s_flag = reinterpret_cast<float*>(c.sm + SM_FLAG);
  float* s_lpart = reinterpret_cast<float*>(c.sm + SM_LPART);
  uint32_t* s_list = reinterpret_cast<uint32_t*>(c.sm + SM_LIST);

  if (tid == 0) {
    for (int i = 0; i < K_SLOTS; ++i) {
      mbar_init(bar_addr(c, B_KFULL + i), 128);
      mbar_init(bar_addr(c, B_KEMPTY + i), 1);
    }
    for (int i = 0; i < V_SLOTS; ++i) {
      mbar_init(bar_addr(c, B_VFULL + i), 64);
      mbar_init(bar_addr(c, B_VEMPTY + i), 1);
    }
    mbar_init(bar_addr(c, B_SFULL), 1);
    mbar_init(bar_addr(c, B_SEMPTY), 128);
    mbar_init(bar_addr(c, B_PFULL), 128);
    mbar_init(bar_addr(c, B_PEMPTY), 1);
    mbar_init(bar_addr(c, B_ODONE), 1);
    mbar_init(bar_addr(c, B_GRP), 128);
    mbar_init(bar_addr(c, B_DRAIN), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    c.info[I_ABORT] = 0;
  }
  if (warp == MMA_WARP) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(c.sb + SM_INFO + 4 * I_TMEM),
                 "r"(TM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  for (int i = tid; i < D_QK; i += NTHREADS) s_normw[i] = __uint_as_float((uint32_t)P.norm_w[i] << 16);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = (uint32_t)c.info[I_TMEM];

  // pipeline counters (each role advances the ones it uses, in the same order)
  uint32_t kq = 0, vq = 0, n_qk = 0, n_pv = 0, n_item_tiles = 0, n_grp = 0;

  for (int item = blockIdx.x; item < P.n_items; item += gridDim.x) {
    const int t = item / P.n_splits;
    const int split = item % P.n_splits;

    // ---------------------------------------------------------- prologue A
    if (warp == SCAN_WARP) {
      // compact the token's valid columns: j < topk_length, index >= 0
      int L = P.topk_length[t];
      L = L < 0 ? 0 : (L > P.topk ? P.topk : L);
      const int32_t* irow = P.indices + (size_t)t * P.topk;
      int count = 0;
      for (int j0 = 0; j0 < L; j0 += 32) {
        const int j = j0 + lane;
        int idx = (j < L) ? irow[j] : -1;
        const bool cmp = j >= P.n_swa_cols;
        bool valid = idx >= 0;
        if (valid && (P.flags & DSA_FLAG_CHECK_INDICES)) {
          const long long nr = cmp ? P.n_cmp_rows : P.n_swa_rows;
          if ((long long)idx >= nr) {
            valid = false;
            atomicOr(P.status, DSA_STATUS_INDEX_OUT_OF_RANGE);
          }
        }
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, valid);
        if (valid) s_list[count + __popc(b & ((1u << lane) - 1u))] = (uint32_t)idx | (cmp ? 0x80000000u : 0u);
        count += __popc(b);
      }
      const int n_tiles_tok = (count + TILE - 1) / TILE;
      const int tps = (n_tiles_tok + P.n_splits - 1) / P.n_splits;
      int tile0 = split * tps, tile1 = tile0 + tps;
      if (tile1 > n_tiles_tok) tile1 = n_tiles_tok;
      const int T = tile1 > tile0 ? tile1 - tile0 : 0;
      const int row0 = tile0 * TILE;
      int nrows = (tile1 * TILE < count ? tile1 * TILE : count) - row0;
      if (T == 0) nrows = 0;
      __syncwarp();
      for (int r = lane; r < nrows; r += 32) prefetch_l2(row_ptr(P, s_list[row0 + r]), ROW_BYTES);
      // warm L2 with the next item's q while this item runs
      const int nxt = item + gridDim.x;
      if (lane == 0 && nxt < P.n_items && nxt / P.n_splits != t)
        prefetch_l2(P.q + (size_t)(nxt / P.n_splits) * P.h_q * D_QK, (uint32_t)(P.h_q * D_QK * 2));
      if (lane == 0) {
        c.info[I_T] = T;
        c.info[I_ROW0] = row0;
        c.info[I_NROWS] = nrows;
      }
    } else if (warp == MMA_WARP) {
      // cos / sin of pos * theta_i for the 32 rotary pairs (fp64 angle)
      const double theta = pow((double)P.rope_base, -2.0 * lane / 64.0);
      double sn, cs;
      sincos((double)P.positions[t] * theta, &sn, &cs);
      s_rope[lane] = make_float2((float)cs, (float)sn);
    } else if (warp == 1) {
      s_mref[lane] = -INFINITY;
      s_mref[lane + 32] = -INFINITY;
      s_lacc[lane] = 0.f;
      s_lacc[lane + 32] = 0.f;
    }
    __syncthreads();

    // ---------------------------------------------------------- prologue B: q~
    {
      const float eps = P.rms_eps;
#pragma unroll 1
      for (int h = warp; h < HP; h += NTHREADS / 32) {
        uint4 raw[3];
        float ss = 0.f;
        const bool live = h < P.h_q;
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          const int ch = lane + 32 * k;
          raw[k] = make_uint4(0, 0, 0, 0);
          if (live && ch < 72) raw[k] = ldg_nc(P.q + ((size_t)t * P.h_q + h) * D_QK + ch * 8);
          const uint32_t w4[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float a = __uint_as_float(w4[e] << 16), b = __uint_as_float(w4[e] & 0xFFFF0000u);
            ss = fmaf(a, a, fmaf(b, b, ss));
          }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
        const float inv = rsqrtf(ss * (1.0f / D_QK) + eps);
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          const int ch = lane + 32 * k;
          if (ch >= 72) continue;
          const uint32_t w4[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
          float x[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            x[2 * e] = __uint_as_float(w4[e] << 16) * inv * s_normw[ch * 8 + 2 * e];
            x[2 * e + 1] = __uint_as_float(w4[e] & 0xFFFF0000u) * inv * s_normw[ch * 8 + 2 * e + 1];
          }
          if (ch >= 64) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 r = s_rope[(ch - 64) * 4 + e];
              const float x0 = x[2 * e], x1 = x[2 * e + 1];
              x[2 * e] = x0 * r.x - x1 * r.y;
              x[2 * e + 1] = x0 * r.y + x1 * r.x;
            }
          }
          uint4 o;
          o.x = pack_f16x2(x[0], x[1]);
          o.y = pack_f16x2(x[2], x[3]);
          o.z = pack_f16x2(x[4], x[5]);
          o.w = pack_f16x2(x[6], x[7]);
          if (!live) o = make_uint4(0, 0, 0, 0);
          const uint32_t atom = ch >> 3, cc = ch & 7;
          sts128(c.sb + SM_Q + atom * 8192 + (h >> 3) * 1024 + (h & 7) * 128 + ((cc ^ (h & 7)) << 4), o);
        }
      }
    }
    fence_async_smem();
    __syncthreads();

    const int T = c.info[I_T];
    const int row0 = c.info[I_ROW0];
    const int nrows = c.info[I_NROWS];
    bool ok = c.info[I_ABORT] == 0;

    // ---------------------------------------------------------- roles
    if (warp == MMA_WARP) {
      // ===== MMA issuer =====
      if (lane == 0 && ok) {
        constexpr uint32_t IDESC_QK = idesc_f16(0, 0);
        constexpr uint32_t IDESC_PV = idesc_f16(1, 1);
        auto pv = [&](int u) -> bool {
          if (!wait_bar(c, B_PFULL, n_pv & 1)) return false;
          tc_fence_after();
          for (int j = 0; j < 4; ++j) {
            const uint32_t slot = vq % V_SLOTS;
            if (!wait_bar(c, B_VFULL + slot, (vq / V_SLOTS) & 1)) return false;
            tc_fence_after();
            const uint32_t vbase = c.sb + SM_V + slot * 32768;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t ad = sdesc(vbase + kk * 2048, 16384, 1024);
              const uint64_t bd = sdesc(c.sb + SM_P + kk * 2048, 16384, 1024);
              mma_ss(tmem + TM_O + 64 * j, ad, bd, IDESC_PV, (u > 0 || kk > 0) ? 1u : 0u);
            }
            tc_commit(bar_addr(c, B_VEMPTY + slot));
            ++vq;
          }
          tc_commit(bar_addr(c, B_PEMPTY));
          ++n_pv;
          return true;
        };
        for (int tt = 0; tt < T && ok; ++tt) {
          if (!wait_bar(c, B_SEMPTY, (n_qk & 1) ^ 1)) { ok = false; break; }
          tc_fence_after();
          for (int hc = 0; hc < HC_PER_TILE && ok; ++hc) {
            const uint32_t slot = kq % K_SLOTS;
            if (!wait_bar(c, B_KFULL + slot, (kq / K_SLOTS) & 1)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t bd = sdesc(c.sb + SM_Q + hc * 8192 + kk * 32, 16, 1024);
              mma_ts(tmem + TM_S, tmem + TM_K + 32 * slot + 8 * kk, bd, IDESC_QK, (hc | kk) ? 1u : 0u);
            }
            tc_commit(bar_addr(c, B_KEMPTY + slot));
            ++kq;
          }
          if (!ok) break;
          tc_commit(bar_addr(c, B_SFULL));
          ++n_qk;
          if (tt >= 1 && !pv(tt - 1)) { ok = false; break; }
        }
        if (ok && T > 0) {
          if (!pv(T - 1)) ok = false;
          else tc_commit(bar_addr(c, B_ODONE));
        }
      }
    } else if (warp >= 4 && warp < 8) {
      // ===== KD: rows -> fp16 K~ -> TMEM ring =====
      const int q4 = warp - 4;
      const int r = q4 * 32 + lane;
      const uint32_t tlane = (uint32_t)(q4 * 32) << 16;
      for (int tt = 0; tt < T && ok; ++tt) {
        const int gr = tt * TILE + r;
        const bool valid = gr < nrows;
        const uint8_t* rp = valid ? row_ptr(P, s_list[row0 + gr]) : nullptr;
        __half2 s2[4];
        {
          uint4 sc = valid ? ldg_nc(rp + D_LAT) : make_uint4(0, 0, 0, 0);
          s2[0] = __float2half2_rn(__uint_as_float(sc.x));
          s2[1] = __float2half2_rn(__uint_as_float(sc.y));
          s2[2] = __float2half2_rn(__uint_as_float(sc.z));
          s2[3] = __float2half2_rn(__uint_as_float(sc.w));
        }
        // two 64-byte load buffers, refilled two half-chunks ahead; the rope chunk
        // (128 bytes of bf16) arrives in both buffers
        uint4 buf[2][4];
#pragma unroll
        for (int p = 0; p < 2; ++p)
#pragma unroll
          for (int i = 0; i < 4; ++i) buf[p][i] = valid ? ldg_nc(rp + 64 * p + 16 * i) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int hc = 0; hc < HC_PER_TILE; ++hc) {
          uint32_t v[32];
          if (hc < 8) {
#pragma unroll
            for (int i = 0; i < 4; ++i) dequant16(buf[hc & 1][i], s2[hc >> 1], v + 8 * i);
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint4 w = buf[i >> 2][i & 3];
              v[4 * i + 0] = bf16x2_to_f16x2(w.x);
              v[4 * i + 1] = bf16x2_to_f16x2(w.y);
              v[4 * i + 2] = bf16x2_to_f16x2(w.z);
              v[4 * i + 3] = bf16x2_to_f16x2(w.w);
            }
          }
          // refill this buffer two half-chunks ahead (latent 0..7, then the rope halves)
          const int nh = hc + 2;
          if (nh < 8) {
#pragma unroll
            for (int i = 0; i < 4; ++i) buf[hc & 1][i] = valid ? ldg_nc(rp + 64 * nh + 16 * i) : make_uint4(0, 0, 0, 0);
          } else if (nh < 10) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              buf[hc & 1][i] = valid ? ldg_nc(rp + 528 + 64 * (nh - 8) + 16 * i) : make_uint4(0, 0, 0, 0);
          }
          const uint32_t slot = kq % K_SLOTS;
          if (!wait_bar_w(c, B_KEMPTY + slot, ((kq / K_SLOTS) & 1) ^ 1)) { ok = false; break; }
          tc_fence_after();
          tmem_st32(tmem + tlane + TM_K + 32 * slot, v);
          tc_wait_st();
          tc_fence_before();
          mbar_arrive(bar_addr(c, B_KFULL + slot));
          ++kq;
        }
      }
    } else if (warp < 2) {
      // ===== VD: rows -> fp16 V~ (MN-major) -> SMEM ring; two rows per thread =====
      for (int tt = 0; tt < T && ok; ++tt) {
        const uint8_t* rp[2];
        bool valid[2];
        float scf[2][4];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int r = warp * 32 + lane + 64 * e;
          const int gr = tt * TILE + r;
          valid[e] = gr < nrows;
          rp[e] = valid[e] ? row_ptr(P, s_list[row0 + gr]) : nullptr;
          const uint4 sc = valid[e] ? ldg_nc(rp[e] + D_LAT) : make_uint4(0, 0, 0, 0);
          scf[e][0] = __uint_as_float(sc.x);
          scf[e][1] = __uint_as_float(sc.y);
          scf[e][2] = __uint_as_float(sc.z);
          scf[e][3] = __uint_as_float(sc.w);
        }
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
          uint4 buf[2][8];
#pragma unroll
          for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int i = 0; i < 8; ++i) buf[e][i] = valid[e] ? ldg_nc(rp[e] + 128 * j + 16 * i) : make_uint4(0, 0, 0, 0);
          const uint32_t slot = vq % V_SLOTS;
          if (!wait_bar_w(c, B_VEMPTY + slot, ((vq / V_SLOTS) & 1) ^ 1)) { ok = false; break; }
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int r = warp * 32 + lane + 64 * e;
            const uint32_t rsw = (uint32_t)(r & 7);
            const uint32_t base = c.sb + SM_V + slot * 32768 + (uint32_t)(r >> 3) * 1024 + rsw * 128;
            const __half2 s2 = __float2half2_rn(scf[e][j]);
#pragma unroll
            for (int a = 0; a < 2; ++a) {
              uint32_t v[32];
#pragma unroll
              for (int i = 0; i < 4; ++i) dequant16(buf[e][4 * a + i], s2, v + 8 * i);
#pragma unroll
              for (int cc = 0; cc < 8; ++cc)
                sts128(base + a * 16384 + ((cc ^ rsw) << 4), make_uint4(v[4 * cc], v[4 * cc + 1], v[4 * cc + 2], v[4 * cc + 3]));
            }
          }
          fence_async_smem();
          mbar_arrive(bar_addr(c, B_VFULL + slot));
          ++vq;
        }
      }
    } else if (warp >= 8 && warp < 12) {
      // ===== SM: softmax, P, rescale; then the epilogue =====
      const int q4 = warp - 8;
      const int r = q4 * 32 + lane;
      const uint32_t tlane = (uint32_t)(q4 * 32) << 16;
      const float c2 = P.score_scale_log2;
      auto grp_sync = [&]() -> bool {
        mbar_arrive(bar_addr(c, B_GRP));
        const bool r_ = wait_bar_w(c, B_GRP, n_grp & 1);
        ++n_grp;
        return r_;
      };
      for (int tt = 0; tt < T && ok; ++tt) {
        const int rows_here = nrows - tt * TILE;
        const bool valid = r < rows_here;
        if (!wait_bar_w(c, B_SFULL, n_qk & 1)) { ok = false; break; }
        tc_fence_after();
        float x[64];
        {
          uint32_t a[32];
          tmem_ld32(tmem + tlane + TM_S, a);
          tc_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] = valid ? __uint_as_float(a[i]) * c2 : -INFINITY;
          tmem_ld32(tmem + tlane + TM_S + 32, a);
          tc_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) x[32 + i] = valid ? __uint_as_float(a[i]) * c2 : -INFINITY;
        }
        tc_fence_before();
        mbar_arrive(bar_addr(c, B_SEMPTY));
        ++n_qk;
        // does any score exceed its head's reference max by more than 2^8?
        float dmax = -INFINITY;
#pragma unroll
        for (int h = 0; h < 64; ++h) dmax = fmaxf(dmax, x[h] - s_mref[h]);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) dmax = fmaxf(dmax, __shfl_xor_sync(0xFFFFFFFFu, dmax, o));
        const float* fl = s_flag + 4 * (n_qk & 1);
        if (lane == 0) s_flag[4 * (n_qk & 1) + q4] = dmax;
        if (!grp_sync()) { ok = false; break; }
        // fold the previous tile's row sums into the running sum (fixed order)
        if (tt > 0 && r < 64) {
          const float* lp = s_lpart + 256 * ((n_pv - 1) & 1);
          s_lacc[r] += ((lp[r] + lp[64 + r]) + lp[128 + r]) + lp[192 + r];
        }
        const float need_v = fmaxf(fmaxf(fl[0], fl[1]), fmaxf(fl[2], fl[3]));
        const bool need = !(need_v <= 8.0f);
        if (need) {
#pragma unroll
          for (int hb = 0; hb < 4; ++hb) {
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = x[16 * hb + i];
            reduce16<true>(v, lane);
            s_red[q4 * 64 + 16 * hb + (lane >> 1)] = v[0];
          }
          if (!grp_sync()) { ok = false; break; }
          if (r < 64) {
            const float tm = fmaxf(fmaxf(s_red[r], s_red[64 + r]), fmaxf(s_red[128 + r], s_red[192 + r]));
            const float mo = s_mref[r];
            const float mn = fmaxf(mo, tm);
            const float al = (mn == -INFINITY) ? 1.f : exp2f(mo - mn);
            s_mref[r] = mn;
            s_alpha[r] = al;
            s_lacc[r] *= al;
          }
          if (!grp_sync()) { ok = false; break; }
        }
        // previous PV must be complete before O is rescaled or P overwritten
        if (!wait_bar_w(c, B_PEMPTY, (n_pv & 1) ^ 1)) { ok = false; break; }
        tc_fence_after();
        // P row r (fp16) into SMEM, heads contiguous (MN-major B operand of PV)
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float p0 = exp2f(x[2 * i] - s_mref[2 * i]);
          const float p1 = exp2f(x[2 * i + 1] - s_mref[2 * i + 1]);
          pk[i] = pack_f16x2(p0, p1);
        }
        {
          const uint32_t rsw = (uint32_t)(r & 7);
          const uint32_t base = c.sb + SM_P + (uint32_t)(r >> 3) * 1024 + rsw * 128;
#pragma unroll
          for (int cc = 0; cc < 8; ++cc)
            sts128(base + ((cc ^ rsw) << 4), make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]));
        }
        // lazy rescale of the O accumulator (only when the reference max moved)
        if (need && tt > 0) {
#pragma unroll 1
          for (int j = 0; j < 4; ++j) {
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
              uint32_t a[32];
              const uint32_t ta = tmem + tlane + TM_O + 64 * j + 32 * half;
              tmem_ld32(ta, a);
              tc_wait_ld();
              const float* al = s_alpha + 32 * half;
#pragma unroll
              for (int i = 0; i < 32; ++i) a[i] = __float_as_uint(__uint_as_float(a[i]) * al[i]);
              tmem_st32(ta, a);
            }
          }
          tc_wait_st();
        }
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(bar_addr(c, B_PFULL));
        ++n_pv;
        // row sums of the rounded P
#pragma unroll
        for (int hb = 0; hb < 4; ++hb) {
          float v[16];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            v[2 * i] = f16lo(pk[8 * hb + i]);
            v[2 * i + 1] = f16hi(pk[8 * hb + i]);
          }
          reduce16<false>(v, lane);
          if ((lane & 1) == 0) s_lpart[256 * ((n_pv - 1) & 1) + 64 * q4 + 16 * hb + (lane >> 1)] = v[0];
        }
      }
      // ---------------------------------------------------------- epilogue
      if (ok && T > 0) {
        ok = wait_bar_w(c, B_ODONE, n_item_tiles & 1);
        tc_fence_after();
      }
      if (ok && !grp_sync()) ok = false;   // every warp's last row sums are written
      if (ok && T > 0 && r < 64) {
        const float* lp = s_lpart + 256 * ((n_pv - 1) & 1);
        s_lacc[r] += ((lp[r] + lp[64 + r]) + lp[128 + r]) + lp[192 + r];
      }
      if (ok && !grp_sync()) ok = false;
      if (ok) {
        const bool is_split = P.n_splits > 1;
        const float ln2 = 0.69314718055994531f;
        // per-head finals for this CTA's rows
        bool last = true;
        if (is_split) {
          // publish the partial (normalised O and LSE in log2 units)
          for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              uint32_t a[32];
              if (T > 0) {
                tmem_ld32(tmem + tlane + TM_O + 64 * j + 32 * half, a);
                tc_wait_ld();
              }
              const int d = 128 * j + r;
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const int h = 32 * half + i;
                const float l = s_lacc[h];
                const float o = (T > 0 && l > 0.f) ? __uint_as_float(a[i]) / l : 0.f;
                P.part_o[(((size_t)t * P.n_splits + split) * HP + h) * D_LAT + d] = o;
              }
            }
          }
          if (r < 64) {
            const float l = s_lacc[r];
            P.part_lse[((size_t)t * P.n_splits + split) * HP + r] = (T > 0 && l > 0.f) ? s_mref[r] + log2f(l) : -INFINITY;
          }
          __threadfence();
          if (!grp_sync()) ok = false;
          if (ok && r == 0) {
            const uint32_t old = atomicAdd(&P.counters[t], 1u);
            const int is_last = (old == (uint32_t)(P.n_splits - 1));
            if (is_last) P.counters[t] = 0u;
            c.info[I_LAST] = is_last;
          }
          if (ok && !grp_sync()) ok = false;
          last = ok && c.info[I_LAST] != 0;
          if (last) __threadfence();
        }
        if (ok && last) {
          // combine weights per head (split) or plain normalisation
          float lse_out = -INFINITY;
          if (r < 64) {
            if (is_split) {
              float M = -INFINITY;
              for (int s = 0; s < P.n_splits; ++s)
                M = fmaxf(M, __ldcg(&P.part_lse[((size_t)t * P.n_splits + s) * HP + r]));
              float den = 0.f;
              for (int s = 0; s < P.n_splits; ++s) {
                const float ls = __ldcg(&P.part_lse[((size_t)t * P.n_splits + s) * HP + r]);
                const float w = (M == -INFINITY) ? 0.f : exp2f(ls - M);
                den += w;
              }
              lse_out = (den > 0.f) ? (M + log2f(den)) * ln2 : -INFINITY;
              s_alpha[r] = M;                    // combine reference per head
              s_lacc[r] = den;                   // combine denominator per head
            } else {
              const float l = s_lacc[r];
              lse_out = (T > 0 && l > 0.f) ? (s_mref[r] + log2f(l)) * ln2 : -INFINITY;
              s_alpha[r] = (T > 0 && l > 0.f) ? 1.f / l : 0.f;
            }
            if (P.out_lse && r < P.h_q) P.out_lse[(size_t)t * P.h_q + r] = lse_out;
          }
          if (!grp_sync()) ok = false;
          for (int j = 0; j < 4 && ok; ++j) {
            float o[64];
            const int d = 128 * j + r;
            if (is_split) {
#pragma unroll
              for (int h = 0; h < 64; ++h) o[h] = 0.f;
#pragma unroll 1
              for (int sp = 0; sp < P.n_splits; ++sp) {
                const size_t base = ((size_t)t * P.n_splits + sp) * HP;
#pragma unroll
                for (int h = 0; h < 64; ++h) {
                  const float M = s_alpha[h];
                  const float w = (M == -INFINITY) ? 0.f : exp2f(__ldcg(&P.part_lse[base + h]) - M);
                  if (w > 0.f) o[h] = fmaf(w, __ldcg(&P.part_o[(base + h) * D_LAT + d]), o[h]);
                }
              }
#pragma unroll
              for (int h = 0; h < 64; ++h) {
                const float den = s_lacc[h];
                o[h] = den > 0.f ? o[h] / den : 0.f;
              }
            } else {
#pragma unroll
              for (int half = 0; half < 2; ++half) {
                uint32_t a[32];
                if (T > 0) {
                  tmem_ld32(tmem + tlane + TM_O + 64 * j + 32 * half, a);
                  tc_wait_ld();
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) o[32 * half + i] = (T > 0) ? __uint_as_float(a[i]) * s_alpha[32 * half + i] : 0.f;
              }
            }
            // inverse RoPE on dims 448..511 (pairs are adjacent lanes)
            if (j == 3 && q4 >= 2) {
              const float2 cs = s_rope[(d - 448) >> 1];
              const bool odd = lane & 1;
#pragma unroll
              for (int h = 0; h < 64; ++h) {
                const float other = __shfl_xor_sync(0xFFFFFFFFu, o[h], 1);
                o[h] = odd ? fmaf(-other, cs.y, o[h] * cs.x) : fmaf(other, cs.y, o[h] * cs.x);
                o[h] += 0.0f;   // a rotated exact zero stays +0 (empty tokens output +0 codes)
              }
            }
            if (P.out_precast) {
#pragma unroll
              for (int h = 0; h < 64; ++h)
                if (h < P.h_q) P.out_precast[((size_t)t * P.h_q + h) * D_LAT + d] = o[h];
            }
            // MXFP8: block = this warp's 32 lanes (32 consecutive dims) for each head
            float* sc = s_red + q4 * 64;
#pragma unroll
            for (int hb = 0; hb < 4; ++hb) {
              float am[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) am[i] = fabsf(o[16 * hb + i]);
              reduce16<true>(am, lane);
              const int h = 16 * hb + (lane >> 1);
              const int ex = (int)((__float_as_uint(am[0]) >> 23) & 0xFF);
              int E = ex - 127 - 8;
              E = E < -127 ? -127 : E;
              if ((lane & 1) == 0) {
                sc[h] = __uint_as_float((uint32_t)(127 - E) << 23);
                if (h < P.h_q) P.out_sf[((size_t)t * P.h_q + h) * 16 + 4 * j + q4] = (uint8_t)(E + 127);
              }
            }
            __syncwarp();
            uint32_t wq[16];
#pragma unroll
            for (int g = 0; g < 16; ++g) {
              const uint32_t lo = f32x2_to_e4m3x2(o[4 * g] * sc[4 * g], o[4 * g + 1] * sc[4 * g + 1]);
              const uint32_t hi = f32x2_to_e4m3x2(o[4 * g + 2] * sc[4 * g + 2], o[4 * g + 3] * sc[4 * g + 3]);
              wq[g] = lo | (hi << 16);
            }
            __syncwarp();
            // 4x4 byte transpose inside lane quads: lane 4k+i gets head 4g+i for dims 4k..4k+3
            const int qi = lane & 3;
            const int dbase = 128 * j + 32 * q4 + 4 * (lane >> 2);
#pragma unroll
            for (int g = 0; g < 16; ++g) {
              uint32_t res = ((wq[g] >> (8 * qi)) & 0xFFu) << (8 * qi);
#pragma unroll
              for (int rr = 1; rr < 4; ++rr) {
                const uint32_t src = __shfl_xor_sync(0xFFFFFFFFu, wq[g], rr);
                res |= ((src >> (8 * qi)) & 0xFFu) << (8 * (qi ^ rr));
              }
              const int h = 4 * g + qi;
              if (h < P.h_q)
                *reinterpret_cast<uint32_t*>(P.out_fp8 + ((size_t)t * P.h_q + h) * D_LAT + dbase) = res;
            }
          }
        }
      }
      if (ok && T > 0) ++n_item_tiles;
    }
    // all roles leave the item here
    if (!ok) c.info[I_ABORT] = 1;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (c.info[I_ABORT]) break;
  }

  // ---------------------------------------------------------- teardown
  __syncthreads();
  if (warp == MMA_WARP) {
    if (c.info[I_ABORT] && lane == 0) {
      // drain whatever the tensor core still has in flight before TMEM is released
      tc_commit(bar_addr(c, B_DRAIN));
      const unsigned long long start = clock64();
      while (!mbar_try(bar_addr(c, B_DRAIN), 0) && clock64() - start < WAIT_LIMIT_CYCLES) {
      }
    }
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TM_COLS) : "memory");
  }
}

// ------------------------------------------------------------------ host side
struct Layout {
  size_t status_off, counters_off, part_o_off, part_lse_off, total;
};

static int pick_splits(int s_q, int topk, int num_sms) {
  if (s_q <= 0) return 1;
  const int tiles = (topk + TILE - 1) / TILE;
  if (tiles <= 1 || s_q >= num_sms) return 1;
  int sp = num_sms / s_q;
  if (sp > tiles) sp = tiles;
  return sp < 1 ? 1 : sp;
}

static Layout layout_for(int s_q, int n_splits) {
  Layout L;
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  L.status_off = 0;
  L.counters_off = 256;
  size_t off = up(L.counters_off + 4 * (size_t)(s_q > 0 ? s_q : 1));
  if (n_splits > 1) {
    L.part_o_off = off;
    off = up(off + (size_t)s_q * n_splits * HP * D_LAT * 4);
    L.part_lse_off = off;
    off = up(off + (size_t)s_q * n_splits * HP * 4);
  } else {
    L.part_o_off = L.part_lse_off = 0;
  }
  L.total = off;
  return L;
}

static int device_sms(int* out_dev) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (out_dev) *out_dev = dev;
  return n;
}

static int check_params(const dsa_params* p) {
  if (!p) return DSA_ERR_INVALID_ARG;
  if (p->s_q < 0 || p->topk < 0 || p->n_swa_cols < 0 || p->n_swa_cols > p->topk) return DSA_ERR_INVALID_ARG;
  if (p->n_swa_rows < 0 || p->n_cmp_rows < 0) return DSA_ERR_INVALID_ARG;
  if (p->n_swa_rows >= (1ll << 31) || p->n_cmp_rows >= (1ll << 31)) return DSA_ERR_UNSUPPORTED_SHAPE;
  if (p->h_q < 1 || p->h_q > DSA_MAX_HEADS) return DSA_ERR_UNSUPPORTED_SHAPE;
  if (p->topk > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED_SHAPE;
  if (!(p->softmax_scale == p->softmax_scale) || !(p->rope_base > 0.f) || !(p->rms_eps >= 0.f))
    return DSA_ERR_INVALID_ARG;
  if (p->flags & ~DSA_FLAG_CHECK_INDICES) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

static bool aligned(const void* ptr, size_t a) { return ((uintptr_t)ptr % a) == 0; }

static int launch(const void* q, const void* kv_swa, const void* kv_cmp, const int32_t* indices,
                  const int32_t* topk_length, const int32_t* positions, const void* norm_w, void* out_fp8,
                  uint8_t* out_sf, float* out_precast, float* lse, const dsa_params* p, void* workspace,
                  size_t workspace_bytes, void* stream) {
  int rc = check_params(p);
  if (rc != DSA_OK) return rc;
  if (p->s_q == 0) return DSA_OK;
  const bool uses_swa = p->n_swa_cols > 0, uses_cmp = p->topk > p->n_swa_cols;
  if (!q || !topk_length || !positions || !norm_w || !out_fp8 || !out_sf || !workspace) return DSA_ERR_INVALID_ARG;
  if (p->topk > 0 && !indices) return DSA_ERR_INVALID_ARG;
  if ((uses_swa && !kv_swa) || (uses_cmp && !kv_cmp)) return DSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || (kv_swa && !aligned(kv_swa, 16)) || (kv_cmp && !aligned(kv_cmp, 16)) ||
      !aligned(out_fp8, 4) || !aligned(indices, 4) || !aligned(workspace, 256) || !aligned(norm_w, 2) ||
      (out_precast && !aligned(out_precast, 4)) || (lse && !aligned(lse, 4)))
    return DSA_ERR_INVALID_ARG;
  int dev = 0;
  const int sms = device_sms(&dev);
  if (sms <= 0) return DSA_ERR_CUDA;
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) return DSA_ERR_UNSUPPORTED_DEVICE;
  const int ns = pick_splits(p->s_q, p->topk, sms);
  const Layout L = layout_for(p->s_q, ns);
  if (workspace_bytes < L.total) return DSA_ERR_WORKSPACE_TOO_SMALL;

  static int attr_done[64] = {0};
  if (dev < 64 && !attr_done[dev]) {
    if (cudaFuncSetAttribute(dsa_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES) !=
        cudaSuccess)
      return DSA_ERR_CUDA;
    attr_done[dev] = 1;
  }
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t* ws = (uint8_t*)workspace;
  if (cudaMemsetAsync(ws, 0, L.counters_off + 4 * (size_t)p->s_q, st) != cudaSuccess) return DSA_ERR_CUDA;

  KParams K;
  K.q = (const uint16_t*)q;
  K.kv_swa = (const uint8_t*)kv_swa;
  K.kv_cmp = (const uint8_t*)kv_cmp;
  K.indices = indices;
  K.topk_length = topk_length;
  K.positions = positions;
  K.norm_w = (const uint16_t*)norm_w;
  K.out_fp8 = (uint8_t*)out_fp8;
  K.out_sf = out_sf;
  K.out_precast = out_precast;
  K.out_lse = lse;
  K.part_o = ns > 1 ? (float*)(ws + L.part_o_off) : nullptr;
  K.part_lse = ns > 1 ? (float*)(ws + L.part_lse_off) : nullptr;
  K.counters = (uint32_t*)(ws + L.counters_off);
  K.status = (uint32_t*)(ws + L.status_off);
  K.s_q = p->s_q;
  K.h_q = p->h_q;
  K.topk = p->topk;
  K.n_swa_cols = p->n_swa_cols;
  K.n_swa_rows = p->n_swa_rows;
  K.n_cmp_rows = p->n_cmp_rows;
  K.score_scale_log2 = p->softmax_scale * 1.4426950408889634f;
  K.rope_base = p->rope_base;
  K.rms_eps = p->rms_eps;
  K.flags = p->flags;
  K.n_splits = ns;
  K.n_items = p->s_q * ns;
  const int grid = K.n_items < sms ? K.n_items : sms;
  dsa_fwd_kernel<<<grid, NTHREADS, SMEM_BYTES, st>>>(K);
  if (cudaGetLastError() != cudaSuccess) return DSA_ERR_CUDA;
  return DSA_OK;
}

}  // namespace dsa

// ------------------------------------------------------------------ C ABI
extern "C" {

int dsa_params_init(dsa_params* p, int32_t s_q, int32_t h_q, int32_t topk, int32_t n_swa_cols, int64_t n_swa_rows,
                    int64_t n_cmp_rows) {
  if (!p) return DSA_ERR_INVALID_ARG;
  p->s_q = s_q;
  p->h_q = h_q;
  p->topk = topk;
  p->n_swa_cols = n_swa_cols;
  p->n_swa_rows = n_swa_rows;
  p->n_cmp_rows = n_cmp_rows;
  p->softmax_scale = 0.041666666666666664f;  // 1/sqrt(576)
  p->rope_base = 10000.f;
  p->rms_eps = 1e-6f;
  p->flags = 0;
  return DSA_OK;
}

int dsa_sparse_attn_num_splits(const dsa_params* p, int num_sms) {
  if (dsa::check_params(p) != DSA_OK) return 0;
  if (num_sms <= 0) num_sms = dsa::device_sms(nullptr);
  if (num_sms <= 0) return 0;
  return dsa::pick_splits(p->s_q, p->topk, num_sms);
}

size_t dsa_sparse_attn_workspace_size(const dsa_params* p, int num_sms) {
  const int ns = dsa_sparse_attn_num_splits(p, num_sms);
  if (ns <= 0) return 0;
  return dsa::layout_for(p->s_q, ns).total;
}

int dsa_sparse_attn_fwd(const void* q, const void* kv_swa, const void* kv_cmp, const int32_t* indices,
                        const int32_t* topk_length, const int32_t* positions, const void* norm_w, void* out_fp8,
                        uint8_t* out_sf, const dsa_params* p, void* workspace, size_t workspace_bytes, void* stream) {
  return dsa::launch(q, kv_swa, kv_cmp, indices, topk_length, positions, norm_w, out_fp8, out_sf, nullptr, nullptr,
                     p, workspace, workspace_bytes, stream);
}

int dsa_sparse_attn_fwd_debug(const void* q, const void* kv_swa, const void* kv_cmp, const int32_t* indices,
                              const int32_t* topk_length, const int32_t* positions, const void* norm_w, void* out_fp8,
                              uint8_t* out_sf, float* out_precast, float* lse, const dsa_params* p, void* workspace,
                              size_t workspace_bytes, void* stream) {
  return dsa::launch(q, kv_swa, kv_cmp, indices, topk_length, positions, norm_w, out_fp8, out_sf, out_precast, lse,
                     p, workspace, workspace_bytes, stream);
}

int dsa_sparse_attn_read_status(const void* workspace, uint32_t* status, void* stream) {
  if (!workspace || !status) return DSA_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaStreamSynchronize(st) != cudaSuccess) return DSA_ERR_CUDA;
  if (cudaMemcpy(status, workspace, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return DSA_ERR_CUDA;
  return DSA_OK;
}

const char* dsa_error_string(int code) {
  switch (code) {
    case DSA_OK: return "ok";
    case DSA_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, or bad parameter)";
    case DSA_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (h_q outside [1,64], topk > 2048, pool >= 2^31 rows)";
    case DSA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small (see dsa_sparse_attn_workspace_size)";
    case DSA_ERR_CUDA: return "CUDA runtime error";
    case DSA_ERR_UNSUPPORTED_DEVICE: return "current device is not compute capability 10.3 (GB300)";
    default: return "unknown error";
  }
}

}  // extern "C"
