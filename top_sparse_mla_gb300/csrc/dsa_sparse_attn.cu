// Fused top-k sparse latent attention for GB300 (sm_103a): q RMSNorm + q RoPE +
// gather of fp8_ds_mla rows by index + QK^T + online softmax + PV + inverse RoPE +
// MXFP8 cast, in one persistent kernel (stages as named on "Deepseek V41 Attention
// MegaKernel", vLLM PR #56344, Purpose).
//
// Work item = (query token, KV split), taken from a global queue.  One CTA of 16 warps
// per SM; the warps are specialised and talk through mbarriers, so consecutive items
// and consecutive tiles overlap:
//
//   PREP  (warps 13-14) take an item; compact its valid index columns into a row list;
//                       rotary table; L2 prefetch of the rows; build q~ = RoPE(RMSNorm(q)
//                       * w) in fp16 as the B operand of QK^T (K-major, 128-byte swizzle)
//   KD    (warps 4-7)   one gathered row per thread -> fp16 K~ (fp32 scale folded) into a
//                       TMEM ring: the A operand of QK^T, lane = row
//   VD    (warps 0-3)   one gathered row per thread -> fp16 V~ into an SMEM ring in
//                       MN-major layout: the A operand of PV
//   QK    (warp 12)     S^T[128 rows x 64 heads]  = K~ . q~^T     (tcgen05, M=128 N=64)
//   PV    (warp 15)     O^T[512 dims x 64 heads] += V~^T . P^T    (tcgen05, M=128 N=64)
//   SM    (warps 8-11)  softmax over S^T (lazy running max, exp2, fp16 P), O rescale,
//                       then the epilogue: O / l, inverse RoPE, MXFP8 cast and stores, or
//                       the split partials and the last split's combine
//
// The two MMA issuers are separate threads so that QK^T of the next tile never waits
// behind PV of the previous one.  S^T and P are double-buffered.
// TMEM: O^T columns 0..255, S^T double buffer 256..383, K~ ring 384..511.
// Every mbarrier wait is bounded; on timeout the CTA raises DSA_STATUS_WAIT_TIMEOUT,
// every role leaves its loop, the tensor core is drained and TMEM freed.

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <math.h>
#include <mutex>
#include <stdint.h>

#include "dsa_sparse_attn.h"
#include "ptx_sm103.cuh"

namespace dsa {

constexpr int D_LAT = 512;
constexpr int D_QK = 576;
constexpr int ROW_BYTES = 656;
constexpr int TILE = 128;           // gathered rows per tile (the M of QK^T)
constexpr int HP = 64;              // heads as seen by the MMAs (padded)
constexpr int NTHREADS = 512;
constexpr int W_VD = 0, W_KD = 4, W_SM = 8, W_QK = 12, W_PREP = 13, N_PREP_WARPS = 2, W_PV = 15;
constexpr int N_PREP = 32 * N_PREP_WARPS;
constexpr int K_SLOTS = 4;          // TMEM ring of 32-column slots (64 dims of K~ each)
constexpr int V_SLOTS = 3;          // SMEM ring of [128 dims x 128 rows] fp16 blocks
constexpr int HC_PER_TILE = 9;      // 8 latent half-chunks (64 dims) + the rope chunk
constexpr int MAX_SPLITS = 16;

// TMEM columns
constexpr uint32_t TM_O = 0;
constexpr uint32_t TM_S = 256;      // + 64 * buffer
constexpr uint32_t TM_K = 384;      // + 32 * slot
constexpr uint32_t TM_COLS = 512;

// shared memory map (offsets from a 1024-aligned base)
constexpr uint32_t SM_Q = 0;                                 // q~: 9 K-atoms x 8 KB
constexpr uint32_t SM_V = SM_Q + 9 * 8192;                   // V~ ring: 3 x 32 KB
constexpr uint32_t SM_P = SM_V + V_SLOTS * 32768;            // P: 2 x 16 KB; epilogue slabs
constexpr uint32_t SM_KDBUF = SM_P + 2 * 16384;              // 4 KD warps x [32 rows x 128 B]
constexpr uint32_t SM_VDSC = SM_KDBUF + 4 * 4096;            // 4 VD warps x [32 rows x 4 scales]
constexpr uint32_t SM_ROPE = SM_VDSC + 4 * 512;              // 2 x 32 x (cos, sin)
constexpr uint32_t SM_ITEM = SM_ROPE + 2 * 32 * 8;           // 2 x item info (8 ints)
constexpr uint32_t SM_NORMW = SM_ITEM + 2 * 32;              // 576 fp32
constexpr uint32_t SM_MREF = SM_NORMW + D_QK * 4;            // 64 fp32 running max (log2 units)
constexpr uint32_t SM_LACC = SM_MREF + 256;                  // 64 fp32 running sum
constexpr uint32_t SM_ALPHA = SM_LACC + 256;                 // 64 fp32 rescale / 1/l
constexpr uint32_t SM_RED = SM_ALPHA + 256;                  // 4 warps x 64 fp32
constexpr uint32_t SM_LPART = SM_RED + 1024;                 // 2 x 4 warps x 64 fp32 row sums
constexpr uint32_t SM_FLAG = SM_LPART + 2048;                // 2 x 4 fp32
constexpr uint32_t SM_MISC = SM_FLAG + 32;                   // misc ints
constexpr uint32_t SM_BAR = SM_MISC + 64;                    // mbarriers
constexpr uint32_t SM_END = SM_BAR + 48 * 8;
constexpr uint32_t SMEM_BYTES = SM_END + 1024;               // + alignment slack
// the epilogue reuses the two P buffers: one [64 heads x 32 dims] fp32 slab per SM warp
// (rows of 128 bytes, 16-byte chunks XOR-swizzled by row), the combine weights after it
constexpr uint32_t EPI_SLAB_BYTES = HP * 32 * 4;
constexpr uint32_t SM_CW = SM_P;                             // MAX_SPLITS x 64 fp32 (combine)
static_assert(4 * EPI_SLAB_BYTES <= 2 * 16384, "epilogue slabs fit in the P buffers");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

enum {
  B_KFULL = 0, B_KEMPTY = B_KFULL + K_SLOTS, B_VFULL = B_KEMPTY + K_SLOTS, B_VEMPTY = B_VFULL + V_SLOTS,
  B_SFULL = B_VEMPTY + V_SLOTS, B_SEMPTY = B_SFULL + 2, B_PFULL = B_SEMPTY + 2, B_PEMPTY = B_PFULL + 2,
  B_ITFULL = B_PEMPTY + 2, B_ITEMPTY = B_ITFULL + 2,
  B_ODONE = B_ITEMPTY + 2, B_OFREE, B_QREADY, B_QFREE, B_GRP, B_PREP, B_DRAIN, B_COUNT
};
static_assert(B_COUNT <= 48, "barrier area");

enum { M_TMEM = 0, M_ABORT, M_LAST };                           // misc ints
enum { IT_ITEM = 0, IT_TOKEN, IT_SPLIT, IT_T, IT_ROW0, IT_NROWS }; // item info ints

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
  float* part_o;        // [s_q][n_splits][64][512]
  float* part_lse;      // [s_q][n_splits][64] (log2 units)
  uint32_t* counters;   // [s_q] split arrivals
  uint32_t* status;
  uint32_t* work;       // global item queue head
  uint32_t* lists;      // [grid][2][DSA_MAX_TOPK] compacted row lists (bit 31: compressed pool)
  int s_q, h_q, topk, n_swa_cols;
  long long n_swa_rows, n_cmp_rows;
  float score_scale_log2;   // softmax_scale * log2(e)
  float rms_eps;
  uint32_t flags;
  int n_splits;
  int n_items;
  // rotary frequency of pair i as a 64-bit fixed-point fraction of a turn:
  // rope_base^(-2i/64) / (2 pi) * 2^64
  unsigned long long rope_turns[32];
};

struct Ctx {
  uint8_t* sm;
  uint32_t sb;
  volatile int* misc;
  uint32_t* status;
};

constexpr unsigned long long WAIT_LIMIT_CYCLES = 4000000000ull;   // ~2 s at 2 GHz

DSA_DEV uint32_t bar(const Ctx& c, int i) { return c.sb + SM_BAR + 8u * (uint32_t)i; }

// Bounded wait: false when the limit passes (raising the abort flag and the status bit)
// or when another thread of the CTA has already aborted.
DSA_DEV bool wait_bar(const Ctx& c, int b, uint32_t parity) {
  const uint32_t addr = bar(c, b);
  if (mbar_try(addr, parity)) return true;
  const unsigned long long start = clock64();
  while (true) {
    if (mbar_try(addr, parity)) return true;
    if (c.misc[M_ABORT]) return false;
    if (clock64() - start > WAIT_LIMIT_CYCLES) {
      atomicOr(c.status, DSA_STATUS_WAIT_TIMEOUT);
      c.misc[M_ABORT] = 1;
      return false;
    }
  }
}
// Warp-collective form: the warp agrees on the outcome, so it never splits before a
// full-warp shuffle or TMEM access.
DSA_DEV bool wait_bar_w(const Ctx& c, int b, uint32_t parity) {
  const bool ok = wait_bar(c, b, parity);
  return __all_sync(0xFFFFFFFFu, ok);
}

DSA_DEV const uint8_t* row_ptr(const KParams& P, uint32_t e) {
  const uint8_t* base = (e & 0x80000000u) ? P.kv_cmp : P.kv_swa;
  return base + (size_t)(e & 0x7FFFFFFFu) * ROW_BYTES;
}

// ================================================================== PREP
// Scan, rotary table, prefetch and q~ for every item, one item ahead of the others.
DSA_DEV void prep_role(const KParams& P, const Ctx& c, int pw, int lane) {
  const int pt = pw * 32 + lane;
  int* s_items = reinterpret_cast<int*>(c.sm + SM_ITEM);
  // volatile: re-read per head group instead of 72 weights held in registers
  const volatile float* s_normw = reinterpret_cast<const volatile float*>(c.sm + SM_NORMW);
  uint32_t n_prep_sync = 0;
  auto prep_sync = [&]() -> bool {
    mbar_arrive(bar(c, B_PREP));
    const bool r = wait_bar_w(c, B_PREP, n_prep_sync & 1);
    ++n_prep_sync;
    return r;
  };
  for (uint32_t seq = 0;; ++seq) {
    const int b = seq & 1;
    int* info = s_items + 8 * b;
    if (!wait_bar_w(c, B_ITEMPTY + b, ((seq >> 1) & 1) ^ 1)) return;
    if (pt == 0) {
      const int item = (int)atomicAdd(P.work, 1u);
      info[IT_ITEM] = item < P.n_items ? item : -1;
    }
    if (!prep_sync()) return;
    const int item = info[IT_ITEM];
    if (item < 0) {
      mbar_arrive(bar(c, B_ITFULL + b));   // tells every role to stop
      return;
    }
    const int t = item / P.n_splits;
    const int split = item % P.n_splits;
    if (pw == 0) {
      // compact the valid columns (j < topk_length, index >= 0), 256 indices per load batch
      uint32_t* list = P.lists + ((size_t)blockIdx.x * 2 + b) * DSA_MAX_TOPK;
      int L = P.topk_length[t];
      L = L < 0 ? 0 : (L > P.topk ? P.topk : L);
      const int32_t* irow = P.indices + (size_t)t * P.topk;
      int count = 0;
      for (int base = 0; base < L; base += 256) {
        int v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int j = base + 32 * k + lane;
          v[k] = (j < L) ? __ldg(irow + j) : -1;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int j = base + 32 * k + lane;
          const bool cmp = j >= P.n_swa_cols;
          bool valid = v[k] >= 0;
          if (valid && (P.flags & DSA_FLAG_CHECK_INDICES)) {
            const long long nr = cmp ? P.n_cmp_rows : P.n_swa_rows;
            if ((long long)v[k] >= nr) {
              valid = false;
              atomicOr(P.status, DSA_STATUS_INDEX_OUT_OF_RANGE);
            }
          }
          const uint32_t bal = __ballot_sync(0xFFFFFFFFu, valid);
          if (valid) list[count + __popc(bal & ((1u << lane) - 1u))] = (uint32_t)v[k] | (cmp ? 0x80000000u : 0u);
          count += __popc(bal);
        }
      }
      const int n_tiles_tok = (count + TILE - 1) / TILE;
      const int tps = (n_tiles_tok + P.n_splits - 1) / P.n_splits;
      const int tile0 = split * tps;
      int tile1 = tile0 + tps;
      if (tile1 > n_tiles_tok) tile1 = n_tiles_tok;
      const int T = tile1 > tile0 ? tile1 - tile0 : 0;
      const int row0 = tile0 * TILE;
      const int nrows = T > 0 ? ((tile1 * TILE < count ? tile1 * TILE : count) - row0) : 0;
      __syncwarp();
      for (int r = lane; r < nrows; r += 32) prefetch_l2(row_ptr(P, list[row0 + r]), ROW_BYTES);
      if (lane == 0) {
        info[IT_TOKEN] = t;
        info[IT_SPLIT] = split;
        info[IT_T] = T;
        info[IT_ROW0] = row0;
        info[IT_NROWS] = nrows;
      }
    } else {
      // cos / sin of positions[t] * theta_i from an exact fixed-point count of turns
      float2* rope = reinterpret_cast<float2*>(c.sm + SM_ROPE) + 32 * b;
      const unsigned long long turns = (unsigned long long)(long long)P.positions[t] * P.rope_turns[lane];
      const float frac = (float)(turns >> 40) * 5.9604644775390625e-08f;   // top 24 bits / 2^24
      float sn, cs;
      sincospif(2.0f * frac, &sn, &cs);
      rope[lane] = make_float2(cs, sn);
      if (lane == 0) prefetch_l2(P.q + (size_t)t * P.h_q * D_QK, (uint32_t)(P.h_q * D_QK * 2));
    }
    if (!prep_sync()) return;
    mbar_arrive(bar(c, B_ITFULL + b));   // rows, table and tile range published

    // q~ for this item, once the previous item's QK^T no longer reads the buffer.
    // Eight lanes per head, four heads per warp at a time, the next four heads' loads
    // in flight while the current ones are normalised and stored.
    if (!wait_bar_w(c, B_QFREE, (seq & 1) ^ 1)) return;
    if (info[IT_T] > 0) {
      const float2* rope = reinterpret_cast<const float2*>(c.sm + SM_ROPE) + 32 * b;
      const float eps = P.rms_eps;
      const int sub = lane >> 3, sl = lane & 7;     // head slot within the group, lane within the head
      uint4 raw[2][9];
      auto load_group = [&](int h0, uint4 (&dst)[9]) {
        const int h = h0 + sub;
#pragma unroll
        for (int k = 0; k < 9; ++k)
          dst[k] = (h < P.h_q) ? ldg_nc(P.q + ((size_t)t * P.h_q + h) * D_QK + (sl + 8 * k) * 8)
                               : make_uint4(0, 0, 0, 0);
      };
      // warp pw builds heads [32 pw, 32 pw + 32), four at a time
      auto process = [&](const uint4 (&cur)[9], int it) {
        const int h = 32 * pw + 4 * it + sub;
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < 9; ++k) {
          const uint32_t w4[4] = {cur[k].x, cur[k].y, cur[k].z, cur[k].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float a = __uint_as_float(w4[e] << 16), bb = __uint_as_float(w4[e] & 0xFFFF0000u);
            ss = fmaf(a, a, fmaf(bb, bb, ss));
          }
        }
        ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 1);
        ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 2);
        ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 4);
        const float inv = rsqrtf(ss * (1.0f / D_QK) + eps);
        const bool live = h < P.h_q;
#pragma unroll
        for (int k = 0; k < 9; ++k) {
          const int ch = sl + 8 * k;           // 16-byte chunk of the head row (8 dims)
          const uint32_t w4[4] = {cur[k].x, cur[k].y, cur[k].z, cur[k].w};
          float x[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            x[2 * e] = __uint_as_float(w4[e] << 16) * inv * s_normw[ch * 8 + 2 * e];
            x[2 * e + 1] = __uint_as_float(w4[e] & 0xFFFF0000u) * inv * s_normw[ch * 8 + 2 * e + 1];
          }
          if (k == 8) {                         // chunks 64..71: the rotary dims 512..575
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 r = rope[(ch - 64) * 4 + e];
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
      };
      load_group(32 * pw, raw[0]);
#pragma unroll 1
      for (int it = 0; it < 8; it += 2) {
        load_group(32 * pw + 4 * (it + 1), raw[1]);
        process(raw[0], it);
        if (it + 2 < 8) load_group(32 * pw + 4 * (it + 2), raw[0]);
        process(raw[1], it + 1);
      }
      fence_async_smem();
    }
    mbar_arrive(bar(c, B_QREADY));
  }
}

// ================================================================== QK issuer
DSA_DEV void qk_role(const KParams& P, const Ctx& c, uint32_t tmem) {
  constexpr uint32_t IDESC_QK = idesc_f16(128, HP, 0, 0);
  const int* s_items = reinterpret_cast<const int*>(c.sm + SM_ITEM);
  uint32_t kq = 0, g = 0;
  for (uint32_t seq = 0;; ++seq) {
    const int b = seq & 1;
    const int* info = s_items + 8 * b;
    if (!wait_bar(c, B_ITFULL + b, (seq >> 1) & 1)) return;
    const int item = info[IT_ITEM];
    const int T = info[IT_T];
    mbar_arrive(bar(c, B_ITEMPTY + b));
    if (item < 0) return;
    if (!wait_bar(c, B_QREADY, seq & 1)) return;
    tc_fence_after();
    for (int tt = 0; tt < T; ++tt) {
      const uint32_t sb = g & 1;
      if (!wait_bar(c, B_SEMPTY + sb, ((g >> 1) & 1) ^ 1)) return;
      tc_fence_after();
      for (int hc = 0; hc < HC_PER_TILE; ++hc) {
        const uint32_t slot = kq % K_SLOTS;
        if (!wait_bar(c, B_KFULL + slot, (kq / K_SLOTS) & 1)) return;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t bd = sdesc(c.sb + SM_Q + hc * 8192 + kk * 32, 16, 1024);
          mma_ts(tmem + TM_S + 64 * sb, tmem + TM_K + 32 * slot + 8 * kk, bd, IDESC_QK, (hc | kk) ? 1u : 0u);
        }
        tc_commit(bar(c, B_KEMPTY + slot));
        ++kq;
      }
      tc_commit(bar(c, B_SFULL + sb));
      ++g;
    }
    tc_commit(bar(c, B_QFREE));   // once per item: q~ may be rebuilt after these MMAs
  }
}

// ================================================================== PV issuer
DSA_DEV void pv_role(const KParams& P, const Ctx& c, uint32_t tmem) {
  constexpr uint32_t IDESC_PV = idesc_f16(128, HP, 1, 1);
  const int* s_items = reinterpret_cast<const int*>(c.sm + SM_ITEM);
  uint32_t vq = 0, g = 0, n_ot = 0;
  for (uint32_t seq = 0;; ++seq) {
    const int b = seq & 1;
    const int* info = s_items + 8 * b;
    if (!wait_bar(c, B_ITFULL + b, (seq >> 1) & 1)) return;
    const int item = info[IT_ITEM];
    const int T = info[IT_T];
    mbar_arrive(bar(c, B_ITEMPTY + b));
    if (item < 0) return;
    for (int tt = 0; tt < T; ++tt) {
      if (tt == 0) {
        // the previous item's epilogue must have read O^T before it is overwritten
        if (n_ot > 0 && !wait_bar(c, B_OFREE, (n_ot - 1) & 1)) return;
        ++n_ot;
      }
      const uint32_t pb = g & 1;
      if (!wait_bar(c, B_PFULL + pb, (g >> 1) & 1)) return;
      tc_fence_after();
      for (int j = 0; j < 4; ++j) {
        const uint32_t slot = vq % V_SLOTS;
        if (!wait_bar(c, B_VFULL + slot, (vq / V_SLOTS) & 1)) return;
        tc_fence_after();
        const uint32_t vbase = c.sb + SM_V + slot * 32768;
        const uint32_t pbase = c.sb + SM_P + pb * 16384;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ad = sdesc(vbase + kk * 2048, 16384, 1024);
          const uint64_t bd = sdesc(pbase + kk * 2048, 16384, 1024);
          mma_ss(tmem + TM_O + 64 * j, ad, bd, IDESC_PV, (tt == 0 && kk == 0) ? 0u : 1u);
        }
        tc_commit(bar(c, B_VEMPTY + slot));
        ++vq;
      }
      tc_commit(bar(c, B_PEMPTY + pb));
      if (tt == T - 1) tc_commit(bar(c, B_ODONE));
      ++g;
    }
  }
}

// ================================================================== KD
// Rows reach the SM with coalesced loads (eight lanes read 128 contiguous bytes of a
// row), pass through a per-warp shared-memory transpose (16-byte chunks XOR-swizzled by
// row) and leave one row per thread, which is what a 32x32b TMEM store needs.
DSA_DEV void kd_role(const KParams& P, const Ctx& c, uint32_t tmem, int q4, int lane) {
  const uint32_t tlane = (uint32_t)(q4 * 32) << 16;
  const int* s_items = reinterpret_cast<const int*>(c.sm + SM_ITEM);
  const uint32_t xb = c.sb + SM_KDBUF + q4 * 4096;       // this warp's transpose buffer
  const int sub = lane >> 3, ch = lane & 7;             // loader view: row 4k + sub, chunk ch
  uint32_t kq = 0;
  for (uint32_t seq = 0;; ++seq) {
    const int b = seq & 1;
    const int* info = s_items + 8 * b;
    if (!wait_bar_w(c, B_ITFULL + b, (seq >> 1) & 1)) return;
    if (info[IT_ITEM] < 0) return;
    const int T = info[IT_T], row0 = info[IT_ROW0], nrows = info[IT_NROWS];
    const uint32_t* list = P.lists + ((size_t)blockIdx.x * 2 + b) * DSA_MAX_TOPK;
    for (int tt = 0; tt < T; ++tt) {
      const int r = q4 * 32 + lane;                     // this thread's row (TMEM lane)
      const bool valid = tt * TILE + r < nrows;
      const uint32_t entry = valid ? __ldg(list + row0 + tt * TILE + r) : 0u;
      const uint8_t* my = row_ptr(P, entry);
      __half2 s2[4];
      {
        const uint4 sc = valid ? ldg_nc(my + D_LAT) : make_uint4(0, 0, 0, 0);
        s2[0] = __float2half2_rn(__uint_as_float(sc.x));
        s2[1] = __float2half2_rn(__uint_as_float(sc.y));
        s2[2] = __float2half2_rn(__uint_as_float(sc.z));
        s2[3] = __float2half2_rn(__uint_as_float(sc.w));
      }
      // the eight rows this lane loads from
      const uint8_t* src[8];
      bool sv[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t e = __shfl_sync(0xFFFFFFFFu, entry, 4 * k + sub);
        sv[k] = __shfl_sync(0xFFFFFFFFu, valid ? 1 : 0, 4 * k + sub) != 0;
        src[k] = row_ptr(P, e) + 16 * ch;
      }
      // five 128-byte batches per row: latent 0..3, then the rope bytes 528..655
      auto load_batch = [&](int bt, uint4 (&L)[8]) {
        const int off = bt < 4 ? 128 * bt : 528;
#pragma unroll
        for (int k = 0; k < 8; ++k) L[k] = sv[k] ? ldg_nc(src[k] + off) : make_uint4(0, 0, 0, 0);
      };
      uint4 L[8];
      load_batch(0, L);
#pragma unroll
      for (int bt = 0; bt < 5; ++bt) {
        // stage the batch: row (4k + sub) chunk ch -> swizzled slot
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t row = 4 * k + sub;
          sts128(xb + row * 128 + (((uint32_t)ch ^ (row & 7)) << 4), L[k]);
        }
        __syncwarp();
        if (bt < 4) load_batch(bt + 1, L);                // next batch in flight
        const int nhalf = bt < 4 ? 2 : 1;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          if (hf >= nhalf) break;
          uint32_t v[32];
          if (bt < 4) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint4 w;
              const uint32_t chunk = (uint32_t)(4 * hf + i);
              asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                           : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                           : "r"(xb + (uint32_t)lane * 128 + ((chunk ^ ((uint32_t)lane & 7)) << 4)));
              dequant16(w, s2[bt], v + 8 * i);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              uint4 w;
              asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                           : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                           : "r"(xb + (uint32_t)lane * 128 + (((uint32_t)i ^ ((uint32_t)lane & 7)) << 4)));
              v[4 * i + 0] = bf16x2_to_f16x2(w.x);
              v[4 * i + 1] = bf16x2_to_f16x2(w.y);
              v[4 * i + 2] = bf16x2_to_f16x2(w.z);
              v[4 * i + 3] = bf16x2_to_f16x2(w.w);
            }
          }
          const uint32_t slot = kq % K_SLOTS;
          if (!wait_bar_w(c, B_KEMPTY + slot, ((kq / K_SLOTS) & 1) ^ 1)) return;
          tc_fence_after();
          tmem_st32(tmem + tlane + TM_K + 32 * slot, v);
          tc_wait_st();
          tc_fence_before();
          mbar_arrive(bar(c, B_KFULL + slot));
          ++kq;
        }
        __syncwarp();                                   // buffer free for the next batch
      }
    }
    mbar_arrive(bar(c, B_ITEMPTY + b));
  }
}

// ================================================================== VD
// Eight lanes per row read 128 contiguous bytes (one d-tile of the latent) and write the
// fp16 values straight into the MN-major V~ block; no thread-per-row mapping is needed.
DSA_DEV void vd_role(const KParams& P, const Ctx& c, int w, int lane) {
  const int* s_items = reinterpret_cast<const int*>(c.sm + SM_ITEM);
  float* s_sc = reinterpret_cast<float*>(c.sm + SM_VDSC + w * 512);   // [32 rows][4 scales]
  const int sub = lane >> 3, ch = lane & 7;
  uint32_t vq = 0;
  for (uint32_t seq = 0;; ++seq) {
    const int b = seq & 1;
    const int* info = s_items + 8 * b;
    if (!wait_bar_w(c, B_ITFULL + b, (seq >> 1) & 1)) return;
    if (info[IT_ITEM] < 0) return;
    const int T = info[IT_T], row0 = info[IT_ROW0], nrows = info[IT_NROWS];
    const uint32_t* list = P.lists + ((size_t)blockIdx.x * 2 + b) * DSA_MAX_TOPK;
    for (int tt = 0; tt < T; ++tt) {
      const int r = w * 32 + lane;
      const bool valid = tt * TILE + r < nrows;
      const uint32_t entry = valid ? __ldg(list + row0 + tt * TILE + r) : 0u;
      {
        const uint4 sc = valid ? ldg_nc(row_ptr(P, entry) + D_LAT) : make_uint4(0, 0, 0, 0);
        __syncwarp();                                   // previous tile's scales consumed
        *reinterpret_cast<uint4*>(s_sc + 4 * lane) = sc;
        __syncwarp();
      }
      const uint8_t* src[8];
      bool sv[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t e = __shfl_sync(0xFFFFFFFFu, entry, 4 * k + sub);
        sv[k] = __shfl_sync(0xFFFFFFFFu, valid ? 1 : 0, 4 * k + sub) != 0;
        src[k] = row_ptr(P, e) + 16 * ch;
      }
      uint4 L[2][8];
#pragma unroll
      for (int k = 0; k < 8; ++k) L[0][k] = sv[k] ? ldg_nc(src[k]) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (j < 3) {
#pragma unroll
          for (int k = 0; k < 8; ++k) L[(j + 1) & 1][k] = sv[k] ? ldg_nc(src[k] + 128 * (j + 1)) : make_uint4(0, 0, 0, 0);
        }
        const uint32_t slot = vq % V_SLOTS;
        if (!wait_bar_w(c, B_VEMPTY + slot, ((vq / V_SLOTS) & 1) ^ 1)) return;
        const uint32_t base = c.sb + SM_V + slot * 32768 + (uint32_t)(ch >> 2) * 16384;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t row = (uint32_t)(w * 32 + 4 * k + sub);
          const __half2 s2 = __float2half2_rn(s_sc[4 * (4 * k + sub) + j]);
          uint32_t v[8];
          dequant16(L[j & 1][k], s2, v);
          // dims [16 ch, 16 ch + 16) of the d-tile = 8-dim chunks 2(ch % 4), +1 of atom ch / 4
          const uint32_t rsw = row & 7;
          const uint32_t rb = base + (row >> 3) * 1024 + rsw * 128;
          const uint32_t c0 = (uint32_t)(2 * (ch & 3));
          sts128(rb + ((c0 ^ rsw) << 4), make_uint4(v[0], v[1], v[2], v[3]));
          sts128(rb + (((c0 + 1) ^ rsw) << 4), make_uint4(v[4], v[5], v[6], v[7]));
        }
        fence_async_smem();
        mbar_arrive(bar(c, B_VFULL + slot));
        ++vq;
      }
    }
    mbar_arrive(bar(c, B_ITEMPTY + b));
  }
}

// ================================================================== SM + epilogue
// Finish 32 consecutive output dims of one head: inverse RoPE, optional pre-cast store,
// MXFP8 (one 32-value block) and the stores.
DSA_DEV void finalize_block(const KParams& P, float (&v)[32], int t, int h, int d0, const float2* rope) {
  if (d0 >= 448) {
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float2 cs = rope[((d0 - 448) >> 1) + k];
      const float x0 = v[2 * k], x1 = v[2 * k + 1];
      v[2 * k] = fmaf(x1, cs.y, x0 * cs.x) + 0.0f;     // +0.0f: a rotated exact zero stays +0
      v[2 * k + 1] = fmaf(-x0, cs.y, x1 * cs.x) + 0.0f;
    }
  }
  const size_t row = (size_t)t * P.h_q + h;
  if (P.out_precast) {
    float4* dst = reinterpret_cast<float4*>(P.out_precast + row * D_LAT + d0);
#pragma unroll
    for (int k = 0; k < 8; ++k) dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
  }
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < 32; ++k) amax = fmaxf(amax, fabsf(v[k]));
  int E = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127 - 8;   // floor(log2 amax) - 8
  E = E < -127 ? -127 : E;
  const float inv = __uint_as_float((uint32_t)(127 - E) << 23);    // 2^-E, exact
  uint32_t wq[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t lo = f32x2_to_e4m3x2(v[4 * k] * inv, v[4 * k + 1] * inv);
    const uint32_t hi = f32x2_to_e4m3x2(v[4 * k + 2] * inv, v[4 * k + 3] * inv);
    wq[k] = lo | (hi << 16);
  }
  uint4* dst = reinterpret_cast<uint4*>(P.out_fp8 + row * D_LAT + d0);
  dst[0] = make_uint4(wq[0], wq[1], wq[2], wq[3]);
  dst[1] = make_uint4(wq[4], wq[5], wq[6], wq[7]);
  P.out_sf[row * 16 + (d0 >> 5)] = (uint8_t)(E + 127);
}

DSA_DEV void sm_role(const KParams& P, const Ctx& c, uint32_t tmem, int q4, int lane) {
  const int r = q4 * 32 + lane;
  const uint32_t tlane = (uint32_t)(q4 * 32) << 16;
  const int* s_items = reinterpret_cast<const int*>(c.sm + SM_ITEM);
  float* s_mref = reinterpret_cast<float*>(c.sm + SM_MREF);
  float* s_lacc = reinterpret_cast<float*>(c.sm + SM_LACC);
  float* s_alpha = reinterpret_cast<float*>(c.sm + SM_ALPHA);
  float* s_red = reinterpret_cast<float*>(c.sm + SM_RED);
  float* s_lpart = reinterpret_cast<float*>(c.sm + SM_LPART);
  float* s_cw = reinterpret_cast<float*>(c.sm + SM_CW);
  float* s_flag = reinterpret_cast<float*>(c.sm + SM_FLAG);
  // this warp's epilogue slab: 64 rows (heads) of 32 fp32 (dims), 16-byte chunks of a row
  // XOR-swizzled by (row & 7) so that both the column writes and the row reads are free
  // of bank conflicts
  uint8_t* slab = c.sm + SM_P + q4 * EPI_SLAB_BYTES;
  const float c2 = P.score_scale_log2;
  const float ln2 = 0.69314718055994531f;
  uint32_t g = 0, n_grp = 0, n_ot = 0;
  auto grp_sync = [&]() -> bool {
    mbar_arrive(bar(c, B_GRP));
    const bool ok = wait_bar_w(c, B_GRP, n_grp & 1);
    ++n_grp;
    return ok;
  };
  auto fold_lpart = [&](uint32_t tile) {
    if (r < 64) {
      const float* lp = s_lpart + 256 * (tile & 1);
      s_lacc[r] += ((lp[r] + lp[64 + r]) + lp[128 + r]) + lp[192 + r];
    }
  };
  for (uint32_t seq = 0;; ++seq) {
    const int b = seq & 1;
    const int* info = s_items + 8 * b;
    if (!wait_bar_w(c, B_ITFULL + b, (seq >> 1) & 1)) return;
    if (info[IT_ITEM] < 0) return;
    const int t = info[IT_TOKEN], split = info[IT_SPLIT], T = info[IT_T], nrows = info[IT_NROWS];
    const float2* rope = reinterpret_cast<const float2*>(c.sm + SM_ROPE) + 32 * b;
    if (r < 64) {
      s_mref[r] = -INFINITY;
      s_lacc[r] = 0.f;
    }
    if (!grp_sync()) return;

    for (int tt = 0; tt < T; ++tt) {
      const uint32_t sb = g & 1;
      const uint32_t ts = tmem + tlane + TM_S + 64 * sb;
      const bool valid = r < nrows - tt * TILE;
      if (!wait_bar_w(c, B_SFULL + sb, (g >> 1) & 1)) return;
      tc_fence_after();
      // pass 1: how far does this tile exceed the reference max of each head?
      float dmax = -INFINITY;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t a[32];
        tmem_ld32(ts + 32 * half, a);
        tc_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float x = valid ? __uint_as_float(a[i]) * c2 : -INFINITY;
          dmax = fmaxf(dmax, x - s_mref[32 * half + i]);
        }
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) dmax = fmaxf(dmax, __shfl_xor_sync(0xFFFFFFFFu, dmax, o));
      if (lane == 0) s_flag[4 * (g & 1) + q4] = dmax;
      if (!grp_sync()) return;
      if (tt > 0) fold_lpart(g - 1);
      const float* fl = s_flag + 4 * (g & 1);
      const float need_v = fmaxf(fmaxf(fl[0], fl[1]), fmaxf(fl[2], fl[3]));
      const bool need = !(need_v <= 8.0f);
      if (need) {
        // exact tile max per head, new reference max, rescale factors
#pragma unroll
        for (int hb = 0; hb < 4; ++hb) {
          uint32_t a[16];
          tmem_ld16(ts + 16 * hb, a);
          tc_wait_ld();
          float v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = valid ? __uint_as_float(a[i]) * c2 : -INFINITY;
          reduce16<true>(v, lane);
          s_red[q4 * 64 + 16 * hb + (lane >> 1)] = v[0];
        }
        if (!grp_sync()) return;
        if (r < 64) {
          const float tm = fmaxf(fmaxf(s_red[r], s_red[64 + r]), fmaxf(s_red[128 + r], s_red[192 + r]));
          const float mo = s_mref[r];
          const float mn = fmaxf(mo, tm);
          const float al = (mn == -INFINITY) ? 1.f : exp2f(mo - mn);
          s_mref[r] = mn;
          s_alpha[r] = al;
          s_lacc[r] *= al;
        }
        if (!grp_sync()) return;
      }
      // P buffer g & 1 is free once the PV two tiles back has completed
      const uint32_t pb = g & 1;
      if (!wait_bar_w(c, B_PEMPTY + pb, ((g >> 1) & 1) ^ 1)) return;
      // pass 2: P = exp2(x - m) in fp16, row r of the MN-major B operand; row sums
      const uint32_t prow = c.sb + SM_P + pb * 16384 + (uint32_t)(r >> 3) * 1024 + (uint32_t)(r & 7) * 128;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t a[32];
        tmem_ld32(ts + 32 * half, a);
        tc_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float x0 = valid ? __uint_as_float(a[2 * i]) * c2 : -INFINITY;
          const float x1 = valid ? __uint_as_float(a[2 * i + 1]) * c2 : -INFINITY;
          pk[i] = pack_f16x2(exp2f(x0 - s_mref[32 * half + 2 * i]), exp2f(x1 - s_mref[32 * half + 2 * i + 1]));
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const uint32_t chunk = (uint32_t)(4 * half + cc);
          sts128(prow + ((chunk ^ (uint32_t)(r & 7)) << 4),
                 make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]));
        }
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          float v[16];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            v[2 * i] = f16lo(pk[8 * hb + i]);
            v[2 * i + 1] = f16hi(pk[8 * hb + i]);
          }
          reduce16<false>(v, lane);
          if ((lane & 1) == 0) s_lpart[256 * (g & 1) + 64 * q4 + 32 * half + 16 * hb + (lane >> 1)] = v[0];
        }
      }
      tc_fence_before();
      mbar_arrive(bar(c, B_SEMPTY + sb));     // S^T fully read
      if (need && tt > 0) {
        // O^T is rescaled once the PV of the previous tile has completed
        if (!wait_bar_w(c, B_PEMPTY + ((g - 1) & 1), ((g - 1) >> 1) & 1)) return;
        tc_fence_after();
#pragma unroll 1
        for (int j = 0; j < 8; ++j) {
          uint32_t a[32];
          const uint32_t ta = tmem + tlane + TM_O + 32 * j;
          tmem_ld32(ta, a);
          tc_wait_ld();
          const float* al = s_alpha + 32 * (j & 1);
#pragma unroll
          for (int i = 0; i < 32; ++i) a[i] = __float_as_uint(__uint_as_float(a[i]) * al[i]);
          tmem_st32(ta, a);
        }
        tc_wait_st();
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(bar(c, B_PFULL + pb));
      ++g;
    }

    // ---------------------------------------------------------- epilogue
    if (T > 0) {
      if (!wait_bar_w(c, B_ODONE, n_ot & 1)) return;
      tc_fence_after();
    }
    if (!grp_sync()) return;                 // last row sums written, P buffers idle
    if (T > 0) fold_lpart(g - 1);
    const bool is_split = P.n_splits > 1;
    if (r < 64) {
      const float l = s_lacc[r];
      const bool any = T > 0 && l > 0.f;
      s_alpha[r] = any ? 1.f / l : 0.f;
      const float lse2 = any ? s_mref[r] + log2f(l) : -INFINITY;
      if (is_split) P.part_lse[((size_t)t * P.n_splits + split) * HP + r] = lse2;
      else if (P.out_lse && r < P.h_q) P.out_lse[(size_t)t * P.h_q + r] = lse2 * ln2;
    }
    if (!grp_sync()) return;
    // this warp's slabs: dims [128j + 32 q4, +32) of every head
    for (int j = 0; j < 4; ++j) {
      const int d0 = 128 * j + 32 * q4;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t a[32];
        if (T > 0) {
          tmem_ld32(tmem + tlane + TM_O + 64 * j + 32 * half, a);
          tc_wait_ld();
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int h = 32 * half + i;
          const float v = (T > 0) ? __uint_as_float(a[i]) * s_alpha[h] : 0.f;
          const uint32_t off = (uint32_t)h * 128 + ((((uint32_t)lane >> 2) ^ (uint32_t)(h & 7)) << 4) + (lane & 3) * 4;
          *reinterpret_cast<float*>(slab + off) = v;
        }
      }
      __syncwarp();
#pragma unroll 1
      for (int e = 0; e < 2; ++e) {
        const int h = lane + 32 * e;
        float v[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float4 f = *reinterpret_cast<const float4*>(slab + h * 128 + ((k ^ (h & 7)) << 4));
          v[4 * k] = f.x;
          v[4 * k + 1] = f.y;
          v[4 * k + 2] = f.z;
          v[4 * k + 3] = f.w;
        }
        if (is_split) {
          float4* dst = reinterpret_cast<float4*>(P.part_o + (((size_t)t * P.n_splits + split) * HP + h) * D_LAT + d0);
#pragma unroll
          for (int k = 0; k < 8; ++k) dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
        } else if (h < P.h_q) {
          finalize_block(P, v, t, h, d0, rope);
        }
      }
      __syncwarp();
    }
    if (T > 0) {
      tc_fence_before();
      mbar_arrive(bar(c, B_OFREE));          // O^T has been read
      ++n_ot;
    }
    if (is_split) {
      // the last split of the token to arrive combines all partials
      __threadfence();
      if (!grp_sync()) return;
      if (r == 0) {
        const uint32_t old = atomicAdd(&P.counters[t], 1u);
        const int last = (old == (uint32_t)(P.n_splits - 1));
        if (last) P.counters[t] = 0u;
        c.misc[M_LAST] = last;
      }
      if (!grp_sync()) return;
      if (c.misc[M_LAST]) {
        __threadfence();
        if (r < 64) {
          const float* pl = P.part_lse + (size_t)t * P.n_splits * HP + r;
          float M = -INFINITY;
          for (int s = 0; s < P.n_splits; ++s) M = fmaxf(M, __ldcg(pl + s * HP));
          float den = 0.f;
          for (int s = 0; s < P.n_splits; ++s) {
            const float w = (M == -INFINITY) ? 0.f : exp2f(__ldcg(pl + s * HP) - M);
            s_cw[s * 64 + r] = w;
            den += w;
          }
          const float inv = den > 0.f ? 1.f / den : 0.f;
          for (int s = 0; s < P.n_splits; ++s) s_cw[s * 64 + r] *= inv;
          if (P.out_lse && r < P.h_q) P.out_lse[(size_t)t * P.h_q + r] = den > 0.f ? (M + log2f(den)) * ln2 : -INFINITY;
        }
        if (!grp_sync()) return;
        for (int j = 0; j < 4; ++j) {
          const int d0 = 128 * j + 32 * q4;
#pragma unroll 1
          for (int e = 0; e < 2; ++e) {
            const int h = lane + 32 * e;
            if (h >= P.h_q) continue;
            float v[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = 0.f;
#pragma unroll 2
            for (int s = 0; s < P.n_splits; ++s) {
              const float w = s_cw[s * 64 + h];
              if (w == 0.f) continue;
              const float4* src =
                  reinterpret_cast<const float4*>(P.part_o + (((size_t)t * P.n_splits + s) * HP + h) * D_LAT + d0);
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const float4 f = __ldcg(src + k);
                v[4 * k] = fmaf(w, f.x, v[4 * k]);
                v[4 * k + 1] = fmaf(w, f.y, v[4 * k + 1]);
                v[4 * k + 2] = fmaf(w, f.z, v[4 * k + 2]);
                v[4 * k + 3] = fmaf(w, f.w, v[4 * k + 3]);
              }
            }
            finalize_block(P, v, t, h, d0, rope);
          }
        }
      }
      if (!grp_sync()) return;               // combine weights no longer needed
    }
    mbar_arrive(bar(c, B_ITEMPTY + b));
  }
}

// ================================================================== the kernel
__global__ void __launch_bounds__(NTHREADS, 1) dsa_fwd_kernel(const __grid_constant__ KParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Ctx c;
  {
    const uint32_t raw = smem_u32(smem_raw);
    c.sm = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  }
  c.sb = smem_u32(c.sm);
  c.misc = reinterpret_cast<volatile int*>(c.sm + SM_MISC);
  c.status = P.status;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < K_SLOTS; ++i) {
      mbar_init(bar(c, B_KFULL + i), 128);
      mbar_init(bar(c, B_KEMPTY + i), 1);
    }
    for (int i = 0; i < V_SLOTS; ++i) {
      mbar_init(bar(c, B_VFULL + i), 128);
      mbar_init(bar(c, B_VEMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(c, B_SFULL + i), 1);
      mbar_init(bar(c, B_SEMPTY + i), 128);
      mbar_init(bar(c, B_PFULL + i), 128);
      mbar_init(bar(c, B_PEMPTY + i), 1);
      mbar_init(bar(c, B_ITFULL + i), N_PREP);
      mbar_init(bar(c, B_ITEMPTY + i), 128 + 128 + 128 + 1 + 1);   // KD, VD, SM, QK, PV
    }
    mbar_init(bar(c, B_ODONE), 1);
    mbar_init(bar(c, B_OFREE), 128);
    mbar_init(bar(c, B_QREADY), N_PREP);
    mbar_init(bar(c, B_QFREE), 1);
    mbar_init(bar(c, B_GRP), 128);
    mbar_init(bar(c, B_PREP), N_PREP);
    mbar_init(bar(c, B_DRAIN), 2);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    c.misc[M_ABORT] = 0;
  }
  if (warp == W_QK) tmem_alloc(c.sb + SM_MISC + 4 * M_TMEM, TM_COLS);
  float* s_normw = reinterpret_cast<float*>(c.sm + SM_NORMW);
  for (int i = tid; i < D_QK; i += NTHREADS) s_normw[i] = __uint_as_float((uint32_t)P.norm_w[i] << 16);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = (uint32_t)c.misc[M_TMEM];

  if (warp == W_PV) {
    if (lane == 0) pv_role(P, c, tmem);
  } else if (warp >= W_PREP) {
    prep_role(P, c, warp - W_PREP, lane);
  } else if (warp == W_QK) {
    if (lane == 0) qk_role(P, c, tmem);
  } else if (warp >= W_SM) {
    sm_role(P, c, tmem, warp - W_SM, lane);
  } else if (warp >= W_KD) {
    kd_role(P, c, tmem, warp - W_KD, lane);
  } else {
    vd_role(P, c, warp - W_VD, lane);
  }

  tc_fence_before();
  __syncthreads();
  if ((warp == W_QK || warp == W_PV) && lane == 0) {
    // every MMA this CTA issued has completed before TMEM is released
    tc_commit(bar(c, B_DRAIN));
    const unsigned long long start = clock64();
    while (!mbar_try(bar(c, B_DRAIN), 0) && clock64() - start < WAIT_LIMIT_CYCLES) {
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == W_QK) {
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
}

// ================================================================== host side
struct Layout {
  size_t status_off, work_off, counters_off, lists_off, part_o_off, part_lse_off, total;
};

static int pick_splits(int s_q, int topk, int num_sms) {
  if (s_q <= 0) return 1;
  const int tiles = (topk + TILE - 1) / TILE;
  if (tiles <= 1 || s_q >= num_sms) return 1;
  int sp = num_sms / s_q;
  if (sp > tiles) sp = tiles;
  if (sp > MAX_SPLITS) sp = MAX_SPLITS;
  return sp < 1 ? 1 : sp;
}

static Layout layout_for(int s_q, int n_splits, int num_sms) {
  Layout L;
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  L.status_off = 0;
  L.work_off = 4;
  L.counters_off = 256;
  size_t off = up(L.counters_off + 4 * (size_t)(s_q > 0 ? s_q : 1));
  L.lists_off = off;
  off = up(off + (size_t)num_sms * 2 * DSA_MAX_TOPK * 4);
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

// rope_base^(-2i/64) / (2 pi) as a 64-bit fraction of a turn (the device multiplies it
// by the position modulo 2^64, which is the angle modulo 2 pi, exactly)
static void rope_turn_table(float base, unsigned long long* out) {
  const long double two_pi = 6.283185307179586476925286766559L;
  for (int i = 0; i < 32; ++i) {
    const long double theta = powl((long double)base, -2.0L * i / 64.0L);
    const long double frac = theta / two_pi;
    const long double f = frac - floorl(frac);
    out[i] = (unsigned long long)(f * 18446744073709551616.0L);
  }
}

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
      !aligned(out_fp8, 16) || !aligned(indices, 4) || !aligned(workspace, 256) || !aligned(norm_w, 2) ||
      (out_precast && !aligned(out_precast, 16)) || (lse && !aligned(lse, 4)))
    return DSA_ERR_INVALID_ARG;
  int dev = 0;
  const int sms = device_sms(&dev);
  if (sms <= 0) return DSA_ERR_CUDA;
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) return DSA_ERR_UNSUPPORTED_DEVICE;
  const int ns = pick_splits(p->s_q, p->topk, sms);
  const Layout L = layout_for(p->s_q, ns, sms);
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
  K.work = (uint32_t*)(ws + L.work_off);
  K.lists = (uint32_t*)(ws + L.lists_off);
  K.s_q = p->s_q;
  K.h_q = p->h_q;
  K.topk = p->topk;
  K.n_swa_cols = p->n_swa_cols;
  K.n_swa_rows = p->n_swa_rows;
  K.n_cmp_rows = p->n_cmp_rows;
  K.score_scale_log2 = p->softmax_scale * 1.4426950408889634f;
  K.rms_eps = p->rms_eps;
  K.flags = p->flags;
  K.n_splits = ns;
  K.n_items = p->s_q * ns;
  rope_turn_table(p->rope_base, K.rope_turns);
  const int grid = K.n_items < sms ? K.n_items : sms;
  dsa_fwd_kernel<<<grid, NTHREADS, SMEM_BYTES, st>>>(K);
  if (cudaGetLastError() != cudaSuccess) return DSA_ERR_CUDA;
  return DSA_OK;
}

// ------------------------------------------------------- allocation-free entry
// Scratch of dsa_sparse_attn_fwd_noalloc, in place of a caller-supplied workspace.
// It is zero-initialised device memory reserved when the module loads; its address is
// looked up once per device and cached.
static __device__ __align__(256) unsigned char g_noalloc_scratch[DSA_NOALLOC_SCRATCH_BYTES];
static std::mutex g_noalloc_mutex;
static void* g_noalloc_ptr[64];

static int noalloc_scratch(int dev, void** out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return DSA_ERR_CUDA;
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return DSA_OK;
}

static int launch_noalloc(const void* q, const void* kv_swa, const void* kv_cmp, const int32_t* indices,
                          const int32_t* topk_length, const int32_t* positions, const void* norm_w, void* out_fp8,
                          uint8_t* out_sf, const dsa_params* p, uint32_t* status_out, void* stream) {
  int rc = check_params(p);
  if (rc != DSA_OK) return rc;
  if (status_out && !aligned(status_out, 4)) return DSA_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (p->s_q == 0) {
    if (status_out && cudaMemsetAsync(status_out, 0, 4, st) != cudaSuccess) return DSA_ERR_CUDA;
    return DSA_OK;
  }
  int dev = 0;
  const int sms = device_sms(&dev);
  if (sms <= 0) return DSA_ERR_CUDA;
  if (dev < 0 || dev >= 64) return DSA_ERR_UNSUPPORTED_DEVICE;
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) return DSA_ERR_UNSUPPORTED_DEVICE;
  const Layout L = layout_for(p->s_q, pick_splits(p->s_q, p->topk, sms), sms);
  if (L.total > (size_t)DSA_NOALLOC_SCRATCH_BYTES) return DSA_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  rc = noalloc_scratch(dev, &scratch);
  if (rc != DSA_OK) return rc;
  // launch() clears the scratch header and the combine counters on `st` first
  rc = launch(q, kv_swa, kv_cmp, indices, topk_length, positions, norm_w, out_fp8, out_sf, nullptr, nullptr, p,
              scratch, DSA_NOALLOC_SCRATCH_BYTES, stream);
  if (rc != DSA_OK) return rc;
  if (status_out && cudaMemcpyAsync(status_out, (const uint8_t*)scratch + L.status_off, 4, cudaMemcpyDeviceToDevice,
                                    st) != cudaSuccess)
    return DSA_ERR_CUDA;
  return DSA_OK;
}

}  // namespace dsa

// ================================================================== C ABI
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
  if (num_sms <= 0) num_sms = dsa::device_sms(nullptr);
  if (num_sms <= 0) return 0;
  return dsa::layout_for(p->s_q, ns, num_sms).total;
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

int dsa_sparse_attn_fwd_noalloc(const void* q, const void* kv_swa, const void* kv_cmp, const int32_t* indices,
                                const int32_t* topk_length, const int32_t* positions, const void* norm_w,
                                void* out_fp8, uint8_t* out_sf, const dsa_params* p, uint32_t* status_out,
                                void* stream) {
  return dsa::launch_noalloc(q, kv_swa, kv_cmp, indices, topk_length, positions, norm_w, out_fp8, out_sf, p,
                             status_out, stream);
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
    case DSA_ERR_SCRATCH_LIMIT:
      return "shape needs more scratch than the no-alloc entry's built-in DSA_NOALLOC_SCRATCH_BYTES";
    default: return "unknown error";
  }
}

}  // extern "C"
