// Fused top-k sparse latent attention for GB300 (sm_103a): q RMSNorm + q RoPE +
// gather of fp8_ds_mla rows by index + QK^T + online softmax + PV + inverse RoPE +
// MXFP8 cast, in one persistent kernel (stages as named on "Deepseek V41 Attention
// MegaKernel", vLLM PR #56344, Purpose).
//
// Precision.  The two contractions run on fp16 tcgen05 MMAs with fp32 accumulation, and
// every operand is either exact in fp16 or carried as an exact-enough hi + lo pair:
//   - the latent tile holds the raw E4M3 codes (exact in fp16); each row's four fp32
//     block scales are applied in fp32, per 128-dim block, outside the MMA: QK^T runs one
//     partial score per block and the softmax warps add the partials times the scales;
//     PV runs one block of output dims per scale block with P scaled by that block's
//     scales (P_b = P * s_b);
//   - q~ = q * w (exact in fp32: 8-bit by 8-bit significands) and P_b go in as hi + lo,
//     both fp16; the MMA's N = 64 holds the work item's 32 heads twice, hi then lo, and
//     the two accumulators are added in fp32.
// A work item is therefore (query token, half of the heads, KV split): 32 heads.
//
// One CTA of 18 warps per SM; the warps are specialised and talk through mbarriers:
//
//   DQ   (warps 0-7)   when an item opens (right after the previous item's last QK^T):
//                      q~ hi/lo of its 32 heads as the B operand of QK^T, with a per-head
//                      power-of-two prescale, and the fp32 RMS statistics of q.  Per tile:
//                      gathered rows -> fp16 codes tile [128 rows x 512 dims] in shared
//                      memory.  The one tile is the A operand of both contractions:
//                      K-major for QK^T (M = rows), MN-major for PV (M = dims).  Raw bytes
//                      are loaded two chunks ahead, rows are prefetched into L2 one tile
//                      ahead; one tile ahead, the rotary part of the rows' keys (into
//                      TMEM) and their block scales (into shared memory).  Between items
//                      (no splits): the MXFP8 finish of output dims 128..383 of the
//                      previous item.
//   SX   (warps 8-15)  two groups of four, 16 heads each; one thread per tile row (TMEM
//                      lane).  Per tile: the five partial scores (four latent blocks,
//                      rope) summed with the row's block scales, the softmax (lazy running
//                      max, exp2), per-warp row sums, P_b hi/lo for the four PV blocks.
//                      Last tile of an item: 1/l and the LSE, then the epilogue of output
//                      dims 0..127 and 384..511, (O_hi + O_lo) / l out of TMEM (all 512
//                      dims as an fp32 partial on the split path)
//   MMA  (warp 16)     T_b[128 rows x 64] = codes_b . q~_b^T for b = 0..3 and the rope
//                      part; O^T_b[128 dims x 64] += codes_b^T . P_b
//   PREP (warp 17)     take an item, compact its valid index columns into a row list,
//                      the per-block reference scale of its rows, rotary table; up to
//                      three items ahead
//
// TMEM: O^T 0..255 (4 blocks x [32 hi | 32 lo]), partial scores 256..447 (three
// buffers), rope keys 448..511 (two).  Shared memory: q~ 72 KB, codes tile 128 KB, one
// 16 KB P buffer.  P_1 and P_2 borrow code chunk 0 once PV of block 0 has read it, so
// the next tile's QK^T takes its chunks in the order 1, 0, 2, 3, the order in which they
// come free.
// With few tokens each token's rows are split over several CTAs, one item per CTA, and
// the launch is cooperative: once its roles are done, every split of a (token, half)
// waits for the others and combines its share of the fp32 partial outputs.
// Every wait is bounded; on timeout the CTA raises DSA_STATUS_WAIT_TIMEOUT, every role
// leaves its loop, the tensor core is drained and TMEM freed.

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
constexpr int HH = 32;              // heads per work item
constexpr int NQ = 64;              // N of both contractions: 32 heads hi, then 32 lo
constexpr int W_SX = 8, W_MMA = 16, W_PREP = 17;
constexpr int NWARPS = 18;
constexpr int NTHREADS = 32 * NWARPS;
constexpr int N_DQ = 256, N_SX = 256;
constexpr int WG_DQ = N_DQ / 32, WG_SX = N_SX / 32;   // warps: the unit of the handoff barriers' counts
constexpr int MAX_SPLITS = 16;
constexpr int NB = 4;              // item buffers: the prep warp runs up to NB - 1 items ahead
constexpr int NSB = 3;             // partial-score buffers in TMEM
constexpr int NPART = 5;           // partial scores per tile: four latent blocks and the rope part

// TMEM columns
constexpr uint32_t TM_O = 0;
constexpr uint32_t TM_S = 256;      // + 64 * buffer
constexpr uint32_t TM_KR = 448;     // + 32 * buffer
constexpr uint32_t TM_COLS = 512;

// shared memory map (offsets from a 1024-aligned base)
constexpr uint32_t SM_Q = 0;                       // q~: 9 K-atoms x [64 rows x 128 B]
constexpr uint32_t SM_V = SM_Q + 9 * 8192;         // codes tile: 4 chunks x 2 halves x 16 KB
constexpr uint32_t SM_P = SM_V + 4 * 32768;        // P_0 / P_2: [128 rows x 64] fp16
constexpr uint32_t SM_ROPE = SM_P + 16384;         // NB x 32 x (cos, sin)
constexpr uint32_t SM_INV = SM_ROPE + NB * 256;    // NB x 32 fp32 score factors
constexpr uint32_t SM_RATIO = SM_INV + NB * 128;   // NB x 32 fp32 latent-to-rope score ratios (FP8 q)
constexpr uint32_t SM_ITEM = SM_RATIO + NB * 128;  // NB x 16 ints
constexpr uint32_t SM_M = SM_ITEM + NB * 64;       // 32 fp32 running max (log2 units)
constexpr uint32_t SM_ALPHA = SM_M + 128;          // 32 fp32 rescale factors
constexpr uint32_t SM_RED = SM_ALPHA + 128;        // 2 groups x 4 warps x 16 fp32
constexpr uint32_t SM_LW = SM_RED + 512;           // 2 x 8 warps x 16 fp32 row-sum partials
constexpr uint32_t SM_EL = SM_LW + 1024;           // 32 fp32 1/l
constexpr uint32_t SM_ELSE = SM_EL + 128;          // 32 fp32 LSE (log2 units)
constexpr uint32_t SM_FLAG = SM_ELSE + 128;        // 2 groups x 2 x 4 fp32
constexpr uint32_t SM_MISC = SM_FLAG + 64;         // misc ints
constexpr uint32_t SM_SCL = SM_MISC + 64;          // 2 x 128 rows x 4 fp32 block scales (a tile's rows)
constexpr uint32_t SM_BAR = SM_SCL + 2 * 128 * 16; // mbarriers
constexpr uint32_t SM_END = SM_BAR + 64 * 8;
constexpr uint32_t SMEM_BYTES = SM_END + 1024;     // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
// after the last item the codes tile area holds the split-combine weights
constexpr uint32_t SM_CW = SM_V;

enum {
  B_VFULL = 0, B_PVD = B_VFULL + 4, B_PFULL = B_PVD + 4, B_SFULL = B_PFULL + 4, B_SFREE = B_SFULL + NSB,
  B_KRFULL = B_SFREE + NSB, B_KRFREE = B_KRFULL + 2, B_ITFULL = B_KRFREE + 2, B_ITEMPTY = B_ITFULL + NB,
  B_ODONE = B_ITEMPTY + NB, B_OFREE, B_QRDY = B_OFREE + 4, B_QFREE = B_QRDY + 5, B_QSTAT, B_LREADY = B_QSTAT + NB,
  B_SXG, B_SXA = B_SXG + 2, B_DRAIN, B_NEVER, B_COUNT
};
static_assert(B_COUNT <= 64, "barrier area");

enum { M_TMEM = 0, M_ABORT, M_COMBINE, M_TOKEN, M_SPLIT, M_HALF };   // misc ints
// item info ints (16 per item buffer); IT_REF / IT_IREF hold 4 floats each
enum { IT_ITEM = 0, IT_TOKEN, IT_HALF, IT_SPLIT, IT_T, IT_ROW0, IT_NROWS, IT_REF = 8, IT_IREF = 12 };

// The QK^T order of the latent chunks (p-th partial -> chunk), the PV event after which
// chunk c of the codes tile may be overwritten by the next tile, and where P_b lives.
// P_0 goes into the shared P buffer; once PV(0) has completed, chunk 0 (two 16 KB halves)
// and the shared buffer take P_1, P_2 and P_3 together, so one handoff per tile gates PV.
// Chunk 1 is then free first (after PV(1)), chunks 0 and 2 after PV(2), chunk 3 after
// PV(3): the next tile's QK^T takes them in the order 1, 0, 2, 3.
DSA_DEV int qk_chunk(int p) { return p == 0 ? 1 : (p == 1 ? 0 : p); }
DSA_DEV int chunk_free_event(int c) { return c == 1 ? 1 : (c == 3 ? 3 : 2); }
DSA_DEV uint32_t p_buffer(int b) {
  return b == 1 ? SM_V : (b == 2 ? SM_V + 16384u : SM_P);
}

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
  float* part_o;        // split partials [s_q][n_splits][64 heads][512 dims]
  float* part_lse;      // [s_q][n_splits][64] (log2 units)
  uint32_t* counters;   // [s_q][n_halves] split arrivals (split path)
  const int32_t* order; // [s_q] tokens, most tiles first (queue path; shares the counters'
                        // region), or null: tokens in order
  uint32_t* status;
  uint32_t* work;       // global item queue head
  uint32_t* lists;      // [grid][NB][DSA_MAX_TOPK] compacted row lists (bit 31: compressed pool)
  int s_q, h_q, topk, n_swa_cols;
  long long n_swa_rows, n_cmp_rows;
  float score_scale_log2;   // softmax_scale * log2(e)
  float rms_eps;
  uint32_t flags;
  // nvfp4_ds_mla (the kernel's V41 instantiation): every kv_cmp value times cmp_scale
  float cmp_scale;
  int n_splits;
  int n_halves;             // 1 when h_q <= 32, else 2
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
// Arrival of a whole warp as one: after the warp's lanes meet (which orders their memory
// operations), lane 0 arrives.  Barriers that warps signal this way count warps, not
// threads, so a 256-thread handoff costs 8 arrive operations instead of 256.
DSA_DEV void arrive_w(const Ctx& c, int b) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar(c, b));
}

// The waiting part of a bounded wait, out of line: one copy serves every wait site (the
// code of all roles shares the SM's instruction caches).  False when the limit passes
// (raising the abort flag and the status bit) or when another thread of the CTA has
// already aborted.
__device__ __noinline__ bool wait_slow(uint32_t addr, uint32_t parity, volatile int* misc, uint32_t* status) {
  const unsigned long long start = clock64();
  while (true) {
    if (mbar_wait_susp(addr, parity)) return true;
    if (misc[M_ABORT]) return false;
    if (clock64() - start > WAIT_LIMIT_CYCLES) {
      atomicOr(status, DSA_STATUS_WAIT_TIMEOUT);
      misc[M_ABORT] = 1;
      return false;
    }
  }
}
// Bounded wait: one try inline, the rest out of line.
DSA_DEV bool wait_bar(const Ctx& c, int b, uint32_t parity) {
  const uint32_t addr = bar(c, b);
  if (mbar_try(addr, parity)) return true;
  return wait_slow(addr, parity, c.misc, c.status);
}
// Warp-collective form: the warp agrees on the outcome, so it never splits before a
// full-warp shuffle or TMEM access.
DSA_DEV bool wait_bar_w(const Ctx& c, int b, uint32_t parity) {
  const bool ok = wait_bar(c, b, parity);
  return __all_sync(0xFFFFFFFFu, ok);
}

// Group barrier of one role on an mbarrier (bounded, unlike bar.sync).
struct Group {
  int b;
  uint32_t n;
  DSA_DEV bool sync(const Ctx& c) {
    arrive_w(c, b);
    const bool ok = wait_bar_w(c, b, n & 1);
    ++n;
    return ok;
  }
};

// The kernel is compiled once per cache format (template argument V41: the
// nvfp4_ds_mla format), so that the format costs no run-time test in the hot loops.
template <bool V41>
struct Fmt {
  static constexpr int d_q = V41 ? DSA_NVFP4_QK_DIMS : D_QK;              // q / norm_w dims
  static constexpr uint32_t swa_row = V41 ? DSA_NVFP4_SWA_ROW_BYTES : ROW_BYTES;
  static constexpr uint32_t cmp_row = V41 ? DSA_NVFP4_CMP_ROW_BYTES : ROW_BYTES;
};
template <bool V41>
DSA_DEV const uint8_t* row_ptr(const KParams& P, uint32_t e) {
  const bool cmp = (e & 0x80000000u) != 0;
  return (cmp ? P.kv_cmp : P.kv_swa) + (size_t)(e & 0x7FFFFFFFu) * (cmp ? Fmt<V41>::cmp_row : Fmt<V41>::swa_row);
}
template <bool V41>
DSA_DEV uint32_t row_bytes(uint32_t e) {
  return (e & 0x80000000u) ? Fmt<V41>::cmp_row : Fmt<V41>::swa_row;
}
// An nvfp4_ds_mla compressed row: its values carry 16-dim E4M3 scales inside the row
// (folded into the fp16 codes by the dequant warps), and one fp32 scale for the pool.
template <bool V41>
DSA_DEV bool fp4_row(uint32_t e) { return V41 && (e & 0x80000000u) != 0; }
// The four fp32 block scales of a row (one per 128 dims) as raw bits: bytes 512..527 of
// an fp8 row; cmp_scale four times for an fp4 row.
template <bool V41>
DSA_DEV uint4 row_scales(const KParams& P, uint32_t e) {
  if (fp4_row<V41>(e)) {
    const uint32_t g = __float_as_uint(P.cmp_scale);
    return make_uint4(g, g, g, g);
  }
  return ldg_nc(row_ptr<V41>(P, e) + D_LAT);
}
DSA_DEV const uint32_t* item_list(const KParams& P, int b) {
  return P.lists + ((size_t)blockIdx.x * NB + b) * DSA_MAX_TOPK;
}
DSA_DEV const int* item_info(const Ctx& c, int b) { return reinterpret_cast<const int*>(c.sm + SM_ITEM) + 16 * b; }
DSA_DEV const float* item_ref(const Ctx& c, int b) {
  return reinterpret_cast<const float*>(c.sm + SM_ITEM) + 16 * b + IT_REF;
}
DSA_DEV const float* item_iref(const Ctx& c, int b) {
  return reinterpret_cast<const float*>(c.sm + SM_ITEM) + 16 * b + IT_IREF;
}

// Output pointers of the MXFP8 finish (passed by value to the out-of-line callers).
struct OutPtrs {
  uint8_t* fp8;
  uint8_t* sf;
  float* precast;
  int h_q;
  int sf_swizzled;   // DSA_FLAG_SF_SWIZZLED
};
DSA_DEV OutPtrs out_ptrs(const KParams& P) {
  return OutPtrs{P.out_fp8, P.out_sf, P.out_precast, P.h_q, (P.flags & DSA_FLAG_SF_SWIZZLED) ? 1 : 0};
}
// Byte offset of the scale code of (token t, head h, 32-dim block blk) in out_sf.  Row
// major: [s_q, h_q, 16].  Swizzled: the [s_q, 16 h_q] scale matrix (m = t, k = 16 h +
// blk) in 128 x 4 tiles of 512 bytes, tiles row-major; inside a tile, (m % 32, m / 32 %
// 4, k % 4) with strides 16, 4, 1 (FlashInfer's 128x4 swizzle, named on "[DSV4.1]
// Combine DSpark decode and prefill kernel optimizations", mHC MXFP8 epilogue).
DSA_DEV size_t sf_offset(const OutPtrs& O, int t, int h, int blk) {
  if (!O.sf_swizzled) return ((size_t)t * O.h_q + h) * 16 + blk;
  const int k = 16 * h + blk;
  return ((size_t)(t >> 7) * (size_t)(4 * O.h_q) + (size_t)(k >> 2)) * 512 + (size_t)((t & 31) * 16 + ((t >> 5) & 3) * 4 + (k & 3));
}

// ================================================================== PREP
// A (token, half) without a valid column on the queue path: o = 0, scale codes 0, LSE
// -inf, written by the prep warp (the item never enters the pipeline).
__device__ __noinline__ void write_empty_item(const KParams& P, int t, int half, int lane) {
  const int h0 = HH * half;
  const int nh = (P.h_q - h0) < HH ? (P.h_q - h0) : HH;
  for (int i = lane; i < nh * 32; i += 32) {
    const int h = h0 + (i >> 5), k = i & 31;
    reinterpret_cast<uint4*>(P.out_fp8 + ((size_t)t * P.h_q + h) * D_LAT)[k] = make_uint4(0, 0, 0, 0);
    if (P.out_precast) {
      float4* pc = reinterpret_cast<float4*>(P.out_precast + ((size_t)t * P.h_q + h) * D_LAT);
#pragma unroll
      for (int u = 0; u < 4; ++u) pc[4 * k + u] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  const OutPtrs O = out_ptrs(P);
  for (int i = lane; i < nh * 16; i += 32) P.out_sf[sf_offset(O, t, h0 + (i >> 4), i & 15)] = 0;
  if (P.out_lse && lane < nh) P.out_lse[(size_t)t * P.h_q + h0 + lane] = -INFINITY;
}

// (cos, sin) of positions[t] * theta_i, from an exact fixed-point count of turns
// (rope_turns[i]: the fraction of theta_i / 2 pi in units of 2^-64; the top 24 bits of the
// product are the fraction of a turn).
DSA_DEV float2 rope_entry_of(const KParams& P, int t, int i) {
  const unsigned long long turns = (unsigned long long)(long long)P.positions[t] * P.rope_turns[i];
  const float frac = (float)(turns >> 40) * 5.9604644775390625e-08f;   // top 24 bits / 2^24
  float sn, cs;
  sincospif(2.0f * frac, &sn, &cs);
  return make_float2(cs, sn);
}

DSA_DEV uint32_t redux_max_u32(uint32_t v) {
  uint32_t r;
  asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}

// Items, row lists, reference scales and rotary tables, ahead of the other roles.
template <bool V41>
DSA_DEV void prep_role(const KParams& P, const Ctx& c, int lane) {
  int* s_items = reinterpret_cast<int*>(c.sm + SM_ITEM);
  const bool split_path = P.n_splits > 1;
  // split path: exactly one item per CTA (the grid has one CTA per item), so the last
  // split of a (token, half) can run its combine with the whole CTA afterwards.
  // Otherwise items come from the global queue: position k is half k % n_halves of the
  // token P.order[k / n_halves] (tokens with the most tiles first, so that the last items
  // handed out are short ones; the halves of a token are adjacent, so the second reads
  // the rows from L2), each fetched one iteration before it is used.
  auto fetch = [&](uint32_t seq) -> int {
    int item = 0;
    if (lane == 0) {
      if (split_path) item = seq == 0 ? (int)blockIdx.x : P.n_items;
      else item = (int)atomicAdd(P.work, 1u);
      item = item < P.n_items ? item : -1;
    }
    return item;
  };
  if ((P.flags & DSA_FLAG_TEST_WAIT_TIMEOUT) && blockIdx.x == 0) {
    // test of the failure path: a wait that runs out, before this CTA takes an item
    wait_slow(bar(c, B_NEVER), 0, c.misc, c.status);
    return;
  }
  int next = fetch(0);
  for (uint32_t seq = 0;; ++seq) {
    const int b = seq % NB;
    int* info = s_items + 16 * b;
    if (!wait_bar_w(c, B_ITEMPTY + b, ((seq / NB) & 1) ^ 1)) return;
    // Take items until one has tiles.  On the queue path an item without a valid column
    // never enters the pipeline: its empty output is written here.  (The dequant warps
    // hold an item until they have converted the first tile of the next item with
    // tiles; a run of items without tiles could otherwise hold every buffer.)  The split
    // path takes its one item as it is: the combine needs every split.
    uint32_t* list = P.lists + ((size_t)blockIdx.x * NB + b) * DSA_MAX_TOPK;
    int item, t = 0, half = 0, split = 0, count = 0, T = 0, tile0 = 0, tile1 = 0;
    while (true) {
      item = __shfl_sync(0xFFFFFFFFu, next, 0);
      if (item < 0) break;
      next = fetch(seq + 1);
      if (split_path) {
        split = item % P.n_splits;
        half = (item / P.n_splits) % P.n_halves;
        t = item / (P.n_splits * P.n_halves);
      } else {
        const int k = item / P.n_halves;
        half = item % P.n_halves;
        t = P.order ? __ldcg(P.order + k) : k;
        split = 0;
      }
      // compact the valid columns (j < topk_length, index >= 0), 512 indices per load batch
      int L = P.topk_length[t];
      L = L < 0 ? 0 : (L > P.topk ? P.topk : L);
      const int32_t* irow = P.indices + (size_t)t * P.topk;
      count = 0;
      for (int base = 0; base < L; base += 512) {
        int v[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int j = base + 32 * k + lane;
          v[k] = (j < L) ? __ldg(irow + j) : -1;
        }
        // (not unrolled: the code of all roles shares the SM's instruction caches)
#pragma unroll 1
        for (int k = 0; k < 16; ++k) {
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
          if (valid) {
            const uint32_t e = (uint32_t)v[k] | (cmp ? 0x80000000u : 0u);
            list[count + __popc(bal & ((1u << lane) - 1u))] = e;
          }
          count += __popc(bal);
        }
      }
      const int n_tiles_tok = (count + TILE - 1) / TILE;
      const int tps = (n_tiles_tok + P.n_splits - 1) / P.n_splits;
      tile0 = split * tps;
      tile1 = tile0 + tps;
      if (tile1 > n_tiles_tok) tile1 = n_tiles_tok;
      T = tile1 > tile0 ? tile1 - tile0 : 0;
      if (split_path || T > 0) break;
      write_empty_item(P, t, half, lane);
    }
    if (item < 0) {
      if (lane == 0) info[IT_ITEM] = -1;
      arrive_w(c, B_ITFULL + b);   // tells every role to stop
      return;
    }
    const int row0 = tile0 * TILE;
    const int nrows = T > 0 ? ((tile1 * TILE < count ? tile1 * TILE : count) - row0) : 0;
    __syncwarp();   // the list entries of the other lanes
    // Reference scale of each latent block: the power of two at or below the largest
    // |scale| of the item's rows, so that P_b = P * scale / reference stays below 2 P.
    float mx[4] = {0.f, 0.f, 0.f, 0.f};
    for (int i = lane; i < nrows; i += 32) {
      const uint4 s = row_scales<V41>(P, __ldcg(list + row0 + i));
      mx[0] = fmaxf(mx[0], fabsf(__uint_as_float(s.x)));
      mx[1] = fmaxf(mx[1], fabsf(__uint_as_float(s.y)));
      mx[2] = fmaxf(mx[2], fabsf(__uint_as_float(s.z)));
      mx[3] = fmaxf(mx[3], fabsf(__uint_as_float(s.w)));
    }
    uint32_t ebits[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      int e = (int)((redux_max_u32(__float_as_uint(mx[k])) >> 23) & 0xFF);
      e = e < 1 ? 1 : (e > 253 ? 253 : e);
      ebits[k] = (uint32_t)e;
    }
    reinterpret_cast<float2*>(c.sm + SM_ROPE)[32 * b + lane] = rope_entry_of(P, t, lane);
    if (lane == 0) {
      info[IT_ITEM] = item;
      info[IT_TOKEN] = t;
      info[IT_HALF] = half;
      info[IT_SPLIT] = split;
      info[IT_T] = T;
      info[IT_ROW0] = row0;
      info[IT_NROWS] = nrows;
    }
    if (lane < 4) {
      info[IT_REF + lane] = (int)(ebits[lane] << 23);            // 2^(e - 127)
      info[IT_IREF + lane] = (int)((254u - ebits[lane]) << 23);  // 2^(127 - e)
    }
    arrive_w(c, B_ITFULL + b);   // rows, tile range, reference scales, rotary table
  }
}

// Finish eight consecutive output dims d0 .. d0 + 7 of head h in one of the four lanes
// (gmask) that share a 32-dim MXFP8 block: inverse RoPE, optional pre-cast store, the
// block amax across the four lanes, the UE8M0 code (stored by the block's first lane) and
// eight E4M3 codes.
DSA_DEV void finalize_eighth(const OutPtrs& O, float (&v)[8], int t, int h, int d0, unsigned gmask, const float2* rope) {
  if (d0 >= 448) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 cs = rope[((d0 - 448) >> 1) + k];
      const float x0 = v[2 * k], x1 = v[2 * k + 1];
      v[2 * k] = fmaf(x1, cs.y, x0 * cs.x) + 0.0f;     // +0.0f: a rotated exact zero stays +0
      v[2 * k + 1] = fmaf(-x0, cs.y, x1 * cs.x) + 0.0f;
    }
  }
  const size_t row = (size_t)t * O.h_q + h;
  if (O.precast) {
    float4* dst = reinterpret_cast<float4*>(O.precast + row * D_LAT + d0);
    dst[0] = make_float4(v[0], v[1], v[2], v[3]);
    dst[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(v[k]));
  amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, 2));
  int E = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127 - 8;   // floor(log2 amax) - 8
  E = E < -127 ? -127 : E;
  const float inv = __uint_as_float((uint32_t)(127 - E) << 23);    // 2^-E, exact
  uint32_t wq[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const uint32_t lo = f32x2_to_e4m3x2(v[4 * k] * inv, v[4 * k + 1] * inv);
    const uint32_t hi = f32x2_to_e4m3x2(v[4 * k + 2] * inv, v[4 * k + 3] * inv);
    wq[k] = lo | (hi << 16);
  }
  *reinterpret_cast<uint2*>(O.fp8 + row * D_LAT + d0) = make_uint2(wq[0], wq[1]);
  if ((d0 & 31) == 0) O.sf[sf_offset(O, t, h, d0 >> 5)] = (uint8_t)(E + 127);
}

// Finish dim d of heads h0..h0+N-1, one head per register; the 32 lanes of the warp hold
// one 32-dim MXFP8 block of each head.  Inverse RoPE with the neighbouring lane, optional
// pre-cast store, block amax across the warp (redux), UE8M0 code, E4M3 codes.  A head's
// stores from the 32 lanes are contiguous.
template <int N>
DSA_DEV void finalize_lanes(const OutPtrs& O, float (&v)[N], int t, int h0, int d, int lane, const float2* rope) {
  if (d >= 448) {
    const float2 cs = rope[(d - 448) >> 1];
    const bool odd = d & 1;
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const float o = __shfl_xor_sync(0xFFFFFFFFu, v[i], 1);
      // pair (x0, x1) rotated by -angle: (x0 c + x1 s, -x0 s + x1 c)
      v[i] = odd ? fmaf(-o, cs.y, v[i] * cs.x) + 0.0f : fmaf(o, cs.y, v[i] * cs.x) + 0.0f;
    }
  }
  const size_t row0 = (size_t)t * O.h_q + h0;
  if (O.precast) {
    float* pc = O.precast + row0 * D_LAT + d;
#pragma unroll
    for (int i = 0; i < N; ++i)
      if (h0 + i < O.h_q) pc[(size_t)i * D_LAT] = v[i];
  }
  uint8_t* out = O.fp8 + row0 * D_LAT + d;
  uint32_t sfw = 0;   // this lane's scale code (lane i < N: head h0 + i)
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    float am0, am1;
    asm volatile("redux.sync.max.abs.f32 %0, %1, 0xffffffff;" : "=f"(am0) : "f"(v[i]));
    asm volatile("redux.sync.max.abs.f32 %0, %1, 0xffffffff;" : "=f"(am1) : "f"(v[i + 1]));
    int e0 = (int)((__float_as_uint(am0) >> 23) & 0xFF) - 127 - 8;   // floor(log2 amax) - 8
    int e1 = (int)((__float_as_uint(am1) >> 23) & 0xFF) - 127 - 8;
    e0 = e0 < -127 ? -127 : e0;
    e1 = e1 < -127 ? -127 : e1;
    const float s0 = __uint_as_float((uint32_t)(127 - e0) << 23), s1 = __uint_as_float((uint32_t)(127 - e1) << 23);
    const uint32_t q = f32x2_to_e4m3x2(v[i] * s0, v[i + 1] * s1);
    if (h0 + i < O.h_q) out[(size_t)i * D_LAT] = (uint8_t)q;
    if (h0 + i + 1 < O.h_q) out[(size_t)(i + 1) * D_LAT] = (uint8_t)(q >> 8);
    sfw = lane == i ? (uint32_t)(e0 + 127) : (lane == i + 1 ? (uint32_t)(e1 + 127) : sfw);
  }
  if (lane < N && h0 + lane < O.h_q) O.sf[sf_offset(O, t, h0 + lane, d >> 5)] = (uint8_t)sfw;
}

// Epilogue of the 128-dim column block cidx of O^T by a warp on TMEM lane quarter q4
// (dims 128 cidx + 32 q4 + lane) for the item's heads hb .. hb + NH * ng - 1, NH at a
// time: (O_hi + O_lo) times the block's reference scale and 1/l from s_il.  The block's
// share is released on OFREE[cidx] once it has been read.  With part set the normalised
// partial is stored instead of finished.  (Out of line: its registers would otherwise
// count against the callers' loops.)
template <int NH>
__device__ __noinline__ void epi_chunk(const Ctx& c, uint32_t tmem, int q4, int lane, int cidx, int hb, int ng, const float* s_il,
                       float ref, const OutPtrs& O, int t, int h0, float* part, const float2* rope) {
  const uint32_t tlane = (uint32_t)(q4 * 32) << 16;
  const int d = 128 * cidx + 32 * q4 + lane;
#pragma unroll 1
  for (int hg = 0; hg < ng; ++hg) {
    const int col = hb + NH * hg;
    uint32_t a[NH], l[NH];
    if constexpr (NH == 16) {
      tmem_ld16(tmem + tlane + TM_O + 64 * cidx + col, a);
      tmem_ld16(tmem + tlane + TM_O + 64 * cidx + HH + col, l);
    } else {
      tmem_ld8(tmem + tlane + TM_O + 64 * cidx + col, a);
      tmem_ld8(tmem + tlane + TM_O + 64 * cidx + HH + col, l);
    }
    tc_wait_ld();
    const float4* il4 = reinterpret_cast<const float4*>(s_il + col);
    float v[NH];
#pragma unroll
    for (int q = 0; q < NH / 4; ++q) {
      const float4 f = il4[q];
      v[4 * q] = (__uint_as_float(a[4 * q]) + __uint_as_float(l[4 * q])) * (ref * f.x);
      v[4 * q + 1] = (__uint_as_float(a[4 * q + 1]) + __uint_as_float(l[4 * q + 1])) * (ref * f.y);
      v[4 * q + 2] = (__uint_as_float(a[4 * q + 2]) + __uint_as_float(l[4 * q + 2])) * (ref * f.z);
      v[4 * q + 3] = (__uint_as_float(a[4 * q + 3]) + __uint_as_float(l[4 * q + 3])) * (ref * f.w);
    }
    if (hg == ng - 1) {
      tc_fence_before();
      arrive_w(c, B_OFREE + cidx);   // this share of O^T has been read
    }
    if (part) {
      float* o = part + (size_t)col * D_LAT + d;
#pragma unroll
      for (int i = 0; i < NH; ++i) o[(size_t)i * D_LAT] = v[i];
    } else {
      finalize_lanes<NH>(O, v, t, h0 + col, d, lane, rope);
    }
  }
}

// ================================================================== q~
// q~ of one item without its RMS factor: q * w times a per-head power of two 2^k, RoPE
// on dims 512..575, as an fp16 hi + lo pair, the B operand of QK^T: row n < 32 holds the
// hi part of the item's head n, row 32 + n its lo part.  q * w is exact in fp32 (two
// 8-bit significands) and has at most 16 significant bits, so hi + lo is exact on the
// latent dims; on the rotated dims it is exact to about 2^-22.  2^k brings the head's
// largest |q * w| into [2^13, 2^14): the rotated pairs stay inside the fp16 range and the
// lo parts stay normal for every value that matters.  The per-head factor
// softmax_scale * log2(e) / (rms(q) 2^k) multiplies the scores instead (the rotation and
// QK^T are linear in q~).  Built by the 256 dequant threads in two passes over q (the
// statistics and the largest magnitude, then the operand): thread er covers head er / 8
// and the 8-dim chunk er % 8 of each of the 9 atoms.  Chunk c of the latent dims (atoms
// 2c, 2c + 1) is announced on QRDY[c], the rotary atom on QRDY[4], so that QK^T can start
// before the whole of q~ is written; the statistics follow on QSTAT[b].
struct QArgs {
  const uint16_t* q;
  const uint16_t* norm_w;
  int h_q;
  float eps, c2;
};

// With FP8Q (DSA_FLAG_FP8_Q) the latent rows of q~ hold E4M3 values instead (hi only, no
// lo part): code = E4M3(fl(q * w) * fl(448 / amax)), amax = the head's largest |q * w| over
// the 512 latent dims, decided in binary32 (the RMS factor cancels: this is the head's
// RMSNorm'd latent divided by its scale amax * rms / 448).  The rope part stays as above,
// and SM_RATIO[b][head] = 2^k / fl(448 / amax) turns the latent scores into the rope
// part's units.
template <bool V41, bool FP8Q>
DSA_DEV void build_q(const QArgs& P, const Ctx& c, int b, int er) {
  constexpr int d_q = Fmt<V41>::d_q;         // 576 (rotary atom 8) or 512 (rotary atom 7)
  const int* info = item_info(c, b);
  const int hs = er >> 3, chn = er & 7;
  const int h = HH * info[IT_HALF] + hs;
  const bool hv = h < P.h_q;
  const uint16_t* qh = P.q + ((size_t)info[IT_TOKEN] * P.h_q + (hv ? h : 0)) * d_q + 8 * chn;
  const uint16_t* wp = P.norm_w + 8 * chn;
  const float2* rope = reinterpret_cast<const float2*>(c.sm + SM_ROPE) + 32 * b;
  constexpr int na = d_q / 64;               // 64-dim atoms of q: 9, or 8
  constexpr int ra = na - 1;                 // the rotary atom
  uint4 raw[9];
#pragma unroll
  for (int a = 0; a < 9; ++a) raw[a] = (hv && a < na) ? ldg_nc(qh + 64 * a) : make_uint4(0, 0, 0, 0);
  // pass 1: sum of squares of q, largest |q * w| (and over the latent dims alone)
  float ss = 0.f, amax = 0.f, amax_lat = 0.f;
#pragma unroll
  for (int a = 0; a < 9; ++a) {
    const uint4 wq = a < na ? ldg_nc(wp + 64 * a) : make_uint4(0, 0, 0, 0);
    const uint32_t x4[4] = {raw[a].x, raw[a].y, raw[a].z, raw[a].w};
    const uint32_t w4[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float x0 = __uint_as_float(x4[e] << 16), x1 = __uint_as_float(x4[e] & 0xFFFF0000u);
      ss = fmaf(x0, x0, fmaf(x1, x1, ss));
      const float m = fmaxf(fabsf(x0 * __uint_as_float(w4[e] << 16)), fabsf(x1 * __uint_as_float(w4[e] & 0xFFFF0000u)));
      amax = fmaxf(amax, m);
      if (FP8Q && a < 8) amax_lat = fmaxf(amax_lat, m);
    }
  }
  ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 1);
  ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 2);
  ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 4);
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
  float rq = 0.f;   // fl(448 / amax_lat): the latent's quantisation factor (FP8Q)
  if constexpr (FP8Q) {
    amax_lat = fmaxf(amax_lat, __shfl_xor_sync(0xFFFFFFFFu, amax_lat, 1));
    amax_lat = fmaxf(amax_lat, __shfl_xor_sync(0xFFFFFFFFu, amax_lat, 2));
    amax_lat = fmaxf(amax_lat, __shfl_xor_sync(0xFFFFFFFFu, amax_lat, 4));
    rq = amax_lat > 0.f ? __fdiv_rn(448.0f, amax_lat) : 0.f;
  }
  const int ea = (int)((__float_as_uint(amax) >> 23) & 0xFF);   // floor(log2 amax) + 127 (normal amax)
  int k = ea == 0 ? 0 : 140 - ea;
  k = k < -100 ? -100 : (k > 100 ? 100 : k);
  const float sk = __uint_as_float((uint32_t)(127 + k) << 23);     // 2^k, exact
  // pass 2: the hi / lo operand rows (unrolled: raw[] stays in registers); with 512-dim
  // q the ninth atom stays unwritten (its QK^T partial is not run) but is announced all
  // the same, so that QRDY keeps one phase per item
#pragma unroll
  for (int a = 0; a < 9; ++a) {
    if (a >= na) {
      arrive_w(c, B_QRDY + 4);
      continue;
    }
    const uint4 wq = ldg_nc(wp + 64 * a);
    const uint32_t x4[4] = {raw[a].x, raw[a].y, raw[a].z, raw[a].w};
    const uint32_t w4[4] = {wq.x, wq.y, wq.z, wq.w};
    if (FP8Q && a < 8) {
      // E4M3 codes of the latent dims, as exact fp16 values in the hi rows only
      uint32_t hw[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float y0 = __fmul_rn(__uint_as_float(x4[e] << 16) * __uint_as_float(w4[e] << 16), rq);
        const float y1 = __fmul_rn(__uint_as_float(x4[e] & 0xFFFF0000u) * __uint_as_float(w4[e] & 0xFFFF0000u), rq);
        hw[e] = e4m3x2_to_f16x2(f32x2_to_e4m3x2(y0, y1));
      }
      const uint32_t atom = c.sb + SM_Q + (uint32_t)a * 8192 + ((uint32_t)chn ^ (uint32_t)(hs & 7)) * 16u;
      sts128(atom + (uint32_t)(hs >> 3) * 1024 + (uint32_t)(hs & 7) * 128, make_uint4(hw[0], hw[1], hw[2], hw[3]));
      if ((a & 1) == 1) {
        fence_async_smem();
        arrive_w(c, B_QRDY + (a >> 1));
      }
      continue;
    }
    float x[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[2 * e] = __uint_as_float(x4[e] << 16) * __uint_as_float(w4[e] << 16) * sk;
      x[2 * e + 1] = __uint_as_float(x4[e] & 0xFFFF0000u) * __uint_as_float(w4[e] & 0xFFFF0000u) * sk;
    }
    if (a == ra) {   // dims 512..575 (or 448..511): the rotary pairs 4 chn + e
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 cs = rope[4 * chn + e];
        const float x0 = x[2 * e], x1 = x[2 * e + 1];
        x[2 * e] = x0 * cs.x - x1 * cs.y;
        x[2 * e + 1] = x0 * cs.y + x1 * cs.x;
      }
    }
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) split_f16x2(x[2 * e], x[2 * e + 1], hw[e], lw[e]);
    const uint32_t atom = c.sb + SM_Q + (uint32_t)a * 8192 + ((uint32_t)chn ^ (uint32_t)(hs & 7)) * 16u;
    sts128(atom + (uint32_t)(hs >> 3) * 1024 + (uint32_t)(hs & 7) * 128, make_uint4(hw[0], hw[1], hw[2], hw[3]));
    sts128(atom + (uint32_t)((HH + hs) >> 3) * 1024 + (uint32_t)(hs & 7) * 128, make_uint4(lw[0], lw[1], lw[2], lw[3]));
    if ((a & 1) == 1 || a == 8) {
      // latent chunk a / 2 (atoms a - 1, a) or the rotary atom is complete
      fence_async_smem();
      arrive_w(c, B_QRDY + (a >> 1));
    }
  }
  float* s_inv = reinterpret_cast<float*>(c.sm + SM_INV) + 32 * b;
  if (chn == 0) s_inv[hs] = hv ? rsqrtf(ss * (1.0f / d_q) + P.eps) * P.c2 * __uint_as_float((uint32_t)(127 - k) << 23)
                               : 0.f;
  if (FP8Q && chn == 0) reinterpret_cast<float*>(c.sm + SM_RATIO)[32 * b + hs] = rq > 0.f ? __fdiv_rn(sk, rq) : 0.f;
  arrive_w(c, B_QSTAT + b);
}

// ================================================================== DQ
// Lane (sub, ch) of warp w converts 16 bytes (16 dims) of rows 16 w + 4 k + sub,
// k = 0..3, per 128-dim chunk: eight lanes read 128 contiguous bytes of a row.  The
// fp16 codes go straight into the 128-byte-swizzled tile (rows of 128 bytes holding 64
// dims); the four rows of one store instruction alternate in row parity, which keeps the
// stores free of bank conflicts.  Chunks are converted in the QK^T order (1, 0, 2, 3);
// raw bytes are loaded two chunks ahead of their conversion (position p of a tile lives
// in register slot p % 2).
// An entry for a row past the end of the item: no list entry has every bit set, since
// pools hold fewer than 2^31 rows.
constexpr uint32_t NO_ROW = 0xFFFFFFFFu;
struct DqRows {
  uint32_t e[4];   // list entries of rows 16 w + 4 k + sub, or NO_ROW
};

DSA_DEV void dq_load_rows(const uint32_t* list, int tt, int nrows, int w, int sub, DqRows& R) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int r = tt * TILE + 16 * w + 4 * k + sub;
    R.e[k] = r < nrows ? __ldcg(list + r) : NO_ROW;
  }
}

// The raw bytes of dims 128 cidx + 16 ch .. + 15 of rows R: 16 E4M3 codes of an fp8 row;
// of an fp4 row, 16 E2M1 values (x, y) and their E4M3 scale (z).
template <bool V41>
DSA_DEV void dq_load_chunk(const KParams& P, uint4 (&dst)[4], int cidx, const DqRows& R, int ch) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t e = R.e[k];
    if (e == NO_ROW) {
      dst[k] = make_uint4(0, 0, 0, 0);
    } else if (fp4_row<V41>(e)) {
      const uint8_t* rp = row_ptr<V41>(P, e);
      const uint2 v = ldg_nc_v2(rp + 64 * cidx + 8 * ch);
      dst[k] = make_uint4(v.x, v.y, ldg_nc_u8(rp + 256 + 8 * cidx + ch), 0);
    } else {
      dst[k] = ldg_nc(row_ptr<V41>(P, e) + 128 * cidx + 16 * ch);
    }
  }
}

// The rotary part of a tile's keys and the rows' block scales, written by the dequant
// warps one tile ahead of their use: warp w takes the tile rows 32 (w % 4) + lane (its
// TMEM lane quarter) and rope dims 32 (w / 4) .. + 31, bf16 -> fp16 into TMEM (the A
// operand of the rope partial, buffer gk % 2); the warps of the first half also store
// the rows' four block scales into shared memory (SCL buffer gk % 2) for the softmax
// warps.  Both are announced on KRFULL.
template <bool V41>
DSA_DEV void dq_rope(const KParams& P, const Ctx& c, uint32_t tmem, const uint32_t* list, int tt, int nrows, int w,
                     int lane, uint32_t gk) {
  const int q4 = w & 3, hh = w >> 2;
  const int r = 32 * q4 + lane;
  const bool valid = tt * TILE + r < nrows;
  const uint32_t e = valid ? __ldcg(list + tt * TILE + r) : NO_ROW;
  const uint32_t kb = gk & 1;
  // The scale table kb was last read by the softmax warps at the start of tile gk - 2.
  // These warps come here for tile gk only after converting every chunk of tile gk - 1,
  // and that waited for PV of tile gk - 2, which needs P of that tile from the softmax
  // warps, long after their read.  So the table is written without a wait (the rotary
  // keys' TMEM buffer, read by the tensor core, still waits for KRFREE below).
  float4* scl = reinterpret_cast<float4*>(c.sm + SM_SCL) + 128 * kb;
  if constexpr (V41) {   // no separate rotary keys: the four block scales only
    if (hh == 0) {
      const uint4 sv = valid ? row_scales<V41>(P, e) : make_uint4(0, 0, 0, 0);
      scl[r] = make_float4(__uint_as_float(sv.x), __uint_as_float(sv.y), __uint_as_float(sv.z), __uint_as_float(sv.w));
    }
    arrive_w(c, B_KRFULL + kb);
    return;
  }
  const uint8_t* src = valid ? row_ptr<V41>(P, e) + D_LAT : nullptr;
  uint4 raw[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) raw[k] = valid ? ldg_nc(src + 16 + 64 * hh + 16 * k) : make_uint4(0, 0, 0, 0);
  if (hh == 0) {
    const uint4 sv = valid ? ldg_nc(src) : make_uint4(0, 0, 0, 0);
    scl[r] = make_float4(__uint_as_float(sv.x), __uint_as_float(sv.y), __uint_as_float(sv.z), __uint_as_float(sv.w));
  }
  uint32_t v[16];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    v[4 * k + 0] = bf16x2_to_f16x2(raw[k].x);
    v[4 * k + 1] = bf16x2_to_f16x2(raw[k].y);
    v[4 * k + 2] = bf16x2_to_f16x2(raw[k].z);
    v[4 * k + 3] = bf16x2_to_f16x2(raw[k].w);
  }
  if (!wait_bar_w(c, B_KRFREE + kb, ((gk >> 1) & 1) ^ 1)) return;
  tc_fence_after();
  tmem_st16(tmem + ((uint32_t)(q4 * 32) << 16) + TM_KR + 32 * kb + 16 * hh, v);
  tc_wait_st();
  tc_fence_before();
  arrive_w(c, B_KRFULL + kb);
}

template <bool V41, bool FP8Q>
DSA_DEV void dq_role(const KParams& P, const Ctx& c, uint32_t tmem, int w, int lane) {
  const int sub = lane >> 3, ch = lane & 7;
  const uint32_t half_off = (uint32_t)(ch >> 2) * 16384;
  const uint32_t c0 = (uint32_t)(2 * (ch & 3));
  const uint32_t pa = c0 + (uint32_t)(ch >> 2), pb = c0 + 1 - (uint32_t)(ch >> 2);   // 16-byte chunks of the two stores
  uint4 raw[2][4];
  DqRows cur, nxt;
  uint32_t g = 0, seq = 0;
  // Without splits the dequant warps finish column blocks 1 (warps 0-3) and 2 (warps
  // 4-7) of each item's O^T, right after converting the next item's first tile: that
  // item's PV waits for O^T to be read, and the warps would wait for that PV anyway.
  // The item's buffers are released after its share.
  const bool share = P.n_splits == 1;
  int pend = -1;          // item (sequence number) whose share is still to do
  uint32_t pend_nq = 0;   // its index among the items with tiles
  uint32_t nq = 0;
  auto do_share = [&]() -> bool {
    const int pbf = pend % NB;
    if (!wait_bar_w(c, B_ODONE, pend_nq & 1)) return false;
    if (!wait_bar_w(c, B_LREADY, pend_nq & 1)) return false;
    tc_fence_after();
    const OutPtrs O = out_ptrs(P);
    const float2* rope = reinterpret_cast<const float2*>(c.sm + SM_ROPE) + 32 * pbf;
    const int* pinfo = item_info(c, pbf);
    const int cidx = 1 + (w >> 2);
    epi_chunk<8>(c, tmem, w & 3, lane, cidx, 0, HH / 8, reinterpret_cast<const float*>(c.sm + SM_EL),
                 item_ref(c, pbf)[cidx], O, pinfo[IT_TOKEN], HH * pinfo[IT_HALF], nullptr, rope);
    arrive_w(c, B_ITEMPTY + pbf);
    pend = -1;
    return true;
  };
  const QArgs qa{P.q, P.norm_w, P.h_q, P.rms_eps, P.score_scale_log2};
  // next item with tiles: its info waited for, its q~ built (once QK^T of the previous
  // item has completed), rows of tile 0 and its first two chunks in flight
  auto open_item = [&]() -> int {   // 1 = opened, 0 = no more items, -1 = aborted
    while (true) {
      const int b = seq % NB;
      if (!wait_bar_w(c, B_ITFULL + b, (seq / NB) & 1)) return -1;
      const int* info = item_info(c, b);
      if (info[IT_ITEM] < 0) return 0;
      if (info[IT_T] > 0) {
        if (nq > 0 && !wait_bar_w(c, B_QFREE, (nq - 1) & 1)) return -1;
        build_q<V41, FP8Q>(qa, c, b, 32 * w + lane);
        dq_rope<V41>(P, c, tmem, item_list(P, b) + info[IT_ROW0], 0, info[IT_NROWS], w, lane, g);
        dq_load_rows(item_list(P, b) + info[IT_ROW0], 0, info[IT_NROWS], w, sub, cur);
        dq_load_chunk<V41>(P, raw[0], qk_chunk(0), cur, ch);
        dq_load_chunk<V41>(P, raw[1], qk_chunk(1), cur, ch);
        return 1;
      }
      arrive_w(c, B_QSTAT + b);   // no q~: the phase still follows the buffer's uses
      arrive_w(c, B_ITEMPTY + b);
      ++seq;
    }
  };
  int r = open_item();
  while (r > 0) {
    const int b = seq % NB;
    const int* info = item_info(c, b);
    const int T = info[IT_T], nrows = info[IT_NROWS];
    const uint32_t* list = item_list(P, b) + info[IT_ROW0];
#pragma unroll 1
    for (int tt = 0; tt < T; ++tt) {
      const bool more = tt + 1 < T;
      // rows of the next tile (of this item, or tile 0 of the next item when its info is
      // already out), to be prefetched into L2 one tile ahead of their loads
      bool pf = more;
      if (more) {
        dq_load_rows(list, tt + 1, nrows, w, sub, nxt);
      } else {
        const int nb = (seq + 1) % NB;
        if (__all_sync(0xFFFFFFFFu, mbar_try(bar(c, B_ITFULL + nb), ((seq + 1) / NB) & 1))) {
          const int* ni = item_info(c, nb);
          if (ni[IT_ITEM] >= 0 && ni[IT_T] > 0) {
            dq_load_rows(item_list(P, nb) + ni[IT_ROW0], 0, ni[IT_NROWS], w, sub, nxt);
            pf = true;
          }
        }
      }
#pragma unroll
      for (int pos = 0; pos < 4; ++pos) {
        const int cidx = qk_chunk(pos);
        // the previous tile's PV has read this chunk (and the P block it held)
        if (!wait_bar_w(c, B_PVD + chunk_free_event(cidx), (g & 1) ^ 1)) return;
        const uint32_t cbase = c.sb + SM_V + (uint32_t)cidx * 32768 + half_off;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          // lanes of the second 64-dim atom (ch >= 4) store their upper eight dims first:
          // the eight lanes of a row then hit eight distinct 16-byte bank groups
          const uint4 rw = raw[pos & 1][k];
          uint32_t o[8];
          if (cur.e[k] != NO_ROW && fp4_row<V41>(cur.e[k])) {
            fp4x16_to_f16(ch >= 4 ? rw.y : rw.x, ch >= 4 ? rw.x : rw.y, rw.z, o);
          } else {
            codes16_to_f16(ch >= 4 ? make_uint4(rw.z, rw.w, rw.x, rw.y) : rw, o);
          }
          const uint32_t row = (uint32_t)(16 * w + 4 * k + sub);
          const uint32_t rsw = row & 7;
          const uint32_t rb = cbase + (row >> 3) * 1024 + rsw * 128;
          sts128(rb + ((pa ^ rsw) << 4), make_uint4(o[0], o[1], o[2], o[3]));
          sts128(rb + ((pb ^ rsw) << 4), make_uint4(o[4], o[5], o[6], o[7]));
        }
        fence_async_smem();
        arrive_w(c, B_VFULL + cidx);
        if (pos == 0 && pf) {
          // the 128-byte lines of each next row (at most six), one line per lane: lane ch
          // takes the line of byte min(128 ch, last byte), for the lines a row starting
          // anywhere on a 16-byte boundary can touch
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t e = nxt.e[k];
            if (e == NO_ROW) continue;
            const uint32_t rb = row_bytes<V41>(e);
            if ((uint32_t)ch < (rb + 112 + 127) / 128)
              prefetch_line_l2(row_ptr<V41>(P, e) + min(128u * (uint32_t)ch, rb - 1));
          }
        }
        // the chunk two positions ahead
        if (pos < 2) {
          dq_load_chunk<V41>(P, raw[pos & 1], qk_chunk(pos + 2), cur, ch);
        } else if (more) {
          dq_load_chunk<V41>(P, raw[pos & 1], qk_chunk(pos - 2), nxt, ch);
        }
      }
      if (more) cur = nxt;
      ++g;
      if (more) dq_rope<V41>(P, c, tmem, list, tt + 1, nrows, w, lane, g);
      if (tt == 0 && pend >= 0 && !do_share()) return;
    }
    if (share) {
      pend = (int)seq;
      pend_nq = nq;
    } else {
      arrive_w(c, B_ITEMPTY + b);
    }
    ++nq;
    ++seq;
    r = open_item();
  }
  if (r == 0 && pend >= 0) do_share();
}

// ================================================================== MMA issuer
// The whole warp runs this role and one elected lane issues each tensor-core
// instruction: with warp-uniform control flow the descriptor arithmetic stays in uniform
// registers.  (Issued from one lane of a divergent branch, every MMA paid conversions
// into uniform registers: 130-160 cycles per M = 128, N = 64, K = 16 MMA against the 48
// its operands take.)
DSA_DEV bool elect_one() {
  uint32_t e;
  asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(e));
  return e != 0;
}
DSA_DEV void issue_ss(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  if (elect_one()) mma_ss(d, adesc, bdesc, idesc, acc);
  __syncwarp();
}
DSA_DEV void issue_ts(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  if (elect_one()) mma_ts(d, a, bdesc, idesc, acc);
  __syncwarp();
}
DSA_DEV void commit(uint32_t bar_addr) {
  if (elect_one()) tc_commit(bar_addr);
  __syncwarp();
}

template <bool V41, bool FP8Q>
DSA_DEV void mma_role(const KParams& P, const Ctx& c, uint32_t tmem) {
  constexpr uint32_t IDESC_QK = idesc_f16(128, NQ, 0, 0);
  // the latent partials: N = 32 with an E4M3 q (its rows hold no lo part)
  constexpr uint32_t IDESC_QK_LAT = FP8Q ? idesc_f16(128, NQ / 2, 0, 0) : IDESC_QK;
  constexpr uint32_t IDESC_PV = idesc_f16(128, NQ, 1, 1);
  // every descriptor of the loop is one of these plus a constant offset (in 16-byte units
  // in the low 14-bit address field; no offset used here carries out of it)
  const uint64_t d_k = sdesc(c.sb + SM_V, 16, 1024);        // codes tile, K-major (QK^T)
  const uint64_t d_v = sdesc(c.sb + SM_V, 16384, 1024);     // codes tile, MN-major (PV)
  const uint64_t d_q = sdesc(c.sb + SM_Q, 16, 1024);        // q~ hi / lo
  uint32_t g = 0, nq = 0, np = 0;
  for (uint32_t seq = 0;; ++seq) {
    const int b = seq % NB;
    if (!wait_bar_w(c, B_ITFULL + b, (seq / NB) & 1)) return;
    const int* info = item_info(c, b);
    const int item = info[IT_ITEM];
    const int T = info[IT_T];
    if (elect_one()) mbar_arrive(bar(c, B_ITEMPTY + b));
    __syncwarp();
    if (item < 0) return;
    if (T == 0) continue;
    for (int tt = 0; tt < T; ++tt) {
      // ---- partial scores T_p = codes_p . q~_p^T, one per latent chunk, then the rope part
#pragma unroll 1
      for (int p = 0; p < 4; ++p) {
        const int cidx = qk_chunk(p);
        const uint32_t sbf = np % NSB;
        if (!wait_bar_w(c, B_SFREE + sbf, ((np / NSB) & 1) ^ 1)) return;
        if (tt == 0 && !wait_bar_w(c, B_QRDY + cidx, nq & 1)) return;
        if (!wait_bar_w(c, B_VFULL + cidx, g & 1)) return;
        tc_fence_after();
        const uint32_t d_s = tmem + TM_S + 64 * sbf;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t aoff = cidx * 32768 + (kk >> 2) * 16384 + (kk & 3) * 32;
          const uint32_t boff = (2 * cidx + (kk >> 2)) * 8192 + (kk & 3) * 32;
          issue_ss(d_s, d_k + (aoff >> 4), d_q + (boff >> 4), IDESC_QK_LAT, kk ? 1u : 0u);
        }
        commit(bar(c, B_SFULL + sbf));
        ++np;
      }
      if constexpr (!V41) {   // (nvfp4_ds_mla keys hold their rotary dims inside the latent chunks)
        const uint32_t sbf = np % NSB;
        const uint32_t kb = g & 1;
        if (!wait_bar_w(c, B_SFREE + sbf, ((np / NSB) & 1) ^ 1)) return;
        if (tt == 0 && !wait_bar_w(c, B_QRDY + 4, nq & 1)) return;
        if (!wait_bar_w(c, B_KRFULL + kb, (g >> 1) & 1)) return;
        tc_fence_after();
        const uint32_t d_s = tmem + TM_S + 64 * sbf;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          issue_ts(d_s, tmem + TM_KR + 32 * kb + 8 * kk, d_q + ((8 * 8192 + kk * 32) >> 4), IDESC_QK, kk ? 1u : 0u);
        commit(bar(c, B_SFULL + sbf));
        commit(bar(c, B_KRFREE + kb));
        ++np;
      }
      if (tt == T - 1) commit(bar(c, B_QFREE));   // q~ may be rebuilt after these MMAs
      // ---- O^T_b += codes_b^T . P_b, one block of output dims per latent block
#pragma unroll 1
      for (int pb = 0; pb < 4; ++pb) {
        if (!wait_bar_w(c, B_PFULL + pb, g & 1)) return;
        tc_fence_after();
        if (tt == 0 && nq > 0) {
          // the previous item's epilogue has read this part of O^T
          if (!wait_bar_w(c, B_OFREE + pb, (nq - 1) & 1)) return;
          tc_fence_after();
        }
        const uint64_t d_p = sdesc(c.sb + p_buffer(pb), 16384, 1024);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          issue_ss(tmem + TM_O + 64 * pb, d_v + ((pb * 32768 + kk * 2048) >> 4), d_p + ((kk * 2048) >> 4), IDESC_PV,
                   (tt > 0 || kk > 0) ? 1u : 0u);
        commit(bar(c, B_PVD + pb));
      }
      if (tt == T - 1) commit(bar(c, B_ODONE));
      ++g;
    }
    ++nq;
  }
}

// ================================================================== SX
// P_b = P * scale_b / reference_b of row r for the group's 16 heads, as hi / lo fp16 into
// the row of the MN-major B operand at `base` (16-byte chunks 2 gq, 2 gq + 1: hi of the
// group's heads; chunks 4 + 2 gq, 5 + 2 gq: their lo).
DSA_DEV void store_pb(uint32_t base, int r, int gq, const float (&p)[16], float f) {
  const uint32_t prow = base + (uint32_t)(r >> 3) * 1024 + (uint32_t)(r & 7) * 128;
  const uint32_t rsw = (uint32_t)(r & 7);
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) split_f16x2(p[8 * j + 2 * e] * f, p[8 * j + 2 * e + 1] * f, hw[e], lw[e]);
    const uint32_t q = (uint32_t)(2 * gq + j);
    sts128(prow + ((q ^ rsw) << 4), make_uint4(hw[0], hw[1], hw[2], hw[3]));
    sts128(prow + (((q + 4u) ^ rsw) << 4), make_uint4(lw[0], lw[1], lw[2], lw[3]));
  }
}

template <bool V41, bool FP8Q>
DSA_DEV void sx_role(const KParams& P, const Ctx& c, uint32_t tmem, int gq, int q4, int lane) {
  const int r = q4 * 32 + lane;
  const int hb = 16 * gq;                       // the group's first head within the item
  const uint32_t tlane = (uint32_t)(q4 * 32) << 16;
  float* s_m = reinterpret_cast<float*>(c.sm + SM_M);
  float* s_alpha = reinterpret_cast<float*>(c.sm + SM_ALPHA);
  float* s_red = reinterpret_cast<float*>(c.sm + SM_RED) + 64 * gq;     // 4 warps x 16
  float* s_flag = reinterpret_cast<float*>(c.sm + SM_FLAG) + 8 * gq;    // 2 x 4
  float* s_lw = reinterpret_cast<float*>(c.sm + SM_LW);                 // 2 x 8 warps x 16
  float* s_el = reinterpret_cast<float*>(c.sm + SM_EL);
  float* s_else = reinterpret_cast<float*>(c.sm + SM_ELSE);
  const float ln2 = 0.69314718055994531f;
  const bool is_split = P.n_splits > 1;
  Group grp{B_SXG + gq, 0};     // the four warps of this group
  Group all{B_SXA, 0};          // both groups
  uint32_t g = 0, seq = 0, nq = 0, np = 0;   // tiles, items, items with tiles, partial scores
  // A split of a (token, half) has stored its partial (or its LSE of -inf): it counts
  // in, and after the CTA's roles have finished every split combines one slice of it
  // (one item per CTA on this path).
  auto count_in = [&](int t, int split, int half) -> bool {
    __threadfence();
    if (!all.sync(c)) return false;
    if (gq == 0 && r == 0) {
      atomicAdd(&P.counters[(size_t)t * P.n_halves + half], 1u);
      c.misc[M_COMBINE] = 1;
      c.misc[M_TOKEN] = t;
      c.misc[M_SPLIT] = split;
      c.misc[M_HALF] = half;
    }
    return true;
  };
  // next item with tiles: its info waited for, the rope and scales of its tile 0 loaded
  auto open_item = [&]() -> int {
    while (true) {
      const int b = seq % NB;
      if (!wait_bar_w(c, B_ITFULL + b, (seq / NB) & 1)) return -1;
      const int* info = item_info(c, b);
      if (info[IT_ITEM] < 0) return 0;
      if (info[IT_T] > 0) return 1;
      if (is_split) {
        // a split without a valid column: LSE -inf, so the combine gives it no weight
        // (on the queue path such items never reach this role: the prep warp writes them)
        const int t = info[IT_TOKEN], half = info[IT_HALF], split = info[IT_SPLIT];
        if (r < 16) P.part_lse[((size_t)t * P.n_splits + split) * 64 + HH * half + hb + r] = -INFINITY;
        if (!count_in(t, split, half)) return -1;
      }
      arrive_w(c, B_ITEMPTY + b);
      ++seq;
    }
  };
  if (open_item() <= 0) return;
  while (true) {
    const int b = seq % NB;
    const int* info = item_info(c, b);
    const int T = info[IT_T], nrows = info[IT_NROWS];
    const int t = info[IT_TOKEN], half = info[IT_HALF], split = info[IT_SPLIT];
    const int h0 = HH * half;
    const uint32_t* list = item_list(P, b) + info[IT_ROW0];
    const float* iref = item_iref(c, b);
    // the next item's q into L2 when its info is already out
    if (gq == 0) {
      const int nb = (seq + 1) % NB;
      if (__all_sync(0xFFFFFFFFu, mbar_try(bar(c, B_ITFULL + nb), ((seq + 1) / NB) & 1))) {
        const int* ni = item_info(c, nb);
        if (ni[IT_ITEM] >= 0 && ni[IT_T] > 0) {
          const int nh0 = HH * ni[IT_HALF];
          const int nh = (P.h_q - nh0) < HH ? (P.h_q - nh0) : HH;
          const uint8_t* qn = reinterpret_cast<const uint8_t*>(P.q + ((size_t)ni[IT_TOKEN] * P.h_q + nh0) * Fmt<V41>::d_q);
          for (int l = r; l < nh * (Fmt<V41>::d_q / 64); l += 128) prefetch_line_l2(qn + 128 * l);
        }
      }
    }
    // the per-head factor of the scores (scale * log2(e) / (rms(q) 2^k)), written with q~
    // (one phase of QSTAT[b] per use of item buffer b: the next needs this buffer released)
    if (!wait_bar_w(c, B_QSTAT + b, (seq / NB) & 1)) return;
    const float* s_inv = reinterpret_cast<const float*>(c.sm + SM_INV) + 32 * b + hb;
    const float* s_ratio = reinterpret_cast<const float*>(c.sm + SM_RATIO) + 32 * b + hb;
    if (r < 16) s_m[hb + r] = -INFINITY;
    float lw = 0.f;   // this warp's row sum of head hb + lane / 2
    if (!grp.sync(c)) return;
#pragma unroll 1
    for (int tt = 0; tt < T; ++tt) {
      const bool valid = r < nrows - tt * TILE;
      // this row's four block scales (written with the tile's rotary keys)
      if (!wait_bar_w(c, B_KRFULL + (g & 1), (g >> 1) & 1)) return;
      const float4 s4 = reinterpret_cast<const float4*>(c.sm + SM_SCL)[128 * (g & 1) + r];
      const float sc[4] = {s4.x, s4.y, s4.z, s4.w};
      // ---- the five partial scores of row r, summed with the block scales
      float y[16];
#pragma unroll
      for (int h = 0; h < 16; ++h) y[h] = 0.f;
      constexpr int npart = V41 ? 4 : NPART;   // nvfp4_ds_mla: no rope partial
#pragma unroll 1
      for (int p = 0; p < npart; ++p) {
        const uint32_t sbf = np % NSB;
        if (!wait_bar_w(c, B_SFULL + sbf, (np / NSB) & 1)) return;
        tc_fence_after();
        const int pc = qk_chunk(p < 4 ? p : 0);
        const float f = p < 4 ? (pc == 0 ? sc[0] : pc == 1 ? sc[1] : pc == 2 ? sc[2] : sc[3]) : 1.0f;
        const uint32_t ts = tmem + tlane + TM_S + 64 * sbf + hb;
        uint32_t a[16], l[16];
        tmem_ld16(ts, a);
        if (!FP8Q || p == 4) tmem_ld16(ts + HH, l);   // (an E4M3 q's latent partials have no lo part)
        tc_wait_ld();
        tc_fence_before();
        arrive_w(c, B_SFREE + sbf);
        if (FP8Q && p < 4) {
#pragma unroll
          for (int i = 0; i < 16; ++i) y[i] = fmaf(f, __uint_as_float(a[i]), y[i]);
        } else if (FP8Q) {
          // the rope partial; the latent sum into the rope part's units first
#pragma unroll
          for (int i = 0; i < 16; ++i) y[i] = fmaf(y[i], s_ratio[i], __uint_as_float(a[i]) + __uint_as_float(l[i]));
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) y[i] = fmaf(f, __uint_as_float(a[i]) + __uint_as_float(l[i]), y[i]);
        }
        ++np;
      }
      // scores in log2 units (without the running max)
#pragma unroll
      for (int h = 0; h < 16; ++h) y[h] = valid ? y[h] * s_inv[h] : -INFINITY;
      bool need = tt == 0;
      if (!need) {
        // optimistic pass with the current reference max; the tile is redone below if it
        // exceeds the max by more than 2^8 somewhere
        float dmax = -INFINITY;
#pragma unroll
        for (int h = 0; h < 16; ++h) dmax = fmaxf(dmax, y[h] - s_m[hb + h]);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) dmax = fmaxf(dmax, __shfl_xor_sync(0xFFFFFFFFu, dmax, o));
        if (lane == 0) s_flag[4 * (g & 1) + q4] = dmax;
        if (!grp.sync(c)) return;
        const float* fl = s_flag + 4 * (g & 1);
        need = !(fmaxf(fmaxf(fl[0], fl[1]), fmaxf(fl[2], fl[3])) <= 8.0f);
      }
      if (need) {
        // exact tile max per head, new reference max, rescale factors
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = y[i];
        reduce16<true>(v, lane);          // lanes 2m, 2m + 1: head hb + m
        if ((lane & 1) == 0) s_red[q4 * 16 + (lane >> 1)] = v[0];
        if (!grp.sync(c)) return;
        if (r < 16) {
          const float tm = fmaxf(fmaxf(s_red[r], s_red[16 + r]), fmaxf(s_red[32 + r], s_red[48 + r]));
          const float mo = s_m[hb + r];
          const float mn = fmaxf(mo, tm);
          s_m[hb + r] = mn;
          s_alpha[hb + r] = (mn == -INFINITY) ? 1.f : exp2f(mo - mn);
        }
        if (!grp.sync(c)) return;
      }
      // ---- P = exp2(score - m) in fp32
#pragma unroll
      for (int h = 0; h < 16; ++h) y[h] = exp2f(y[h] - s_m[hb + h]);
      if (need && tt > 0) {
        // the group's columns of O^T rescaled once PV of the previous tile has completed
        if (!wait_bar_w(c, B_PVD + 3, (g & 1) ^ 1)) return;
        tc_fence_after();
#pragma unroll 1
        for (int j = 0; j < 8; ++j) {
          uint32_t a[16];
          const uint32_t ta = tmem + tlane + TM_O + 64 * (j >> 1) + HH * (j & 1) + hb;   // block j / 2, hi or lo
          tmem_ld16(ta, a);
          tc_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) a[i] = __float_as_uint(__uint_as_float(a[i]) * s_alpha[hb + i]);
          tmem_st16(ta, a);
        }
        tc_wait_st();
      }
      // ---- P_b hi / lo for the four PV blocks: P_0 in the shared buffer (last read by
      // PV(3) of the previous tile), P_1 .. P_3 once PV(0) of this tile has completed
      // (chunk 0 and the shared buffer).  The row sums go between P_0 and P_1.
#pragma unroll 1
      for (int pb = 0; pb < 4; ++pb) {
        if (pb < 2 && !wait_bar_w(c, B_PVD + (pb == 0 ? 3 : 0), pb == 0 ? ((g & 1) ^ 1) : (g & 1))) return;
        const float f = (pb == 0 ? sc[0] : pb == 1 ? sc[1] : pb == 2 ? sc[2] : sc[3]) * iref[pb];
        store_pb(c.sb + p_buffer(pb), r, gq, y, valid ? f : 0.f);
        fence_async_smem();
        tc_fence_before();
        arrive_w(c, B_PFULL + pb);
        if (pb == 0) {
          // this warp's row sums (lanes 2m, 2m + 1: head hb + m)
          float v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = valid ? y[i] : 0.f;
          reduce16<false>(v, lane);
          lw = fmaf(lw, (need && tt > 0) ? s_alpha[hb + (lane >> 1)] : 1.f, v[0]);
        }
      }
      ++g;
      if (tt + 1 < T) continue;
      // ---- the item's last tile: 1/l, LSE and the epilogue of this group's heads
      if ((lane & 1) == 0) s_lw[(nq & 1) * 128 + (4 * gq + q4) * 16 + (lane >> 1)] = lw;
      if (!grp.sync(c)) return;
      if (!wait_bar_w(c, B_ODONE, nq & 1)) return;
      tc_fence_after();
      if (r < 16) {
        const float* lwb = s_lw + (nq & 1) * 128 + 64 * gq + r;
        const float l = (lwb[0] + lwb[16]) + (lwb[32] + lwb[48]);
        const bool any = l > 0.f;
        s_else[hb + r] = any ? s_m[hb + r] + log2f(l) : -INFINITY;
        s_el[hb + r] = any ? 1.f / l : 0.f;
      }
      if (!grp.sync(c)) return;
      if (r < 16 && h0 + hb + r < P.h_q) {
        if (is_split) P.part_lse[((size_t)t * P.n_splits + split) * 64 + h0 + hb + r] = s_else[hb + r];
        else if (P.out_lse) P.out_lse[(size_t)t * P.h_q + h0 + hb + r] = s_else[hb + r] * ln2;
      }
      // without splits column blocks 1 and 2 are finished by the dequant warps once 1/l
      // is out
      if (!is_split) arrive_w(c, B_LREADY);
      const OutPtrs O = out_ptrs(P);
      const float2* rope = reinterpret_cast<const float2*>(c.sm + SM_ROPE) + 32 * b;
      float* part = is_split ? P.part_o + (((size_t)t * P.n_splits + split) * 64 + h0) * D_LAT : nullptr;
      const float* ref = item_ref(c, b);
      const int nblk = is_split ? 4 : 2;
#pragma unroll 1
      for (int bi = 0; bi < nblk; ++bi) {
        const int cidx = is_split ? bi : 3 * bi;
        epi_chunk<16>(c, tmem, q4, lane, cidx, hb, 1, s_el, ref[cidx], O, t, h0, part, rope);
      }
      if (is_split && !count_in(t, split, half)) return;
    }
    arrive_w(c, B_ITEMPTY + b);
    ++seq;
    ++nq;
    if (open_item() <= 0) return;
  }
}

// Combine of one (token, half)'s split partials: split `part` takes the slice
// part / n_splits of its (head, 32-dim block) units, four threads per unit (eight dims
// each); weights exp2(lse_s - M) / sum over splits.  The token's rotary table is already
// in s_rope (written while the splits were still arriving).
DSA_DEV void combine_token(const KParams& P, const Ctx& c, int t, int half, int part, int tid) {
  float* s_cw = reinterpret_cast<float*>(c.sm + SM_CW);       // [MAX_SPLITS][32]
  float* s_lse = s_cw + MAX_SPLITS * HH;                       // [32]
  const float2* s_rope = reinterpret_cast<const float2*>(s_lse + HH);   // [32] (cos, sin)
  const int ns = P.n_splits;
  const int h0 = HH * half;
  const float ln2 = 0.69314718055994531f;
  if (tid < HH) {
    const float* pl = P.part_lse + (size_t)t * ns * 64 + h0 + tid;
    float lv[MAX_SPLITS];
#pragma unroll
    for (int s = 0; s < MAX_SPLITS; ++s) lv[s] = s < ns ? __ldcg(pl + s * 64) : -INFINITY;
    float M = -INFINITY;
#pragma unroll
    for (int s = 0; s < MAX_SPLITS; ++s) M = fmaxf(M, lv[s]);
    float den = 0.f;
#pragma unroll
    for (int s = 0; s < MAX_SPLITS; ++s) {
      lv[s] = (M == -INFINITY || s >= ns) ? 0.f : exp2f(lv[s] - M);
      den += lv[s];
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
    for (int s = 0; s < MAX_SPLITS; ++s)
      if (s < ns) s_cw[s * HH + tid] = lv[s] * inv;
    s_lse[tid] = den > 0.f ? (M + log2f(den)) * ln2 : -INFINITY;
  }
  __syncthreads();
  if (part == 0 && P.out_lse && tid < HH && h0 + tid < P.h_q) P.out_lse[(size_t)t * P.h_q + h0 + tid] = s_lse[tid];
  const int nh = (P.h_q - h0) < HH ? (P.h_q - h0) : HH;
  const int u0 = part * nh * 16 / ns, u1 = (part + 1) * nh * 16 / ns;
  const int q = tid & 3;                                         // this thread's eight dims of the unit
  const unsigned gmask = 0xFu << (tid & 28);                     // the unit's four lanes
  for (int u = u0 + (tid >> 2); u < u1; u += NTHREADS / 4) {
    const int hh = u >> 4, blk = u & 15;
    float v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = 0.f;
    const float* base = P.part_o + ((size_t)t * ns * 64 + h0 + hh) * D_LAT + 32 * blk + 8 * q;
    // four splits' loads in flight at a time
#pragma unroll 1
    for (int s0 = 0; s0 < ns; s0 += 4) {
      float w[4];
      float4 f[4][2];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int sp = s0 + j;
        w[j] = sp < ns ? s_cw[sp * HH + hh] : 0.f;
        const float4* src = reinterpret_cast<const float4*>(base + (size_t)sp * 64 * D_LAT);
        f[j][0] = w[j] != 0.f ? __ldcg(src) : make_float4(0.f, 0.f, 0.f, 0.f);
        f[j][1] = w[j] != 0.f ? __ldcg(src + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[0] = fmaf(w[j], f[j][0].x, v[0]);
        v[1] = fmaf(w[j], f[j][0].y, v[1]);
        v[2] = fmaf(w[j], f[j][0].z, v[2]);
        v[3] = fmaf(w[j], f[j][0].w, v[3]);
        v[4] = fmaf(w[j], f[j][1].x, v[4]);
        v[5] = fmaf(w[j], f[j][1].y, v[5]);
        v[6] = fmaf(w[j], f[j][1].z, v[6]);
        v[7] = fmaf(w[j], f[j][1].w, v[7]);
      }
    }
    finalize_eighth(out_ptrs(P), v, t, h0 + hh, 32 * blk + 8 * q, gmask, s_rope);
  }
}

// ================================================================== the kernel
// Queue path, before the fused kernel: clears the workspace header (status word, queue
// head) and writes the order in which the queue hands out tokens, those with the most
// 128-row tiles first.  With items of mixed length taken from one queue, the CTAs that
// draw long items last finish late; longest-first leaves only short items for the end.
// The tile count comes from topk_length alone (sentinels are not counted).  A stable
// counting sort over the 17 possible tile counts: tokens of equal count keep their
// order.  Each warp counts equal keys with one match, so a batch of equal lengths costs
// one shared-memory atomic per warp.  The fused kernel is launched as this grid's
// programmatic dependent: it may start its prologue at once, and it waits for this
// grid's writes before it takes an item.
constexpr int ORDER_THREADS = 1024;
constexpr int ORDER_MAX_TOKENS = 65536;   // beyond this the queue takes tokens in order
__global__ void __launch_bounds__(ORDER_THREADS, 1) dsa_order_kernel(const int32_t* __restrict__ topk_length,
                                                                     int s_q, int topk, uint32_t* header,
                                                                     int32_t* order) {
  constexpr int NK = DSA_MAX_TOPK / TILE + 1, NW = ORDER_THREADS / 32;
  __shared__ int s_next[NK];      // first free slot of each tile count
  __shared__ int s_cnt[NW][NK];   // per warp: tokens of each count in the current chunk
  __shared__ int s_off[NW][NK];   // per warp: where those tokens go
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // launched as a producer's programmatic dependent (DSA_FLAG_AFTER_PRODUCER): nothing is
  // read before that kernel has completed; a no-op otherwise
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const unsigned lt = (1u << lane) - 1u;
  auto key = [&](int t) {
    if (t >= s_q) return -1;
    const int len = min(max(topk_length[t], 0), topk);
    return (len + TILE - 1) / TILE;
  };
  if (tid < NK) s_next[tid] = 0;
  for (int i = tid; i < NW * NK; i += ORDER_THREADS) (&s_cnt[0][0])[i] = 0;
  if (tid < 64) header[tid] = 0;   // the 256-byte header: status word, queue head
  __syncthreads();
  for (int c0 = 0; c0 < s_q; c0 += ORDER_THREADS) {
    const int k = key(c0 + tid);
    const unsigned same = __match_any_sync(0xFFFFFFFFu, k);
    if (k >= 0 && (same & lt) == 0) atomicAdd(&s_next[k], __popc(same));
  }
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int k = NK - 1; k >= 0; --k) {
      const int n = s_next[k];
      s_next[k] = run;
      run += n;
    }
  }
  __syncthreads();
  for (int c0 = 0; c0 < s_q; c0 += ORDER_THREADS) {
    const int t = c0 + tid, k = key(t);
    const unsigned same = __match_any_sync(0xFFFFFFFFu, k);
    if (k >= 0 && (same & lt) == 0) s_cnt[w][k] = __popc(same);
    __syncthreads();
    if (tid < NK) {   // one thread per count: the warps' slots in warp order
      int run = s_next[tid];
      for (int j = 0; j < NW; ++j) {
        s_off[j][tid] = run;
        run += s_cnt[j][tid];
        s_cnt[j][tid] = 0;
      }
      s_next[tid] = run;
    }
    __syncthreads();
    if (k >= 0) order[s_off[w][k] + __popc(same & lt)] = t;
  }
}

template <bool V41, bool FP8Q>
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
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar(c, B_VFULL + i), WG_DQ);
      mbar_init(bar(c, B_PVD + i), 1);
      mbar_init(bar(c, B_PFULL + i), WG_SX);
      // O^T blocks 1 and 2 are read by four dequant warps each, blocks 0 and 3 (all four
      // on the split path) by the eight softmax warps (counts in warps)
      mbar_init(bar(c, B_OFREE + i), (P.n_splits == 1 && (i == 1 || i == 2)) ? 4 : WG_SX);
    }
    for (int i = 0; i < NSB; ++i) {
      mbar_init(bar(c, B_SFULL + i), 1);
      mbar_init(bar(c, B_SFREE + i), WG_SX);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(c, B_KRFULL + i), WG_DQ);
      mbar_init(bar(c, B_KRFREE + i), 1);
    }
    for (int i = 0; i < NB; ++i) {
      mbar_init(bar(c, B_ITFULL + i), 1);
      mbar_init(bar(c, B_ITEMPTY + i), WG_DQ + WG_SX + 1);
      mbar_init(bar(c, B_QSTAT + i), WG_DQ);
    }
    mbar_init(bar(c, B_ODONE), 1);
    for (int i = 0; i < 5; ++i) mbar_init(bar(c, B_QRDY + i), WG_DQ);
    mbar_init(bar(c, B_QFREE), 1);
    mbar_init(bar(c, B_LREADY), WG_SX);
    mbar_init(bar(c, B_SXG), 4);
    mbar_init(bar(c, B_SXG + 1), 4);
    mbar_init(bar(c, B_SXA), WG_SX);
    mbar_init(bar(c, B_DRAIN), 1);
    mbar_init(bar(c, B_NEVER), 1);   // nothing arrives: the failure-path test waits on it
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    c.misc[M_ABORT] = 0;
    c.misc[M_COMBINE] = 0;
  }
  if (warp == W_MMA) tmem_alloc(c.sb + SM_MISC + 4 * M_TMEM, TM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = (uint32_t)c.misc[M_TMEM];
  // launched as the order kernel's programmatic dependent (queue path): its header and
  // order are visible after this; a no-op for a launch without that dependency
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp < W_SX) {
    dq_role<V41, FP8Q>(P, c, tmem, warp, lane);
  } else if (warp < W_MMA) {
    sx_role<V41, FP8Q>(P, c, tmem, (warp - W_SX) >> 2, warp & 3, lane);
  } else if (warp == W_MMA) {
    mma_role<V41, FP8Q>(P, c, tmem);
  } else if (warp == W_PREP) {
    prep_role<V41>(P, c, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == W_MMA && lane == 0) {
    // every MMA this CTA issued has completed before TMEM is released
    tc_commit(bar(c, B_DRAIN));
    const unsigned long long start = clock64();
    while (!mbar_wait_susp(bar(c, B_DRAIN), 0) && clock64() - start < WAIT_LIMIT_CYCLES) {
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == W_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
  if (P.n_splits > 1 && c.misc[M_COMBINE] && !c.misc[M_ABORT]) {
    // every split of the (token, half) has stored its partial (the splits are
    // co-resident: this path is a cooperative launch); bounded wait on the arrival count
    const int t = c.misc[M_TOKEN], half = c.misc[M_HALF];
    if (tid >= 32 && tid < 64) {
      // the token's rotary table for the combine (the item buffers are gone), while the
      // other splits are still arriving
      float2* s_rope = reinterpret_cast<float2*>(c.sm + SM_CW) + (MAX_SPLITS * HH + HH) / 2;
      s_rope[tid - 32] = rope_entry_of(P, t, tid - 32);
    }
    if (tid == 0) {
      const volatile uint32_t* cnt = P.counters + (size_t)t * P.n_halves + half;
      const unsigned long long start = clock64();
      while (*cnt < (uint32_t)P.n_splits) {
        __nanosleep(64);
        if (clock64() - start > WAIT_LIMIT_CYCLES) {
          atomicOr(c.status, DSA_STATUS_WAIT_TIMEOUT);
          c.misc[M_ABORT] = 1;
          break;
        }
      }
      __threadfence();
    }
    __syncthreads();
    if (!c.misc[M_ABORT]) combine_token(P, c, t, half, c.misc[M_SPLIT], tid);
  }
}

// ================================================================== host side
struct Layout {
  size_t status_off, work_off, counters_off, lists_off, part_o_off, part_lse_off, total;
};

static int halves_for(int h_q) { return h_q > HH ? 2 : 1; }

static int pick_splits(int s_q, int h_q, int topk, int num_sms) {
  if (s_q <= 0) return 1;
  const int tiles = (topk + TILE - 1) / TILE;
  const long long base = (long long)s_q * halves_for(h_q);
  if (tiles <= 1 || base >= num_sms) return 1;
  int sp = (int)(num_sms / base);
  if (sp > tiles) sp = tiles;
  if (sp > MAX_SPLITS) sp = MAX_SPLITS;
  return sp < 1 ? 1 : sp;
}

static Layout layout_for(int s_q, int h_q, int n_splits, int num_sms) {
  Layout L;
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  L.status_off = 0;
  L.work_off = 4;
  L.counters_off = 256;
  // one int32 per (token, half): the split path's arrival counters, or the queue's order
  size_t off = up(L.counters_off + 4 * (size_t)(s_q > 0 ? s_q : 1) * halves_for(h_q));
  L.lists_off = off;
  off = up(off + (size_t)num_sms * NB * DSA_MAX_TOPK * 4);
  if (n_splits > 1) {
    L.part_o_off = off;
    off = up(off + (size_t)s_q * n_splits * 64 * D_LAT * 4);
    L.part_lse_off = off;
    off = up(off + (size_t)s_q * n_splits * 64 * 4);
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
  if (p->kv_format != DSA_KV_FP8_DS_MLA && p->kv_format != DSA_KV_NVFP4_DS_MLA) return DSA_ERR_INVALID_ARG;
  if ((p->flags & DSA_FLAG_FP8_Q) && p->kv_format != DSA_KV_FP8_DS_MLA) return DSA_ERR_INVALID_ARG;
  if (!(p->cmp_scale == p->cmp_scale) || p->cmp_scale == INFINITY || p->cmp_scale == -INFINITY)
    return DSA_ERR_INVALID_ARG;
  if (p->flags & ~(DSA_FLAG_CHECK_INDICES | DSA_FLAG_TEST_WAIT_TIMEOUT | DSA_FLAG_AFTER_PRODUCER | DSA_FLAG_SF_SWIZZLED |
                   DSA_FLAG_FP8_Q))
    return DSA_ERR_INVALID_ARG;
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

// The fused kernel's dynamic shared-memory limit, raised once per device (any host
// thread may make the first call).
static std::mutex g_attr_mutex;
static bool g_attr_done[DSA_MAX_DEVICES];

static int ensure_smem_attr(int dev) {
  if (dev < 0 || dev >= DSA_MAX_DEVICES) return DSA_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_attr_mutex);
  if (!g_attr_done[dev]) {
    if (cudaFuncSetAttribute(dsa_fwd_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES) != cudaSuccess ||
        cudaFuncSetAttribute(dsa_fwd_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES) != cudaSuccess ||
        cudaFuncSetAttribute(dsa_fwd_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES) != cudaSuccess)
      return DSA_ERR_CUDA;
    g_attr_done[dev] = true;
  }
  return DSA_OK;
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
      !aligned(out_fp8, 16) || !aligned(indices, 4) || !aligned(workspace, 256) || !aligned(norm_w, 16) ||
      (out_precast && !aligned(out_precast, 16)) || (lse && !aligned(lse, 4)))
    return DSA_ERR_INVALID_ARG;
  int dev = 0;
  const int sms = device_sms(&dev);
  if (sms <= 0) return DSA_ERR_CUDA;
  if (dev >= DSA_MAX_DEVICES) return DSA_ERR_UNSUPPORTED_DEVICE;
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) return DSA_ERR_UNSUPPORTED_DEVICE;
  const int nh = halves_for(p->h_q);
  const int ns = pick_splits(p->s_q, p->h_q, p->topk, sms);
  const Layout L = layout_for(p->s_q, p->h_q, ns, sms);
  if (workspace_bytes < L.total) return DSA_ERR_WORKSPACE_TOO_SMALL;
  rc = ensure_smem_attr(dev);
  if (rc != DSA_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t* ws = (uint8_t*)workspace;
  const bool ordered = ns == 1 && p->s_q <= ORDER_MAX_TOKENS;
  if (ordered) {
    // header and the queue's order (in the counters' region, which the queue path does not use)
    cudaLaunchConfig_t ocfg = {};
    ocfg.gridDim = dim3(1);
    ocfg.blockDim = dim3(ORDER_THREADS);
    ocfg.stream = st;
    cudaLaunchAttribute oattr[1];
    oattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    oattr[0].val.programmaticStreamSerializationAllowed = 1;
    ocfg.attrs = oattr;
    ocfg.numAttrs = (p->flags & DSA_FLAG_AFTER_PRODUCER) ? 1 : 0;
    if (cudaLaunchKernelEx(&ocfg, dsa_order_kernel, topk_length, p->s_q, p->topk, (uint32_t*)ws,
                           (int32_t*)(ws + L.counters_off)) != cudaSuccess)
      return DSA_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return DSA_ERR_CUDA;
  } else {
    // header and the split arrival counters
    const size_t n = ns > 1 ? L.counters_off + 4 * (size_t)p->s_q * nh : L.counters_off;
    if (cudaMemsetAsync(ws, 0, n, st) != cudaSuccess) return DSA_ERR_CUDA;
  }

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
  K.order = ordered ? (const int32_t*)(ws + L.counters_off) : nullptr;
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
  K.cmp_scale = p->cmp_scale;
  K.n_splits = ns;
  K.n_halves = nh;
  K.n_items = p->s_q * nh * ns;
  rope_turn_table(p->rope_base, K.rope_turns);
  const int grid = K.n_items < sms ? K.n_items : sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = st;
  // the split path waits across CTAs for the combine: a cooperative launch keeps its
  // CTAs (one per item, at most one per SM) co-resident.  The ordered queue path starts
  // while the order kernel runs, as its programmatic dependent.
  cudaLaunchAttribute attr[1];
  if (ns > 1) {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  } else {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = (ns > 1 || ordered) ? 1 : 0;
  // one instantiation per cache format, and the fp8_ds_mla one also with an E4M3 q
  void (*kernel)(KParams) = p->kv_format == DSA_KV_NVFP4_DS_MLA ? dsa_fwd_kernel<true, false>
                            : (p->flags & DSA_FLAG_FP8_Q)       ? dsa_fwd_kernel<false, true>
                                                                : dsa_fwd_kernel<false, false>;
  if (cudaLaunchKernelEx(&cfg, kernel, K) != cudaSuccess) return DSA_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return DSA_ERR_CUDA;
  return DSA_OK;
}

// ------------------------------------------------------- allocation-free entry
// Scratch of dsa_sparse_attn_fwd_noalloc, in place of a caller-supplied workspace.
// It is zero-initialised device memory reserved when the module loads; its address is
// looked up once per device and cached.
static __device__ __align__(256) unsigned char g_noalloc_scratch[DSA_NOALLOC_SCRATCH_BYTES];
static std::mutex g_noalloc_mutex;
static void* g_noalloc_ptr[DSA_MAX_DEVICES];

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
  if (dev < 0 || dev >= DSA_MAX_DEVICES) return DSA_ERR_UNSUPPORTED_DEVICE;
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) return DSA_ERR_UNSUPPORTED_DEVICE;
  const Layout L = layout_for(p->s_q, p->h_q, pick_splits(p->s_q, p->h_q, p->topk, sms), sms);
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
  p->kv_format = DSA_KV_FP8_DS_MLA;
  p->cmp_scale = 1.0f;
  return DSA_OK;
}

int dsa_sparse_attn_num_splits(const dsa_params* p, int num_sms) {
  if (dsa::check_params(p) != DSA_OK) return 0;
  if (num_sms <= 0) num_sms = dsa::device_sms(nullptr);
  if (num_sms <= 0) return 0;
  return dsa::pick_splits(p->s_q, p->h_q, p->topk, num_sms);
}

size_t dsa_sparse_attn_workspace_size(const dsa_params* p, int num_sms) {
  const int ns = dsa_sparse_attn_num_splits(p, num_sms);
  if (ns <= 0) return 0;
  if (num_sms <= 0) num_sms = dsa::device_sms(nullptr);
  if (num_sms <= 0) return 0;
  return dsa::layout_for(p->s_q, p->h_q, ns, num_sms).total;
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
    case DSA_ERR_UNSUPPORTED_DEVICE:
      return "current device is not compute capability 10.3 (GB300), or its ordinal is >= DSA_MAX_DEVICES";
    case DSA_ERR_SCRATCH_LIMIT:
      return "shape needs more scratch than the no-alloc entry's built-in DSA_NOALLOC_SCRATCH_BYTES";
    default: return "unknown error";
  }
}

}  // extern "C"
