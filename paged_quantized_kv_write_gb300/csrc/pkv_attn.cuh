// The attention kernel shared by paged_decode_attention and
// paged_prefill_attention: PagedAttention over a paged, optionally quantized
// KV cache.
//
// What it computes (softmax(q K^T / sqrt(d)) V per query head, GQA groups
// sharing one KV head: "KV Cache Optimization: 3x Faster LLM Inference",
// GQA section; the per-head walk over logical blocks -> physical blocks ->
// K, V -> scores -> softmax -> weighted sum: "KV Cache Compression & Paged
// Attention", Implementation Details):
//   out[b,h] = sum_t exp(s_t - max) V_t / sum_t exp(s_t - max),
//   s_t = softmax_scale * q[b,h] . K_t, t < context_lens[b] (decode) or
//   t <= the query's position (prefill, causal),
//   K_t, V_t read at block_tables[b][t / bs], offset t % bs, dequantized.
//
// Design (GB300, sm_103a):
//  * A warp owns up to 8 score columns: the G query heads of one KV head
//    (decode) or 8/G query tokens times those G heads (prefill).  They are
//    the N=8 columns of an mma.sync.m16n8k16: S^T[t, c] = K_tile(16 x D) .
//    Q^T(D x 8) and O^T[d, c] += V_tile^T(D x 16) . P^T(16 x 8), fp32
//    accumulate.  Each K/V element is read once from shared memory, converted
//    in registers and used for all 8 columns.
//  * Each warp stages its tiles in a private shared-memory ring with 16-byte
//    cp.async copies (K rows, V rows, INT4 scale rows, block scales), a few
//    tiles ahead, so several KB per warp are in flight from HBM.  The 16-byte
//    chunks are XOR-swizzled per row so the fragment reads hit all 32 banks.
//  * FP8 codes become exact f16 (cvt.rn.f16x2.e4m3x2 / e5m2x2); INT8 and INT4
//    codes become f16 subnormals ((x + 128) 2^-24, n 2^-24) whose offset and
//    2^24 are taken off after the sums; scales are applied outside the
//    products (block scales per tile; INT4: per token and group, with the
//    zero points through one more product on each side).
//  * The probabilities P enter the second product as a hi + lo pair of 16-bit
//    values (P = hi + lo to ~2^-17 relative), so rounding P to 16 bits costs
//    no accuracy (INT4: P' = p * scale formed exactly as an f16 hi + lo pair).
//  * Decode splits long contexts into partitions: each writes (max, sum,
//    O/sum) per head to a workspace that pkv_lse_reduce merges.  A CTA's 4
//    warps either share a partition's tiles (merging in shared memory) or
//    each own (partition, KV head) units.
#pragma once

#include <limits.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>

#include "pkv_common.cuh"
#include "pkv_encode.cuh"
#include "pkv_internal.h"
#include "pkv_tcgen05.cuh"

namespace pkv {
namespace {

// ring depth (tiles in flight per warp, plus the one being computed); build-time knobs
#ifndef PKV_STAGES_HALF
#define PKV_STAGES_HALF 2
#endif
#ifndef PKV_STAGES_FP8
#define PKV_STAGES_FP8 2
#endif
#ifndef PKV_STAGES_INT4
#define PKV_STAGES_INT4 2
#endif
// CTAs per SM the register allocation must allow (__launch_bounds__ minimum)
#ifndef PKV_MINB_HALF
#define PKV_MINB_HALF 3
#endif
#ifndef PKV_MINB_QUANT
#define PKV_MINB_QUANT 3
#endif
#ifndef PKV_MINB_INT4
#define PKV_MINB_INT4 PKV_MINB_QUANT
#endif

#ifndef PKV_DECODE_WARPS
#define PKV_DECODE_WARPS 4
#endif
constexpr int kDecodeWarps = PKV_DECODE_WARPS;   // warps per CTA (each walks its own tiles)
constexpr int kTile = 16;            // tokens per tile (the mma M / K extent)
constexpr int kMaxDevices = 64;
// partitions per CTA (0: choose), and the longest run of tokens one CTA takes
#ifndef PKV_PPC
#define PKV_PPC 0
#endif
#ifndef PKV_RUN_TOKENS
#define PKV_RUN_TOKENS 2048
#endif
#ifndef PKV_RUN_TOKENS_WU
#define PKV_RUN_TOKENS_WU 512
#endif
// warp-owned units from this many waves of warp-units (large: never)
#ifndef PKV_WU_WAVES
#define PKV_WU_WAVES 3
#endif
// 16-token sub-tiles per ring stage (one softmax step covers them all)
#ifndef PKV_SUB_HALF
#define PKV_SUB_HALF 1
#endif
#ifndef PKV_SUB_QUANT
#define PKV_SUB_QUANT 2
#endif
#ifndef PKV_SUB_INT4
#define PKV_SUB_INT4 PKV_SUB_QUANT
#endif
constexpr float kLog2e = 1.4426950408889634f;

template <int KV, int D> struct Geo {
  static constexpr bool kHalf = (KV == PKV_F16 || KV == PKV_BF16);
  static constexpr int kRowBytes = kHalf ? 2 * D : (is_blk8(KV) ? D : D / 2);
  static constexpr int kCpr = kRowBytes / 16;                   // 16-byte chunks per row
  static constexpr int kTileBytes = kTile * kRowBytes;          // one of K or V
  static constexpr int kScaleRowBytes = (KV == PKV_INT4_G32) ? (D / 32) * 4 : 0;
  static constexpr int kScaleTileBytes = kTile * kScaleRowBytes;
  // A stage holds kSub 16-token sub-tiles, each K rows | V rows | K scale rows |
  // V scale rows, then 16 B of misc per sub-tile (FP8 K and V scale, valid flag).
  static constexpr int kSub = kHalf ? PKV_SUB_HALF : (KV == PKV_INT4_G32 ? PKV_SUB_INT4 : PKV_SUB_QUANT);
  static constexpr int kTileTok = kTile * kSub;                 // tokens per stage
  static constexpr int kSubBytes = 2 * kTileBytes + 2 * kScaleTileBytes;
  static constexpr int kMiscOffset = kSub * kSubBytes;
  static constexpr int kStageBytes = kSub * kSubBytes + 16 * kSub;
  static constexpr int kStages =
      kHalf ? PKV_STAGES_HALF : (is_blk8(KV) ? PKV_STAGES_FP8 : PKV_STAGES_INT4);
  static constexpr int kWarpRing = kStages * kStageBytes;
  static constexpr int kRingBytes = kDecodeWarps * kWarpRing;
  // merge buffer: one warp's state, lane-major with an odd stride (no bank conflicts)
  static constexpr int kMbStride = (D / 16) * 4 + 5;
  static constexpr int kMbufBytes = kWarp * kMbStride * 4;
  static constexpr int kSmemBytes = kRingBytes + kMbufBytes;
  static constexpr int kMinBlocks =
      kHalf ? PKV_MINB_HALF : (KV == PKV_INT4_G32 ? PKV_MINB_INT4 : PKV_MINB_QUANT);
};

// 2^x on the SFU (ex2.approx; 2^-inf = +0).  Scores and probabilities use it
// consistently, so the softmax stays exact up to its ~2 ulp.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// XOR swizzle of the 16-byte chunk position within a row (see the bank
// analysis in the fragment readers below).
template <int KV, int D>
__device__ __forceinline__ int swz(int r) {
  if constexpr (KV == PKV_F16 || KV == PKV_BF16 || (is_blk8(KV) && D == 128)) {
    return (((r ^ (r >> 1)) & 1) << 2) | ((r >> 2) & 1);
  } else if constexpr (KV == PKV_INT4_G32) {
    return D == 128 ? ((r >> 1) & 3) : ((r >> 2) & 1);
  } else {
    return 0;
  }
}

template <int KV, int D>
__device__ __forceinline__ uint32_t chunk_off(int row, int ch) {
  using G = Geo<KV, D>;
  return static_cast<uint32_t>((row * G::kCpr + (ch ^ swz<KV, D>(row))) * 16);
}

// INT4 ldmatrix row addresses of one lane within a sub-tile (bytes from its
// base).  K (no .trans): lane l gives token l % 8 of group l / 8 (D = 64:
// token l % 8 + 8 ((l / 8) >> 1), group (l / 8) & 1), so matrix j returns,
// for lane (q4, c4), bytes 4c4..4c4+3 of group j of token q4; tokens 8..15
// sit kInt4K1 bytes further (the swizzle repeats every 8 rows).
// V (.trans): matrix m of call c is tokens 8 (m & 1) + 0..7 of group
// 2c + (m >> 1), so lane (q4, c4) gets bytes 2q4, 2q4 + 1 of tokens 2c4 and
// 2c4 + 1 (or + 8).  kz: row (lane % 16) of the K scale tile; the V scale
// tile's row sits kScaleTileBytes further.
struct Int4Lanes {
  uint32_t k0, v0, v1, kz;
};
constexpr uint32_t kInt4K1 = 8 * 64;          // 8 rows of 64 bytes (D = 128)
template <int KV, int D>
__device__ __forceinline__ Int4Lanes int4_lanes(int lane) {
  Int4Lanes o = {0u, 0u, 0u, 0u};
  if constexpr (KV == PKV_INT4_G32) {
    using G = Geo<KV, D>;
    const int r = lane & 7, m = lane >> 3;
    if constexpr (D == 128) {
      o.k0 = chunk_off<KV, D>(r, m);
      o.v0 = G::kTileBytes + chunk_off<KV, D>(r + 8 * (m & 1), m >> 1);
      o.v1 = G::kTileBytes + chunk_off<KV, D>(r + 8 * (m & 1), 2 + (m >> 1));
    } else {
      o.k0 = chunk_off<KV, D>(r + 8 * (m >> 1), m & 1);
      o.v0 = G::kTileBytes + chunk_off<KV, D>(r + 8 * (m & 1), m >> 1);
    }
    o.kz = 2 * G::kTileBytes + (lane & 15) * G::kScaleRowBytes;
  }
  return o;
}

struct Params {
  const uint16_t* q;
  uint8_t* k_cache;           // written only by the fused write
  uint8_t* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  void* scales;
  const uint16_t* k_new;      // fused write: [num_seqs][Hkv][D] in the q dtype, or null
  const uint16_t* v_new;
  const int64_t* slot_mapping;
  void* out;
  float* ws_out;
  float* ws_ml;
  int* dev_status;
  int max_blocks_per_seq;
  int num_seqs;
  int num_blocks;
  int num_q_heads;
  int num_kv_heads;
  int block_size;
  int partition_size;
  int num_partitions;
  int parts_per_cta;
  float softmax_scale;
  const int32_t* q_start;     // prefill: [num_seqs + 1] offsets of each chunk's queries in q
  int max_query_len;          // prefill: queries j >= max_query_len of a chunk are not computed
  // balanced split: the number of warps the tiles are split over
  int bal_warps;
};

// Issue the copies of one 16-token sub-tile into its place in a stage
// (lane-parallel).  `rowp` locates it: (physical block * Hkv + kvh) << 4 |
// (offset in the block / 16), or -1 for a block id out of range; `live` is
// false past the unit's end.  `stage` is the sub-tile's shared-memory base,
// `misc_smem`/`misc` its 16-byte misc slot.  Sub-tiles that copy nothing are
// marked empty.  L1: also allocate the rows in L1 (prefill, where the CTA's
// warps stream the same tiles; decode reads each tile once and runs faster
// without).
template <int KV, int D, bool L1 = false>
__device__ __forceinline__ void issue_tile(const Params& p, int rowp, bool live, uint32_t stage,
                                           uint32_t misc_smem, int* misc, int lane) {
  using G = Geo<KV, D>;
  const bool ok = rowp >= 0;
  if (lane == 0) misc[2] = (live && ok) ? 1 : 0;
  if (!live) return;
  if (!ok) {
    if (lane == 0) flag_status(p.dev_status, PKV_ERR_DEVICE_BOUNDS);
    return;
  }
  const int blk = rowp >> 4;                               // physical block * Hkv + kvh
  const int64_t row0 = static_cast<int64_t>(blk) * p.block_size + ((rowp & 15) << 4);
  const uint8_t* ksrc = p.k_cache + row0 * G::kRowBytes;
  const uint8_t* vsrc = p.v_cache + row0 * G::kRowBytes;
  constexpr int kChunks = G::kTileBytes / 16;
#pragma unroll
  for (int i = 0; i < (kChunks + kWarp - 1) / kWarp; ++i) {
    const int ch = lane + i * kWarp;
    if (kChunks % kWarp == 0 || ch < kChunks) {
      const int r = ch / G::kCpr, c = ch % G::kCpr;
      const uint32_t o = chunk_off<KV, D>(r, c);
      if constexpr (L1) {
        cp_async_16_ca(stage + o, ksrc + ch * 16);
        cp_async_16_ca(stage + G::kTileBytes + o, vsrc + ch * 16);
      } else {
        cp_async_16(stage + o, ksrc + ch * 16);
        cp_async_16(stage + G::kTileBytes + o, vsrc + ch * 16);
      }
    }
  }
  if constexpr (KV == PKV_INT4_G32) {
    // (scale, zero) rows of the tile's 16 tokens, K then V: contiguous runs
    constexpr int kSc = G::kScaleTileBytes / 16;            // 16 (D=128) or 8 (D=64)
    const uint16_t* sc = static_cast<const uint16_t*>(p.scales);
    const int64_t per_kv = static_cast<int64_t>(p.num_blocks) * p.num_kv_heads * p.block_size *
                           (D / 32) * 2;
    const uint8_t* ksc = reinterpret_cast<const uint8_t*>(sc + row0 * (D / 32) * 2);
    const uint8_t* vsc = reinterpret_cast<const uint8_t*>(sc + per_kv + row0 * (D / 32) * 2);
    if (lane < kSc) {
      cp_async_16(stage + 2 * G::kTileBytes + lane * 16, ksc + lane * 16);
    } else if (lane >= 16 && lane < 16 + kSc) {
      cp_async_16(stage + 2 * G::kTileBytes + G::kScaleTileBytes + (lane - 16) * 16,
                  vsc + (lane - 16) * 16);
    }
  } else if constexpr (is_blk8(KV)) {
    const float* sc = static_cast<const float*>(p.scales);
    const int64_t idx = blk;
    const int64_t per_kv = static_cast<int64_t>(p.num_blocks) * p.num_kv_heads;
    const uint32_t mo = misc_smem;
    if (lane == 0) asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(mo), "l"(sc + idx) : "memory");
    if (lane == 1) asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(mo + 4), "l"(sc + per_kv + idx) : "memory");
  }
}

// Fused write: store sequence b's new token for KV head kvh (one warp), as
// paged_kv_write would.  The slot must be -1 (nothing to write) or the slot of
// position ctx - 1 through b's block table: only then is the row read by this
// CTA alone; any other slot is flagged and left unwritten.
template <int KV, int QT, int D>
__device__ __forceinline__ void fused_write(const Params& p, int b, int kvh, int ctx, int lane) {
  // the slot, the table entry of position ctx - 1 and the new K and V rows are
  // independent loads: issued together, they cost one memory latency
  const int64_t row = static_cast<int64_t>(b) * p.num_kv_heads + kvh;
  const int64_t slot = p.slot_mapping[b];
  const int t = ctx - 1;
  const int logical = ctx > 0 ? t / p.block_size : 0;
  const int phys = ctx > 0 ? p.block_tables[static_cast<int64_t>(b) * p.max_blocks_per_seq + logical]
                           : -1;
  const RowWords<D> kw = load_row_words<D>(p.k_new + row * D, lane);
  const RowWords<D> vw = load_row_words<D>(p.v_new + row * D, lane);
  if (slot == -1) return;
  int64_t expect = -2;
  if (ctx > 0 && phys >= 0 && phys < p.num_blocks)
    expect = static_cast<int64_t>(phys) * p.block_size + (t - logical * p.block_size);
  if (slot != expect) {
    if (lane == 0) flag_status(p.dev_status, PKV_ERR_DEVICE_BOUNDS);
    return;
  }
  const int64_t block = slot / p.block_size;
  const int offset = static_cast<int>(slot - block * p.block_size);
  encode_token_head_words<KV, QT, D>(kw, vw, p.k_cache, p.v_cache, p.scales, p.num_blocks,
                                     p.num_kv_heads, p.block_size, block, kvh, offset, lane);
}

// One unit of work: partition `part` of sequence b, KV head kvh.
struct Unit {
  int b, kvh, part, tok_begin, tok_end, ntiles;
};

// Unit = partition `part` of sequence b, KV head kvh.
template <int kTok>
__device__ __forceinline__ Unit make_unit(const Params& p, int b, int kvh, int ctx, int part) {
  Unit u;
  u.b = b;
  u.kvh = kvh;
  u.part = part;
  u.tok_begin = u.part * p.partition_size;
  u.tok_end = min(ctx, u.tok_begin + p.partition_size);
  u.ntiles = ctx > 0 ? (u.tok_end - u.tok_begin + kTok - 1) / kTok : 0;
  return u;
}

// ---------------------------------------------------------------- balanced split
// (kBalMaxSeqs, pkv_internal.h: the most sequences the balanced split takes;
// its tile prefix lives in the CTA's merge buffer, which warp-owned units
// leave unused)
static_assert((kBalMaxSeqs + 1) * 4 <= Geo<PKV_F16, 64>::kMbufBytes, "prefix fits the buffer");

// pfx[b] = Hkv * sum over b' < b of ceil(min(ctx_b', cap) / kTok) for b <= B:
// the first tile of sequence b's first pair in the list of all pairs' tiles.
// Every thread of the CTA calls it (two barriers); CTA 0 also flags contexts
// longer than their table rows.
template <int kTok>
__device__ __forceinline__ void bal_prefix(const Params& p, int* pfx, int cap) {
  constexpr int kThreads = kDecodeWarps * kWarp;
  __shared__ int warp_sum[kDecodeWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = p.num_seqs;
  const int per = (B + kThreads - 1) / kThreads;          // consecutive sequences per thread
  auto tiles_of = [&](int bb) -> int {
    int c = p.context_lens[bb];
    if (c > cap) {
      if (blockIdx.x == 0) flag_status(p.dev_status, PKV_ERR_DEVICE_BOUNDS);
      c = cap;
    }
    return c > 0 ? (c + kTok - 1) / kTok : 0;
  };
  int local = 0;
  for (int i = 0; i < per; ++i)
    if (tid * per + i < B) local += tiles_of(tid * per + i);
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  int run = incl - local;
  for (int w = 0; w < warp; ++w) run += warp_sum[w];
  const int hkv = p.num_kv_heads;
  for (int i = 0; i < per; ++i) {
    const int bb = tid * per + i;
    if (bb < B) {
      pfx[bb] = run * hkv;
      run += tiles_of(bb);
    }
  }
  if (tid == kThreads - 1) pfx[B] = run * hkv;
  __syncthreads();
}

// The pair (b * Hkv + kvh) holding tile t of the list (0 <= t < pfx[B]).
__device__ __forceinline__ int bal_pair_of(const int* pfx, int B, int hkv, int t) {
  int lo = 0, hi = B;                                     // pfx[lo] <= t < pfx[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pfx[mid] <= t) lo = mid;
    else hi = mid;
  }
  const int nt = (pfx[lo + 1] - pfx[lo]) / hkv;
  return lo * hkv + (t - pfx[lo]) / nt;
}

// Warp w's piece of pair `pair`: the pair's tiles that fall in [lo, hi) (none
// for a pair without tokens).  Its partial result goes to workspace slot
// w + pair, distinct for every (warp, pair) since consecutive pairs share at
// most one warp.
template <int kTok>
__device__ __forceinline__ Unit bal_unit(const Params& p, const int* pfx, int cap, int pair,
                                         int lo, int hi, int w) {
  const int hkv = p.num_kv_heads;
  Unit u;
  u.b = pair / hkv;
  u.kvh = pair - u.b * hkv;
  const int nt = (pfx[u.b + 1] - pfx[u.b]) / hkv;
  const int base = pfx[u.b] + u.kvh * nt;
  const int tlo = max(lo, base) - base, thi = min(hi, base + nt) - base;
  const int ctx = max(0, min(p.context_lens[u.b], cap));
  u.part = w + pair;
  u.tok_begin = tlo * kTok;
  u.ntiles = max(0, thi - tlo);
  u.tok_end = min(ctx, thi * kTok);
  return u;
}

// The warp's query columns as the B operand of S^T = K Q^T (column n = q4:
// row `qrow` of q, rows of the operand = d in the order the K fragments use;
// columns without a query (head_ok false) are zero), plus the f16 scaling.  INT4 also gets the B operand of its
// zero-point product (zq, hi + lo f16 words; see the score code) and the
// factor zscale that product's sums are taken back with.  INT8 gets qoff8:
// 128 * the sum over d of q as the mma sees it, for heads 2c4 and 2c4 + 1
// (its codes enter as x + 128).
template <int KV, int QT, int D>
__device__ __forceinline__ void load_q(const uint16_t* qrow, bool head_ok, int q4, int c4,
                                       uint32_t (&qb)[D / 16][2], float& qexp,
                                       uint32_t (&zq)[2], float& zscale, float (&qoff8)[2]) {
  constexpr bool kHalf = (KV == PKV_F16 || KV == PKV_BF16);
  qexp = 1.f;
  if constexpr (kHalf) {
#pragma unroll
    for (int jp = 0; jp < D / 32; ++jp) {
      uint4 v = head_ok ? ld_global_nc_v4(qrow + 8 * (4 * jp + c4)) : make_uint4(0, 0, 0, 0);
      qb[2 * jp][0] = v.x; qb[2 * jp][1] = v.y;
      qb[2 * jp + 1][0] = v.z; qb[2 * jp + 1][1] = v.w;
    }
    zq[0] = zq[1] = 0u;
    zscale = 0.f;
    qoff8[0] = qoff8[1] = 0.f;
  } else {
    // each thread's 32 d values, as float
    float qf[32];
    qoff8[0] = qoff8[1] = 0.f;
    if constexpr (is_blk8(KV)) {
      // d = 16*(4i + c4) + 0..15 for i < D/64
#pragma unroll
      for (int i = 0; i < D / 64; ++i) {
#pragma unroll
        for (int hlf = 0; hlf < 2; ++hlf) {
          uint4 v = head_ok ? ld_global_nc_v4(qrow + 16 * (4 * i + c4) + 8 * hlf) : make_uint4(0, 0, 0, 0);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            qf[16 * i + 8 * hlf + 2 * k] = Half16<QT>::to_float(w[k] & 0xFFFF);
            qf[16 * i + 8 * hlf + 2 * k + 1] = Half16<QT>::to_float(w[k] >> 16);
          }
        }
      }
    } else {
      // INT4: d = 32*grp + 8*c4 + 0..7
#pragma unroll
      for (int grp = 0; grp < D / 32; ++grp) {
        uint4 v = head_ok ? ld_global_nc_v4(qrow + 32 * grp + 8 * c4) : make_uint4(0, 0, 0, 0);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          qf[8 * grp + 2 * k] = Half16<QT>::to_float(w[k] & 0xFFFF);
          qf[8 * grp + 2 * k + 1] = Half16<QT>::to_float(w[k] >> 16);
        }
      }
    }
    constexpr int NQ = D / 4;                  // values per thread: 32 (D=128) or 16 (D=64)
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < NQ; ++i) amax = fmaxf(amax, fabsf(qf[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    // keep |q| * 2^-e below 2^15 so the f16 copy is exact in the normal range
    int e = 0;
    if (amax >= 32768.f) e = ilogbf(amax) - 14;
    const float qs = ldexpf(1.f, -e);
    qexp = ldexpf(1.f, e);
    if constexpr (is_blk8(KV)) {
      zq[0] = zq[1] = 0u;
      zscale = 0.f;
      // k-step 4i+h: lo pair = d 16(4i+c4) + 4h + {0,1}, hi pair = + 4h + {2,3}
      float s16 = 0.f;
#pragma unroll
      for (int i = 0; i < D / 64; ++i)
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          qb[4 * i + h][0] = Half16<PKV_F16>::pack_rn(qf[16 * i + 4 * h] * qs, qf[16 * i + 4 * h + 1] * qs);
          qb[4 * i + h][1] = Half16<PKV_F16>::pack_rn(qf[16 * i + 4 * h + 2] * qs, qf[16 * i + 4 * h + 3] * qs);
          const float2 a = Half16<PKV_F16>::unpack(qb[4 * i + h][0]);
          const float2 c = Half16<PKV_F16>::unpack(qb[4 * i + h][1]);
          s16 += (a.x + a.y) + (c.x + c.y);
        }
      if constexpr (KV == PKV_INT8) {
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) s16 += __shfl_xor_sync(0xffffffffu, s16, o);  // head q4
        qoff8[0] = 128.f * __shfl_sync(0xffffffffu, s16, (2 * c4) * 4);
        qoff8[1] = 128.f * __shfl_sync(0xffffffffu, s16, (2 * c4 + 1) * 4);
      }
    } else {
      // k-step 2grp+h: lo pair = d (8c4 + 2h, 8c4 + 2h + 4), hi pair = (8c4 + 2h + 1, 8c4 + 2h + 5).
      // The hi pairs meet K codes taken as 16 n (high nibbles, no shift), so
      // their q enters divided by 16.
      float zsel = 0.f;                        // sum of q over group c4 of head q4
#pragma unroll
      for (int grp = 0; grp < D / 32; ++grp) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float* x = qf + 8 * grp;
          qb[2 * grp + h][0] = Half16<PKV_F16>::pack_rn(x[2 * h] * qs, x[2 * h + 4] * qs);
          qb[2 * grp + h][1] =
              Half16<PKV_F16>::pack_rn(x[2 * h + 1] * (qs * 0.0625f), x[2 * h + 5] * (qs * 0.0625f));
        }
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) s += qf[8 * grp + k] + qf[8 * grp + k + 4];
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (grp == c4) zsel = s;
      }
      // Zero-point product: the (scale, zero) words of a token's scale row are
      // its A operand (k = 2g: scale of group g, k = 2g + 1: zero of group g),
      // so its B operand is 0 at k = 2c4 and sum(q of group c4) at k = 2c4 + 1,
      // as an f16 hi + lo pair (relative error ~2^-22).  The sum enters times
      // qs / 32, clear of the f16 range (|q qs| < 2^15, 32 terms).
      const float zv = zsel * (qs * 0.03125f);
      const __half zh = __float2half_rn(zv);
      const __half zl = __float2half_rn(zv - __half2float(zh));
      zq[0] = static_cast<uint32_t>(__half_as_ushort(zh)) << 16;
      zq[1] = static_cast<uint32_t>(__half_as_ushort(zl)) << 16;
      zscale = qexp * 32.f;
    }
  }
}

// Fold state B (mb, lb, ob) into state A for the thread's two head columns.
template <int MT>
__device__ __forceinline__ void merge_state(float (&ma)[2], float (&la)[2], float (&oa)[MT][4],
                                            const float* mb, const float* lb, const float* ob) {
  float fa[2], fb[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float M = fmaxf(ma[h], mb[h]);
    fa[h] = ma[h] == -INFINITY ? 0.f : fast_exp2(ma[h] - M);
    fb[h] = mb[h] == -INFINITY ? 0.f : fast_exp2(mb[h] - M);
    la[h] = la[h] * fa[h] + lb[h] * fb[h];
    ma[h] = M;
  }
#pragma unroll
  for (int i = 0; i < MT; ++i) {
    oa[i][0] = oa[i][0] * fa[0] + ob[4 * i + 0] * fb[0];
    oa[i][1] = oa[i][1] * fa[1] + ob[4 * i + 1] * fb[1];
    oa[i][2] = oa[i][2] * fa[0] + ob[4 * i + 2] * fb[0];
    oa[i][3] = oa[i][3] * fa[1] + ob[4 * i + 3] * fb[1];
  }
}

// Decode kernel.  CTA = (run of PPC consecutive partitions, KV head,
// sequence).  The warps share each partition's 16-token tiles (tile t goes to
// warp t % W) and keep their copy rings running across partition boundaries,
// so the next partition's tiles are already in flight while a partition's
// four warp states are merged; Q and the setup are paid once per run.
//
// Two ways to share the work (WU):
//  WU = false: the CTA's units are partitions [blockIdx.x * PPC, +PPC); the
//    four warps share each partition's tiles and merge their states at its end.
//  WU = true (split-KV with many partitions): each warp owns whole units: warp
//    w takes KV head blockIdx.y * W + w of partitions [blockIdx.x * PPC, +PPC),
//    streams their tiles alone and writes its own partial results -- no
//    merges, no barriers, and every warp of a CTA has the same token count.
// PF (prefill, chunked): CTA = (run of 4 query groups, KV head, sequence).
//    Warp w owns query group blockIdx.x * 4 + w: the 8/G query tokens
//    [j0, j0 + 8/G) of the sequence's chunk times the G heads of the KV head
//    are its 8 columns; it streams the cache from token 0 up to its last
//    query's position and masks each column causally.  No partitions, no
//    merges, no barriers (as WU).
template <int KV, int QT, int D, bool WU, bool PF = false, bool BAL = false>
__global__ void __launch_bounds__(kDecodeWarps * kWarp, Geo<KV, D>::kMinBlocks)
paged_decode_kernel(const Params p) {
  using G = Geo<KV, D>;
  constexpr bool kHalf = G::kHalf;
  constexpr int MT = D / 16;                 // m-tiles of O^T (and k-steps of S^T)
  // mma operand type: the cache's type for 16-bit caches, f16 for FP8/INT4
  constexpr int MMA_T = kHalf ? KV : PKV_F16;
  // P enters the second product as 16-bit values times kPScale (clear of f16
  // subnormals).  kTau: the running max is only raised (and O rescaled) when a
  // tile's max exceeds it by more than kTau (log2 units), so P <= 2^kTau; the
  // f16 cases keep kPScale * 2^kTau (* 16 for the FP8 scale ratio) below 2^15.
  constexpr float kPScale = (KV == PKV_BF16 || KV == PKV_INT4_G32) ? 1.f
                                                                   : (KV == PKV_F16 ? 256.f : 64.f);
  constexpr float kTau = (KV == PKV_BF16) ? 8.f : (KV == PKV_F16 ? 6.f : (is_blk8(KV) ? 4.f : 0.f));

  extern __shared__ __align__(128) uint8_t smem[];
  pdl_wait();                 // the cache may have been written by the previous kernel
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int q4 = lane >> 2, c4 = lane & 3;   // mma groupID / thread-in-group
  const int group = p.num_q_heads / p.num_kv_heads;
  const int cap = p.max_blocks_per_seq * p.block_size;

  static_assert(!PF || WU, "prefill runs with warp-owned units");
  static_assert(!BAL || (WU && !PF), "the balanced split is a warp-owned decode mode");
  // Balanced split: the tiles of every (sequence, KV head) pair, in pair order
  // (sequence-major), are one list; warp w of the W = p.bal_warps warps takes
  // tiles [w T / W, (w + 1) T / W) of the T in all.  pfx[b] (in the merge
  // buffer, unused by warp-owned units) is the number of tiles of the pairs
  // before sequence b's first: Hkv * sum over b' < b of ceil(ctx_b' / tile).
  int* pfx = reinterpret_cast<int*>(smem + G::kRingBytes);
  int bal_lo = 0, bal_hi = 0, bal_p0 = 0, bal_w = 0;
  if constexpr (BAL) {
    bal_prefix<G::kTileTok>(p, pfx, cap);
    const int64_t T = pfx[p.num_seqs];
    bal_w = static_cast<int>(blockIdx.x) * kDecodeWarps + warp;
    bal_lo = static_cast<int>(static_cast<int64_t>(bal_w) * T / p.bal_warps);
    bal_hi = static_cast<int>(static_cast<int64_t>(bal_w + 1) * T / p.bal_warps);
    if (bal_hi > bal_lo) bal_p0 = bal_pair_of(pfx, p.num_seqs, p.num_kv_heads, bal_lo);
  }
  const int kvh = PF ? static_cast<int>(blockIdx.y)
                     : (BAL ? 0
                            : (WU ? static_cast<int>(blockIdx.y) * kDecodeWarps + warp
                                  : static_cast<int>(blockIdx.y)));
  const int b = BAL ? 0 : blockIdx.z;
  if (WU && !BAL && kvh >= p.num_kv_heads) return;
  int ctx = BAL ? 0 : p.context_lens[b];
  if (!BAL && ctx > cap) {
    // a context longer than its table row can hold is clamped (and flagged)
    if (lane == 0 && blockIdx.x == 0 && kvh == 0) flag_status(p.dev_status, PKV_ERR_DEVICE_BOUNDS);
    ctx = cap;
  }
  // prefill: this warp's queries j0 .. j0 + qpw - 1 of the chunk, query j at
  // position pos0 + j (pos0 = ctx - nq), the cache tokens they see [0, pf_end);
  // queries from max_query_len on are not computed (nqc = computed queries).
  // A chunk longer than the context is flagged; its queries at negative
  // positions see nothing and give zeros.
  const int qpw = PF ? kWarp / 4 / group : 0;               // 8 / G query tokens per warp
  int nq = 0, nqc = 0, j0 = 0, pos0 = 0, pf_end = 0;
  if constexpr (PF) {
    nq = p.q_start[b + 1] - p.q_start[b];
    nqc = min(nq, p.max_query_len);
    j0 = (static_cast<int>(blockIdx.x) * kDecodeWarps + warp) * qpw;
    if (j0 >= nqc) return;                                   // no query for this warp
    pos0 = ctx - nq;
    if (pos0 < 0 && j0 == 0 && lane == 0) flag_status(p.dev_status, PKV_ERR_DEVICE_BOUNDS);
    pf_end = max(0, pos0 + min(j0 + qpw, nqc));
  }
  const int nparts_seq = (PF || BAL) ? 1 : (ctx > 0 ? (ctx + p.partition_size - 1) / p.partition_size : 1);
  // unit j -> partition; tiles of a unit this warp takes: kFirst, kFirst + kStride, ...
  constexpr int kStride = WU ? 1 : kDecodeWarps;
  const int kFirst = WU ? 0 : warp;
  const int pbase = (PF || BAL) ? 0 : static_cast<int>(blockIdx.x) * p.parts_per_cta;
  auto part_of = [&](int j) -> int { return pbase + j; };
  int nunits;
  if constexpr (BAL) {
    // the pairs this warp's tiles touch: bal_p0 .. the pair of its last tile
    nunits = bal_hi > bal_lo
                 ? bal_pair_of(pfx, p.num_seqs, p.num_kv_heads, bal_hi - 1) - bal_p0 + 1
                 : 0;
    if (nunits == 0 && bal_lo < pfx[p.num_seqs]) {
      // more warps than tiles: a warp without tiles still sits between the
      // owners of tile bal_lo's pair, so it leaves an empty piece (max -inf,
      // sum 0, zero rows) in its slot for the merge
      const int pair = bal_pair_of(pfx, p.num_seqs, p.num_kv_heads, bal_lo);
      const int64_t row0 = static_cast<int64_t>(bal_w + pair) * group;
      for (int g = 0; g < group; ++g) {
        for (int d = lane; d < D; d += kWarp) p.ws_out[(row0 + g) * D + d] = 0.f;
        if (lane == 0) {
          p.ws_ml[(row0 + g) * 2] = -INFINITY;
          p.ws_ml[(row0 + g) * 2 + 1] = 0.f;
        }
      }
    }
  } else {
    nunits = PF ? 1 : min(p.parts_per_cta, nparts_seq - pbase);
  }
  if (nunits <= 0) return;                 // the whole CTA (same b and partitions for all
                                           // warps), or (balanced) a warp without tiles
  auto unit_at = [&](int j) -> Unit {
    if constexpr (BAL) {
      return bal_unit<G::kTileTok>(p, pfx, cap, bal_p0 + j, bal_lo, bal_hi, bal_w);
    } else if constexpr (PF) {
      Unit u;
      u.b = b;
      u.kvh = kvh;
      u.part = 0;
      u.tok_begin = 0;
      u.tok_end = pf_end;
      u.ntiles = (pf_end + G::kTileTok - 1) / G::kTileTok;
      return u;
    } else {
      return make_unit<G::kTileTok>(p, b, kvh, ctx, part_of(j));
    }
  };

  uint8_t* ring_ptr = smem + warp * G::kWarpRing;
  const uint32_t ring = smem_u32(ring_ptr);
  float* mbuf = reinterpret_cast<float*>(smem + G::kRingBytes);                 // [32][kMbStride]

  // ---------------------------------------------------------------- issue cursor
  // Walks (unit, tile) pairs with tile = warp, warp + W, ... < ntiles, in unit
  // order.  The cache rows of the warp's 16-token sub-tiles of a unit are
  // looked up 32 at a time, one per lane (lane l of window k: the warp's
  // sub-tile 32k + l, i.e. sub-tile (32k + l) % kSub of its tile (32k + l) /
  // kSub), as (physical block * Hkv + kvh) << 4 | (offset in the block / 16),
  // or -1 when the sub-tile is past the unit or its block id is out of range;
  // window 0 of the next unit is prefetched on entering a unit.
  int iu = -1, it = 0, i_tb = 0, i_next_tb = -1, i_win = 0;
  Unit iunit;
  iunit.ntiles = 0;
  auto window = [&](const Unit& u, int k) -> int {
    const int sidx = 32 * k + lane;
    const int tile = kFirst + kStride * (sidx / G::kSub);
    const int tok = u.tok_begin + tile * G::kTileTok + (sidx % G::kSub) * kTile;
    if (tile >= u.ntiles || tok >= u.tok_end) return -1;
    const int32_t* trow = p.block_tables + static_cast<int64_t>(u.b) * p.max_blocks_per_seq;
    const int logical = tok / p.block_size;
    const int phys = __ldg(trow + logical);
    if (phys < 0 || phys >= p.num_blocks) return -1;
    return ((phys * p.num_kv_heads + u.kvh) << 4) | ((tok - logical * p.block_size) >> 4);
  };
  auto next_window_unit = [&](int j) -> int {          // window 0 of unit j (or -1s)
    return j < nunits ? window(unit_at(j), 0) : -1;
  };
  // advance to the next pair this warp issues; false when the stream is done
  auto issue_advance = [&]() -> bool {
    it += kStride;
    while (it >= iunit.ntiles) {
      if (iu + 1 >= nunits) return false;
      ++iu;
      iunit = unit_at(iu);
      it = kFirst;
      i_tb = i_next_tb;                                  // prefetched window 0 of unit iu
      i_win = 0;
      i_next_tb = next_window_unit(iu + 1);
    }
    const int k = (it - kFirst) / kStride * G::kSub;     // the warp's first sub-tile index
    if ((k >> 5) != i_win) {                              // beyond 32 sub-tiles: next window
      i_win = k >> 5;
      i_tb = window(iunit, i_win);
    }
    return true;
  };
  int s_issue = 0;                                       // ring stage the next pair goes to
  auto issue_next = [&]() {
    if (issue_advance()) {
      const int k = (it - kFirst) / kStride * G::kSub;
      const uint32_t sb = ring + s_issue * G::kStageBytes;
      uint8_t* sp = ring_ptr + s_issue * G::kStageBytes;
#pragma unroll
      for (int u = 0; u < G::kSub; ++u) {
        const int rowp = __shfl_sync(0xffffffffu, i_tb, (k + u) & 31);
        issue_tile<KV, D, PF>(p, rowp, iunit.tok_begin + it * G::kTileTok + u * kTile < iunit.tok_end,
                          sb + u * G::kSubBytes, sb + G::kMiscOffset + 16 * u,
                          reinterpret_cast<int*>(sp + G::kMiscOffset + 16 * u), lane);
      }
    }
    s_issue = s_issue + 1 == G::kStages ? 0 : s_issue + 1;
    cp_async_commit();
  };
  // Fused write: the CTA (warp-owned units: the warp) holding b's last
  // partition stores b's new token for its KV head before issuing any copy.
  // Balanced split: the warp holding a pair's last tile, for each such pair,
  // before it issues that tile.  A piece's last tile is the new token's; when
  // it sits among the first kStages tiles of the warp's stream (issued before
  // the loop) the token is written first, otherwise only after those first
  // copies are on their way, so that the write's latency overlaps theirs.
  auto bal_writes = [&](bool early) {
    int pos = 0;                                   // tiles of the stream before piece j's end
#pragma unroll 1
    for (int j = 0; j < nunits; ++j) {
      const Unit u = unit_at(j);
      pos += u.ntiles;
      const int cb = max(0, min(p.context_lens[u.b], cap));
      if (u.ntiles > 0 && u.tok_end == cb && (pos <= G::kStages) == early)
        fused_write<KV, QT, D>(p, u.b, u.kvh, cb, lane);
    }
    __syncwarp();
  };
  if constexpr (BAL) {
    if (p.slot_mapping != nullptr) bal_writes(true);
  } else if (p.slot_mapping != nullptr && pbase + nunits == nparts_seq) {
    if (WU || warp == 0) fused_write<KV, QT, D>(p, b, kvh, ctx, lane);
    if constexpr (WU) {
      __syncwarp();
    } else {
      __syncthreads();
    }
  }

  // the first advance enters unit 0 (it + W >= ntiles = 0) with its prefetched window
  it = 0;
  i_next_tb = next_window_unit(0);
#pragma unroll 1
  for (int s = 0; s < G::kStages; ++s) issue_next();
  if constexpr (BAL) {
    if (p.slot_mapping != nullptr) bal_writes(false);
  }

  // INT4: this lane's ldmatrix row addresses within a sub-tile
  const Int4Lanes i4 = int4_lanes<KV, D>(lane);
  // prefill: the last token this thread's columns 2c4, 2c4 + 1 see (their
  // query's position); columns without a query are left unmasked (zero q)
  int lim[2] = {INT_MAX, INT_MAX};
  bool col_q[2] = {false, false}, col_zero[2] = {false, false};
  if constexpr (PF) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int jj = (2 * c4 + h) / group;
      col_q[h] = jj < qpw && j0 + jj < nqc;
      if (col_q[h]) {
        const int pos = pos0 + j0 + jj;
        if (pos >= 0) lim[h] = pos;
        else col_zero[h] = true;                  // a query at a negative position
      }
    }
  }

  // ---------------------------------------------------------------- state
  uint32_t qb[MT][2];
  float qexp = 1.f;
  uint32_t zq[2];                            // INT4: B operand of the zero-point product
  float zscale;
  float qoff8[2];                            // INT8: 128 * sum of q (heads 2c4, 2c4 + 1)
  float zp[2];                               // INT8: running sum of P' (heads 2c4, 2c4 + 1)
  float oacc[MT][4];
  float mrow[2], lrow[2];
  float zc[4];                               // INT4: zero-point sums (C fragment)
  float vref, inv_vref;                      // FP8: oacc is in units of vref / kPScale
  int s_cons = 0;                            // ring stage of the next pair to compute
  // this lane's query column q4: decode, head q4 of the group; prefill, token
  // j0 + q4 / G of the chunk, head q4 % G
  bool q_ok;
  int64_t q_row;
  if constexpr (PF) {
    const int jj = q4 / group;
    q_ok = jj < qpw && j0 + jj < nqc && pos0 + j0 + jj >= 0;
    q_row = static_cast<int64_t>(p.q_start[b]) + j0 + (q_ok ? jj : 0);
  } else {
    q_ok = q4 < group;
    q_row = b;
  }
  if constexpr (!BAL) {
    const uint16_t* qrow = p.q + (q_row * p.num_q_heads + kvh * group + (q_ok ? q4 % group : 0)) * D;
    load_q<KV, QT, D>(qrow, q_ok, q4, c4, qb, qexp, zq, zscale, qoff8);
  }

#pragma unroll 1
  for (int cu = 0; cu < nunits; ++cu) {
    const Unit unit = unit_at(cu);
    if constexpr (BAL) {
      // each piece may belong to another sequence and KV head: its own q
      const uint16_t* qrow =
          p.q + ((static_cast<int64_t>(unit.b) * p.num_q_heads + unit.kvh * group +
                  (q_ok ? q4 : 0)) * D);
      load_q<KV, QT, D>(qrow, q_ok, q4, c4, qb, qexp, zq, zscale, qoff8);
    }
#pragma unroll
    for (int i = 0; i < MT; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
    mrow[0] = mrow[1] = -INFINITY;           // running max (log2 units), heads 2c4, 2c4+1
    lrow[0] = lrow[1] = 0.f;                 // this thread's share of the running sum
    zc[0] = zc[1] = zc[2] = zc[3] = 0.f;
    zp[0] = zp[1] = 0.f;
    vref = 0.f;
    inv_vref = 0.f;
    const float base = p.softmax_scale * kLog2e * qexp;
    const float kq24 = qexp * 16777216.f;    // INT4: undoes the codes' 2^-24 and q's scaling
    const int tok_end = unit.tok_end;

#pragma unroll 1
    for (int ct = kFirst; ct < unit.ntiles; ct += kStride) {
      cp_async_wait<G::kStages - 1>();
      __syncwarp();
      const int stage = s_cons;
      const uint32_t stb = ring + stage * G::kStageBytes;
      const uint8_t* st_ptr = ring_ptr + stage * G::kStageBytes;
      const int* misc0 = reinterpret_cast<const int*>(st_ptr + G::kMiscOffset);
      const int t0 = unit.tok_begin + ct * G::kTileTok;
      // sub-tile u covers tokens [t0 + 16u, t0 + 16u + 16)
      int nval[G::kSub];
      bool any_valid = false;
#pragma unroll
      for (int u = 0; u < G::kSub; ++u) {
        nval[u] = misc0[4 * u + 2] ? max(0, min(kTile, tok_end - (t0 + kTile * u))) : 0;
        any_valid |= nval[u] > 0;
      }

      if (any_valid) {
        float scs[G::kSub][4];
#pragma unroll
        for (int u = 0; u < G::kSub; ++u) {
          const uint32_t st = stb + u * G::kSubBytes;
          const int* misc = misc0 + 4 * u;
          const int nvalid = nval[u];
            // ------------------------------------------------ S^T = K_tile Q^T
            float sc[4] = {0.f, 0.f, 0.f, 0.f};
            float sc2[4] = {0.f, 0.f, 0.f, 0.f};     // second chain: halves the mma dependency depth
            if constexpr (kHalf) {
#pragma unroll
              for (int jp = 0; jp < D / 32; ++jp) {
                // thread reads chunk 4jp+c4 of rows q4 and q4+8: words = d pairs
                const uint4 r0 = ld_shared_v4(st + chunk_off<KV, D>(q4, 4 * jp + c4));
                const uint4 r1 = ld_shared_v4(st + chunk_off<KV, D>(q4 + 8, 4 * jp + c4));
                const uint32_t a0[4] = {r0.x, r1.x, r0.y, r1.y};
                mma_16816<MMA_T>(sc, a0, qb[2 * jp][0], qb[2 * jp][1]);
                const uint32_t a1[4] = {r0.z, r1.z, r0.w, r1.w};
                mma_16816<MMA_T>(sc2, a1, qb[2 * jp + 1][0], qb[2 * jp + 1][1]);
              }
            } else if constexpr (is_blk8(KV)) {
#pragma unroll
              for (int i = 0; i < D / 64; ++i) {
                const uint4 r0 = ld_shared_v4(st + chunk_off<KV, D>(q4, 4 * i + c4));
                const uint4 r1 = ld_shared_v4(st + chunk_off<KV, D>(q4 + 8, 4 * i + c4));
                const uint32_t w0[4] = {b8_prep<KV>(r0.x), b8_prep<KV>(r0.y), b8_prep<KV>(r0.z),
                                        b8_prep<KV>(r0.w)};
                const uint32_t w1[4] = {b8_prep<KV>(r1.x), b8_prep<KV>(r1.y), b8_prep<KV>(r1.z),
                                        b8_prep<KV>(r1.w)};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                  const uint32_t a[4] = {b8_lo<KV>(w0[h]), b8_lo<KV>(w1[h]), b8_hi<KV>(w0[h]),
                                         b8_hi<KV>(w1[h])};
                  if (h & 1)
                    mma_16816<PKV_F16>(sc2, a, qb[4 * i + h][0], qb[4 * i + h][1]);
                  else
                    mma_16816<PKV_F16>(sc, a, qb[4 * i + h][0], qb[4 * i + h][1]);
                }
              }
            } else {
              // INT4: one fresh accumulator per 32-element group for the codes
              // (taken as n 2^-24 and 16 n 2^-24, met by q and q / 16), then
              // s = 2^24 qexp sum_g scale_t,g acc_g + zero-point product.
              constexpr int NG = D / 32;
              constexpr int SR = G::kScaleRowBytes;
              const uint32_t ksc = st + 2 * G::kTileBytes;
              uint32_t w0[NG], w1[NG];               // codes of tokens q4, q4 + 8 per group
              {
                uint32_t r[4];
                ldmatrix_x4(st + i4.k0, r);
                if constexpr (D == 128) {
                  w0[0] = r[0]; w0[1] = r[1]; w0[2] = r[2]; w0[3] = r[3];
                  ldmatrix_x4(st + i4.k0 + kInt4K1, r);
                  w1[0] = r[0]; w1[1] = r[1]; w1[2] = r[2]; w1[3] = r[3];
                } else {
                  w0[0] = r[0]; w0[1] = r[1]; w1[0] = r[2]; w1[1] = r[3];
                }
              }
              uint32_t sz0[NG], sz1[NG];             // (scale, zero) words of tokens q4, q4 + 8
              uint64_t sc01 = tc::f2_pack(0.f, 0.f), sc23 = tc::f2_pack(0.f, 0.f);
              if constexpr (D == 128) {
                const uint4 a = ld_shared_v4(ksc + q4 * SR), c = ld_shared_v4(ksc + (q4 + 8) * SR);
                sz0[0] = a.x; sz0[1] = a.y; sz0[2] = a.z; sz0[3] = a.w;
                sz1[0] = c.x; sz1[1] = c.y; sz1[2] = c.z; sz1[3] = c.w;
              } else {
                const uint2 a = ld_shared_v2(ksc + q4 * SR), c = ld_shared_v2(ksc + (q4 + 8) * SR);
                sz0[0] = a.x; sz0[1] = a.y; sz1[0] = c.x; sz1[1] = c.y;
              }
              // zero-point product: rows = tokens, k = the scale row's 16-bit
              // columns (word c4 = scale and zero of group c4)
              float zs[4] = {0.f, 0.f, 0.f, 0.f};
              {
                uint32_t za[4] = {0u, 0u, 0u, 0u};
                if constexpr (D == 128) {
                  uint32_t r[2];
                  ldmatrix_x2(st + i4.kz, r);
                  za[0] = r[0]; za[1] = r[1];
                } else {
                  if (c4 < NG) {
                    za[0] = ld_shared_b32(ksc + q4 * SR + 4 * c4);
                    za[1] = ld_shared_b32(ksc + (q4 + 8) * SR + 4 * c4);
                  }
                }
                mma_16816<PKV_F16>(zs, za, zq[0], 0u);
                mma_16816<PKV_F16>(zs, za, zq[1], 0u);
              }
#pragma unroll
              for (int grp = 0; grp < NG; ++grp) {
                float g4[4] = {0.f, 0.f, 0.f, 0.f};
                const uint32_t w0s = w0[grp] >> 8, w1s = w1[grp] >> 8;
                const uint32_t a0[4] = {nib_lo(w0[grp]), nib_lo(w1[grp]), nib_hi(w0[grp]), nib_hi(w1[grp])};
                mma_16816<PKV_F16>(g4, a0, qb[2 * grp][0], qb[2 * grp][1]);
                const uint32_t a1[4] = {nib_lo(w0s), nib_lo(w1s), nib_hi(w0s), nib_hi(w1s)};
                mma_16816<PKV_F16>(g4, a1, qb[2 * grp + 1][0], qb[2 * grp + 1][1]);
                const float s0 = __low2float(*reinterpret_cast<const __half2*>(&sz0[grp]));
                const float s1 = __low2float(*reinterpret_cast<const __half2*>(&sz1[grp]));
                sc01 = tc::f2_fma(tc::f2_pack(s0, s0), tc::f2_pack(g4[0], g4[1]), sc01);
                sc23 = tc::f2_fma(tc::f2_pack(s1, s1), tc::f2_pack(g4[2], g4[3]), sc23);
              }
              {
                const uint64_t q2 = tc::f2_pack(kq24, kq24), z2 = tc::f2_pack(zscale, zscale);
                const float2 a = tc::f2_unpack(tc::f2_fma(sc01, q2, tc::f2_mul(tc::f2_pack(zs[0], zs[1]), z2)));
                const float2 c = tc::f2_unpack(tc::f2_fma(sc23, q2, tc::f2_mul(tc::f2_pack(zs[2], zs[3]), z2)));
                sc[0] = a.x; sc[1] = a.y; sc[2] = c.x; sc[3] = c.y;
              }
            }

#pragma unroll
            for (int k = 0; k < 4; ++k) sc[k] += sc2[k];
            if constexpr (KV == PKV_INT8) {
              // codes entered as (x + 128) 2^-24: sum q x = 2^24 acc - 128 sum q
              sc[0] = sc[0] * 16777216.f - qoff8[0];
              sc[1] = sc[1] * 16777216.f - qoff8[1];
              sc[2] = sc[2] * 16777216.f - qoff8[0];
              sc[3] = sc[3] * 16777216.f - qoff8[1];
            }

          // ---------------------------------------------- scale and mask
          float mult = base;
          if constexpr (is_blk8(KV)) {
            mult *= reinterpret_cast<const float*>(misc)[0];
          } else if constexpr (KV == PKV_INT4_G32) {
            mult = p.softmax_scale * kLog2e;     // qexp already folded into the group sums
          }
          const bool v0 = q4 < nvalid, v1 = q4 + 8 < nvalid;
          if constexpr (PF) {
            // causal: column c sees tokens <= lim[c] (rows q4 and q4 + 8)
            const int ta = t0 + kTile * u + q4, tb = ta + 8;
            scs[u][0] = (v0 && ta <= lim[0]) ? sc[0] * mult : -INFINITY;
            scs[u][1] = (v0 && ta <= lim[1]) ? sc[1] * mult : -INFINITY;
            scs[u][2] = (v1 && tb <= lim[0]) ? sc[2] * mult : -INFINITY;
            scs[u][3] = (v1 && tb <= lim[1]) ? sc[3] * mult : -INFINITY;
          } else {
            scs[u][0] = v0 ? sc[0] * mult : -INFINITY;
            scs[u][1] = v0 ? sc[1] * mult : -INFINITY;
            scs[u][2] = v1 ? sc[2] * mult : -INFINITY;
            scs[u][3] = v1 ? sc[3] * mult : -INFINITY;
          }
        }

        // ------------------------------------------------ online softmax over the tile
        // this lane's rows' max per head (the eight lanes of a head column are
        // reduced only when the running max has to move)
        float tmax0 = -INFINITY, tmax1 = -INFINITY;
#pragma unroll
        for (int u = 0; u < G::kSub; ++u) {
          tmax0 = fmaxf(tmax0, fmaxf(scs[u][0], scs[u][2]));
          tmax1 = fmaxf(tmax1, fmaxf(scs[u][1], scs[u][3]));
        }
        // Lazy rescale: the running max moves (and O, l, the INT4 zero sums are
        // rescaled) only when some head's tile max exceeds it by more than kTau,
        // or when the FP8 reference V scale must be rebased.  Some lane's row
        // max exceeds its head's running max + kTau exactly when the head's
        // tile max does, so the test needs no reduction across lanes.
        // A block whose FP8 scale is 0 was never written: its V rows dequantize
        // to 0 and add nothing (its scores still count in the softmax sum).
        bool von[G::kSub];
        float vfac[G::kSub];                     // FP8: a sub-tile's V scale / vref
        bool rebase = false;
        float vmax = 0.f;
#pragma unroll
        for (int u = 0; u < G::kSub; ++u) {
          von[u] = nval[u] > 0;
          vfac[u] = 1.f;
          if constexpr (is_blk8(KV)) {
            const float vs = reinterpret_cast<const float*>(misc0 + 4 * u)[1];
            von[u] = von[u] && vs > 0.f;
            if (von[u]) {
              vfac[u] = vs * inv_vref;           // 0 while no reference is set
              rebase |= !(vfac[u] >= 0.0625f && vfac[u] <= 16.f);
              vmax = fmaxf(vmax, vs);
            }
          }
        }
        const bool grow = tmax0 > mrow[0] + kTau || tmax1 > mrow[1] + kTau;
        if (__any_sync(0xffffffffu, grow) || rebase) {
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) {
            tmax0 = fmaxf(tmax0, __shfl_xor_sync(0xffffffffu, tmax0, o));
            tmax1 = fmaxf(tmax1, __shfl_xor_sync(0xffffffffu, tmax1, o));
          }
          const float mnew0 = fmaxf(mrow[0], tmax0), mnew1 = fmaxf(mrow[1], tmax1);
          // mnew is finite: at least one token of the tile is valid
          float alpha0 = fast_exp2(mrow[0] - mnew0), alpha1 = fast_exp2(mrow[1] - mnew1);
          mrow[0] = mnew0; mrow[1] = mnew1;
          lrow[0] *= alpha0; lrow[1] *= alpha1;
          if constexpr (KV == PKV_INT4_G32) { zc[0] *= alpha0; zc[1] *= alpha1; }
          if constexpr (is_blk8(KV)) {
            if (rebase) {
              // new reference: the tile's largest V scale; O_true = oacc * vref /
              // kPScale stays invariant across the rebase
              const float r = __frcp_rn(vmax);
              const float f = vref > 0.f ? vref * r : 1.f;
              alpha0 *= f; alpha1 *= f;
              vref = vmax; inv_vref = r;
#pragma unroll
              for (int u = 0; u < G::kSub; ++u)
                vfac[u] = reinterpret_cast<const float*>(misc0 + 4 * u)[1] * r;
            }
          }
#pragma unroll
          for (int i = 0; i < MT; ++i) {
            oacc[i][0] *= alpha0; oacc[i][1] *= alpha1;
            oacc[i][2] *= alpha0; oacc[i][3] *= alpha1;
          }
          if constexpr (KV == PKV_INT8) { zp[0] *= alpha0; zp[1] *= alpha1; }
        }

#pragma unroll
        for (int u = 0; u < G::kSub; ++u) {
          const uint32_t st = stb + u * G::kSubBytes;
          const int nvalid = nval[u];
          const bool v_on = von[u];
          const float pr[4] = {fast_exp2(scs[u][0] - mrow[0]), fast_exp2(scs[u][1] - mrow[1]),
                               fast_exp2(scs[u][2] - mrow[0]), fast_exp2(scs[u][3] - mrow[1])};
          lrow[0] += pr[0] + pr[2];
          lrow[1] += pr[1] + pr[3];
          const float vfac_u = vfac[u];
            // ------------------------------------------------ O^T += V_tile^T P^T
            const uint32_t vt = st + G::kTileBytes;
            // rows (tokens) this thread's V fragments cover: 2c4, 2c4+1, 2c4+8, 2c4+9
            const int tA = 2 * c4, tB = 2 * c4 + 1, tC = 2 * c4 + 8, tE = 2 * c4 + 9;
            const bool partial = nvalid < kTile;
            const uint32_t mA = (tA < nvalid) ? 0xFFFFFFFFu : 0u, mB = (tB < nvalid) ? 0xFFFFFFFFu : 0u;
            const uint32_t mC = (tC < nvalid) ? 0xFFFFFFFFu : 0u, mE = (tE < nvalid) ? 0xFFFFFFFFu : 0u;

            if (v_on) {
            if constexpr (KV != PKV_INT4_G32) {
              // P as B fragments (hi + lo split)
              using H = Half16<MMA_T>;
              const float ps = kPScale * vfac_u;
              const float pp[4] = {pr[0] * ps, pr[1] * ps, pr[2] * ps, pr[3] * ps};
              const uint32_t h01 = H::pack_rn(pp[0], pp[1]), h23 = H::pack_rn(pp[2], pp[3]);
              const float2 f01 = H::unpack(h01), f23 = H::unpack(h23);
              const uint32_t l01 = H::pack_rn(pp[0] - f01.x, pp[1] - f01.y);
              const uint32_t l23 = H::pack_rn(pp[2] - f23.x, pp[3] - f23.y);
              const uint32_t bh0 = movmatrix_trans(h01), bh1 = movmatrix_trans(h23);
              const uint32_t bl0 = movmatrix_trans(l01), bl1 = movmatrix_trans(l23);
              if constexpr (KV == PKV_INT8) {
                // the P' the products see (hi + lo, within 2^-22): their sum
                // takes the codes' offset of 128 off in the epilogue
                zp[0] += pp[0] + pp[2];
                zp[1] += pp[1] + pp[3];
              }

              if constexpr (kHalf) {
#pragma unroll
                for (int hc = 0; hc < D / 64; ++hc) {
                  // chunk (D/64 == 2 ? 2*q4 + hc : q4): d = 16*q4 + 8*hc + 0..7 (D=128) or 8*q4 + 0..7
                  const int ch = (D == 128) ? 2 * q4 + hc : q4;
                  uint4 A = ld_shared_v4(vt + chunk_off<KV, D>(tA, ch));
                  uint4 B = ld_shared_v4(vt + chunk_off<KV, D>(tB, ch));
                  uint4 C = ld_shared_v4(vt + chunk_off<KV, D>(tC, ch));
                  uint4 E = ld_shared_v4(vt + chunk_off<KV, D>(tE, ch));
                  if (partial) {
                    A.x &= mA; A.y &= mA; A.z &= mA; A.w &= mA;
                    B.x &= mB; B.y &= mB; B.z &= mB; B.w &= mB;
                    C.x &= mC; C.y &= mC; C.z &= mC; C.w &= mC;
                    E.x &= mE; E.y &= mE; E.z &= mE; E.w &= mE;
                  }
                  const uint32_t wa[4] = {A.x, A.y, A.z, A.w}, wb[4] = {B.x, B.y, B.z, B.w};
                  const uint32_t wc[4] = {C.x, C.y, C.z, C.w}, we[4] = {E.x, E.y, E.z, E.w};
#pragma unroll
                  for (int k = 0; k < 4; ++k) {
                    const int i = 4 * hc + k;                       // m-tile: d = base + 2i (+1)
                    const uint32_t a[4] = {__byte_perm(wa[k], wb[k], 0x5410), __byte_perm(wa[k], wb[k], 0x7632),
                                           __byte_perm(wc[k], we[k], 0x5410), __byte_perm(wc[k], we[k], 0x7632)};
                    mma_16816<MMA_T>(oacc[i], a, bh0, bh1);
                    mma_16816<MMA_T>(oacc[i], a, bl0, bl1);
                  }
                }
              } else {
                // FP8: d = base(q4) + 0..15 (D=128) or 8*q4 + 0..7 (D=64)
                constexpr int NW = D / 32;                          // words per token: 4 or 2
                uint32_t wa[NW], wb[NW], wc[NW], we[NW];
                if constexpr (D == 128) {
                  const int pi = ((q4 & 1) << 1) | ((q4 >> 1) & 1) | (q4 & 4);
                  const uint4 A = ld_shared_v4(vt + chunk_off<KV, D>(tA, pi));
                  const uint4 B = ld_shared_v4(vt + chunk_off<KV, D>(tB, pi));
                  const uint4 C = ld_shared_v4(vt + chunk_off<KV, D>(tC, pi));
                  const uint4 E = ld_shared_v4(vt + chunk_off<KV, D>(tE, pi));
                  wa[0] = A.x; wa[1] = A.y; wa[2] = A.z; wa[3] = A.w;
                  wb[0] = B.x; wb[1] = B.y; wb[2] = B.z; wb[3] = B.w;
                  wc[0] = C.x; wc[1] = C.y; wc[2] = C.z; wc[3] = C.w;
                  we[0] = E.x; we[1] = E.y; we[2] = E.z; we[3] = E.w;
                } else {
                  const uint2 A = ld_shared_v2(vt + tA * G::kRowBytes + 8 * q4);
                  const uint2 B = ld_shared_v2(vt + tB * G::kRowBytes + 8 * q4);
                  const uint2 C = ld_shared_v2(vt + tC * G::kRowBytes + 8 * q4);
                  const uint2 E = ld_shared_v2(vt + tE * G::kRowBytes + 8 * q4);
                  wa[0] = A.x; wa[1] = A.y; wb[0] = B.x; wb[1] = B.y;
                  wc[0] = C.x; wc[1] = C.y; we[0] = E.x; we[1] = E.y;
                }
                if constexpr (is_fp8(KV)) {
                  // stale FP8 bytes past the context may be NaN codes (p is 0
                  // there, but 0 * NaN is not); INT8 codes are always finite
                  if (partial) {
#pragma unroll
                    for (int k = 0; k < NW; ++k) { wa[k] &= mA; wb[k] &= mB; wc[k] &= mC; we[k] &= mE; }
                  }
                }
#pragma unroll
                for (int k = 0; k < NW; ++k) {
                  // token pairs (tA, tB), (tC, tE) byte-interleaved per d
                  const uint32_t x01 = b8_prep<KV>(__byte_perm(wa[k], wb[k], 0x5140));
                  const uint32_t x23 = b8_prep<KV>(__byte_perm(wa[k], wb[k], 0x7362));
                  const uint32_t y01 = b8_prep<KV>(__byte_perm(wc[k], we[k], 0x5140));
                  const uint32_t y23 = b8_prep<KV>(__byte_perm(wc[k], we[k], 0x7362));
                  const uint32_t a0[4] = {b8_lo<KV>(x01), b8_hi<KV>(x01), b8_lo<KV>(y01), b8_hi<KV>(y01)};
                  mma_16816<PKV_F16>(oacc[2 * k], a0, bh0, bh1);
                  mma_16816<PKV_F16>(oacc[2 * k], a0, bl0, bl1);
                  const uint32_t a1[4] = {b8_lo<KV>(x23), b8_hi<KV>(x23), b8_lo<KV>(y23), b8_hi<KV>(y23)};
                  mma_16816<PKV_F16>(oacc[2 * k + 1], a1, bh0, bh1);
                  mma_16816<PKV_F16>(oacc[2 * k + 1], a1, bl0, bl1);
                }
              }
            } else {
              // INT4: O^T += V_codes^T P'_g^T per group g, with P'_g = p * scale_t,g
              // formed on the B operand (f16), and the zero points through one
              // more product: rows = the V scale row's 16-bit columns (scale and
              // zero of each group), k = tokens, times P^T.
              constexpr int NG = D / 32;
              constexpr int SR = G::kScaleRowBytes;
              const uint32_t vsc = st + 2 * G::kTileBytes + G::kScaleTileBytes;
              using H = Half16<PKV_F16>;
              // P^T as B fragments: head q4, tokens 2c4 + {0, 1} (bp0) and + 8 (bp1),
              // as an f16 hi + lo pair (p = hi + lo to ~2^-22)
              const uint32_t ph01 = H::pack_rn(pr[0], pr[1]), ph23 = H::pack_rn(pr[2], pr[3]);
              const float2 f01 = H::unpack(ph01), f23 = H::unpack(ph23);
              const uint32_t bp0 = movmatrix_trans(ph01);
              const uint32_t bp1 = movmatrix_trans(ph23);
              const uint32_t bl0 = movmatrix_trans(H::pack_rn(pr[0] - f01.x, pr[1] - f01.y));
              const uint32_t bl1 = movmatrix_trans(H::pack_rn(pr[2] - f23.x, pr[3] - f23.y));
              // Scale pairs per group: tokens (tA, tB) -> sp0, (tC, tE) -> sp1.
              // Rows past the context may hold stale scale bits (p is 0 there,
              // but 0 * inf is not): their scales and zeros are masked to 0.
              // (one mask per B register: low half token tA / tC, high half tB / tE)
              const uint32_t mAB = (mA & 0xFFFFu) | (mB & 0xFFFF0000u);
              const uint32_t mCE = (mC & 0xFFFFu) | (mE & 0xFFFF0000u);
              uint32_t pb0[NG], pb1[NG];
#pragma unroll
              for (int half = 0; half < 2; ++half) {
                const int t0 = half ? tC : tA, t1 = half ? tE : tB;
                uint32_t s0[NG], s1[NG];
                if constexpr (D == 128) {
                  const uint4 a = ld_shared_v4(vsc + t0 * SR), c = ld_shared_v4(vsc + t1 * SR);
                  s0[0] = a.x; s0[1] = a.y; s0[2] = a.z; s0[3] = a.w;
                  s1[0] = c.x; s1[1] = c.y; s1[2] = c.z; s1[3] = c.w;
                } else {
                  const uint2 a = ld_shared_v2(vsc + t0 * SR), c = ld_shared_v2(vsc + t1 * SR);
                  s0[0] = a.x; s0[1] = a.y; s1[0] = c.x; s1[1] = c.y;
                }
#pragma unroll
                for (int g = 0; g < NG; ++g)
                  (half ? pb1 : pb0)[g] = __byte_perm(s0[g], s1[g], 0x5410);
              }
              // the zero-point product's A operand: column q4 of the scale rows of
              // tokens (tA, tB) and (tC, tE)
              uint32_t zr[2];
              if constexpr (D == 128) {
                ldmatrix_x2_trans(st + i4.kz + G::kScaleTileBytes, zr);
              } else {
                zr[0] = zr[1] = 0u;
                if (q4 < 2 * NG) {
                  zr[0] = __byte_perm(ld_shared_u16(vsc + tA * SR + 2 * q4),
                                      ld_shared_u16(vsc + tB * SR + 2 * q4), 0x5410);
                  zr[1] = __byte_perm(ld_shared_u16(vsc + tC * SR + 2 * q4),
                                      ld_shared_u16(vsc + tE * SR + 2 * q4), 0x5410);
                }
              }
              if (partial) {
#pragma unroll
                for (int g = 0; g < NG; ++g) { pb0[g] &= mAB; pb1[g] &= mCE; }
                zr[0] &= mAB;
                zr[1] &= mCE;
              }
              {
                const uint32_t za[4] = {zr[0], 0u, zr[1], 0u};
                mma_16816<PKV_F16>(zc, za, bp0, bp1);
                mma_16816<PKV_F16>(zc, za, bl0, bl1);
              }
              // codes: x = tokens (tA, tB), y = (tC, tE), 2 bytes each (d = 32 g + 4 q4 + 0..3)
              uint32_t xv[NG], yv[NG];
              {
                uint32_t r[4];
                ldmatrix_x4_trans(st + i4.v0, r);
                xv[0] = r[0]; yv[0] = r[1]; xv[1] = r[2]; yv[1] = r[3];
                if constexpr (D == 128) {
                  ldmatrix_x4_trans(st + i4.v1, r);
                  xv[2] = r[0]; yv[2] = r[1]; xv[3] = r[2]; yv[3] = r[3];
                }
              }
#pragma unroll
              for (int grp = 0; grp < NG; ++grp) {
                // P'_g = p * scale as an exact f16 hi + lo pair: hi = f16(p_hi s),
                // its rounding error p_hi s - hi by one fused multiply-add (exact),
                // lo = f16(p_lo s + that error)
                const uint32_t b0 = hmul2(bp0, pb0[grp]), b1 = hmul2(bp1, pb1[grp]);
                const uint32_t l0 = hfma2(bl0, pb0[grp], hfma2(bp0, pb0[grp], hneg2(b0)));
                const uint32_t l1 = hfma2(bl1, pb1[grp], hfma2(bp1, pb1[grp], hneg2(b1)));
                // rows q4 (even d) take n 2^-24, rows q4 + 8 (odd d) 16 n 2^-24
                const uint32_t x = xv[grp], y = yv[grp], xs = x >> 8, ys = y >> 8;
                const uint32_t a0[4] = {nib_lo(x), nib_hi(x), nib_lo(y), nib_hi(y)};
                mma_16816<PKV_F16>(oacc[2 * grp], a0, b0, b1);
                mma_16816<PKV_F16>(oacc[2 * grp], a0, l0, l1);
                const uint32_t a1[4] = {nib_lo(xs), nib_hi(xs), nib_lo(ys), nib_hi(ys)};
                mma_16816<PKV_F16>(oacc[2 * grp + 1], a1, b0, b1);
                mma_16816<PKV_F16>(oacc[2 * grp + 1], a1, l0, l1);
              }
            }
            }  // v_on
        }
      }

      __syncwarp();
      issue_next();
      s_cons = s_cons + 1 == G::kStages ? 0 : s_cons + 1;
    }

    // -------------------------------------------------------------- unit epilogue
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      lrow[0] += __shfl_xor_sync(0xffffffffu, lrow[0], o);
      lrow[1] += __shfl_xor_sync(0xffffffffu, lrow[1], o);
    }
    if constexpr (KV == PKV_INT8) {
      // codes entered as (x + 128) 2^-24: O = 2^24 acc - 128 sum_t P'_t
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        zp[0] += __shfl_xor_sync(0xffffffffu, zp[0], o);
        zp[1] += __shfl_xor_sync(0xffffffffu, zp[1], o);
      }
#pragma unroll
      for (int i = 0; i < MT; ++i) {
        oacc[i][0] = oacc[i][0] * 16777216.f - 128.f * zp[0];
        oacc[i][1] = oacc[i][1] * 16777216.f - 128.f * zp[1];
        oacc[i][2] = oacc[i][2] * 16777216.f - 128.f * zp[0];
        oacc[i][3] = oacc[i][3] * 16777216.f - 128.f * zp[1];
      }
    }
    // INT4 codes entered as n 2^-24 (rows q4 + 8, odd d: 16 n 2^-24)
    float post = (KV == PKV_INT4_G32) ? 16777216.f : 1.f / kPScale;
    if constexpr (is_blk8(KV)) post *= vref;
    const float post_odd = (KV == PKV_INT4_G32) ? 1048576.f : post;
#pragma unroll
    for (int i = 0; i < MT; ++i) {
      oacc[i][0] *= post; oacc[i][1] *= post;
      oacc[i][2] *= post_odd; oacc[i][3] *= post_odd;
    }
    if constexpr (KV == PKV_INT4_G32) {
      // zero-point sums: row 2g + 1 of the product (lane (2g + 1) * 4 + c4)
      // holds group g for this thread's heads 2c4, 2c4 + 1
#pragma unroll
      for (int g = 0; g < D / 32; ++g) {
        const float z0 = __shfl_sync(0xffffffffu, zc[0], (2 * g + 1) * 4 + c4);
        const float z1 = __shfl_sync(0xffffffffu, zc[1], (2 * g + 1) * 4 + c4);
        oacc[2 * g][0] += z0; oacc[2 * g][2] += z0;
        oacc[2 * g][1] += z1; oacc[2 * g][3] += z1;
        oacc[2 * g + 1][0] += z0; oacc[2 * g + 1][2] += z0;
        oacc[2 * g + 1][1] += z1; oacc[2 * g + 1][3] += z1;
      }
    }

    // merge the warps' states in registers (lane i of every warp holds the same
    // output positions), passing them through one buffer: 1 -> 0, 3 -> 2, 2 -> 0
    float* mb = mbuf + lane * G::kMbStride;
    auto put = [&]() {
#pragma unroll
      for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int k = 0; k < 4; ++k) mb[4 * i + k] = oacc[i][k];
      mb[4 * MT + 0] = mrow[0]; mb[4 * MT + 1] = mrow[1];
      mb[4 * MT + 2] = lrow[0]; mb[4 * MT + 3] = lrow[1];
    };
    auto take = [&]() { merge_state<MT>(mrow, lrow, oacc, mb + 4 * MT, mb + 4 * MT + 2, mb); };
    if constexpr (!WU) {
      if (warp == 1) put();
      __syncthreads();
      if (warp == 0) take();
      __syncthreads();
      if (warp == 3) put();
      __syncthreads();
      if (warp == 2) take();
      __syncthreads();
      if (warp == 2) put();
      __syncthreads();
      if (warp == 0) take();
    }
    if (WU || warp == 0) {
      const int64_t head0 = static_cast<int64_t>(unit.b) * p.num_q_heads + unit.kvh * group;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int g = 2 * c4 + h;
        int64_t head;
        float inv;
        if constexpr (PF) {
          // column g: query token j0 + g / G of the chunk, head g % G
          if (!col_q[h]) continue;
          head = (static_cast<int64_t>(p.q_start[unit.b]) + j0 + g / group) * p.num_q_heads +
                 unit.kvh * group + g % group;
          inv = (lrow[h] > 0.f && !col_zero[h]) ? 1.f / lrow[h] : 0.f;
        } else {
          if (g >= group) continue;
          head = head0 + g;
          inv = lrow[h] > 0.f ? 1.f / lrow[h] : 0.f;
        }
        // balanced split: slot (piece slot, head in the group), else (head, partition)
        const int64_t slot = BAL ? static_cast<int64_t>(unit.part) * group + g
                                 : head * p.num_partitions + unit.part;
#pragma unroll
        for (int i = 0; i < MT; ++i) {
          int d0;
          if constexpr (KV == PKV_INT4_G32) {
            d0 = 32 * (i >> 1) + 4 * q4 + 2 * (i & 1);
          } else if constexpr (is_blk8(KV) && D == 128) {
            d0 = 16 * (((q4 & 1) << 1) | ((q4 >> 1) & 1) | (q4 & 4)) + 2 * i;
          } else {
            d0 = (D == 128 ? 16 : 8) * q4 + 2 * i;
          }
          const float v0 = oacc[i][h] * inv, v1 = oacc[i][2 + h] * inv;
          if (!BAL && p.num_partitions == 1) {
            uint32_t* outp = reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.out) + head * D + d0);
            *outp = Half16<QT>::pack_rn(v0, v1);
          } else {
            *reinterpret_cast<float2*>(p.ws_out + slot * D + d0) = make_float2(v0, v1);
          }
        }
        if ((BAL || p.num_partitions > 1) && q4 == 0) {
          p.ws_ml[slot * 2] = mrow[h];
          p.ws_ml[slot * 2 + 1] = lrow[h];
        }
      }
    }
    if constexpr (!WU) __syncthreads();      // the buffer is free for the next unit
  }
  pdl_launch_dependents();
  cp_async_wait<0>();
}

}  // namespace
}  // namespace pkv
