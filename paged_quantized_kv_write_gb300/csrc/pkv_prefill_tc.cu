// Chunked-prefill attention on the fifth-generation tensor cores (tcgen05,
// accumulators in tensor memory) for one-byte caches (FP8 E4M3, FP8 E5M2,
// INT8) at head_dim 64 and 128: prefill_tc8_kernel.  (16-bit caches take the
// warp-role kernel of pkv_prefill_ws.cu.)  Chunked prefill is a dense
// contraction (every cached token meets a whole chunk of queries), unlike the
// decode step, so it runs where the dense tensor throughput is: "Optimizing
// KV-Cache Memory Footprint in High-Throughput LLM Serving", section 5, pairs
// PagedAttention with GQA and chunked prefill; query j of a chunk of n over c
// cached tokens sits at position c - n + j and sees tokens 0 .. c - n + j.
//
// One CTA (one warpgroup, 128 threads; two CTAs per SM) takes 128 query rows
// -- 128/G query tokens of one sequence times the G query heads of one KV
// head -- and walks that KV head's cache in 64-token tiles:
//   1. the tile's K and V codes come in through the block table and are
//      converted to f16 operands in shared memory, K as a K-major operand and
//      V as an MN-major one (token rows as they are stored);
//   2. S = Q K^T: eight tcgen05.mma (M 128, N 64, K 16) into tensor memory;
//   3. thread r reads row r of S from tensor memory, applies the causal mask
//      and the online softmax (running max raised lazily, by more than
//      2^8 only), and writes row r of P as a 16-bit hi + lo pair back into
//      tensor memory (two tokens per 32-bit column);
//   4. O += P V: eight tcgen05.mma (M 128, N = head_dim, K 16) into tensor
//      memory, hi then lo, with P read from tensor memory as the A operand;
// and finally reads O from tensor memory, divides by the row sums and writes
// the output rows.  The other operands sit in shared memory in the canonical
// layouts without swizzle, built from 8 x 16-byte core matrices: K-major
// (Q, K) with the next core matrix along K 128 bytes on (leading byte
// offset) and the next 8-row group further (stride byte offset); MN-major (V)
// with 8 tokens x 8 head_dim values per core matrix, the next token group 128
// bytes on and the next 8 head_dim values 1024 bytes on.  Every wait for the
// tensor cores is bounded: when one runs out the launch ORs
// PKV_ERR_DEVICE_TIMEOUT into dev_status, stops, and still frees its tensor
// memory.
#include <math.h>
#include <stdlib.h>
#include <stdint.h>

#include "pagedkv.h"
#include "pkv_common.cuh"
#include "pkv_internal.h"
#include "pkv_tcgen05.cuh"

namespace pkv {
namespace {
using namespace tc;

constexpr int kTcThreads = 128;      // one warpgroup; thread r owns query row r
constexpr int kTcRows = 128;         // MMA M
constexpr int kTcKv = 64;            // KV tokens per tile
constexpr float kTcTau = 8.f;        // lazy rescale threshold (log2 units)

// Shared-memory plans (bytes; operand tiles 1024-byte aligned) and tensor
// memory (S: columns [0, 64); O: [64, 64 + D)) for head_dim D.
template <int D> struct TcPlan {
  // S [0, 64), O [64, 64 + D), P hi and lo [64 + D, 128 + D)
  static constexpr uint32_t kTmemCols = 256;
  static constexpr int kQBytes = kTcRows * D * 2;
  static constexpr int kKBytes = kTcKv * D * 2;
  static constexpr int kVBytes = kTcKv * D * 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  // Q, K, one V tile, the per-token scales of two tiles (by tile parity: K
  // scales, V scales, V max per half-tile), barriers
  static constexpr int kSc8Floats = 2 * kTcKv + 8;
  static constexpr int kOffV8 = kOffK + kKBytes;
  static constexpr int kOffS8 = kOffV8 + kVBytes;
  static constexpr int kOffBar8 = kOffS8 + 2 * kSc8Floats * 4;
  static constexpr int kSmem8 = kOffBar8 + 32;
  static_assert(2 * (kSmem8 + 1024) <= 233472, "two CTAs per SM");
};

struct TcParams {
  const uint16_t* q;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* q_start;
  const float* scales;        // one-byte caches: fp32 [2][num_blocks][num_kv_heads]
  int max_query_len;          // queries j >= max_query_len of a chunk are not computed
  void* out;
  int* dev_status;
  int max_blocks_per_seq;
  int num_blocks;
  int num_q_heads;
  int num_kv_heads;
  int block_size;
  float softmax_scale;
};

// ----------------------------------------------------------------------------
// One-byte caches (FP8 E4M3, FP8 E5M2, INT8; one fp32 scale per block and KV
// head).  The tiles and tensor-core steps of the file's header, with f16
// operands:
//   * the codes of the next tile are fetched into registers one tile ahead
//     (16-byte loads through the block table) and converted exactly to f16
//     into the K-major K tile and the MN-major V tile (E4M3 and E5M2 by cvt,
//     INT8 as 1024 + (x + 128) - 1152 in f16);
//   * q in bf16 enters as f16 with a power-of-two scale per row (exact for
//     every value above 2^-28 of the row's largest), taken off in the softmax
//     multiplier;
//   * a token's K block scale multiplies its score column; its V block scale
//     multiplies its column of P, in units of a running reference scale vu
//     (the largest V scale seen so far): P'' = p s_V / vu <= 2^8.  When a tile
//     raises vu, O and the row sum (kept in the same units) are rescaled, and
//     the output O / l is free of vu;
//   * P'' goes to tensor memory as a hi + lo pair, and the softmax works
//     on packed fp32 pairs (two scores per fma / add / mul / sub).
template <int KV, int QT, int D>
__global__ void __launch_bounds__(kTcThreads, 2) prefill_tc8_kernel(const TcParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  using PL = TcPlan<D>;
  pdl_wait();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int group = p.num_q_heads / p.num_kv_heads;
  const int qpb = kTcRows / group;
  const int nq = p.q_start[b + 1] - p.q_start[b];
  const int nqc = min(nq, p.max_query_len);            // queries computed
  const int j0 = static_cast<int>(blockIdx.x) * qpb;
  if (j0 >= nqc) return;
  const int cap = p.max_blocks_per_seq * p.block_size;
  int ctx = p.context_lens[b];
  if (ctx > cap) {
    if (tid == 0 && blockIdx.x == 0 && kvh == 0) flag_status(p.dev_status, PKV_ERR_DEVICE_BOUNDS);
    ctx = cap;
  }
  const int pos0 = ctx - nq;
  if (pos0 < 0 && j0 == 0 && tid == 0 && kvh == 0) flag_status(p.dev_status, PKV_ERR_DEVICE_BOUNDS);
  const int jj = tid / group, g = tid % group;
  const bool row_q = j0 + jj < nqc;
  const int pos = pos0 + j0 + jj;
  const bool row_ok = row_q && pos >= 0;
  const int last_j = min(j0 + qpb, nqc) - 1;
  const int kv_end = max(0, min(ctx, pos0 + last_j + 1));
  const int ntiles = (kv_end + kTcKv - 1) / kTcKv;

  const uint32_t sb = smem_u32(smem);
  const uint32_t bar_s = sb + PL::kOffBar8, bar_o = sb + PL::kOffBar8 + 8;
  volatile uint32_t* tslot = reinterpret_cast<volatile uint32_t*>(smem + PL::kOffBar8 + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + PL::kOffBar8 + 20);
  float* scb = reinterpret_cast<float*>(smem + PL::kOffS8);   // [2][PL::kSc8Floats]

  if (warp == 0) {
    tmem_alloc(sb + PL::kOffBar8 + 16, PL::kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    mbar_init_fence();
    *abort_flag = 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tmem_s = tmem, tmem_o = tmem + 64, tmem_p = tmem + 64 + D;
  const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;

  // Q row tid as f16 (bf16 q: times 2^qe, the row's largest magnitude in [2^13, 2^14))
  int qe = 0;
  {
    const uint16_t* qrow =
        p.q + ((static_cast<int64_t>(p.q_start[b]) + j0 + (row_q ? jj : 0)) * p.num_q_heads +
               kvh * group + g) * D;
    if constexpr (QT == PKV_F16) {
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint32_t dst = sb + PL::kOffQ + core_off(tid, c, D / 8);
        if (row_ok) cp_async_16(dst, qrow + 8 * c);
        else st_shared_v4(dst, make_uint4(0, 0, 0, 0));
      }
      cp_async_commit();
    } else {
      float amax = 0.f;
      if (row_ok) {
#pragma unroll 4
        for (int c = 0; c < D / 8; ++c) {
          const uint4 v = ld_global_nc_v4(qrow + 8 * c);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i)
            amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[i] << 16)),
                                     fabsf(__uint_as_float(w[i] & 0xFFFF0000u))));
        }
      }
      if (amax > 0.f && amax <= 3.0e38f) {
        int ex;
        frexpf(amax, &ex);                             // amax = f 2^ex, f in [0.5, 1)
        qe = 14 - ex;
      }
#pragma unroll 4
      for (int c = 0; c < D / 8; ++c) {
        uint4 o = make_uint4(0, 0, 0, 0);
        if (row_ok) {
          const uint4 v = ld_global_nc_v4(qrow + 8 * c);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
          uint32_t h[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            h[i] = Half16<PKV_F16>::pack_rn(ldexpf(__uint_as_float(w[i] << 16), qe),
                                            ldexpf(__uint_as_float(w[i] & 0xFFFF0000u), qe));
          o = make_uint4(h[0], h[1], h[2], h[3]);
        }
        st_shared_v4(sb + PL::kOffQ + core_off(tid, c, D / 8), o);
      }
    }
  }

  const float mult = ldexpf(p.softmax_scale * 1.4426950408889634f, -qe);
  constexpr uint32_t kIdescS = umma_idesc(false, kTcRows, kTcKv, false);
  constexpr uint32_t kIdescO = umma_idesc(false, kTcRows, D, true);
  float m = -INFINITY, l = 0.f;                       // l in units of 1 / vu
  float vu = 1.f, lg_vu = 0.f;                         // V reference scale (1 until one is seen) and its log2
  bool vu_set = false;
  bool failed = false;
  int s_commits = 0, o_commits = 0;
  const int32_t* trow = p.block_tables + static_cast<int64_t>(b) * p.max_blocks_per_seq;
  const int64_t per_kv = static_cast<int64_t>(p.num_blocks) * p.num_kv_heads;

  // this thread's share of a tile: item tid + 128 j (j < D / 32) is 16-byte
  // code chunk (item >> 3) % (D / 16) of token 8 ((item >> 3) / (D / 16)) + (tid & 7)
  constexpr int kRc = D / 16, kNj = D / 32;
  const int lr = tid & 7, lrc = (tid >> 3) % kRc;
  auto tgroup = [&](int j) { return ((tid >> 3) + 16 * j) / kRc; };
  uint4 kraw[4], vraw[4];
  auto fetch = [&](int t) {
#pragma unroll
    for (int j = 0; j < kNj; ++j) {
      const int abs_t = t * kTcKv + 8 * tgroup(j) + lr;
      kraw[j] = make_uint4(0, 0, 0, 0);
      vraw[j] = make_uint4(0, 0, 0, 0);
      if (abs_t < kv_end) {
        const int logical = abs_t / p.block_size;
        const int phys = __ldg(trow + logical);
        if (phys >= 0 && phys < p.num_blocks) {
          const int64_t row = (static_cast<int64_t>(phys) * p.num_kv_heads + kvh) * p.block_size +
                              (abs_t - logical * p.block_size);
          kraw[j] = ld_global_nc_v4(p.k_cache + row * D + lrc * 16);
          vraw[j] = ld_global_nc_v4(p.v_cache + row * D + lrc * 16);
        } else if (lrc == 0) {
          flag_status(p.dev_status, PKV_ERR_DEVICE_BOUNDS);
        }
      }
    }
  };
  // threads 0-63: the K and V scales of token tid of tile t (0 past the range;
  // for a token in an out-of-range block, which takes no part, a K scale of
  // NaN and a V scale of 0), and per warp the largest V scale and whether
  // any of its tokens is in an out-of-range block
  auto put_scales = [&](int t) {
    if (tid < kTcKv) {
      const int abs_t = t * kTcKv + tid;
      float ks = 0.f, vs = 0.f;
      bool bad = false;
      if (abs_t < kv_end) {
        const int phys = __ldg(trow + abs_t / p.block_size);
        if (phys >= 0 && phys < p.num_blocks) {
          const int64_t idx = static_cast<int64_t>(phys) * p.num_kv_heads + kvh;
          ks = __ldg(p.scales + idx);
          vs = __ldg(p.scales + per_kv + idx);
        } else {
          ks = __int_as_float(0x7fc00000);
          bad = true;
        }
      }
      float* sc = scb + (t & 1) * PL::kSc8Floats;
      sc[tid] = ks;
      sc[kTcKv + tid] = vs;
      float vm = vs;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, o));
      const bool any_bad = __any_sync(0xffffffffu, bad);
      if (lane == 0) {
        sc[2 * kTcKv + warp] = vm;
        sc[2 * kTcKv + 2 + warp] = any_bad ? 1.f : 0.f;
      }
    }
  };
  // codes in registers -> f16 operand tile (K: K-major; V: MN-major)
  auto convert = [&](const uint4 (&raw)[4], bool is_v) {
    const uint32_t base = sb + (is_v ? PL::kOffV8 : PL::kOffK) + (lr << 4);
#pragma unroll
    for (int j = 0; j < kNj; ++j) {
      const int tb = tgroup(j);
      uint4 lo, hi;
      codes16_to_f16<KV>(raw[j], lo, hi);
      const int c0 = 2 * lrc, c1 = 2 * lrc + 1;
      const uint32_t o0 = is_v ? ((c0 * (kTcKv / 8) + tb) << 7) : ((tb * (D / 8) + c0) << 7);
      const uint32_t o1 = is_v ? ((c1 * (kTcKv / 8) + tb) << 7) : ((tb * (D / 8) + c1) << 7);
      st_shared_v4(base + o0, lo);
      st_shared_v4(base + o1, hi);
    }
  };
  if (ntiles > 0) {
    fetch(0);
    put_scales(0);
  }
  if constexpr (QT == PKV_F16) cp_async_wait<0>();

  for (int t = 0; t < ntiles; ++t) {
    const int t0 = t * kTcKv;
    // 1. K(t) into its operand tile (the previous S has finished with it)
    convert(kraw, false);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) { failed = true; break; }
    // 2. S = Q K^T
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        umma(tmem_s, umma_desc(sb + PL::kOffQ + kk * 256, 128, (D / 8) * 128),
             umma_desc(sb + PL::kOffK + kk * 256, 128, (D / 8) * 128), kIdescS, kk > 0);
      umma_commit(bar_s);
    }
    ++s_commits;
    // 3. the previous P V has finished with O, P and the V tile: V(t) goes in,
    //    and the next tile's codes and scales are requested
    if (t > 0 && !mbar_wait(bar_o, (t - 1) & 1)) {
      flag_status(p.dev_status, PKV_ERR_DEVICE_TIMEOUT);
      *abort_flag = 1;
    }
    tc_fence_after();
    convert(vraw, true);
    if (t + 1 < ntiles) {
      fetch(t + 1);
      put_scales(t + 1);
    }
    if (!mbar_wait(bar_s, t & 1)) {
      flag_status(p.dev_status, PKV_ERR_DEVICE_TIMEOUT);
      *abort_flag = 1;
    }
    tc_fence_after();
    // 4. row tid of S times each column's K scale
    const float* sc = scb + (t & 1) * PL::kSc8Floats;
    float s[kTcKv];
    {
      float a[32];
      tmem_ld32(tmem_s + lane_base, a);
#pragma unroll
      for (int i = 0; i < 32; ++i) s[i] = a[i];
      tmem_ld32(tmem_s + lane_base + 32, a);
#pragma unroll
      for (int i = 0; i < 32; ++i) s[32 + i] = a[i];
    }
#pragma unroll
    for (int c4 = 0; c4 < kTcKv / 4; ++c4) {
      const float4 ks = *reinterpret_cast<const float4*>(sc + 4 * c4);
      const float2 a = f2_unpack(f2_mul(f2_pack(s[4 * c4], s[4 * c4 + 1]), f2_pack(ks.x, ks.y)));
      const float2 c = f2_unpack(f2_mul(f2_pack(s[4 * c4 + 2], s[4 * c4 + 3]), f2_pack(ks.z, ks.w)));
      s[4 * c4] = a.x;
      s[4 * c4 + 1] = a.y;
      s[4 * c4 + 2] = c.x;
      s[4 * c4 + 3] = c.y;
    }
    const bool bad_tile = sc[2 * kTcKv + 2] != 0.f || sc[2 * kTcKv + 3] != 0.f;
    const bool full = t0 + kTcKv <= kv_end && t0 + kTcKv - 1 <= pos0 + j0 && !bad_tile;
    float tmax, pmul;
    if (full) {
      float e;
      if (mult >= 0.f) {
        e = -INFINITY;
#pragma unroll
        for (int c = 0; c < kTcKv; ++c) e = fmaxf(e, s[c]);
      } else {
        e = INFINITY;
#pragma unroll
        for (int c = 0; c < kTcKv; ++c) e = fminf(e, s[c]);
      }
      tmax = e * mult;
      pmul = mult;
    } else {
      tmax = -INFINITY;
#pragma unroll
      for (int c = 0; c < kTcKv; ++c) {
        const int abs_t = t0 + c;
        const bool valid = abs_t < kv_end && (!row_ok || abs_t <= pos) && sc[c] == sc[c];
        s[c] = valid ? s[c] * mult : -INFINITY;
        tmax = fmaxf(tmax, s[c]);
      }
      pmul = 1.f;
    }
    // 5. online softmax (lazy max) and the V reference (same in every thread)
    const bool raise = tmax > m + kTcTau;
    float alpha = 1.f;
    if (raise) {
      const float mn = fmaxf(m, tmax);
      alpha = ex2_ftz(m - mn);
      m = mn;
    }
    const float vmax = fmaxf(sc[2 * kTcKv], sc[2 * kTcKv + 1]);
    const bool rebase = vmax > (vu_set ? vu : 0.f);
    if (rebase) {
      alpha *= vu_set ? vu / vmax : 1.f / vmax;
      vu = vmax;
      lg_vu = __log2f(vmax);
      vu_set = true;
    }
    l *= alpha;
    if (t > 0 && (__any_sync(0xffffffffu, raise) || rebase)) {
#pragma unroll
      for (int k = 0; k < D / 32; ++k) {
        float o[32];
        tmem_ld32(tmem_o + lane_base + 32 * k, o);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] *= alpha;
        tmem_st32(tmem_o + lane_base + 32 * k, o);
      }
    }
    // P / vu = 2^(x - m - log2 vu); P'' = (P / vu) s_V as an f16 hi + lo pair
    const float moff = m + lg_vu;
    // (score pairs as packed fp32: one fused multiply-add, one add to the
    // pair of row-sum halves, one multiply and one subtraction per two scores)
    const uint64_t pm2 = f2_pack(pmul, pmul), nm2 = f2_pack(-moff, -moff);
    uint64_t l2 = f2_pack(0.f, 0.f);
#pragma unroll
    for (int c8 = 0; c8 < kTcKv / 8; ++c8) {
      const float4 va = *reinterpret_cast<const float4*>(sc + kTcKv + 8 * c8);
      const float4 vb = *reinterpret_cast<const float4*>(sc + kTcKv + 8 * c8 + 4);
      const float vsc[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 x = f2_unpack(f2_fma(f2_pack(s[8 * c8 + 2 * k], s[8 * c8 + 2 * k + 1]), pm2, nm2));
        const uint64_t pp = f2_pack(ex2_ftz(x.x), ex2_ftz(x.y));
        l2 = f2_add(l2, pp);
        const uint64_t qq = f2_mul(pp, f2_pack(vsc[2 * k], vsc[2 * k + 1]));
        const float2 q = f2_unpack(qq);
        hw[k] = Half16<PKV_F16>::pack_rn(q.x, q.y);
        const float2 f = Half16<PKV_F16>::unpack(hw[k]);
        const float2 d = f2_unpack(f2_sub(qq, f2_pack(f.x, f.y)));
        lw[k] = Half16<PKV_F16>::pack_rn(d.x, d.y);
      }
      tmem_st4(tmem_p + lane_base + 4 * c8, hw[0], hw[1], hw[2], hw[3]);
      tmem_st4(tmem_p + lane_base + kTcKv / 2 + 4 * c8, lw[0], lw[1], lw[2], lw[3]);
    }
    {
      const float2 lh = f2_unpack(l2);
      l += lh.x + lh.y;
    }
    tmem_store_wait();
    fence_proxy_async_smem();                          // the V tile's converted rows
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) { failed = true; break; }
    // 6. O += P'' V (hi, then lo)
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kTcKv / 16; ++kk)
        umma_ts(tmem_o, tmem_p + kk * 8, umma_desc(sb + PL::kOffV8 + kk * 256, 128, (kTcKv / 8) * 128),
                kIdescO, t > 0 || kk > 0);
#pragma unroll
      for (int kk = 0; kk < kTcKv / 16; ++kk)
        umma_ts(tmem_o, tmem_p + kTcKv / 2 + kk * 8,
                umma_desc(sb + PL::kOffV8 + kk * 256, 128, (kTcKv / 8) * 128), kIdescO, 1u);
      umma_commit(bar_o);
    }
    ++o_commits;
  }

  if (o_commits > 0 && !mbar_wait(bar_o, (o_commits - 1) & 1)) {
    flag_status(p.dev_status, PKV_ERR_DEVICE_TIMEOUT);
    failed = true;
  }
  if (s_commits > 0 && !mbar_wait(bar_s, (s_commits - 1) & 1)) {
    flag_status(p.dev_status, PKV_ERR_DEVICE_TIMEOUT);
    failed = true;
  }
  tc_fence_after();
  const bool all_ok = __syncthreads_and(!failed) != 0;
  uint16_t* orow = static_cast<uint16_t*>(p.out) +
                   ((static_cast<int64_t>(p.q_start[b]) + j0 + jj) * p.num_q_heads + kvh * group + g) * D;
  if (row_q && !(all_ok && ntiles > 0)) {
    for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = make_uint4(0, 0, 0, 0);
  }
  if (all_ok && ntiles > 0) {
    const float inv = (row_ok && l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
    for (int k = 0; k < D / 32; ++k) {
      float o[32];
      tmem_ld32(tmem_o + lane_base + 32 * k, o);       // warp-collective: every row
      if (row_q) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint4 w;
          w.x = Half16<QT>::pack_rn(o[8 * c] * inv, o[8 * c + 1] * inv);
          w.y = Half16<QT>::pack_rn(o[8 * c + 2] * inv, o[8 * c + 3] * inv);
          w.z = Half16<QT>::pack_rn(o[8 * c + 4] * inv, o[8 * c + 5] * inv);
          w.w = Half16<QT>::pack_rn(o[8 * c + 6] * inv, o[8 * c + 7] * inv);
          reinterpret_cast<uint4*>(orow + 32 * k)[c] = w;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, PL::kTmemCols);
  pdl_launch_dependents();
}

template <typename Kern>
cudaError_t launch_tc(Kern kern, int smem_bytes, const PrefillArgs& a, cudaStream_t st) {
  TcParams p;
  p.q = static_cast<const uint16_t*>(a.q);
  p.k_cache = static_cast<const uint8_t*>(a.k_cache);
  p.v_cache = static_cast<const uint8_t*>(a.v_cache);
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.q_start = a.q_start;
  p.scales = static_cast<const float*>(a.scales);
  p.out = a.out;
  p.dev_status = a.dev_status;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_blocks = a.num_blocks;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.block_size = a.block_size;
  p.softmax_scale = a.softmax_scale;
  p.max_query_len = a.max_query_len;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  const int group = a.num_q_heads / a.num_kv_heads;
  const int qpb = kTcRows / group;
  const dim3 grid(static_cast<unsigned>((a.max_query_len + qpb - 1) / qpb),
                  static_cast<unsigned>(a.num_kv_heads), static_cast<unsigned>(a.num_seqs));
  return launch_pdl(kern, grid, dim3(kTcThreads), smem_bytes, st, p);
}

template <int KV, int D>
cudaError_t launch_tc8(const PrefillArgs& a, cudaStream_t st) {
  constexpr int kSmem = TcPlan<D>::kSmem8;
  return a.q_dtype == PKV_F16 ? launch_tc(prefill_tc8_kernel<KV, PKV_F16, D>, kSmem, a, st)
                              : launch_tc(prefill_tc8_kernel<KV, PKV_BF16, D>, kSmem, a, st);
}

template <int D>
cudaError_t launch_tc_d(const PrefillArgs& a, cudaStream_t st) {
  switch (a.kv_dtype) {
    case PKV_FP8_E4M3: return launch_tc8<PKV_FP8_E4M3, D>(a, st);
    case PKV_FP8_E5M2: return launch_tc8<PKV_FP8_E5M2, D>(a, st);
    case PKV_INT8: return launch_tc8<PKV_INT8, D>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool prefill_tc_supported(const PrefillArgs& a) {
  return is_blk8(a.kv_dtype) && (a.head_dim == 64 || a.head_dim == 128);
}

cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t st) {
  if (a.num_seqs == 0 || a.max_query_len == 0) return cudaSuccess;
  return a.head_dim == 64 ? launch_tc_d<64>(a, st) : launch_tc_d<128>(a, st);
}

}  // namespace pkv
