// Decode-phase PagedAttention for one-byte caches (FP8 E4M3, FP8 E5M2, INT8;
// one fp32 scale per block and KV head) with head_dim 128 on the
// fifth-generation tensor cores, accumulators in tensor memory: the
// dequantized tiles feed the tensor cores from shared memory, and the
// softmax runs with one thread per token.  It computes what
// paged_decode_kernel (the mma.sync kernel) computes and is kept as a
// comparator (PKV_DECODE_MODE=tc) in the test build (libpagedkv_test.so,
// compiled with PKV_TEST_HOOKS) only, never chosen by the library: on GB300 it
// runs about 2.7x slower, because each CTA works through one serial chain
// per tile (row lookup, code loads, conversion, S, softmax vote, P V) and
// only three such chains fit on an SM, against twelve independent copy rings
// per SM in the mma.sync kernel.
//
// The computation is the one "KV Cache Compression & Paged Attention"
// (myaihardware.com, section "Implementation Details") describes for the
// kernel: walk the sequence's logical blocks, translate each through the
// block table, and attend over the dequantized K and V of each block; the
// block-wise scales are those of "Reducing LLM Inference Latency: KV Cache
// Quantization and PagedAttention in vLLM" (section "Block-Wise Scaling
// Factors").  Long contexts are split into partitions whose partial results
// the log-sum-exp merge combines.
//
// One CTA (one warpgroup, 128 threads, three CTAs per SM) takes one unit:
// partition `part` of sequence b, KV head kvh.  It walks the unit in tiles of
// 128 tokens; thread t owns token t of a tile (tensor-memory lane t of S^T)
// and head_dim row t of O^T:
//   1. the codes of the next tile are fetched into registers one tile ahead
//      (16-byte loads, 64 contiguous bytes per row and instruction, row
//      addresses through the block table) and converted exactly to f16 into
//      the K tile (K-major: rows = tokens) and the V tile (MN-major A
//      operand of O^T: rows = head_dim);
//   2. S^T = K Q^T: eight tcgen05.mma (M 128 tokens, N 16: the G <= 8 query
//      heads, the other 8 columns unused, K 16) into tensor memory;
//   3. thread t takes row t of S^T, scales it by its block's K scale, and runs
//      the online softmax with a running max per head that is shared by the
//      whole CTA and raised lazily (a barrier vote; the per-head maximum is
//      reduced only when some score passes the running max by more than 2^8);
//   4. P'' = p s_V / s_ref (s_ref: the largest V scale of the unit's blocks)
//      goes to shared memory as an f16 hi + lo pair in the K-major layout of
//      the B operand P^T (rows = heads);
//   5. O^T += V^T P^T: 2 x 8 tcgen05.mma (M 128 head_dim rows, N 16, K 16).
// At the end thread t divides row t of O^T by the per-head sums and writes
// the output (one partition) or the partition's normalised partial result
// and its (max, sum) for the merge.  Every wait on the tensor cores is
// bounded (PKV_ERR_DEVICE_TIMEOUT, outputs zero, tensor memory freed).
#include "pkv_attn.cuh"
#include "pkv_tcgen05.cuh"

namespace pkv {
namespace {
using namespace tc;

constexpr int kDtThreads = 128;
constexpr int kDtTok = 128;                 // tokens per tile (MMA M of S^T)
constexpr int kDtD = 128;                   // head_dim (MMA M of O^T)
constexpr int kDtN = 16;                    // MMA N: query heads, zero-padded
constexpr int kDtH = 8;                     // query heads held per thread (G <= 8)
constexpr uint32_t kDtTmemCols = 32;        // S^T: columns [0, 16); O^T: [16, 32)
constexpr float kDtTau = 8.f;

// shared memory (bytes): K and V f16 tiles, Q (8 head rows; the MMA's rows
// 8-15 alias them through a zero stride offset and feed only unused
// columns), P^T hi and lo (likewise), then reduction scratch and barriers
constexpr int kDtKBytes = kDtTok * kDtD * 2;          // 32 KiB
constexpr int kDtVBytes = kDtTok * kDtD * 2;          // 32 KiB
constexpr int kDtQBytes = kDtH * kDtD * 2;            // 2 KiB
constexpr int kDtPBytes = kDtH * kDtTok * 2;          // 2 KiB each
constexpr int kDtOffK = 0;
constexpr int kDtOffV = kDtOffK + kDtKBytes;
constexpr int kDtOffQ = kDtOffV + kDtVBytes;
constexpr int kDtOffPh = kDtOffQ + kDtQBytes;
constexpr int kDtOffPl = kDtOffPh + kDtPBytes;
constexpr int kDtOffRed = kDtOffPl + kDtPBytes;       // float [4 warps][8 heads]
constexpr int kDtOffQe = kDtOffRed + 4 * kDtH * 4;    // int [8]: q row exponents
constexpr int kDtOffBar = kDtOffQe + kDtH * 4;        // 2 mbarriers, tmem address, abort flag
constexpr int kDtSmem = kDtOffBar + 32;
static_assert(3 * (kDtSmem + 1024) <= 233472, "three CTAs per SM");

__device__ __forceinline__ uint4 ld_global_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

template <int KV, int QT>
__global__ void __launch_bounds__(kDtThreads, 3) decode_tc_kernel(const Params p) {
  extern __shared__ __align__(1024) uint8_t dtc_smem[];
  uint8_t* smem = dtc_smem;
  pdl_wait();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int part = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int group = p.num_q_heads / p.num_kv_heads;
  const int cap = p.max_blocks_per_seq * p.block_size;
  int ctx = p.context_lens[b];
  if (ctx > cap) {
    if (tid == 0 && part == 0 && kvh == 0) flag_status(p.dev_status, PKV_ERR_DEVICE_BOUNDS);
    ctx = cap;
  }
  const int nparts_seq = ctx > 0 ? (ctx + p.partition_size - 1) / p.partition_size : 1;
  if (part >= nparts_seq) return;                     // the whole CTA: past this sequence
  const Unit unit = make_unit<kDtTok>(p, b, kvh, ctx, part);
  const int ntiles = unit.ntiles;

  // the new token first (the CTA holding the sequence's last partition)
  if (p.slot_mapping != nullptr && part == nparts_seq - 1) {
    if (warp == 0) fused_write<KV, QT, kDtD>(p, b, kvh, ctx, lane);
    __syncthreads();
  }

  const uint32_t sb = smem_u32(smem);
  const uint32_t bar_s = sb + kDtOffBar, bar_o = sb + kDtOffBar + 8;
  volatile uint32_t* tslot = reinterpret_cast<volatile uint32_t*>(smem + kDtOffBar + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kDtOffBar + 20);
  float* red = reinterpret_cast<float*>(smem + kDtOffRed);
  int* qe_sm = reinterpret_cast<int*>(smem + kDtOffQe);
  const int64_t per_kv = static_cast<int64_t>(p.num_blocks) * p.num_kv_heads;
  const float* scales = static_cast<const float*>(p.scales);
  const int32_t* trow = p.block_tables + static_cast<int64_t>(b) * p.max_blocks_per_seq;

  if (warp == 0) {
    tmem_alloc(sb + kDtOffBar + 16, kDtTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    mbar_init_fence();
    *abort_flag = 0;
  }

  // Q: thread (h = tid / 16, chunk c = tid % 16) takes 8 values of head h; a
  // bf16 q enters as f16 times 2^qe_h (the row's largest magnitude in
  // [2^13, 2^14)), an f16 q as it is; heads past G are zero
  {
    const int h = tid >> 4, c = tid & 15;
    const bool hok = h < group;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (hok) v = ld_global_nc_v4(p.q + (static_cast<int64_t>(b) * p.num_q_heads + kvh * group + h) * kDtD + 8 * c);
    int qe = 0;
    uint4 o = v;
    if constexpr (QT == PKV_BF16) {
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[i] << 16)), fabsf(__uint_as_float(w[i] & 0xFFFF0000u))));
#pragma unroll
      for (int o2 = 8; o2 > 0; o2 >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o2));
      if (amax > 0.f && amax <= 3.0e38f) {
        int ex;
        frexpf(amax, &ex);
        qe = 14 - ex;
      }
      uint32_t hh[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        hh[i] = Half16<PKV_F16>::pack_rn(ldexpf(__uint_as_float(w[i] << 16), qe),
                                         ldexpf(__uint_as_float(w[i] & 0xFFFF0000u), qe));
      o = make_uint4(hh[0], hh[1], hh[2], hh[3]);
    }
    st_shared_v4(sb + kDtOffQ + core_off(h, c, kDtD / 8), o);
    if (c == 0) qe_sm[h] = qe;
  }
  // the unit's V reference scale: the largest V scale of its blocks
  {
    const int blk0 = unit.tok_begin / p.block_size;
    const int nblk = unit.tok_end > unit.tok_begin ? (unit.tok_end - 1) / p.block_size - blk0 + 1 : 0;
    float vm = 0.f;
    for (int j = tid; j < nblk; j += kDtThreads) {
      const int phys = __ldg(trow + blk0 + j);
      if (phys >= 0 && phys < p.num_blocks) vm = fmaxf(vm, scales[per_kv + static_cast<int64_t>(phys) * p.num_kv_heads + kvh]);
    }
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, o2));
    if (lane == 0) red[warp] = vm;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tmem_s = tmem, tmem_o = tmem + kDtN;
  const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
  const float vref = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  const float inv_vref = vref > 0.f ? 1.f / vref : 0.f;
  float mult[kDtH];
#pragma unroll
  for (int h = 0; h < kDtH; ++h) mult[h] = ldexpf(p.softmax_scale * 1.4426950408889634f, -qe_sm[h]);
  __syncthreads();                                    // red[] is reused below

  constexpr uint32_t kIdescS = umma_idesc(false, kDtTok, kDtN, false);
  // O^T: A = V^T MN-major (bit 15), B = P^T K-major
  constexpr uint32_t kIdescO = umma_idesc(false, kDtD, kDtN, false) | (1u << 15);

  // this thread's loads: rows 8 (i / 2) + (lane & 7) of the warp's 32 tokens,
  // 16-byte chunk 4 (i & 1) + (lane >> 3), i = 0..7
  const int lk = lane & 7, lj = lane >> 3;
  uint4 kraw[8], vraw[8];
  float ks_next = 0.f, vs_next = 0.f;
  bool ok_next = false;
  // the row's byte offset in a cache tensor (or -1) for token t of tile i
  auto token_row = [&](int i, int t, float& ks, float& vs) -> int64_t {
    const int abs_t = unit.tok_begin + i * kDtTok + t;
    ks = 0.f;
    vs = 0.f;
    if (abs_t >= unit.tok_end) return -1;
    const int logical = abs_t / p.block_size;
    const int phys = __ldg(trow + logical);
    if (phys < 0 || phys >= p.num_blocks) {
      flag_status(p.dev_status, PKV_ERR_DEVICE_BOUNDS);
      return -1;
    }
    const int64_t bh = static_cast<int64_t>(phys) * p.num_kv_heads + kvh;
    ks = scales[bh];
    vs = scales[per_kv + bh];
    return (bh * p.block_size + (abs_t - logical * p.block_size)) * kDtD;
  };
  auto fetch = [&](int i) {
    const int64_t my = token_row(i, tid, ks_next, vs_next);
    ok_next = my >= 0;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int src_lane = 8 * (r >> 1) + lk;
      const int64_t off = __shfl_sync(0xffffffffu, my, src_lane);
      const int c = 4 * (r & 1) + lj;
      if (off >= 0) {
        kraw[r] = ld_global_v4(p.k_cache + off + 16 * c);
        vraw[r] = ld_global_v4(p.v_cache + off + 16 * c);
      } else {
        kraw[r] = make_uint4(0, 0, 0, 0);
        vraw[r] = make_uint4(0, 0, 0, 0);
      }
    }
  };
  // codes -> f16 tiles.  Load r of this thread: token 32 warp + 8 (r / 2) + lk,
  // raw chunk c = 4 (r & 1) + lj -> f16 chunks 2c, 2c + 1.
  auto convert_k = [&]() {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int tok = 32 * warp + 8 * (r >> 1) + lk, c = 4 * (r & 1) + lj;
      uint4 lo, hi;
      codes16_to_f16<KV>(kraw[r], lo, hi);
      st_shared_v4(sb + kDtOffK + core_off(tok, 2 * c, kDtD / 8), lo);
      st_shared_v4(sb + kDtOffK + core_off(tok, 2 * c + 1, kDtD / 8), hi);
    }
  };
  auto convert_v = [&]() {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int tok = 32 * warp + 8 * (r >> 1) + lk, c = 4 * (r & 1) + lj;
      uint4 lo, hi;
      codes16_to_f16<KV>(vraw[r], lo, hi);
      // MN-major: head_dim group m (8 values) of token group tok / 8 at
      // (m * 16 + tok / 8) * 128, token tok % 8 at 16 (tok % 8)
      const uint32_t base = sb + kDtOffV + ((tok & 7) << 4);
      st_shared_v4(base + (((2 * c) * (kDtTok / 8) + (tok >> 3)) << 7), lo);
      st_shared_v4(base + (((2 * c + 1) * (kDtTok / 8) + (tok >> 3)) << 7), hi);
    }
  };

  float m[kDtH], l[kDtH];
#pragma unroll
  for (int h = 0; h < kDtH; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
  }
  bool failed = false;
  int s_commits = 0, o_commits = 0;
  if (ntiles > 0) fetch(0);

  for (int i = 0; i < ntiles; ++i) {
    const float ks = ks_next, vs = vs_next;
    const bool tok_ok = ok_next;
    // 1. K(i) into its tile (the previous S^T has finished with it)
    convert_k();
    // 2. the previous P V has finished with the V tile, P and O: V(i) in
    if (i > 0 && !mbar_wait(bar_o, (i - 1) & 1)) {
      flag_status(p.dev_status, PKV_ERR_DEVICE_TIMEOUT);
      *abort_flag = 1;
    }
    tc_fence_after();
    convert_v();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) { failed = true; break; }
    // 3. S^T = K Q^T (Q rows 8-15 alias rows 0-7: zero stride offset)
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kDtD / 16; ++kk)
        umma(tmem_s, umma_desc(sb + kDtOffK + kk * 256, 128, (kDtD / 8) * 128),
             umma_desc(sb + kDtOffQ + kk * 256, 128, 0), kIdescS, kk > 0);
      umma_commit(bar_s);
    }
    ++s_commits;
    // 4. the next tile's codes, while the tensor cores work
    if (i + 1 < ntiles) fetch(i + 1);
    if (!mbar_wait(bar_s, i & 1)) {
      flag_status(p.dev_status, PKV_ERR_DEVICE_TIMEOUT);
      *abort_flag = 1;
    }
    tc_fence_after();
    float x[kDtH];
    tmem_ld8(tmem_s + lane_base, x);
    const float kf = tok_ok ? ks : 0.f;
#pragma unroll
    for (int h = 0; h < kDtH; ++h) x[h] = (tok_ok && h < group) ? x[h] * kf * mult[h] : -INFINITY;
    // 5. lazy running max per head, shared by the CTA
    bool over = false;
#pragma unroll
    for (int h = 0; h < kDtH; ++h) over |= x[h] > m[h] + kDtTau;
    if (__syncthreads_or(over)) {
      float tm[kDtH];
#pragma unroll
      for (int h = 0; h < kDtH; ++h) {
        tm[h] = x[h];
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) tm[h] = fmaxf(tm[h], __shfl_xor_sync(0xffffffffu, tm[h], o2));
      }
      if (lane == 0) {
#pragma unroll
        for (int h = 0; h < kDtH; ++h) red[warp * kDtH + h] = tm[h];
      }
      __syncthreads();
      float alpha[kDtH];
#pragma unroll
      for (int h = 0; h < kDtH; ++h) {
        const float t4 = fmaxf(fmaxf(red[h], red[kDtH + h]), fmaxf(red[2 * kDtH + h], red[3 * kDtH + h]));
        const float mn = fmaxf(m[h], t4);
        alpha[h] = mn == -INFINITY ? 1.f : ex2_ftz(m[h] - mn);
        m[h] = mn;
        l[h] *= alpha[h];
      }
      __syncthreads();                                 // red[] is free again
      if (i > 0) {                                     // row tid of O^T (O is stable: step 2)
        float o[8];
        tmem_ld8(tmem_o + lane_base, o);
#pragma unroll
        for (int h = 0; h < kDtH; ++h) o[h] *= alpha[h];
        tmem_st8(tmem_o + lane_base, o);
      }
    }
    // 6. P'' = p s_V / s_ref as an f16 hi + lo pair, column tid of P^T
    const float vf = vs * inv_vref;
    const uint32_t pcol = ((tid >> 3) << 7) + ((tid & 7) << 1);
#pragma unroll
    for (int h = 0; h < kDtH; ++h) {
      // (a head with no score yet, or past G, has m = -inf: p = 0)
      const float pr = m[h] == -INFINITY ? 0.f : ex2_ftz(x[h] - m[h]);
      l[h] += pr;
      const float q2 = pr * vf;
      const __half hi = __float2half_rn(q2);
      const __half lo = __float2half_rn(q2 - __half2float(hi));
      st_shared_u16(sb + kDtOffPh + pcol + (h << 4), __half_as_ushort(hi));
      st_shared_u16(sb + kDtOffPl + pcol + (h << 4), __half_as_ushort(lo));
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) { failed = true; break; }
    // 7. O^T += V^T P^T (hi, then lo); V^T is MN-major: the next 16 tokens
    //    256 bytes on, the next 8 head_dim rows (kDtTok / 8) * 128 bytes on
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kDtTok / 16; ++kk)
        umma(tmem_o, umma_desc(sb + kDtOffV + kk * 256, 128, (kDtTok / 8) * 128),
             umma_desc(sb + kDtOffPh + kk * 256, 128, 0), kIdescO, i > 0 || kk > 0);
#pragma unroll
      for (int kk = 0; kk < kDtTok / 16; ++kk)
        umma(tmem_o, umma_desc(sb + kDtOffV + kk * 256, 128, (kDtTok / 8) * 128),
             umma_desc(sb + kDtOffPl + kk * 256, 128, 0), kIdescO, 1u);
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
  // per-head sums over the CTA's tokens
#pragma unroll
  for (int h = 0; h < kDtH; ++h) {
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) l[h] += __shfl_xor_sync(0xffffffffu, l[h], o2);
  }
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < kDtH; ++h) red[warp * kDtH + h] = l[h];
  }
  const bool all_ok = __syncthreads_and(!failed) != 0;
  float ltot[kDtH];
#pragma unroll
  for (int h = 0; h < kDtH; ++h) ltot[h] = red[h] + red[kDtH + h] + red[2 * kDtH + h] + red[3 * kDtH + h];
  float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (all_ok && ntiles > 0) tmem_ld8(tmem_o + lane_base, o);   // warp-collective
  const int d = tid;
  const int64_t head0 = static_cast<int64_t>(b) * p.num_q_heads + kvh * group;
#pragma unroll
  for (int h = 0; h < kDtH; ++h) {
    if (h >= group) break;
    const bool live = all_ok && ntiles > 0 && ltot[h] > 0.f;
    const float val = live ? o[h] * vref / ltot[h] : 0.f;
    const int64_t head = head0 + h;
    if (p.num_partitions == 1) {
      static_cast<uint16_t*>(p.out)[head * kDtD + d] =
          QT == PKV_F16 ? __half_as_ushort(__float2half_rn(val))
                        : __bfloat16_as_ushort(__float2bfloat16_rn(val));
    } else {
      const int64_t slot = head * p.num_partitions + unit.part;
      p.ws_out[slot * kDtD + d] = val;
      if (d == 0) {
        p.ws_ml[slot * 2] = live ? m[h] : -INFINITY;
        p.ws_ml[slot * 2 + 1] = live ? ltot[h] : 0.f;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kDtTmemCols);
  pdl_launch_dependents();
}

template <int KV, int QT>
cudaError_t launch_tc_typed(const DecodeArgs& a, cudaStream_t st) {
  Params p = {};
  p.q = static_cast<const uint16_t*>(a.q);
  p.k_cache = static_cast<uint8_t*>(const_cast<void*>(a.k_cache));
  p.v_cache = static_cast<uint8_t*>(const_cast<void*>(a.v_cache));
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.scales = const_cast<void*>(a.scales);
  p.k_new = static_cast<const uint16_t*>(a.k_new);
  p.v_new = static_cast<const uint16_t*>(a.v_new);
  p.slot_mapping = a.slot_mapping;
  p.out = a.out;
  p.ws_out = a.ws_out;
  p.ws_ml = a.ws_ml;
  p.dev_status = a.dev_status;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_seqs = a.num_seqs;
  p.num_blocks = a.num_blocks;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.block_size = a.block_size;
  p.partition_size = a.partition_size;
  p.num_partitions = a.num_partitions;
  p.softmax_scale = a.softmax_scale;
  p.parts_per_cta = 1;
  auto kern = decode_tc_kernel<KV, QT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kDtSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(a.num_partitions), static_cast<unsigned>(a.num_kv_heads),
                  static_cast<unsigned>(a.num_seqs));
  e = launch_pdl(kern, grid, dim3(kDtThreads), kDtSmem, st, p);
  if (e != cudaSuccess || a.num_partitions == 1) return e;
  return launch_lse_reduce(a, st);
}

template <int KV>
cudaError_t launch_tc_kv(const DecodeArgs& a, cudaStream_t st) {
  return a.q_dtype == PKV_F16 ? launch_tc_typed<KV, PKV_F16>(a, st) : launch_tc_typed<KV, PKV_BF16>(a, st);
}

}  // namespace

bool decode_tc_supported(const DecodeArgs& a) {
  return is_blk8(a.kv_dtype) && a.head_dim == kDtD && a.num_q_heads / a.num_kv_heads <= kDtH;
}

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t st) {
  switch (a.kv_dtype) {
    case PKV_FP8_E4M3: return launch_tc_kv<PKV_FP8_E4M3>(a, st);
    case PKV_FP8_E5M2: return launch_tc_kv<PKV_FP8_E5M2>(a, st);
    case PKV_INT8: return launch_tc_kv<PKV_INT8>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
