// Launch side of the decode kernel (pkv_attn.cuh) and the log-sum-exp merge
// of split-KV partitions: launch configuration, work split and partitions per
// CTA.  Included by one translation unit per cache-dtype family
// (pkv_decode_half.cu, pkv_decode_byte.cu, pkv_decode_int4.cu) so they
// compile in parallel; pkv_decode.cu dispatches between them.
#pragma once

#include "pkv_attn.cuh"

namespace pkv {
namespace {

// One lane's EPT values of row i of a partial output, i < np.
template <int EPT>
__device__ __forceinline__ void load_partial(const float* src, float (&v)[EPT]) {
  if constexpr (EPT == 4) {
    const float4 x = __ldcg(reinterpret_cast<const float4*>(src));
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  } else {
    const float2 x = __ldcg(reinterpret_cast<const float2*>(src));
    v[0] = x.x; v[1] = x.y;
  }
}

// Log-sum-exp merge of np partial states: state i is (m_i, l_i) at
// ml + ml_step * i and its normalised output row at o + o_step * i (this
// lane's EPT values).  The warp takes the chunks of 32 states from base0 in
// steps of bstride; acc = sum_i l_i 2^(m_i - M) O_i and L = this lane's share
// of sum_i l_i 2^(m_i - M), M the largest m_i of all np states.  The first
// chunk's states and its first kPre rows are loaded together, before M is
// known, so that the merge waits for one round of loads rather than three.
template <int EPT, int kPre, int kStep>
__device__ __forceinline__ void merge_states(const float* ml, int64_t ml_step, const float* o,
                                             int64_t o_step, int np, int base0, int bstride,
                                             int lane, float (&acc)[EPT], float& L) {
  const int i0 = base0 + lane;
  float2 st0 = make_float2(-INFINITY, 0.f);
  if (i0 < np) st0 = __ldcg(reinterpret_cast<const float2*>(ml + ml_step * i0));
  float v0[kPre][EPT];
#pragma unroll
  for (int u = 0; u < kPre; ++u)
    if (base0 + u < np) load_partial<EPT>(o + static_cast<int64_t>(base0 + u) * o_step, v0[u]);
  float M = -INFINITY;
  for (int i = lane; i < np; i += kWarp) M = fmaxf(M, i == i0 ? st0.x : __ldcg(ml + ml_step * i));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
#pragma unroll
  for (int e = 0; e < EPT; ++e) acc[e] = 0.f;
  L = 0.f;
  if (M == -INFINITY) return;
  for (int base = base0; base < np; base += bstride) {
    float2 st = st0;
    if (base != base0) {
      const int i = base + lane;
      st = i < np ? __ldcg(reinterpret_cast<const float2*>(ml + ml_step * i))
                  : make_float2(-INFINITY, 0.f);
    }
    const float wgt = st.x == -INFINITY ? 0.f : st.y * exp2f(st.x - M);
    L += wgt;
    const int n = min(kWarp, np - base);
    int j = 0;
    if (base == base0) {
#pragma unroll
      for (int u = 0; u < kPre; ++u) {
        const float wj = __shfl_sync(0xffffffffu, wgt, u);
        if (u < n) {
#pragma unroll
          for (int e = 0; e < EPT; ++e) acc[e] = fmaf(wj, v0[u][e], acc[e]);
        }
      }
      j = kPre;
    }
    for (; j < n; j += kStep) {
      float v[kStep][EPT];
#pragma unroll
      for (int u = 0; u < kStep; ++u)
        if (j + u < n) load_partial<EPT>(o + static_cast<int64_t>(base + j + u) * o_step, v[u]);
#pragma unroll
      for (int u = 0; u < kStep; ++u) {
        const float wj = __shfl_sync(0xffffffffu, wgt, (j + u) & 31);
        if (j + u < n) {
#pragma unroll
          for (int e = 0; e < EPT; ++e) acc[e] = fmaf(wj, v[u][e], acc[e]);
        }
      }
    }
  }
}

// Merge the partitions of one (sequence, q head): M = max m_p,
// L = sum l_p 2^(m_p - M), out = sum l_p 2^(m_p - M) O_p / L.
//
// One CTA per (sequence, q head) with W warps.  Lane l of every warp keeps
// head_dim values [EPT l, EPT l + EPT) of the sum.  The partitions are taken
// in blocks of 32: lane j computes the weight of partition 32k + j of its
// warp's block k, the warp then walks the block with eight independent
// 16-byte (8-byte at head_dim 64) loads in flight per lane, each weight
// handed out by a shuffle; the W warps' sums meet in shared memory.
template <int QT, int D, int W>
__global__ void __launch_bounds__(32 * W)
pkv_lse_reduce(const Params p) {
  constexpr int EPT = D / kWarp;                   // 4 (D = 128) or 2 (D = 64)
  __shared__ float s_acc[W][D];
  __shared__ float s_l[W];
  pdl_wait();                                      // the partials of the decode kernel
  const int64_t head = blockIdx.x;                 // b * Hq + h
  const int b = static_cast<int>(head / p.num_q_heads);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ctx = min(p.context_lens[b], p.max_blocks_per_seq * p.block_size);
  const int np = max(1, (ctx + p.partition_size - 1) / p.partition_size);
  const float* ml = p.ws_ml + head * p.num_partitions * 2;
  const float* o = p.ws_out + head * p.num_partitions * D + EPT * lane;
  constexpr int64_t ml_step = 2, o_step = D;
  float acc[EPT];
  float L;
  merge_states<EPT, 8, 8>(ml, ml_step, o, o_step, np, warp * kWarp, W * kWarp, lane, acc, L);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  if constexpr (W > 1) {
#pragma unroll
    for (int e = 0; e < EPT; ++e) s_acc[warp][EPT * lane + e] = acc[e];
    if (lane == 0) s_l[warp] = L;
    __syncthreads();
    if (warp != 0) return;
#pragma unroll
    for (int w = 1; w < W; ++w) {
#pragma unroll
      for (int e = 0; e < EPT; ++e) acc[e] += s_acc[w][EPT * lane + e];
      L += s_l[w];
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  uint16_t* outp = static_cast<uint16_t*>(p.out) + head * D + EPT * lane;
  if constexpr (EPT == 4) {
    *reinterpret_cast<uint2*>(outp) = make_uint2(Half16<QT>::pack_rn(acc[0] * inv, acc[1] * inv),
                                                 Half16<QT>::pack_rn(acc[2] * inv, acc[3] * inv));
  } else {
    *reinterpret_cast<uint32_t*>(outp) = Half16<QT>::pack_rn(acc[0] * inv, acc[1] * inv);
  }
}

// The merge of the balanced split: one CTA per (sequence, KV head) pair, warp
// g merging query head g of the group.  The pair's tile range and the warps
// that hold its pieces come from the tile prefix, which the CTA computes from
// context_lens (a CTA-wide scan) before it waits for the decode kernel, so
// that this chain overlaps the decode kernel's end; then each warp merges its
// head's pieces (slots w + pair, see bal_unit) as pkv_lse_reduce does.
template <int QT, int D, int kTok>
__global__ void __launch_bounds__(8 * kWarp, 4)
pkv_bal_merge(const Params p) {
  constexpr int EPT = D / kWarp;
  __shared__ int s_before[8], s_all[8];            // per warp: tiles before sequence b, in all
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthreads = blockDim.x, nwarps = nthreads / kWarp;
  const int hkv = p.num_kv_heads, group = p.num_q_heads / hkv;
  const int b = static_cast<int>(blockIdx.x) / hkv, kvh = static_cast<int>(blockIdx.x) - b * hkv;
  const int cap = p.max_blocks_per_seq * p.block_size;
  auto tiles_of = [&](int bb) -> int {
    const int c = min(p.context_lens[bb], cap);
    return c > 0 ? (c + kTok - 1) / kTok : 0;
  };
  int before = 0, all = 0;
  for (int bb = tid; bb < p.num_seqs; bb += nthreads) {
    const int t = tiles_of(bb);
    all += t;
    if (bb < b) before += t;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, o);
    all += __shfl_xor_sync(0xffffffffu, all, o);
  }
  if (lane == 0) {
    s_before[warp] = before;
    s_all[warp] = all;
  }
  __syncthreads();
  before = 0;
  all = 0;
  for (int w = 0; w < nwarps; ++w) {
    before += s_before[w];
    all += s_all[w];
  }
  const int nt = tiles_of(b);
  const int t0 = before * hkv + kvh * nt;          // the pair's first tile in the list
  const int64_t T = static_cast<int64_t>(all) * hkv;
  pdl_wait();                                      // the pieces of the decode kernel
  if (warp >= group) return;
  const int pair = b * hkv + kvh;
  int np = 0, first = 0;
  if (nt > 0) {
    const int64_t Wn = p.bal_warps;
    const int w0 = static_cast<int>((static_cast<int64_t>(t0 + 1) * Wn - 1) / T);
    const int w1 = static_cast<int>((static_cast<int64_t>(t0 + nt) * Wn - 1) / T);
    np = w1 - w0 + 1;
    first = w0 + pair;
  } else if (kvh == 0 && warp == 0 && lane == 0 && p.slot_mapping != nullptr &&
             p.slot_mapping[b] != -1) {
    // a sequence without tokens has no slot to write (as the other splits flag it)
    flag_status(p.dev_status, PKV_ERR_DEVICE_BOUNDS);
  }
  const int g = warp;
  const float* ml = p.ws_ml + (static_cast<int64_t>(first) * group + g) * 2;
  const float* o = p.ws_out + (static_cast<int64_t>(first) * group + g) * D + EPT * lane;
  const int64_t ml_step = 2 * group, o_step = static_cast<int64_t>(group) * D;
  float acc[EPT];
  float L;
  merge_states<EPT, 4, 4>(ml, ml_step, o, o_step, np, 0, kWarp, lane, acc, L);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const int64_t head = static_cast<int64_t>(b) * p.num_q_heads + kvh * group + g;
  uint16_t* outp = static_cast<uint16_t*>(p.out) + head * D + EPT * lane;
  if constexpr (EPT == 4) {
    *reinterpret_cast<uint2*>(outp) = make_uint2(Half16<QT>::pack_rn(acc[0] * inv, acc[1] * inv),
                                                 Half16<QT>::pack_rn(acc[2] * inv, acc[3] * inv));
  } else {
    *reinterpret_cast<uint32_t*>(outp) = Half16<QT>::pack_rn(acc[0] * inv, acc[1] * inv);
  }
}

// the merge for a call's partition count: warps per (sequence, q head)
template <int QT, int D>
cudaError_t launch_lse_typed(const Params& p, int num_heads, cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>(num_heads));
  if (p.num_partitions <= 32) return launch_pdl(pkv_lse_reduce<QT, D, 1>, grid, dim3(32), 0, st, p);
  if (p.num_partitions <= 64) return launch_pdl(pkv_lse_reduce<QT, D, 2>, grid, dim3(64), 0, st, p);
  return launch_pdl(pkv_lse_reduce<QT, D, 4>, grid, dim3(128), 0, st, p);
}

inline Params params_of(const DecodeArgs& a) {
  Params p;
  p.q = static_cast<const uint16_t*>(a.q);
  // the caches are written only by the fused write (a.slot_mapping set), which
  // the C ABI allows only for caller-writable buffers
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
  p.q_start = nullptr;
  p.max_query_len = 0;
  p.parts_per_cta = 1;
  p.bal_warps = 0;
  return p;
}

// SMs x resident CTAs of `kern` on the current device (looked up once per
// device, with the shared-memory opt-in set on the way)
template <typename K>
cudaError_t kernel_slots(K kern, size_t smem, std::atomic<int>* slots_per_dev, int* slots) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  *slots = slots_per_dev[dev].load(std::memory_order_relaxed);
  if (*slots == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int occ = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kDecodeWarps * kWarp, smem);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    *slots = max(1, occ) * max(1, sms);
    slots_per_dev[dev].store(*slots, std::memory_order_relaxed);
  }
  return cudaSuccess;
}

// The balanced split: one resident wave of CTAs (at most kBalMaxWarps warps),
// each warp an equal share of all pairs' tiles, then the merge of the pieces.
template <int KV, int QT, int D>
cudaError_t launch_bal(const DecodeArgs& a, cudaStream_t st) {
  using G = Geo<KV, D>;
  Params p = params_of(a);
  auto kern = paged_decode_kernel<KV, QT, D, true, false, true>;
  static std::atomic<int> slots_per_dev[kMaxDevices];
  int slots = 0;
  cudaError_t e = kernel_slots(kern, G::kSmemBytes, slots_per_dev, &slots);
  if (e != cudaSuccess) return e;
  const int ctas = std::min(slots, kBalMaxWarps / kDecodeWarps);
  p.bal_warps = ctas * kDecodeWarps;
  const BalLayout L = bal_layout(a.num_seqs, a.num_q_heads, a.num_kv_heads, a.head_dim);
  uint8_t* base = static_cast<uint8_t*>(a.ws_base);
  p.ws_out = reinterpret_cast<float*>(base);
  p.ws_ml = reinterpret_cast<float*>(base + L.ml_off);
  e = launch_pdl(kern, dim3(ctas), dim3(kDecodeWarps * kWarp), G::kSmemBytes, st, p);
  if (e != cudaSuccess) return e;
  // one CTA per (sequence, KV head), a warp per query head of the group (at
  // least 4 warps, which the prefix scan needs)
  const int group = a.num_q_heads / a.num_kv_heads;
  return launch_pdl(pkv_bal_merge<QT, D, G::kTileTok>,
                    dim3(static_cast<unsigned>(a.num_seqs * a.num_kv_heads)),
                    dim3(kWarp * std::max(4, group)), 0, st, p);
}

template <int KV, int QT, int D, bool WU>
cudaError_t launch_mode(const DecodeArgs& a, cudaStream_t st) {
  using G = Geo<KV, D>;
  Params p = params_of(a);
  auto kern = paged_decode_kernel<KV, QT, D, WU>;
  // per device, once: the shared-memory opt-in and the resident CTAs per SM
  static std::atomic<int> slots_per_dev[kMaxDevices];     // SMs x resident CTAs (0: unknown)
  int slots = 0;
  cudaError_t e = kernel_slots(kern, G::kSmemBytes, slots_per_dev, &slots);
  if (e != cudaSuccess) return e;
  // partitions per CTA (per warp with WU): runs of up to PKV_RUN_TOKENS tokens
  // per warp stream, as long as the grid keeps at least four waves of CTAs
  const int heads_per_cta = WU ? kDecodeWarps : 1;
  const int64_t head_groups = (a.num_kv_heads + heads_per_cta - 1) / heads_per_cta;
  int ppc = PKV_PPC;
  if (ppc <= 0) {
    ppc = 1;
    const int64_t groups = static_cast<int64_t>(a.num_seqs) * head_groups;
    const int run = WU ? PKV_RUN_TOKENS_WU : PKV_RUN_TOKENS;
    while (ppc * 2 * a.partition_size <= run && ppc * 2 <= a.num_partitions &&
           ((a.num_partitions + ppc * 2 - 1) / (ppc * 2)) * groups >= 4 * static_cast<int64_t>(slots))
      ppc *= 2;
  }
  ppc = std::max(1, std::min(ppc, a.num_partitions));
  p.parts_per_cta = ppc;
  dim3 grid((a.num_partitions + ppc - 1) / ppc, static_cast<unsigned>(head_groups), a.num_seqs);
  e = launch_pdl(kern, grid, dim3(kDecodeWarps * kWarp), G::kSmemBytes, st, p);
  if (e != cudaSuccess || a.num_partitions == 1) return e;
  return launch_lse_typed<QT, D>(p, a.num_seqs * a.num_q_heads, st);
}

// Warp-owned units when the split-KV work has enough (partition, sequence, KV
// head) units for several waves of warps (PKV_WU_WAVES x SMs x 16 warps), in
// the balanced split when the call allows it; shared partitions otherwise.
template <int KV, int QT, int D>
cudaError_t launch_typed(const DecodeArgs& a, cudaStream_t st) {
  static std::atomic<int> sms_per_dev[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int sms = sms_per_dev[dev].load(std::memory_order_relaxed);
  if (sms == 0) {
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    sms_per_dev[dev].store(sms, std::memory_order_relaxed);
  }
  const int64_t units = static_cast<int64_t>(a.num_partitions) * a.num_seqs * a.num_kv_heads;
  bool wu = a.num_partitions > 1 && units >= static_cast<int64_t>(PKV_WU_WAVES) * sms * 16;
  // PKV_DECODE_MODE=shared|warp overrides the choice (both give the same
  // results).  The test build also takes =simt, the CUDA-core comparator
  // (16-bit, FP8 and INT8 caches without the fused write; other calls keep
  // the tensor path), and =tc, the tcgen05 comparator for one-byte caches.
  // Where warp-owned units would be chosen, the balanced split takes the work
  // instead when it can (measured on GB300: config 4 198.6 -> 184.3 us,
  // config 5 188.4 -> 184.3, config 3 110.5 -> 108.5 for the attention call).
  const bool bal_ok = a.ws_base != nullptr &&
                      bal_eligible(a.num_seqs, a.num_kv_heads, a.max_blocks_per_seq,
                                   a.block_size, a.num_partitions);
  bool bal = wu && bal_ok;
  if (const char* m = getenv("PKV_DECODE_MODE")) {
    // shared / warp: the partitioned splits (shared or warp-owned partitions);
    // balanced: the balanced split wherever it can run
    if (!strcmp(m, "shared")) wu = bal = false;
    if (!strcmp(m, "warp")) { wu = true; bal = false; }
    if (!strcmp(m, "balanced")) bal = bal_ok;
#ifdef PKV_TEST_HOOKS
    if (!strcmp(m, "simt") && KV != PKV_INT4_G32 && a.slot_mapping == nullptr)
      return launch_simt(a, st);
    if (!strcmp(m, "tc") && decode_tc_supported(a)) return launch_decode_tc(a, st);
#endif
  }
  if (bal) return launch_bal<KV, QT, D>(a, st);
  return wu ? launch_mode<KV, QT, D, true>(a, st) : launch_mode<KV, QT, D, false>(a, st);
}

template <int KV, int QT>
cudaError_t launch_d(const DecodeArgs& a, cudaStream_t st) {
  return a.head_dim == 64 ? launch_typed<KV, QT, 64>(a, st) : launch_typed<KV, QT, 128>(a, st);
}

}  // namespace
}  // namespace pkv
