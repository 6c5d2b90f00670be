// paged_decode_attention: decode-phase PagedAttention (the kernel is in
// pkv_attn.cuh) plus the log-sum-exp merge of split-KV partitions, the launch
// configuration and the partition-size heuristic.
#include "pkv_attn.cuh"

namespace pkv {
namespace {

// Merge the partitions of one (sequence, q head): M = max m_p,
// L = sum l_p 2^(m_p - M), out = sum l_p 2^(m_p - M) O_p / L.
template <int QT, int D>
__global__ void __launch_bounds__(D)
pkv_lse_reduce(const Params p) {
  pdl_wait();                                      // the partials of the decode kernel
  const int64_t head = blockIdx.x;                 // b * Hq + h
  const int b = static_cast<int>(head / p.num_q_heads);
  const int d = threadIdx.x;
  const int ctx = min(p.context_lens[b], p.max_blocks_per_seq * p.block_size);
  const int np = max(1, (ctx + p.partition_size - 1) / p.partition_size);
  const float* ml = p.ws_ml + head * p.num_partitions * 2;
  const float* o = p.ws_out + head * p.num_partitions * D;
  float M = -INFINITY;
  for (int i = 0; i < np; ++i) M = fmaxf(M, ml[2 * i]);
  float L = 0.f, acc = 0.f;
  if (M != -INFINITY) {
    for (int i = 0; i < np; ++i) {
      const float m = ml[2 * i];
      if (m == -INFINITY) continue;
      const float w = ml[2 * i + 1] * exp2f(m - M);
      L += w;
      acc += w * o[i * D + d];
    }
  }
  const float val = L > 0.f ? acc / L : 0.f;
  uint16_t* outp = static_cast<uint16_t*>(p.out);
  if constexpr (QT == PKV_F16) {
    outp[head * D + d] = __half_as_ushort(__float2half_rn(val));
  } else {
    outp[head * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(val));
  }
}

template <int KV, int QT, int D, bool WU>
cudaError_t launch_mode(const DecodeArgs& a, cudaStream_t st) {
  using G = Geo<KV, D>;
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
  auto kern = paged_decode_kernel<KV, QT, D, WU>;
  // per device, once: the shared-memory opt-in and the resident CTAs per SM
  static std::atomic<int> slots_per_dev[kMaxDevices];     // SMs x resident CTAs (0: unknown)
  p.parts_per_cta = 1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int slots = slots_per_dev[dev].load(std::memory_order_relaxed);
  if (slots == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::kSmemBytes);
    if (e != cudaSuccess) return e;
    int occ = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kDecodeWarps * kWarp,
                                                      G::kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    slots = max(1, occ) * max(1, sms);
    slots_per_dev[dev].store(slots, std::memory_order_relaxed);
  }
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
  return launch_pdl(pkv_lse_reduce<QT, D>, dim3(a.num_seqs * a.num_q_heads), dim3(D), 0, st, p);
}

// Warp-owned units when the split-KV work has enough (partition, sequence, KV
// head) units for several waves of warps (PKV_WU_WAVES x SMs x 16 warps);
// shared partitions otherwise.
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
  // results); =simt runs the CUDA-core comparator instead (16-bit, FP8 and
  // INT8 caches without the fused write; other calls keep the tensor path)
  if (const char* m = getenv("PKV_DECODE_MODE")) {
    if (!strcmp(m, "shared")) wu = false;
    if (!strcmp(m, "warp")) wu = true;
    if (!strcmp(m, "simt") && KV != PKV_INT4_G32 && a.slot_mapping == nullptr)
      return launch_simt(a, st);
    if (!strcmp(m, "tc") && decode_tc_supported(a)) return launch_decode_tc(a, st);
  }
  return wu ? launch_mode<KV, QT, D, true>(a, st) : launch_mode<KV, QT, D, false>(a, st);
}

template <int KV, int QT>
cudaError_t launch_d(const DecodeArgs& a, cudaStream_t st) {
  return a.head_dim == 64 ? launch_typed<KV, QT, 64>(a, st) : launch_typed<KV, QT, 128>(a, st);
}

}  // namespace

// the log-sum-exp merge of a split-KV call's partitions (also used by the
// SIMT comparator)
cudaError_t launch_lse_reduce(const DecodeArgs& a, cudaStream_t st) {
  Params p = {};
  p.context_lens = a.context_lens;
  p.out = a.out;
  p.ws_out = a.ws_out;
  p.ws_ml = a.ws_ml;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_q_heads = a.num_q_heads;
  p.block_size = a.block_size;
  p.partition_size = a.partition_size;
  p.num_partitions = a.num_partitions;
  const dim3 grid(a.num_seqs * a.num_q_heads);
  if (a.q_dtype == PKV_F16) {
    return a.head_dim == 64 ? launch_pdl(pkv_lse_reduce<PKV_F16, 64>, grid, dim3(64), 0, st, p)
                            : launch_pdl(pkv_lse_reduce<PKV_F16, 128>, grid, dim3(128), 0, st, p);
  }
  return a.head_dim == 64 ? launch_pdl(pkv_lse_reduce<PKV_BF16, 64>, grid, dim3(64), 0, st, p)
                          : launch_pdl(pkv_lse_reduce<PKV_BF16, 128>, grid, dim3(128), 0, st, p);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
  if (a.num_seqs == 0) return cudaSuccess;
  switch (a.kv_dtype) {
    case PKV_F16: return launch_d<PKV_F16, PKV_F16>(a, st);
    case PKV_BF16: return launch_d<PKV_BF16, PKV_BF16>(a, st);
    case PKV_FP8_E4M3:
      return a.q_dtype == PKV_F16 ? launch_d<PKV_FP8_E4M3, PKV_F16>(a, st)
                                  : launch_d<PKV_FP8_E4M3, PKV_BF16>(a, st);
    case PKV_FP8_E5M2:
      return a.q_dtype == PKV_F16 ? launch_d<PKV_FP8_E5M2, PKV_F16>(a, st)
                                  : launch_d<PKV_FP8_E5M2, PKV_BF16>(a, st);
    case PKV_INT8:
      return a.q_dtype == PKV_F16 ? launch_d<PKV_INT8, PKV_F16>(a, st)
                                  : launch_d<PKV_INT8, PKV_BF16>(a, st);
    default:
      return a.q_dtype == PKV_F16 ? launch_d<PKV_INT4_G32, PKV_F16>(a, st)
                                  : launch_d<PKV_INT4_G32, PKV_BF16>(a, st);
  }
}

int resolve_partition_size(int num_seqs, int num_q_heads, int num_kv_heads,
                           int max_blocks_per_seq, int block_size, int requested) {
  if (requested > 0) return ((requested + kTile - 1) / kTile) * kTile;
  // Measured on GB300: grids with enough units for warp-owned units run best
  // with 512-token partitions, shared-partition grids with 1024 (fewer merges);
  // few (sequence, KV head) pairs need short partitions to fill 152 SMs.
  // The unit threshold below is the one the launch uses for 152 SMs.
  const int64_t max_ctx = static_cast<int64_t>(max_blocks_per_seq) * block_size;
  const int64_t pairs = static_cast<int64_t>(num_seqs) * num_kv_heads;
  const int64_t wu_units = static_cast<int64_t>(PKV_WU_WAVES) * 152 * 16;
  int part;
  if (pairs * ((max_ctx + 511) / 512) >= wu_units)
    part = 512;
  else if (pairs * ((max_ctx + 1023) / 1024) >= 4 * 152)
    part = 1024;
  else if (pairs * ((max_ctx + 511) / 512) >= 2 * 152)
    part = 512;
  else
    part = 256;
  if (max_ctx <= part) part = static_cast<int>(((max_ctx + kTile - 1) / kTile) * kTile);
  if (part <= 0) part = kTile;
  (void)num_q_heads;
  return part;
}

}  // namespace pkv
