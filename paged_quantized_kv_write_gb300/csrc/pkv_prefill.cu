// paged_prefill_attention: chunked-prefill PagedAttention.  A chunk of new
// query tokens per sequence (already written to the cache) attends causally
// over everything in the cache up to each query's own position -- the
// multi-token counterpart of the decode step.  "Optimizing KV-Cache Memory
// Footprint in High-Throughput LLM Serving", section 5 (Production Benchmarks
// & Implementation), pairs PagedAttention with GQA and chunked prefill; the
// causal rule is the usual one for prefill (query j of a chunk of n over a
// context of c tokens sits at position c - n + j and sees tokens 0..c - n + j).
//
// Two kernels compute it.  16-bit and one-byte caches go to the warp-role
// tcgen05 kernel of pkv_prefill_ws.cu (two 128-row Q tiles per CTA against
// 128-token tiles, accumulators in tensor memory; one-byte codes converted to
// f16 operands by its load warps).  INT4 caches, or any call under
// PKV_PREFILL_MODE=mma, run the
// decode kernel of pkv_attn.cuh in its PF mode: a warp's 8 score columns are
// 8/G query tokens times the G query heads of one KV head, each column masked
// at its query's position; the warp streams the cache from token 0 to its
// last query's position through the same copy ring, dequantization and online
// softmax as a decode step.
#include "pkv_attn.cuh"

namespace pkv {
namespace {

template <int KV, int QT, int D>
cudaError_t launch_prefill_t(const PrefillArgs& a, cudaStream_t st) {
  using G = Geo<KV, D>;
  Params p = {};
  p.q = static_cast<const uint16_t*>(a.q);
  p.k_cache = static_cast<uint8_t*>(const_cast<void*>(a.k_cache));   // read only
  p.v_cache = static_cast<uint8_t*>(const_cast<void*>(a.v_cache));
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.scales = const_cast<void*>(a.scales);
  p.out = a.out;
  p.dev_status = a.dev_status;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_seqs = a.num_seqs;
  p.num_blocks = a.num_blocks;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.block_size = a.block_size;
  p.partition_size = a.max_blocks_per_seq * a.block_size;   // one partition: the whole context
  p.num_partitions = 1;
  p.parts_per_cta = 1;
  p.softmax_scale = a.softmax_scale;
  p.q_start = a.q_start;
  p.max_query_len = a.max_query_len;
  auto kern = paged_decode_kernel<KV, QT, D, true, true>;
  static std::atomic<int> attr_set[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!attr_set[dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(1, std::memory_order_relaxed);
  }
  const int group = a.num_q_heads / a.num_kv_heads;
  const int qpw = kWarp / 4 / group;                        // query tokens per warp
  const int64_t qgroups = (static_cast<int64_t>(a.max_query_len) + qpw - 1) / qpw;
  const dim3 grid(static_cast<unsigned>((qgroups + kDecodeWarps - 1) / kDecodeWarps),
                  static_cast<unsigned>(a.num_kv_heads), static_cast<unsigned>(a.num_seqs));
  return launch_pdl(kern, grid, dim3(kDecodeWarps * kWarp), G::kSmemBytes, st, p);
}

template <int KV, int QT>
cudaError_t launch_prefill_d(const PrefillArgs& a, cudaStream_t st) {
  return a.head_dim == 64 ? launch_prefill_t<KV, QT, 64>(a, st) : launch_prefill_t<KV, QT, 128>(a, st);
}

template <int KV>
cudaError_t launch_prefill_q(const PrefillArgs& a, cudaStream_t st) {
  if constexpr (KV == PKV_F16 || KV == PKV_BF16) {
    return launch_prefill_d<KV, KV>(a, st);
  } else {
    return a.q_dtype == PKV_F16 ? launch_prefill_d<KV, PKV_F16>(a, st)
                                : launch_prefill_d<KV, PKV_BF16>(a, st);
  }
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t st) {
  if (a.num_seqs == 0 || a.max_query_len == 0) return cudaSuccess;
  // 16-bit and one-byte caches run on the tcgen05 kernel (pkv_prefill_ws.cu);
  // PKV_PREFILL_MODE=mma keeps them on this one
  const char* mode = getenv("PKV_PREFILL_MODE");
  const bool mma = mode && !strcmp(mode, "mma");
  if (prefill_ws_supported(a) && !mma) return launch_prefill_ws(a, st);
  switch (a.kv_dtype) {
    case PKV_F16: return launch_prefill_q<PKV_F16>(a, st);
    case PKV_BF16: return launch_prefill_q<PKV_BF16>(a, st);
    case PKV_FP8_E4M3: return launch_prefill_q<PKV_FP8_E4M3>(a, st);
    case PKV_FP8_E5M2: return launch_prefill_q<PKV_FP8_E5M2>(a, st);
    case PKV_INT8: return launch_prefill_q<PKV_INT8>(a, st);
    default: return launch_prefill_q<PKV_INT4_G32>(a, st);
  }
}

}  // namespace pkv
