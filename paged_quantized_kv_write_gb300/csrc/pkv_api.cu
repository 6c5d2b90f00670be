// C ABI of the pagedkv library: argument validation and dispatch.  Every
// check that can fail runs before anything is launched; the entry points
// never allocate, never synchronize and never abort.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "pagedkv.h"
#include "pkv_internal.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool ok_head_dim(int d) { return d == 64 || d == 128; }
bool ok_block_size(int bs) { return bs >= 16 && bs <= 256 && bs % 16 == 0; }
bool ok_kv_dtype(int t) { return t >= PKV_F16 && t <= PKV_INT8; }
bool ok_half_dtype(int t) { return t == PKV_F16 || t == PKV_BF16; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Split-KV partial results are (sequence, q head, partition) rows of
// head_dim + 2 floats.  Bounding their count at 2^40 keeps every byte count
// derived from it far inside int64 and size_t (at most 2^27 partitions of
// 2^31 rows each, so the product itself cannot overflow).
bool workspace_fits(int num_seqs, int num_q_heads, int num_kv_heads, int max_blocks_per_seq,
                    int block_size, int partition_size) {
  const int part = pkv::resolve_partition_size(num_seqs, num_q_heads, num_kv_heads,
                                               max_blocks_per_seq, block_size, partition_size);
  if (part <= 0) return false;
  const int64_t np = ceil_div(static_cast<int64_t>(max_blocks_per_seq) * block_size, part);
  const int64_t heads = static_cast<int64_t>(num_seqs) * num_q_heads;
  return heads <= 0x7FFFFFFF && np <= 0x7FFFFFFF && heads * np <= (int64_t(1) << 40);
}

// paged_decode_attention, and its fused-write form when slot_mapping is set
int decode_impl(const void* q, int q_dtype, const void* k_new, const void* v_new,
                const int64_t* slot_mapping, const void* k_cache, const void* v_cache,
                const int32_t* block_tables, int max_blocks_per_seq,
                const int32_t* context_lens, int num_seqs, const void* scales, int kv_dtype,
                int num_blocks, void* out, float softmax_scale, int num_q_heads,
                int num_kv_heads, int head_dim, int block_size, int partition_size,
                void* workspace, size_t workspace_bytes, int* dev_status, void* stream) {
  if (num_seqs < 0 || num_blocks <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      max_blocks_per_seq <= 0 || partition_size < 0)
    return PKV_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads) return PKV_ERR_INVALID_ARG;
  if (!ok_half_dtype(q_dtype) || !ok_kv_dtype(kv_dtype)) return PKV_ERR_UNSUPPORTED;
  if ((kv_dtype == PKV_F16 || kv_dtype == PKV_BF16) && q_dtype != kv_dtype)
    return PKV_ERR_UNSUPPORTED;
  if (!ok_head_dim(head_dim) || !ok_block_size(block_size)) return PKV_ERR_UNSUPPORTED;
  if (num_q_heads / num_kv_heads > 8) return PKV_ERR_UNSUPPORTED;
  if (num_seqs > 65535 || num_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;
  // the merge runs one CTA per (sequence, q head) on a 1-D grid
  if (static_cast<int64_t>(num_seqs) * num_q_heads > 0x7FFFFFFF) return PKV_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_blocks_per_seq) * block_size > 0x7FFFFFFF) return PKV_ERR_UNSUPPORTED;
  // the kernel locates a 16-token sub-tile as (block * Hkv + head) << 4 | offset / 16
  if (static_cast<int64_t>(num_blocks) * num_kv_heads >= (int64_t(1) << 27)) return PKV_ERR_UNSUPPORTED;
  if (!(softmax_scale == softmax_scale)) return PKV_ERR_INVALID_ARG;
  if (!workspace_fits(num_seqs, num_q_heads, num_kv_heads, max_blocks_per_seq, block_size,
                      partition_size))
    return PKV_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
    return PKV_ERR_INVALID_ARG;
  const bool quant = kv_dtype != PKV_F16 && kv_dtype != PKV_BF16;
  if (quant && !scales) return PKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
      (reinterpret_cast<uintptr_t>(context_lens) & 3u) || (quant && !aligned16(scales)))
    return PKV_ERR_INVALID_ARG;
  const int part = pkv::resolve_partition_size(num_seqs, num_q_heads, num_kv_heads,
                                               max_blocks_per_seq, block_size, partition_size);
  const int64_t np = ceil_div(static_cast<int64_t>(max_blocks_per_seq) * block_size, part);
  if (np > 0x7FFFFFFF) return PKV_ERR_UNSUPPORTED;
  float* ws_out = nullptr;
  float* ws_ml = nullptr;
  if (np > 1) {
    const size_t need = paged_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads,
                                                     head_dim, max_blocks_per_seq, block_size,
                                                     partition_size);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return PKV_ERR_WORKSPACE;
    const int64_t out_bytes = static_cast<int64_t>(num_seqs) * num_q_heads * np * head_dim * 4;
    ws_out = static_cast<float*>(workspace);
    ws_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + ceil_div(out_bytes, 256) * 256);
  }
  if (slot_mapping && (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new) ||
                       (reinterpret_cast<uintptr_t>(slot_mapping) & 7u)))
    return PKV_ERR_INVALID_ARG;
  pkv::DecodeArgs a{q, q_dtype, k_cache, v_cache, block_tables, max_blocks_per_seq,
                    context_lens, num_seqs, scales, kv_dtype, num_blocks, out, softmax_scale,
                    num_q_heads, num_kv_heads, head_dim, block_size, part,
                    static_cast<int>(np), ws_out, ws_ml, dev_status};
  a.k_new = k_new;
  a.v_new = v_new;
  a.slot_mapping = slot_mapping;
  a.ws_base = np > 1 ? workspace : nullptr;
  a.ws_bytes = np > 1 ? workspace_bytes : 0;
  cudaError_t e = pkv::launch_decode(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

extern "C" {

int paged_kv_write(const void* k_new, const void* v_new, int new_dtype,
                   const int64_t* slot_mapping, int64_t num_tokens,
                   void* k_cache, void* v_cache, void* scales, int kv_dtype,
                   int num_blocks, int num_kv_heads, int head_dim, int block_size,
                   int* dev_status, void* stream) {
  if (num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0) return PKV_ERR_INVALID_ARG;
  if (!ok_half_dtype(new_dtype) || !ok_kv_dtype(kv_dtype)) return PKV_ERR_UNSUPPORTED;
  if ((kv_dtype == PKV_F16 || kv_dtype == PKV_BF16) && new_dtype != kv_dtype)
    return PKV_ERR_UNSUPPORTED;
  if (!ok_head_dim(head_dim) || !ok_block_size(block_size)) return PKV_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
  const bool quant = kv_dtype != PKV_F16 && kv_dtype != PKV_BF16;
  if (quant && !scales) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) || (quant && !aligned16(scales)))
    return PKV_ERR_INVALID_ARG;
  if (static_cast<int64_t>(num_blocks) * block_size > (int64_t(1) << 40)) return PKV_ERR_INVALID_ARG;
  // one warp per (token, KV head), eight per CTA, on a 1-D grid (num_tokens is
  // bounded first so that the product cannot overflow)
  if (num_tokens > (int64_t(1) << 34) || ceil_div(num_tokens * num_kv_heads, 8) > 0x7FFFFFFF)
    return PKV_ERR_UNSUPPORTED;
  pkv::WriteArgs a{k_new, v_new, new_dtype, slot_mapping, num_tokens, k_cache, v_cache,
                   scales, kv_dtype, num_blocks, num_kv_heads, head_dim, block_size, dev_status};
  cudaError_t e = pkv::launch_kv_write(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int paged_kv_copy_blocks(void* k_cache, void* v_cache, void* scales, int kv_dtype,
                         const int32_t* block_pairs, int num_pairs, int num_blocks,
                         int num_kv_heads, int head_dim, int block_size, int* dev_status,
                         void* stream) {
  if (num_pairs < 0 || num_blocks <= 0 || num_kv_heads <= 0) return PKV_ERR_INVALID_ARG;
  if (!ok_kv_dtype(kv_dtype)) return PKV_ERR_UNSUPPORTED;
  if (!ok_head_dim(head_dim) || !ok_block_size(block_size)) return PKV_ERR_UNSUPPORTED;
  if (num_pairs == 0) return PKV_OK;
  if (!k_cache || !v_cache || !block_pairs) return PKV_ERR_INVALID_ARG;
  const bool quant = kv_dtype != PKV_F16 && kv_dtype != PKV_BF16;
  if (quant && !scales) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || (reinterpret_cast<uintptr_t>(block_pairs) & 3u) ||
      (quant && !aligned16(scales)))
    return PKV_ERR_INVALID_ARG;
  // chunks of one block's K + V rows per grid column (<= 65535)
  const int64_t block_bytes = static_cast<int64_t>(num_kv_heads) * block_size * 2 * head_dim;
  if (2 * block_bytes / 16 > int64_t(65535) * 1024) return PKV_ERR_UNSUPPORTED;
  pkv::CopyArgs a{k_cache, v_cache, scales, kv_dtype, block_pairs, num_pairs, num_blocks,
                  num_kv_heads, head_dim, block_size, dev_status};
  cudaError_t e = pkv::launch_copy_blocks(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int paged_decode_partition_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                int max_blocks_per_seq, int block_size, int partition_size) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_blocks_per_seq <= 0 ||
      !ok_block_size(block_size) || partition_size < 0)
    return 0;
  return pkv::resolve_partition_size(num_seqs, num_q_heads, num_kv_heads, max_blocks_per_seq,
                                     block_size, partition_size);
}

size_t paged_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                    int head_dim, int max_blocks_per_seq, int block_size,
                                    int partition_size) {
  const int part = paged_decode_partition_size(num_seqs, num_q_heads, num_kv_heads,
                                               max_blocks_per_seq, block_size, partition_size);
  if (part <= 0 || !ok_head_dim(head_dim) || num_seqs > 65535 || num_q_heads > 65535 * 8 ||
      static_cast<int64_t>(max_blocks_per_seq) * block_size > 0x7FFFFFFF ||
      !workspace_fits(num_seqs, num_q_heads, num_kv_heads, max_blocks_per_seq, block_size,
                      partition_size))
    return 0;   // arguments the calls reject
  const int64_t np = ceil_div(static_cast<int64_t>(max_blocks_per_seq) * block_size, part);
  if (np <= 1) return 0;
  const int64_t heads = static_cast<int64_t>(num_seqs) * num_q_heads;
  const int64_t out_bytes = heads * np * head_dim * 4;
  const int64_t ml_bytes = heads * np * 2 * 4;
  size_t bytes = static_cast<size_t>(ceil_div(out_bytes, 256) * 256 + ml_bytes);
  // room for the balanced split's layout too, when the call may take it
  if (num_q_heads % num_kv_heads == 0 &&
      pkv::bal_eligible(num_seqs, num_kv_heads, max_blocks_per_seq, block_size,
                        static_cast<int>(np)))
    bytes = std::max(bytes, pkv::bal_layout(num_seqs, num_q_heads, num_kv_heads, head_dim).bytes);
  return bytes;
}

int paged_decode_attention(const void* q, int q_dtype,
                           const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           const int32_t* context_lens, int num_seqs,
                           const void* scales, int kv_dtype, int num_blocks,
                           void* out, float softmax_scale,
                           int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                           int partition_size, void* workspace, size_t workspace_bytes,
                           int* dev_status, void* stream) {
  return decode_impl(q, q_dtype, nullptr, nullptr, nullptr, k_cache, v_cache, block_tables,
                     max_blocks_per_seq, context_lens, num_seqs, scales, kv_dtype, num_blocks,
                     out, softmax_scale, num_q_heads, num_kv_heads, head_dim, block_size,
                     partition_size, workspace, workspace_bytes, dev_status, stream);
}

int paged_prefill_attention(const void* q, int q_dtype, const int32_t* q_start,
                            int max_query_len, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* context_lens, int num_seqs, const void* scales,
                            int kv_dtype, int num_blocks, void* out, float softmax_scale,
                            int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                            int* dev_status, void* stream) {
  if (num_seqs < 0 || num_blocks <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      max_blocks_per_seq <= 0 || max_query_len < 0)
    return PKV_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads) return PKV_ERR_INVALID_ARG;
  if (!ok_half_dtype(q_dtype) || !ok_kv_dtype(kv_dtype)) return PKV_ERR_UNSUPPORTED;
  if ((kv_dtype == PKV_F16 || kv_dtype == PKV_BF16) && q_dtype != kv_dtype)
    return PKV_ERR_UNSUPPORTED;
  if (!ok_head_dim(head_dim) || !ok_block_size(block_size)) return PKV_ERR_UNSUPPORTED;
  const int group = num_q_heads / num_kv_heads;
  if (8 % group) return PKV_ERR_UNSUPPORTED;                 // G in {1, 2, 4, 8}
  if (num_seqs > 65535 || num_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_blocks_per_seq) * block_size > 0x7FFFFFFF) return PKV_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(num_blocks) * num_kv_heads >= (int64_t(1) << 27)) return PKV_ERR_UNSUPPORTED;
  if (!(softmax_scale == softmax_scale)) return PKV_ERR_INVALID_ARG;
  if (num_seqs == 0 || max_query_len == 0) return PKV_OK;
  if (!q || !q_start || !k_cache || !v_cache || !block_tables || !context_lens || !out)
    return PKV_ERR_INVALID_ARG;
  const bool quant = kv_dtype != PKV_F16 && kv_dtype != PKV_BF16;
  if (quant && !scales) return PKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
      (reinterpret_cast<uintptr_t>(context_lens) & 3u) ||
      (reinterpret_cast<uintptr_t>(q_start) & 3u) || (quant && !aligned16(scales)))
    return PKV_ERR_INVALID_ARG;
  pkv::PrefillArgs a{q, q_dtype, q_start, max_query_len, k_cache, v_cache, block_tables,
                     max_blocks_per_seq, context_lens, num_seqs, scales, kv_dtype, num_blocks,
                     out, softmax_scale, num_q_heads, num_kv_heads, head_dim, block_size,
                     dev_status};
  cudaError_t e = pkv::launch_prefill(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int paged_decode_attention_with_write(const void* q, int q_dtype, const void* k_new,
                                      const void* v_new, const int64_t* slot_mapping,
                                      void* k_cache, void* v_cache,
                                      const int32_t* block_tables, int max_blocks_per_seq,
                                      const int32_t* context_lens, int num_seqs, void* scales,
                                      int kv_dtype, int num_blocks, void* out,
                                      float softmax_scale, int num_q_heads, int num_kv_heads,
                                      int head_dim, int block_size, int partition_size,
                                      void* workspace, size_t workspace_bytes, int* dev_status,
                                      void* stream) {
  if (num_seqs > 0 && !slot_mapping) return PKV_ERR_INVALID_ARG;
  return decode_impl(q, q_dtype, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables,
                     max_blocks_per_seq, context_lens, num_seqs, scales, kv_dtype, num_blocks,
                     out, softmax_scale, num_q_heads, num_kv_heads, head_dim, block_size,
                     partition_size, workspace, workspace_bytes, dev_status, stream);
}

const char* paged_kv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case PKV_ERR_CUDA: return "CUDA launch failed";
    case PKV_ERR_DEVICE_BOUNDS: return "block id or slot outside the pool";
    case PKV_ERR_WORKSPACE: return "workspace missing or too small";
    case PKV_ERR_DEVICE_TIMEOUT: return "a kernel's wait for its own asynchronous work timed out";
    default: return "unknown status";
  }
}

int paged_kv_version(void) { return 100; }

}  // extern "C"
