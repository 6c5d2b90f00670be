// Host-side argument bundles passed from the C ABI to the kernel launchers.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pkv {

struct WriteArgs {
  const void* k_new;
  const void* v_new;
  int new_dtype;
  const int64_t* slot_mapping;
  int64_t num_tokens;
  void* k_cache;
  void* v_cache;
  void* scales;
  int kv_dtype;
  int num_blocks;
  int num_kv_heads;
  int head_dim;
  int block_size;
  int* dev_status;
};

struct DecodeArgs {
  const void* q;
  int q_dtype;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  int max_blocks_per_seq;
  const int32_t* context_lens;
  int num_seqs;
  const void* scales;
  int kv_dtype;
  int num_blocks;
  void* out;
  float softmax_scale;
  int num_q_heads;
  int num_kv_heads;
  int head_dim;
  int block_size;
  int partition_size;   // resolved, multiple of 16
  int num_partitions;   // grid.x: ceil(max_blocks_per_seq * block_size / partition_size)
  float* ws_out;        // [num_seqs][num_q_heads][num_partitions][head_dim]
  float* ws_ml;         // [num_seqs][num_q_heads][num_partitions][2]
  int* dev_status;
  // fused write (null for attention alone): new K/V [num_seqs][Hkv][D] in q_dtype
  const void* k_new = nullptr;
  const void* v_new = nullptr;
  const int64_t* slot_mapping = nullptr;
  // the whole caller workspace (the balanced split lays it out its own way)
  void* ws_base = nullptr;
  size_t ws_bytes = 0;
};

// Balanced split of the decode work (warp-owned, equal tile counts per warp):
// at most kBalMaxSeqs sequences, at most kBalMaxWarps warps (152 SMs x 4 CTAs
// x 4 warps).  Its workspace: partial rows [slots][G][D] floats, then
// (max, sum) [slots][G][2], with slots = kBalMaxWarps + num_seqs *
// num_kv_heads (the second part 256-byte aligned).
constexpr int kBalMaxSeqs = 512;
constexpr int kBalMaxWarps = 152 * 4 * 4;
struct BalLayout {
  size_t ml_off, bytes;
};
inline BalLayout bal_layout(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim) {
  const size_t slots = static_cast<size_t>(kBalMaxWarps) + static_cast<size_t>(num_seqs) * num_kv_heads;
  const size_t rows = slots * static_cast<size_t>(num_q_heads / num_kv_heads);
  BalLayout L;
  L.ml_off = (rows * head_dim * 4 + 255) / 256 * 256;
  L.bytes = L.ml_off + rows * 2 * 4;
  return L;
}
// whether a call may take the balanced split (the tile list must fit int)
inline bool bal_eligible(int num_seqs, int num_kv_heads, int max_blocks_per_seq, int block_size,
                         int num_partitions) {
  if (num_partitions <= 1 || num_seqs > kBalMaxSeqs) return false;
  const int64_t tiles = (static_cast<int64_t>(max_blocks_per_seq) * block_size + 15) / 16;
  return static_cast<int64_t>(num_seqs) * num_kv_heads * tiles < (int64_t(1) << 30);
}

struct PrefillArgs {
  const void* q;                 // [q_start[num_seqs]][num_q_heads][head_dim]
  int q_dtype;
  const int32_t* q_start;        // [num_seqs + 1]
  int max_query_len;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  int max_blocks_per_seq;
  const int32_t* context_lens;
  int num_seqs;
  const void* scales;
  int kv_dtype;
  int num_blocks;
  void* out;
  float softmax_scale;
  int num_q_heads;
  int num_kv_heads;
  int head_dim;
  int block_size;
  int* dev_status;
};

struct CopyArgs {
  void* k_cache;
  void* v_cache;
  void* scales;
  int kv_dtype;
  const int32_t* block_pairs;   // [num_pairs][2] (src, dst)
  int num_pairs;
  int num_blocks;
  int num_kv_heads;
  int head_dim;
  int block_size;
  int* dev_status;
};

cudaError_t launch_kv_write(const WriteArgs& a, cudaStream_t st);
cudaError_t launch_copy_blocks(const CopyArgs& a, cudaStream_t st);
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t st);
cudaError_t launch_lse_reduce(const DecodeArgs& a, cudaStream_t st);
// 16-bit and one-byte caches: the tcgen05 prefill with warp roles (pkv_prefill_ws.cu)
bool prefill_ws_supported(const PrefillArgs& a);
cudaError_t launch_prefill_ws(const PrefillArgs& a, cudaStream_t st);
#ifdef PKV_TEST_HOOKS
// comparators, built into the test library only: decode on the tcgen05 tensor
// cores (one-byte caches, head_dim 128, G <= 8) and on the CUDA cores
bool decode_tc_supported(const DecodeArgs& a);
cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_simt(const DecodeArgs& a, cudaStream_t st);
#endif
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st);
// the decode launchers per cache-dtype family (one translation unit each)
cudaError_t launch_decode_half(const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_decode_byte(const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_decode_int4(const DecodeArgs& a, cudaStream_t st);

int resolve_partition_size(int num_seqs, int num_q_heads, int num_kv_heads,
                           int max_blocks_per_seq, int block_size, int requested);

}  // namespace pkv
