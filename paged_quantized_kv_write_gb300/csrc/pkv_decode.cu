// paged_decode_attention: dispatch to the per-dtype launchers (the kernel is
// in pkv_attn.cuh, its launch side and the log-sum-exp merge of split-KV
// partitions in pkv_decode_launch.cuh), the merge for the test build's SIMT
// comparator, and the partition-size heuristic.
#include "pkv_decode_launch.cuh"

namespace pkv {

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
  const int heads = a.num_seqs * a.num_q_heads;
  if (a.q_dtype == PKV_F16) {
    return a.head_dim == 64 ? launch_lse_typed<PKV_F16, 64>(p, heads, st)
                            : launch_lse_typed<PKV_F16, 128>(p, heads, st);
  }
  return a.head_dim == 64 ? launch_lse_typed<PKV_BF16, 64>(p, heads, st)
                          : launch_lse_typed<PKV_BF16, 128>(p, heads, st);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
  if (a.num_seqs == 0) return cudaSuccess;
  switch (a.kv_dtype) {
    case PKV_F16:
    case PKV_BF16: return launch_decode_half(a, st);
    case PKV_FP8_E4M3:
    case PKV_FP8_E5M2:
    case PKV_INT8: return launch_decode_byte(a, st);
    default: return launch_decode_int4(a, st);
  }
}

int resolve_partition_size(int num_seqs, int num_q_heads, int num_kv_heads,
                           int max_blocks_per_seq, int block_size, int requested) {
  // requests beyond 2^30 tokens (more than any context the calls accept) are
  // clamped first, so rounding up to whole tiles cannot overflow
  if (requested > 0) return ((std::min(requested, 1 << 30) + kTile - 1) / kTile) * kTile;
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
