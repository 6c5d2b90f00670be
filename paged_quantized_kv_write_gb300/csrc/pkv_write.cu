// paged_kv_write: store new K/V rows at their physical slots, quantizing on
// the way in.
//
// One warp owns one (token, KV head) and handles K then V (the encoder and
// the encodings are in pkv_encode.cuh).  FP8 runs as two launches: tokens at
// block offset 0 first (they set the block scales), then the rest.
#include "pkv_common.cuh"
#include "pkv_encode.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kWriteWarps = 8;   // warps (token-head rows) per CTA

// PHASE 0: only tokens at block offset 0; 1: only the others; 2: all tokens.
template <int KV, int NEW, int D, int PHASE>
__global__ void __launch_bounds__(kWriteWarps * kWarp)
kv_write_kernel(const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
                const int64_t* __restrict__ slot_mapping, int64_t num_tokens,
                uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
                void* __restrict__ scales, int num_blocks, int num_kv_heads, int block_size,
                int* __restrict__ dev_status) {
  pdl_wait();                 // inputs and cache may come from the previous kernel
  pdl_launch_dependents();
  const int lane = threadIdx.x & (kWarp - 1);
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kWriteWarps + (threadIdx.x >> 5);
  if (row >= num_tokens * num_kv_heads) return;
  const int64_t tok = row / num_kv_heads;
  const int head = static_cast<int>(row - tok * num_kv_heads);
  const int64_t slot = slot_mapping[tok];
  if (slot < 0) {
    if (slot != -1 && lane == 0 && head == 0 && PHASE != 1) flag_status(dev_status, PKV_ERR_DEVICE_BOUNDS);
    return;
  }
  const int64_t nslots = static_cast<int64_t>(num_blocks) * block_size;
  if (slot >= nslots) {
    if (lane == 0 && head == 0 && PHASE != 1) flag_status(dev_status, PKV_ERR_DEVICE_BOUNDS);
    return;
  }
  const int64_t block = slot / block_size;
  const int offset = static_cast<int>(slot - block * block_size);
  if (PHASE == 0 && offset != 0) return;
  if (PHASE == 1 && offset == 0) return;
  encode_token_head<KV, NEW, D>(k_new + row * D, v_new + row * D, k_cache, v_cache, scales,
                                num_blocks, num_kv_heads, block_size, block, head, offset, lane);
}

template <int KV, int NEW, int D, int PHASE>
cudaError_t launch_one(const WriteArgs& a, cudaStream_t st) {
  const int64_t rows = a.num_tokens * a.num_kv_heads;
  const int64_t grid = (rows + kWriteWarps - 1) / kWriteWarps;
  return launch_pdl(kv_write_kernel<KV, NEW, D, PHASE>, dim3(static_cast<unsigned>(grid)),
                    dim3(kWriteWarps * kWarp), 0, st, static_cast<const uint16_t*>(a.k_new),
                    static_cast<const uint16_t*>(a.v_new), a.slot_mapping, a.num_tokens,
                    static_cast<uint8_t*>(a.k_cache), static_cast<uint8_t*>(a.v_cache), a.scales,
                    a.num_blocks, a.num_kv_heads, a.block_size, a.dev_status);
}

template <int KV, int NEW, int D>
cudaError_t launch_kv(const WriteArgs& a, cudaStream_t st) {
  if constexpr (is_blk8(KV)) {
    // offset-0 tokens set the block scales; the rest read them afterwards
    cudaError_t e = launch_one<KV, NEW, D, 0>(a, st);
    if (e != cudaSuccess) return e;
    return launch_one<KV, NEW, D, 1>(a, st);
  } else {
    return launch_one<KV, NEW, D, 2>(a, st);
  }
}

template <int NEW, int D>
cudaError_t dispatch_kv(const WriteArgs& a, cudaStream_t st) {
  switch (a.kv_dtype) {
    case PKV_F16: return launch_kv<PKV_F16, NEW, D>(a, st);
    case PKV_BF16: return launch_kv<PKV_BF16, NEW, D>(a, st);
    case PKV_FP8_E4M3: return launch_kv<PKV_FP8_E4M3, NEW, D>(a, st);
    case PKV_FP8_E5M2: return launch_kv<PKV_FP8_E5M2, NEW, D>(a, st);
    case PKV_INT8: return launch_kv<PKV_INT8, NEW, D>(a, st);
    default: return launch_kv<PKV_INT4_G32, NEW, D>(a, st);
  }
}

}  // namespace

cudaError_t launch_kv_write(const WriteArgs& a, cudaStream_t st) {
  if (a.num_tokens == 0) return cudaSuccess;
  if (a.new_dtype == PKV_F16)
    return a.head_dim == 64 ? dispatch_kv<PKV_F16, 64>(a, st) : dispatch_kv<PKV_F16, 128>(a, st);
  return a.head_dim == 64 ? dispatch_kv<PKV_BF16, 64>(a, st) : dispatch_kv<PKV_BF16, 128>(a, st);
}

}  // namespace pkv
