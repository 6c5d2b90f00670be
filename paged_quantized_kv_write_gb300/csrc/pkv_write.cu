// paged_kv_write: store new K/V rows at their physical slots, quantizing on
// the way in.
//
// One warp owns one (token, KV head) and handles K then V (the encoder and
// the encodings are in pkv_encode.cuh).
//
// One-byte formats (FP8 E4M3/E5M2, INT8) take one scale per (block, KV head)
// from the absolute maximum of the block ("Block-Wise Scaling Factors",
// snippet-4).  A call that writes a block's offset-0 slot opens the block,
// and its scale is taken over every token that call writes into it.  That
// needs the whole call's rows before any code is written, so the write runs
// as three launches over the caller's scale array, which doubles as the
// accumulator:
//   open   offset-0 tokens: atomicMax(word, 0x80000000 | bits(row amax)).
//          Any kept scale is a positive float, below every mark as an
//          unsigned word, so the mark replaces it.
//   grow   other tokens: if their block's word carries the mark,
//          atomicMax(word, mark | bits(row amax)); blocks with a kept scale
//          (sign clear) are left alone.
//   encode every token: the scale is the word, or max(amax / max_finite,
//          1e-12) of a marked word; the offset-0 token stores it.
// Stored scales are never negative, so the sign bit is free for the mark.
#include "pkv_common.cuh"
#include "pkv_encode.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kWriteWarps = 8;   // warps (token-head rows) per CTA

enum WritePhase { kOpen = 0, kGrow = 1, kEncode = 2 };

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
    if (slot != -1 && lane == 0 && head == 0 && PHASE == kEncode)
      flag_status(dev_status, PKV_ERR_DEVICE_BOUNDS);
    return;
  }
  const int64_t nslots = static_cast<int64_t>(num_blocks) * block_size;
  if (slot >= nslots) {
    if (lane == 0 && head == 0 && PHASE == kEncode) flag_status(dev_status, PKV_ERR_DEVICE_BOUNDS);
    return;
  }
  const int64_t block = slot / block_size;
  const int offset = static_cast<int>(slot - block * block_size);
  if constexpr (PHASE == kEncode) {
    encode_token_head<KV, NEW, D, is_blk8(KV) ? kScaleFromWord : kScaleOwnRow>(
        k_new + row * D, v_new + row * D, k_cache, v_cache, scales, num_blocks, num_kv_heads,
        block_size, block, head, offset, lane);
  } else {
    if ((PHASE == kOpen) != (offset == 0)) return;
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      unsigned int* word = reinterpret_cast<unsigned int*>(scales) +
                           (static_cast<int64_t>(which) * num_blocks + block) * num_kv_heads + head;
      if constexpr (PHASE == kGrow) {
        uint32_t w = 0;
        if (lane == 0) w = __ldcg(word);
        if (!(__shfl_sync(0xffffffffu, w, 0) & kOpenMark)) continue;   // a kept scale
      }
      const float amax = row_amax<NEW, D>((which ? v_new : k_new) + row * D, lane);
      if (lane == 0) atomicMax(word, kOpenMark | __float_as_uint(amax));
    }
  }
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
    // open the blocks whose offset-0 slot this call writes, grow their amax
    // over the call's other rows, then encode with the finished scales
    cudaError_t e = launch_one<KV, NEW, D, kOpen>(a, st);
    if (e == cudaSuccess) e = launch_one<KV, NEW, D, kGrow>(a, st);
    if (e != cudaSuccess) return e;
    return launch_one<KV, NEW, D, kEncode>(a, st);
  } else {
    return launch_one<KV, NEW, D, kEncode>(a, st);
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
