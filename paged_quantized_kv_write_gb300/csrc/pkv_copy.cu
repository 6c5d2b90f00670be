// Whole-block copies inside the paged KV pool: copy-on-write and beam forks.
//
// "KV Cache Compression & Paged Attention Deep Dive" (www.myaihardware.com),
// sections "PagedAttention: Operating System-Inspired Memory Management for
// LLMs" (copy-on-write for beam search, shared prefixes pointing at the same
// physical pages) and "Implementation Details: PagedAttention Kernel and Page
// Table" (reference counts kept for copy-on-write): a shared block is copied
// into a fresh one before a sequence writes into it.  The block manager
// (reference counts, the free list) decides which copies to make; this kernel
// performs them.
//
// One copy moves, for the pair (src, dst): the K rows and the V rows of all
// KV heads of the block (each a contiguous run of Hkv * bs * row bytes in the
// [num_blocks][Hkv][bs][row] layout) and the block's scales (FP8, INT8: Hkv
// floats per K and V; INT4: Hkv * bs * D/32 (scale, zero) pairs per K and V, also
// contiguous).  The bytes are copied as they are: a copied block dequantizes
// to exactly what its source did.
//
// Grid: x = pair, y = chunk of the pair's 16-byte units; each thread keeps
// kUnroll 16-byte loads in flight before storing them.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedkv.h"
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kUnroll = 4;
constexpr int kUnitsPerCta = kCopyThreads * kUnroll;        // 16-byte units per CTA

struct CopyParams {
  uint8_t* k_cache;
  uint8_t* v_cache;
  uint8_t* scales;
  const int32_t* pairs;        // [num_pairs][2] (src, dst)
  int* dev_status;
  int64_t block_units;         // 16-byte units of one block's K (or V) rows
  int64_t scale_bytes;         // bytes of one block's K (or V) scales (0: none)
  int64_t scale_plane;         // bytes of the whole K scale plane (V's follows)
  int num_blocks;
  int fp8_scales;              // scales in 4-byte pieces (FP8) rather than 16-byte units
};

__device__ __forceinline__ void st_global_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(const CopyParams p) {
  pdl_wait();                              // the pool may have been written just before
  const int pair = blockIdx.x;
  const int src = p.pairs[2 * pair], dst = p.pairs[2 * pair + 1];
  const bool ok = src >= 0 && src < p.num_blocks && dst >= 0 && dst < p.num_blocks;
  if (!ok) {
    if (blockIdx.y == 0 && threadIdx.x == 0) flag_status(p.dev_status, PKV_ERR_DEVICE_BOUNDS);
  } else if (src != dst) {
    // K units [0, block_units), V units [block_units, 2 block_units)
    const int64_t total = 2 * p.block_units;
    const int64_t base = static_cast<int64_t>(blockIdx.y) * kUnitsPerCta + threadIdx.x;
    uint4 v[kUnroll];
#pragma unroll
    for (int i = 0; i < kUnroll; ++i) {
      const int64_t u = base + i * kCopyThreads;
      if (u < total) {
        const bool is_v = u >= p.block_units;
        const int64_t w = is_v ? u - p.block_units : u;
        const uint8_t* c = is_v ? p.v_cache : p.k_cache;
        v[i] = ld_global_nc_v4(c + (static_cast<int64_t>(src) * p.block_units + w) * 16);
      }
    }
#pragma unroll
    for (int i = 0; i < kUnroll; ++i) {
      const int64_t u = base + i * kCopyThreads;
      if (u < total) {
        const bool is_v = u >= p.block_units;
        const int64_t w = is_v ? u - p.block_units : u;
        uint8_t* c = is_v ? p.v_cache : p.k_cache;
        st_global_v4(c + (static_cast<int64_t>(dst) * p.block_units + w) * 16, v[i]);
      }
    }
    // the scales, by the first chunk's CTA
    if (blockIdx.y == 0 && p.scale_bytes > 0) {
      for (int which = 0; which < 2; ++which) {
        const uint8_t* s = p.scales + which * p.scale_plane + static_cast<int64_t>(src) * p.scale_bytes;
        uint8_t* d = p.scales + which * p.scale_plane + static_cast<int64_t>(dst) * p.scale_bytes;
        if (p.fp8_scales) {
          for (int64_t i = threadIdx.x; i < p.scale_bytes / 4; i += kCopyThreads)
            reinterpret_cast<float*>(d)[i] = reinterpret_cast<const float*>(s)[i];
        } else {
          for (int64_t i = threadIdx.x; i < p.scale_bytes / 16; i += kCopyThreads)
            st_global_v4(d + 16 * i, ld_global_nc_v4(s + 16 * i));
        }
      }
    }
  }
  pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_copy_blocks(const CopyArgs& a, cudaStream_t st) {
  CopyParams p;
  p.k_cache = static_cast<uint8_t*>(a.k_cache);
  p.v_cache = static_cast<uint8_t*>(a.v_cache);
  p.scales = static_cast<uint8_t*>(a.scales);
  p.pairs = a.block_pairs;
  p.dev_status = a.dev_status;
  p.num_blocks = a.num_blocks;
  const int64_t rows = static_cast<int64_t>(a.num_kv_heads) * a.block_size;
  int64_t row_bytes = 2 * a.head_dim;
  p.scale_bytes = 0;
  p.fp8_scales = 0;
  if (is_blk8(a.kv_dtype)) {
    row_bytes = a.head_dim;
    p.scale_bytes = 4 * static_cast<int64_t>(a.num_kv_heads);
    p.fp8_scales = 1;
  } else if (a.kv_dtype == PKV_INT4_G32) {
    row_bytes = a.head_dim / 2;
    p.scale_bytes = rows * (a.head_dim / 32) * 4;
  }
  p.block_units = rows * row_bytes / 16;
  p.scale_plane = static_cast<int64_t>(a.num_blocks) * p.scale_bytes;
  const int64_t chunks = (2 * p.block_units + kUnitsPerCta - 1) / kUnitsPerCta;
  const dim3 grid(static_cast<unsigned>(a.num_pairs), static_cast<unsigned>(chunks));
  return launch_pdl(copy_blocks_kernel, grid, dim3(kCopyThreads), 0, st, p);
}

}  // namespace pkv
