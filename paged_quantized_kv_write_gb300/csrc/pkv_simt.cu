// A SIMT comparator for the decode kernel, selected with PKV_DECODE_MODE=simt:
// the same computation with CUDA-core FMAs and warp-shuffle reductions in
// place of mma.sync, in the shape the pages describe for vLLM's kernel ("KV
// Cache Compression & Paged Attention", Implementation Details: per token,
// dot products of q with the gathered K row, softmax, weighted sum of V).
// It exists to measure what the tensor-core formulation buys; the library
// never picks it by itself, and only the test build (libpagedkv_test.so,
// compiled with PKV_TEST_HOOKS) contains it.
//
// One warp owns one (sequence, KV head, partition) unit, like the tensor
// kernel's warp-owned mode: lane l holds elements [EPL*l, EPL*l + EPL) of q
// (all G heads, fp32) and of the output accumulators.  16-token tiles of K
// and V rows are staged in a per-warp shared-memory ring with 16-byte
// cp.async copies; every token is then consumed in turn: EPL * G FMAs for the
// partial dot products, a 5-step xor-shuffle all-reduce per head, an online
// softmax update per head (fp32, every lane keeps the same state), and
// EPL * G FMAs for the output.  Partitions are merged by the same
// log-sum-exp kernel as the tensor path.  16-bit, FP8 and INT8 caches.
#include <math.h>
#include <stdint.h>

#include "pagedkv.h"
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kSimtWarps = 4;
constexpr int kSimtTile = 16;      // tokens per staged tile
constexpr int kSimtStages = 2;
constexpr float kLog2eS = 1.4426950408889634f;

template <int KV, int D>
struct SimtGeo {
  static constexpr bool kHalf = KV == PKV_F16 || KV == PKV_BF16;
  static constexpr int kEpl = D / kWarp;                    // elements per lane: 4 or 2
  static constexpr int kRow = kHalf ? 2 * D : D;            // bytes per token row
  static constexpr int kTileBytes = kSimtTile * kRow;       // K (or V) rows of a tile
  static constexpr int kStageBytes = 2 * kTileBytes + 16;   // + K scale, V scale, valid
  static constexpr int kWarpRing = kSimtStages * kStageBytes;
  static constexpr int kSmem = kSimtWarps * kWarpRing;
};

struct SimtParams {
  const uint16_t* q;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const float* scales;
  void* out;
  float* ws_out;
  float* ws_ml;
  int* dev_status;
  int max_blocks_per_seq;
  int num_blocks;
  int num_q_heads;
  int num_kv_heads;
  int block_size;
  int partition_size;
  int num_partitions;
  float softmax_scale;
};

// this lane's EPL elements of a token row in shared memory, as fp32
template <int KV, int D>
__device__ __forceinline__ void load_row(uint32_t row_smem, int lane, float (&x)[D / kWarp]) {
  constexpr int EPL = D / kWarp;
  if constexpr (KV == PKV_F16 || KV == PKV_BF16) {
    if constexpr (EPL == 4) {
      const uint2 w = ld_shared_v2(row_smem + 8 * lane);
      const float2 a = Half16<KV>::unpack(w.x), b = Half16<KV>::unpack(w.y);
      x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
    } else {
      const float2 a = Half16<KV>::unpack(ld_shared_b32(row_smem + 4 * lane));
      x[0] = a.x; x[1] = a.y;
    }
  } else {
    uint32_t w;
    if constexpr (EPL == 4) {
      w = ld_shared_b32(row_smem + 4 * lane);
    } else {
      w = ld_shared_u16(row_smem + 2 * lane);
    }
    if constexpr (KV == PKV_INT8) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) x[e] = static_cast<float>(static_cast<int8_t>(w >> (8 * e)));
    } else {
      const float2 a = Half16<PKV_F16>::unpack(fp8x2_to_f16x2<KV>(static_cast<uint16_t>(w & 0xFFFFu)));
      x[0] = a.x; x[1] = a.y;
      if constexpr (EPL == 4) {
        const float2 b = Half16<PKV_F16>::unpack(fp8x2_to_f16x2<KV>(static_cast<uint16_t>(w >> 16)));
        x[2] = b.x; x[3] = b.y;
      }
    }
  }
}

template <int KV, int QT, int D>
__global__ void __launch_bounds__(kSimtWarps * kWarp)
simt_decode_kernel(const SimtParams p) {
  using G = SimtGeo<KV, D>;
  constexpr int EPL = G::kEpl;
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_wait();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int kvh = static_cast<int>(blockIdx.y) * kSimtWarps + warp;
  const int part = blockIdx.x, b = blockIdx.z;
  if (kvh >= p.num_kv_heads) return;
  const int group = p.num_q_heads / p.num_kv_heads;
  const int cap = p.max_blocks_per_seq * p.block_size;
  int ctx = p.context_lens[b];
  if (ctx > cap) {
    if (lane == 0 && part == 0 && kvh == 0) flag_status(p.dev_status, PKV_ERR_DEVICE_BOUNDS);
    ctx = cap;
  }
  const int t_begin = part * p.partition_size;
  const int t_end = min(ctx, t_begin + p.partition_size);
  if (t_begin >= max(ctx, 1)) return;                       // a partition past this context
  const uint32_t ring = smem_u32(smem + warp * G::kWarpRing);
  uint8_t* ring_ptr = smem + warp * G::kWarpRing;

  // q of the G heads, this lane's elements, fp32
  float q[8][EPL];
#pragma unroll
  for (int h = 0; h < 8; ++h)
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      q[h][e] = 0.f;
      if (h < group) {
        const uint16_t* qrow = p.q + (static_cast<int64_t>(b) * p.num_q_heads + kvh * group + h) * D;
        q[h][e] = Half16<QT>::to_float(qrow[EPL * lane + e]);
      }
    }
  float o[8][EPL], m[8], l[8];
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[h][e] = 0.f;
  }

  const int ntiles = t_end > t_begin ? (t_end - t_begin + kSimtTile - 1) / kSimtTile : 0;
  // stage tile i into ring stage s (all lanes); marks the stage valid or empty
  auto issue = [&](int i, int s) {
    const uint32_t sb = ring + s * G::kStageBytes;
    int* misc = reinterpret_cast<int*>(ring_ptr + s * G::kStageBytes + 2 * G::kTileBytes);
    if (i < ntiles) {
      const int t0 = t_begin + i * kSimtTile;
      const int logical = t0 / p.block_size;
      const int phys = __ldg(p.block_tables + static_cast<int64_t>(b) * p.max_blocks_per_seq + logical);
      const bool ok = phys >= 0 && phys < p.num_blocks;
      if (lane == 0) misc[2] = ok ? 1 : 0;
      if (!ok) {
        if (lane == 0) flag_status(p.dev_status, PKV_ERR_DEVICE_BOUNDS);
      } else {
        const int64_t row0 = (static_cast<int64_t>(phys) * p.num_kv_heads + kvh) * p.block_size +
                             (t0 - logical * p.block_size);
        const uint8_t* ks = p.k_cache + row0 * G::kRow;
        const uint8_t* vs = p.v_cache + row0 * G::kRow;
        constexpr int kChunks = G::kTileBytes / 16;
#pragma unroll
        for (int c = lane; c < kChunks; c += kWarp) {
          cp_async_16(sb + 16 * c, ks + 16 * c);
          cp_async_16(sb + G::kTileBytes + 16 * c, vs + 16 * c);
        }
        if constexpr (is_blk8(KV)) {
          const int64_t idx = static_cast<int64_t>(phys) * p.num_kv_heads + kvh;
          const int64_t per_kv = static_cast<int64_t>(p.num_blocks) * p.num_kv_heads;
          const uint32_t mo = sb + 2 * G::kTileBytes;
          if (lane == 0) asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(mo), "l"(p.scales + idx) : "memory");
          if (lane == 1) asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(mo + 4), "l"(p.scales + per_kv + idx) : "memory");
        }
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int s = 0; s < kSimtStages; ++s) issue(s, s);

  const float base = p.softmax_scale * kLog2eS;
  for (int i = 0; i < ntiles; ++i) {
    const int s = i % kSimtStages;
    cp_async_wait<kSimtStages - 1>();
    __syncwarp();
    const uint32_t sb = ring + s * G::kStageBytes;
    const uint8_t* sp = ring_ptr + s * G::kStageBytes + 2 * G::kTileBytes;
    const bool valid = reinterpret_cast<const int*>(sp)[2] != 0;
    float kscale = 1.f, vscale = 1.f;
    if constexpr (is_blk8(KV)) {
      kscale = reinterpret_cast<const float*>(sp)[0];
      vscale = reinterpret_cast<const float*>(sp)[1];
    }
    const int t0 = t_begin + i * kSimtTile;
    const int n = valid ? min(kSimtTile, t_end - t0) : 0;
    const float mult = base * kscale;
    for (int j = 0; j < n; ++j) {
      float kx[EPL], vx[EPL];
      load_row<KV, D>(sb + j * G::kRow, lane, kx);
      load_row<KV, D>(sb + G::kTileBytes + j * G::kRow, lane, vx);
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        if (h >= group) continue;
        float d = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) d = fmaf(q[h][e], kx[e], d);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
        const float sc = d * mult;                           // log2 units
        const float mn = fmaxf(m[h], sc);
        const float a = exp2f(m[h] - mn), pw = exp2f(sc - mn);
        m[h] = mn;
        l[h] = l[h] * a + pw;
        const float pv = pw * vscale;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[h][e] = fmaf(o[h][e], a, pv * vx[e]);
      }
    }
    __syncwarp();
    issue(i + kSimtStages, s);
  }
  cp_async_wait<0>();

  // output (one partition) or this partition's (max, sum, O / sum)
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    if (h >= group) continue;
    const int64_t head = static_cast<int64_t>(b) * p.num_q_heads + kvh * group + h;
    const float inv = l[h] > 0.f ? 1.f / l[h] : 0.f;
    if (p.num_partitions == 1) {
      uint16_t* outp = static_cast<uint16_t*>(p.out) + head * D + EPL * lane;
#pragma unroll
      for (int e = 0; e < EPL; e += 2)
        *reinterpret_cast<uint32_t*>(outp + e) = Half16<QT>::pack_rn(o[h][e] * inv, o[h][e + 1] * inv);
    } else {
      const int64_t slot = head * p.num_partitions + part;
#pragma unroll
      for (int e = 0; e < EPL; ++e) p.ws_out[slot * D + EPL * lane + e] = o[h][e] * inv;
      if (lane == 0) {
        p.ws_ml[slot * 2] = m[h];
        p.ws_ml[slot * 2 + 1] = l[h];
      }
    }
  }
  pdl_launch_dependents();
}

template <int KV, int QT, int D>
cudaError_t launch_simt_t(const DecodeArgs& a, cudaStream_t st) {
  using G = SimtGeo<KV, D>;
  SimtParams p;
  p.q = static_cast<const uint16_t*>(a.q);
  p.k_cache = static_cast<const uint8_t*>(a.k_cache);
  p.v_cache = static_cast<const uint8_t*>(a.v_cache);
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.scales = static_cast<const float*>(a.scales);
  p.out = a.out;
  p.ws_out = a.ws_out;
  p.ws_ml = a.ws_ml;
  p.dev_status = a.dev_status;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_blocks = a.num_blocks;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.block_size = a.block_size;
  p.partition_size = a.partition_size;
  p.num_partitions = a.num_partitions;
  p.softmax_scale = a.softmax_scale;
  auto kern = simt_decode_kernel<KV, QT, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::kSmem);
  if (e != cudaSuccess) return e;
  const dim3 grid(a.num_partitions, (a.num_kv_heads + kSimtWarps - 1) / kSimtWarps, a.num_seqs);
  e = launch_pdl(kern, grid, dim3(kSimtWarps * kWarp), G::kSmem, st, p);
  if (e != cudaSuccess || a.num_partitions == 1) return e;
  return launch_lse_reduce(a, st);
}

template <int KV, int QT>
cudaError_t launch_simt_d(const DecodeArgs& a, cudaStream_t st) {
  return a.head_dim == 64 ? launch_simt_t<KV, QT, 64>(a, st) : launch_simt_t<KV, QT, 128>(a, st);
}

}  // namespace

// The SIMT comparator for 16-bit, FP8 and INT8 caches (no fused write);
// cudaErrorNotSupported for the rest.
cudaError_t launch_simt(const DecodeArgs& a, cudaStream_t st) {
  if (a.slot_mapping != nullptr) return cudaErrorNotSupported;
  switch (a.kv_dtype) {
    case PKV_F16: return launch_simt_d<PKV_F16, PKV_F16>(a, st);
    case PKV_BF16: return launch_simt_d<PKV_BF16, PKV_BF16>(a, st);
    case PKV_FP8_E4M3:
      return a.q_dtype == PKV_F16 ? launch_simt_d<PKV_FP8_E4M3, PKV_F16>(a, st)
                                  : launch_simt_d<PKV_FP8_E4M3, PKV_BF16>(a, st);
    case PKV_FP8_E5M2:
      return a.q_dtype == PKV_F16 ? launch_simt_d<PKV_FP8_E5M2, PKV_F16>(a, st)
                                  : launch_simt_d<PKV_FP8_E5M2, PKV_BF16>(a, st);
    case PKV_INT8:
      return a.q_dtype == PKV_F16 ? launch_simt_d<PKV_INT8, PKV_F16>(a, st)
                                  : launch_simt_d<PKV_INT8, PKV_BF16>(a, st);
    default:
      return cudaErrorNotSupported;
  }
}

}  // namespace pkv
