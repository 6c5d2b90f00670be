// paged_kv_write: store new K/V rows at their physical slots, quantizing on
// the way in.
//
// One warp owns one (token, KV head) and handles K then V; lane l holds the
// EPL = head_dim/32 consecutive elements [EPL*l, EPL*l + EPL) of the row, so
// a warp reads and writes each row with one coalesced access.
//
// Encodings (the formats' definitions; block-wise FP8 scale from snippet-4
// of "Reducing LLM Inference Latency ... PagedAttention in vLLM"; INT4
// group-wise from section 4 of "Optimizing KV-Cache Memory Footprint"):
//  FP8  scale = max(amax / max_finite, 1e-12) (fp32; max_finite 448 for E4M3,
//       57344 for E5M2), set by the token at block offset 0;
//       code = cvt.rn.satfinite.{e4m3,e5m2}(x / scale), IEEE fp32 division.
//  INT4 per 32-element group: scale = fp16(fp32(max - min + 0) / 15),
//       zero = fp16(min + 0), code = clamp(rint((x - zero) / scale), 0, 15).
// Every fp32 step uses an explicitly rounded intrinsic so the codes are the
// same bits whatever the compiler contracts.
#include "pkv_common.cuh"
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
  constexpr int EPL = D / kWarp;                       // elements per lane: 2 or 4
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
  const int64_t cache_row = (block * num_kv_heads + head) * block_size + offset;

#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const uint16_t* src = (which ? v_new : k_new) + row * D + lane * EPL;
    uint8_t* cache = which ? v_cache : k_cache;
    uint16_t raw[EPL];
    if constexpr (EPL == 4) {
      uint2 w = *reinterpret_cast<const uint2*>(src);
      raw[0] = w.x & 0xFFFF; raw[1] = w.x >> 16; raw[2] = w.y & 0xFFFF; raw[3] = w.y >> 16;
    } else {
      uint32_t w = *reinterpret_cast<const uint32_t*>(src);
      raw[0] = w & 0xFFFF; raw[1] = w >> 16;
    }

    if constexpr (KV == PKV_F16 || KV == PKV_BF16) {
      uint16_t* dst = reinterpret_cast<uint16_t*>(cache) + cache_row * D + lane * EPL;
      if constexpr (EPL == 4) {
        *reinterpret_cast<uint2*>(dst) =
            make_uint2(raw[0] | (uint32_t(raw[1]) << 16), raw[2] | (uint32_t(raw[3]) << 16));
      } else {
        *reinterpret_cast<uint32_t*>(dst) = raw[0] | (uint32_t(raw[1]) << 16);
      }
    } else if constexpr (is_fp8(KV)) {
      float x[EPL];
#pragma unroll
      for (int e = 0; e < EPL; ++e) x[e] = Half16<NEW>::to_float(raw[e]);
      float* sp = reinterpret_cast<float*>(scales) +
                  (static_cast<int64_t>(which) * num_blocks + block) * num_kv_heads + head;
      float s;
      if (offset == 0) {
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        s = fmaxf(__fdiv_rn(amax, fp8_max<KV>()), 1e-12f);
        if (lane == 0) *sp = s;
      } else {
        s = *sp;
      }
      uint8_t* dst = cache + cache_row * D + lane * EPL;
      if constexpr (EPL == 4) {
        uint32_t lo = fp8x2_from_f32<KV>(__fdiv_rn(x[0], s), __fdiv_rn(x[1], s));
        uint32_t hi = fp8x2_from_f32<KV>(__fdiv_rn(x[2], s), __fdiv_rn(x[3], s));
        *reinterpret_cast<uint32_t*>(dst) = lo | (hi << 16);
      } else {
        *reinterpret_cast<uint16_t*>(dst) = fp8x2_from_f32<KV>(__fdiv_rn(x[0], s), __fdiv_rn(x[1], s));
      }
    } else {  // INT4_G32
      constexpr int LPG = 32 / EPL;                    // lanes per 32-element group
      float x[EPL];
#pragma unroll
      for (int e = 0; e < EPL; ++e) x[e] = Half16<NEW>::to_float(raw[e]);
      float mn = x[0], mx = x[0];
#pragma unroll
      for (int e = 1; e < EPL; ++e) { mn = fminf(mn, x[e]); mx = fmaxf(mx, x[e]); }
#pragma unroll
      for (int o = LPG / 2; o > 0; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      }
      const __half sh = __float2half_rn(__fdiv_rn(__fadd_rn(__fsub_rn(mx, mn), 0.0f), 15.0f));
      const __half zh = __float2half_rn(__fadd_rn(mn, 0.0f));
      const float sf = __half2float(sh), zf = __half2float(zh);
      uint32_t codes = 0;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        float c = 0.f;
        if (sf != 0.f) c = fminf(fmaxf(rintf(__fdiv_rn(__fsub_rn(x[e], zf), sf)), 0.f), 15.f);
        codes |= static_cast<uint32_t>(c) << (4 * e);
      }
      uint8_t* dst = cache + cache_row * (D / 2) + lane * (EPL / 2);
      if constexpr (EPL == 4) {
        *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(codes);
      } else {
        *dst = static_cast<uint8_t>(codes);
      }
      if ((lane % LPG) == 0) {
        const int group = lane / LPG;
        uint16_t* pair = reinterpret_cast<uint16_t*>(scales) +
                         2 * ((((static_cast<int64_t>(which) * num_blocks + block) * num_kv_heads +
                                head) * block_size + offset) * (D / 32) + group);
        const uint32_t packed = __half_as_ushort(sh) | (uint32_t(__half_as_ushort(zh)) << 16);
        *reinterpret_cast<uint32_t*>(pair) = packed;
      }
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
  if constexpr (is_fp8(KV)) {
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
