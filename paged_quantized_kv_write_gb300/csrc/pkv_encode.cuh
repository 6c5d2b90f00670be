// Quantize-on-write of one (token, KV head): the K row and the V row of one
// token for one KV head, encoded into the cache by one warp.  Shared by the
// write kernel and by the decode kernel's fused write.
//
// Lane l holds the EPL = head_dim/32 consecutive elements [EPL*l, EPL*l + EPL)
// of a row, so each row is read and written with one coalesced access.
// Encodings (the formats' definitions; block-wise FP8 scale from snippet-4
// of "Reducing LLM Inference Latency ... PagedAttention in vLLM"; INT4
// group-wise from section 4 of "Optimizing KV-Cache Memory Footprint"):
//  FP8  scale = max(amax / max_finite, 1e-12) (fp32; max_finite 448 for E4M3,
//       57344 for E5M2), amax over every token that the call opening the
//       block (writing its offset-0 slot) writes into it; later calls keep it;
//       code = cvt.rn.satfinite.{e4m3,e5m2}(x / scale), IEEE fp32 division.
//  INT8 the same block-wise rule with 127: code = clamp(rint(x / scale),
//       -127, 127), round half to even, two's complement byte.
//  INT4 per 32-element group: scale = fp16(fp32(max - min + 0) / 15),
//       zero = fp16(min + 0), code = clamp(rint((x - zero) / scale), 0, 15).
// Every fp32 step uses an explicitly rounded intrinsic so the codes are the
// same bits whatever the compiler contracts.
#pragma once

#include "pkv_common.cuh"

namespace pkv {

// Where a one-byte format's block scale comes from when a row is encoded.
enum ScaleSource {
  // The call writes one token into the block (the fused decode write): the
  // token at offset 0 opens the block with its own amax; others read the
  // stored scale.
  kScaleOwnRow = 0,
  // The write kernel's encode pass: the block's scale word holds either a
  // kept scale (sign bit clear) or, for a block this call opened, the open
  // mark 0x80000000 | bits(amax) of every row the call writes into it.  The
  // offset-0 token stores the finished scale; a row that meets the mark
  // finishes it the same way, so the order of the two does not matter.
  kScaleFromWord = 1,
};

constexpr uint32_t kOpenMark = 0x80000000u;

// max(amax / max_finite, 1e-12) in fp32, the block-wise rule of snippet-4.
template <int KV>
__device__ __forceinline__ float block_scale_from_amax(float amax) {
  return fmaxf(__fdiv_rn(amax, KV == PKV_INT8 ? 127.f : fp8_max<KV>()), 1e-12f);
}

// max |x| over the token's row for this head (a warp, EPL values per lane);
// NaN elements are passed over (fmaxf), as a plain max search does.
template <int NEW, int D>
__device__ __forceinline__ float row_amax(const uint16_t* __restrict__ src, int lane) {
  constexpr int EPL = D / kWarp;
  float amax = 0.f;
  if constexpr (EPL == 4) {
    const uint2 w = *reinterpret_cast<const uint2*>(src + lane * EPL);
    amax = fmaxf(fmaxf(fabsf(Half16<NEW>::to_float(w.x & 0xFFFF)),
                       fabsf(Half16<NEW>::to_float(w.x >> 16))),
                 fmaxf(fabsf(Half16<NEW>::to_float(w.y & 0xFFFF)),
                       fabsf(Half16<NEW>::to_float(w.y >> 16))));
  } else {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(src + lane * EPL);
    amax = fmaxf(fabsf(Half16<NEW>::to_float(w & 0xFFFF)), fabsf(Half16<NEW>::to_float(w >> 16)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  return amax;
}

// This lane's EPL = D/32 consecutive 16-bit values of a row, as 32-bit words.
template <int D>
struct RowWords {
  uint32_t w[D / kWarp / 2];
};
template <int D>
__device__ __forceinline__ RowWords<D> load_row_words(const uint16_t* __restrict__ src, int lane) {
  RowWords<D> r;
  if constexpr (D / kWarp == 4) {
    const uint2 v = *reinterpret_cast<const uint2*>(src + lane * 4);
    r.w[0] = v.x;
    r.w[1] = v.y;
  } else {
    r.w[0] = *reinterpret_cast<const uint32_t*>(src + lane * 2);
  }
  return r;
}

// The encoding of one (token, KV head) from this lane's words of its K and V
// rows (see encode_token_head).
template <int KV, int NEW, int D, int SRC = kScaleOwnRow>
__device__ __forceinline__ void encode_token_head_words(const RowWords<D>& kw,
                                                        const RowWords<D>& vw,
                                                        uint8_t* __restrict__ k_cache,
                                                        uint8_t* __restrict__ v_cache,
                                                        void* __restrict__ scales, int num_blocks,
                                                        int num_kv_heads, int block_size,
                                                        int64_t block, int head, int offset,
                                                        int lane) {
  constexpr int EPL = D / kWarp;                       // elements per lane: 2 or 4
  const int64_t cache_row = (block * num_kv_heads + head) * block_size + offset;
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const RowWords<D>& words = which ? vw : kw;
    uint8_t* cache = which ? v_cache : k_cache;
    uint16_t raw[EPL];
#pragma unroll
    for (int e = 0; e < EPL / 2; ++e) {
      raw[2 * e] = words.w[e] & 0xFFFF;
      raw[2 * e + 1] = words.w[e] >> 16;
    }

    if constexpr (KV == PKV_F16 || KV == PKV_BF16) {
      uint16_t* dst = reinterpret_cast<uint16_t*>(cache) + cache_row * D + lane * EPL;
      if constexpr (EPL == 4) {
        *reinterpret_cast<uint2*>(dst) =
            make_uint2(raw[0] | (uint32_t(raw[1]) << 16), raw[2] | (uint32_t(raw[3]) << 16));
      } else {
        *reinterpret_cast<uint32_t*>(dst) = raw[0] | (uint32_t(raw[1]) << 16);
      }
    } else if constexpr (is_blk8(KV)) {
      float x[EPL];
#pragma unroll
      for (int e = 0; e < EPL; ++e) x[e] = Half16<NEW>::to_float(raw[e]);
      float* sp = reinterpret_cast<float*>(scales) +
                  (static_cast<int64_t>(which) * num_blocks + block) * num_kv_heads + head;
      float s;
      if constexpr (SRC == kScaleFromWord) {
        uint32_t word = 0;
        if (lane == 0) word = __ldcg(reinterpret_cast<const unsigned int*>(sp));
        word = __shfl_sync(0xffffffffu, word, 0);
        s = (word & kOpenMark) ? block_scale_from_amax<KV>(__uint_as_float(word & ~kOpenMark))
                               : __uint_as_float(word);
        if (offset == 0 && lane == 0) *sp = s;
      } else if (offset == 0) {
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        s = block_scale_from_amax<KV>(amax);
        if (lane == 0) *sp = s;
      } else {
        s = *sp;
      }
      uint8_t* dst = cache + cache_row * D + lane * EPL;
      if constexpr (KV == PKV_INT8) {
        uint32_t codes = 0;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          const float r = rintf(__fdiv_rn(x[e], s));
          const float c = r == r ? fminf(fmaxf(r, -127.f), 127.f) : 0.f;   // NaN -> 0
          codes |= (static_cast<uint32_t>(static_cast<int>(c)) & 0xFFu) << (8 * e);
        }
        if constexpr (EPL == 4) {
          *reinterpret_cast<uint32_t*>(dst) = codes;
        } else {
          *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(codes);
        }
      } else if constexpr (EPL == 4) {
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

// k_src / v_src: the token's rows for this head (D values of dtype NEW).
// block, offset: where the token goes; cache_row = (block * Hkv + head) * bs + offset.
template <int KV, int NEW, int D, int SRC = kScaleOwnRow>
__device__ __forceinline__ void encode_token_head(const uint16_t* __restrict__ k_src,
                                                  const uint16_t* __restrict__ v_src,
                                                  uint8_t* __restrict__ k_cache,
                                                  uint8_t* __restrict__ v_cache,
                                                  void* __restrict__ scales, int num_blocks,
                                                  int num_kv_heads, int block_size, int64_t block,
                                                  int head, int offset, int lane) {
  const RowWords<D> kw = load_row_words<D>(k_src, lane);
  const RowWords<D> vw = load_row_words<D>(v_src, lane);
  encode_token_head_words<KV, NEW, D, SRC>(kw, vw, k_cache, v_cache, scales, num_blocks,
                                           num_kv_heads, block_size, block, head, offset, lane);
}

}  // namespace pkv
