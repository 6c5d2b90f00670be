// Device helpers shared by the write and decode kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedkv.h"

namespace pkv {

constexpr int kWarp = 32;

// ------------------------------------------------------------------ status
__device__ __forceinline__ void flag_status(int* dev_status, int code) {
  if (dev_status) atomicOr(dev_status, code);
}

// ------------------------------------------------------------------ 16-bit floats
template <int DT> struct Half16;
template <> struct Half16<PKV_F16> {
  using T = __half;
  using T2 = __half2;
  static __device__ __forceinline__ float to_float(uint16_t b) {
    return __half2float(__ushort_as_half(b));
  }
  static __device__ __forceinline__ uint32_t pack_rn(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  static __device__ __forceinline__ float2 unpack(uint32_t w) {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    return __half22float2(h);
  }
};
template <> struct Half16<PKV_BF16> {
  using T = __nv_bfloat16;
  using T2 = __nv_bfloat162;
  static __device__ __forceinline__ float to_float(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
  static __device__ __forceinline__ uint32_t pack_rn(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  static __device__ __forceinline__ float2 unpack(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  }
};

__device__ __forceinline__ float half_bits_to_float(uint16_t b, int dtype) {
  return dtype == PKV_F16 ? Half16<PKV_F16>::to_float(b) : Half16<PKV_BF16>::to_float(b);
}

// ------------------------------------------------------------------ FP8 E4M3
// Two fp32 values -> two E4M3 codes (round to nearest even, saturating to
// +-448).  Result: low byte = code of `lo`, high byte = code of `hi`.
__device__ __forceinline__ uint16_t e4m3x2_from_f32(float lo, float hi) {
  uint16_t r;
  // PTX: the first source operand lands in the upper byte.
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two E4M3 codes (low byte, high byte) -> f16x2 (exact: every E4M3 value is an f16).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t codes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(codes));
  return r;
}

// The same for OCP E5M2 (largest finite 57344; every E5M2 value is an f16).
__device__ __forceinline__ uint16_t e5m2x2_from_f32(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t e5m2x2_to_f16x2(uint16_t codes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(r) : "h"(codes));
  return r;
}

// FP8 cache formats, by dtype tag
__host__ __device__ constexpr bool is_fp8(int kv) { return kv == PKV_FP8_E4M3 || kv == PKV_FP8_E5M2; }
// one byte per element and one fp32 scale per (block, KV head): FP8 and INT8
__host__ __device__ constexpr bool is_blk8(int kv) { return is_fp8(kv) || kv == PKV_INT8; }
template <int KV> __device__ __forceinline__ float fp8_max() { return KV == PKV_FP8_E5M2 ? 57344.f : 448.f; }
template <int KV> __device__ __forceinline__ uint16_t fp8x2_from_f32(float lo, float hi) {
  if constexpr (KV == PKV_FP8_E5M2) return e5m2x2_from_f32(lo, hi);
  else return e4m3x2_from_f32(lo, hi);
}
template <int KV> __device__ __forceinline__ uint32_t fp8x2_to_f16x2(uint16_t codes) {
  if constexpr (KV == PKV_FP8_E5M2) return e5m2x2_to_f16x2(codes);
  else return e4m3x2_to_f16x2(codes);
}

// One-byte codes of a 32-bit word (bytes 0..3) as f16x2 operands, by format:
// FP8 converts exactly; INT8 codes x become (x + 128) 2^-24 (the XOR with
// 0x80 in b8_prep makes x + 128 an unsigned byte, which placed in the low
// mantissa bits of a zero-exponent f16 is that subnormal), so INT8 sums carry
// an offset of 128 per code that the caller takes off.
template <int KV> __device__ __forceinline__ uint32_t b8_prep(uint32_t w) {
  if constexpr (KV == PKV_INT8) return w ^ 0x80808080u;
  else return w;
}
// bytes 0, 1 of a prepared word
template <int KV> __device__ __forceinline__ uint32_t b8_lo(uint32_t w) {
  if constexpr (KV == PKV_INT8) return __byte_perm(w, 0u, 0x4140);
  else return fp8x2_to_f16x2<KV>(static_cast<uint16_t>(w & 0xFFFFu));
}
// bytes 2, 3 of a prepared word
template <int KV> __device__ __forceinline__ uint32_t b8_hi(uint32_t w) {
  if constexpr (KV == PKV_INT8) return __byte_perm(w, 0u, 0x4342);
  else return fp8x2_to_f16x2<KV>(static_cast<uint16_t>(w >> 16));
}

// ------------------------------------------------------------------ INT4
// Codes as f16 subnormals.  A nibble n placed in the low mantissa bits of an
// f16 with a zero exponent field is exactly n * 2^-24, so one AND turns two
// packed nibbles into an f16x2 operand with no offset to take off:
//   nib_lo: the nibbles at bits 0-3 and 16-19 of w -> n * 2^-24
//   nib_hi: the nibbles at bits 4-7 and 20-23      -> 16 n * 2^-24
// The products with them are exact in fp32; the caller undoes 2^24 (and the
// 16 of the high nibbles) once, after the sums.
__device__ __forceinline__ uint32_t nib_lo(uint32_t w) { return w & 0x000F000Fu; }
__device__ __forceinline__ uint32_t nib_hi(uint32_t w) { return w & 0x00F000F0u; }

// f16x2 product, round to nearest
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
// f16x2 a * b + c with one rounding
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  __half2 r = __hfma2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b),
                      *reinterpret_cast<__half2*>(&c));
  return *reinterpret_cast<uint32_t*>(&r);
}
// f16x2 negation (sign flip)
__device__ __forceinline__ uint32_t hneg2(uint32_t a) { return a ^ 0x80008000u; }

// ------------------------------------------------------------------ tensor cores
// D = A(16x16, row) * B(16x8, col) + D, fp32 accumulate (mma.sync m16n8k16).
template <int DT>
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4],
                                          uint32_t b0, uint32_t b1) {
  if constexpr (DT == PKV_BF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// Transpose an 8x8 matrix of 16-bit values held in the mma fragment layout
// (lane holds row lane/4, columns 2*(lane%4), +1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

// ------------------------------------------------------------------ dependent launches
// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may start while the previous kernel in the
// stream finishes; pdl_wait() blocks until that kernel has completed and its
// memory is visible (it returns at once when there is none).
// pdl_launch_dependents() lets the next such kernel begin launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch `kern` on `st` with programmatic stream serialization enabled.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ------------------------------------------------------------------ async copies
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async_16(uint32_t dst_smem, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst_smem), "l"(src)
               : "memory");
}
// the same, also allocating the line in L1
__device__ __forceinline__ void cp_async_16_ca(uint32_t dst_smem, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(dst_smem), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 ld_shared_v2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t ld_shared_b32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t ld_shared_u16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

// ldmatrix: 8x8 matrices of 16-bit values, one 16-byte row per lane address
// (lanes 8j..8j+7 give the rows of matrix j).  Without .trans lane l receives
// row l/4, columns 2(l%4), +1 of each matrix; with .trans, rows 2(l%4), +1 of
// column l/4.
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x2(uint32_t addr, uint32_t (&r)[2]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x2_trans(uint32_t addr, uint32_t (&r)[2]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr));
}

__device__ __forceinline__ uint4 ld_global_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

}  // namespace pkv
