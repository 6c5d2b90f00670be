// Decode attention for one-byte caches (FP8 E4M3, FP8 E5M2, INT8): the instantiations of the decode
// kernel's launch side (pkv_decode_launch.cuh) for this family.
#include "pkv_decode_launch.cuh"

namespace pkv {

cudaError_t launch_decode_byte(const DecodeArgs& a, cudaStream_t st) {
  const bool f16q = a.q_dtype == PKV_F16;
  switch (a.kv_dtype) {
    case PKV_FP8_E4M3:
      return f16q ? launch_d<PKV_FP8_E4M3, PKV_F16>(a, st) : launch_d<PKV_FP8_E4M3, PKV_BF16>(a, st);
    case PKV_FP8_E5M2:
      return f16q ? launch_d<PKV_FP8_E5M2, PKV_F16>(a, st) : launch_d<PKV_FP8_E5M2, PKV_BF16>(a, st);
    default:
      return f16q ? launch_d<PKV_INT8, PKV_F16>(a, st) : launch_d<PKV_INT8, PKV_BF16>(a, st);
  }
}

}  // namespace pkv
