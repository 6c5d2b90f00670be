// Decode attention for 16-bit caches (F16, BF16): the instantiations of the decode
// kernel's launch side (pkv_decode_launch.cuh) for this family.
#include "pkv_decode_launch.cuh"

namespace pkv {

cudaError_t launch_decode_half(const DecodeArgs& a, cudaStream_t st) {
  return a.kv_dtype == PKV_F16 ? launch_d<PKV_F16, PKV_F16>(a, st)
                               : launch_d<PKV_BF16, PKV_BF16>(a, st);
}

}  // namespace pkv
