// Decode attention for INT4 group-32 caches: the instantiations of the decode
// kernel's launch side (pkv_decode_launch.cuh) for this family.
#include "pkv_decode_launch.cuh"

namespace pkv {

cudaError_t launch_decode_int4(const DecodeArgs& a, cudaStream_t st) {
  return a.q_dtype == PKV_F16 ? launch_d<PKV_INT4_G32, PKV_F16>(a, st)
                              : launch_d<PKV_INT4_G32, PKV_BF16>(a, st);
}

}  // namespace pkv
