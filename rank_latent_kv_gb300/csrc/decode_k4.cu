// Decode kernels whose key records have 4 hi octet(s) (key class 4), for
// every value class and both value storage kinds.
#include "decode_kernel.cuh"

namespace palu {

template <>
DecodeKernel decode_kernel_for<4>(int vc, bool vq) {
  switch (vc) {
    case 1: return vq ? latent_decode_kernel<4, 1, true> : latent_decode_kernel<4, 1, false>;
    case 2: return vq ? latent_decode_kernel<4, 2, true> : latent_decode_kernel<4, 2, false>;
    case 3: return vq ? latent_decode_kernel<4, 3, true> : latent_decode_kernel<4, 3, false>;
    case 4: return vq ? latent_decode_kernel<4, 4, true> : latent_decode_kernel<4, 4, false>;
    default: return nullptr;
  }
}

}  // namespace palu
