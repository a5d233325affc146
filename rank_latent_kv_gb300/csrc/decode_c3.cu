// Decode kernels for key records of class 3 (ceil(octets / 4) = 3) that
// serve every octet count of their class; used when either side has more
// than 8 octets.
#include "decode_kernel.cuh"

namespace palu {

template <>
DecodeKernel decode_kernel_class<3>(int vc, bool vq) {
  switch (vc) {
    case 1: return vq ? latent_decode_kernel<3, 1, true, 0, 0> : latent_decode_kernel<3, 1, false, 0, 0>;
    case 2: return vq ? latent_decode_kernel<3, 2, true, 0, 0> : latent_decode_kernel<3, 2, false, 0, 0>;
    case 3: return vq ? latent_decode_kernel<3, 3, true, 0, 0> : latent_decode_kernel<3, 3, false, 0, 0>;
    case 4: return vq ? latent_decode_kernel<3, 4, true, 0, 0> : latent_decode_kernel<3, 4, false, 0, 0>;
    default: return nullptr;
  }
}

}  // namespace palu
