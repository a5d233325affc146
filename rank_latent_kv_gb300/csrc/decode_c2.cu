// Decode kernels for key records of class 2 (ceil(octets / 4) = 2) that
// serve every octet count of their class; used when either side has more
// than 8 octets.
#include "decode_kernel.cuh"

namespace palu {

template <>
DecodeKernel decode_kernel_class<2>(int vc, bool vq) {
  switch (vc) {
    case 3: return vq ? latent_decode_kernel<2, 3, true, 0, 0> : latent_decode_kernel<2, 3, false, 0, 0>;
    case 4: return vq ? latent_decode_kernel<2, 4, true, 0, 0> : latent_decode_kernel<2, 4, false, 0, 0>;
    default: return nullptr;
  }
}

}  // namespace palu
