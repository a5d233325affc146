// Decode kernels for key records of exactly 3 octet(s), for value records of
// 1..8 octets (both storage kinds).
#include "decode_kernel.cuh"

namespace palu {

template <>
DecodeKernel decode_kernel_exact<3>(int ve, bool vq) {
  switch (ve) {
    case 1: return vq ? latent_decode_kernel<1, 1, true, 3, 1> : latent_decode_kernel<1, 1, false, 3, 1>;
    case 2: return vq ? latent_decode_kernel<1, 1, true, 3, 2> : latent_decode_kernel<1, 1, false, 3, 2>;
    case 3: return vq ? latent_decode_kernel<1, 1, true, 3, 3> : latent_decode_kernel<1, 1, false, 3, 3>;
    case 4: return vq ? latent_decode_kernel<1, 1, true, 3, 4> : latent_decode_kernel<1, 1, false, 3, 4>;
    case 5: return vq ? latent_decode_kernel<1, 2, true, 3, 5> : latent_decode_kernel<1, 2, false, 3, 5>;
    case 6: return vq ? latent_decode_kernel<1, 2, true, 3, 6> : latent_decode_kernel<1, 2, false, 3, 6>;
    case 7: return vq ? latent_decode_kernel<1, 2, true, 3, 7> : latent_decode_kernel<1, 2, false, 3, 7>;
    case 8: return vq ? latent_decode_kernel<1, 2, true, 3, 8> : latent_decode_kernel<1, 2, false, 3, 8>;
    default: return nullptr;
  }
}

}  // namespace palu
