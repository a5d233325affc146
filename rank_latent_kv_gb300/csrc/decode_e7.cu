// Decode kernels for key records of exactly 7 octet(s), for value records of
// 1..8 octets (both storage kinds).
#include "decode_kernel.cuh"

namespace palu {

template <>
DecodeKernel decode_kernel_exact<7>(int ve, bool vq) {
  switch (ve) {
    case 1: return vq ? latent_decode_kernel<2, 1, true, 7, 1> : latent_decode_kernel<2, 1, false, 7, 1>;
    case 2: return vq ? latent_decode_kernel<2, 1, true, 7, 2> : latent_decode_kernel<2, 1, false, 7, 2>;
    case 3: return vq ? latent_decode_kernel<2, 1, true, 7, 3> : latent_decode_kernel<2, 1, false, 7, 3>;
    case 4: return vq ? latent_decode_kernel<2, 1, true, 7, 4> : latent_decode_kernel<2, 1, false, 7, 4>;
    case 5: return vq ? latent_decode_kernel<2, 2, true, 7, 5> : latent_decode_kernel<2, 2, false, 7, 5>;
    case 6: return vq ? latent_decode_kernel<2, 2, true, 7, 6> : latent_decode_kernel<2, 2, false, 7, 6>;
    case 7: return vq ? latent_decode_kernel<2, 2, true, 7, 7> : latent_decode_kernel<2, 2, false, 7, 7>;
    case 8: return vq ? latent_decode_kernel<2, 2, true, 7, 8> : latent_decode_kernel<2, 2, false, 7, 8>;
    default: return nullptr;
  }
}

}  // namespace palu
