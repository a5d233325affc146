// Decode kernels for key records of exactly 6 octet(s), for value records of
// 1..8 octets (both storage kinds).
#include "decode_kernel.cuh"

namespace palu {

template <>
DecodeKernel decode_kernel_exact<6>(int ve, bool vq) {
  switch (ve) {
    case 1: return vq ? latent_decode_kernel<2, 1, true, 6, 1> : latent_decode_kernel<2, 1, false, 6, 1>;
    case 2: return vq ? latent_decode_kernel<2, 1, true, 6, 2> : latent_decode_kernel<2, 1, false, 6, 2>;
    case 3: return vq ? latent_decode_kernel<2, 1, true, 6, 3> : latent_decode_kernel<2, 1, false, 6, 3>;
    case 4: return vq ? latent_decode_kernel<2, 1, true, 6, 4> : latent_decode_kernel<2, 1, false, 6, 4>;
    case 5: return vq ? latent_decode_kernel<2, 2, true, 6, 5> : latent_decode_kernel<2, 2, false, 6, 5>;
    case 6: return vq ? latent_decode_kernel<2, 2, true, 6, 6> : latent_decode_kernel<2, 2, false, 6, 6>;
    case 7: return vq ? latent_decode_kernel<2, 2, true, 6, 7> : latent_decode_kernel<2, 2, false, 6, 7>;
    case 8: return vq ? latent_decode_kernel<2, 2, true, 6, 8> : latent_decode_kernel<2, 2, false, 6, 8>;
    default: return nullptr;
  }
}

}  // namespace palu
