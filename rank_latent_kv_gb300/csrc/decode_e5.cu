// Decode kernels for key records of exactly 5 octet(s), for value records of
// 1..8 octets (both storage kinds).
#include "decode_kernel.cuh"

namespace palu {

template <>
DecodeKernel decode_kernel_exact<5>(int ve, bool vq) {
  switch (ve) {
    case 1: return vq ? latent_decode_kernel<2, 1, true, 5, 1> : latent_decode_kernel<2, 1, false, 5, 1>;
    case 2: return vq ? latent_decode_kernel<2, 1, true, 5, 2> : latent_decode_kernel<2, 1, false, 5, 2>;
    case 3: return vq ? latent_decode_kernel<2, 1, true, 5, 3> : latent_decode_kernel<2, 1, false, 5, 3>;
    case 4: return vq ? latent_decode_kernel<2, 1, true, 5, 4> : latent_decode_kernel<2, 1, false, 5, 4>;
    case 5: return vq ? latent_decode_kernel<2, 2, true, 5, 5> : latent_decode_kernel<2, 2, false, 5, 5>;
    case 6: return vq ? latent_decode_kernel<2, 2, true, 5, 6> : latent_decode_kernel<2, 2, false, 5, 6>;
    case 7: return vq ? latent_decode_kernel<2, 2, true, 5, 7> : latent_decode_kernel<2, 2, false, 5, 7>;
    case 8: return vq ? latent_decode_kernel<2, 2, true, 5, 8> : latent_decode_kernel<2, 2, false, 5, 8>;
    default: return nullptr;
  }
}

}  // namespace palu
