// Decode kernels for key records of exactly 2 octet(s), for value records of
// 1..8 octets (both storage kinds).
#include "decode_kernel.cuh"

namespace palu {

template <>
DecodeKernel decode_kernel_exact<2>(int ve, bool vq) {
  switch (ve) {
    case 1: return vq ? latent_decode_kernel<1, 1, true, 2, 1> : latent_decode_kernel<1, 1, false, 2, 1>;
    case 2: return vq ? latent_decode_kernel<1, 1, true, 2, 2> : latent_decode_kernel<1, 1, false, 2, 2>;
    case 3: return vq ? latent_decode_kernel<1, 1, true, 2, 3> : latent_decode_kernel<1, 1, false, 2, 3>;
    case 4: return vq ? latent_decode_kernel<1, 1, true, 2, 4> : latent_decode_kernel<1, 1, false, 2, 4>;
    case 5: return vq ? latent_decode_kernel<1, 2, true, 2, 5> : latent_decode_kernel<1, 2, false, 2, 5>;
    case 6: return vq ? latent_decode_kernel<1, 2, true, 2, 6> : latent_decode_kernel<1, 2, false, 2, 6>;
    case 7: return vq ? latent_decode_kernel<1, 2, true, 2, 7> : latent_decode_kernel<1, 2, false, 2, 7>;
    case 8: return vq ? latent_decode_kernel<1, 2, true, 2, 8> : latent_decode_kernel<1, 2, false, 2, 8>;
    default: return nullptr;
  }
}

}  // namespace palu
