// Decode kernels for key records of exactly 8 octet(s), for value records of
// 1..8 octets (both storage kinds).
#include "decode_kernel.cuh"

namespace palu {

template <>
DecodeKernel decode_kernel_exact<8>(int ve, bool vq) {
  switch (ve) {
    case 1: return vq ? latent_decode_kernel<2, 1, true, 8, 1> : latent_decode_kernel<2, 1, false, 8, 1>;
    case 2: return vq ? latent_decode_kernel<2, 1, true, 8, 2> : latent_decode_kernel<2, 1, false, 8, 2>;
    case 3: return vq ? latent_decode_kernel<2, 1, true, 8, 3> : latent_decode_kernel<2, 1, false, 8, 3>;
    case 4: return vq ? latent_decode_kernel<2, 1, true, 8, 4> : latent_decode_kernel<2, 1, false, 8, 4>;
    case 5: return vq ? latent_decode_kernel<2, 2, true, 8, 5> : latent_decode_kernel<2, 2, false, 8, 5>;
    case 6: return vq ? latent_decode_kernel<2, 2, true, 8, 6> : latent_decode_kernel<2, 2, false, 8, 6>;
    case 7: return vq ? latent_decode_kernel<2, 2, true, 8, 7> : latent_decode_kernel<2, 2, false, 8, 7>;
    case 8: return vq ? latent_decode_kernel<2, 2, true, 8, 8> : latent_decode_kernel<2, 2, false, 8, 8>;
    default: return nullptr;
  }
}

}  // namespace palu
