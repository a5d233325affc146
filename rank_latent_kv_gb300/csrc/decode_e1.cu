// Decode kernels for key records of exactly 1 octet(s), for value records of
// 1..8 octets (both storage kinds).
#include "decode_kernel.cuh"

namespace palu {

template <>
DecodeKernel decode_kernel_exact<1>(int ve, bool vq) {
  switch (ve) {
    case 1: return vq ? latent_decode_kernel<1, 1, true, 1, 1> : latent_decode_kernel<1, 1, false, 1, 1>;
    case 2: return vq ? latent_decode_kernel<1, 1, true, 1, 2> : latent_decode_kernel<1, 1, false, 1, 2>;
    case 3: return vq ? latent_decode_kernel<1, 1, true, 1, 3> : latent_decode_kernel<1, 1, false, 1, 3>;
    case 4: return vq ? latent_decode_kernel<1, 1, true, 1, 4> : latent_decode_kernel<1, 1, false, 1, 4>;
    case 5: return vq ? latent_decode_kernel<1, 2, true, 1, 5> : latent_decode_kernel<1, 2, false, 1, 5>;
    case 6: return vq ? latent_decode_kernel<1, 2, true, 1, 6> : latent_decode_kernel<1, 2, false, 1, 6>;
    case 7: return vq ? latent_decode_kernel<1, 2, true, 1, 7> : latent_decode_kernel<1, 2, false, 1, 7>;
    case 8: return vq ? latent_decode_kernel<1, 2, true, 1, 8> : latent_decode_kernel<1, 2, false, 1, 8>;
    default: return nullptr;
  }
}

}  // namespace palu
