// Decode kernels for key and value records of exactly 10 octets (3 of
// 4-bit channels and 7 of 2-bit ones: ranks 66-75 at a hi fraction of 0.25,
// the long-context workload's rank 74 among them), so every record offset is
// a compile-time constant instead of the class kernels' run-time ones.
#include "decode_kernel.cuh"

namespace palu {

DecodeKernel decode_kernel_wide(int ke, int ve, int kc, int vc, bool vq) {
  if (ke == 10 && ve == 10 && kc == 3 && vc == 3)
    return vq ? latent_decode_kernel<3, 3, true, 10, 10> : latent_decode_kernel<3, 3, false, 10, 10>;
  return nullptr;
}

}  // namespace palu
