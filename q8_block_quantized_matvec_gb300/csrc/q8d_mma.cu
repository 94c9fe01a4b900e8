// Tensor-core (tcgen05) path of q8d_matmul_small_m for m >= 9.
#include "q8d_internal.cuh"

namespace q8d {

int mma_small_m_launch(const float*, int, const uint8_t*, float*, int, int, int, int, cudaStream_t) {
  return Q8D_EUNSUPPORTED;
}

}  // namespace q8d
