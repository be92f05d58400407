// Verification attention (Vegas): the head_dim 64 kernels (see verify_impl.cuh).
#include "verify_impl.cuh"

namespace sfi {

cudaError_t launch_verify_d64(const VerifyArgs& va, int G, cudaStream_t st) {
  return launch_verify_d<64>(va, G, st);
}

}  // namespace sfi
