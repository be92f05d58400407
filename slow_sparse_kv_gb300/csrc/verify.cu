// Verification attention (Vegas): launcher and the head_dim 128 kernels; the
// head_dim 64 kernels are compiled in verify_d64.cu.  The kernel design is
// described in verify_impl.cuh.
#include "verify_impl.cuh"

namespace sfi {

cudaError_t launch_verify_d64(const VerifyArgs& va, int G, cudaStream_t st);

cudaError_t launch_verify(const VerifyArgs& va, int D, int G, cudaStream_t st) {
  if (D == 128) return launch_verify_d<128>(va, G, st);
  if (D == 64) return launch_verify_d64(va, G, st);
  return cudaErrorInvalidValue;
}

int verify_stage_rows() { return VerifyCfg<128>::SR; }

}  // namespace sfi
