// Instantiations of the split-K decode attention kernel for f32 caches
// (head_dim 64 and 128; 1, 2, 4 or 8 query heads per KV head).
#include "attn_kernel.cuh"

namespace sfi {

cudaError_t launch_attn_f32(const AttnArgs& a, int D, int G, cudaStream_t st, bool pdl) {
#define SFI_CASE(DD, GG) \
  if (D == DD && G == GG) return launch_attn_t<float, DD, GG>(a, st, pdl);
  SFI_CASE(64, 1) SFI_CASE(64, 2) SFI_CASE(64, 4) SFI_CASE(64, 8)
  SFI_CASE(128, 1) SFI_CASE(128, 2) SFI_CASE(128, 4) SFI_CASE(128, 8)
#undef SFI_CASE
  return cudaErrorInvalidValue;
}

int attn_stage_rows_f32(int D) {
  return D == 64 ? AttnCfg<float, 64, 4>::SR : AttnCfg<float, 128, 4>::SR;
}

}  // namespace sfi
