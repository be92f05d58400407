// Warp-aggregated shared-memory histogram update of the selector kernels.
// Score distributions are very skewed (many lanes hit the same bin), so the
// lanes of a warp that share a bin add their count with one atomic from the
// lowest of them.
#pragma once

#include "common.cuh"

namespace sfi {

// Every lane of the warp must call this (active or not).
__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t bin, bool active) {
  const unsigned m = __ballot_sync(kFull, active);
  if (active) {
    const unsigned peers = __match_any_sync(m, bin);
    const int leader = __ffs(peers) - 1;
    if ((threadIdx.x & 31) == leader) atomicAdd(hist + bin, uint32_t(__popc(peers)));
  }
}

}  // namespace sfi
