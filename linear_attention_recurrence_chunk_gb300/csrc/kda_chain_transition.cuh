// Launcher of the 32-column inter-chunk pass with the output epilogue, in
// transition form (kda_chain_transition.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "kda_internal.cuh"

namespace kda {

// Enqueues the gated chain over the records of the prep kernel: one CTA per
// (sequence, head, 32 value columns), the DV/32 CTAs of a head one thread-block
// cluster; p.out_gate must be set.  The tensor maps are those of the records:
// [w; q e^G] (64 x 128 boxes), P (64 x 64), K~^T (64 x 128), u (32 x 64,
// 64-byte swizzle) and e^{G_last} (128 x 1).
cudaError_t launch_chain_transition_gated(const CUtensorMap& mWQ, const CUtensorMap& mP, const CUtensorMap& mKT,
                                          const CUtensorMap& mU, const CUtensorMap& mGam, const ChunkProblem& p,
                                          const ChunkMap& map, cudaStream_t stream);

}  // namespace kda
