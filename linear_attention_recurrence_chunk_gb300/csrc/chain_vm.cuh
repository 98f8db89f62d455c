// Launcher of the value-major inter-chunk chain (kda_chain_vm.cu), called by
// the tensor-core prefill path once the per-(chunk, head) records are written.
#pragma once

#include <cuda.h>

#include "kda_internal.cuh"

namespace kda {

// One CTA per (sequence, head) over all d_v = 128 value columns, without the
// output epilogue (p.out_gate must be null).  The tensor maps are the records'
// 2D maps: [w; q e^G] boxes of 64 x 128, P of 64 x 64, (k e^{G_last - G})^T of
// 64 x 128, u of 64 x 64 (128-byte swizzle), e^{G_last} of 128 x 1; and the 3D
// map of o, [tokens][H][128] bf16, boxes of 64 values x 1 head x 64 tokens
// with 128-byte swizzle.
cudaError_t launch_chain_vm(const CUtensorMap& mWQ, const CUtensorMap& mP, const CUtensorMap& mKT,
                            const CUtensorMap& mU, const CUtensorMap& mGam, const CUtensorMap& mO,
                            const ChunkProblem& p, const ChunkMap& map, cudaStream_t stream);

}  // namespace kda
