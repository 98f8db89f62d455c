// Value-major inter-chunk chain of the tensor-core prefill, for d_v = 128 (the
// plain call), as a kernel of its own: one CTA of 16 consumer warps per
// (sequence, head).  The device code and its design are in chain_vm_body.cuh.
#include "chain_vm.cuh"
#include "chain_vm_body.cuh"

namespace kda {
namespace {

using W16 = vm::VmWarps<16>;

__global__ void __launch_bounds__(W16::kThreads, 1)
    chunk_chain_vm_tc(const __grid_constant__ CUtensorMap tmWQ, const __grid_constant__ CUtensorMap tmP,
                      const __grid_constant__ CUtensorMap tmKT, const __grid_constant__ CUtensorMap tmU,
                      const __grid_constant__ CUtensorMap tmGam, const __grid_constant__ CUtensorMap tmO,
                      const int32_t* __restrict__ cu, int32_t num_seqs, int64_t T_seq, int32_t H, ChunkMap map,
                      const float* __restrict__ s0, float* __restrict__ s_final, vm::bf16* __restrict__ o,
                      int32_t* dev_err) {
  vm::chain_body<16>(tmWQ, tmP, tmKT, tmU, tmGam, tmO, cu, num_seqs, T_seq, H, map, s0, s_final, o, dev_err,
                     (int)blockIdx.x, nullptr);
}

}  // namespace

cudaError_t launch_chain_vm(const CUtensorMap& mWQ, const CUtensorMap& mP, const CUtensorMap& mKT,
                            const CUtensorMap& mU, const CUtensorMap& mGam, const CUtensorMap& mO,
                            const ChunkProblem& p, const ChunkMap& map, cudaStream_t stream) {
  if (p.d_v != vm::DV || p.d_k != vm::DK || p.out_gate) return cudaErrorInvalidValue;
  cudaError_t e =
      cudaFuncSetAttribute(chunk_chain_vm_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)vm::VmSmem::kAlloc);
  if (e != cudaSuccess) return e;
  prof_begin(stream, "chunk_chain_vm_tc");
  chunk_chain_vm_tc<<<(unsigned)p.num_seqs * (unsigned)p.H, W16::kThreads, vm::VmSmem::kAlloc, stream>>>(
      mWQ, mP, mKT, mU, mGam, mO, p.cu, p.num_seqs, p.T_seq, p.H, map, p.s0, p.s_final, static_cast<vm::bf16*>(p.o),
      p.dev_err);
  prof_end(stream);
  return cudaGetLastError();
}

}  // namespace kda
