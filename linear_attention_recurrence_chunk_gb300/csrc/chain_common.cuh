// Small device helpers shared by the tensor-core prefill kernels (prep and the
// inter-chunk chains): packing of fp32 pairs into 16-bit words, stores of
// 16-column row slices, the bounded-wait budget and the non-finite report.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "kda_internal.cuh"
#include "tc_ptx.cuh"

namespace kda {
namespace tcu {

constexpr long long kWaitLimit = 2000000000LL;   // ~1 s of SM clocks per bounded wait

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// V_new = u - w S for eight value columns: u as four fp16 pairs (one 16-byte
// load), w S as fp32 from TMEM.  w S is rounded to fp16 and the difference taken
// in packed fp16 arithmetic (round-to-nearest), two instructions per pair; the
// extra rounding of w S leaves the path's error unchanged (checked against the
// oracle by the CPU emulation of the rounding scheme).
__device__ __forceinline__ uint32_t sub_f16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint4 vnew_f16x8(uint4 u, const float* ws) {
  return make_uint4(sub_f16x2(u.x, pack_f16x2(ws[0], ws[1])), sub_f16x2(u.y, pack_f16x2(ws[2], ws[3])),
                    sub_f16x2(u.z, pack_f16x2(ws[4], ws[5])), sub_f16x2(u.w, pack_f16x2(ws[6], ws[7])));
}

// 16 fp32 values (value columns 16 hf .. 16 hf + 15) of K row `k` of an MN-major
// SW64 operand, as fp16, in two 16-byte stores.
__device__ __forceinline__ void store_mn_half(uint8_t* tile, int k, int hf, const float (&x)[16]) {
#pragma unroll
  for (int j = 0; j < 2; ++j)
    *reinterpret_cast<uint4*>(tile + tc::sw64_chunk_offset(k, 2 * hf + j)) =
        make_uint4(pack_f16x2(x[8 * j + 0], x[8 * j + 1]), pack_f16x2(x[8 * j + 2], x[8 * j + 3]),
                   pack_f16x2(x[8 * j + 4], x[8 * j + 5]), pack_f16x2(x[8 * j + 6], x[8 * j + 7]));
}

// 16 fp32 values as bf16 to global memory (two 16-byte stores).
__device__ __forceinline__ void store_bf16x16(__nv_bfloat16* dst, const float (&x)[16]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int j = 0; j < 2; ++j)
    d[j] = make_uint4(pack_bf16x2(x[8 * j + 0], x[8 * j + 1]), pack_bf16x2(x[8 * j + 2], x[8 * j + 3]),
                      pack_bf16x2(x[8 * j + 4], x[8 * j + 5]), pack_bf16x2(x[8 * j + 6], x[8 * j + 7]));
}

// Whole warp: records kDevErrNonFinite in the device error word (unless a code is
// already there) when any lane's accumulated x * 0 checks are not 0, i.e. some
// o or state value it wrote was inf or NaN (an fp16 operand of the chain out of
// range, or non-finite inputs).
__device__ __forceinline__ void report_nonfinite(float acc, int32_t* dev_err) {
  if (__any_sync(0xffffffffu, !(acc == 0.f)) && (threadIdx.x & 31) == 0)
    atomicCAS(dev_err, 0, (int32_t)kDevErrNonFinite);
}

}  // namespace tcu
}  // namespace kda
