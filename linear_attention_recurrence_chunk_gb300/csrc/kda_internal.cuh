// Internal declarations shared by the library's translation units (not part of
// the public C ABI in include/kda.h).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// Codes written to the per-device error word (see kda_device_error()).
enum DeviceError : int32_t {
  kDevErrNone = 0,
  kDevErrBadSeqlens = 1,   // cu_seqlens not starting at 0, decreasing, or not ending at T
  kDevErrTimeout = 2,      // a bounded wait on an mbarrier ran out
};

// Chunk length of the prefill (tokens per chunk) and the sub-tile length whose
// cumulative log-decay stays within (-80, 0] because every log-decay is > -5.
constexpr int kChunk = 64;
constexpr int kSub = 16;

// The per-channel log-decay: g_min * Sigmoid(logit), g_min = -5.
__device__ __forceinline__ float log_decay(float logit) { return -5.0f / (1.0f + expf(-logit)); }

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Sequence -> chunk map built on the device from cu_seqlens (or from B, T).
struct ChunkMap {
  int32_t* seq_chunk0;   // [num_seqs + 1] first global chunk of each sequence (exclusive scan)
  int32_t* chunk_seq;    // [max_chunks] sequence of each global chunk
  int32_t max_chunks;    // upper bound used to size the grid
};

// Problem description handed to the launchers (validated by the API layer).
struct ChunkProblem {
  const void* q;
  const void* k;
  const void* v;
  const void* g;
  const float* beta;
  const float* s0;
  const int32_t* cu;     // device cu_seqlens or nullptr (then sequence s = [s*T, s*T+T))
  int32_t num_seqs;
  int64_t T_seq;         // tokens per sequence when cu == nullptr
  int64_t total_tokens;
  int32_t H, d_k, d_v;
  kda_dtype dt;
  void* o;
  float* s_final;
  int32_t* dev_err;
};

// Workspace layout (all offsets 256-byte aligned).
struct Workspace {
  size_t bytes;
  size_t off_seq_chunk0, off_chunk_seq, off_inter;
  int32_t max_chunks;
  size_t inter_bytes_per_chunk_head;
};
Workspace chunk_workspace_layout(int64_t total_tokens, int32_t num_seqs, int32_t H, int32_t d_k, int32_t d_v,
                                 kda_dtype dt);

// Measurement hook: event pair around one launch when profiling is on.
void prof_begin(cudaStream_t s, const char* name);
void prof_end(cudaStream_t s);

cudaError_t launch_chunk_fwd(const ChunkProblem& p, const Workspace& ws, void* workspace, cudaStream_t stream);

cudaError_t launch_decode_step(const void* q, const void* k, const void* v, const void* g, const float* beta,
                               float* state, int32_t N, int32_t H, int32_t d_k, int32_t d_v, kda_dtype dt,
                               void* o, cudaStream_t stream);

}  // namespace kda
