// Internal declarations shared by the library's translation units (not part of
// the public C ABI in include/kda.h).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// Codes written to the per-device error word (see kda_device_error()).
enum DeviceError : int32_t {
  kDevErrNone = 0,
  kDevErrBadSeqlens = 1,   // cu_seqlens not starting at 0, decreasing, or not ending at T
  kDevErrTimeout = 2,      // a bounded wait on an mbarrier ran out
  kDevErrNonFinite = 3,    // an output or final-state value came out inf or NaN (fp16 chain range exceeded)
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

// Sequence -> chunk map built on the device from cu_seqlens (or from B, T),
// plus where the state snapshots of each sequence go.
struct ChunkMap {
  int32_t* seq_chunk0;   // [num_seqs + 1] first global chunk of each sequence (exclusive scan)
  int4* chunk_info;      // [max_chunks] per global chunk: (sequence, rows, first token low, high word)
  int32_t* seq_order;    // [num_seqs] sequences by decreasing chunk count (the chain's launch order)
  int32_t max_chunks;    // upper bound used to size the grid
  // State snapshots (page "Kimi K3：架构、训练与百万 Token Agentic RL 技术解读" §9: the
  // recurrent state kept every 512 tokens for the prefix cache): with
  // snap_every > 0, the state after every snap_every full chunks of a sequence
  // is written to snaps [slot][H][d_k][d_v], slot = snap_slot0[s] + m - 1 for
  // the m-th snapshot of sequence s.
  float* snaps;
  int32_t* snap_slot0;   // [num_seqs + 1] first snapshot slot of each sequence (exclusive scan)
  int32_t snap_every;    // chunks between snapshots, 0 = none
};

// Snapshot slot of the state after local chunk i (0-based) of sequence s, whose
// length is len tokens, or -1 when no snapshot is taken there.
__device__ __forceinline__ int64_t snapshot_slot(const ChunkMap& m, int32_t s, int32_t i, int64_t len) {
  if (m.snap_every <= 0 || (i + 1) % m.snap_every != 0 || (int64_t)(i + 1) * kChunk > len) return -1;
  return (int64_t)m.snap_slot0[s] + (i + 1) / m.snap_every - 1;
}

// Where chunk j of the map lives in the packed token array.
struct ChunkPos {
  int32_t seq;
  int64_t t0;
  int32_t len;
};

__device__ __forceinline__ bool locate_chunk(const ChunkMap& m, const int32_t* cu, int32_t num_seqs, int64_t T_seq,
                                             int32_t j, ChunkPos& p) {
  (void)cu;
  (void)T_seq;
  if (j >= m.seq_chunk0[num_seqs]) return false;
  const int4 ci = m.chunk_info[j];
  p.seq = ci.x;
  p.len = ci.y;
  p.t0 = (int64_t)(((uint64_t)(uint32_t)ci.w << 32) | (uint32_t)ci.z);
  return p.len > 0;
}

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
  float* snaps;          // state snapshots or nullptr
  int32_t snap_every;    // chunks between snapshots (0 = none)
  const void* out_gate;       // output epilogue: gate logits [tokens][H][d_v] or nullptr (none)
  const float* norm_weight;   // its RMSNorm weight [H][d_v] or nullptr (ones)
  float eps_rms;
  int32_t decay_map;     // KDA_DECAY_BOUNDED or KDA_DECAY_SOFTPLUS (tensor-core path only)
  int32_t diag_pairs;    // nonzero: diagonal blocks of A and P by position pairs (tensor-core path only)
  int32_t* dev_err;
};

// Output epilogue of page "Kimi K3：架构、训练与百万 Token Agentic RL 技术解读" §3.2,
// applied before o is written: o = Sigmoid(gate) * o~ / sqrt(mean(o~^2) + eps) * w,
// per token and head over d_v.
struct OutEpilogue {
  const __nv_bfloat16* gate;   // [tokens][H][d_v] or nullptr (no epilogue)
  const float* weight;         // [H][d_v] or nullptr (ones)
  float eps;
};

// Workspace layout (all offsets 256-byte aligned).  `tc` selects the bf16
// tensor-core path (d_k = 128), whose per-(chunk, head) records are split into
// separate arrays so that each can be read with 2D TMA tiles.
struct Workspace {
  size_t bytes;
  size_t off_seq_chunk0, off_chunk_info, off_seq_order, off_snap_slot0, off_inter;
  int32_t max_chunks;
  size_t inter_bytes_per_chunk_head;
  bool tc;
  size_t off_wq, off_p, off_kt, off_u, off_gam;   // tensor-core path arrays
  size_t off_flags;                                // tensor-core path: int32 [R] record publication flags
};

// fp16 records of the tensor-core path, R = max_chunks * H records each.
struct TcRecords {
  __half* wq;           // [R][128][d_k]: rows 0-63 w = X Diag(beta)(k e^G), rows 64-127 q e^G
  __half* p;            // [R][64][64]:   P (inclusive lower triangle)
  __half* kt;           // [R][d_k][64]:  (k e^{G_last - G})^T, tokens contiguous
  __half* u;            // [R][64][d_v]:  u = X Diag(beta) V
  float* gam;           // [R][d_k]:      e^{G_last}
};
bool tc_path_supported(int32_t d_k, int32_t d_v, kda_dtype dt);
size_t tc_record_bytes(int32_t d_k, int32_t d_v);
cudaError_t launch_chunk_tc(const ChunkProblem& p, const Workspace& ws, const ChunkMap& map, char* base,
                            cudaStream_t stream);
Workspace chunk_workspace_layout(int64_t total_tokens, int32_t num_seqs, int32_t H, int32_t d_k, int32_t d_v,
                                 kda_dtype dt);

// Measurement hook: event pair around one launch when profiling is on.
// Device address of this device's error word.
cudaError_t device_error_ptr(int32_t** ptr);
void prof_begin(cudaStream_t s, const char* name);
void prof_end(cudaStream_t s);

cudaError_t launch_chunk_fwd(const ChunkProblem& p, const Workspace& ws, void* workspace, cudaStream_t stream);

cudaError_t launch_decode_step(const void* q, const void* k, const void* v, const void* g, const float* beta,
                               float* state, int32_t N, int32_t H, int32_t d_k, int32_t d_v, kda_dtype dt,
                               void* o, cudaStream_t stream);

// Fused decode layer step (validated by the API layer).
struct DecodeLayerProblem {
  const void* q_in;
  const void* k_in;
  const void* v_in;
  const void* z;
  const float* A_log;
  const float* beta_logit;
  void* conv_cache;
  const float* conv_weight;
  int32_t conv_width;
  float* state;
  const void* out_gate;
  const float* norm_weight;
  float eps_l2, eps_rms;
  int32_t N, H, d_k, d_v;
  kda_dtype dt;
  void* o;
};
cudaError_t launch_decode_layer(const DecodeLayerProblem& p, cudaStream_t stream);

}  // namespace kda
