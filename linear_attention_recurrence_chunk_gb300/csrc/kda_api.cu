// C ABI of the KDA recurrence library: argument validation, workspace sizing,
// the per-device error word and dispatch to the kernel launchers.
#include <limits.h>
#include <stdint.h>

#include "kda_internal.cuh"

namespace {

// Per-device error word (one instance per device that loads the module).
__device__ int32_t g_kda_device_error = 0;

cudaError_t device_error_word(int32_t** ptr) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(ptr), g_kda_device_error);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

bool head_dims_supported(int32_t d_k, int32_t d_v) {
  return (d_k == 64 || d_k == 128) && (d_v == 64 || d_v == 128);
}

size_t dtype_bytes(kda_dtype dt) { return dt == KDA_F32 ? 4 : 2; }

// [a, a+na) and [b, b+nb) overlap (byte ranges; empty ranges never overlap)
bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// Shared shape checks of kda_chunk_fwd and its workspace query.
kda_status check_chunk_shape(int64_t B, int64_t T, int32_t H, int32_t d_k, int32_t d_v, int32_t num_seqs,
                             kda_dtype dt, bool varlen) {
  if (dt != KDA_F32 && dt != KDA_BF16) return KDA_ERR_INVALID_ARG;
  if (B < 0 || T < 0 || H <= 0 || num_seqs < 0) return KDA_ERR_INVALID_ARG;
  if (varlen ? (B != 1 || num_seqs < 1) : (num_seqs != B)) return KDA_ERR_INVALID_ARG;
  if (B * T > (int64_t)INT32_MAX - 1) return KDA_ERR_INVALID_ARG;
  if ((int64_t)num_seqs * H > (int64_t)INT32_MAX / 2 || H > 65535) return KDA_ERR_INVALID_ARG;
  if (!head_dims_supported(d_k, d_v)) return KDA_ERR_UNSUPPORTED;
  return KDA_OK;
}

// Measurement hook state (host side).
constexpr int kProfMax = 4096;
struct ProfRecord {
  const char* name;
  cudaEvent_t ev[2];
};
bool g_prof_on = false;
int g_prof_n = 0;          // timed records in use
int g_prof_launches = 0;   // launches seen since the last collect
ProfRecord g_prof[kProfMax] = {};

}  // namespace

namespace kda {

void prof_begin(cudaStream_t s, const char* name) {
  if (!g_prof_on) return;
  ++g_prof_launches;
  if (g_prof_n >= kProfMax) return;
  ProfRecord& r = g_prof[g_prof_n];
  if (!r.ev[0]) {
    if (cudaEventCreate(&r.ev[0]) != cudaSuccess || cudaEventCreate(&r.ev[1]) != cudaSuccess) return;
  }
  r.name = name;
  cudaEventRecord(r.ev[0], s);
}

void prof_end(cudaStream_t s) {
  if (!g_prof_on || g_prof_n >= kProfMax || !g_prof[g_prof_n].name) return;
  cudaEventRecord(g_prof[g_prof_n].ev[1], s);
  ++g_prof_n;
}

cudaError_t device_error_ptr(int32_t** ptr) { return device_error_word(ptr); }

}  // namespace kda

extern "C" {

const char* kda_status_string(kda_status s) {
  switch (s) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
    case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
    case KDA_ERR_DEVICE_TIMEOUT: return "KDA_ERR_DEVICE_TIMEOUT";
    case KDA_ERR_NONFINITE: return "KDA_ERR_NONFINITE";
  }
  return "KDA_ERR_UNKNOWN";
}

size_t kda_chunk_fwd_workspace_size(int64_t B, int64_t T, int32_t H, int32_t d_k, int32_t d_v, int32_t num_seqs,
                                    kda_dtype dt) {
  // The varlen form (B = 1, num_seqs sequences) and the batched form
  // (num_seqs = B) need the same space for the same total token count.
  const bool varlen = !(num_seqs == B);
  if (check_chunk_shape(B, T, H, d_k, d_v, num_seqs, dt, varlen) != KDA_OK) return SIZE_MAX;
  return kda::chunk_workspace_layout(B * T, num_seqs, H, d_k, d_v, dt).bytes;
}

}  // extern "C"

namespace {

// kda_chunk_fwd with optional state snapshots every snapshot_interval tokens
// (snapshots == nullptr and snapshot_interval == 0: none).
kda_status chunk_fwd_impl(const void* q, const void* k, const void* v, const void* g, const float* beta,
                          const float* initial_state, const int32_t* cu_seqlens, int32_t num_seqs, int64_t B,
                          int64_t T, int32_t H, int32_t d_k, int32_t d_v, kda_dtype dt, void* o,
                          float* final_state, float* snapshots, int32_t snapshot_interval,
                          int64_t snapshot_capacity, const void* out_gate, const float* norm_weight, float eps_rms,
                          void* workspace, size_t workspace_bytes, cudaStream_t stream,
                          int32_t decay_map = KDA_DECAY_BOUNDED, int32_t diag_pairs = 0) {
  const bool varlen = cu_seqlens != nullptr;
  kda_status st = check_chunk_shape(B, T, H, d_k, d_v, num_seqs, dt, varlen);
  if (st != KDA_OK) return st;
  const int64_t tokens = B * T;
  if (tokens > 0 && (!q || !k || !v || !g || !beta || !o)) return KDA_ERR_INVALID_ARG;
  if (!workspace) return KDA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, g, initial_state, o, final_state};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return KDA_ERR_INVALID_ARG;
  if ((beta && !aligned4(beta)) || (cu_seqlens && !aligned4(cu_seqlens))) return KDA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return KDA_ERR_INVALID_ARG;
  const kda::Workspace ws = kda::chunk_workspace_layout(tokens, num_seqs, H, d_k, d_v, dt);
  if (workspace_bytes < ws.bytes) return KDA_ERR_INVALID_ARG;

  // o must not overlap any input; the workspace must not overlap anything.
  const size_t eb = dtype_bytes(dt);
  const size_t nqk = (size_t)tokens * H * d_k * eb, nv = (size_t)tokens * H * d_v * eb;
  const size_t nb = (size_t)tokens * H * sizeof(float);
  const size_t ns = (size_t)num_seqs * H * d_k * d_v * sizeof(float);
  const size_t ncu = varlen ? sizeof(int32_t) * ((size_t)num_seqs + 1) : 0;
  struct Range { const void* p; size_t n; };
  const Range inputs[] = {{q, nqk}, {k, nqk}, {g, nqk}, {v, nv}, {beta, nb}, {initial_state, ns},
                          {cu_seqlens, ncu}};
  for (const Range& r : inputs) {
    if (overlaps(o, nv, r.p, r.n)) return KDA_ERR_INVALID_ARG;
    if (overlaps(final_state, ns, r.p, r.n) && r.p != initial_state) return KDA_ERR_INVALID_ARG;
    if (overlaps(workspace, ws.bytes, r.p, r.n)) return KDA_ERR_INVALID_ARG;
  }
  if (overlaps(o, nv, final_state, ns) || overlaps(workspace, ws.bytes, o, nv) ||
      overlaps(workspace, ws.bytes, final_state, ns))
    return KDA_ERR_INVALID_ARG;
  if (final_state && initial_state && final_state != initial_state && overlaps(final_state, ns, initial_state, ns))
    return KDA_ERR_INVALID_ARG;

  // Snapshots: every snapshot_interval tokens (a positive multiple of the
  // 64-token chunk) of each sequence; floor(T / interval) slots per batched
  // sequence, floor(total tokens / interval) bound the varlen total.
  if (snapshot_interval != 0 || snapshots) {
    if (snapshot_interval <= 0 || snapshot_interval % kda::kChunk != 0 || snapshot_capacity < 0)
      return KDA_ERR_INVALID_ARG;
    const int64_t need = varlen ? tokens / snapshot_interval : B * (T / snapshot_interval);
    if (snapshot_capacity < need || (need > 0 && !snapshots)) return KDA_ERR_INVALID_ARG;
    if (snapshots && !aligned16(snapshots)) return KDA_ERR_INVALID_ARG;
    const size_t nsnap = (size_t)snapshot_capacity * H * d_k * d_v * sizeof(float);
    const Range all[] = {{q, nqk}, {k, nqk}, {g, nqk}, {v, nv}, {beta, nb}, {initial_state, ns},
                         {cu_seqlens, ncu}, {o, nv}, {final_state, ns}, {workspace, ws.bytes}};
    for (const Range& r : all)
      if (overlaps(snapshots, nsnap, r.p, r.n)) return KDA_ERR_INVALID_ARG;
  }

  // Output epilogue: on the bf16 tensor-core path (d_k = 128) only.
  if (out_gate || norm_weight) {
    if (!out_gate) return KDA_ERR_INVALID_ARG;
    if (!kda::tc_path_supported(d_k, d_v, dt)) return KDA_ERR_UNSUPPORTED;
    if (!aligned16(out_gate) || (norm_weight && !aligned16(norm_weight))) return KDA_ERR_INVALID_ARG;
    if (!(eps_rms >= 0.f && eps_rms < 1e30f)) return KDA_ERR_INVALID_ARG;
    const Range gr[] = {{out_gate, nv}, {norm_weight, norm_weight ? (size_t)H * d_v * sizeof(float) : 0}};
    for (const Range& r : gr) {
      if (overlaps(o, nv, r.p, r.n) || overlaps(final_state, ns, r.p, r.n) || overlaps(workspace, ws.bytes, r.p, r.n))
        return KDA_ERR_INVALID_ARG;
      if (snapshots && overlaps(snapshots, (size_t)snapshot_capacity * H * d_k * d_v * sizeof(float), r.p, r.n))
        return KDA_ERR_INVALID_ARG;
    }
  }

  // Decay-map ablation: on the bf16 tensor-core path (d_k = 128) only; the
  // unbounded map needs the pair path for the diagonal blocks.
  if (decay_map != KDA_DECAY_BOUNDED && decay_map != KDA_DECAY_SOFTPLUS) return KDA_ERR_INVALID_ARG;
  if (diag_pairs != 0 && diag_pairs != 1) return KDA_ERR_INVALID_ARG;
  if (decay_map != KDA_DECAY_BOUNDED || diag_pairs) {
    if (!kda::tc_path_supported(d_k, d_v, dt)) return KDA_ERR_UNSUPPORTED;
    if (decay_map == KDA_DECAY_SOFTPLUS && !diag_pairs) return KDA_ERR_UNSUPPORTED;
  }

  if (num_seqs == 0) return KDA_OK;

  int32_t* dev_err = nullptr;
  if (device_error_word(&dev_err) != cudaSuccess) return KDA_ERR_CUDA;

  kda::ChunkProblem p{};
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta; p.s0 = initial_state;
  p.cu = cu_seqlens; p.num_seqs = num_seqs; p.T_seq = varlen ? 0 : T; p.total_tokens = tokens;
  p.H = H; p.d_k = d_k; p.d_v = d_v; p.dt = dt; p.o = o; p.s_final = final_state; p.dev_err = dev_err;
  p.snaps = snapshots;
  p.snap_every = snapshots ? snapshot_interval / kda::kChunk : 0;
  p.out_gate = out_gate;
  p.norm_weight = norm_weight;
  p.eps_rms = eps_rms;
  p.decay_map = decay_map;
  p.diag_pairs = diag_pairs;
  return kda::launch_chunk_fwd(p, ws, workspace, stream) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace

extern "C" {

kda_status kda_chunk_fwd(const void* q, const void* k, const void* v, const void* g, const float* beta,
                         const float* initial_state, const int32_t* cu_seqlens, int32_t num_seqs, int64_t B,
                         int64_t T, int32_t H, int32_t d_k, int32_t d_v, kda_dtype dt, void* o, float* final_state,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return chunk_fwd_impl(q, k, v, g, beta, initial_state, cu_seqlens, num_seqs, B, T, H, d_k, d_v, dt, o,
                        final_state, nullptr, 0, 0, nullptr, nullptr, 0.f, workspace, workspace_bytes, stream);
}

kda_status kda_chunk_fwd_gated(const void* q, const void* k, const void* v, const void* g, const float* beta,
                               const float* initial_state, const int32_t* cu_seqlens, int32_t num_seqs, int64_t B,
                               int64_t T, int32_t H, int32_t d_k, int32_t d_v, kda_dtype dt, void* o,
                               float* final_state, const void* out_gate, const float* norm_weight, float eps_rms,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!out_gate) return KDA_ERR_INVALID_ARG;
  return chunk_fwd_impl(q, k, v, g, beta, initial_state, cu_seqlens, num_seqs, B, T, H, d_k, d_v, dt, o,
                        final_state, nullptr, 0, 0, out_gate, norm_weight, eps_rms, workspace, workspace_bytes,
                        stream);
}

kda_status kda_chunk_fwd_decay_variant(const void* q, const void* k, const void* v, const void* g, const float* beta,
                                       const float* initial_state, const int32_t* cu_seqlens, int32_t num_seqs,
                                       int64_t B, int64_t T, int32_t H, int32_t d_k, int32_t d_v, kda_dtype dt,
                                       void* o, float* final_state, int32_t decay_map, int32_t diag_by_pairs,
                                       void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return chunk_fwd_impl(q, k, v, g, beta, initial_state, cu_seqlens, num_seqs, B, T, H, d_k, d_v, dt, o,
                        final_state, nullptr, 0, 0, nullptr, nullptr, 0.f, workspace, workspace_bytes, stream,
                        decay_map, diag_by_pairs);
}

kda_status kda_chunk_fwd_snapshots(const void* q, const void* k, const void* v, const void* g, const float* beta,
                                   const float* initial_state, const int32_t* cu_seqlens, int32_t num_seqs,
                                   int64_t B, int64_t T, int32_t H, int32_t d_k, int32_t d_v, kda_dtype dt, void* o,
                                   float* final_state, float* snapshots, int32_t snapshot_interval,
                                   int64_t snapshot_capacity, void* workspace, size_t workspace_bytes,
                                   cudaStream_t stream) {
  if (snapshot_interval <= 0) return KDA_ERR_INVALID_ARG;
  return chunk_fwd_impl(q, k, v, g, beta, initial_state, cu_seqlens, num_seqs, B, T, H, d_k, d_v, dt, o,
                        final_state, snapshots, snapshot_interval, snapshot_capacity, nullptr, nullptr, 0.f,
                        workspace, workspace_bytes, stream);
}

kda_status kda_decode_step(const void* q, const void* k, const void* v, const void* g, const float* beta,
                           float* state, int32_t N, int32_t H, int32_t d_k, int32_t d_v, kda_dtype dt, void* o,
                           cudaStream_t stream) {
  if (dt != KDA_F32 && dt != KDA_BF16) return KDA_ERR_INVALID_ARG;
  if (N < 0 || H <= 0) return KDA_ERR_INVALID_ARG;
  if ((int64_t)N * H > (int64_t)INT32_MAX) return KDA_ERR_INVALID_ARG;
  if (!head_dims_supported(d_k, d_v)) return KDA_ERR_UNSUPPORTED;
  if (N == 0) return KDA_OK;
  const void* ptrs[] = {q, k, v, g, state, o};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return KDA_ERR_INVALID_ARG;
  if (!beta || !aligned4(beta)) return KDA_ERR_INVALID_ARG;
  const size_t eb = dtype_bytes(dt), heads = (size_t)N * H;
  const size_t nqk = heads * d_k * eb, nv = heads * d_v * eb, ns = heads * d_k * d_v * sizeof(float);
  struct Range { const void* p; size_t n; };
  const Range others[] = {{q, nqk}, {k, nqk}, {g, nqk}, {v, nv}, {beta, heads * sizeof(float)}};
  for (const Range& r : others) {
    if (overlaps(o, nv, r.p, r.n) || overlaps(state, ns, r.p, r.n)) return KDA_ERR_INVALID_ARG;
  }
  if (overlaps(o, nv, state, ns)) return KDA_ERR_INVALID_ARG;
  return kda::launch_decode_step(q, k, v, g, beta, state, N, H, d_k, d_v, dt, o, stream) == cudaSuccess
             ? KDA_OK
             : KDA_ERR_CUDA;
}

kda_status kda_decode_layer_step(const void* q_in, const void* k_in, const void* v_in, const void* z,
                                 const float* A_log, const float* beta_logit, void* conv_cache,
                                 const float* conv_weight, int32_t conv_width, float* state, const void* out_gate,
                                 const float* norm_weight, float eps_l2, float eps_rms, int32_t N, int32_t H,
                                 int32_t d_k, int32_t d_v, kda_dtype dt, void* o, cudaStream_t stream) {
  if (dt != KDA_F32 && dt != KDA_BF16) return KDA_ERR_INVALID_ARG;
  if (N < 0 || H <= 0 || (int64_t)N * H > (int64_t)INT32_MAX) return KDA_ERR_INVALID_ARG;
  if (conv_width < 1 || conv_width > 8) return KDA_ERR_INVALID_ARG;
  if (!(eps_l2 >= 0.f && eps_l2 < 1e30f) || !(eps_rms >= 0.f && eps_rms < 1e30f)) return KDA_ERR_INVALID_ARG;
  if (!head_dims_supported(d_k, d_v)) return KDA_ERR_UNSUPPORTED;
  if (N == 0) return KDA_OK;
  const size_t eb = dtype_bytes(dt), heads = (size_t)N * H, ch = (size_t)2 * d_k + d_v;
  const bool need_cache = conv_width > 1;
  const void* req[] = {q_in, k_in, v_in, z, A_log, beta_logit, conv_weight, state, o};
  for (const void* p : req)
    if (!p) return KDA_ERR_INVALID_ARG;
  if (need_cache && !conv_cache) return KDA_ERR_INVALID_ARG;
  if (!aligned16(state)) return KDA_ERR_INVALID_ARG;
  const void* elem[] = {q_in, k_in, v_in, z, conv_cache, out_gate, o};
  for (const void* p : elem)
    if (p && (reinterpret_cast<uintptr_t>(p) % eb) != 0) return KDA_ERR_INVALID_ARG;
  const void* f32s[] = {A_log, beta_logit, conv_weight, norm_weight};
  for (const void* p : f32s)
    if (p && !aligned4(p)) return KDA_ERR_INVALID_ARG;
  struct Range { const void* p; size_t n; };
  const size_t nqk = heads * d_k * eb, nv = heads * d_v * eb, ns = heads * d_k * d_v * sizeof(float);
  const size_t ncache = need_cache ? heads * (size_t)(conv_width - 1) * ch * eb : 0;
  const Range reads[] = {{q_in, nqk}, {k_in, nqk}, {v_in, nv}, {z, nqk}, {A_log, (size_t)H * 4},
                         {beta_logit, heads * 4}, {conv_weight, (size_t)H * ch * conv_width * 4},
                         {out_gate, out_gate ? nv : 0}, {norm_weight, norm_weight ? (size_t)H * d_v * 4 : 0}};
  for (const Range& r : reads) {   // the three outputs overlap no input and no other output
    if (overlaps(o, nv, r.p, r.n) || overlaps(state, ns, r.p, r.n) || overlaps(conv_cache, ncache, r.p, r.n))
      return KDA_ERR_INVALID_ARG;
  }
  if (overlaps(o, nv, state, ns) || overlaps(o, nv, conv_cache, ncache) || overlaps(state, ns, conv_cache, ncache))
    return KDA_ERR_INVALID_ARG;
  kda::DecodeLayerProblem p{q_in, k_in, v_in, z, A_log, beta_logit, conv_cache, conv_weight, conv_width, state,
                            out_gate, norm_weight, eps_l2, eps_rms, N, H, d_k, d_v, dt, o};
  return kda::launch_decode_layer(p, stream) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_profile_enable(int32_t on) {
  g_prof_on = on != 0;
  return KDA_OK;
}

int32_t kda_profile_collect(char* names, float* ms, int32_t max_records) {
  const int32_t seen = g_prof_launches;
  for (int i = 0; i < g_prof_n; ++i) {
    ProfRecord& r = g_prof[i];
    if (i < max_records) {
      float t = -1.f;
      if (cudaEventSynchronize(r.ev[1]) != cudaSuccess || cudaEventElapsedTime(&t, r.ev[0], r.ev[1]) != cudaSuccess)
        t = -1.f;
      if (ms) ms[i] = t;
      if (names) {
        int j = 0;
        for (; j < 63 && r.name[j]; ++j) names[64 * i + j] = r.name[j];
        names[64 * i + j] = 0;
      }
    }
    r.name = nullptr;
  }
  g_prof_n = 0;
  g_prof_launches = 0;
  return seen;
}

kda_status kda_device_error(cudaStream_t stream, int32_t* code) {
  if (!code) return KDA_ERR_INVALID_ARG;
  int32_t* dev_err = nullptr;
  if (device_error_word(&dev_err) != cudaSuccess) return KDA_ERR_CUDA;
  int32_t h = 0;
  if (cudaMemcpyAsync(&h, dev_err, sizeof h, cudaMemcpyDeviceToHost, stream) != cudaSuccess) return KDA_ERR_CUDA;
  if (cudaMemsetAsync(dev_err, 0, sizeof h, stream) != cudaSuccess) return KDA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return KDA_ERR_CUDA;
  *code = h;
  if (h == 0) return KDA_OK;
  if (h == kda::kDevErrBadSeqlens) return KDA_ERR_INVALID_ARG;
  if (h == kda::kDevErrNonFinite) return KDA_ERR_NONFINITE;
  return KDA_ERR_DEVICE_TIMEOUT;
}

}  // extern "C"
