/*
 * kda.h -- C ABI of the KDA (Kimi Delta Attention) recurrence library for one
 * GB300 GPU (sm_103a).
 *
 * The operation (per sequence and head; S is d_k x d_v, rows = key channels):
 *
 *     log alpha_t = -5 * Sigmoid(g_t)                      (per key channel)
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t                                       (after the update)
 *
 * Sources: page "Kimi K3：架构、训练与百万 Token Agentic RL 技术解读", §3.1 (the KDA
 * equation; Diag(alpha) scales the rows of S), §3.2 (decay, read, write the
 * beta-weighted error, read out from the updated state; the single-token
 * interface (x_t, S_{t-1}) -> (y_t, S_t)), §3.3 (chunked prefill
 * (X_[c], S_in) -> (Y_[c], S_out) with S_in[c+1] = S_out[c]; the lower-bounded
 * decay with g_min = -5); page "Kimi K3 架构篇：一文详解 2.8 万亿参数的巨型怪兽",
 * sections "KDA 到底在算什么" and "最被低估的一个细节：下界衰减".
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller, dense and
 *    contiguous in the layouts given below, 16-byte aligned (beta and
 *    cu_seqlens: 4-byte aligned) unless an entry point states otherwise
 *    (kda_decode_layer_step needs 16 bytes for the state only).  The library
 *    allocates no memory; kda_chunk_fwd and its variants take their scratch
 *    space from the caller.
 *  - Calls are asynchronous on `stream` (0 = legacy default stream).  Argument
 *    errors are detected on the host and returned before anything is launched.
 *    A launch failure returns KDA_ERR_CUDA.  Conditions only the device can see
 *    (a malformed cu_seqlens array, a bounded device-side wait that ran out,
 *    an inf or NaN in the tensor-core prefill's outputs) set a per-device error
 *    word instead; read and clear it with kda_device_error() after the work has
 *    finished.
 *  - q and k are used as given (any L2 normalisation happens upstream); g is
 *    the raw decay logit (any per-head scale is already folded into it); beta is
 *    the write strength, already in (0, 1), as fp32.  No 1/sqrt(d_k) factor is
 *    applied to q.  o has the input dtype; states are always fp32.
 *    (kda_decode_layer_step instead starts from the token's projections and
 *    applies the conv, activations, norms and gate scale itself.)
 *  - Supported head sizes: d_k, d_v in {64, 128}; other values return
 *    KDA_ERR_UNSUPPORTED.
 */
#ifndef KDA_GB300_KDA_H
#define KDA_GB300_KDA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1,    /* bad pointer, size, alignment, alias or workspace */
  KDA_ERR_UNSUPPORTED = 2,    /* valid request outside what the kernels cover (head size) */
  KDA_ERR_CUDA = 3,           /* a CUDA runtime call or a launch failed */
  KDA_ERR_DEVICE_TIMEOUT = 4, /* a bounded device-side wait gave up (see kda_device_error) */
  KDA_ERR_NONFINITE = 5       /* an output or final state came out inf / NaN (see kda_device_error) */
} kda_status;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

/* Decay map of the gate logits g (kda_chunk_fwd_decay_variant):
 *  KDA_DECAY_BOUNDED   log alpha = -5 Sigmoid(g), the lower-bounded decay of page
 *                      "Kimi K3：架构、训练与百万 Token Agentic RL 技术解读" §3.3 (what
 *                      every other entry point applies);
 *  KDA_DECAY_SOFTPLUS  log alpha = -Softplus(g) = -ln(1 + e^g), the unbounded map of
 *                      the predecessor model that page "Kimi K3 架构篇：一文详解 2.8 万亿参数的
 *                      巨型怪兽" contrasts with the bound ("最被低估的一个细节：下界衰减"). */
typedef enum { KDA_DECAY_BOUNDED = 0, KDA_DECAY_SOFTPLUS = 1 } kda_decay_map;

/* Human-readable name of a status code (static string, never NULL). */
KDA_API const char* kda_status_string(kda_status s);

/*
 * Bytes of device scratch memory kda_chunk_fwd needs for this problem size
 * (same arguments as kda_chunk_fwd; with cu_seqlens, pass B = 1, T = total
 * packed tokens and num_seqs = number of sequences).  Returns SIZE_MAX when the
 * arguments are invalid or unsupported.
 */
KDA_API size_t kda_chunk_fwd_workspace_size(int64_t B, int64_t T, int32_t H, int32_t d_k, int32_t d_v,
                                    int32_t num_seqs, kda_dtype dt);

/*
 * Chunked prefill: runs the recurrence over whole sequences, chunk by chunk
 * (page "Kimi K3：架构、训练与百万 Token Agentic RL 技术解读" §3.3: intra-chunk work as
 * matrix products, the state passed only across chunk boundaries).
 *
 *  q, k, g   [B, T, H, d_k]   dtype dt (token-major, heads interleaved)
 *  v, o      [B, T, H, d_v]   dtype dt
 *  beta      [B, T, H]        fp32
 *  initial_state [S, H, d_k, d_v] fp32 (d_v contiguous) or NULL for zeros
 *  final_state   [S, H, d_k, d_v] fp32, or NULL when not wanted; it may be the
 *                same pointer as initial_state (updated in place)
 *  Without cu_seqlens: S = B = num_seqs sequences of T tokens each.
 *  With cu_seqlens (device int32[num_seqs + 1]): B must be 1, the T tokens are
 *    num_seqs packed sequences, sequence s covering tokens
 *    [cu_seqlens[s], cu_seqlens[s+1]); the array must start at 0, never
 *    decrease and end at T.  A malformed array is detected on the device: no
 *    output is written and kda_device_error() then reports
 *    KDA_ERR_INVALID_ARG.  Empty sequences are allowed.
 *  o must not overlap any input.  T = 0 (or an empty sequence) writes the
 *  initial state (or zeros) to final_state.
 *  workspace: device memory of at least kda_chunk_fwd_workspace_size(...)
 *  bytes, 256-byte aligned, owned by the caller; its contents on entry do not
 *  matter and on return are unspecified.  Two calls in flight at once need two
 *  workspaces.
 *  Range of the bf16 path with d_k = 128 (the tensor-core path): the chain's
 *  intermediates u = (I + A)^{-1} Diag(beta) V, V_new = u - w S, beta v and the
 *  copy of the state the tensor cores multiply are held in fp16, whose largest
 *  finite value is 65504.  On inputs like the benchmark's (unit-norm q, k)
 *  |u| and |V_new| reach about 1-2x max|v| and the state about |S_0| plus
 *  max|v|, so |v| and |S| must stay below about 3e4 (2e4 leaves margin).
 *  Beyond that a value becomes inf; the chain then reports
 *  KDA_ERR_NONFINITE through kda_device_error() (it checks every o and final
 *  state value it writes), and o / final_state hold inf or NaN.  fp32 inputs
 *  and d_k = 64 run in fp32 throughout and have no such limit.
 */
KDA_API kda_status kda_chunk_fwd(const void* q, const void* k, const void* v, const void* g, const float* beta,
                         const float* initial_state, const int32_t* cu_seqlens, int32_t num_seqs,
                         int64_t B, int64_t T, int32_t H, int32_t d_k, int32_t d_v, kda_dtype dt,
                         void* o, float* final_state, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream);

/*
 * Chunked prefill that also keeps the recurrent state every
 * `snapshot_interval` tokens of each sequence: the state snapshots that page
 * "Kimi K3：架构、训练与百万 Token Agentic RL 技术解读" §9 stores every 512 tokens so that a
 * prefix cache can resume a sequence at any such boundary without recomputing
 * it.  Arguments, layouts, results and errors are those of kda_chunk_fwd, plus:
 *  snapshots          device fp32 [slots][H][d_k][d_v] (d_v contiguous), owned by
 *                     the caller, 16-byte aligned, overlapping no other argument.
 *                     Snapshot m (m = 1 .. floor(len_s / snapshot_interval)) of
 *                     sequence s is the state after its first m * snapshot_interval
 *                     tokens, stored at slot first(s) + m - 1, where first(s) is the
 *                     number of snapshots of the sequences before s (sequence
 *                     order).  Without cu_seqlens that is slot
 *                     s * floor(T / snapshot_interval) + m - 1.  Slots beyond the
 *                     snapshots taken are not written.
 *  snapshot_interval  tokens between snapshots, a positive multiple of 64.
 *  snapshot_capacity  slots available in `snapshots`; must be at least
 *                     B * floor(T / snapshot_interval) (batched) or
 *                     floor(T / snapshot_interval) (cu_seqlens, an upper bound of
 *                     the total), else KDA_ERR_INVALID_ARG before anything is
 *                     launched.  `snapshots` may be NULL only when that bound is 0.
 * The snapshot at a sequence's last token (length a multiple of the interval)
 * equals its final state.  Uses the same workspace as kda_chunk_fwd.
 */
KDA_API kda_status kda_chunk_fwd_snapshots(const void* q, const void* k, const void* v, const void* g,
                                           const float* beta, const float* initial_state,
                                           const int32_t* cu_seqlens, int32_t num_seqs, int64_t B, int64_t T,
                                           int32_t H, int32_t d_k, int32_t d_v, kda_dtype dt, void* o,
                                           float* final_state, float* snapshots, int32_t snapshot_interval,
                                           int64_t snapshot_capacity, void* workspace, size_t workspace_bytes,
                                           cudaStream_t stream);

/*
 * Chunked prefill with the output epilogue of page "Kimi K3：架构、训练与百万 Token
 * Agentic RL 技术解读" §3.2 applied before o is written (the input of the output
 * projection W_o):  o = Sigmoid(out_gate) * o~ / sqrt(mean(o~^2) + eps_rms) * w,
 * per token and head over d_v, where o~ is kda_chunk_fwd's output.  Arguments,
 * layouts, results and errors are those of kda_chunk_fwd, plus:
 *  out_gate     [B, T, H, d_v] dtype dt (W_g x), 16-byte aligned, required;
 *  norm_weight  [H, d_v] fp32, 16-byte aligned, or NULL for ones;
 *  eps_rms      >= 0.
 * Supported on the bf16 path with d_k = 128 (d_v = 64 or 128); other head sizes
 * or fp32 inputs return KDA_ERR_UNSUPPORTED.  The RMS needs a token's whole
 * row, and the epilogue is always applied inside the inter-chunk pass before
 * o is written: where that pass holds all d_v columns of a head per CTA (many
 * heads) directly, else (few heads: 32 columns per CTA) the CTAs of a head run
 * as one thread-block cluster and exchange each row's partial sums of squares
 * through distributed shared memory.
 */
KDA_API kda_status kda_chunk_fwd_gated(const void* q, const void* k, const void* v, const void* g,
                                       const float* beta, const float* initial_state, const int32_t* cu_seqlens,
                                       int32_t num_seqs, int64_t B, int64_t T, int32_t H, int32_t d_k, int32_t d_v,
                                       kda_dtype dt, void* o, float* final_state, const void* out_gate,
                                       const float* norm_weight, float eps_rms, void* workspace,
                                       size_t workspace_bytes, cudaStream_t stream);

/*
 * Chunked prefill under a chosen decay map and diagonal-block path: the
 * ablation of the lower bound (page "Kimi K3 架构篇：一文详解 2.8 万亿参数的巨型怪兽",
 * "最被低估的一个细节：下界衰减": without a lower bound the factors e^{-G} inside a
 * 16-token tile leave the floating-point range, so the diagonal tiles have to be
 * formed pair by pair instead of on the tensor cores).  Arguments, layouts,
 * results and errors are those of kda_chunk_fwd, plus:
 *  decay_map      KDA_DECAY_BOUNDED or KDA_DECAY_SOFTPLUS (else KDA_ERR_INVALID_ARG);
 *  diag_by_pairs  0: the diagonal 16x16 blocks of the intra-chunk matrices on the
 *                 tensor cores (valid only with KDA_DECAY_BOUNDED, else
 *                 KDA_ERR_UNSUPPORTED); 1: each entry of those blocks summed over
 *                 the key channels on the CUDA cores with one exponential
 *                 e^{G_r - G_i} <= 1 per position pair and channel (any map);
 *                 other values: KDA_ERR_INVALID_ARG.
 * Supported on the bf16 path with d_k = 128 (d_v = 64 or 128); other head sizes
 * or fp32 inputs return KDA_ERR_UNSUPPORTED.  With KDA_DECAY_BOUNDED and
 * diag_by_pairs = 0 it is kda_chunk_fwd.  Logits above 8.8e29 are taken as
 * 8.8e29 under KDA_DECAY_SOFTPLUS (the decay factors they feed are 0 either way).
 */
KDA_API kda_status kda_chunk_fwd_decay_variant(const void* q, const void* k, const void* v, const void* g,
                                               const float* beta, const float* initial_state,
                                               const int32_t* cu_seqlens, int32_t num_seqs, int64_t B, int64_t T,
                                               int32_t H, int32_t d_k, int32_t d_v, kda_dtype dt, void* o,
                                               float* final_state, int32_t decay_map, int32_t diag_by_pairs,
                                               void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * One decode step for N independent sequences (one new token each), the
 * single-token interface of page "Kimi K3：架构、训练与百万 Token Agentic RL 技术解读"
 * §3.2 restricted to the recurrence: (q, k, v, g, beta, S_{t-1}) -> (o_t, S_t).
 *
 *  q, k, g [N, H, d_k] dtype dt;  v, o [N, H, d_v] dtype dt;  beta [N, H] fp32
 *  state   [N, H, d_k, d_v] fp32, read and overwritten in place with S_t.
 *  o must not overlap any input or the state.  N = 0 is a no-op.
 */
KDA_API kda_status kda_decode_step(const void* q, const void* k, const void* v, const void* g, const float* beta,
                           float* state, int32_t N, int32_t H, int32_t d_k, int32_t d_v, kda_dtype dt,
                           void* o, cudaStream_t stream);

/*
 * Fused decode step of a whole KDA layer from the token's per-head
 * projections, for N sequences (page "Kimi K3：架构、训练与百万 Token Agentic RL 技术解读"
 * §3.2: the interface (x_t, S_{t-1}, C^conv_{t-1}) -> (y_t, S_t, C^conv_t) and the
 * input branches; §3.3: the lower-bounded gate; §3.2: the gated output), up to
 * the output projection W_o:
 *   [q; k; v] = Swish(ShortConv([q_in; k_in; v_in]))  per channel, causal, width
 *               conv_width: y = sum_j w[j] x_{t-W+1+j} (tap W-1 on the current token)
 *   q, k      = q / sqrt(|q|^2 + eps_l2), k / sqrt(|k|^2 + eps_l2)
 *   log alpha = -5 Sigmoid(exp(A_log[h]) z),  beta = Sigmoid(beta_logit)
 *   S, o~     = the kda_decode_step recurrence on these
 *   o         = Sigmoid(out_gate) * o~ / sqrt(mean(o~^2) + eps_rms) * norm_weight
 *               (per head over d_v), or o = o~ when out_gate is NULL.
 *  q_in, k_in, z [N, H, d_k], v_in [N, H, d_v], out_gate [N, H, d_v]: dtype dt
 *      (the projections W_q x, W_k x, W_v x, the gate input z, W_g x);
 *  A_log [H], beta_logit [N, H]: fp32;
 *  conv_cache [N, H, conv_width - 1, 2 d_k + d_v] dtype dt, read and updated in
 *      place: the previous conv_width - 1 inputs of the q, k, v channels (in that
 *      order), oldest first; zeros for a new sequence; may be NULL when
 *      conv_width = 1;
 *  conv_weight [H, 2 d_k + d_v, conv_width] fp32;  conv_width in 1..8;
 *  state [N, H, d_k, d_v] fp32, 16-byte aligned, updated in place;
 *  norm_weight [H, d_v] fp32 or NULL (ones);  eps_l2, eps_rms >= 0;
 *  o [N, H, d_v] dtype dt.
 * Other arrays need their element alignment.  o, state and conv_cache overlap no
 * input and no one another.  N = 0 is a no-op.  Errors as kda_decode_step.
 */
KDA_API kda_status kda_decode_layer_step(const void* q_in, const void* k_in, const void* v_in, const void* z,
                                         const float* A_log, const float* beta_logit, void* conv_cache,
                                         const float* conv_weight, int32_t conv_width, float* state,
                                         const void* out_gate, const float* norm_weight, float eps_l2,
                                         float eps_rms, int32_t N, int32_t H, int32_t d_k, int32_t d_v,
                                         kda_dtype dt, void* o, cudaStream_t stream);

/*
 * Reads and clears this device's error word (on the current device), after
 * waiting for `stream`.  *code receives the raw word (0 = none).  Returns
 * KDA_OK when it was 0, KDA_ERR_INVALID_ARG for a malformed cu_seqlens,
 * KDA_ERR_DEVICE_TIMEOUT for a device-side wait that ran out,
 * KDA_ERR_NONFINITE when a tensor-core prefill wrote an inf or NaN output or
 * final state (the fp16 range of kda_chunk_fwd exceeded, or non-finite
 * inputs), KDA_ERR_CUDA if the read itself failed.  The word keeps the first
 * non-finite report and the last of the other codes.
 */
KDA_API kda_status kda_device_error(cudaStream_t stream, int32_t* code);

/*
 * Failure-detection check (the pages have no counterpart).  Launches one small
 * kernel on `stream` that waits on a shared-memory mbarrier nothing ever
 * arrives at, with the same bounded wait the tensor-core kernels use, limited
 * to `limit_cycles` SM clock cycles (1 .. 1e9).  When the limit runs out the
 * kernel sets this device's error word and returns, so that a following
 * kda_device_error() reports KDA_ERR_DEVICE_TIMEOUT and the CUDA context stays
 * usable.  Returns KDA_ERR_INVALID_ARG for a limit out of range (nothing is
 * launched) and KDA_ERR_CUDA if the launch fails.
 */
KDA_API kda_status kda_check_wait_timeout(int64_t limit_cycles, cudaStream_t stream);

/*
 * Allocation-free variant of kda_chunk_fwd (the pages have no counterpart).
 *
 * For callers that cannot call cudaMalloc, for example a serving engine that
 * reserves almost all device memory for its caches at start-up, or a plug-in
 * whose host owns the device allocator.  Arguments, layouts, results and
 * error behaviour are those of kda_chunk_fwd, except that there is no
 * workspace argument: the scratch space is a fixed array of
 * KDA_NOALLOC_SCRATCH_BYTES bytes that the library keeps in device memory on
 * every GPU that loads it, until the process exits.  The caller still
 * provides every input and output.
 *  - A problem whose kda_chunk_fwd_workspace_size(...) exceeds
 *    KDA_NOALLOC_SCRATCH_BYTES is rejected with KDA_ERR_INVALID_ARG before
 *    anything is launched.  The 64 MiB hold about 55,000 head-tokens on the
 *    bf16 tensor-core path (d_k = d_v = 128: one sequence of ~1,700 tokens at
 *    H = 32, ~57,000 at H = 1; each 64-token chunk of each head takes ~74 KB)
 *    and about 27,000 on the fp32 path at d = 128 (~830 tokens at H = 32).
 *    Larger problems need kda_chunk_fwd with a caller workspace.
 *  - The first call on a device looks up the array's device address with
 *    cudaGetSymbolAddress (on the current device) and caches it; make that
 *    first call before any stream capture.  The cache assumes the device's
 *    primary context for the life of the process: do not use this entry
 *    point on a device after cudaDeviceReset.
 *  - Nothing is allocated or freed by the call.
 *  - All calls share the one array: calls whose work overlaps on the GPU
 *    (other streams, other host threads) race on it and must not overlap.
 *    Its contents on entry do not matter.
 */
#define KDA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
KDA_API kda_status kda_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const void* g,
                                         const float* beta, const float* initial_state, const int32_t* cu_seqlens,
                                         int32_t num_seqs, int64_t B, int64_t T, int32_t H, int32_t d_k,
                                         int32_t d_v, kda_dtype dt, void* o, float* final_state,
                                         cudaStream_t stream);

/*
 * Measurement hook (the pages have no counterpart: it exists so that a
 * benchmark can time each kernel of a call on the stream it runs on).
 * kda_profile_enable(1) makes every later launch of this library record a
 * CUDA event pair around itself on its stream (at most 4096 pairs are kept;
 * later launches are counted but not timed); kda_profile_enable(0) stops it.
 * kda_profile_collect() waits for the recorded events, writes up to
 * max_records kernel names (NUL-terminated, 64 bytes each) and durations in
 * milliseconds, returns the number of launches seen since the last collect
 * (timed or not) and clears the record.  Host-side bookkeeping only; not
 * thread safe; the events are created once and reused.
 */
KDA_API kda_status kda_profile_enable(int32_t on);
KDA_API int32_t kda_profile_collect(char* names, float* ms, int32_t max_records);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_KDA_H */
