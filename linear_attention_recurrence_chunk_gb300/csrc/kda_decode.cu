// Fused single-token decode step of the KDA recurrence.
//
// Page "Kimi K3：架构、训练与百万 Token Agentic RL 技术解读" §3.2 gives the step as
// decay -> read -> write error -> read out:
//   S_bar = Diag(alpha) S,  v_hat = S_bar^T k,  S = S_bar + beta k (v - v_hat)^T,  o = S^T q.
// Since S^T q = S_bar^T q + (k.q) beta (v - v_hat), the read-out needs only the
// column sums S_bar^T k and S_bar^T q of the decayed state, so each state is
// read from HBM once and written once:
//   delta = beta (v - S_bar^T k),  o = S_bar^T q + (k.q) delta,  S = S_bar + k delta^T.
//
// One CTA per (sequence, head).  256 threads: a warp row of d_v/4 threads
// covers one state row with float4 accesses (512 B per row for d_v = 128), and
// the d_k rows are spread over the remaining thread dimension; every thread
// holds its d_k*d_v/1024 float4s in registers between the read and the write.
// The state streams through with evict-first hints (it is touched once per step).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kDecodeThreads = 256;

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(kDecodeThreads) decode_step_kernel(const T* __restrict__ q,
                                                                     const T* __restrict__ k,
                                                                     const T* __restrict__ v,
                                                                     const T* __restrict__ g,
                                                                     const float* __restrict__ beta,
                                                                     float* __restrict__ state,
                                                                     T* __restrict__ o) {
  constexpr int TX = DV / 4;                 // float4 columns of a state row
  constexpr int TY = kDecodeThreads / TX;    // rows processed side by side
  constexpr int RPT = DK / TY;               // rows per thread
  static_assert(RPT * TY == DK, "row split");

  __shared__ float s_k[DK], s_q[DK], s_alpha[DK];
  __shared__ __align__(16) float s_red[2][TY][DV];
  __shared__ __align__(16) float s_delta[DV];
  __shared__ float s_kq;

  const int64_t head = blockIdx.x;          // n * H + h
  const int tid = threadIdx.x;
  const int tx = tid % TX;
  const int ty = tid / TX;

  // Issue the state loads first: they do not depend on the token vectors.
  float4* st = reinterpret_cast<float4*>(state + head * DK * DV);
  float4 S[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) S[i] = __ldcs(st + (ty + i * TY) * TX + tx);

  for (int i = tid; i < DK; i += kDecodeThreads) {
    s_k[i] = to_f32(k[head * DK + i]);
    s_q[i] = to_f32(q[head * DK + i]);
    s_alpha[i] = expf(log_decay(to_f32(g[head * DK + i])));
  }
  __syncthreads();

  if (tid < 32) {  // k . q
    float acc = 0.f;
    for (int i = tid; i < DK; i += 32) acc += s_k[i] * s_q[i];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (tid == 0) s_kq = acc;
  }

  float4 vh = make_float4(0.f, 0.f, 0.f, 0.f), aq = vh;
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int row = ty + i * TY;
    const float al = s_alpha[row], kr = s_k[row], qr = s_q[row];
    S[i].x *= al; S[i].y *= al; S[i].z *= al; S[i].w *= al;
    vh.x += S[i].x * kr; vh.y += S[i].y * kr; vh.z += S[i].z * kr; vh.w += S[i].w * kr;
    aq.x += S[i].x * qr; aq.y += S[i].y * qr; aq.z += S[i].z * qr; aq.w += S[i].w * qr;
  }
  reinterpret_cast<float4*>(&s_red[0][ty][0])[tx] = vh;
  reinterpret_cast<float4*>(&s_red[1][ty][0])[tx] = aq;
  __syncthreads();

  if (tid < DV) {
    float vhat = 0.f, a = 0.f;
#pragma unroll
    for (int y = 0; y < TY; ++y) {
      vhat += s_red[0][y][tid];
      a += s_red[1][y][tid];
    }
    const float d = beta[head] * (to_f32(v[head * DV + tid]) - vhat);
    s_delta[tid] = d;
    o[head * DV + tid] = from_f32<T>(a + s_kq * d);
  }
  __syncthreads();

  const float4 d4 = reinterpret_cast<const float4*>(s_delta)[tx];
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const float kr = s_k[ty + i * TY];
    S[i].x += kr * d4.x; S[i].y += kr * d4.y; S[i].z += kr * d4.z; S[i].w += kr * d4.w;
    __stcs(st + (ty + i * TY) * TX + tx, S[i]);
  }
}

// ---------------------------------------------------------------------------
// Fused decode layer step: the token's input branches, the recurrence step and
// the output gate of page "Kimi K3：架构、训练与百万 Token Agentic RL 技术解读" §3.2-§3.3
// in one kernel, from the per-head projections of the token:
//   [q; k; v] = Swish(ShortConv([W_q x; W_k x; W_v x]))   (causal depthwise, width W,
//               the conv cache holds the W-1 previous inputs, oldest first)
//   q, k     <- L2Norm(q), L2Norm(k)
//   log alpha = -5 Sigmoid(e^{A^h} z),  beta = Sigmoid(beta logit)
//   the recurrence step above,  then optionally  o = Sigmoid(gate) * RMSNorm(o) * w.
// One CTA per (sequence, head) as above; threads take the 2 d_k + d_v conv
// channels while the state loads are in flight.
template <typename T>
struct LayerArgs {
  const T* q_in;
  const T* k_in;
  const T* v_in;
  const T* z;
  const float* A_log;
  const float* beta_logit;
  T* conv_cache;              // [N, H, W-1, 2 d_k + d_v]
  const float* conv_weight;   // [H, 2 d_k + d_v, W]
  int32_t W;
  float* state;
  const T* out_gate;          // [N, H, d_v] or nullptr
  const float* norm_weight;   // [H, d_v] or nullptr (ones)
  float eps_l2, eps_rms;
  int32_t H;
  T* o;
};

__device__ __forceinline__ float sigmoidf_(float x) { return 1.f / (1.f + expf(-x)); }

// Loads issued where they stand (the compiler may not sink them past the work
// that follows), for the per-token values of the layer step.
__device__ __forceinline__ float ld_f32_early(const float* p) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ float ld_early(const float* p) { return ld_f32_early(p); }
__device__ __forceinline__ float ld_early(const __nv_bfloat16* p) {
  unsigned short b;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(b) : "l"(p));
  return __uint_as_float((uint32_t)b << 16);
}

// Streaming (evict-first) 16-byte load issued where it stands: the compiler may
// not sink it past the front-end work that follows.
__device__ __forceinline__ float4 ld_cs_early(const float4* p) {
  float4 v;
  asm volatile("ld.global.cs.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
  return v;
}

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(kDecodeThreads) decode_layer_kernel(const LayerArgs<T> a) {
  constexpr int TX = DV / 4;
  constexpr int TY = kDecodeThreads / TX;
  constexpr int RPT = DK / TY;
  constexpr int CH = 2 * DK + DV;   // conv channels of a head: q, then k, then v
  static_assert(RPT * TY == DK, "row split");

  __shared__ float s_k[DK], s_q[DK], s_alpha[DK], s_v[DV];
  __shared__ __align__(16) float s_red[2][TY][DV];
  __shared__ __align__(16) float s_delta[DV];
  __shared__ float s_kq, s_scale[2], s_ss[DV / 32];

  const int64_t head = blockIdx.x;   // n * H + h
  const int h = (int)(head % a.H);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tx = tid % TX;
  const int ty = tid / TX;

  float4* st = reinterpret_cast<float4*>(a.state + head * DK * DV);
  float4 S[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) S[i] = ld_cs_early(st + (ty + i * TY) * TX + tx);

  // Every per-token value besides the state, issued up front: the gate input,
  // beta's logit, the output gate and its norm weight.
  const float zraw = tid < DK ? ld_early(a.z + head * DK + tid) : 0.f;
  const float blog = ld_f32_early(a.beta_logit + head);
  const float alog = ld_f32_early(a.A_log + h);
  float graw = 0.f, nwv = 1.f;
  if (tid < DV && a.out_gate) {
    graw = ld_early(a.out_gate + head * DV + tid);
    if (a.norm_weight) nwv = ld_f32_early(a.norm_weight + h * DV + tid);
  }

  // Input branches: conv over the cached inputs and the new one, cache shifted,
  // Swish.  Every load of the thread's channels (the input, up to kMaxConv - 1
  // cached inputs and kMaxConv taps each) is issued before any store.
  constexpr int kMaxConv = 8;
  constexpr int kChIter = (CH + kDecodeThreads - 1) / kDecodeThreads;
  const int W = a.W;
  T xr[kChIter], xv[kChIter][kMaxConv - 1];
  float wcur[kChIter], wp[kChIter][kMaxConv - 1];   // the current token's tap, the earlier taps
#pragma unroll
  for (int it = 0; it < kChIter; ++it) {
    const int c = tid + it * kDecodeThreads;
    const bool ok = c < CH;
    const int cs = ok ? c : 0;
    xr[it] = cs < DK ? a.q_in[head * DK + cs] : (cs < 2 * DK ? a.k_in[head * DK + cs - DK] : a.v_in[head * DV + cs - 2 * DK]);
    const float* wc = a.conv_weight + ((int64_t)h * CH + cs) * W;
    const T* cc = a.conv_cache + head * (int64_t)(W - 1) * CH + cs;
    wcur[it] = wc[W - 1];
#pragma unroll
    for (int j = 0; j < kMaxConv - 1; ++j) {
      const bool tap = ok && j < W - 1;
      wp[it][j] = tap ? wc[j] : 0.f;
      xv[it][j] = tap ? cc[(int64_t)j * CH] : T(0.f);
    }
  }
#pragma unroll
  for (int it = 0; it < kChIter; ++it) {
    const int c = tid + it * kDecodeThreads;
    if (c < CH) {
      float y = wcur[it] * to_f32(xr[it]);
#pragma unroll
      for (int j = 0; j < kMaxConv - 1; ++j) y += wp[it][j] * to_f32(xv[it][j]);   // zero beyond tap W - 2
      T* cc = a.conv_cache + head * (int64_t)(W - 1) * CH + c;
#pragma unroll
      for (int j = 1; j < kMaxConv - 1; ++j)
        if (j < W - 1) cc[(int64_t)(j - 1) * CH] = xv[it][j];
      if (W > 1) cc[(int64_t)(W - 2) * CH] = xr[it];
      const float act = y * sigmoidf_(y);
      if (c < DK) s_q[c] = act;
      else if (c < 2 * DK) s_k[c - DK] = act;
      else s_v[c - 2 * DK] = act;
    }
  }
  if (tid < DK) s_alpha[tid] = expf(-5.f * sigmoidf_(expf(alog) * zraw));
  __syncthreads();

  if (warp < 2) {   // L2Norm scales of q (warp 0) and k (warp 1)
    const float* x = warp == 0 ? s_q : s_k;
    float acc = 0.f;
    for (int i = lane; i < DK; i += 32) acc += x[i] * x[i];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) s_scale[warp] = rsqrtf(acc + a.eps_l2);
  }
  __syncthreads();
  for (int i = tid; i < DK; i += kDecodeThreads) {
    s_q[i] *= s_scale[0];
    s_k[i] *= s_scale[1];
  }
  __syncthreads();

  if (tid < 32) {   // k . q
    float acc = 0.f;
    for (int i = tid; i < DK; i += 32) acc += s_k[i] * s_q[i];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (tid == 0) s_kq = acc;
  }

  float4 vh = make_float4(0.f, 0.f, 0.f, 0.f), aq = vh;
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int row = ty + i * TY;
    const float al = s_alpha[row], kr = s_k[row], qr = s_q[row];
    S[i].x *= al; S[i].y *= al; S[i].z *= al; S[i].w *= al;
    vh.x += S[i].x * kr; vh.y += S[i].y * kr; vh.z += S[i].z * kr; vh.w += S[i].w * kr;
    aq.x += S[i].x * qr; aq.y += S[i].y * qr; aq.z += S[i].z * qr; aq.w += S[i].w * qr;
  }
  reinterpret_cast<float4*>(&s_red[0][ty][0])[tx] = vh;
  reinterpret_cast<float4*>(&s_red[1][ty][0])[tx] = aq;
  __syncthreads();

  float ov = 0.f;
  if (tid < DV) {
    float vhat = 0.f, acc = 0.f;
#pragma unroll
    for (int y = 0; y < TY; ++y) {
      vhat += s_red[0][y][tid];
      acc += s_red[1][y][tid];
    }
    const float d = sigmoidf_(blog) * (s_v[tid] - vhat);
    s_delta[tid] = d;
    ov = acc + s_kq * d;
  }
  if (a.out_gate) {   // RMSNorm over the head's d_v outputs, weight, Sigmoid gate
    if (tid < DV) {
      float sq = ov * ov;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
      if (lane == 0) s_ss[warp] = sq;
    }
    __syncthreads();
    if (tid < DV) {
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < DV / 32; ++w) tot += s_ss[w];
      ov = ov * rsqrtf(tot / DV + a.eps_rms) * nwv * sigmoidf_(graw);
    }
  }
  if (tid < DV) a.o[head * DV + tid] = from_f32<T>(ov);
  __syncthreads();

  const float4 d4 = reinterpret_cast<const float4*>(s_delta)[tx];
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const float kr = s_k[ty + i * TY];
    S[i].x += kr * d4.x; S[i].y += kr * d4.y; S[i].z += kr * d4.z; S[i].w += kr * d4.w;
    __stcs(st + (ty + i * TY) * TX + tx, S[i]);
  }
}

template <typename T>
cudaError_t launch_layer_typed(const LayerArgs<T>& a, int32_t N, int32_t d_k, int32_t d_v, cudaStream_t stream) {
  const dim3 grid((unsigned)((int64_t)N * a.H));
  prof_begin(stream, "decode_layer");
  if (d_k == 128 && d_v == 128)
    decode_layer_kernel<128, 128, T><<<grid, kDecodeThreads, 0, stream>>>(a);
  else if (d_k == 128 && d_v == 64)
    decode_layer_kernel<128, 64, T><<<grid, kDecodeThreads, 0, stream>>>(a);
  else if (d_k == 64 && d_v == 128)
    decode_layer_kernel<64, 128, T><<<grid, kDecodeThreads, 0, stream>>>(a);
  else
    decode_layer_kernel<64, 64, T><<<grid, kDecodeThreads, 0, stream>>>(a);
  prof_end(stream);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(const void* q, const void* k, const void* v, const void* g, const float* beta,
                         float* state, int32_t N, int32_t H, int32_t d_k, int32_t d_v, void* o,
                         cudaStream_t stream) {
  const dim3 grid((unsigned)((int64_t)N * H));
  const T* qq = static_cast<const T*>(q);
  const T* kk = static_cast<const T*>(k);
  const T* vv = static_cast<const T*>(v);
  const T* gg = static_cast<const T*>(g);
  T* oo = static_cast<T*>(o);
  prof_begin(stream, "decode_step");
  if (d_k == 128 && d_v == 128)
    decode_step_kernel<128, 128, T><<<grid, kDecodeThreads, 0, stream>>>(qq, kk, vv, gg, beta, state, oo);
  else if (d_k == 128 && d_v == 64)
    decode_step_kernel<128, 64, T><<<grid, kDecodeThreads, 0, stream>>>(qq, kk, vv, gg, beta, state, oo);
  else if (d_k == 64 && d_v == 128)
    decode_step_kernel<64, 128, T><<<grid, kDecodeThreads, 0, stream>>>(qq, kk, vv, gg, beta, state, oo);
  else
    decode_step_kernel<64, 64, T><<<grid, kDecodeThreads, 0, stream>>>(qq, kk, vv, gg, beta, state, oo);
  prof_end(stream);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_step(const void* q, const void* k, const void* v, const void* g, const float* beta,
                               float* state, int32_t N, int32_t H, int32_t d_k, int32_t d_v, kda_dtype dt,
                               void* o, cudaStream_t stream) {
  if (dt == KDA_F32) return launch_typed<float>(q, k, v, g, beta, state, N, H, d_k, d_v, o, stream);
  return launch_typed<__nv_bfloat16>(q, k, v, g, beta, state, N, H, d_k, d_v, o, stream);
}

cudaError_t launch_decode_layer(const DecodeLayerProblem& p, cudaStream_t stream) {
  if (p.dt == KDA_F32) {
    const LayerArgs<float> a{static_cast<const float*>(p.q_in), static_cast<const float*>(p.k_in),
                             static_cast<const float*>(p.v_in), static_cast<const float*>(p.z), p.A_log, p.beta_logit,
                             static_cast<float*>(p.conv_cache), p.conv_weight, p.conv_width, p.state,
                             static_cast<const float*>(p.out_gate), p.norm_weight, p.eps_l2, p.eps_rms, p.H,
                             static_cast<float*>(p.o)};
    return launch_layer_typed<float>(a, p.N, p.d_k, p.d_v, stream);
  }
  using B = __nv_bfloat16;
  const LayerArgs<B> a{static_cast<const B*>(p.q_in), static_cast<const B*>(p.k_in), static_cast<const B*>(p.v_in),
                       static_cast<const B*>(p.z), p.A_log, p.beta_logit, static_cast<B*>(p.conv_cache),
                       p.conv_weight, p.conv_width, p.state, static_cast<const B*>(p.out_gate), p.norm_weight,
                       p.eps_l2, p.eps_rms, p.H, static_cast<B*>(p.o)};
  return launch_layer_typed<B>(a, p.N, p.d_k, p.d_v, stream);
}

}  // namespace kda
