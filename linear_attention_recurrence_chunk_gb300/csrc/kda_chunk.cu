// Chunked prefill of the KDA recurrence: sequence->chunk map, intra-chunk
// preparation (gate, cumulative decay, UT/WY transform) and the inter-chunk
// state pass.  This file holds the fp32 SIMT instantiation; the bf16 tensor-core
// kernels live in kda_chunk_tc.cu and use the same workspace map.
//
// Page "Kimi K3：架构、训练与百万 Token Agentic RL 技术解读" §3.3 states the chunked
// form as (X_[c], S_in) -> (Y_[c], S_out) with the state handed from chunk to
// chunk, and the lower-bounded decay that keeps a 16-token tile's cumulative
// log-decay in (-80, 0).  Unrolling the §3.1 recurrence over one chunk of C
// tokens (rows r, state S_0 entering the chunk, G_r = inclusive cumulative
// log-decay from the chunk start, per key channel) gives, exactly:
//   A_ri   = beta_r (k_r * e^{G_r}) . (k_i * e^{-G_i})        for i < r
//   X      = (I + A)^{-1}                                      (unit lower triangular)
//   w      = X Diag(beta) (k * e^{G}),   u = X Diag(beta) V
//   V_new  = u - w S_0                                         (the beta-weighted errors)
//   O      = (q * e^{G}) S_0 + P V_new,  P_ri = (q_r * e^{G_r}) . (k_i * e^{-G_i}), i <= r
//   S_out  = Diag(e^{G_last}) S_0 + (k * e^{G_last - G})^T V_new
// Every factor e^{+-G} is taken relative to the start of the 16-row sub-tile of
// row r (block-row referencing): the row factor e^{G_r - G_ref} <= 1 and the
// column factor e^{G_ref - G_i} <= e^{80} for columns in the same sub-tile and
// <= 1 for earlier ones, which is the range argument of §3.3.
#include "kda_internal.cuh"

#include <algorithm>

namespace kda {

// ---------------------------------------------------------------------------
// Sequence -> chunk map (one CTA).  Validates cu_seqlens; on a malformed
// array it raises the device error word and maps zero chunks.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) chunk_map_kernel(const int32_t* __restrict__ cu, int32_t num_seqs,
                                                         int64_t T_seq, int64_t total, int32_t* seq_chunk0,
                                                         int4* chunk_info, int32_t* seq_order, int32_t max_chunks,
                                                         int32_t snap_every, int32_t* snap_slot0,
                                                         int32_t* dev_err) {
  __shared__ int32_t s_scan[1024];
  __shared__ int32_t s_carry;
  const int tid = threadIdx.x;
  int bad = 0;
  if (cu != nullptr) {
    if (tid == 0 && (cu[0] != 0 || (int64_t)cu[num_seqs] != total)) bad = 1;
    for (int s = tid; s < num_seqs; s += blockDim.x)
      if (cu[s + 1] < cu[s]) bad = 1;
  }
  bad = __syncthreads_or(bad);
  if (bad) {
    // zero chunks everywhere and a negative total: every later kernel of the
    // call sees the mark and writes nothing.
    if (tid == 0) atomicExch(dev_err, (int32_t)kDevErrBadSeqlens);
    for (int s = tid; s < num_seqs; s += blockDim.x) seq_chunk0[s] = 0;
    if (tid == 0) seq_chunk0[num_seqs] = -1;
    return;
  }
  // Exclusive scans over the sequences: pass 0 the chunk counts (-> seq_chunk0),
  // pass 1 the snapshot counts, floor(len / (64 snap_every)) (-> snap_slot0).
  int32_t n_chunks = 0;
  for (int pass = 0; pass < (snap_every > 0 ? 2 : 1); ++pass) {
    int32_t* dst = pass == 0 ? seq_chunk0 : snap_slot0;
    if (tid == 0) s_carry = 0;
    __syncthreads();
    for (int base = 0; base < num_seqs; base += blockDim.x) {
      const int s = base + tid;
      int32_t n = 0;
      if (s < num_seqs) {
        const int64_t len = cu ? (int64_t)(cu[s + 1] - cu[s]) : T_seq;
        n = pass == 0 ? (int32_t)((len + kChunk - 1) / kChunk) : (int32_t)(len / ((int64_t)kChunk * snap_every));
      }
      s_scan[tid] = n;
      __syncthreads();
      for (int off = 1; off < (int)blockDim.x; off <<= 1) {  // inclusive Hillis-Steele scan
        const int32_t add = tid >= off ? s_scan[tid - off] : 0;
        __syncthreads();
        s_scan[tid] += add;
        __syncthreads();
      }
      const int32_t start = s_carry + s_scan[tid] - n;
      if (s < num_seqs) dst[s] = start;
      __syncthreads();
      if (tid == blockDim.x - 1) s_carry += s_scan[tid];
      __syncthreads();
    }
    if (pass == 0) n_chunks = min(s_carry, max_chunks);
    else if (tid == 0) dst[num_seqs] = s_carry;
    __syncthreads();
  }
  if (tid == 0) seq_chunk0[num_seqs] = n_chunks;
  __syncthreads();
  // Per chunk: its sequence (the last s with seq_chunk0[s] <= j, which skips
  // empty sequences), row count and first token.
  for (int32_t j = tid; j < n_chunks; j += blockDim.x) {
    int32_t lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
      const int32_t mid = (lo + hi + 1) >> 1;
      if (seq_chunk0[mid] <= j) lo = mid;
      else hi = mid - 1;
    }
    const int64_t start = cu ? (int64_t)cu[lo] : (int64_t)lo * T_seq;
    const int64_t end = cu ? (int64_t)cu[lo + 1] : start + T_seq;
    const int64_t t0 = start + (int64_t)(j - seq_chunk0[lo]) * kChunk;
    chunk_info[j] = make_int4(lo, (int32_t)min((int64_t)kChunk, end - t0), (int32_t)(uint32_t)(uint64_t)t0,
                              (int32_t)(uint32_t)((uint64_t)t0 >> 32));
  }
  // Launch order of the sequential chains: longest first (ties by index), so
  // that the longest chains start in the first wave.  Beyond kRankedSeqs
  // sequences the order is the identity.
  constexpr int32_t kRankedSeqs = 4096;
  for (int32_t s = tid; s < num_seqs; s += blockDim.x) {
    int32_t rank = s;
    if (num_seqs <= kRankedSeqs) {
      const int32_t n = seq_chunk0[s + 1] - seq_chunk0[s];
      rank = 0;
      for (int32_t t = 0; t < num_seqs; ++t) {
        const int32_t nt = seq_chunk0[t + 1] - seq_chunk0[t];
        rank += (nt > n || (nt == n && t < s)) ? 1 : 0;
      }
    }
    seq_order[rank] = s;
  }
}

// Intermediate record of one (chunk, head) in the workspace (fp32 SIMT path).
template <int DK, int DV>
struct InterF32 {
  static constexpr int kW = 0;                       // w      [C][DK]
  static constexpr int kU = kW + kChunk * DK;        // u      [C][DV]
  static constexpr int kQh = kU + kChunk * DV;       // q*e^G  [C][DK]
  static constexpr int kKt = kQh + kChunk * DK;      // k*e^{G_last-G} [C][DK]
  static constexpr int kP = kKt + kChunk * DK;       // P      [C][C]
  static constexpr int kGamma = kP + kChunk * kChunk;  // e^{G_last} [DK]
  static constexpr int kFloats = kGamma + DK;
};

// ---------------------------------------------------------------------------
// Kernel (a)+(b), SIMT: one CTA per (chunk, head).
// ---------------------------------------------------------------------------
constexpr int kPrepThreads = 256;

template <int DK, int DV>
struct PrepSmem {
  static constexpr int LDK = DK + 1, LDV = DV + 1, LDC = kChunk + 1;
  static constexpr int oK = 0;
  static constexpr int oQ = oK + kChunk * LDK;
  static constexpr int oG = oQ + kChunk * LDK;
  static constexpr int oV = oG + kChunk * LDK;
  static constexpr int oKc = oV + kChunk * LDV;
  static constexpr int oKr = oKc + kChunk * LDK;
  static constexpr int oQr = oKr + kSub * LDK;
  static constexpr int oA = oQr + kSub * LDK;
  static constexpr int oX = oA + kChunk * LDC;
  static constexpr int oY = oX + kChunk * LDC;
  static constexpr int oBeta = oY + 3 * kSub * kSub;
  static constexpr int kFloats = oBeta + kChunk;
  static constexpr size_t kBytes = sizeof(float) * kFloats;
};

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(kPrepThreads) chunk_prep_simt(const T* __restrict__ q, const T* __restrict__ k,
                                                                const T* __restrict__ v, const T* __restrict__ g,
                                                                const float* __restrict__ beta,
                                                                const int32_t* __restrict__ cu, int32_t num_seqs,
                                                                int64_t T_seq, int32_t H, ChunkMap map,
                                                                float* __restrict__ inter) {
  using L = PrepSmem<DK, DV>;
  using R = InterF32<DK, DV>;
  constexpr int C = kChunk, LDK = L::LDK, LDV = L::LDV, LDC = L::LDC;
  extern __shared__ float sm[];
  float* sK = sm + L::oK;
  float* sQ = sm + L::oQ;
  float* sG = sm + L::oG;
  float* sV = sm + L::oV;
  float* sKc = sm + L::oKc;
  float* sKr = sm + L::oKr;
  float* sQr = sm + L::oQr;
  float* sA = sm + L::oA;
  float* sX = sm + L::oX;
  float* sY = sm + L::oY;
  float* sBeta = sm + L::oBeta;

  ChunkPos pos;
  if (!locate_chunk(map, cu, num_seqs, T_seq, blockIdx.x, pos)) return;
  const int h = blockIdx.y;
  const int tid = threadIdx.x;
  float* rec = inter + ((int64_t)blockIdx.x * H + h) * R::kFloats;

  // 1. load the chunk (rows past the sequence end are zero, with zero decay)
  for (int idx = tid; idx < C * DK; idx += kPrepThreads) {
    const int r = idx / DK, c = idx % DK;
    float kv = 0.f, qv = 0.f, lg = 0.f;
    if (r < pos.len) {
      const int64_t off = ((pos.t0 + r) * H + h) * DK + c;
      kv = to_f32(k[off]);
      qv = to_f32(q[off]);
      lg = log_decay(to_f32(g[off]));
    }
    sK[r * LDK + c] = kv;
    sQ[r * LDK + c] = qv;
    sG[r * LDK + c] = lg;
  }
  for (int idx = tid; idx < C * DV; idx += kPrepThreads) {
    const int r = idx / DV, c = idx % DV;
    sV[r * LDV + c] = r < pos.len ? to_f32(v[((pos.t0 + r) * H + h) * DV + c]) : 0.f;
  }
  for (int r = tid; r < C; r += kPrepThreads) sBeta[r] = r < pos.len ? beta[(pos.t0 + r) * H + h] : 0.f;
  for (int idx = tid; idx < C * LDC; idx += kPrepThreads) sX[idx] = 0.f;
  __syncthreads();

  // 2. inclusive cumulative log-decay within the chunk, per key channel
  for (int c = tid; c < DK; c += kPrepThreads) {
    float run = 0.f;
    for (int r = 0; r < C; ++r) {
      run += sG[r * LDK + c];
      sG[r * LDK + c] = run;
    }
  }
  __syncthreads();

  // 3. A (strictly lower, beta-weighted) and P (inclusive lower), one 16-row
  //    block-row at a time, referenced to the block-row's start.
  for (int a = 0; a < C / kSub; ++a) {
    const int r0 = a * kSub, ncols = r0 + kSub;
    for (int idx = tid; idx < ncols * DK; idx += kPrepThreads) {
      const int i = idx / DK, c = idx % DK;
      const float gref = a ? sG[(r0 - 1) * LDK + c] : 0.f;
      sKc[i * LDK + c] = sK[i * LDK + c] * expf(gref - sG[i * LDK + c]);
    }
    for (int idx = tid; idx < kSub * DK; idx += kPrepThreads) {
      const int rr = idx / DK, c = idx % DK;
      const float gref = a ? sG[(r0 - 1) * LDK + c] : 0.f;
      const float e = expf(sG[(r0 + rr) * LDK + c] - gref);
      sKr[rr * LDK + c] = sK[(r0 + rr) * LDK + c] * e;
      sQr[rr * LDK + c] = sQ[(r0 + rr) * LDK + c] * e;
    }
    __syncthreads();
    for (int p = tid; p < kSub * C; p += kPrepThreads) {
      const int rr = p / C, i = p % C, r = r0 + rr;
      float av = 0.f, pv = 0.f;
      if (i <= r) {
        float da = 0.f, dp = 0.f;
        for (int c = 0; c < DK; ++c) {
          const float kc = sKc[i * LDK + c];
          da += sKr[rr * LDK + c] * kc;
          dp += sQr[rr * LDK + c] * kc;
        }
        av = i < r ? sBeta[r] * da : 0.f;
        pv = dp;
      }
      sA[r * LDC + i] = av;
      rec[R::kP + r * C + i] = pv;
    }
    __syncthreads();
  }

  // 4. X = (I + A)^{-1} by blocked forward substitution.
  //    4a. the four 16x16 unit-lower diagonal blocks, one column per thread
  if (tid < C) {
    const int base = (tid / kSub) * kSub, j = tid % kSub;
    for (int r = j; r < kSub; ++r) {
      float acc = (r == j) ? 1.f : 0.f;
      for (int i = j; i < r; ++i) acc -= sA[(base + r) * LDC + base + i] * sX[(base + i) * LDC + base + j];
      sX[(base + r) * LDC + base + j] = acc;
    }
  }
  __syncthreads();
  //    4b. X_ab = -X_aa sum_{b<=m<a} A_am X_mb, block-row after block-row
  for (int a = 1; a < C / kSub; ++a) {
    for (int e = tid; e < a * kSub * kSub; e += kPrepThreads) {
      const int b = e / (kSub * kSub), rr = (e / kSub) % kSub, cc = e % kSub;
      float acc = 0.f;
      for (int m = b * kSub; m < a * kSub; ++m) acc += sA[(a * kSub + rr) * LDC + m] * sX[m * LDC + b * kSub + cc];
      sY[e] = acc;
    }
    __syncthreads();
    for (int e = tid; e < a * kSub * kSub; e += kPrepThreads) {
      const int b = e / (kSub * kSub), rr = (e / kSub) % kSub, cc = e % kSub;
      float acc = 0.f;
      for (int t = 0; t <= rr; ++t) acc += sX[(a * kSub + rr) * LDC + a * kSub + t] * sY[b * kSub * kSub + t * kSub + cc];
      sX[(a * kSub + rr) * LDC + b * kSub + cc] = -acc;
    }
    __syncthreads();
  }

  // 5. w = X Diag(beta)(k * e^G), u = X Diag(beta) V
  for (int idx = tid; idx < C * DK; idx += kPrepThreads) {
    const int i = idx / DK, c = idx % DK;
    sKc[i * LDK + c] = sBeta[i] * sK[i * LDK + c] * expf(sG[i * LDK + c]);
  }
  for (int idx = tid; idx < C * DV; idx += kPrepThreads) {
    const int i = idx / DV, c = idx % DV;
    sV[i * LDV + c] *= sBeta[i];
  }
  __syncthreads();
  for (int idx = tid; idx < C * DK; idx += kPrepThreads) {
    const int r = idx / DK, c = idx % DK;
    float acc = 0.f;
    for (int i = 0; i <= r; ++i) acc += sX[r * LDC + i] * sKc[i * LDK + c];
    rec[R::kW + idx] = acc;
  }
  for (int idx = tid; idx < C * DV; idx += kPrepThreads) {
    const int r = idx / DV, c = idx % DV;
    float acc = 0.f;
    for (int i = 0; i <= r; ++i) acc += sX[r * LDC + i] * sV[i * LDV + c];
    rec[R::kU + idx] = acc;
  }

  // 6. q * e^G, k * e^{G_last - G} and e^{G_last}.  Padded rows carry zero
  //    decay, so row C-1 holds the cumulative decay of the last real token.
  for (int idx = tid; idx < C * DK; idx += kPrepThreads) {
    const int r = idx / DK, c = idx % DK;
    const float gl = sG[(C - 1) * LDK + c], gr = sG[r * LDK + c];
    rec[R::kQh + idx] = sQ[r * LDK + c] * expf(gr);
    rec[R::kKt + idx] = sK[r * LDK + c] * expf(gl - gr);
  }
  for (int c = tid; c < DK; c += kPrepThreads) rec[R::kGamma + c] = expf(sG[(C - 1) * LDK + c]);
}

// ---------------------------------------------------------------------------
// Kernel (c), SIMT: one CTA per (sequence, head, block of BV value columns),
// walking the sequence's chunks in order with the fp32 state in shared memory.
// ---------------------------------------------------------------------------
constexpr int kChainThreads = 256;
constexpr int kChainBV = 32;

template <int DK>
struct ChainSmem {
  static constexpr int oS = 0;                          // S     [DK][BV]
  static constexpr int oW = oS + DK * kChainBV;         // w     [C][DK]
  static constexpr int oQh = oW + kChunk * DK;          // q e^G [C][DK]
  static constexpr int oKt = oQh + kChunk * DK;         // K~    [C][DK]
  static constexpr int oP = oKt + kChunk * DK;          // P     [C][C]
  static constexpr int oU = oP + kChunk * kChunk;       // u     [C][BV]
  static constexpr int oVn = oU + kChunk * kChainBV;    // V_new [C][BV]
  static constexpr int oGam = oVn + kChunk * kChainBV;  // gamma [DK]
  static constexpr int kFloats = oGam + DK;
  static constexpr size_t kBytes = sizeof(float) * kFloats;
};

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(kChainThreads) chunk_chain_simt(const int32_t* __restrict__ cu, int32_t num_seqs,
                                                                  int64_t T_seq, int32_t H, ChunkMap map,
                                                                  const float* __restrict__ inter,
                                                                  const float* __restrict__ s0,
                                                                  float* __restrict__ s_final, T* __restrict__ o) {
  using L = ChainSmem<DK>;
  using R = InterF32<DK, DV>;
  constexpr int C = kChunk, BV = kChainBV;
  constexpr int NW = kChainThreads / 32;
  extern __shared__ float sm[];
  float* sS = sm + L::oS;
  float* sW = sm + L::oW;
  float* sQh = sm + L::oQh;
  float* sKt = sm + L::oKt;
  float* sP = sm + L::oP;
  float* sU = sm + L::oU;
  float* sVn = sm + L::oVn;
  float* sGam = sm + L::oGam;

  if (map.seq_chunk0[num_seqs] < 0) return;  // malformed cu_seqlens: write nothing
  const int s = blockIdx.x, h = blockIdx.y, n0 = blockIdx.z * BV;
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int64_t state_off = ((int64_t)s * H + h) * DK * DV;

  for (int idx = tid; idx < DK * BV; idx += kChainThreads) {
    const int c = idx / BV, n = idx % BV;
    sS[idx] = s0 ? s0[state_off + (int64_t)c * DV + n0 + n] : 0.f;
  }
  const int32_t j0 = map.seq_chunk0[s], j1 = map.seq_chunk0[s + 1];
  const int64_t seq_start = cu ? (int64_t)cu[s] : (int64_t)s * T_seq;
  const int64_t seq_end = cu ? (int64_t)cu[s + 1] : seq_start + T_seq;
  __syncthreads();

  for (int32_t j = j0; j < j1; ++j) {
    const float* rec = inter + ((int64_t)j * H + h) * R::kFloats;
    const int64_t t0 = seq_start + (int64_t)(j - j0) * C;
    const int len = (int)min((int64_t)C, seq_end - t0);
    for (int idx = tid; idx < C * DK / 4; idx += kChainThreads) {
      reinterpret_cast<float4*>(sW)[idx] = reinterpret_cast<const float4*>(rec + R::kW)[idx];
      reinterpret_cast<float4*>(sQh)[idx] = reinterpret_cast<const float4*>(rec + R::kQh)[idx];
      reinterpret_cast<float4*>(sKt)[idx] = reinterpret_cast<const float4*>(rec + R::kKt)[idx];
    }
    for (int idx = tid; idx < C * C / 4; idx += kChainThreads)
      reinterpret_cast<float4*>(sP)[idx] = reinterpret_cast<const float4*>(rec + R::kP)[idx];
    for (int idx = tid; idx < C * BV; idx += kChainThreads) {
      const int r = idx / BV, n = idx % BV;
      sU[idx] = rec[R::kU + r * DV + n0 + n];
    }
    for (int c = tid; c < DK; c += kChainThreads) sGam[c] = rec[R::kGamma + c];
    __syncthreads();

    // V_new = u - w S   (lane = value column, warps over rows)
    for (int r = warp; r < C; r += NW) {
      float acc = sU[r * BV + lane];
      for (int c = 0; c < DK; ++c) acc -= sW[r * DK + c] * sS[c * BV + lane];
      sVn[r * BV + lane] = acc;
    }
    __syncthreads();
    // O = (q e^G) S + P V_new
    for (int r = warp; r < C; r += NW) {
      float acc = 0.f;
      for (int c = 0; c < DK; ++c) acc += sQh[r * DK + c] * sS[c * BV + lane];
      for (int i = 0; i <= r; ++i) acc += sP[r * C + i] * sVn[i * BV + lane];
      if (r < len) o[((t0 + r) * H + h) * DV + n0 + lane] = from_f32<T>(acc);
    }
    // S = Diag(e^{G_last}) S + K~^T V_new
    float snew[DK / NW];
#pragma unroll
    for (int ii = 0; ii < DK / NW; ++ii) {
      const int c = warp + ii * NW;
      float acc = sGam[c] * sS[c * BV + lane];
      for (int r = 0; r < C; ++r) acc += sKt[r * DK + c] * sVn[r * BV + lane];
      snew[ii] = acc;
    }
    __syncthreads();
#pragma unroll
    for (int ii = 0; ii < DK / NW; ++ii) sS[(warp + ii * NW) * BV + lane] = snew[ii];
    const int64_t slot = snapshot_slot(map, s, j - j0, seq_end - seq_start);
    if (slot >= 0) {
#pragma unroll
      for (int ii = 0; ii < DK / NW; ++ii)
        map.snaps[((slot * H + h) * DK + warp + ii * NW) * DV + n0 + lane] = snew[ii];
    }
    __syncthreads();
  }

  if (s_final) {
    for (int idx = tid; idx < DK * BV; idx += kChainThreads) {
      const int c = idx / BV, n = idx % BV;
      s_final[state_off + (int64_t)c * DV + n0 + n] = sS[idx];
    }
  }
}

// ---------------------------------------------------------------------------
// Workspace layout and launch.
// ---------------------------------------------------------------------------
static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static size_t inter_floats(int32_t d_k, int32_t d_v) {
  return (size_t)3 * kChunk * d_k + (size_t)kChunk * d_v + (size_t)kChunk * kChunk + d_k;
}

Workspace chunk_workspace_layout(int64_t total_tokens, int32_t num_seqs, int32_t H, int32_t d_k, int32_t d_v,
                                 kda_dtype dt) {
  Workspace w{};
  const int64_t max_chunks = (total_tokens + kChunk - 1) / kChunk + num_seqs;
  w.max_chunks = (int32_t)max_chunks;
  w.tc = tc_path_supported(d_k, d_v, dt);
  w.inter_bytes_per_chunk_head = w.tc ? tc_record_bytes(d_k, d_v) : sizeof(float) * inter_floats(d_k, d_v);
  w.off_seq_chunk0 = 0;
  w.off_chunk_info = align256(sizeof(int32_t) * ((size_t)num_seqs + 1));
  w.off_seq_order = w.off_chunk_info + align256(sizeof(int4) * (size_t)std::max<int64_t>(max_chunks, 1));
  w.off_snap_slot0 = w.off_seq_order + align256(sizeof(int32_t) * (size_t)std::max<int32_t>(num_seqs, 1));
  w.off_inter = w.off_snap_slot0 + align256(sizeof(int32_t) * ((size_t)num_seqs + 1));
  const size_t R = (size_t)max_chunks * (size_t)H;
  if (w.tc) {
    w.off_wq = w.off_inter;
    w.off_p = w.off_wq + align256(R * 128 * d_k * 2);
    w.off_kt = w.off_p + align256(R * kChunk * kChunk * 2);
    w.off_u = w.off_kt + align256(R * d_k * kChunk * 2);
    w.off_gam = w.off_u + align256(R * kChunk * d_v * 2);
    w.off_flags = w.off_gam + align256(R * d_k * 4);
    w.bytes = w.off_flags + align256(R * 4);
  } else {
    w.bytes = w.off_inter + align256(w.inter_bytes_per_chunk_head * R);
  }
  return w;
}

template <int DK, int DV, typename T>
static cudaError_t launch_simt(const ChunkProblem& p, const Workspace& ws, const ChunkMap& map, float* inter,
                               cudaStream_t stream) {
  const size_t prep_smem = PrepSmem<DK, DV>::kBytes;
  const size_t chain_smem = ChainSmem<DK>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(chunk_prep_simt<DK, DV, T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)prep_smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(chunk_chain_simt<DK, DV, T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)chain_smem);
  if (e != cudaSuccess) return e;
  if (ws.max_chunks > 0 && p.total_tokens > 0) {
    prof_begin(stream, "chunk_prep_simt");
    chunk_prep_simt<DK, DV, T><<<dim3(ws.max_chunks, p.H), kPrepThreads, prep_smem, stream>>>(
        static_cast<const T*>(p.q), static_cast<const T*>(p.k), static_cast<const T*>(p.v),
        static_cast<const T*>(p.g), p.beta, p.cu, p.num_seqs, p.T_seq, p.H, map, inter);
    prof_end(stream);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  prof_begin(stream, "chunk_chain_simt");
  chunk_chain_simt<DK, DV, T><<<dim3(p.num_seqs, p.H, DV / kChainBV), kChainThreads, chain_smem, stream>>>(
      p.cu, p.num_seqs, p.T_seq, p.H, map, inter, p.s0, p.s_final, static_cast<T*>(p.o));
  prof_end(stream);
  return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_simt_dims(const ChunkProblem& p, const Workspace& ws, const ChunkMap& map, float* inter,
                                    cudaStream_t stream) {
  if (p.d_k == 128 && p.d_v == 128) return launch_simt<128, 128, T>(p, ws, map, inter, stream);
  if (p.d_k == 128 && p.d_v == 64) return launch_simt<128, 64, T>(p, ws, map, inter, stream);
  if (p.d_k == 64 && p.d_v == 128) return launch_simt<64, 128, T>(p, ws, map, inter, stream);
  return launch_simt<64, 64, T>(p, ws, map, inter, stream);
}

cudaError_t launch_chunk_fwd(const ChunkProblem& p, const Workspace& ws, void* workspace, cudaStream_t stream) {
  char* base = static_cast<char*>(workspace);
  ChunkMap map;
  map.seq_chunk0 = reinterpret_cast<int32_t*>(base + ws.off_seq_chunk0);
  map.chunk_info = reinterpret_cast<int4*>(base + ws.off_chunk_info);
  map.seq_order = reinterpret_cast<int32_t*>(base + ws.off_seq_order);
  map.max_chunks = ws.max_chunks;
  map.snaps = p.snap_every > 0 ? p.snaps : nullptr;
  map.snap_slot0 = reinterpret_cast<int32_t*>(base + ws.off_snap_slot0);
  map.snap_every = p.snaps ? p.snap_every : 0;
  float* inter = reinterpret_cast<float*>(base + ws.off_inter);

  prof_begin(stream, "chunk_map");
  chunk_map_kernel<<<1, 1024, 0, stream>>>(p.cu, p.num_seqs, p.T_seq, p.total_tokens, map.seq_chunk0,
                                           map.chunk_info, map.seq_order, map.max_chunks, map.snap_every,
                                           map.snap_slot0, p.dev_err);
  prof_end(stream);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (ws.tc) return launch_chunk_tc(p, ws, map, base, stream);
  if (p.dt == KDA_F32) return launch_simt_dims<float>(p, ws, map, inter, stream);
  return launch_simt_dims<__nv_bfloat16>(p, ws, map, inter, stream);
}

}  // namespace kda
