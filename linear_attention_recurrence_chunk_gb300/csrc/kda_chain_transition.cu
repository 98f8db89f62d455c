// Inter-chunk pass of the tensor-core prefill with the output epilogue fused
// (kda_chunk_fwd_gated), in transition form, 32 value columns per CTA.
//
// With the per-chunk records of the prep kernel ([w; q e^G], P, K~^T =
// (k e^{G_last - G})^T, u, e^{G_last}) the state update of one chunk,
//     S' = Diag(e^{G_last}) S + K~^T (u - w S),
// is rewritten with the chunk's transition matrix M = K~^T w (d_k x d_k) as
//     S' = Diag(e^{G_last}) S - M S + K~^T u.
// The two forms are equal (the chunked algebra of page "Kimi K3：架构、训练与百万
// Token Agentic RL 技术解读" §3.3, the intra-chunk work as matrix products with the
// state handed across chunk boundaries).  In the transition form the only work
// that depends on S is one product, M S, so the state's critical path per chunk is
// that product plus the fp32 update: M and K~^T u of the next chunk, and the read
// out o = (q e^G) S + P (u - w S) of the current one, are formed while the state
// hand-off runs.
//
// Per chunk i the MMA warp issues, in this order (fp16 operands, fp32 in TMEM):
//   D_S[i%2]  += (-M_i) S_i            A = -M_i in TMEM, B = S_i (shared memory)
//   D_M        = K~_{i+1}^T w_{i+1}     the next chunk's transition (N = d_k)
//   D_S[(i+1)%2] = K~_{i+1}^T u_{i+1}
//   D12[(i-1)%4] += [. ; P_{i-1}] V_new_{i-1}      (o rows of the previous chunk)
//   D12[i%4]   = [w_i; q_i e^G] S_i                 (rows 0-63: w S, 64-127: q e^G S)
// Warp roles (20 warps):
//   0-7    state: S = e^{G_last} S + D_S in fp32 registers (key channel = TMEM
//          lane, 16 value columns per thread), its fp16 copy the next B operand;
//   8, 9   V_new = u - w S (TMEM lanes 0-63) into the B operand of the o product;
//   10, 11, 18, 19  o rows (TMEM lanes 64-127, 16 columns each) through the
//          output epilogue (Sigmoid gate times the per-head RMSNorm of o and its
//          weight) to global memory: the DV/32 CTAs of a head form a cluster,
//          and each o warp sends its 32 rows' partial sums of squares to every
//          CTA of it as one bulk shared-memory copy counted on the receiver's
//          mbarrier;
//   12-15  transition drain: D_M (fp32) -> -M as fp16 in TMEM, the A operand of
//          the next state product;
//   16     TMA producer: three stages of records (a stage is free once the
//          chunk's [w; q e^G] S has completed) and four P tiles (read a chunk
//          later, by the o product), plus L2 prefetches of later records;
//   17     MMA issue (whole warp, one elected lane).
// Every wait is bounded; on expiry a role stops, reports KDA_ERR_DEVICE_TIMEOUT
// through the device error word, and the CTA drains its MMAs and loads and
// frees TMEM before it returns.
#include <cuda.h>

#include "chain_common.cuh"
#include "kda_chain_transition.cuh"
#include "kda_internal.cuh"
#include "tc_ptx.cuh"

namespace kda {
namespace {

using bf16 = __nv_bfloat16;
using f16 = __half;
using tcu::kWaitLimit;
using tcu::pack_bf16x2;
using tcu::pack_f16x2;
using tcu::report_nonfinite;
using tcu::store_mn_half;

constexpr int C = kChunk;   // tokens per chunk
constexpr int DK = 128;     // key dim of the tensor-core path
constexpr int NC = 32;      // value columns per CTA
constexpr int kMaxRanks = 4;

constexpr int kStateWarps = 8;
constexpr int kVnWarp0 = 8, kOWarp0 = 10, kMWarp0 = 12, kTmaWarp = 16, kMmaWarp = 17, kOWarp1 = 18;
constexpr int kOWarps = 4;
constexpr int kThreads = 32 * 20;

// TMEM columns (fp32 accumulators unless noted)
constexpr int kNB = 4;                  // o buffers (D12)
constexpr uint32_t kColDS = 0;          // D_S[2], 32 columns each
constexpr uint32_t kColD12 = 64;        // D12[4], 32 columns each
constexpr uint32_t kColDM = 192;        // D_M, 128 columns
constexpr uint32_t kColAM = 320;        // -M as fp16 pairs, [2] x 64 columns
constexpr uint32_t kTmemCols = 512;

// fp16 operands, M = 128; B MN-major (value columns or key channels contiguous)
constexpr uint32_t kIdN32 = tc::idesc_f16_f32(128, NC) | (1u << 16);
constexpr uint32_t kIdN128 = tc::idesc_f16_f32(128, DK) | (1u << 16);

struct TransitionSmem {
  // one stage (1024-byte aligned tiles, 128-byte swizzle unless noted)
  static constexpr uint32_t oWQ = 0;         // [w; q e^G] 128 x 128: two 64-column atoms of 16 KB
  static constexpr uint32_t oKT = 32768;     // K~^T 128 x 64
  static constexpr uint32_t oU = 49152;      // u 64 x 32, 64-byte swizzle
  static constexpr uint32_t oGam = 53248;    // e^{G_last}, 128 fp32
  static constexpr uint32_t kStage = 54272;
  static constexpr int kStages = 3, kPBufs = 4;
  static constexpr uint32_t kTx = 32768 + 16384 + C * NC * 2 + DK * 4 + C * C * 2;   // with the chunk's P tile
  static constexpr uint32_t oS = kStages * kStage;   // state operands [2]: 128 keys x 32 columns, 64-byte swizzle
  // P tiles [4], 64 x 64; the o product's A operand is the 16 KB ending at one
  // (rows 0-63: the block before it, finite fp16 data that only adds to the
  // w S rows of D12, which have been read by then)
  static constexpr uint32_t oP = oS + 2 * 8192;
  static constexpr uint32_t oVN = oP + kPBufs * 8192;   // V_new operand: 64 tokens x 32 columns, 64-byte swizzle
  static constexpr uint32_t oWgt = oVN + 4096;          // output epilogue: the CTA's 32 norm weights
  static constexpr uint32_t oStg = oWgt + NC * 4;       // output epilogue: row sums to send, fp32 [2 parities][4 warps][32]
  // output epilogue: partial row sums of squares, fp32 [2 parities][kMaxRanks][2 column halves][64 rows]
  static constexpr uint32_t oRss = oStg + 2 * kOWarps * 32 * 4;
  static constexpr uint32_t oBar = oRss + 2 * kMaxRanks * 2 * 64 * 4;
  static constexpr uint32_t oTmem = oBar + 8 * 32;
  static constexpr uint32_t kBytes = oTmem + 16;
  static constexpr uint32_t kAlloc = kBytes + 1024;   // slack to align the base to 1024
  static_assert(kStage % 1024 == 0 && oP % 1024 == 0 && oU % 1024 == 0 && oS % 1024 == 0 && oVN % 1024 == 0,
                "operand alignment");
  static_assert(kAlloc <= 232448, "fits the shared-memory limit");
};

// The two bf16 values of a packed word as floats, without going through memory.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

template <int DV>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_chain_transition_tc(const __grid_constant__ CUtensorMap tmWQ, const __grid_constant__ CUtensorMap tmP,
                       const __grid_constant__ CUtensorMap tmKT, const __grid_constant__ CUtensorMap tmU,
                       const __grid_constant__ CUtensorMap tmGam, const int32_t* __restrict__ cu, int32_t num_seqs,
                       int64_t T_seq, int32_t H, ChunkMap map, const float* __restrict__ s0,
                       float* __restrict__ s_final, bf16* __restrict__ o, OutEpilogue ep, int32_t* dev_err) {
  using L = TransitionSmem;
  constexpr int kRanks = DV / NC;   // CTAs per head: the cluster
  static_assert(kRanks <= kMaxRanks, "row-sum slots");
  if (map.seq_chunk0[num_seqs] < 0) return;   // malformed cu_seqlens: every CTA of a cluster alike
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::oBar);
  uint64_t* full = bar;          // [3] a stage's tiles (and its P tile) landed (TMA transaction count)
  uint64_t* d12f = bar + 3;      // [3] [w; q e^G] S of the stage's chunk has completed: the last MMA reading the stage
  uint64_t* cons = bar + 6;      // [3] the state and V_new warps are done reading a stage
  uint64_t* dsf = bar + 9;       // [2] the state product of a chunk has completed
  uint64_t* s_ready = bar + 11;  // the state warps have stored the next state operand
  uint64_t* vn_ready = bar + 12; // the V_new warps have stored V_new
  uint64_t* ofull = bar + 13;    // [4] a chunk's o rows are complete in D12
  uint64_t* dfree = bar + 17;    // [4] the o warps have read a D12 buffer
  uint64_t* dm_full = bar + 21;  // D_M holds the next transition
  uint64_t* am_full = bar + 22;  // -M is in TMEM (and D_M has been read)
  uint64_t* drain = bar + 23;    // every MMA has completed (end of kernel)
  uint64_t* rs = bar + 24;       // [2] gated: the row sums of every o warp of the cluster have landed
  float* rss = reinterpret_cast<float*>(sm + L::oRss);
  float* sWgt = reinterpret_cast<float*>(sm + L::oWgt);
  float* sStg = reinterpret_cast<float*>(sm + L::oStg);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::oTmem);

  // one-dimensional grid, sequence-rank major: all blocks of the longest chain first
  const int blk = (int)(blockIdx.x % (unsigned)(H * kRanks));
  const int s = map.seq_order[blockIdx.x / (unsigned)(H * kRanks)], h = blk / kRanks, n0 = (blk % kRanks) * NC;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int32_t j0 = map.seq_chunk0[s];
  const int32_t nch = map.seq_chunk0[s + 1] - j0;
  const int64_t seq_start = cu ? (int64_t)cu[s] : (int64_t)s * T_seq;
  const int64_t seq_end = cu ? (int64_t)cu[s + 1] : seq_start + T_seq;

  if (tid == 0) {
    for (int i = 0; i < L::kStages; ++i) {
      tc::mbar_init(full + i, 1);
      tc::mbar_init(d12f + i, 1);
      tc::mbar_init(cons + i, kStateWarps + 2);
    }
    tc::mbar_init(dsf, 1);
    tc::mbar_init(dsf + 1, 1);
    tc::mbar_init(s_ready, kStateWarps);
    tc::mbar_init(vn_ready, 2);
    for (int b = 0; b < kNB; ++b) {
      tc::mbar_init(ofull + b, 1);
      tc::mbar_init(dfree + b, kOWarps);
    }
    tc::mbar_init(dm_full, 1);
    tc::mbar_init(am_full, 4);
    tc::mbar_init(drain, 1);
    tc::mbar_init(rs, 1);   // one local arrival (with the expected bytes) per phase
    tc::mbar_init(rs + 1, 1);
    tc::fence_mbar_init();
  }
  for (int i = tid; i < 512; i += kThreads)   // the second state operand (the rows before P tile 0)
    reinterpret_cast<uint4*>(sm + L::oS + 8192)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (tid < NC) sWgt[tid] = ep.weight ? ep.weight[(int64_t)h * DV + n0 + tid] : 1.f;
  if (warp == 0) {
    tc::tmem_alloc(tslot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  // the cluster's barriers are initialised before any CTA of it sends row sums
  tc::cluster_sync_all();
  const uint32_t tmem = *tslot;

  if (warp == kTmaWarp) {
    // ---------------- TMA producer
    if (lane == 0) {
      tc::tma_prefetch_desc(&tmWQ);
      tc::tma_prefetch_desc(&tmP);
      tc::tma_prefetch_desc(&tmKT);
      tc::tma_prefetch_desc(&tmU);
      tc::tma_prefetch_desc(&tmGam);
      constexpr int kPf = 6;   // chunks between an L2 prefetch and the load of the same records
      auto prefetch = [&](int i) {
        const int64_t rec = (int64_t)(j0 + i) * H + h;
        tc::tma_prefetch_l2_2d(&tmWQ, 0, (int32_t)(rec * 128));
        tc::tma_prefetch_l2_2d(&tmWQ, 64, (int32_t)(rec * 128));
        tc::tma_prefetch_l2_2d(&tmKT, 0, (int32_t)(rec * DK));
        tc::tma_prefetch_l2_2d(&tmP, 0, (int32_t)(rec * C));
        tc::tma_prefetch_l2_2d(&tmU, n0, (int32_t)(rec * C));
        tc::tma_prefetch_l2_2d(&tmGam, 0, (int32_t)rec);
      };
      for (int i = 0; i < kPf && i < nch; ++i) prefetch(i);
      int issued = 0;
      for (int i = 0; i < nch; ++i) {
        const int st = i % L::kStages;
        const uint32_t ph = (uint32_t)(i / L::kStages - 1) & 1u;
        // a stage is refilled once [w; q e^G] S of chunk i - 3 has completed (after
        // the o product of chunk i - 4, the last reader of P tile i % 4) and the
        // consumer warps are done reading it
        if (i >= L::kStages && !(tc::mbar_wait(d12f + st, ph, kWaitLimit) && tc::mbar_wait(cons + st, ph, kWaitLimit))) {
          atomicExch(dev_err, (int32_t)kDevErrTimeout);
          break;
        }
        const int64_t rec = (int64_t)(j0 + i) * H + h;
        uint8_t* stg = sm + st * L::kStage;
        tc::mbar_arrive_expect_tx(full + st, L::kTx);
        tc::tma_load_2d(stg + L::oWQ, &tmWQ, 0, (int32_t)(rec * 128), full + st);
        tc::tma_load_2d(stg + L::oWQ + 16384, &tmWQ, 64, (int32_t)(rec * 128), full + st);
        tc::tma_load_2d(stg + L::oKT, &tmKT, 0, (int32_t)(rec * DK), full + st);
        tc::tma_load_2d(stg + L::oU, &tmU, n0, (int32_t)(rec * C), full + st);
        tc::tma_load_2d(stg + L::oGam, &tmGam, 0, (int32_t)rec, full + st);
        tc::tma_load_2d(sm + L::oP + 8192 * (i % L::kPBufs), &tmP, 0, (int32_t)(rec * C), full + st);
        ++issued;
        if (i + kPf < nch) prefetch(i + kPf);
      }
      // never leave loads in flight: wait (bounded) until the last ones landed
      for (int i = (issued > L::kStages ? issued - L::kStages : 0); i < issued; ++i)
        tc::mbar_wait(full + i % L::kStages, (uint32_t)(i / L::kStages) & 1u, kWaitLimit);
    }
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issue (whole warp, warp-uniform operands, one elected lane)
    const uint64_t dA0 = tc::desc_kmajor_sw128(tc::smem_u32(sm));                      // stage 0, K-major tiles
    const uint64_t dW0 = tc::desc_mnmajor_sw128_atoms(tc::smem_u32(sm + L::oWQ), 16384);   // w rows as an MN-major B
    const uint64_t dS0 = tc::desc_mnmajor_sw64(tc::smem_u32(sm + L::oS));
    const uint64_t dV0 = tc::desc_mnmajor_sw64(tc::smem_u32(sm + L::oVN));
    auto wait_all = [&](uint64_t* b, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, tc::mbar_wait(b, parity, kWaitLimit));
    };
    // chunk j's transition M_j (stage j % 3)
    auto issue_m = [&](int j) {
      const int st = j % L::kStages;
      const uint64_t dKT = dA0 + ((uint64_t)(st * L::kStage + L::oKT) >> 4);
      const uint64_t dW = dW0 + ((uint64_t)(st * L::kStage) >> 4);
#pragma unroll
      for (int kk = 0; kk < C / 16; ++kk)
        tc::mma_16bit_w(tmem + kColDM, dKT + ((kk * 32) >> 4), dW + ((kk * 2048) >> 4), kIdN128, kk > 0);
      tc::mma_commit_w(dm_full);
    };
    // the K~^T u start of chunk j's state product (state accumulator j % 2)
    auto issue_init = [&](int j) {
      const int st = j % L::kStages;
      const uint64_t dKT = dA0 + ((uint64_t)(st * L::kStage + L::oKT) >> 4);
      const uint64_t dU = tc::desc_mnmajor_sw64(tc::smem_u32(sm + st * L::kStage + L::oU));
#pragma unroll
      for (int kk = 0; kk < C / 16; ++kk)
        tc::mma_16bit_w(tmem + kColDS + (uint32_t)(j & 1) * NC, dKT + ((kk * 32) >> 4), dU + ((kk * 1024) >> 4),
                        kIdN32, kk > 0);
    };
    // chunk j's o rows: D12 += [. ; P_j] V_new_j
    auto issue_pv = [&](int j) {
      const uint64_t dPt = dA0 + ((uint64_t)(L::oP + 8192 * (j % L::kPBufs) - 8192) >> 4);
      const uint32_t d12 = tmem + kColD12 + (uint32_t)(j % kNB) * NC;
#pragma unroll
      for (int kk = 0; kk < C / 16; ++kk)
        tc::mma_16bit_w(d12, dPt + ((kk * 32) >> 4), dV0 + ((kk * 1024) >> 4), kIdN32, 1u);
      tc::mma_commit_w(ofull + (j % kNB));
    };
    bool ok = true, issued = false;
    if (nch > 0) {
      ok = wait_all(full, 0);
      if (ok) {
        tc::tc_fence_after();
        issue_m(0);
        issue_init(0);
        issued = true;
      }
    }
    for (int i = 0; i < nch && ok; ++i) {
      const int sb = i & 1;   // state accumulator, state operand, transition buffer
      // the drain of M_i has read D_M and the state warps have read D_S[(i+1)%2]
      ok = wait_all(am_full, (uint32_t)i & 1u) && wait_all(s_ready, (uint32_t)i & 1u);
      if (!ok) break;
      tc::tc_fence_after();
      const uint64_t dS = dS0 + ((uint64_t)(sb * 8192) >> 4);
      const uint32_t aM = tmem + kColAM + (uint32_t)sb * 64;
#pragma unroll
      for (int kk = 0; kk < DK / 16; ++kk)   // the state product: D_S += (-M) S
        tc::mma_16bit_ta_w(tmem + kColDS + (uint32_t)sb * NC, aM + 8 * kk, dS + ((kk * 1024) >> 4), kIdN32, 1u);
      tc::mma_commit_w(dsf + sb);
      if (i + 1 < nch) {
        ok = wait_all(full + (i + 1) % L::kStages, (uint32_t)((i + 1) / L::kStages) & 1u);
        if (!ok) break;
        tc::tc_fence_after();
        issue_m(i + 1);
        issue_init(i + 1);
      }
      if (i >= 1) {
        ok = wait_all(vn_ready, (uint32_t)(i - 1) & 1u);
        if (!ok) break;
        tc::tc_fence_after();
        issue_pv(i - 1);
      }
      if (i >= kNB) {
        ok = wait_all(dfree + (i % kNB), (uint32_t)((i / kNB) - 1) & 1u);
        if (!ok) break;
        tc::tc_fence_after();
      }
      const uint64_t dA = dA0 + ((uint64_t)((i % L::kStages) * L::kStage) >> 4);
      const uint32_t d12 = tmem + kColD12 + (uint32_t)(i % kNB) * NC;
#pragma unroll
      for (int kk = 0; kk < DK / 16; ++kk)   // [w; q e^G] S
        tc::mma_16bit_w(d12, dA + ((((kk >> 2) * 16384) + (kk & 3) * 32) >> 4), dS + ((kk * 1024) >> 4), kIdN32,
                        kk > 0);
      tc::mma_commit_w(d12f + i % L::kStages);
    }
    if (ok && nch > 0) {
      ok = wait_all(vn_ready, (uint32_t)(nch - 1) & 1u);
      if (ok) {
        tc::tc_fence_after();
        issue_pv(nch - 1);
      }
    }
    if (!ok && lane == 0) atomicExch(dev_err, (int32_t)kDevErrTimeout);
    if (issued) {   // no MMA may still be writing TMEM when it is freed
      tc::mma_commit_w(drain);
      wait_all(drain, 0);
    }
  } else if (warp >= kMWarp0 && warp < kOWarp1) {
    // ---------------- transition drain: D_M (fp32) -> -M (fp16 pairs) in TMEM
    const uint32_t tl = (uint32_t)(32 * (warp & 3));
    bool bad = false;
    for (int j = 0; j < nch; ++j) {
      bad |= !tc::mbar_wait(dm_full, (uint32_t)j & 1u, kWaitLimit);
      if (__any_sync(0xffffffffu, bad)) {
        bad = true;
        break;
      }
      tc::tc_fence_after();
#pragma unroll
      for (int b = 0; b < DK / 32; ++b) {
        float m[32];
        tc::tmem_ld32(tc::tmem_addr(tmem, tl, kColDM + 32 * b), m);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = pack_f16x2(m[2 * e], m[2 * e + 1]) ^ 0x80008000u;   // negated
        tc::tmem_st16(tc::tmem_addr(tmem, tl, kColAM + (uint32_t)(j & 1) * 64 + 16 * b), pk);
      }
      tc::tmem_st_wait();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(am_full);
    }
    if (bad && lane == 0) atomicExch(dev_err, (int32_t)kDevErrTimeout);
  } else if (warp >= kOWarp0) {
    // ---------------- o rows (TMEM lanes 64-127, token r of the chunk), value columns 16 hf .. 16 hf + 15
    const int q = warp & 3, r = 32 * (q - 2) + lane, hf = warp >= kOWarp1 ? 1 : 0;
    const uint32_t tl = (uint32_t)(32 * q);
    const uint32_t crank = tc::cluster_ctarank();
    float nonfinite = 0.f;
    const int wi = 2 * hf + (q - 2);   // this warp's slot: 32 rows, 16 columns
    // The row's gate logits: prefetched into L2 kGatePf chunks ahead, loaded into
    // registers a chunk ahead.
    constexpr int kGatePf = 4;
    uint4 gnext[2] = {};
    auto gate_row = [&](int i) -> const bf16* {   // null past the sequence
      const int64_t t0 = seq_start + (int64_t)i * C;
      return (i < nch && r < seq_end - t0) ? ep.gate + ((t0 + r) * H + h) * DV + n0 + 16 * hf : nullptr;
    };
    auto load_gate = [&](int i) {   // issued where it stands
      if (const bf16* gp = gate_row(i)) {
#pragma unroll
        for (int k = 0; k < 2; ++k) gnext[k] = ld_nc_v4(gp + 8 * k);
      }
    };
    auto prefetch_gate = [&](int i) {
      if (const bf16* gp = gate_row(i)) asm volatile("prefetch.global.L2 [%0];" ::"l"(gp));
    };
    for (int k = 0; k < kGatePf; ++k) prefetch_gate(k);
    load_gate(0);
    bool bad = false;
    int i = 0;
    for (; i < nch; ++i) {
      const int b = i % kNB;
      const int64_t t0 = seq_start + (int64_t)i * C;
      const int64_t len = min((int64_t)C, seq_end - t0);
      bad |= !tc::mbar_wait(ofull + b, (uint32_t)(i / kNB) & 1u, kWaitLimit);
      if (__any_sync(0xffffffffu, bad)) {
        bad = true;
        break;
      }
      tc::tc_fence_after();
      float ov[16];
      tc::tmem_ld16(tc::tmem_addr(tmem, tl, kColD12 + (uint32_t)b * NC + 16 * hf), ov);
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(dfree + b);
      {
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) ss = fmaf(ov[e], ov[e], ss);
        const int par = i & 1;
        // The warp's 32 row sums go to every CTA of the cluster as one 128-byte
        // bulk copy per destination, counted on the destination's barrier; the
        // staging row of this parity is rewritten once the copies of chunk i - 2
        // (the group before the latest) have read it.
        float* stg = sStg + (par * 2 + wi) * 32;
        if (lane == 0 && i >= 2) tc::bulk_wait_read1();
        __syncwarp();
        stg[lane] = ss;
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          // this CTA expects 128 bytes from each (rank, o warp) of the cluster in this phase
          if (warp == kOWarp0) tc::mbar_arrive_expect_tx(rs + par, (uint32_t)kRanks * kOWarps * 128u);
          float* slot = rss + ((par * kMaxRanks + (int)crank) * 2 + hf) * 64 + 32 * (q - 2);
#pragma unroll
          for (uint32_t d = 0; d < (uint32_t)kRanks; ++d)
            tc::bulk_copy_s2c(tc::mapa_shared(slot, d), stg, 128u, tc::mapa_shared(rs + par, d));
          tc::bulk_commit();
        }
        uint4 gcur[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) gcur[k] = gnext[k];
        load_gate(i + 1);
        prefetch_gate(i + kGatePf);
        // the gate and the weight while the other CTAs' row sums arrive
        const float* wt = sWgt + 16 * hf;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const uint32_t gw[4] = {gcur[k].x, gcur[k].y, gcur[k].z, gcur[k].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c0 = 8 * k + 2 * e;
            ov[c0] *= __fdividef(wt[c0], 1.f + __expf(-bf16_lo(gw[e])));
            ov[c0 + 1] *= __fdividef(wt[c0 + 1], 1.f + __expf(-bf16_hi(gw[e])));
          }
        }
        bad |= !tc::mbar_wait(rs + par, (uint32_t)(i >> 1) & 1u, kWaitLimit);
        if (__any_sync(0xffffffffu, bad)) {
          bad = true;
          break;
        }
        float tot = 0.f;
#pragma unroll
        for (int d = 0; d < 2 * kRanks; ++d) tot += rss[(par * kMaxRanks * 2 + d) * 64 + r];
        const float sc = rsqrtf(tot * (1.f / DV) + ep.eps);
#pragma unroll
        for (int e = 0; e < 16; ++e) ov[e] *= sc;
      }
      if (r < len) {
        uint4* dst = reinterpret_cast<uint4*>(o + ((t0 + r) * H + h) * DV + n0 + 16 * hf);
#pragma unroll
        for (int k = 0; k < 2; ++k)
          dst[k] = make_uint4(pack_bf16x2(ov[8 * k + 0], ov[8 * k + 1]), pack_bf16x2(ov[8 * k + 2], ov[8 * k + 3]),
                              pack_bf16x2(ov[8 * k + 4], ov[8 * k + 5]), pack_bf16x2(ov[8 * k + 6], ov[8 * k + 7]));
#pragma unroll
        for (int e = 0; e < 16; ++e) nonfinite = fmaf(ov[e], 0.f, nonfinite);
      }
    }
    if (lane == 0) tc::bulk_wait0();   // every row-sum copy of this warp has completed
    if (i < nch || bad) {
      if (lane == 0) atomicExch(dev_err, (int32_t)kDevErrTimeout);
    } else {
      report_nonfinite(nonfinite, dev_err);
    }
  } else if (warp >= kVnWarp0) {
    // ---------------- V_new = u - w S (TMEM lanes 0-63, token r of the chunk)
    const int q = warp & 3, r = 32 * q + lane;
    const uint32_t tl = (uint32_t)(32 * q);
    bool bad = false;
    for (int i = 0; i < nch; ++i) {
      const int st = i % L::kStages;
      bad |= !tc::mbar_wait(d12f + st, (uint32_t)(i / L::kStages) & 1u, kWaitLimit);
      if (__any_sync(0xffffffffu, bad)) {
        bad = true;
        break;
      }
      uint4 uraw[4];   // u of the stage, read before anything else so that the stage is released early
      const uint8_t* ub = sm + st * L::kStage + L::oU;
#pragma unroll
      for (int k = 0; k < 4; ++k) uraw[k] = *reinterpret_cast<const uint4*>(ub + tc::sw64_chunk_offset(r, k));
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(cons + st);
      tc::tc_fence_after();
      float d[32];
      tc::tmem_ld32(tc::tmem_addr(tmem, tl, kColD12 + (uint32_t)(i % kNB) * NC), d);
      uint8_t* vb = sm + L::oVN;   // one buffer: the o product of chunk i - 1 preceded [w; q e^G] S of chunk i
#pragma unroll
      for (int k = 0; k < 4; ++k)
        *reinterpret_cast<uint4*>(vb + tc::sw64_chunk_offset(r, k)) = tcu::vnew_f16x8(uraw[k], d + 8 * k);
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(vn_ready);
    }
    if (bad && lane == 0) atomicExch(dev_err, (int32_t)kDevErrTimeout);
  } else {
    // ---------------- state: key channel c (TMEM lane), value columns 16 hf .. 16 hf + 15
    const int q = warp & 3, hf = warp >> 2;
    const int c = 32 * q + lane;
    const uint32_t tl = (uint32_t)(32 * q);
    float S[16];
    {
      const int64_t off = (((int64_t)s * H + h) * DK + c) * DV + n0 + 16 * hf;
#pragma unroll
      for (int n = 0; n < 16; n += 4) {
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (s0) x = *reinterpret_cast<const float4*>(s0 + off + n);
        S[n] = x.x;
        S[n + 1] = x.y;
        S[n + 2] = x.z;
        S[n + 3] = x.w;
      }
    }
    store_mn_half(sm + L::oS, c, hf, S);
    tc::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(s_ready);
    bool bad = false;
    int i = 0;
    for (; i < nch; ++i) {
      const int st = i % L::kStages, sb = i & 1;
      bad |= !tc::mbar_wait(full + st, (uint32_t)(i / L::kStages) & 1u, kWaitLimit);
      if (__any_sync(0xffffffffu, bad)) {
        bad = true;
        break;
      }
      const float gam = reinterpret_cast<const float*>(sm + st * L::kStage + L::oGam)[c];
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(cons + st);   // e^{G_last} of the stage has been read
      bad |= !tc::mbar_wait(dsf + sb, (uint32_t)(i >> 1) & 1u, kWaitLimit);
      if (__any_sync(0xffffffffu, bad)) {
        bad = true;
        break;
      }
      tc::tc_fence_after();
      float d[16];
      tc::tmem_ld16(tc::tmem_addr(tmem, tl, kColDS + (uint32_t)sb * NC + 16 * hf), d);
#pragma unroll
      for (int n = 0; n < 16; ++n) S[n] = fmaf(gam, S[n], d[n]);
      const bool more = i + 1 < nch;
      if (more) {
        store_mn_half(sm + L::oS + (sb ^ 1) * 8192, c, hf, S);
        tc::fence_proxy_async_smem();
      }
      tc::tc_fence_before();
      __syncwarp();
      if (more && lane == 0) tc::mbar_arrive(s_ready);
      if (const int64_t slot = snapshot_slot(map, s, i, seq_end - seq_start); slot >= 0) {
        float* dst = map.snaps + ((slot * H + h) * DK + c) * DV + n0 + 16 * hf;
#pragma unroll
        for (int n = 0; n < 16; n += 4) *reinterpret_cast<float4*>(dst + n) = make_float4(S[n], S[n + 1], S[n + 2], S[n + 3]);
      }
    }
    if (i < nch || bad) {
      if (lane == 0) atomicExch(dev_err, (int32_t)kDevErrTimeout);
    } else {
      float nonfinite = 0.f;
#pragma unroll
      for (int n = 0; n < 16; ++n) nonfinite = fmaf(S[n], 0.f, nonfinite);
      report_nonfinite(nonfinite, dev_err);
      if (s_final) {
        float* dst = s_final + (((int64_t)s * H + h) * DK + c) * DV + n0 + 16 * hf;
#pragma unroll
        for (int n = 0; n < 16; n += 4) *reinterpret_cast<float4*>(dst + n) = make_float4(S[n], S[n + 1], S[n + 2], S[n + 3]);
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
  // no CTA of the cluster leaves while another may still send it row sums
  tc::cluster_sync_all();
}

template <int DV>
cudaError_t launch_transition(const CUtensorMap& mWQ, const CUtensorMap& mP, const CUtensorMap& mKT,
                              const CUtensorMap& mU, const CUtensorMap& mGam, const ChunkProblem& p, const ChunkMap& map,
                              cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(chunk_chain_transition_tc<DV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)TransitionSmem::kAlloc);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.num_seqs * p.H * (DV / NC), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = TransitionSmem::kAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];   // the DV / 32 CTAs of a head (consecutive blocks) form one cluster
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = DV / NC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const OutEpilogue ep{static_cast<const bf16*>(p.out_gate), p.norm_weight, p.eps_rms};
  prof_begin(stream, "chunk_chain_transition_tc");
  e = cudaLaunchKernelEx(&cfg, chunk_chain_transition_tc<DV>, mWQ, mP, mKT, mU, mGam, p.cu, p.num_seqs, p.T_seq, p.H,
                         map, p.s0, p.s_final, static_cast<bf16*>(p.o), ep, p.dev_err);
  prof_end(stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chain_transition_gated(const CUtensorMap& mWQ, const CUtensorMap& mP, const CUtensorMap& mKT,
                                          const CUtensorMap& mU, const CUtensorMap& mGam, const ChunkProblem& p,
                                          const ChunkMap& map, cudaStream_t stream) {
  if (p.d_v == 128) return launch_transition<128>(mWQ, mP, mKT, mU, mGam, p, map, stream);
  return launch_transition<64>(mWQ, mP, mKT, mU, mGam, p, map, stream);
}

}  // namespace kda
