// Tensor-core chunked prefill for bf16 inputs with d_k = 128 (d_v = 64 or 128).
//
// After the sequence -> chunk map, prep then a chain kernel, or, for few
// (sequence, head) chains with d_v = 128, both in one launch (chunk_fused_tc at
// the end of this file: the chains, in the value-major form of
// chain_vm_body.cuh, trail the prep CTAs chunk by chunk):
//
//  chunk_prep_tc   persistent over (64-token chunk, head) tasks in chunk-major
//                  order, the next raw rows arriving by TMA during the current
//                  task: gate, cumulative log-decay, the exp(+-G) scalings as
//                  bf16 operand tiles (128-byte swizzle), then the
//                  beta-weighted decayed k k^T matrix A and the read-out matrix
//                  P as tcgen05 products (M = 128, fp32 in TMEM) while the
//                  threads write the q e^G and K~^T records and the
//                  [beta k e^G | beta V] operand; X = (I + A)^{-1} (diagonal
//                  blocks in registers, blocks below on mma.sync), then
//                  w, u = X [beta k e^G | beta V] on tcgen05, drained and stored
//                  by TMA during the next task.  Records: fp16 [w; q e^G], P,
//                  (k e^{G_last - G})^T, u and fp32 e^{G_last}.  The bounded
//                  map runs it with two task streams per CTA, a task in two
//                  64-channel passes (chunk_prep_split_tc, prep_split_body.cuh,
//                  also chunk_fused_tc's prep role); the single-stream kernel
//                  below runs the ablation's pair paths.
//
//  chunk_chain_tc  one CTA per (sequence, head, 32 value columns); the wide
//  (_wide_tc)      form takes 64 or all value columns per CTA (the value-major
//                  chain, kda_chain_vm.cu, all 128 without the epilogue).  Walks the
//                  sequence's chunks in order with the fp32 state block in
//                  registers, feeding tcgen05 MMAs (fp32 accumulators in TMEM,
//                  issued by one warp) from TMA-staged fp16 tiles
//                  (double-buffered by a producer warp):
//                     group 1:  D12 = [w; q e^G] . S                (M=128, K=d_k)
//                               V_new = u - D12[0:64]
//                     group 2:  D12 += [0; P] . V_new               (M=128, K=64)
//                               D3   = (k e^{G_last-G})^T . V_new   (M=128, K=64)
//                     o = D12[64:128];   S = Diag(e^{G_last}) S + D3
//
// Precision.  The sub-tile operands of A and P need bf16's exponent range (the
// factors reach e^80); everything the chain multiplies is bounded by 1 or by
// the size of v and S, so it is stored in fp16, whose 10-bit mantissa is 4x
// finer than bf16's.  P multiplies V_new (O(|v|)) into o, which is an order
// of magnitude smaller than v, so P's diagonal sub-tiles get a two-term bf16
// split on both operands (hi*hi + hi*lo + lo*hi, about 16 bits); below the
// diagonal every factor is <= 1 and single bf16 products suffice.  With plain
// bf16 everywhere the largest output error reached ~5% of rms(o); with this
// split it is ~0.6%.
//
// The algebra (page "Kimi K3：架构、训练与百万 Token Agentic RL 技术解读" §3.3: intra-chunk
// work as matrix products, the state passed across chunk boundaries) is
// derived in kda_chunk.cu.  The sub-tile factors follow the 16-token bound of
// the same section: within a 16-row block the row factor e^{G_r - G_s} <= 1 and
// the column factor e^{G_s - G_i} <= e^{80} (G_s = cumulative decay just before
// the block); across blocks both factors are <= 1.
#include <cudaTypedefs.h>

#include <algorithm>
#include <type_traits>
#include <mutex>

#include "kda_internal.cuh"

#include <cstdlib>
#include "tc_ptx.cuh"
#include "chain_common.cuh"
#include "chain_vm.cuh"
#include "chain_vm_body.cuh"
#include "prep_split_body.cuh"

namespace kda {
namespace {

using bf16 = __nv_bfloat16;
using f16 = __half;
constexpr int C = kChunk;         // 64 tokens per chunk
constexpr int DK = 128;           // key dim of this path
constexpr int BV = 32;            // value columns per chain CTA
using tcu::kWaitLimit;
using tcu::pack_bf16x2;
using tcu::pack_f16x2;
using tcu::report_nonfinite;
using tcu::store_bf16x16;
using tcu::store_mn_half;

// Helpers shared with the two-stream prep (prep_split_body.cuh).
using ps::ex2_approx;
using ps::kv_off;
using ps::later_row0;
using ps::ld_early_f32;
using ps::ld_early_v4;
using ps::ldsm_x4;
using ps::ldsm_x4_t;
using ps::mma16816_f16;
using ps::rcp_approx;
using ps::split_bf16x2;
using ps::xs_off;
using ps::kPublishBatch;
using ps::publish_records;

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// log2 of the unbounded decay, -Softplus(x) / ln 2 = -log2(1 + 2^y) with
// y = x log2(e), as -(max(y, 0) + log2(1 + 2^{-|y|})) so that nothing
// overflows; y is capped at 2^100 (logits above 8.8e29), which keeps a chunk's
// sum finite (the factors it feeds are then 0 either way).
__device__ __forceinline__ float fast_log2_softplus_decay(float x) {
  float y = x * 1.4426950408889634f;
  y = y > 1.2676506e30f ? 1.2676506e30f : y;   // NaN passes through
  return -(fmaxf(y, 0.f) + lg2_approx(1.f + ex2_approx(-fabsf(y))));
}
template <bool kSoftplus>
__device__ __forceinline__ float log2_decay(float x) {
  return kSoftplus ? fast_log2_softplus_decay(x) : ps::log2_decay_bounded(x);
}

// --------------------------------------------------------------- prep kernel
constexpr int kPrepTcThreads = 512;

// Variants of the prep kernel (the decay-map ablation):
//   kPrepBounded       -5 Sigmoid gate, diagonal 16x16 blocks of A and P on the
//                      tensor cores with the sub-tile-start reference, whose
//                      factors e^{G_s - G_i} stay below e^80 only because of the
//                      lower bound (page "Kimi K3：架构、训练与百万 Token Agentic RL 技术解读",
//                      §3.3 "lower-bounded decay");
//   kPrepBoundedPairs  the same gate, diagonal blocks by position pairs;
//   kPrepSoftplusPairs the unbounded -Softplus gate of the predecessor model
//                      (page "Kimi K3 架构篇：一文详解 2.8 万亿参数的巨型怪兽", section
//                      "最被低估的一个细节：下界衰减"), which only the pair path can take.
// The pair path forms each diagonal-block entry as a sum over the key channels
// of k_r k_i e^{G_r - G_i} (and q_r k_i e^{G_r - G_i}) on the CUDA cores, one
// exponential per pair and channel, with every exponent <= 0.
constexpr int kPrepBounded = 0, kPrepBoundedPairs = 1, kPrepSoftplusPairs = 2;

template <int DV, int kVariant = kPrepBounded>
struct PrepTcSmem {
  static constexpr bool kPairs = kVariant != kPrepBounded;
  static constexpr int LDX = C + 8;           // fp16 row stride of A's off-diagonal blocks
  static constexpr int kWuN = DK + DV;        // columns of [w | u]
  static constexpr int LDA = C + 1;           // fp32 row stride of A's diagonal blocks
  // Operands of the A / P products on the tensor cores: bf16, K-major (key
  // channels contiguous), 128-byte swizzle, one atom per 64 channels.
  //   row operand, 192 rows:    0-63  k e^{G - G_s},  64-127 q e^{G - G_s} (high part),
  //                             128-191 its low part
  //   column operand, 224 rows: 0-63  k e^{G_s - G} of the own sub-tile (high part),
  //                             64-127 its low part,
  //                             128 + kOff[a'] + i  k_i e^{G_s(a') - G_i} for the later
  //                             sub-tiles a' = 1..3 (columns i < 16 a', high part only)
  static constexpr int kRowRows = 192, kColRows = 224;
  static constexpr size_t kRowAtom = (size_t)kRowRows * 128, kColAtom = (size_t)kColRows * 128;
  // raw input rows of the next task (TMA, bf16 [64][d]), staged during this one
  static constexpr size_t oRawG = 0;
  static constexpr size_t oRawK = oRawG + (size_t)C * DK * 2;
  static constexpr size_t oRawQ = oRawK + (size_t)C * DK * 2;
  static constexpr size_t oRawV = oRawQ + (size_t)C * DK * 2;
  static constexpr size_t oRow = (oRawV + (size_t)C * DV * 2 + 1023) / 1024 * 1024;
  static constexpr size_t oCol = oRow + (DK / 64) * kRowAtom;
  // [beta k e^G | beta V], fp16, the B operand of [w | u] = X (...): MN-major,
  // 128-byte swizzle, 64-column atoms [64 tokens][128 B] of 8 KB
  static constexpr size_t oKV = oCol + (DK / 64) * kColAtom;
  static constexpr size_t oPst = oKV + (size_t)(kWuN / 64) * 8192;   // fp16 [64][64] P, 128-byte swizzle (TMA store)
  static constexpr size_t oTot = oPst + (size_t)C * C * 2;           // fp32 [8][DK] group sums
  static constexpr size_t oBeta = oTot + (size_t)8 * DK * 4;         // fp32 [64]
  static constexpr size_t oBar = oBeta + (size_t)C * 4;              // mbarriers: raw rows, [w | u], A / P products
  static constexpr size_t oTmem = oBar + 24;                          // TMEM base address
  static constexpr size_t kBytes = oTmem + 8;
  static constexpr size_t kAlloc = kBytes + 1024;                    // slack to align the base to 1 KB
  // reused once the A / P products are done
  static constexpr size_t oA = oRow;                                  // fp32 [64][LDA]  A, diagonal blocks
  // X, fp16 [128][64] (rows 64-127 zero), K-major with 128-byte swizzle: the A operand of [w | u]
  static constexpr size_t oXb = (oA + (size_t)C * LDA * 4 + 1023) / 1024 * 1024;
  static constexpr size_t oAh = oXb + (size_t)2 * C * C * 2;         // fp16 [64][LDX]  A, blocks below them
  static constexpr size_t oYh = oAh + (size_t)C * LDX * 2;           // fp16 [7][16][24] scratch blocks of the inverse
  static_assert(oYh + 7 * 16 * 24 * 2 <= oKV, "aliases fit in the operand area");
  static_assert(oKV + (size_t)(kWuN / 64) * 8192 <= oPst, "the [w | u] tiles fit the area of its operand");
  static_assert((oRow % 1024) == 0 && (oCol % 1024) == 0 && (kRowAtom % 1024) == 0 && (kColAtom % 1024) == 0 &&
                    (oXb % 1024) == 0 && (oKV % 1024) == 0 && (oPst % 1024) == 0 && (oBar % 8) == 0 &&
                    (oRawV % 1024) == 0,
                "TMA, tcgen05 operand and mbarrier alignment");
  static_assert(kAlloc <= 232448, "fits the 227 KB shared-memory limit");
  // The pair path keeps the per-token decays (fp32 [64][DK], rows 0-31 and 32-63)
  // in column-operand rows 0-127 of the two channel atoms, which its product
  // does not read.
  static constexpr size_t oAlpha0 = oCol, oAlpha1 = oCol + kColAtom;
  static_assert(32 * DK * 4 <= 128 * 128, "half of the decays fits 128 operand rows");
};

// (r, i) of the s-th strictly lower pair of a 16x16 block (0 <= s < 120), the
// order the pair path enumerates them in: rows r = 1..15, and in each row the
// columns i = r-1 down to 0, s = r (r - 1) / 2 + (r - 1 - i).
__device__ __forceinline__ void pair_unrank(int s, int& r, int& i) {
  r = 1;
  while ((r + 1) * r / 2 <= s) ++r;
  i = r - 1 - (s - r * (r - 1) / 2);
}

// Byte offset of (row, channel) in a K-major 128-byte-swizzled operand whose
// 64-channel atoms hold `rows` rows each.
__device__ __forceinline__ uint32_t opnd_off(int rows, int row, int ch) {
  return (uint32_t)(ch >> 6) * (uint32_t)rows * 128u + tc::sw128_offset(row, ch & 63);
}


// One CTA's share of the prep tasks, cta + i * ncta (chunk-major), run by the
// whole CTA.  With `ready`, the records are published (publish_records) in
// groups of kPublishBatch, each at the earliest two tasks of this CTA later, when
// its [w | u] stores, issued a task later, are complete (the CTA's records are
// consecutive tasks, ncta apart).
template <int DV, int kVariant>
__device__ __forceinline__ void prep_body(const CUtensorMap& tmG, const CUtensorMap& tmK, const CUtensorMap& tmQ,
                                          const CUtensorMap& tmV, const CUtensorMap& tmWs, const CUtensorMap& tmUs,
                                          const CUtensorMap& tmPs, const float* __restrict__ beta, int32_t num_seqs,
                                          int32_t H, const ChunkMap& map, const TcRecords& out, int64_t n_tasks,
                                          int32_t* __restrict__ dev_err, int cta, int ncta,
                                          int32_t* __restrict__ ready) {
  using L = PrepTcSmem<DV, kVariant>;
  constexpr int LDX = L::LDX, LDA = L::LDA;
  constexpr bool kPairs = L::kPairs, kSoftplus = kVariant == kPrepSoftplusPairs;
  // TMEM column of the first block below the diagonal (the pair path's
  // product holds those blocks only)
  constexpr int kLaterCol = kPairs ? 0 : 2 * C;
  constexpr int NTH = kPrepTcThreads;
  // TMEM: the A / P accumulators (columns 0-287) and, after them, the [w | u]
  // accumulator (columns 0-255, rows 0-63 in lanes 0-63)
  constexpr uint32_t kTmemCols = 512;
  constexpr uint32_t kIdescWU = tc::idesc_f16_f32(128, L::kWuN) | (1u << 16);   // B (KV) MN-major
  constexpr int kWuIssuer = 2;   // warp that issues [w | u]
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sRow = smem + L::oRow;   // row operand of the A / P products
  uint8_t* sCol = smem + L::oCol;   // column operand
  uint8_t* sKV = smem + L::oKV;
  uint8_t* sPst = smem + L::oPst;
  float* sTot = reinterpret_cast<float*>(smem + L::oTot);
  float* sBeta = reinterpret_cast<float*>(smem + L::oBeta);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::oBar);
  float* sA = reinterpret_cast<float*>(smem + L::oA);
  uint8_t* sX = smem + L::oXb;
  f16* sAh = reinterpret_cast<f16*>(smem + L::oAh);
  f16* sYh = reinterpret_cast<f16*>(smem + L::oYh);
  const bf16* rawG = reinterpret_cast<const bf16*>(smem + L::oRawG);
  const bf16* rawK = reinterpret_cast<const bf16*>(smem + L::oRawK);
  const bf16* rawQ = reinterpret_cast<const bf16*>(smem + L::oRawQ);
  const bf16* rawV = reinterpret_cast<const bf16*>(smem + L::oRawV);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;

  if (tid == 0) {
    tc::mbar_init(bar, 1);       // raw rows staged
    tc::mbar_init(bar + 1, 1);   // [w | u] products done
    tc::mbar_init(bar + 2, 1);   // A / P products done
    tc::fence_mbar_init();
    tc::tma_prefetch_desc(&tmG);
    tc::tma_prefetch_desc(&tmK);
    tc::tma_prefetch_desc(&tmQ);
    tc::tma_prefetch_desc(&tmV);
  }
  if (warp == 0) {
    tc::tmem_alloc(reinterpret_cast<uint32_t*>(smem + L::oTmem), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<const uint32_t*>(smem + L::oTmem);

  // [w | u] of a task is multiplied on the tensor cores after its inverse and
  // read out of TMEM in the next task, after its gate and scan (or after the
  // last task): the warps of lane quarters 0 and 1 take rows 32(w%4)..+31 and
  // columns 64(w/4)..+63 into 64-column tiles (128-byte swizzle) in the area of
  // the product's own B operand, free once the product is done, which thread 0
  // stores to the record with TMA; the tiles are released (bulk read wait)
  // before that area is rewritten.
  // In the fused kernel (with `ready`) the records are read back within a few chunks
  // from L2: they are stored with evict-last priority and the inputs, read once,
  // loaded with evict-first; alone, prep keeps the default priority.
  const uint64_t pol_in = ready ? tc::l2_policy_evict_first() : tc::l2_policy_evict_normal();
  const uint64_t pol_rec = ready ? tc::l2_policy_evict_last() : tc::l2_policy_evict_normal();
  bool wu_pending = false, bulk_pending = false;   // bulk_pending: thread 0 has record stores in flight
  // thread 0, with `ready`: the record that is complete after the next drain, the
  // oldest complete one not yet published and how many are waiting
  int64_t pub_rec = -1, unpub = -1;
  int n_unpub = 0;
  uint32_t wu_parity = 0, ap_parity = 0;
  int64_t wu_rec = 0;
  // Returns the OR over the CTA of `raw_bad` (taken at the drain's CTA
  // barrier, or at one of its own when nothing is pending); sets drain_ok.
  bool drain_ok = true;
  auto wu_drain = [&](bool raw_bad) -> bool {
    drain_ok = true;
    if (!wu_pending) return __syncthreads_or(raw_bad);
    const bool okw = tc::mbar_wait(bar + 1, wu_parity, kWaitLimit);
    wu_parity ^= 1u;
    wu_pending = false;
    tc::tc_fence_after();
    uint8_t* stg = smem + L::oKV;   // tile t (columns 64t..64t+63) at stg + 8 KB * t, in the product's own
                                    // operand area (rewritten only after the pre-product barrier)
    const int qw = warp & 3, cg = warp >> 2;
    if (qw < 2 && 64 * cg < L::kWuN) {
      const int r = 32 * qw + lane;
#pragma unroll
      for (int qt = 0; qt < 4; ++qt) {   // 16 columns at a time (the gate/scan registers are live here)
        float v[16];
        tc::tmem_ld16(tc::tmem_addr(tmem, (uint32_t)(32 * qw), (uint32_t)(64 * cg + 16 * qt)), v);
#pragma unroll
        for (int j = 0; j < 2; ++j)
          *reinterpret_cast<uint4*>(stg + cg * 8192 + xs_off(r, 16 * qt + 8 * j)) =
              make_uint4(pack_f16x2(v[8 * j + 0], v[8 * j + 1]), pack_f16x2(v[8 * j + 2], v[8 * j + 3]),
                         pack_f16x2(v[8 * j + 4], v[8 * j + 5]), pack_f16x2(v[8 * j + 6], v[8 * j + 7]));
      }
    }
    tc::fence_proxy_async_smem();   // the tiles, written by the threads, read by the TMA unit
    tc::tc_fence_before();
    const bool any_raw_bad = __syncthreads_or(raw_bad);
    if (ready && tid == 0) {   // the record two tasks back is complete once all but the last group are
      if (pub_rec >= 0) {
        if (unpub < 0) unpub = pub_rec;
        if (++n_unpub == kPublishBatch) {
          tc::bulk_wait1();
          publish_records(ready, unpub, pub_rec, ncta);
          unpub = -1;
          n_unpub = 0;
        }
      }
      pub_rec = wu_rec;   // complete once its [w | u] stores, issued below, are
    }
    if (tid == 0 && okw) {
#pragma unroll
      for (int t = 0; t < L::kWuN / 64; ++t) {
        if (t < DK / 64)
          tc::tma_store_2d_hint(&tmWs, 64 * t, (int32_t)(wu_rec * 128), stg + t * 8192, pol_rec);
        else
          tc::tma_store_2d_hint(&tmUs, 64 * (t - DK / 64), (int32_t)(wu_rec * C), stg + t * 8192, pol_rec);
      }
      tc::bulk_commit();
      bulk_pending = true;
    }
    drain_ok = okw;
    return any_raw_bad;
  };

  // This CTA's tasks are cta + i * ncta; (chunk, head) of the
  // next two are tracked incrementally, without 64-bit divisions.
  const int32_t n_chunks = map.seq_chunk0[num_seqs];   // negative after malformed cu_seqlens
  const int32_t dj = (int32_t)((unsigned)ncta / (unsigned)H), dh = (int32_t)((unsigned)ncta % (unsigned)H);
  int32_t j_next = (int32_t)((unsigned)cta / (unsigned)H), h_next = (int32_t)((unsigned)cta % (unsigned)H);
  auto advance = [&](int32_t& jt, int32_t& ht) {
    jt += dj;
    ht += dh;
    if (ht >= H) {
      ht -= H;
      ++jt;
    }
  };
  // Chunk record of a task: one 16-byte load, fetched two tasks ahead.
  auto fetch = [&](int64_t t, int32_t jt) -> int4 {
    return (t < n_tasks && jt < n_chunks) ? ld_early_v4(map.chunk_info + jt) : make_int4(0, 0, 0, 0);
  };
  // Staging of a task's raw rows: 64 tokens of one head of g, k, q, v by TMA
  // (zero-filled past the token array; rows past the sequence end are masked
  // by the gate and by beta = 0).  The barrier is armed by thread 0 before the
  // CTA barrier that precedes the four copies, which lanes 0 of warps 12-15
  // issue.  beta of the next task is loaded into a register of threads 0-63
  // at the start of the current one.
  auto arm = [&](int4 ci) {
    if (ci.y > 0 && tid == 0) tc::mbar_arrive_expect_tx(bar, (uint32_t)C * (3 * DK + DV) * 2);
  };
  // `which_mask`: bit t selects tensor t (g, k, q, v); the pair path stages g
  // and v a task ahead as usual, k and q once it has read the current ones.
  auto issue = [&](int32_t ht, int4 ci, unsigned which_mask = 15u) {
    if (ci.y <= 0 || warp < 12 || warp >= 16 || lane != 0) return;
    const int which = warp - 12;
    if (!((which_mask >> which) & 1u)) return;
    const CUtensorMap* m = which == 0 ? &tmG : (which == 1 ? &tmK : (which == 2 ? &tmQ : &tmV));
    tc::tma_load_3d_hint(smem + L::oRawG + (size_t)which * C * DK * 2, m, 0, ht, ci.z, bar, pol_in);
  };
  auto load_beta = [&](int32_t ht, int4 ci) -> float {
    return (tid < ci.y) ? ld_early_f32(beta + ((int64_t)(uint32_t)ci.z + tid) * H + ht) : 0.f;   // ci.y <= 64
  };
  int4 ci_next = fetch(cta, j_next);
  float beta_next = tid < C ? load_beta(h_next, ci_next) : 0.f;
  int32_t j_next2 = j_next, h_next2 = h_next;
  advance(j_next2, h_next2);
  int4 ci_next2 = fetch((int64_t)cta + ncta, j_next2);
  arm(ci_next);
  __syncthreads();
  issue(h_next, ci_next);
  uint32_t parity = 0;

  bool failed = false;
  // Persistent: tasks (chunk j, head h) in chunk-major order, strided over the grid.
  for (int64_t task = cta; task < n_tasks; task += ncta) {
    const int4 ci = ci_next;
    const float beta_cur = beta_next;
    ci_next = ci_next2;   // the next task (record fetched a task ago)
    j_next = j_next2;
    h_next = h_next2;
    if (tid < C) beta_next = load_beta(h_next, ci_next);
    advance(j_next2, h_next2);
    ci_next2 = fetch(task + 2 * (int64_t)ncta, j_next2);
    if (ci.y <= 0) {
      arm(ci_next);
      __syncthreads();
      issue(h_next, ci_next);
      continue;
    }
    const int len = ci.y;
    const int64_t rec = task;   // == j * H + h
    f16* o_wq = out.wq + rec * 128 * DK;
    f16* o_kt = out.kt + rec * DK * C;
    float* o_gam = out.gam + rec * DK;

    // 1. Thread -> channel pair (c, c+1) and the 8 rows r0..r0+7 of sub-tile a.
    //    Gate and inclusive cumulative sum over the thread's rows, in registers;
    //    the raw k, q, v of the thread are read before the area is reused.
    const int rg = tid >> 6, a = rg >> 1, c = (tid & 63) * 2, r0 = 8 * rg;
    if (tid < C) sBeta[tid] = beta_cur;   // visible after the next CTA barrier
    // (A copy that never landed leaves stale rows here; the CTA barrier of the
    // drain below tells every thread, and nothing read from them is used.)
    const bool ok = tc::mbar_wait(bar, parity, kWaitLimit);
    float2 G[8];
    {
      float2 run = make_float2(0.f, 0.f);
      if (r0 + 8 <= len) {   // every row of the thread is a token (warp-uniform)
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) {
          const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(rawG + (r0 + rr) * DK + c);
          run.x += log2_decay<kSoftplus>(__low2float(x));
          run.y += log2_decay<kSoftplus>(__high2float(x));
          G[rr] = run;
        }
      } else {               // rows past the sequence end carry no decay
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) {
          const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(rawG + (r0 + rr) * DK + c);
          if (r0 + rr < len) {
            run.x += log2_decay<kSoftplus>(__low2float(x));
            run.y += log2_decay<kSoftplus>(__high2float(x));
          }
          G[rr] = run;
        }
      }
      *reinterpret_cast<float2*>(sTot + rg * DK + c) = run;
    }
    __nv_bfloat162 kq[8], qq[8];
#pragma unroll
    for (int rr = 0; rr < 8; ++rr) {
      kq[rr] = *reinterpret_cast<const __nv_bfloat162*>(rawK + (r0 + rr) * DK + c);
      qq[rr] = *reinterpret_cast<const __nv_bfloat162*>(rawQ + (r0 + rr) * DK + c);
    }
    constexpr int kPerV = C * (DV / 8) / NTH;   // 2 or 1
    uint4 vraw[kPerV];
#pragma unroll
    for (int e2 = 0; e2 < kPerV; ++e2) {
      const int idx = tid + e2 * NTH;
      vraw[e2] = *reinterpret_cast<const uint4*>(rawV + (idx / (DV / 8)) * DV + (idx % (DV / 8)) * 8);
    }
    arm(ci_next);
    // The previous task's [w | u], whose product ran during the steps above.
    // The drain's CTA barrier also ends every raw read, makes the group sums
    // visible and tells every thread whether a raw-row copy failed to land.
    if (wu_drain(!ok)) {   // a staging copy never landed: report, drain, stop
      if (tid == 0) atomicExch(dev_err, (int32_t)kDevErrTimeout);
      tc::mbar_wait(bar, parity, kWaitLimit);
      failed = true;
      break;
    }
    if (!drain_ok && tid == 0) atomicExch(dev_err, (int32_t)kDevErrTimeout);
    parity ^= 1u;
    issue(h_next, ci_next, kPairs ? 0x9u : 15u);   // the pair path reads k and q until its epilogue

    // 2. Offsets from the group sums: G_s(a') = cumulative decay before sub-tile
    //    a', G_last; then the per-thread factors e^{G_s(a') - G_s(a)}, a' >= a.
    float2 gsA[4], gl;
    {
      float2 acc = make_float2(0.f, 0.f), excl = acc;
#pragma unroll
      for (int r2 = 0; r2 < 8; ++r2) {
        if ((r2 & 1) == 0) gsA[r2 >> 1] = acc;
        if (r2 == rg) excl = acc;
        const float2 t2 = *reinterpret_cast<const float2*>(sTot + r2 * DK + c);
        acc.x += t2.x;
        acc.y += t2.y;
      }
      gl = acc;
      if constexpr (kPairs) {   // the per-token decay alpha_r = 2^{G_r - G_{r-1}} for the pair path, from the
                                // thread's own partial sums (small exponents)
        float* adst = reinterpret_cast<float*>(smem + (rg < 4 ? L::oAlpha0 : L::oAlpha1)) + (r0 & 31) * DK + c;
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) {
          const float2 prev = rr ? G[rr - 1] : make_float2(0.f, 0.f);
          *reinterpret_cast<float2*>(adst + rr * DK) =
              make_float2(ex2_approx(G[rr].x - prev.x), ex2_approx(G[rr].y - prev.y));
        }
      }
#pragma unroll
      for (int rr = 0; rr < 8; ++rr) {
        G[rr].x += excl.x;
        G[rr].y += excl.y;
      }
    }
    float2 gs = gsA[0];   // G_s(a), selected without a dynamic register index
#pragma unroll
    for (int a2 = 1; a2 < 4; ++a2)
      if (a2 == a) gs = gsA[a2];
    float2 om[4];
#pragma unroll
    for (int a2 = 0; a2 < 4; ++a2)
      om[a2] = (!kPairs && a2 > a) ? make_float2(ex2_approx(gsA[a2].x - gs.x), ex2_approx(gsA[a2].y - gs.y))
                                   : make_float2(a2 == a ? 1.f : 0.f, a2 == a ? 1.f : 0.f);
    if (rg == 0) {
      tc::st_global_hint(o_gam + c, __float_as_uint(ex2_approx(gl.x)), pol_rec);
      tc::st_global_hint(o_gam + c + 1, __float_as_uint(ex2_approx(gl.y)), pol_rec);
    }

    // 3. The operands of the A / P products (every 16-bit operand is stored as
    //    a 32-bit pair).
#pragma unroll
    for (int rr = 0; rr < 8; ++rr) {
      const int r = r0 + rr;
      const float2 gr = G[rr];
      const float e0 = ex2_approx(gr.x - gs.x), e1 = ex2_approx(gr.y - gs.y);   // e^{G_r - G_s} in (e^-80, 1]: normal
      const float k0 = __low2float(kq[rr]), k1 = __high2float(kq[rr]);
      const float q0 = __low2float(qq[rr]), q1 = __high2float(qq[rr]);
      *reinterpret_cast<uint32_t*>(sRow + opnd_off(L::kRowRows, r, c)) = pack_bf16x2(k0 * e0, k1 * e1);
      if constexpr (kPairs) {   // blocks below the diagonal only: every factor e^{G_a - G_b} <= 1, one ex2 each
        *reinterpret_cast<uint32_t*>(sRow + opnd_off(L::kRowRows, C + r, c)) = pack_bf16x2(q0 * e0, q1 * e1);
#pragma unroll
        for (int a2 = 1; a2 < 4; ++a2) {
          if (a2 > a)
            *reinterpret_cast<uint32_t*>(sCol + opnd_off(L::kColRows, 2 * C + later_row0(a2) + r, c)) =
                pack_bf16x2(k0 * ex2_approx(gsA[a2].x - gr.x), k1 * ex2_approx(gsA[a2].y - gr.y));
        }
        continue;
      }
      const float f0 = rcp_approx(e0), f1 = rcp_approx(e1);                     // e^{G_s - G_r} in [1, e^80)
      uint32_t hi, lo;
      split_bf16x2(q0 * e0, q1 * e1, hi, lo);
      *reinterpret_cast<uint32_t*>(sRow + opnd_off(L::kRowRows, C + r, c)) = hi;
      *reinterpret_cast<uint32_t*>(sRow + opnd_off(L::kRowRows, 2 * C + r, c)) = lo;
      const float kf0 = k0 * f0, kf1 = k1 * f1;
      split_bf16x2(kf0, kf1, hi, lo);   // own sub-tile: high and low parts
      *reinterpret_cast<uint32_t*>(sCol + opnd_off(L::kColRows, r, c)) = hi;
      *reinterpret_cast<uint32_t*>(sCol + opnd_off(L::kColRows, C + r, c)) = lo;
#pragma unroll
      for (int a2 = 1; a2 < 4; ++a2) {   // later sub-tiles: factors <= 1, high part only
        if (a2 > a)
          *reinterpret_cast<uint32_t*>(sCol + opnd_off(L::kColRows, 2 * C + later_row0(a2) + r, c)) =
              pack_bf16x2(kf0 * om[a2].x, kf1 * om[a2].y);
      }
    }
    if (bulk_pending) {   // thread 0: the P and [w | u] tiles stored so far have been read by the TMA unit
      tc::bulk_wait_read0();   // (both areas are rewritten after the barrier below)
      bulk_pending = false;
    }
    tc::fence_proxy_async_smem();   // the operands, written by the threads, read by the MMAs
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();

    // 4. A and P on the tensor cores (bf16 operands, fp32 accumulators in TMEM):
    //      D1 = [k e^G ; q e^G high] (M = 128) x (column operand)^T (N = 224, K = d_k)
    //      D2 = [q e^G high ; low]   (M = 128) x (own sub-tile, high part)^T (N = 64)
    //    A_ri = beta_r D1[r][..] (rows 0-63); P_ri = D1[64 + r][..], plus, on the
    //    diagonal blocks, the low-part products D1[64 + r][64 + i] + D2[64 + r][i].
    if (tid == 0) {   // one thread issues (a whole-warp issue measured 3 % slower here)
      const uint64_t dR = tc::desc_kmajor_sw128(tc::smem_u32(sRow));
      // the pair path multiplies by the later sub-tiles' rows only (128-223: N = 96)
      const uint64_t dC = tc::desc_kmajor_sw128(tc::smem_u32(sCol + (kPairs ? 2 * C * 128 : 0)));
      constexpr uint32_t kId1 = tc::idesc_bf16_f32(128, kPairs ? L::kColRows - 2 * C : L::kColRows),
                         kId2 = tc::idesc_bf16_f32(128, C);
#pragma unroll
      for (int kk = 0; kk < DK / 16; ++kk) {
        const uint64_t oR = (((kk >> 2) * L::kRowAtom) + (kk & 3) * 32) >> 4;
        const uint64_t oC = (((kk >> 2) * L::kColAtom) + (kk & 3) * 32) >> 4;
        tc::mma_16bit(tmem, dR + oR, dC + oC, kId1, kk > 0);
      }
#pragma unroll
      for (int kk = 0; kk < (kPairs ? 0 : DK / 16); ++kk) {
        const uint64_t oR = (((kk >> 2) * L::kRowAtom) + C * 128 + (kk & 3) * 32) >> 4;
        const uint64_t oC = (((kk >> 2) * L::kColAtom) + (kk & 3) * 32) >> 4;
        tc::mma_16bit(tmem + L::kColRows, dR + oR, dC + oC, kId2, kk > 0);
      }
      tc::mma_commit(bar + 2);
    }

    // While they run: [beta k e^G | beta V] (the operand of [w | u]), and the
    // record's q e^G rows and (k e^{G_last - G})^T, with G taken from the chunk
    // start (2^G and 2^{G_last - G} directly).
    {
      uint32_t kt0[4], kt1[4];   // K~^T rows c and c+1, tokens r0..r0+7, fp16 pairs
      float bw[8];   // beta of the thread's rows (two broadcast loads)
      *reinterpret_cast<float4*>(bw) = *reinterpret_cast<const float4*>(sBeta + r0);
      *reinterpret_cast<float4*>(bw + 4) = *reinterpret_cast<const float4*>(sBeta + r0 + 4);
#pragma unroll
      for (int rr = 0; rr < 8; ++rr) {
        const int r = r0 + rr;
        const float2 gr = G[rr];
        const float eg0 = ex2_approx(gr.x), eg1 = ex2_approx(gr.y);                 // e^{G_r}
        const float el0 = ex2_approx(gl.x - gr.x), el1 = ex2_approx(gl.y - gr.y);   // e^{G_last - G_r}
        const float k0 = __low2float(kq[rr]), k1 = __high2float(kq[rr]);
        const float q0 = __low2float(qq[rr]), q1 = __high2float(qq[rr]);
        const float br = bw[rr];
        *reinterpret_cast<uint32_t*>(sKV + kv_off(r, c)) = pack_f16x2(br * k0 * eg0, br * k1 * eg1);
        tc::st_global_hint(o_wq + (C + r) * DK + c, pack_f16x2(q0 * eg0, q1 * eg1), pol_rec);
        const __half2 kt = __floats2half2_rn(k0 * el0, k1 * el1);
        const uint32_t lo16 = *reinterpret_cast<const uint16_t*>(&kt.x), hi16 = *reinterpret_cast<const uint16_t*>(&kt.y);
        if (rr & 1) {
          kt0[rr >> 1] |= lo16 << 16;
          kt1[rr >> 1] |= hi16 << 16;
        } else {
          kt0[rr >> 1] = lo16;
          kt1[rr >> 1] = hi16;
        }
      }
      tc::st_global_hint(o_kt + c * C + r0, make_uint4(kt0[0], kt0[1], kt0[2], kt0[3]), pol_rec);
      tc::st_global_hint(o_kt + (c + 1) * C + r0, make_uint4(kt1[0], kt1[1], kt1[2], kt1[3]), pol_rec);
#pragma unroll
      for (int e2 = 0; e2 < kPerV; ++e2) {   // beta V (beta is 0 on rows past the sequence end)
        const int idx = tid + e2 * NTH;
        const int r = idx / (DV / 8), c8 = (idx % (DV / 8)) * 8;
        const bf16* x = reinterpret_cast<const bf16*>(&vraw[e2]);
        const float br = sBeta[r];
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) pk[e] = pack_f16x2(br * __bfloat162float(x[2 * e]), br * __bfloat162float(x[2 * e + 1]));
        *reinterpret_cast<uint4*>(sKV + kv_off(r, DK + c8)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
    }
    // 4b. The pair path: the diagonal 16x16 blocks of A and P from the raw k, q
    //     and the per-token decays, on the CUDA cores while the products run.
    //     Warp w takes a quarter (w % 4) of the 256 entries of sub-tile w / 4:
    //     entries 2s and 2s + 1 are A and P of the s-th strictly lower pair
    //     (r, i), entries 240 + d the P diagonal (d, d).  A lane sums over its 4
    //     key channels, with the pair's decay e^{G_r - G_i} = prod_{i<m<=r} alpha_m
    //     carried along the row as i descends (one product per pair, every
    //     factor <= 1, so no exponent can leave the range whatever the map);
    //     the warp then reduces over lanes in halving steps (each lane keeps half
    //     of the entries it still holds, plus its partner's copy of them), so
    //     lane l ends with the warp's entries 2l and 2l + 1.
    float pv[2] = {0.f, 0.f};
    if constexpr (kPairs) {
      const int sa = warp >> 2, part = warp & 3, c4 = 4 * lane, row0 = 16 * sa;
      auto alpha_row = [&](int row) -> float4 {   // row within the sub-tile
        const int rc = row0 + row;
        const float* base = reinterpret_cast<const float*>(smem + (rc < 32 ? L::oAlpha0 : L::oAlpha1));
        return *reinterpret_cast<const float4*>(base + (rc & 31) * DK + c4);
      };
      auto unpack = [](uint2 w, float (&x)[4]) {
        x[0] = __uint_as_float(w.x << 16);
        x[1] = __uint_as_float(w.x & 0xffff0000u);
        x[2] = __uint_as_float(w.y << 16);
        x[3] = __uint_as_float(w.y & 0xffff0000u);
      };
      auto ld_bf4 = [&](const bf16* base, int row) -> uint2 {
        return *reinterpret_cast<const uint2*>(base + (row0 + row) * DK + c4);
      };
      // A cursor: pair (r, i), k and q of row r (as floats), and e = e^{G_r - G_i}
      // per channel.
      struct Cursor {
        int r, i;
        float k[4], q[4];
        float4 e;
      };
      auto start = [&](Cursor& cu, int sidx) {
        pair_unrank(sidx, cu.r, cu.i);
        unpack(ld_bf4(rawK, cu.r), cu.k);
        unpack(ld_bf4(rawQ, cu.r), cu.q);
        cu.e = alpha_row(cu.r);
        for (int m = cu.r - 1; m > cu.i; --m) {   // a start inside the row
          const float4 am = alpha_row(m);
          cu.e = make_float4(cu.e.x * am.x, cu.e.y * am.y, cu.e.z * am.z, cu.e.w * am.w);
        }
      };
      auto advance = [&](Cursor& cu) {   // warp-uniform: every lane walks the same pairs
        if (cu.i == 0) {                  // next row, first pair (r + 1, r)
          ++cu.r;
          cu.i = cu.r - 1;
          unpack(ld_bf4(rawK, cu.r), cu.k);
          unpack(ld_bf4(rawQ, cu.r), cu.q);
          cu.e = alpha_row(cu.r);
        } else {                          // (r, i - 1): one more factor alpha_i
          const float4 am = alpha_row(cu.i);
          cu.e = make_float4(cu.e.x * am.x, cu.e.y * am.y, cu.e.z * am.z, cu.e.w * am.w);
          --cu.i;
        }
      };
      auto term = [&](const Cursor& cu, float& av, float& pw) {
        float ki[4];
        unpack(ld_bf4(rawK, cu.i), ki);
        const float e[4] = {cu.e.x, cu.e.y, cu.e.z, cu.e.w};
        av = 0.f;
        pw = 0.f;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const float t = ki[ch] * e[ch];
          av = fmaf(cu.k[ch], t, av);
          pw = fmaf(cu.q[ch], t, pw);
        }
      };
      auto diag = [&](int d) -> float {   // P (d, d): the factor is e^0
        float kr[4], qr[4];
        unpack(ld_bf4(rawK, d), kr);
        unpack(ld_bf4(rawQ, d), qr);
        return fmaf(qr[3], kr[3], fmaf(qr[2], kr[2], fmaf(qr[1], kr[1], qr[0] * kr[0])));
      };
      // pairs 32 part + m (lower half of the entries) and 32 part + 16 + m (upper half)
      const bool hi_pairs = part < 3;   // part 3: 8 upper pairs (s = 112..119), then the P diagonal
      Cursor lo, hi;
      start(lo, 32 * part);
      start(hi, 32 * part + 16);
      const bool up = (lane & 16) != 0;
      float keep[32];
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        float a_lo, p_lo, a_hi, p_hi;
        term(lo, a_lo, p_lo);
        if (hi_pairs || m < 8) {
          term(hi, a_hi, p_hi);
        } else {
          a_hi = diag(2 * (m - 8));
          p_hi = diag(2 * (m - 8) + 1);
        }
        const float xa = __shfl_xor_sync(0xffffffffu, up ? a_lo : a_hi, 16);
        const float xp = __shfl_xor_sync(0xffffffffu, up ? p_lo : p_hi, 16);
        keep[2 * m] = (up ? a_hi : a_lo) + xa;
        keep[2 * m + 1] = (up ? p_hi : p_lo) + xp;
        if (m < 15) {
          advance(lo);
          if (hi_pairs || m < 7) advance(hi);
        }
      }
#pragma unroll
      for (int msk = 8, n = 32; msk >= 1; msk >>= 1, n >>= 1) {
        const bool hb = (lane & msk) != 0;
#pragma unroll
        for (int j = 0; j < n / 2; ++j) {
          const float x = __shfl_xor_sync(0xffffffffu, hb ? keep[j] : keep[n / 2 + j], msk);
          keep[j] = (hb ? keep[n / 2 + j] : keep[j]) + x;
        }
      }
      pv[0] = keep[0];
      pv[1] = keep[1];
    }

    // 5. A and P out of TMEM: A to shared memory, P to the record tile.
    {
      const bool okap = tc::mbar_wait(bar + 2, ap_parity, kWaitLimit);
      ap_parity ^= 1u;
      if (!okap) atomicExch(dev_err, (int32_t)kDevErrTimeout);
      tc::tc_fence_after();
      // Warp -> TMEM lane quarter q (rows 32(q%2).. of A for q < 2, of P for
      // q >= 2) and 16-column block b; each lane holds one row r of sub-tile ar.
      const int q = warp & 3, b = warp >> 2;
      const uint32_t tl = (uint32_t)(32 * q);
      const int rr = 32 * (q & 1) + lane, ar = rr >> 4;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const int ap = 2 * (q & 1) + part;   // the sub-tile of lanes 16 part .. 16 part + 15
        float v[16];
        if (q < 2) {
          if (b > ap || (kPairs && b == ap)) continue;   // the pair path writes the diagonal blocks
          tc::tmem_ld16(tc::tmem_addr(tmem, tl, b == ap ? 16 * b : kLaterCol + later_row0(ap) + 16 * b), v);
          if (ar != ap) continue;
          const float br = sBeta[rr];
          if (b == ap) {   // diagonal block, fp32 (only its strictly lower part is read)
#pragma unroll
            for (int i = 0; i < 16; ++i) sA[rr * LDA + 16 * b + i] = br * v[i];
          } else {         // below the diagonal, fp16
            uint4* dst = reinterpret_cast<uint4*>(sAh + rr * LDX + 16 * b);
#pragma unroll
            for (int j = 0; j < 2; ++j)
              dst[j] = make_uint4(pack_f16x2(br * v[8 * j + 0], br * v[8 * j + 1]), pack_f16x2(br * v[8 * j + 2], br * v[8 * j + 3]),
                                  pack_f16x2(br * v[8 * j + 4], br * v[8 * j + 5]), pack_f16x2(br * v[8 * j + 6], br * v[8 * j + 7]));
          }
        } else {
          if (b > ap) {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = 0.f;
          } else if (b == ap) {
            if constexpr (kPairs) continue;
            float w2[16];
            tc::tmem_ld16(tc::tmem_addr(tmem, tl, 16 * b), v);
            tc::tmem_ld16(tc::tmem_addr(tmem, tl, C + 16 * b), w2);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] += w2[i];
            tc::tmem_ld16(tc::tmem_addr(tmem, tl, L::kColRows + 16 * b), w2);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = i <= (rr & 15) ? v[i] + w2[i] : 0.f;   // inclusive lower triangle
          } else {
            tc::tmem_ld16(tc::tmem_addr(tmem, tl, kLaterCol + later_row0(ap) + 16 * b), v);
          }
          if (ar != ap) continue;
#pragma unroll
          for (int j = 0; j < 2; ++j)
            *reinterpret_cast<uint4*>(sPst + xs_off(rr, 16 * b + 8 * j)) =
                make_uint4(pack_f16x2(v[8 * j + 0], v[8 * j + 1]), pack_f16x2(v[8 * j + 2], v[8 * j + 3]),
                           pack_f16x2(v[8 * j + 4], v[8 * j + 5]), pack_f16x2(v[8 * j + 6], v[8 * j + 7]));
        }
      }
    }
    if constexpr (kPairs) {   // the pair path's entries: A (beta-weighted, fp32) and P (fp16, zero above)
      const int sa = warp >> 2, part = warp & 3;
      if (part < 3 || lane < 24) {
        int r, i;
        pair_unrank(32 * part + lane, r, i);
        const int R = 16 * sa + r, I = 16 * sa + i;
        sA[R * LDA + I] = sBeta[R] * pv[0];
        *reinterpret_cast<f16*>(sPst + xs_off(R, I)) = __float2half_rn(pv[1]);
        *reinterpret_cast<f16*>(sPst + xs_off(I, R)) = __float2half_rn(0.f);
      } else {
        const int R = 16 * sa + 2 * (lane - 24);
        *reinterpret_cast<f16*>(sPst + xs_off(R, R)) = __float2half_rn(pv[0]);
        *reinterpret_cast<f16*>(sPst + xs_off(R + 1, R + 1)) = __float2half_rn(pv[1]);
      }
    }
    tc::tc_fence_before();
    tc::fence_proxy_async_smem();   // the P tile, written by the threads, read by the TMA unit
    __syncthreads();
    if (tid == 0) {   // P to the record (the tile is released before the next task's product barrier)
      tc::tma_store_2d_hint(&tmPs, 0, (int32_t)(rec * C), sPst, pol_rec);
      tc::bulk_commit();
      bulk_pending = true;
    }
    if constexpr (kPairs) issue(h_next, ci_next, 0x6u);   // k and q of this task are no longer read

    // 6. X = (I + A)^{-1}, in fp16 (the precision w and u are formed in):
    //    diagonal 16x16 blocks (only their strictly lower parts are read) by
    //    forward substitution in fp32, one column per thread in registers;
    //    then the blocks below them on tensor cores, in two stages of
    //    dependent 16x16 products (T blocks rounded to fp16 like X):
    //      1: X_10 = -X_11 A_10 X_00,  X_32 = -X_33 A_32 X_22,  T_21 = A_21 X_11,  T_31 = A_31 X_11
    //      2: X_20 = -X_22 T_20,  X_21 = -X_22 T_21,  X_30 = -(X_32 T_20 + X_33 T_30),
    //         X_31 = -(X_32 T_21 + X_33 T_31),  with T_a0 = A_a0 X_00 + A_a1 X_10.
    if (warp < C / kSub && lane < kSub) {   // block `warp`, column `lane`
      const int base = warp * kSub, jc = lane;
      float xc[kSub];
#pragma unroll
      for (int r = 0; r < kSub; ++r) xc[r] = (r == jc) ? 1.f : 0.f;
      // right-looking: once x_i is final it is folded into every later row, so
      // the dependent chain is 16 steps long (rows above jc stay exactly 0)
#pragma unroll
      for (int i = 0; i < kSub - 1; ++i) {
#pragma unroll
        for (int r = i + 1; r < kSub; ++r) xc[r] -= sA[(base + r) * LDA + base + i] * xc[i];
      }
#pragma unroll
      for (int r = 0; r < kSub; ++r) *reinterpret_cast<f16*>(sX + xs_off(base + r, base + jc)) = __float2half_rn(xc[r]);
    }
    constexpr int kZeroThreads = NTH - 32 * (C / kSub);   // the warps not inverting a block
    if (tid >= NTH - kZeroThreads) {
      const int z = tid - (NTH - kZeroThreads);
      for (int idx = z; idx < 6 * 32; idx += kZeroThreads) {   // zeros above the block diagonal of X (16-byte chunks)
        const int blk = idx >> 5, e = idx & 31;
        const int ra = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
        const int rb = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
        *reinterpret_cast<uint4*>(sX + xs_off(16 * ra + (e >> 1), 16 * rb + 8 * (e & 1))) = make_uint4(0u, 0u, 0u, 0u);
      }
      for (int idx = z; idx < C * 8; idx += kZeroThreads)   // rows 64-127 of the MMA's A tile are zero
        *reinterpret_cast<uint4*>(sX + C * 128 + idx * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
    {
      // m16n8k16 fragments: A_am (row-major, fp16 [64][LDX]), X_am as the A
      // operand, X_mb or a [16][24] scratch block as the B operand (two n-tiles).
      auto ld_a = [&](int ra, int m, uint32_t (&f)[4]) {
        ldsm_x4(tc::smem_u32(sAh + (16 * ra + (lane & 15)) * LDX + 16 * m + (lane >> 4) * 8), f[0], f[1], f[2], f[3]);
      };
      auto ld_xa = [&](int ra, int m, uint32_t (&f)[4]) {
        ldsm_x4(tc::smem_u32(sX + xs_off(16 * ra + (lane & 15), 16 * m + (lane >> 4) * 8)), f[0], f[1], f[2], f[3]);
      };
      auto ld_xb = [&](int m, int rb, uint32_t (&f)[4]) {
        ldsm_x4_t(tc::smem_u32(sX + xs_off(16 * m + (lane & 7) + ((lane >> 3) & 1) * 8, 16 * rb + (lane >> 4) * 8)),
                  f[0], f[1], f[2], f[3]);
      };
      auto ld_tb = [&](const f16* t, uint32_t (&f)[4]) {
        ldsm_x4_t(tc::smem_u32(t + ((lane & 7) + ((lane >> 3) & 1) * 8) * 24 + (lane >> 4) * 8), f[0], f[1], f[2], f[3]);
      };
      auto mma_nn = [&](float (&y)[2][4], const uint32_t (&fa)[4], const uint32_t (&fb)[4]) {
        mma16816_f16(y[0], fa[0], fa[1], fa[2], fa[3], fb[0], fb[1]);
        mma16816_f16(y[1], fa[0], fa[1], fa[2], fa[3], fb[2], fb[3]);
      };
      auto st_t = [&](f16* t, const float (&y)[2][4]) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          *reinterpret_cast<uint32_t*>(t + gq * 24 + 8 * nt + 2 * tq) = pack_f16x2(y[nt][0], y[nt][1]);
          *reinterpret_cast<uint32_t*>(t + (gq + 8) * 24 + 8 * nt + 2 * tq) = pack_f16x2(y[nt][2], y[nt][3]);
        }
      };
      auto st_x = [&](int ra, int rb, const float (&y)[2][4]) {   // X_ab = -y
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          *reinterpret_cast<uint32_t*>(sX + xs_off(16 * ra + gq, 16 * rb + 8 * nt + 2 * tq)) = pack_f16x2(-y[nt][0], -y[nt][1]);
          *reinterpret_cast<uint32_t*>(sX + xs_off(16 * ra + gq + 8, 16 * rb + 8 * nt + 2 * tq)) = pack_f16x2(-y[nt][2], -y[nt][3]);
        }
      };
      constexpr int kBlk = 16 * 24;   // one scratch block: 0, 1 stage-1 products, 2 T_21, 3 T_31, 4, 5 T_20, 6 T_30
      uint32_t fa[4], fb[4];
      if (warp < 2) {   // stage 1: X_10 (warp 0), X_32 (warp 1)
        const int ra = warp == 0 ? 1 : 3, rb = ra - 1;
        float y[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        ld_a(ra, rb, fa);
        ld_xb(rb, rb, fb);
        mma_nn(y, fa, fb);
        f16* yb = sYh + warp * kBlk;
        st_t(yb, y);
        __syncwarp();
        float x[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        ld_xa(ra, ra, fa);
        ld_tb(yb, fb);
        mma_nn(x, fa, fb);
        st_x(ra, rb, x);
      } else if (warp < 4) {   // stage 1: T_21 (warp 2), T_31 (warp 3)
        float y[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        ld_a(warp, 1, fa);
        ld_xb(1, 1, fb);
        mma_nn(y, fa, fb);
        st_t(sYh + warp * kBlk, y);
      }
      __syncthreads();
      float x[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      if (warp == 1) {          // X_21 = -X_22 T_21
        ld_xa(2, 2, fa);
        ld_tb(sYh + 2 * kBlk, fb);
        mma_nn(x, fa, fb);
        st_x(2, 1, x);
      } else if (warp == 3) {   // X_31 = -(X_32 T_21 + X_33 T_31)
        ld_xa(3, 2, fa);
        ld_tb(sYh + 2 * kBlk, fb);
        mma_nn(x, fa, fb);
        ld_xa(3, 3, fa);
        ld_tb(sYh + 3 * kBlk, fb);
        mma_nn(x, fa, fb);
        st_x(3, 1, x);
      } else if (warp == 0 || warp == 2) {   // X_20 (warp 0), X_30 (warp 2): both form T_20
        float t[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        ld_a(2, 0, fa);
        ld_xb(0, 0, fb);
        mma_nn(t, fa, fb);
        ld_a(2, 1, fa);
        ld_xb(1, 0, fb);
        mma_nn(t, fa, fb);
        f16* t20 = sYh + (warp == 0 ? 4 : 5) * kBlk;
        st_t(t20, t);
        if (warp == 2) {
          float t3[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
          ld_a(3, 0, fa);
          ld_xb(0, 0, fb);
          mma_nn(t3, fa, fb);
          ld_a(3, 1, fa);
          ld_xb(1, 0, fb);
          mma_nn(t3, fa, fb);
          st_t(sYh + 6 * kBlk, t3);
        }
        __syncwarp();
        if (warp == 0) {
          ld_xa(2, 2, fa);
          ld_tb(t20, fb);
          mma_nn(x, fa, fb);
          st_x(2, 0, x);
        } else {
          ld_xa(3, 2, fa);
          ld_tb(t20, fb);
          mma_nn(x, fa, fb);
          ld_xa(3, 3, fa);
          ld_tb(sYh + 6 * kBlk, fb);
          mma_nn(x, fa, fb);
          st_x(3, 0, x);
        }
      }
    }

    // 7. [w | u] = X [beta k e^G | beta V] on the tensor cores (M = 128 with X's rows
    //    64-127 zero, N = d_k + d_v, K = 64; fp32 accumulator in TMEM lanes 0-63), read out
    //    at the start of the next task.  (As an M = 64 product, whose rows reach every lane
    //    quarter, all 16 warps could drain it, but that measured slower.)
    tc::fence_proxy_async_smem();   // X and the operand written by the threads, seen by the MMAs
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (tid == 32 * kWuIssuer) {   // lane 0 of warp 2, which has no part in the next drain: it catches up there
      const uint64_t dX = tc::desc_kmajor_sw128(tc::smem_u32(sX));
      const uint64_t dKV = tc::desc_mnmajor_sw128_atoms(tc::smem_u32(sKV), 8192);
#pragma unroll
      for (int kk = 0; kk < C / 16; ++kk)
        tc::mma_16bit(tmem, dX + ((kk * 32) >> 4), dKV + ((kk * 2048) >> 4), kIdescWU, kk > 0);
      tc::mma_commit(bar + 1);
    }
    wu_pending = true;
    wu_rec = rec;
    // No barrier here: until the next task's first one the threads write only
    // sBeta, whose last readers (the A / P epilogue, the operand of [w | u])
    // finished before the barrier above (a barrier here cost 7 %).
  }
  wu_drain(false);   // the last task's [w | u]
  if (!drain_ok && tid == 0) atomicExch(dev_err, (int32_t)kDevErrTimeout);
  if (bulk_pending) tc::bulk_wait0();   // thread 0: every record store has completed
  if (ready && tid == 0 && pub_rec >= 0) publish_records(ready, unpub >= 0 ? unpub : pub_rec, pub_rec, ncta);
  (void)failed;
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

template <int DV, int kVariant>
__global__ void __launch_bounds__(kPrepTcThreads, 1)
    chunk_prep_tc(const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmWs, const __grid_constant__ CUtensorMap tmUs,
                  const __grid_constant__ CUtensorMap tmPs,
                  const float* __restrict__ beta, int32_t num_seqs, int32_t H, ChunkMap map, TcRecords out,
                  int64_t n_tasks, int32_t* __restrict__ dev_err) {
  prep_body<DV, kVariant>(tmG, tmK, tmQ, tmV, tmWs, tmUs, tmPs, beta, num_seqs, H, map, out, n_tasks, dev_err,
                          (int)blockIdx.x, (int)gridDim.x, nullptr);
}

// The bounded map's prep with two task streams per CTA (prep_split_body.cuh):
// the default prep of the plain, gated and snapshot calls.  The single-stream
// kernel above runs the pair-path variants of the decay-map ablation.
template <int DV>
__global__ void __launch_bounds__(ps::kThreads, 1)
    chunk_prep_split_tc(const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmWs,
                        const __grid_constant__ CUtensorMap tmUs, const __grid_constant__ CUtensorMap tmPs,
                        const bf16* __restrict__ v, const float* __restrict__ beta, int32_t num_seqs, int32_t H,
                        ChunkMap map, TcRecords out, int64_t n_tasks, int32_t* __restrict__ dev_err) {
  ps::prep_split_body<DV>(tmG, tmK, tmQ, tmWs, tmUs, tmPs, v, beta, num_seqs, H, map, out, n_tasks, dev_err,
                          (int)blockIdx.x, (int)gridDim.x, nullptr);
}

// -------------------------------------------------------------- chain kernel
// Warp roles: 8 consumer warps (warp w reads TMEM lanes 32(w%4)..+31 and the
// value columns 16(w/4)..+15 of the CTA's block), one TMA producer warp and one
// MMA-issuing warp.  Without the output epilogue the consumer warps of lanes
// 64-127 also write the o rows.  With it, four o warps do: TMEM lanes 64-127
// are readable by warps 2 and 3 mod 4 only, so warps 10 and 11 take value
// columns 0-15 of the o rows and warps 14 and 15 columns 16-31 (12 and 13 have
// no role).  (Dedicated o warps without the epilogue measured 9 % slower.)
constexpr int kChainConsumerWarps = 8;
constexpr int kChainTmaWarp = 8, kChainMmaWarp = 9;
constexpr int kChainOWarp0 = 10, kChainOWarp1 = 14, kChainOWarps = 4;
constexpr int chain_threads(bool gated) { return 32 * (gated ? 16 : kChainConsumerWarps + 2); }
// D12 buffers: one per chunk parity, four with the o warps (which may read a
// chunk's rows while later chunks are formed)
constexpr int chain_buffers(bool gated) { return gated ? 4 : 2; }
constexpr int kMaxRanks = 4;    // CTAs of a head at most (d_v / 32)
// K-major A (TMA-staged tiles), MN-major B (the state block / V_new written by the threads), fp16,
// M = 128, N = 32.
constexpr uint32_t kIdescMN = tc::idesc_f16_f32(128, BV) | (1u << 16);
constexpr uint32_t kTmemD12 = 0;    // D12 buffers of 32 columns, then D3

struct ChainTcSmem {
  // one pipeline stage (all tiles 1024-byte aligned, 128-byte swizzle unless noted)
  static constexpr uint32_t oWQ = 0;           // [w; q e^G] 128 x 128: two 64-column atoms of 16 KB
  static constexpr uint32_t oPZ = 32768;       // [0; P] 128 x 64 (rows 0-63 stay zero)
  static constexpr uint32_t oKT = 49152;       // (k e^{G_last-G})^T 128 x 64
  static constexpr uint32_t oU = 65536;        // u block 64 x 32, 64-byte swizzle (64 B rows)
  static constexpr uint32_t oGam = 69632;      // e^{G_last}, 128 fp32
  static constexpr uint32_t kStage = 71680;    // 70 KB, keeps the next stage 1024-aligned
  static constexpr uint32_t kTxBytes = 32768 + 8192 + 16384 + 64 * BV * 2 + DK * 4;
  static constexpr uint32_t oS = 2 * kStage;   // state block as MN-major B operand: [128 keys][32 value cols]
  static constexpr uint32_t oVN = oS + 8192;   // V_new as MN-major B operand: [64 tokens][32 value cols]
  // output epilogue: the CTA's 32 norm weights, the row sums of squares to send
  // (fp32 [2 parities][4 o warps][32]) and those received (fp32 [2 parities]
  // [kMaxRanks][2 column halves][64 rows])
  static constexpr uint32_t oWgt = oVN + 4096;
  static constexpr uint32_t oStg = oWgt + BV * 4;
  static constexpr uint32_t oRss = oStg + 2 * kChainOWarps * 32 * 4;
  // full[2], empty[2], mma1, mma2, drain, vn_ready, s_ready, cons[2]; with the output
  // epilogue ofull[4], dfree[4], rs[2]
  static constexpr uint32_t oBar = oRss + 2 * kMaxRanks * 2 * 64 * 4;
  static constexpr uint32_t oTmem = oBar + 21 * 8;
  static constexpr uint32_t kBytes = oTmem + 16;
  static constexpr uint32_t kAlloc = kBytes + 1024;   // slack to align the base to 1024
};

// Inter-chunk pass of one (sequence, head, 32-column value block): the state
// lives in fp32 registers of the consumer threads (key channel = TMEM lane),
// its fp16 copy is the B operand of both MMA groups of the next chunk.
//   group 1: D12 = [w; q e^G] S                       (rows 0-63: w S, 64-127: q e^G S)
//   V_new  = u - (w S)                                 (consumers, to SMEM)
//   group 2: D12 += [0; P] V_new (o rows), D3 = K~^T V_new
//   S      = e^{G_last} S + D3                          (consumers)
// With kGated the o rows of a chunk are read by the four o warps once its o
// product has completed, and they apply the output epilogue (Sigmoid gate times
// the per-head RMSNorm of o and its weight) first: a token's d_v outputs are
// spread over the DV/32 CTAs of its head, which the launch groups into one
// thread-block cluster, and each o warp sends its 32 rows' partial sums of
// squares to every CTA of it as one bulk shared-memory copy counted on the
// receiver's mbarrier.
template <int DV, bool kGated>
__global__ void __launch_bounds__(chain_threads(kGated), 1)
    chunk_chain_tc(const __grid_constant__ CUtensorMap tmWQ, const __grid_constant__ CUtensorMap tmP,
                   const __grid_constant__ CUtensorMap tmKT, const __grid_constant__ CUtensorMap tmU,
                   const __grid_constant__ CUtensorMap tmGam, const int32_t* __restrict__ cu, int32_t num_seqs,
                   int64_t T_seq, int32_t H, ChunkMap map, const float* __restrict__ s0, float* __restrict__ s_final,
                   bf16* __restrict__ o, OutEpilogue ep, int32_t* dev_err) {
  using L = ChainTcSmem;
  constexpr int kRanks = DV / BV;                    // CTAs per head (the cluster with kGated)
  static_assert(kRanks <= kMaxRanks, "row-sum slots");
  constexpr uint32_t kNBuf = chain_buffers(kGated);  // D12 buffers
  constexpr uint32_t kTmemD3 = kTmemD12 + kNBuf * BV;
  constexpr uint32_t kTmemCols = kGated ? 256 : 128;
  constexpr int kThreads = chain_threads(kGated);
  static_assert(kTmemD3 + BV <= kTmemCols, "TMEM columns");
  if (map.seq_chunk0[num_seqs] < 0) return;   // malformed cu_seqlens: write nothing
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L::oBar);
  uint64_t* empty = full + 2;
  uint64_t* mma1 = full + 4;
  uint64_t* mma2 = full + 5;
  uint64_t* drain = full + 6;
  uint64_t* vn_ready = full + 7;   // the 4 V_new warps have stored their rows
  uint64_t* s_ready = full + 8;    // the 8 consumer warps have stored the state and read TMEM
  uint64_t* cons = full + 9;       // [2] the 8 consumer warps are done reading a stage (gam, u)
  uint64_t* ofull = full + 11;     // [4] a chunk's o rows are complete in its D12 buffer
  uint64_t* dfree = full + 15;     // [4] the o warps have read a D12 buffer
  uint64_t* rs = full + 19;        // [2] output epilogue: the row sums of every o warp of the cluster have landed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::oTmem);
  uint8_t* sS = sm + L::oS;
  uint8_t* sVN = sm + L::oVN;
  float* sWgt = reinterpret_cast<float*>(sm + L::oWgt);
  float* sStg = reinterpret_cast<float*>(sm + L::oStg);
  float* rss = reinterpret_cast<float*>(sm + L::oRss);

  // one-dimensional grid, sequence-rank major: all blocks of the longest chain first
  const int blk = (int)(blockIdx.x % (unsigned)(H * (DV / BV)));
  const int s = map.seq_order[blockIdx.x / (unsigned)(H * (DV / BV))], h = blk / (DV / BV), n0 = (blk % (DV / BV)) * BV;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int32_t j0 = map.seq_chunk0[s];
  const int32_t nch = map.seq_chunk0[s + 1] - j0;
  const int64_t seq_start = cu ? (int64_t)cu[s] : (int64_t)s * T_seq;
  const int64_t seq_end = cu ? (int64_t)cu[s + 1] : seq_start + T_seq;

  if (tid == 0) {
    for (int i = 0; i < 7; ++i) tc::mbar_init(full + i, 1);
    tc::mbar_init(vn_ready, 4);                      // one arrival per V_new warp
    tc::mbar_init(s_ready, kChainConsumerWarps);     // one arrival per consumer warp
    tc::mbar_init(cons, kChainConsumerWarps);        // one arrival per consumer warp and chunk
    tc::mbar_init(cons + 1, kChainConsumerWarps);
    for (int b = 0; b < (int)kNBuf; ++b) {
      tc::mbar_init(ofull + b, 1);
      tc::mbar_init(dfree + b, kChainOWarps);
    }
    tc::mbar_init(rs, 1);   // one local arrival (with the expected bytes) per phase
    tc::mbar_init(rs + 1, 1);
    tc::fence_mbar_init();
  }
  if (kGated && tid < BV) sWgt[tid] = ep.weight ? ep.weight[(int64_t)h * DV + n0 + tid] : 1.f;
  // rows 0-63 of both [0; P] tiles are zero for the whole kernel
  for (int i = tid; i < 2 * 512; i += kThreads) {
    const int st = i >> 9, off = (i & 511) * 16;
    *reinterpret_cast<uint4*>(sm + st * L::kStage + L::oPZ + off) = make_uint4(0u, 0u, 0u, 0u);
  }
  if (warp == 0) {
    tc::tmem_alloc(tslot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  // the cluster's barriers are initialised before any CTA of it sends row sums
  if constexpr (kGated) tc::cluster_sync_all();
  const uint32_t tmem = *tslot;

  if (warp == kChainTmaWarp) {
    // ---------------- TMA producer
    if (lane == 0) {
      tc::tma_prefetch_desc(&tmWQ);
      tc::tma_prefetch_desc(&tmP);
      tc::tma_prefetch_desc(&tmKT);
      tc::tma_prefetch_desc(&tmU);
      tc::tma_prefetch_desc(&tmGam);
      int issued = 0;
      for (int i = 0; i < nch; ++i) {
        const int st = i & 1;
        // a stage is refilled once the MMAs and every consumer warp are done with
        // its previous chunk: a consumer can then never see this barrier two phases
        // ahead of the chunk it waits for
        if (i >= 2 && !(tc::mbar_wait(empty + st, ((i >> 1) - 1) & 1, kWaitLimit) &&
                        tc::mbar_wait(cons + st, ((i >> 1) - 1) & 1, kWaitLimit))) {
          atomicExch(dev_err, (int32_t)kDevErrTimeout);
          break;
        }
        const int64_t rec = (int64_t)(j0 + i) * H + h;
        uint8_t* stg = sm + st * L::kStage;
        tc::mbar_arrive_expect_tx(full + st, L::kTxBytes);
        tc::tma_load_2d(stg + L::oWQ, &tmWQ, 0, (int32_t)(rec * 128), full + st);
        tc::tma_load_2d(stg + L::oWQ + 16384, &tmWQ, 64, (int32_t)(rec * 128), full + st);
        tc::tma_load_2d(stg + L::oPZ + 8192, &tmP, 0, (int32_t)(rec * C), full + st);
        tc::tma_load_2d(stg + L::oKT, &tmKT, 0, (int32_t)(rec * DK), full + st);
        tc::tma_load_2d(stg + L::oU, &tmU, n0, (int32_t)(rec * C), full + st);
        tc::tma_load_2d(stg + L::oGam, &tmGam, 0, (int32_t)rec, full + st);
        ++issued;
      }
      // never leave loads in flight: wait (bounded) until the last ones landed
      for (int i = (issued > 2 ? issued - 2 : 0); i < issued; ++i) tc::mbar_wait(full + (i & 1), (i >> 1) & 1, kWaitLimit);
    }
  } else if (warp == kChainMmaWarp) {
    // ---------------- MMA issue: the whole warp runs this loop with warp-uniform
    // operands and one elected lane issues (fast back-to-back issue).
    // Descriptors: the B tiles never move; A tiles differ per stage only by the
    // stage offset, K slices by constant offsets added to the start-address field.
    const uint64_t dS0 = tc::desc_mnmajor_sw64(tc::smem_u32(sS));
    const uint64_t dV0 = tc::desc_mnmajor_sw64(tc::smem_u32(sVN));
    const uint64_t dA0 = tc::desc_kmajor_sw128(tc::smem_u32(sm));   // stage 0 base
    auto wait_all = [&](uint64_t* b, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, tc::mbar_wait(b, parity, kWaitLimit));
    };
    bool ok = true, issued = false;
    for (int i = 0; i < nch && ok; ++i) {
      const int st = i & 1;
      ok = wait_all(full + st, (i >> 1) & 1) && wait_all(s_ready, i & 1);
      if (!ok) break;
      tc::tc_fence_after();
      if (kGated && i >= (int)kNBuf) {   // the o warps have read what this buffer held kNBuf chunks ago
        ok = wait_all(dfree + i % (int)kNBuf, (uint32_t)((i / (int)kNBuf) - 1) & 1u);
        if (!ok) break;
        tc::tc_fence_after();
      }
      const uint64_t dA = dA0 + ((uint64_t)(st * L::kStage) >> 4);
      const uint32_t d12 = tmem + kTmemD12 + (uint32_t)(i % (int)kNBuf) * BV;
#pragma unroll
      for (int kk = 0; kk < DK / 16; ++kk)   // group 1
        tc::mma_16bit_w(d12, dA + (((kk >> 2) * 16384 + (kk & 3) * 32) >> 4), dS0 + ((kk * 1024) >> 4), kIdescMN,
                        kk > 0);
      tc::mma_commit_w(mma1);
      issued = true;
      ok = wait_all(vn_ready, i & 1);
      if (!ok) break;
      tc::tc_fence_after();
      // group 2: the state product first, committed on its own, then the o rows
#pragma unroll
      for (int kk = 0; kk < C / 16; ++kk)
        tc::mma_16bit_w(tmem + kTmemD3, dA + ((L::oKT + kk * 32) >> 4), dV0 + ((kk * 1024) >> 4), kIdescMN, kk > 0);
      tc::mma_commit_w(mma2);
#pragma unroll
      for (int kk = 0; kk < C / 16; ++kk)
        tc::mma_16bit_w(d12, dA + ((L::oPZ + kk * 32) >> 4), dV0 + ((kk * 1024) >> 4), kIdescMN, 1u);
      tc::mma_commit_w(empty + st);
      if constexpr (kGated) tc::mma_commit_w(ofull + i % (int)kNBuf);
    }
    if (!ok && lane == 0) atomicExch(dev_err, (int32_t)kDevErrTimeout);
    if (issued) {   // no MMA may still be writing TMEM when it is freed
      tc::mma_commit_w(drain);
      wait_all(drain, 0);
    }
  } else if (warp < kChainConsumerWarps) {
    // ---------------- consumers: TMEM lane quarter q, value columns 16 hf .. 16 hf + 15
    const int q = warp & 3, hf = warp >> 2;
    const int c = 32 * q + lane;   // key channel of this thread's state row; token row for V_new / o
    const uint32_t tl = (uint32_t)(32 * q);
    float S[16];
    {
      const int64_t off = (((int64_t)s * H + h) * DK + c) * DV + n0 + 16 * hf;
#pragma unroll
      for (int n = 0; n < 16; n += 4) {
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (s0) x = *reinterpret_cast<const float4*>(s0 + off + n);
        S[n] = x.x; S[n + 1] = x.y; S[n + 2] = x.z; S[n + 3] = x.w;
      }
    }
    store_mn_half(sS, c, hf, S);
    tc::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(s_ready);
    float nonfinite = 0.f;   // stays 0 unless an o or state value is inf or NaN (x * 0 is then NaN)
    const int r = c - 64;    // without the epilogue, consumer warps q >= 2 write the o rows: token row
    bool bad = false;
    int i = 0;
    int64_t prev_t0 = 0;
    int64_t prev_len = 0;
    for (; i < nch; ++i) {
      const int st = i & 1;
      const uint8_t* stg = sm + st * L::kStage;
      bad |= !tc::mbar_wait(full + st, (i >> 1) & 1, kWaitLimit);
      if (__any_sync(0xffffffffu, bad)) {   // warp-uniform, so that no lane is left at a __syncwarp
        bad = true;
        break;
      }
      const float gam = reinterpret_cast<const float*>(stg + L::oGam)[c];
      if (q >= 2) {
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(cons + st);   // this warp reads nothing more of the stage
      }
      if (!kGated && q >= 2) {
        // previous chunk's o rows (tokens 32(q-2)+lane) from the other buffer,
        // read while the state product is issued: its o product completed
        // before this chunk's group 1 (mma1)
        bad |= !tc::mbar_wait(vn_ready, i & 1, kWaitLimit);
        bad |= !tc::mbar_wait(mma1, i & 1, kWaitLimit);
        if (__any_sync(0xffffffffu, bad)) {   // warp-uniform, so that no lane is left at a __syncwarp
          bad = true;
          break;
        }
        tc::tc_fence_after();
        if (i > 0) {
          float ov[16];
          tc::tmem_ld16(tc::tmem_addr(tmem, tl, kTmemD12 + (uint32_t)(st ^ 1) * BV + 16 * hf), ov);
          if (r < prev_len) {
            store_bf16x16(o + ((prev_t0 + r) * H + h) * DV + n0 + 16 * hf, ov);
#pragma unroll
            for (int e = 0; e < 16; ++e) nonfinite = fmaf(ov[e], 0.f, nonfinite);
          }
        }
      }
      if (q < 2) {   // V_new rows (tokens) 0-63: u - w S
        bad |= !tc::mbar_wait(mma1, i & 1, kWaitLimit);
        if (__any_sync(0xffffffffu, bad)) {   // warp-uniform, so that no lane is left at a __syncwarp
          bad = true;
          break;
        }
        tc::tc_fence_after();
        float d[16];
        tc::tmem_ld16(tc::tmem_addr(tmem, tl, kTmemD12 + (uint32_t)(i % (int)kNBuf) * BV + 16 * hf), d);
#pragma unroll
        for (int q4 = 0; q4 < 2; ++q4) {
          const uint4 raw = *reinterpret_cast<const uint4*>(stg + L::oU + tc::sw64_chunk_offset(c, 2 * hf + q4));
          *reinterpret_cast<uint4*>(sVN + tc::sw64_chunk_offset(c, 2 * hf + q4)) = tcu::vnew_f16x8(raw, d + 8 * q4);
        }
        tc::fence_proxy_async_smem();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive(vn_ready);
          tc::mbar_arrive(cons + st);   // u and gam of the stage have been read
        }
      }
      bad |= !tc::mbar_wait(mma2, i & 1, kWaitLimit);
      if (__any_sync(0xffffffffu, bad)) {   // warp-uniform, so that no lane is left at a __syncwarp
        bad = true;
        break;
      }
      tc::tc_fence_after();
      {
        float d[16];
        tc::tmem_ld16(tc::tmem_addr(tmem, tl, kTmemD3 + 16 * hf), d);
#pragma unroll
        for (int n = 0; n < 16; ++n) S[n] = gam * S[n] + d[n];
        store_mn_half(sS, c, hf, S);
        tc::fence_proxy_async_smem();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(s_ready);
      }
      if (const int64_t slot = snapshot_slot(map, s, i, seq_end - seq_start); slot >= 0) {
        float* dst = map.snaps + ((slot * H + h) * DK + c) * DV + n0 + 16 * hf;
#pragma unroll
        for (int n = 0; n < 16; n += 4) *reinterpret_cast<float4*>(dst + n) = make_float4(S[n], S[n + 1], S[n + 2], S[n + 3]);
      }
      prev_t0 = seq_start + (int64_t)i * C;
      prev_len = min((int64_t)C, seq_end - prev_t0);
    }
    if (!kGated && i == nch && !bad && nch > 0 && q >= 2) {   // the last chunk's o, once the final drain has completed
      bad = __any_sync(0xffffffffu, !tc::mbar_wait(drain, 0, kWaitLimit));
      tc::tc_fence_after();
      if (!bad) {
        float ov[16];
        tc::tmem_ld16(tc::tmem_addr(tmem, tl, kTmemD12 + (uint32_t)((nch - 1) & 1) * BV + 16 * hf), ov);
        if (r < prev_len) {
          store_bf16x16(o + ((prev_t0 + r) * H + h) * DV + n0 + 16 * hf, ov);
#pragma unroll
          for (int e = 0; e < 16; ++e) nonfinite = fmaf(ov[e], 0.f, nonfinite);
        }
      }
    }
    if (i < nch || bad) {
      atomicExch(dev_err, (int32_t)kDevErrTimeout);
    } else {
#pragma unroll
      for (int n = 0; n < 16; ++n) nonfinite = fmaf(S[n], 0.f, nonfinite);
      report_nonfinite(nonfinite, dev_err);
    }
    if (i == nch && !bad && s_final) {
      float* dst = s_final + (((int64_t)s * H + h) * DK + c) * DV + n0 + 16 * hf;
#pragma unroll
      for (int n = 0; n < 16; n += 4) *reinterpret_cast<float4*>(dst + n) = make_float4(S[n], S[n + 1], S[n + 2], S[n + 3]);
    }
  } else if (kGated && (warp & 3) >= 2) {
    // ---------------- o rows (TMEM lanes 64-127, token r of the chunk), value columns 16 hf .. 16 hf + 15
    const int q = warp & 3, r = 32 * (q - 2) + lane, hf = warp >= kChainOWarp1 ? 1 : 0;
    const int wi = 2 * hf + (q - 2);   // this warp's slot in the row-sum exchange
    const uint32_t tl = (uint32_t)(32 * q);
    const uint32_t crank = kGated ? tc::cluster_ctarank() : 0u;
    float nonfinite = 0.f;   // stays 0 unless an o value is inf or NaN (x * 0 is then NaN)
    // gate logits of the row: prefetched into L2 a few chunks ahead, into registers a chunk ahead
    constexpr int kGatePf = 4;
    uint4 gnext[2] = {};
    auto gate_row = [&](int i) -> const bf16* {   // null past the sequence
      const int64_t t0 = seq_start + (int64_t)i * C;
      return (i < nch && r < seq_end - t0) ? ep.gate + ((t0 + r) * H + h) * DV + n0 + 16 * hf : nullptr;
    };
    auto load_gate = [&](int i) {   // issued where it stands
      if (const bf16* gp = gate_row(i)) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int4 v = ld_early_v4(reinterpret_cast<const int4*>(gp) + k);
          gnext[k] = make_uint4((uint32_t)v.x, (uint32_t)v.y, (uint32_t)v.z, (uint32_t)v.w);
        }
      }
    };
    for (int k = 0; k < kGatePf; ++k)
      if (const bf16* gp = gate_row(k)) asm volatile("prefetch.global.L2 [%0];" ::"l"(gp));
    load_gate(0);
    bool bad = false;
    int i = 0;
    for (; i < nch; ++i) {
      const int b = i % (int)kNBuf;
      const int64_t t0 = seq_start + (int64_t)i * C;
      const int64_t len = min((int64_t)C, seq_end - t0);
      bad |= !tc::mbar_wait(ofull + b, (uint32_t)(i / (int)kNBuf) & 1u, kWaitLimit);
      if (__any_sync(0xffffffffu, bad)) {
        bad = true;
        break;
      }
      tc::tc_fence_after();
      float ov[16];
      tc::tmem_ld16(tc::tmem_addr(tmem, tl, kTmemD12 + (uint32_t)b * BV + 16 * hf), ov);
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
        float* stg = sStg + (par * kChainOWarps + wi) * 32;
        if (lane == 0 && i >= 2) tc::bulk_wait_read1();
        __syncwarp();
        stg[lane] = ss;
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          // this CTA expects 128 bytes from each (rank, o warp) of the cluster in this phase
          if (warp == kChainOWarp0) tc::mbar_arrive_expect_tx(rs + par, (uint32_t)kRanks * kChainOWarps * 128u);
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
        if (const bf16* gp = gate_row(i + kGatePf)) asm volatile("prefetch.global.L2 [%0];" ::"l"(gp));
        // the gate and the weight while the other CTAs' row sums arrive (bf16
        // pairs unpacked with shifts, the sigmoid with the fast exponential and divide)
        const float* wt = sWgt + 16 * hf;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const uint32_t gw[4] = {gcur[k].x, gcur[k].y, gcur[k].z, gcur[k].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c0 = 8 * k + 2 * e;
            ov[c0] *= __fdividef(wt[c0], 1.f + __expf(-__uint_as_float(gw[e] << 16)));
            ov[c0 + 1] *= __fdividef(wt[c0 + 1], 1.f + __expf(-__uint_as_float(gw[e] & 0xffff0000u)));
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
        store_bf16x16(o + ((t0 + r) * H + h) * DV + n0 + 16 * hf, ov);
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
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
  // no CTA of the cluster leaves while another may still send it row sums
  if constexpr (kGated) tc::cluster_sync_all();
}

// ------------------------------------------------------- wide chain kernel
// The same inter-chunk pass with NC = 64 or 128 value columns per CTA: the
// per-chunk A tiles are read and the MMAs issued once per NC columns instead
// of once per 32.  Used when the 32-column grid would exceed one wave of the
// GPU and the value-major chain does not apply (d_v = 64, or the output
// epilogue fused), and for a forced 64-column width.  Consumer warp w reads TMEM lanes 32(w%4)..+31 and value columns
// 32(w/4)..+31 of the block; the state block and V_new are MN-major B operands
// of NC/32 atoms of 32 columns.
template <int NC>
struct ChainWideSmem {
  static constexpr int DV = NC;              // value columns held by one CTA
  static constexpr int kConsumerWarps = 4 * (DV / 32);
  static constexpr int kThreads = 32 * (kConsumerWarps + 2);
  static constexpr int kTmaWarp = kConsumerWarps, kMmaWarp = kConsumerWarps + 1;
  static constexpr uint32_t kTmemCols = DV == 128 ? 512 : 256;   // D12 x 3 + D3, DV columns each
  static constexpr uint32_t oWQ = 0;           // [w; q e^G] 128 x 128: two 64-column atoms of 16 KB
  static constexpr uint32_t oPZ = 32768;       // [0; P] 128 x 64 (rows 0-63 stay zero)
  static constexpr uint32_t oKT = 49152;       // (k e^{G_last-G})^T 128 x 64
  static constexpr uint32_t oU = 65536;        // u 64 x DV: DV/64 atoms [64 rows][128 B], 128-byte swizzle
  static constexpr uint32_t oGam = oU + 64 * DV * 2;   // e^{G_last}, 128 fp32
  static constexpr uint32_t kStage = (oGam + DK * 4 + 1023) / 1024 * 1024;
  static constexpr uint32_t kTxBytes = 32768 + 8192 + 16384 + 64 * DV * 2 + DK * 4;
  static constexpr uint32_t kSAtom = DK * 64, kVAtom = C * 64;   // MN atom strides
  static constexpr uint32_t oS = 2 * kStage;                      // state block, DV/32 atoms
  static constexpr uint32_t oVN = oS + (DV / 32) * kSAtom;        // V_new, DV/32 atoms
  static constexpr uint32_t oBar = oVN + (DV / 32) * kVAtom;      // full[2], empty[2], mma1, mma2, drain, vn_ready, s_ready, rs[2], cons[2]
  static constexpr uint32_t oTmem = oBar + 13 * 8;
  static constexpr uint32_t oRss = oTmem + 16;                    // output epilogue: fp32 [2][DV/32][64] row sums of squares
  static constexpr uint32_t kBytes = oRss + 2 * (DV / 32) * 64 * 4;
  static constexpr uint32_t kAlloc = kBytes + 1024;
  static_assert(kAlloc <= 232448, "fits the 227 KB shared-memory limit");
};

// 32 fp32 values of K row `k` of one 32-column MN-major SW64 atom, as fp16.
__device__ __forceinline__ void store_mn_atom_row(uint8_t* atom, int k, const float (&x)[32]) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
    *reinterpret_cast<uint4*>(atom + tc::sw64_chunk_offset(k, j)) =
        make_uint4(pack_f16x2(x[8 * j + 0], x[8 * j + 1]), pack_f16x2(x[8 * j + 2], x[8 * j + 3]),
                   pack_f16x2(x[8 * j + 4], x[8 * j + 5]), pack_f16x2(x[8 * j + 6], x[8 * j + 7]));
}

template <int DV, int NC, bool kGated>
__global__ void __launch_bounds__(ChainWideSmem<NC>::kThreads, 1)
    chunk_chain_wide_tc(const __grid_constant__ CUtensorMap tmWQ, const __grid_constant__ CUtensorMap tmP,
                        const __grid_constant__ CUtensorMap tmKT, const __grid_constant__ CUtensorMap tmU,
                        const __grid_constant__ CUtensorMap tmGam, const int32_t* __restrict__ cu,
                        int32_t num_seqs, int64_t T_seq, int32_t H, ChunkMap map, const float* __restrict__ s0,
                        float* __restrict__ s_final, bf16* __restrict__ o, OutEpilogue ep, int32_t* dev_err) {
  using L = ChainWideSmem<NC>;
  constexpr uint32_t kIdesc = tc::idesc_f16_f32(128, NC) | (1u << 16);
  constexpr uint32_t kD3 = 3 * NC;   // D12 buffers 0-2 (chunk i in buffer i % 3), then D3
  if (map.seq_chunk0[num_seqs] < 0) return;   // malformed cu_seqlens: write nothing
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L::oBar);
  uint64_t* empty = full + 2;
  uint64_t* mma1 = full + 4;
  uint64_t* mma2 = full + 5;
  uint64_t* drain = full + 6;
  uint64_t* vn_ready = full + 7;
  uint64_t* s_ready = full + 8;
  uint64_t* rs_full = full + 9;   // [2] output epilogue: row sums of squares of a chunk published
  uint64_t* cons = full + 11;     // [2] every consumer warp is done reading a stage (gam, u)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::oTmem);
  float* rss = reinterpret_cast<float*>(sm + L::oRss);
  uint8_t* sS = sm + L::oS;
  uint8_t* sVN = sm + L::oVN;

  // one-dimensional grid, sequence-rank major: all blocks of the longest chain first
  const int blk = (int)(blockIdx.x % (unsigned)(H * (DV / NC)));
  const int s = map.seq_order[blockIdx.x / (unsigned)(H * (DV / NC))], h = blk / (DV / NC), n0 = (blk % (DV / NC)) * NC;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int32_t j0 = map.seq_chunk0[s];
  const int32_t nch = map.seq_chunk0[s + 1] - j0;
  const int64_t seq_start = cu ? (int64_t)cu[s] : (int64_t)s * T_seq;
  const int64_t seq_end = cu ? (int64_t)cu[s + 1] : seq_start + T_seq;

  if (tid == 0) {
    for (int i = 0; i < 7; ++i) tc::mbar_init(full + i, 1);
    tc::mbar_init(vn_ready, L::kConsumerWarps / 2);   // one arrival per V_new warp
    tc::mbar_init(s_ready, L::kConsumerWarps);        // one arrival per consumer warp
    tc::mbar_init(rs_full, L::kConsumerWarps / 2);    // one arrival per o warp
    tc::mbar_init(rs_full + 1, L::kConsumerWarps / 2);
    tc::mbar_init(cons, L::kConsumerWarps);
    tc::mbar_init(cons + 1, L::kConsumerWarps);
    tc::fence_mbar_init();
  }
  for (int i = tid; i < 2 * 512; i += L::kThreads) {   // rows 0-63 of both [0; P] tiles stay zero
    const int st = i >> 9, off = (i & 511) * 16;
    *reinterpret_cast<uint4*>(sm + st * L::kStage + L::oPZ + off) = make_uint4(0u, 0u, 0u, 0u);
  }
  if (warp == 0) {
    tc::tmem_alloc(tslot, L::kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == L::kTmaWarp) {
    if (lane == 0) {
      tc::tma_prefetch_desc(&tmWQ);
      tc::tma_prefetch_desc(&tmP);
      tc::tma_prefetch_desc(&tmKT);
      tc::tma_prefetch_desc(&tmU);
      tc::tma_prefetch_desc(&tmGam);
      int issued = 0;
      for (int i = 0; i < nch; ++i) {
        const int st = i & 1;
        // a stage is refilled once the MMAs and every consumer warp are done with
        // its previous chunk: a consumer can then never see this barrier two phases
        // ahead of the chunk it waits for
        if (i >= 2 && !(tc::mbar_wait(empty + st, ((i >> 1) - 1) & 1, kWaitLimit) &&
                        tc::mbar_wait(cons + st, ((i >> 1) - 1) & 1, kWaitLimit))) {
          atomicExch(dev_err, (int32_t)kDevErrTimeout);
          break;
        }
        const int64_t rec = (int64_t)(j0 + i) * H + h;
        uint8_t* stg = sm + st * L::kStage;
        tc::mbar_arrive_expect_tx(full + st, L::kTxBytes);
        tc::tma_load_2d(stg + L::oWQ, &tmWQ, 0, (int32_t)(rec * 128), full + st);
        tc::tma_load_2d(stg + L::oWQ + 16384, &tmWQ, 64, (int32_t)(rec * 128), full + st);
        tc::tma_load_2d(stg + L::oPZ + 8192, &tmP, 0, (int32_t)(rec * C), full + st);
        tc::tma_load_2d(stg + L::oKT, &tmKT, 0, (int32_t)(rec * DK), full + st);
#pragma unroll
        for (int a = 0; a < NC / 64; ++a)
          tc::tma_load_2d(stg + L::oU + a * 8192, &tmU, n0 + 64 * a, (int32_t)(rec * C), full + st);
        tc::tma_load_2d(stg + L::oGam, &tmGam, 0, (int32_t)rec, full + st);
        ++issued;
      }
      for (int i = (issued > 2 ? issued - 2 : 0); i < issued; ++i) tc::mbar_wait(full + (i & 1), (i >> 1) & 1, kWaitLimit);
    }
  } else if (warp == L::kMmaWarp) {
    // the whole warp runs the issue loop (warp-uniform operands, one elected lane issues)
    const uint64_t dS0 = tc::desc_mnmajor_sw64_atoms(tc::smem_u32(sS), L::kSAtom);
    const uint64_t dV0 = tc::desc_mnmajor_sw64_atoms(tc::smem_u32(sVN), L::kVAtom);
    const uint64_t dA0 = tc::desc_kmajor_sw128(tc::smem_u32(sm));
    auto wait_all = [&](uint64_t* b, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, tc::mbar_wait(b, parity, kWaitLimit));
    };
    bool ok = true, issued = false;
    for (int i = 0; i < nch && ok; ++i) {
      const int st = i & 1;
      ok = wait_all(full + st, (i >> 1) & 1) && wait_all(s_ready, i & 1);
      if (!ok) break;
      tc::tc_fence_after();
      const uint64_t dA = dA0 + ((uint64_t)(st * L::kStage) >> 4);
      const uint32_t d12 = tmem + (uint32_t)(i % 3) * NC;
#pragma unroll
      for (int kk = 0; kk < DK / 16; ++kk)   // group 1
        tc::mma_16bit_w(d12, dA + (((kk >> 2) * 16384 + (kk & 3) * 32) >> 4), dS0 + ((kk * 1024) >> 4), kIdesc,
                        kk > 0);
      tc::mma_commit_w(mma1);
      issued = true;
      ok = wait_all(vn_ready, i & 1);
      if (!ok) break;
      tc::tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < C / 16; ++kk)   // group 2
        tc::mma_16bit_w(d12, dA + ((L::oPZ + kk * 32) >> 4), dV0 + ((kk * 1024) >> 4), kIdesc, 1u);
#pragma unroll
      for (int kk = 0; kk < C / 16; ++kk)
        tc::mma_16bit_w(tmem + kD3, dA + ((L::oKT + kk * 32) >> 4), dV0 + ((kk * 1024) >> 4), kIdesc, kk > 0);
      tc::mma_commit_w(mma2);
      tc::mma_commit_w(empty + st);
    }
    if (!ok && lane == 0) atomicExch(dev_err, (int32_t)kDevErrTimeout);
    if (issued) {
      tc::mma_commit_w(drain);
      wait_all(drain, 0);
    }
  } else {
    const int q = warp & 3, cg = warp >> 2;   // TMEM lane quarter, 32-column group
    const int c = 32 * q + lane;
    const uint32_t tl = (uint32_t)(32 * q);
    // o rows (tokens t0 + r, r = c - 64 < len) of local chunk j from D12 buffer
    // `buf`, with the optional output epilogue: each o warp publishes its 32
    // columns' sum of squares per row, the row's total over the NC/32 column
    // groups gives the RMS, then the weight and the Sigmoid gate scale the row
    // (the gate logits are loaded where used, at this kernel's register limit
    // holding them longer spilled and measured slower; they are prefetched into
    // L2 kGatePf chunks ahead and into L1 a chunk ahead).
    constexpr int kGatePf = 3;
    float nonfinite = 0.f;   // stays 0 unless an o or state value is inf or NaN (x * 0 is then NaN)
    auto prefetch_gate = [&](int j, bool l1) {
      const int64_t t0 = seq_start + (int64_t)j * C;
      const int r = c - 64;
      if (j < nch && r < seq_end - t0) {
        const bf16* gp = ep.gate + ((t0 + r) * H + h) * DV + n0 + 32 * cg;
        if (l1) asm volatile("prefetch.global.L1 [%0];" ::"l"(gp));
        else asm volatile("prefetch.global.L2 [%0];" ::"l"(gp));
      }
    };
    if constexpr (kGated) {
      if (q >= 2) {
        for (int j = 0; j < kGatePf; ++j) prefetch_gate(j, false);
        prefetch_gate(0, true);
      }
    }
    auto emit_o = [&](uint32_t buf, int64_t t0, int64_t len, int j) -> bool {
      const int r = c - 64;
      float sc = 1.f;
      if constexpr (kGated) {   // the next chunk's gate rows into L1, a later one's into L2
        prefetch_gate(j + 1, true);
        prefetch_gate(j + kGatePf, false);
      }
      if constexpr (kGated) {   // first pass over TMEM: this warp's share of the row's sum of squares
        float ss = 0.f;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          float ov[16];
          tc::tmem_ld16(tc::tmem_addr(tmem, tl, buf * NC + 32 * cg + 16 * hf), ov);
#pragma unroll
          for (int e = 0; e < 16; ++e) ss += ov[e] * ov[e];
        }
        float* rp = rss + (j & 1) * (NC / 32) * 64;
        rp[cg * 64 + r] = ss;
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(rs_full + (j & 1));
        if (!tc::mbar_wait(rs_full + (j & 1), (uint32_t)(j >> 1) & 1u, kWaitLimit)) return false;
        float tot = 0.f;
#pragma unroll
        for (int g2 = 0; g2 < NC / 32; ++g2) tot += rp[g2 * 64 + r];
        sc = rsqrtf(tot * (1.f / DV) + ep.eps);
      }
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float ov[16];
        tc::tmem_ld16(tc::tmem_addr(tmem, tl, buf * NC + 32 * cg + 16 * hf), ov);
        if (r < len) {
          const int col0 = n0 + 32 * cg + 16 * hf;
          if constexpr (kGated) {
            const uint4* gp = reinterpret_cast<const uint4*>(ep.gate + ((t0 + r) * H + h) * DV + col0);
#pragma unroll
            for (int v8 = 0; v8 < 2; ++v8) {
              const uint4 raw = gp[v8];
              const uint32_t gw[4] = {raw.x, raw.y, raw.z, raw.w};   // bf16 pairs, unpacked by shifts
              float4 w0 = make_float4(1.f, 1.f, 1.f, 1.f), w1 = w0;
              if (ep.weight) {
                w0 = *reinterpret_cast<const float4*>(ep.weight + (int64_t)h * DV + col0 + 8 * v8);
                w1 = *reinterpret_cast<const float4*>(ep.weight + (int64_t)h * DV + col0 + 8 * v8 + 4);
              }
              const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float x = (e & 1) ? __uint_as_float(gw[e >> 1] & 0xffff0000u) : __uint_as_float(gw[e >> 1] << 16);
                ov[8 * v8 + e] *= __fdividef(sc * wv[e], 1.f + __expf(-x));
              }
            }
          }
          store_bf16x16(o + ((t0 + r) * H + h) * DV + col0, ov);
#pragma unroll
          for (int e = 0; e < 16; ++e) nonfinite = fmaf(ov[e], 0.f, nonfinite);
        }
      }
      return true;
    };
    float S[32];
    {
      const int64_t off = (((int64_t)s * H + h) * DK + c) * DV + n0 + 32 * cg;
#pragma unroll
      for (int n = 0; n < 32; n += 4) {
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (s0) x = *reinterpret_cast<const float4*>(s0 + off + n);
        S[n] = x.x; S[n + 1] = x.y; S[n + 2] = x.z; S[n + 3] = x.w;
      }
    }
    store_mn_atom_row(sS + cg * L::kSAtom, c, S);
    tc::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(s_ready);
    bool bad = false;
    int i = 0;
    int64_t prev_t0 = 0;
    int64_t prev_len = 0;
    for (; i < nch; ++i) {
      const int st = i & 1;
      const uint8_t* stg = sm + st * L::kStage;
      bad |= !tc::mbar_wait(full + st, (i >> 1) & 1, kWaitLimit);
      if (__any_sync(0xffffffffu, bad)) {   // warp-uniform, so that no lane is left at a __syncwarp
        bad = true;
        break;
      }
      const float gam = reinterpret_cast<const float*>(stg + L::oGam)[c];
      if (q >= 2) {
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(cons + st);   // this warp reads nothing more of the stage
      }
      bad |= !tc::mbar_wait(mma1, i & 1, kWaitLimit);
      if (__any_sync(0xffffffffu, bad)) {   // warp-uniform, so that no lane is left at a __syncwarp
        bad = true;
        break;
      }
      tc::tc_fence_after();
      if (q < 2) {   // V_new rows (tokens) 0-63: u - w S, in two 16-column halves
        const uint8_t* uat = stg + L::oU + (cg >> 1) * 8192;   // the 64-column atom of this column group
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          float d[16];
          tc::tmem_ld16(tc::tmem_addr(tmem, tl, (uint32_t)(i % 3) * NC + 32 * cg + 16 * hf), d);
#pragma unroll
          for (int q4 = 0; q4 < 2; ++q4) {
            const uint4 raw =
                *reinterpret_cast<const uint4*>(uat + tc::sw128_offset(c, 32 * (cg & 1) + 16 * hf + 8 * q4));
            *reinterpret_cast<uint4*>(sVN + cg * L::kVAtom + tc::sw64_chunk_offset(c, 2 * hf + q4)) =
                tcu::vnew_f16x8(raw, d + 8 * q4);
          }
        }
        tc::fence_proxy_async_smem();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive(vn_ready);
          tc::mbar_arrive(cons + st);   // u and gam of the stage have been read
        }
      }
      bad |= !tc::mbar_wait(mma2, i & 1, kWaitLimit);
      if (__any_sync(0xffffffffu, bad)) {   // warp-uniform, so that no lane is left at a __syncwarp
        bad = true;
        break;
      }
      tc::tc_fence_after();
      {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          float d[16];
          tc::tmem_ld16(tc::tmem_addr(tmem, tl, kD3 + 32 * cg + 16 * hf), d);
#pragma unroll
          for (int n = 0; n < 16; ++n) S[16 * hf + n] = gam * S[16 * hf + n] + d[n];
        }
        store_mn_atom_row(sS + cg * L::kSAtom, c, S);
        tc::fence_proxy_async_smem();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(s_ready);
      }
      if (const int64_t slot = snapshot_slot(map, s, i, seq_end - seq_start); slot >= 0) {
        float* dst = map.snaps + ((slot * H + h) * DK + c) * DV + n0 + 32 * cg;
#pragma unroll
        for (int n = 0; n < 32; n += 4) *reinterpret_cast<float4*>(dst + n) = make_float4(S[n], S[n + 1], S[n + 2], S[n + 3]);
      }
      // The previous chunk's o rows are emitted after the state hand-off (off the
      // chain's critical path): their buffer, (i - 1) % 3, is next written by the
      // first group of chunk i + 2, issued only after this warp's next hand-off.
      // Meanwhile the MMAs and the TMA producer may run a chunk ahead; the stage
      // release barrier (cons) keeps the producer from refilling the stage this
      // warp reads next before the warp has waited for it.
      if (i > 0 && q >= 2) {
        bad |= !emit_o((uint32_t)((i - 1) % 3), prev_t0, prev_len, i - 1);
        if (__any_sync(0xffffffffu, bad)) {
          bad = true;
          break;
        }
      }
      prev_t0 = seq_start + (int64_t)i * C;
      prev_len = min((int64_t)C, seq_end - prev_t0);
    }
    if (i == nch && !bad && nch > 0 && q >= 2) {   // the last chunk's o
      bad = __any_sync(0xffffffffu, !emit_o((uint32_t)((nch - 1) % 3), prev_t0, prev_len, nch - 1));
    }
    if (i < nch || bad) {
      atomicExch(dev_err, (int32_t)kDevErrTimeout);
    } else {
#pragma unroll
      for (int n = 0; n < 32; ++n) nonfinite = fmaf(S[n], 0.f, nonfinite);
      report_nonfinite(nonfinite, dev_err);
    }
    if (i == nch && !bad && s_final) {
      float* dst = s_final + (((int64_t)s * H + h) * DK + c) * DV + n0 + 32 * cg;
#pragma unroll
      for (int n = 0; n < 32; n += 4) *reinterpret_cast<float4*>(dst + n) = make_float4(S[n], S[n + 1], S[n + 2], S[n + 3]);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, L::kTmemCols);
}

// ------------------------------------------------------------- fused kernel
// Prep and the value-major chain in one persistent launch (cooperative, one
// CTA per SM, so that every CTA is resident at once): CTAs 0 .. n_chain-1 run
// the chains of the (sequence, head) pairs, each loading a chunk's record only
// once it has been published; the other CTAs run the prep tasks in chunk-major
// order and publish each record when its stores have completed.  The chains
// then trail prep by a few chunks (their records still in L2) instead of
// waiting for the whole prep pass, and prep never waits for a chain, so every
// wait ends.
__global__ void __launch_bounds__(kPrepTcThreads, 1)
    chunk_fused_tc(const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmQ, const bf16* __restrict__ v,
                   const __grid_constant__ CUtensorMap tmWs, const __grid_constant__ CUtensorMap tmUs,
                   const __grid_constant__ CUtensorMap tmPs, const __grid_constant__ CUtensorMap tmWQ,
                   const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmKT,
                   const __grid_constant__ CUtensorMap tmU, const __grid_constant__ CUtensorMap tmGam,
                   const __grid_constant__ CUtensorMap tmO, const float* __restrict__ beta,
                   const int32_t* __restrict__ cu, int32_t num_seqs, int64_t T_seq, int32_t H, ChunkMap map,
                   TcRecords out, int64_t n_tasks, const float* __restrict__ s0, float* __restrict__ s_final,
                   bf16* __restrict__ o, int32_t* __restrict__ dev_err, int32_t* __restrict__ ready, int32_t n_chain) {
  static_assert(vm::VmWarps<8>::kThreads <= kPrepTcThreads && ps::kThreads == kPrepTcThreads,
                "the chain role fits the prep CTA");
  if ((int)blockIdx.x < n_chain)
    vm::chain_body<8>(tmWQ, tmP, tmKT, tmU, tmGam, tmO, cu, num_seqs, T_seq, H, map, s0, s_final, o, dev_err,
                      (int)blockIdx.x, ready, &out);
  else
    ps::prep_split_body<128>(tmG, tmK, tmQ, tmWs, tmUs, tmPs, v, beta, num_seqs, H, map, out, n_tasks, dev_err,
                             (int)blockIdx.x - n_chain, (int)gridDim.x - n_chain, ready);
}
constexpr size_t kFusedSmem =
    ps::Smem<128>::kAlloc > vm::VmSmem::kAlloc ? ps::Smem<128>::kAlloc : vm::VmSmem::kAlloc;

// --------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2D tensor map over a row-major [rows][inner] array.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, size_t esize, void* base, uint64_t inner, uint64_t rows,
              uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * esize};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3D tensor map over a token-major [tokens][H][inner] bf16 array, one box =
// 64 tokens of one head and box_inner of its inner elements: the inputs (whole
// rows, no swizzle) and the output o (64-value boxes, 128-byte swizzle).
bool make_input_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t H, uint64_t tokens,
                    uint32_t box_inner = 0, CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_NONE) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {inner, H, tokens};
  const cuuint64_t strides[2] = {inner * 2, H * inner * 2};
  const cuuint32_t box[3] = {box_inner ? box_inner : (cuuint32_t)inner, 1, (cuuint32_t)C};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The 32-column chain: with the output epilogue (kGated) the DV/32 CTAs of a head
// (consecutive blocks) form one thread-block cluster.
template <int DV, bool kGated>
cudaError_t launch_chain_narrow(const CUtensorMap& mWQ, const CUtensorMap& mP, const CUtensorMap& mKT,
                                const CUtensorMap& mU, const CUtensorMap& mGam, const ChunkProblem& p,
                                const ChunkMap& map, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(chunk_chain_tc<DV, kGated>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)ChainTcSmem::kAlloc);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.num_seqs * p.H * (DV / BV), 1, 1);
  cfg.blockDim = dim3(chain_threads(kGated), 1, 1);
  cfg.dynamicSmemBytes = ChainTcSmem::kAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (kGated) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = DV / BV;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  const OutEpilogue ep = kGated ? OutEpilogue{static_cast<const bf16*>(p.out_gate), p.norm_weight, p.eps_rms}
                                : OutEpilogue{nullptr, nullptr, 0.f};
  prof_begin(stream, kGated ? "chunk_chain_tc_gated" : "chunk_chain_tc");
  e = cudaLaunchKernelEx(&cfg, chunk_chain_tc<DV, kGated>, mWQ, mP, mKT, mU, mGam, p.cu, p.num_seqs, p.T_seq, p.H,
                         map, p.s0, p.s_final, static_cast<bf16*>(p.o), ep, p.dev_err);
  prof_end(stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int DV, int NC, bool kGated>
cudaError_t launch_chain_wide_nc(const CUtensorMap& mWQ, const CUtensorMap& mP, const CUtensorMap& mKT,
                                 const CUtensorMap& mU, const CUtensorMap& mGam, const ChunkProblem& p,
                                 const ChunkMap& map, cudaStream_t stream) {
  using W = ChainWideSmem<NC>;
  cudaError_t e =
      cudaFuncSetAttribute(chunk_chain_wide_tc<DV, NC, kGated>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)W::kAlloc);
  if (e != cudaSuccess) return e;
  prof_begin(stream, "chunk_chain_wide_tc");
  const OutEpilogue ep = kGated ? OutEpilogue{static_cast<const bf16*>(p.out_gate), p.norm_weight, p.eps_rms}
                                : OutEpilogue{nullptr, nullptr, 0.f};
  chunk_chain_wide_tc<DV, NC, kGated><<<(unsigned)p.num_seqs * p.H * (DV / NC), W::kThreads, W::kAlloc, stream>>>(
      mWQ, mP, mKT, mU, mGam, p.cu, p.num_seqs, p.T_seq, p.H, map, p.s0, p.s_final, static_cast<bf16*>(p.o), ep,
      p.dev_err);
  prof_end(stream);
  return cudaGetLastError();
}

template <int DV>
cudaError_t launch_chain_wide(bool fuse_epilogue, const CUtensorMap& mWQ, const CUtensorMap& mP,
                              const CUtensorMap& mKT, const CUtensorMap& mU, const CUtensorMap& mGam,
                              const ChunkProblem& p, const ChunkMap& map, cudaStream_t stream) {
  // (all 128 value columns without the epilogue run in the value-major chain)
  constexpr int kFull = DV == 128 ? 128 : 64;
  if (fuse_epilogue) return launch_chain_wide_nc<DV, kFull, true>(mWQ, mP, mKT, mU, mGam, p, map, stream);
  return launch_chain_wide_nc<DV, 64, false>(mWQ, mP, mKT, mU, mGam, p, map, stream);
}

template <int DV>
cudaError_t launch_tc(const ChunkProblem& p, const Workspace& ws, const ChunkMap& map, char* base,
                      cudaStream_t stream) {
  TcRecords rec;
  rec.wq = reinterpret_cast<f16*>(base + ws.off_wq);
  rec.p = reinterpret_cast<f16*>(base + ws.off_p);
  rec.kt = reinterpret_cast<f16*>(base + ws.off_kt);
  rec.u = reinterpret_cast<f16*>(base + ws.off_u);
  rec.gam = reinterpret_cast<float*>(base + ws.off_gam);
  const uint64_t R = (uint64_t)ws.max_chunks * (uint64_t)p.H;
  const uint64_t Rr = R > 0 ? R : 1;
  cudaError_t e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  // The records as the chains read them: [w; q e^G] boxes of 64 x 128, P of 64 x 64,
  // (k e^{G_last - G})^T of 64 x 128, u of u_cols x 64, e^{G_last} of 128 x 1.
  CUtensorMap mWQ, mP, mKT, mU, mGam;
  auto chain_maps = [&](uint32_t u_cols) -> bool {
    return make_map(&mWQ, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, rec.wq, DK, Rr * 128, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_map(&mP, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, rec.p, C, Rr * C, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_map(&mKT, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, rec.kt, C, Rr * DK, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_map(&mU, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, rec.u, DV, Rr * C, u_cols, 64,
                    u_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B) &&
           make_map(&mGam, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, rec.gam, DK, Rr, DK, 1, CU_TENSOR_MAP_SWIZZLE_NONE);
  };
  // Prep and the value-major chain fused (chunk_fused_tc) when the (sequence, head)
  // chains are few enough to leave most SMs to prep: d_v = 128, the plain call,
  // the bounded map.  KDA_FUSED=0, or a forced chain width, runs the two passes.
  const int64_t n_chain = (int64_t)p.num_seqs * p.H;
  bool fused = DV == 128 && !p.out_gate && p.decay_map == KDA_DECAY_BOUNDED && !p.diag_pairs && ws.max_chunks > 0 &&
               p.total_tokens > 0 && n_chain <= sms / 4 && !std::getenv("KDA_CHAIN_COLUMNS");
  if (const char* env = std::getenv("KDA_FUSED")) fused = fused && std::atoi(env) != 0;
  // The bounded map's prep runs two task streams per CTA over 64-channel halves
  // of g, k, q (chunk_prep_split_tc); the pair-path variants, or KDA_PREP_STREAMS=1,
  // run the single-stream kernel over whole rows.
  bool split = p.decay_map == KDA_DECAY_BOUNDED && !p.diag_pairs;
  if (const char* env = std::getenv("KDA_PREP_STREAMS")) split = split && std::atoi(env) != 1;
  fused = fused && split;
  if (ws.max_chunks > 0 && p.total_tokens > 0) {
    CUtensorMap mG, mK, mQ, mV;
    const uint64_t tok = (uint64_t)p.total_tokens;
    const uint32_t box = split ? (uint32_t)ps::KH : 0u;
    if (!make_input_map(&mG, p.g, DK, p.H, tok, box) || !make_input_map(&mK, p.k, DK, p.H, tok, box) ||
        !make_input_map(&mQ, p.q, DK, p.H, tok, box) || !make_input_map(&mV, p.v, DV, p.H, tok))
      return cudaErrorInvalidValue;
    CUtensorMap mWs, mUs, mPs;   // record stores of [w | u] and P: 64 x 64 boxes, 128-byte swizzle
    if (!make_map(&mWs, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, rec.wq, DK, R * 128, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mUs, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, rec.u, DV, R * C, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mPs, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, rec.p, C, R * C, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    const int64_t n_tasks = (int64_t)ws.max_chunks * p.H;
    if constexpr (DV == 128) {
      if (fused) {
        CUtensorMap mO;   // o rows by TMA store: 64 tokens x 64 values per box
        if (!chain_maps(64) || !make_input_map(&mO, p.o, DV, p.H, tok, 64, CU_TENSOR_MAP_SWIZZLE_128B))
          return cudaErrorInvalidValue;
        int32_t* flags = reinterpret_cast<int32_t*>(base + ws.off_flags);
        if ((e = cudaMemsetAsync(flags, 0, R * sizeof(int32_t), stream)) != cudaSuccess) return e;
        if ((e = cudaFuncSetAttribute(chunk_fused_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFusedSmem)) !=
            cudaSuccess)
          return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)sms, 1, 1);   // one CTA per SM, all resident (cooperative)
        cfg.blockDim = dim3(kPrepTcThreads, 1, 1);
        cfg.dynamicSmemBytes = kFusedSmem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        prof_begin(stream, "chunk_fused_tc");
        e = cudaLaunchKernelEx(&cfg, chunk_fused_tc, mG, mK, mQ, static_cast<const bf16*>(p.v), mWs, mUs, mPs, mWQ,
                               mP, mKT, mU, mGam, mO, p.beta,
                               p.cu, p.num_seqs, p.T_seq, p.H, map, rec, n_tasks, p.s0, p.s_final,
                               static_cast<bf16*>(p.o), p.dev_err, flags, (int32_t)n_chain);
        prof_end(stream);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
      }
    }
    const int grid = (int)std::min<int64_t>(n_tasks, sms);
    auto prep = [&](auto variant_tag, const char* name) -> cudaError_t {
      constexpr int kV = decltype(variant_tag)::value;
      const size_t smem = PrepTcSmem<DV, kV>::kAlloc;
      cudaError_t err = cudaFuncSetAttribute(chunk_prep_tc<DV, kV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (err != cudaSuccess) return err;
      prof_begin(stream, name);
      chunk_prep_tc<DV, kV><<<grid, kPrepTcThreads, smem, stream>>>(mG, mK, mQ, mV, mWs, mUs, mPs, p.beta, p.num_seqs,
                                                                    p.H, map, rec, n_tasks, p.dev_err);
      prof_end(stream);
      return cudaGetLastError();
    };
    if (split) {
      const size_t smem = ps::Smem<DV>::kAlloc;
      if ((e = cudaFuncSetAttribute(chunk_prep_split_tc<DV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem)) != cudaSuccess)
        return e;
      // two task streams per CTA: as many CTAs as SMs, or half the tasks (rounded up)
      const int grid2 = (int)std::min<int64_t>((n_tasks + 1) / 2, sms);
      prof_begin(stream, "chunk_prep_tc");
      chunk_prep_split_tc<DV><<<grid2, ps::kThreads, smem, stream>>>(mG, mK, mQ, mWs, mUs, mPs,
                                                                     static_cast<const bf16*>(p.v), p.beta, p.num_seqs,
                                                                     p.H, map, rec, n_tasks, p.dev_err);
      prof_end(stream);
      e = cudaGetLastError();
    } else if (p.decay_map == KDA_DECAY_SOFTPLUS)
      e = prep(std::integral_constant<int, kPrepSoftplusPairs>{}, "chunk_prep_tc_softplus_pairs");
    else if (p.diag_pairs)
      e = prep(std::integral_constant<int, kPrepBoundedPairs>{}, "chunk_prep_tc_pairs");
    else
      e = prep(std::integral_constant<int, kPrepBounded>{}, "chunk_prep_tc_single");
    if (e != cudaSuccess) return e;
  }
  // Chain variant: 32 value columns per CTA (the most CTAs, for few long
  // chains) unless that grid exceeds one wave of the GPU; then one CTA per
  // (sequence, head) with all DV columns, which reads the per-chunk tiles and
  // issues the MMAs once per head: the value-major chain for d_v = 128 without
  // the output epilogue, the wide chain otherwise.  KDA_CHAIN_COLUMNS=32, 64 or
  // DV forces a width.
  int ncol = (int64_t)p.num_seqs * p.H * (DV / BV) > sms ? DV : BV;
  if (const char* env = std::getenv("KDA_CHAIN_COLUMNS")) {
    const int cols = std::atoi(env);
    if (cols == BV || cols == 64 || cols == DV) ncol = cols;
  }
  // The output epilogue needs a token's d_v outputs: fused into the chain, either
  // the 32-column chain (the CTAs of a head exchange row sums within their
  // cluster) or the wide chain holding all d_v columns (the 64-column width is
  // not used with it).
  if (p.out_gate && ncol != BV) ncol = DV;
  const bool fuse = p.out_gate && ncol == DV;
  const bool wide = ncol != BV;
  if (!chain_maps(wide ? 64 : BV)) return cudaErrorInvalidValue;
  if (DV == 128 && ncol == DV && !p.out_gate) {
    CUtensorMap mO = {};   // o rows by TMA store: 64 tokens x 64 values per box (unused without tokens)
    if (p.total_tokens > 0 &&
        !make_input_map(&mO, p.o, DV, p.H, (uint64_t)p.total_tokens, 64, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    return launch_chain_vm(mWQ, mP, mKT, mU, mGam, mO, p, map, stream);
  }
  if (wide) return launch_chain_wide<DV>(fuse, mWQ, mP, mKT, mU, mGam, p, map, stream);
  return p.out_gate ? launch_chain_narrow<DV, true>(mWQ, mP, mKT, mU, mGam, p, map, stream)
                    : launch_chain_narrow<DV, false>(mWQ, mP, mKT, mU, mGam, p, map, stream);
}

}  // namespace

bool tc_path_supported(int32_t d_k, int32_t d_v, kda_dtype dt) {
  return dt == KDA_BF16 && d_k == DK && (d_v == 64 || d_v == 128);
}

size_t tc_record_bytes(int32_t d_k, int32_t d_v) {
  return (size_t)128 * d_k * 2 + (size_t)C * C * 2 + (size_t)d_k * C * 2 + (size_t)C * d_v * 2 + (size_t)d_k * 4;
}

cudaError_t launch_chunk_tc(const ChunkProblem& p, const Workspace& ws, const ChunkMap& map, char* base,
                            cudaStream_t stream) {
  if (p.d_v == 128) return launch_tc<128>(p, ws, map, base, stream);
  return launch_tc<64>(p, ws, map, base, stream);
}

}  // namespace kda
