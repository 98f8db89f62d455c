// Prep of the tensor-core prefill (bf16, d_k = 128, bounded decay map) with two
// independent task streams per CTA.
//
// What a task computes is the chunk form of page "Kimi K3：架构、训练与百万 Token
// Agentic RL 技术解读" §3.3 for one (64-token chunk, head): the gate
// -5 Sigmoid(g) and its cumulative sum G, the beta-weighted decayed k k^T
// matrix A and the read-out matrix P (diagonal 16-token sub-tiles referenced
// to the sub-tile start, whose column factors stay below e^80 only because of
// the lower bound), X = (I + A)^{-1}, and w, u = X [beta k e^G | beta V].  It
// writes the same fp16 records as the single-stream prep kernel: [w; q e^G],
// P, (k e^{G_last - G})^T, u and fp32 e^{G_last}.
//
// Layout of the work.  The 512 threads of a CTA form two groups of 8 warps.
// Each group runs its own stream of tasks (its own shared-memory half, its own
// 256 TMEM columns, its own mbarriers and named barrier), so that while one
// group is in the serial part of a task (the A / P epilogue, the inverse on 4
// warps, the [w | u] issue) the other one keeps the SM's issue slots busy with
// the elementwise phases of its own task.  Within a group a task runs as two
// passes over 64 key channels each (the half of every operand that fits the
// group's 111 KB): gate and cumulative sum, offsets, the bf16 operand tiles,
// the A / P products over those channels (K = 64 of 128) and the records of
// those channels; the second pass waits for the first pass's products before
// rewriting the operand tiles.  Then the epilogue, the inverse and [w | u].
//
// TMEM of a group (256 columns, 128 lanes):
//   0-159    D1 = [k e^{G-G_s} ; (q e^{G-G_s})_hi] x [own sub-tile hi ; later sub-tiles]^T
//   160-223  Dc = [k ; q_hi] x (own lo)^T + [q_hi ; q_lo] x (own hi)^T: in lanes 64-127
//            the two correction products of P's diagonal sub-tiles (lanes 0-63 unused)
//   0-127    after the epilogue: w (lanes 0-63, from A = [X ; 0]) and u (lanes 64-127,
//            columns 0..d_v-1, from A = [0 ; X] accumulated onto the zeros the w product
//            left there), drained by all 8 warps at the start of the next task.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "chain_common.cuh"
#include "kda_internal.cuh"
#include "tc_ptx.cuh"

namespace kda {
namespace ps {

using bf16 = __nv_bfloat16;
using f16 = __half;
constexpr int C = kChunk;               // 64 tokens per chunk
constexpr int DK = 128;                 // key channels
constexpr int KH = 64;                  // key channels per pass
constexpr int kGroupThreads = 256;      // one task stream
constexpr int kThreads = 2 * kGroupThreads;
constexpr uint32_t kGroupCols = 256;    // TMEM columns of a group
constexpr int LDX = C + 8;              // fp16 row stride of A's blocks below the diagonal
constexpr int LDA = kSub + 1;           // fp32 row stride of A's diagonal blocks
constexpr int kLater = 64;              // column-operand row (D1 column) of the later sub-tiles' rows
constexpr int kLo = 160;                // column-operand row of the own sub-tile's low part; Dc's column

// ------------------------------------------------------------ small helpers
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// log2 of the bounded decay, -5 Sigmoid(x) / ln 2 (G is kept in base-2 units, so
// that every factor 2^{G_a - G_b} is one ex2.approx); a huge -x gives exp = inf
// and a reciprocal of 0, i.e. no decay.
__device__ __forceinline__ float log2_decay_bounded(float x) {
  return __fdividef(-5.f * 1.4426950408889634f, 1.f + __expf(-x));
}
// A thread's elementwise work is on channel pairs: fp32 pairs in one register pair,
// multiplied and added by the packed fp32x2 instructions of sm_100 (one
// instruction per pair, each half rounded as the scalar operation would be).
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 splat2(float x) { return make_float2(x, x); }
__device__ __forceinline__ float2 ex2_pair(float2 x) { return make_float2(ex2_approx(x.x), ex2_approx(x.y)); }
__device__ __forceinline__ float2 bf2_to_f2(__nv_bfloat162 x) { return __bfloat1622float2(x); }
__device__ __forceinline__ uint32_t pack_bf16_pair(float2 x) {
  const __nv_bfloat162 v = __float22bfloat162_rn(x);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_f16_pair(float2 x) {
  const __half2 v = __float22half2_rn(x);
  return *reinterpret_cast<const uint32_t*>(&v);
}
// log2 of the bounded decay of a channel pair, -5 Sigmoid(x) / ln 2: e^{-x} as
// 2^{-x log2 e}, then -5 / ln 2 times the approximate reciprocal of 1 + e^{-x}
// (a huge -x gives inf and a reciprocal of 0: no decay).
__device__ __forceinline__ float2 log2_decay_bounded2(float2 x) {
  const float2 den = add2(ex2_pair(mul2(x, splat2(-1.4426950408889634f))), splat2(1.f));
  return mul2(make_float2(rcp_approx(den.x), rcp_approx(den.y)), splat2(-5.f * 1.4426950408889634f));
}
// bf16 (hi, lo) split of a pair: hi = x rounded to bf16, lo = x - hi (exact in
// fp32) rounded to bf16; both as bf16x2 words.
__device__ __forceinline__ void split_bf16_pair(float2 x, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __float22bfloat162_rn(x);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = pack_bf16_pair(fma2(__bfloat1622float2(h), splat2(-1.f), x));
}
// bf16 pair (hi, lo) of each of two floats, packed as bf16x2 words.
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - __low2float(h), x1 - __high2float(h));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}
// Global loads issued where they stand (not sunk to the first use).
__device__ __forceinline__ float ld_early_f32(const float* p) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ int4 ld_early_v4(const int4* p) {
  int4 v;
  asm volatile("ld.global.nc.v4.s32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 ld_early_v4_hint(const void* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}
// m16n8k16 helpers of the inverse's blocks below the diagonal.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void mma16816_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Byte offset of element (row, col) of a [rows][64] 16-bit tile, K-major, 128-byte swizzle.
__device__ __forceinline__ uint32_t xs_off(int row, int col) { return tc::sw128_offset(row, col); }
// Byte offset of element (k, n) of the [beta k e^G | beta V] operand: MN-major (n
// contiguous), 128-byte swizzle, 64-column atoms [64 k][128 B].
__device__ __forceinline__ uint32_t kv_off(int k, int n) {
  return (uint32_t)(n >> 6) * 8192u + (uint32_t)k * 128u + (((((uint32_t)n & 63u) >> 3) ^ ((uint32_t)k & 7u)) << 4) +
         ((uint32_t)n & 7u) * 2u;
}
// Column-operand row of column i of later sub-tile a' = 1..3, minus kLater.
__device__ __forceinline__ int later_row0(int a2) { return a2 == 1 ? 0 : (a2 == 2 ? 16 : 48); }

// Record publication for the fused kernel (see prep_split_body): one release
// fence, then a store of 1 into the flag of each record first, first + step, .., last.
// The single-stream prep publishes four records per fence; the two-stream prep,
// whose control thread is off the inverse's path, publishes each record.
constexpr int kPublishBatch = 4;
constexpr int kSplitPublishBatch = 1;
__device__ __forceinline__ void publish_records(int32_t* ready, int64_t first, int64_t last, int64_t step) {
  asm volatile("fence.proxy.async.global;" ::: "memory");
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
  for (int64_t r = first; r <= last; r += step)
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(ready + r), "r"(1u) : "memory");
}

// Shared memory of one group (the CTA holds two, kStride apart, then the TMEM
// address slot).
template <int DV>
struct Smem {
  static constexpr int kRowRows = 192, kColRows = 224;
  static constexpr int kWuN = DK + DV;
  // Operands of the A / P products for one pass (64 channels, one 128-byte
  // swizzle atom), bf16, K-major:
  //   row operand:    0-63 k e^{G - G_s}, 64-127 q e^{G - G_s} (high part), 128-191 its low part
  //   column operand: 0-63 k e^{G_s - G} of the own sub-tile (high part),
  //                   64 + later_row0(a') + i  k_i e^{G_s(a') - G_i} for the later sub-tiles
  //                   a' = 1..3 (columns i < 16 a', high part only), 160-223 own sub-tile low part
  static constexpr size_t oRow = 0;
  static constexpr size_t oCol = oRow + (size_t)kRowRows * 128;
  // [beta k e^G | beta V], fp16, the B operand of [w | u] (MN-major, 64-column atoms)
  static constexpr size_t oKV = oCol + (size_t)kColRows * 128;
  // raw g, k, q of one pass (TMA, bf16 [64 tokens][64 channels] each), staged a pass ahead
  static constexpr size_t oRaw = oKV + (size_t)(kWuN / 64) * 8192;
  static constexpr size_t oTot = oRaw + (size_t)3 * C * KH * 2;   // fp32 [8][64] row-group sums
  static constexpr size_t oBeta = oTot + (size_t)8 * KH * 4;       // fp32 [64]
  static constexpr size_t oBar = oBeta + (size_t)C * 4;            // mbarriers: raw rows, [w | u], A / P
  static constexpr size_t kBytes = oBar + 3 * 8;
  static constexpr size_t kStride = (kBytes + 1023) / 1024 * 1024;
  static constexpr size_t kAlloc = 2 * kStride + 16 + 1024;       // + TMEM slot, + slack to align to 1 KB
  // Reused from the A / P epilogue to the [w | u] issue (the operand area is free once
  // the products are done):
  static constexpr size_t oA = 0;          // fp32 [64][LDA]: A's diagonal blocks (columns within the block)
  static constexpr size_t oZ0 = 5120;      // 8 KB of zeros: [0 ; X] starts here
  static constexpr size_t oXb = 13312;     // X, fp16 [64][64], 128-byte swizzle: [X ; 0] starts here
  static constexpr size_t oZ1 = 21504;     // 8 KB of zeros
  static constexpr size_t oAh = 29696;     // fp16 [64][LDX]: A, blocks below the diagonal
  static constexpr size_t oYh = oAh + (size_t)C * LDX * 2;   // fp16 [7][16][24] scratch blocks of the inverse
  static constexpr size_t oPst = 45056;    // fp16 [64][64] P, 128-byte swizzle (TMA store)
  static_assert(oA + (size_t)C * LDA * 4 <= oZ0 && oZ0 + 8192 == oXb && oXb + 8192 == oZ1 && oZ1 + 8192 <= oAh,
                "X between its zero blocks");
  static_assert(oYh + 7 * 16 * 24 * 2 <= oPst && oPst + (size_t)C * C * 2 <= oKV, "aliases fit the operand area");
  static_assert((oCol % 1024) == 0 && (oKV % 1024) == 0 && (oZ0 % 1024) == 0 && (oXb % 1024) == 0 &&
                    (oPst % 1024) == 0 && (oRaw % 1024) == 0 && (oBar % 8) == 0,
                "TMA, tcgen05 operand and mbarrier alignment");
  static_assert(kAlloc <= 232448, "two groups fit the 227 KB shared-memory limit");
};

// One CTA's share of the tasks (chunk j, head h), record index j * H + h, in
// chunk-major order: group g of CTA `cta` takes tasks (2 cta + g) + i * 2 ncta.
// With `ready` (the fused kernel) the records are published, kSplitPublishBatch
// at a time, once every store of theirs has completed: the [w | u] record of a
// task is stored at the start of the next one, so a record joins the batch in
// the next task's epilogue, right after that task's P store, and is published
// once the group's control thread has waited for all but that most recent bulk
// group.
template <int DV>
__device__ __forceinline__ void prep_split_body(const CUtensorMap& tmG, const CUtensorMap& tmK, const CUtensorMap& tmQ,
                                                const CUtensorMap& tmWs, const CUtensorMap& tmUs, const CUtensorMap& tmPs,
                                                const bf16* __restrict__ v, const float* __restrict__ beta,
                                                int32_t num_seqs, int32_t H, const ChunkMap& map, const TcRecords& out,
                                                int64_t n_tasks, int32_t* __restrict__ dev_err, int cta, int ncta,
                                                int32_t* __restrict__ ready) {
  using L = Smem<DV>;
  constexpr int NG = kGroupThreads;
  constexpr int kPerV = DV / 64;   // 16-byte chunks of v per thread and pass
  constexpr uint32_t kIdD1 = tc::idesc_bf16_f32(128, 160), kIdDc = tc::idesc_bf16_f32(128, 64);
  constexpr uint32_t kIdW = tc::idesc_f16_f32(128, DK) | (1u << 16);   // B (KV) MN-major
  constexpr uint32_t kIdU = tc::idesc_f16_f32(128, DV) | (1u << 16);
  constexpr int kWuIssuer = 2;   // warp of the group that issues [w | u]
  using tcu::kWaitLimit;
  using tcu::pack_bf16x2;
  using tcu::pack_f16x2;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, grp = tid >> 8, gt = tid & (NG - 1), gw = gt >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const uint32_t bar_id = 1u + (uint32_t)grp;   // the group's named barrier
  // The group's control thread (lane 0 of its warp 4, which only writes zeros
  // during the inverse): raw-row loads, the A / P products, the record stores,
  // their bulk-group waits and the publication.
  const bool ctl = gt == 128;
  uint8_t* smem = base + (size_t)grp * L::kStride;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + 2 * L::kStride);
  uint8_t* sRow = smem + L::oRow;
  uint8_t* sCol = smem + L::oCol;
  uint8_t* sKV = smem + L::oKV;
  uint8_t* sPst = smem + L::oPst;
  uint8_t* sX = smem + L::oXb;
  float* sTot = reinterpret_cast<float*>(smem + L::oTot);
  float* sBeta = reinterpret_cast<float*>(smem + L::oBeta);
  float* sA = reinterpret_cast<float*>(smem + L::oA);
  f16* sAh = reinterpret_cast<f16*>(smem + L::oAh);
  f16* sYh = reinterpret_cast<f16*>(smem + L::oYh);
  const bf16* rawG = reinterpret_cast<const bf16*>(smem + L::oRaw);
  const bf16* rawK = rawG + C * KH;
  const bf16* rawQ = rawK + C * KH;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::oBar);   // 0 raw rows, 1 [w | u], 2 A / P

  auto gsync = [&]() { asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(NG) : "memory"); };

  if (gt == 0) {
    tc::mbar_init(bar, 1);
    tc::mbar_init(bar + 1, 1);
    tc::mbar_init(bar + 2, 1);
    tc::fence_mbar_init();
  }
  if (tid == 0) {
    tc::tma_prefetch_desc(&tmG);
    tc::tma_prefetch_desc(&tmK);
    tc::tma_prefetch_desc(&tmQ);
  }
  if (tid < 32) {
    tc::tmem_alloc(tmem_slot, 2 * kGroupCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tm = *tmem_slot + (uint32_t)grp * kGroupCols;

  // In the fused kernel (with `ready`) the records are read back within a few
  // chunks from L2: stored with evict-last priority, the inputs (read once)
  // loaded with evict-first; alone, prep keeps the default priority.
  const uint64_t pol_in = ready ? tc::l2_policy_evict_first() : tc::l2_policy_evict_normal();
  const uint64_t pol_rec = ready ? tc::l2_policy_evict_last() : tc::l2_policy_evict_normal();
  const int vc = 2 * cta + grp, nv = 2 * ncta;   // this group's first task and the task stride
  bool wu_pending = false, bulk_pending = false;   // bulk_pending: the control thread has record stores in flight
  // control thread, with `ready`: the record whose [w | u] stores were issued this task,
  // and the batch of records waiting for publication
  int64_t pub_rec = -1, batch_first = -1, batch_last = -1, wu_rec = 0;
  int batch_n = 0;
  uint32_t raw_par = 0, wu_par = 0, ap_par = 0;

  // [w | u] of the previous task out of TMEM into 64-column fp16 tiles (128-byte
  // swizzle) in the area of its B operand: warp (q, half) takes TMEM lanes
  // 32q..32q+31 (w rows for q < 2, u rows for q >= 2) and columns 64 half..+63.
  // Returns false if the product did not complete in time.
  auto wu_drain_tiles = [&]() -> bool {
    if (!wu_pending) return true;
    const bool okw = tc::mbar_wait(bar + 1, wu_par, kWaitLimit);
    wu_par ^= 1u;
    wu_pending = false;
    tc::tc_fence_after();
    const int q = gw & 3, half = gw >> 2;
    if (q < 2 || 64 * half < DV) {
      const int r = 32 * (q & 1) + lane;
      uint8_t* tile = sKV + (size_t)((q < 2 ? 0 : DK / 64) + half) * 8192;
#pragma unroll
      for (int qt = 0; qt < 4; ++qt) {
        float x[16];
        tc::tmem_ld16(tc::tmem_addr(tm, (uint32_t)(32 * q), (uint32_t)(64 * half + 16 * qt)), x);
#pragma unroll
        for (int j = 0; j < 2; ++j)
          *reinterpret_cast<uint4*>(tile + xs_off(r, 16 * qt + 8 * j)) =
              make_uint4(pack_f16x2(x[8 * j + 0], x[8 * j + 1]), pack_f16x2(x[8 * j + 2], x[8 * j + 3]),
                         pack_f16x2(x[8 * j + 4], x[8 * j + 5]), pack_f16x2(x[8 * j + 6], x[8 * j + 7]));
      }
    }
    return okw;
  };
  // After the group barrier that follows wu_drain_tiles: the control thread stores the tiles
  // to the record (and does the publication bookkeeping of the fused kernel).
  auto wu_store = [&](bool drained, bool okw) {
    if (!ctl || !drained) return;
    if (ready) pub_rec = wu_rec;   // complete once its [w | u] stores, issued below, are
    if (okw) {
#pragma unroll
      for (int t = 0; t < L::kWuN / 64; ++t) {
        if (t < DK / 64)
          tc::tma_store_2d_hint(&tmWs, 64 * t, (int32_t)(wu_rec * 128), sKV + t * 8192, pol_rec);
        else
          tc::tma_store_2d_hint(&tmUs, 64 * (t - DK / 64), (int32_t)(wu_rec * C), sKV + t * 8192, pol_rec);
      }
      tc::bulk_commit();
      bulk_pending = true;
    }
  };

  // This group's tasks are vc + i * nv; (chunk, head) of the next two are
  // tracked incrementally, without 64-bit divisions.
  const int32_t n_chunks = map.seq_chunk0[num_seqs];   // negative after malformed cu_seqlens
  const int32_t dj = (int32_t)((unsigned)nv / (unsigned)H), dh = (int32_t)((unsigned)nv % (unsigned)H);
  int32_t j_next = (int32_t)((unsigned)vc / (unsigned)H), h_next = (int32_t)((unsigned)vc % (unsigned)H);
  auto advance = [&](int32_t& jt, int32_t& ht) {
    jt += dj;
    ht += dh;
    if (ht >= H) {
      ht -= H;
      ++jt;
    }
  };
  auto fetch = [&](int64_t t, int32_t jt) -> int4 {
    return (t < n_tasks && jt < n_chunks) ? ld_early_v4(map.chunk_info + jt) : make_int4(0, 0, 0, 0);
  };
  // Thread 0: raw g, k, q of pass `h` of a task (channels 64h..64h+63 of 64 tokens
  // of one head, zero-filled past the token array; rows past the sequence end are
  // masked by the gate and by beta = 0).
  auto raw_issue = [&](int32_t ht, int4 ci, int h) {
    if (ci.y <= 0) return;
    tc::mbar_arrive_expect_tx(bar, (uint32_t)(3 * C * KH * 2));
    tc::tma_load_3d_hint(smem + L::oRaw, &tmG, KH * h, ht, ci.z, bar, pol_in);
    tc::tma_load_3d_hint(smem + L::oRaw + C * KH * 2, &tmK, KH * h, ht, ci.z, bar, pol_in);
    tc::tma_load_3d_hint(smem + L::oRaw + 2 * C * KH * 2, &tmQ, KH * h, ht, ci.z, bar, pol_in);
  };
  auto load_beta = [&](int32_t ht, int4 ci) -> float {
    return (gt < ci.y) ? ld_early_f32(beta + ((int64_t)(uint32_t)ci.z + gt) * H + ht) : 0.f;   // ci.y <= 64
  };
  int4 ci_next = fetch(vc, j_next);
  float beta_next = gt < C ? load_beta(h_next, ci_next) : 0.f;
  int32_t j_next2 = j_next, h_next2 = h_next;
  advance(j_next2, h_next2);
  int4 ci_next2 = fetch((int64_t)vc + nv, j_next2);
  if (ctl) raw_issue(h_next, ci_next, 0);

  // Thread -> channel pair (c, c+1) of the pass and the 8 rows r0..r0+7 of sub-tile a.
  const int rg = gw, a = rg >> 1, c = 2 * lane, r0 = 8 * rg;
  bool failed = false;
  for (int64_t task = vc; task < n_tasks; task += nv) {
    const int4 ci = ci_next;
    const int32_t h_cur = h_next;
    const float beta_cur = beta_next;
    ci_next = ci_next2;
    j_next = j_next2;
    h_next = h_next2;
    if (gt < C) beta_next = load_beta(h_next, ci_next);
    advance(j_next2, h_next2);
    ci_next2 = fetch(task + 2 * (int64_t)nv, j_next2);
    if (ci.y <= 0) {   // group-uniform
      if (ctl) raw_issue(h_next, ci_next, 0);
      continue;
    }
    const int len = ci.y;
    const int64_t rec = task;   // == j * H + h
    const int64_t tok0 = (int64_t)(uint32_t)ci.z;
    f16* o_wq = out.wq + rec * 128 * DK;
    f16* o_kt = out.kt + rec * DK * C;
    float* o_gam = out.gam + rec * DK;
    if (gt < C) sBeta[gt] = beta_cur;   // visible after the next group barrier

#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      const int cg = KH * h + c;   // the thread's first channel
      // v of the columns this pass stores into the [w | u] operand, loaded now, used in step 5
      uint4 vraw[kPerV];
#pragma unroll
      for (int e2 = 0; e2 < kPerV; ++e2) {
        const int idx = gt + e2 * NG, r = idx / (DV / 16);
        const int col = (idx % (DV / 16)) * 8 + (DV / 2) * h;
        vraw[e2] = r < len ? ld_early_v4_hint(v + ((tok0 + r) * H + h_cur) * DV + col, pol_in) : make_uint4(0, 0, 0, 0);
      }
      // 1. Gate and inclusive cumulative sum over the thread's rows, in registers;
      //    the raw k, q of the thread read before the area is reused.
      const uint32_t rp = raw_par;
      const bool ok = tc::mbar_wait(bar, rp, kWaitLimit);
      raw_par ^= 1u;
      float2 G[8];
      {
        float2 run = make_float2(0.f, 0.f);
        if (r0 + 8 <= len) {   // every row of the thread is a token (warp-uniform)
#pragma unroll
          for (int rr = 0; rr < 8; ++rr) {
            const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(rawG + (r0 + rr) * KH + c);
            run = add2(run, log2_decay_bounded2(bf2_to_f2(x)));
            G[rr] = run;
          }
        } else {               // rows past the sequence end carry no decay
#pragma unroll
          for (int rr = 0; rr < 8; ++rr) {
            const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(rawG + (r0 + rr) * KH + c);
            if (r0 + rr < len) run = add2(run, log2_decay_bounded2(bf2_to_f2(x)));
            G[rr] = run;
          }
        }
        *reinterpret_cast<float2*>(sTot + rg * KH + c) = run;
      }
      __nv_bfloat162 kq[8], qq[8];
#pragma unroll
      for (int rr = 0; rr < 8; ++rr) {
        kq[rr] = *reinterpret_cast<const __nv_bfloat162*>(rawK + (r0 + rr) * KH + c);
        qq[rr] = *reinterpret_cast<const __nv_bfloat162*>(rawQ + (r0 + rr) * KH + c);
      }
      // The previous task's [w | u] (first pass), whose product ran during the steps above.
      bool drained = false, okw = true;
      if (h == 0) {
        drained = wu_pending;
        okw = wu_drain_tiles();
        // the P tile of the previous task (in the operand area) has been read by the TMA unit
        if (ctl && bulk_pending) tc::bulk_wait_read0();
      }
      tc::fence_proxy_async_smem();   // drain tiles, written by the threads, read by the TMA unit
      tc::tc_fence_before();
      // The barrier ends every raw read, makes the row-group sums visible and tells
      // every thread whether a raw-row copy failed to land.
      const bool any_bad = tc::bar_sync_or(bar_id, NG, !ok);
      wu_store(drained, okw);
      if (drained && !okw && ctl) atomicExch(dev_err, (int32_t)kDevErrTimeout);
      if (any_bad) {   // a staging copy never landed: report, let it finish, stop
        if (ctl) atomicExch(dev_err, (int32_t)kDevErrTimeout);
        tc::mbar_wait(bar, rp, kWaitLimit);
        if (h == 1) tc::mbar_wait(bar + 2, ap_par, kWaitLimit);   // the first pass's products
        failed = true;
        break;
      }
      if (ctl) {   // the raw rows of the next pass
        if (h == 0)
          raw_issue(h_cur, ci, 1);
        else
          raw_issue(h_next, ci_next, 0);
      }

      // 2. Offsets from the row-group sums: G_s(a') = cumulative decay before
      //    sub-tile a', G_last; the per-thread factors e^{G_s(a') - G_s(a)}, a' > a.
      float2 gsA[4], gl;
      {
        float2 acc = make_float2(0.f, 0.f), excl = acc;
#pragma unroll
        for (int r2 = 0; r2 < 8; ++r2) {
          if ((r2 & 1) == 0) gsA[r2 >> 1] = acc;
          if (r2 == rg) excl = acc;
          acc = add2(acc, *reinterpret_cast<const float2*>(sTot + r2 * KH + c));
        }
        gl = acc;
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) G[rr] = add2(G[rr], excl);
      }
      float2 gs = gsA[0];   // G_s(a), selected without a dynamic register index
#pragma unroll
      for (int a2 = 1; a2 < 4; ++a2)
        if (a2 == a) gs = gsA[a2];
      const float2 ngs = make_float2(-gs.x, -gs.y);
      float2 om[4];
#pragma unroll
      for (int a2 = 0; a2 < 4; ++a2) om[a2] = a2 > a ? ex2_pair(add2(gsA[a2], ngs)) : splat2(a2 == a ? 1.f : 0.f);
      if (rg == 0) {
        tc::st_global_hint(o_gam + cg, __float_as_uint(ex2_approx(gl.x)), pol_rec);
        tc::st_global_hint(o_gam + cg + 1, __float_as_uint(ex2_approx(gl.y)), pol_rec);
      }

      // 3. The operand tiles of this pass (the second pass first waits for the first
      //    pass's products, which read the same tiles).
      if (h == 1) {
        if (!tc::mbar_wait(bar + 2, ap_par, kWaitLimit) && ctl) atomicExch(dev_err, (int32_t)kDevErrTimeout);
        ap_par ^= 1u;
      }
#pragma unroll
      for (int rr = 0; rr < 8; ++rr) {
        const int r = r0 + rr;
        const float2 e = ex2_pair(add2(G[rr], ngs));   // e^{G_r - G_s} in (e^-80, 1]
        const float2 k = bf2_to_f2(kq[rr]), q = bf2_to_f2(qq[rr]);
        *reinterpret_cast<uint32_t*>(sRow + xs_off(r, c)) = pack_bf16_pair(mul2(k, e));
        const float2 f = make_float2(rcp_approx(e.x), rcp_approx(e.y));   // e^{G_s - G_r} in [1, e^80)
        uint32_t hi, lo;
        split_bf16_pair(mul2(q, e), hi, lo);
        *reinterpret_cast<uint32_t*>(sRow + xs_off(C + r, c)) = hi;
        *reinterpret_cast<uint32_t*>(sRow + xs_off(2 * C + r, c)) = lo;
        const float2 kf = mul2(k, f);
        split_bf16_pair(kf, hi, lo);   // own sub-tile: high and low parts
        *reinterpret_cast<uint32_t*>(sCol + xs_off(r, c)) = hi;
        *reinterpret_cast<uint32_t*>(sCol + xs_off(kLo + r, c)) = lo;
#pragma unroll
        for (int a2 = 1; a2 < 4; ++a2) {   // later sub-tiles: factors <= 1, high part only
          if (a2 > a)
            *reinterpret_cast<uint32_t*>(sCol + xs_off(kLater + later_row0(a2) + r, c)) =
                pack_bf16_pair(mul2(kf, om[a2]));
        }
      }
      if (ctl && bulk_pending) {   // the [w | u] tiles stored above have been read (the
        tc::bulk_wait_read0();         // operand area of [w | u] is rewritten after the barrier)
        bulk_pending = false;
      }
      tc::fence_proxy_async_smem();   // the operands, written by the threads, read by the MMAs
      tc::tc_fence_before();
      gsync();
      tc::tc_fence_after();

      // 4. This pass's K = 64 of the A / P products (bf16 operands, fp32 in TMEM).
      if (ctl) {
        const uint64_t dR = tc::desc_kmajor_sw128(tc::smem_u32(sRow));
        const uint64_t dC = tc::desc_kmajor_sw128(tc::smem_u32(sCol));
        constexpr uint64_t kRowQ = (uint64_t)(C * 128) >> 4, kColLo = (uint64_t)(kLo * 128) >> 4;
#pragma unroll
        for (int kk = 0; kk < KH / 16; ++kk) {
          const uint64_t oK = (uint64_t)(kk * 32) >> 4;
          const uint32_t acc = (h > 0 || kk > 0) ? 1u : 0u;
          tc::mma_16bit(tm, dR + oK, dC + oK, kIdD1, acc);                       // D1
          tc::mma_16bit(tm + kLo, dR + oK, dC + kColLo + oK, kIdDc, acc);        // Dc: [k ; q_hi] (own lo)^T
          tc::mma_16bit(tm + kLo, dR + kRowQ + oK, dC + oK, kIdDc, 1u);          //   + [q_hi ; q_lo] (own hi)^T
        }
        tc::mma_commit(bar + 2);
      }

      // 5. While they run: [beta k e^G | beta V] (the operand of [w | u]) and the
      //    record's q e^G rows and (k e^{G_last - G})^T of this pass's channels.
      {
        uint32_t kt0[4], kt1[4];   // K~^T rows cg and cg+1, tokens r0..r0+7, fp16 pairs
        float bw[8];
        *reinterpret_cast<float4*>(bw) = *reinterpret_cast<const float4*>(sBeta + r0);
        *reinterpret_cast<float4*>(bw + 4) = *reinterpret_cast<const float4*>(sBeta + r0 + 4);
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) {
          const int r = r0 + rr;
          const float2 eg = ex2_pair(G[rr]);                            // e^{G_r}
          const float2 el = ex2_pair(fma2(G[rr], splat2(-1.f), gl));    // e^{G_last - G_r}
          const float2 k = bf2_to_f2(kq[rr]), q = bf2_to_f2(qq[rr]);
          const float2 keg = mul2(k, eg);
          *reinterpret_cast<uint32_t*>(sKV + kv_off(r, cg)) = pack_f16_pair(mul2(keg, splat2(bw[rr])));
          tc::st_global_hint(o_wq + (C + r) * DK + cg, pack_f16_pair(mul2(q, eg)), pol_rec);
          const uint32_t kt = pack_f16_pair(mul2(k, el));   // channels cg, cg + 1 of token r
          if (rr & 1) {   // tokens r - 1, r of each channel as one fp16 pair
            kt0[rr >> 1] = __byte_perm(kt0[rr >> 1], kt, 0x5410);
            kt1[rr >> 1] = __byte_perm(kt1[rr >> 1], kt, 0x7632);
          } else {
            kt0[rr >> 1] = kt;
            kt1[rr >> 1] = kt;
          }
        }
        tc::st_global_hint(o_kt + cg * C + r0, make_uint4(kt0[0], kt0[1], kt0[2], kt0[3]), pol_rec);
        tc::st_global_hint(o_kt + (cg + 1) * C + r0, make_uint4(kt1[0], kt1[1], kt1[2], kt1[3]), pol_rec);
#pragma unroll
        for (int e2 = 0; e2 < kPerV; ++e2) {   // beta V (beta is 0 on rows past the sequence end)
          const int idx = gt + e2 * NG, r = idx / (DV / 16);
          const int col = (idx % (DV / 16)) * 8 + (DV / 2) * h;
          const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&vraw[e2]);
          const float2 br = splat2(sBeta[r]);
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) pk[e] = pack_f16_pair(mul2(bf2_to_f2(x[e]), br));
          *reinterpret_cast<uint4*>(sKV + kv_off(r, DK + col)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
    }
    if (failed) break;

    // 6. A and P out of TMEM: A to shared memory (diagonal blocks fp32, blocks below
    //    them fp16, beta-weighted), P to the record tile.  Warp -> TMEM lane quarter q
    //    (rows 32(q%2).. of A for q < 2, of P for q >= 2) and 16-column blocks 2(w/4),
    //    2(w/4)+1; each lane holds one row r of sub-tile ar.
    {
      if (!tc::mbar_wait(bar + 2, ap_par, kWaitLimit) && ctl) atomicExch(dev_err, (int32_t)kDevErrTimeout);
      ap_par ^= 1u;
      tc::tc_fence_after();
      const int q = gw & 3;
      const uint32_t tl = (uint32_t)(32 * q);
      const int rr = 32 * (q & 1) + lane, ar = rr >> 4;
#pragma unroll
      for (int bb = 0; bb < 2; ++bb) {
        const int b = 2 * (gw >> 2) + bb;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          const int ap = 2 * (q & 1) + part;   // the sub-tile of lanes 16 part .. 16 part + 15
          float x[16];
          if (q < 2) {
            if (b > ap) continue;
            tc::tmem_ld16(tc::tmem_addr(tm, tl, b == ap ? 16 * b : kLater + later_row0(ap) + 16 * b), x);
            if (ar != ap) continue;
            const float2 br = splat2(sBeta[rr]);
            float2 y[8];   // beta_r A_ri
#pragma unroll
            for (int i = 0; i < 8; ++i) y[i] = mul2(make_float2(x[2 * i], x[2 * i + 1]), br);
            if (b == ap) {   // diagonal block, fp32 (only its strictly lower part is read)
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                sA[rr * LDA + 2 * i] = y[i].x;
                sA[rr * LDA + 2 * i + 1] = y[i].y;
              }
            } else {         // below the diagonal, fp16
              uint4* dst = reinterpret_cast<uint4*>(sAh + rr * LDX + 16 * b);
#pragma unroll
              for (int j = 0; j < 2; ++j)
                dst[j] = make_uint4(pack_f16_pair(y[4 * j + 0]), pack_f16_pair(y[4 * j + 1]), pack_f16_pair(y[4 * j + 2]),
                                    pack_f16_pair(y[4 * j + 3]));
            }
          } else {
            if (b > ap) {
#pragma unroll
              for (int i = 0; i < 16; ++i) x[i] = 0.f;
            } else if (b == ap) {   // hi x hi + (hi x lo + lo x hi), inclusive lower triangle
              float w2[16];
              tc::tmem_ld16(tc::tmem_addr(tm, tl, 16 * b), x);
              tc::tmem_ld16(tc::tmem_addr(tm, tl, kLo + 16 * b), w2);
#pragma unroll
              for (int i = 0; i < 16; ++i) x[i] = i <= (rr & 15) ? x[i] + w2[i] : 0.f;
            } else {
              tc::tmem_ld16(tc::tmem_addr(tm, tl, kLater + later_row0(ap) + 16 * b), x);
            }
            if (ar != ap) continue;
#pragma unroll
            for (int j = 0; j < 2; ++j)
              *reinterpret_cast<uint4*>(sPst + xs_off(rr, 16 * b + 8 * j)) =
                  make_uint4(pack_f16x2(x[8 * j + 0], x[8 * j + 1]), pack_f16x2(x[8 * j + 2], x[8 * j + 3]),
                             pack_f16x2(x[8 * j + 4], x[8 * j + 5]), pack_f16x2(x[8 * j + 6], x[8 * j + 7]));
          }
        }
      }
    }
    tc::tc_fence_before();
    tc::fence_proxy_async_smem();   // the P tile, written by the threads, read by the TMA unit
    gsync();
    if (ctl) {   // P to the record (the tile is released before the next task's first barrier)
      tc::tma_store_2d_hint(&tmPs, 0, (int32_t)(rec * C), sPst, pol_rec);
      tc::bulk_commit();
      bulk_pending = true;
      if (ready && pub_rec >= 0) {   // the previous task's record: its P and [w | u] stores are
        if (batch_first < 0) batch_first = pub_rec;   // the groups before this P store
        batch_last = pub_rec;
        pub_rec = -1;
        if (++batch_n == kSplitPublishBatch) {
          tc::bulk_wait1();
          publish_records(ready, batch_first, batch_last, nv);
          batch_first = -1;
          batch_n = 0;
        }
      }
    }

    // 7. X = (I + A)^{-1} in fp16: diagonal 16x16 blocks by forward substitution in
    //    fp32 (warp = block, lane = column, in registers), then the blocks below them
    //    in two stages of dependent 16x16 products on mma.sync:
    //      1: X_10 = -X_11 A_10 X_00,  X_32 = -X_33 A_32 X_22,  T_21 = A_21 X_11,  T_31 = A_31 X_11
    //      2: X_20 = -X_22 T_20,  X_21 = -X_22 T_21,  X_30 = -(X_32 T_20 + X_33 T_30),
    //         X_31 = -(X_32 T_21 + X_33 T_31),  with T_a0 = A_a0 X_00 + A_a1 X_10.
    //    Meanwhile warps 4-7 write the zeros of X above its block diagonal and the two
    //    zero blocks around X.
    if (gw < C / kSub) {
      if (lane < kSub) {
        const int base = gw * kSub, jc = lane;
        float xc[kSub];
#pragma unroll
        for (int r = 0; r < kSub; ++r) xc[r] = (r == jc) ? 1.f : 0.f;
#pragma unroll
        for (int i = 0; i < kSub - 1; ++i) {
#pragma unroll
          for (int r = i + 1; r < kSub; ++r) xc[r] -= sA[(base + r) * LDA + i] * xc[i];
        }
#pragma unroll
        for (int r = 0; r < kSub; ++r)
          *reinterpret_cast<f16*>(sX + xs_off(base + r, base + jc)) = __float2half_rn(xc[r]);
      }
    } else {
      const int z = gt - 32 * (C / kSub);
      constexpr int kZeroThreads = NG - 32 * (C / kSub);
      for (int idx = z; idx < 6 * 32; idx += kZeroThreads) {   // zeros above the block diagonal of X
        const int blk = idx >> 5, e = idx & 31;
        const int ra = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
        const int rb = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
        *reinterpret_cast<uint4*>(sX + xs_off(16 * ra + (e >> 1), 16 * rb + 8 * (e & 1))) = make_uint4(0u, 0u, 0u, 0u);
      }
      for (int idx = z; idx < 1024; idx += kZeroThreads)   // the zero blocks before and after X
        *reinterpret_cast<uint4*>(smem + (idx < 512 ? L::oZ0 + (size_t)idx * 16 : L::oZ1 + (size_t)(idx - 512) * 16)) =
            make_uint4(0u, 0u, 0u, 0u);
    }
    gsync();
    {
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
          *reinterpret_cast<uint32_t*>(sX + xs_off(16 * ra + gq, 16 * rb + 8 * nt + 2 * tq)) =
              pack_f16x2(-y[nt][0], -y[nt][1]);
          *reinterpret_cast<uint32_t*>(sX + xs_off(16 * ra + gq + 8, 16 * rb + 8 * nt + 2 * tq)) =
              pack_f16x2(-y[nt][2], -y[nt][3]);
        }
      };
      constexpr int kBlk = 16 * 24;   // scratch block: 0, 1 stage-1 products, 2 T_21, 3 T_31, 4, 5 T_20, 6 T_30
      uint32_t fa[4], fb[4];
      if (gw < 2) {   // stage 1: X_10 (warp 0), X_32 (warp 1)
        const int ra = gw == 0 ? 1 : 3, rb = ra - 1;
        float y[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        ld_a(ra, rb, fa);
        ld_xb(rb, rb, fb);
        mma_nn(y, fa, fb);
        f16* yb = sYh + gw * kBlk;
        st_t(yb, y);
        __syncwarp();
        float x[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        ld_xa(ra, ra, fa);
        ld_tb(yb, fb);
        mma_nn(x, fa, fb);
        st_x(ra, rb, x);
      } else if (gw < 4) {   // stage 1: T_21 (warp 2), T_31 (warp 3)
        float y[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        ld_a(gw, 1, fa);
        ld_xb(1, 1, fb);
        mma_nn(y, fa, fb);
        st_t(sYh + gw * kBlk, y);
      }
      gsync();
      float x[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      if (gw == 1) {          // X_21 = -X_22 T_21
        ld_xa(2, 2, fa);
        ld_tb(sYh + 2 * kBlk, fb);
        mma_nn(x, fa, fb);
        st_x(2, 1, x);
      } else if (gw == 3) {   // X_31 = -(X_32 T_21 + X_33 T_31)
        ld_xa(3, 2, fa);
        ld_tb(sYh + 2 * kBlk, fb);
        mma_nn(x, fa, fb);
        ld_xa(3, 3, fa);
        ld_tb(sYh + 3 * kBlk, fb);
        mma_nn(x, fa, fb);
        st_x(3, 1, x);
      } else if (gw == 0 || gw == 2) {   // X_20 (warp 0), X_30 (warp 2): both form T_20
        float t[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        ld_a(2, 0, fa);
        ld_xb(0, 0, fb);
        mma_nn(t, fa, fb);
        ld_a(2, 1, fa);
        ld_xb(1, 0, fb);
        mma_nn(t, fa, fb);
        f16* t20 = sYh + (gw == 0 ? 4 : 5) * kBlk;
        st_t(t20, t);
        if (gw == 2) {
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
        if (gw == 0) {
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

    // 8. [w | u] = X [beta k e^G | beta V] on the tensor cores, w and u stacked in 128
    //    TMEM columns: w = [X ; 0] (beta k e^G) into lanes 0-63 (lanes 64-127 get
    //    zeros), then u = [0 ; X] (beta V) added into lanes 64-127 of its d_v columns.
    //    Read out at the start of the next task.
    tc::fence_proxy_async_smem();   // X and the operand written by the threads, seen by the MMAs
    tc::tc_fence_before();
    gsync();
    tc::tc_fence_after();
    if (gw == kWuIssuer && lane == 0) {   // warp 2 has no part in step 1's drain before its barrier
      const uint64_t dXw = tc::desc_kmajor_sw128(tc::smem_u32(sX));
      const uint64_t dXu = tc::desc_kmajor_sw128(tc::smem_u32(smem + L::oZ0));
      const uint64_t dKw = tc::desc_mnmajor_sw128_atoms(tc::smem_u32(sKV), 8192);
      const uint64_t dKu = tc::desc_mnmajor_sw128_atoms(tc::smem_u32(sKV + (DK / 64) * 8192), 8192);
#pragma unroll
      for (int kk = 0; kk < C / 16; ++kk)
        tc::mma_16bit(tm, dXw + ((kk * 32) >> 4), dKw + ((kk * 2048) >> 4), kIdW, kk > 0);
#pragma unroll
      for (int kk = 0; kk < C / 16; ++kk)
        tc::mma_16bit(tm, dXu + ((kk * 32) >> 4), dKu + ((kk * 2048) >> 4), kIdU, 1u);
      tc::mma_commit(bar + 1);
    }
    wu_pending = true;
    wu_rec = rec;
    // No barrier here: until the next task's first one the threads write only sBeta
    // (its last readers finished before the barrier above) and read the raw rows.
  }
  {   // the last task's [w | u]
    const bool drained = wu_pending;
    const bool okw = wu_drain_tiles();
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    gsync();
    wu_store(drained, okw);
    if (drained && !okw && ctl) atomicExch(dev_err, (int32_t)kDevErrTimeout);
  }
  if (ctl) tc::bulk_wait0();   // every record store of the group has completed
  if (ready && ctl) {
    if (pub_rec >= 0) {
      if (batch_first < 0) batch_first = pub_rec;
      batch_last = pub_rec;
    }
    if (batch_first >= 0) publish_records(ready, batch_first, batch_last, nv);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (tid < 32) tc::tmem_dealloc(*tmem_slot, 2 * kGroupCols);
}

}  // namespace ps
}  // namespace kda
