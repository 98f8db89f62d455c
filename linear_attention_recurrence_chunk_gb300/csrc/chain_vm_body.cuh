// Device code of the value-major inter-chunk chain of the tensor-core prefill, for d_v = 128 (the
// plain call): one CTA per (sequence, head) walks the sequence's chunks with all
// value columns.
//
// The products of the chain (page "Kimi K3：架构、训练与百万 Token Agentic RL 技术解读"
// §3.3, chunked prefill with the state carried across chunk boundaries) are
// taken transposed, value column = TMEM lane:
//
//   group 1:  VN   = u^T I - S^T w^T          (M = 128 values, N = 64 tokens, K = 64, then d_k)
//             V_new^T = VN, to fp16               (threads)
//   group 2:  D3   = V_new^T K~                  (M = 128, N = d_k, K = 64 tokens)
//             O    = -S^T (q e^G)^T - V_new^T P^T (the o rows, negated; N = 64)
//             S^T  = S^T Diag(e^{G_last}) + D3   (threads, fp32 in registers)
//
// so that both operands the threads produce, S^T and V_new^T, are the A
// operands of the next products and go straight back into TMEM (tcgen05.st)
// instead of through shared memory: each hand-off is a TMEM read, a rounding
// to fp16 (and for the state the decay and sum), a TMEM write and an mbarrier
// arrive.  The products that need a minus sign take the instruction's negate-B
// flag, u enters the accumulator through a product with the identity (u as an
// MN-major A operand, as stored), so V_new = u - w S is formed in fp32 and
// rounded to fp16 once, and the o rows come out negated.  The o product, off
// the chain's path, runs after the state product, from its own copy of S^T
// (two TMEM buffers, by chunk parity).  The records are read as the other
// chains read them: [w; q e^G] (rows x keys), P (rows x tokens) and K~^T
// (keys x tokens) are K-major B operands as stored.
//
// The records of a chunk arrive by TMA in two rings released separately:
// [w; q e^G] and u (three slots, free once group 1 has run) and K~^T, P with
// e^{G_last} (two slots, free once group 2 has run), so that the larger part
// is requested about two chunk steps before it is used.
//
// Warp roles: consumers 0 .. n-1 (n = 8 or 16; warp w: value lanes
// 32(w%4)..+31; for V_new 256/n tokens, for the state 512/n keys, held in fp32
// registers); four o warps (one per lane quarter: read a chunk's o^T out of
// TMEM into a shared-memory tile that TMA stores as o rows); the TMA producer
// (lane 0 feeds the first ring, lane 16 the second); the MMA issuer.  The output epilogue is not fused here: its per-row
// normalisation over all 128 values would fall on these four warps alone.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "chain_common.cuh"
#include "kda_internal.cuh"
#include "tc_ptx.cuh"

namespace kda {
namespace vm {

using bf16 = __nv_bfloat16;
using tcu::kWaitLimit;
using tcu::pack_bf16x2;
using tcu::pack_f16x2;
using tcu::report_nonfinite;

constexpr int C = kChunk;   // 64 tokens per chunk
constexpr int DK = 128, DV = 128;
constexpr int kOWarps = 4;
constexpr int kSlotsA = 3, kSlotsB = 2;
constexpr int kGamSlots = 4;   // e^{G_last} ring: a chunk's factors stay until its state update has used them

// TMEM columns (512 allocated)
constexpr uint32_t kVN = 0;      // V_new^T, 64 columns (fp32)
constexpr uint32_t kO = 64;      // two buffers of 64 (chunk parity): -o^T
constexpr uint32_t kD3 = 192;    // (K~^T V_new)^T, 128 columns
constexpr uint32_t kSA = 320;    // two buffers of 64 (chunk parity): S^T as the fp16 A operand (pairs of keys)
constexpr uint32_t kVA = 448;    // V_new^T as the fp16 A operand: 32 columns (pairs of tokens)
constexpr uint32_t kTmemCols = 512;

struct VmSmem {
  // ring A slot: [w; q e^G] (128 rows x 128 keys, two 64-key atoms of 16 KB), then
  // u (64 tokens x 128 values, two 64-value atoms of 8 KB); 128-byte swizzle
  static constexpr uint32_t kSlotA = 49152, kAU = 32768;
  static constexpr uint32_t kTxA = 49152;
  // ring B slot: (k e^{G_last - G})^T (128 keys x 64 tokens), then P (64 x 64)
  static constexpr uint32_t oB = kSlotsA * kSlotA, kSlotB = 24576, kBP = 16384;
  static constexpr uint32_t kTxB = 24576 + DK * 4;   // with e^{G_last} into its own ring
  static constexpr uint32_t oI = oB + kSlotsB * kSlotB;   // the 64 x 64 identity, fp16, K-major, 128-byte swizzle
  static constexpr uint32_t oGam = oI + 8192;             // fp32 [kGamSlots][DK]
  // o staging, bf16: the two 64-value boxes of the TMA store, [64 tokens][128 B]
  // each, 128-byte swizzle
  static constexpr uint32_t oO = oGam + kGamSlots * DK * 4 + 2048;   // 1024-aligned
  static constexpr uint32_t oBar = oO + 2 * 8192;
  static constexpr uint32_t oTmem = oBar + 19 * 8;
  static constexpr uint32_t kBytes = oTmem + 8;
  static constexpr uint32_t kAlloc = kBytes + 1024;   // slack to align the base to 1024
  static_assert(kAlloc <= 232448, "fits the 227 KB shared-memory limit");
  static_assert(oB % 1024 == 0 && oI % 1024 == 0 && oGam % 512 == 0 && oO % 1024 == 0 && oBar % 8 == 0, "alignment");
};


// Warp roles for kCons consumer warps (8 or 16): consumers 0 .. kCons-1, o warps
// kCons .. kCons+3, the TMA producer kCons+4, the MMA issuer kCons+5.
template <int kCons>
struct VmWarps {
  static_assert(kCons == 8 || kCons == 16, "consumer warps");
  static constexpr int kConsumerWarps = kCons, kOWarp0 = kCons, kTmaWarp = kCons + 4, kMmaWarp = kCons + 5;
  static constexpr int kThreads = 32 * (kCons + 6);
  static constexpr int KPW = 512 / kCons;   // state keys per consumer warp
  static constexpr int TPW = 256 / kCons;   // V_new tokens per consumer warp
};

// Waits (bounded) until the record of a chunk has been published by the prep
// role of the fused kernel (a release store of 1 after the record's stores
// completed), then orders the TMA reads that follow after it.
__device__ __forceinline__ bool wait_record(const int32_t* flag) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
  if (v == 0) {
    const long long t0 = clock64();
    do {
      if (clock64() - t0 > kWaitLimit) return false;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    } while (v == 0);
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

// The chain of (sequence, head) `chain_idx` (sequence-rank major order), run by
// the whole CTA.  `ready` (or null) holds the publication flags of the records,
// [max_chunks * H], when the records are written concurrently by the fused
// kernel's prep role; the records are then loaded with evict-first priority and,
// given `recs`, their L2 lines dropped once consumed (nothing reads them again).
template <int kCons>
__device__ __forceinline__ void chain_body(const CUtensorMap& tmWQ, const CUtensorMap& tmP, const CUtensorMap& tmKT,
                                           const CUtensorMap& tmU, const CUtensorMap& tmGam, const CUtensorMap& tmO,
                                           const int32_t* __restrict__ cu, int32_t num_seqs, int64_t T_seq, int32_t H,
                                           const ChunkMap& map, const float* __restrict__ s0,
                                           float* __restrict__ s_final, bf16* __restrict__ o, int32_t* dev_err,
                                           int chain_idx, const int32_t* __restrict__ ready,
                                           const TcRecords* recs = nullptr) {
  using W = VmWarps<kCons>;
  constexpr int kConsumerWarps = W::kConsumerWarps, kOWarp0 = W::kOWarp0, kTmaWarp = W::kTmaWarp,
                kMmaWarp = W::kMmaWarp;
  using L = VmSmem;
  constexpr uint32_t kIdN64 = tc::idesc_f16_f32(128, 64), kIdN128 = tc::idesc_f16_f32(128, 128);
  constexpr uint32_t kIdU = kIdN64 | (1u << 15);       // u^T I: A (u) MN-major
  constexpr uint32_t kIdNeg64 = kIdN64 | (1u << 14);    // B negated
  if (map.seq_chunk0[num_seqs] < 0) return;   // malformed cu_seqlens: write nothing
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* fullA = reinterpret_cast<uint64_t*>(sm + L::oBar);   // [3] a ring-A slot has landed
  uint64_t* emptyA = fullA + 3;    // [3] the products are done with a ring-A slot
  uint64_t* fullB = fullA + 6;     // [2] a ring-B slot (and its e^{G_last}) has landed
  uint64_t* emptyB = fullA + 8;    // [2] group 2 is done with a ring-B slot
  uint64_t* mma1 = fullA + 10;     // group 1 complete: V_new^T in VN
  uint64_t* mma2 = fullA + 11;     // the state product complete
  uint64_t* drain = fullA + 12;    // every MMA complete (kernel end)
  uint64_t* vn_ready = fullA + 13; // the consumer warps have written V_new^T
  uint64_t* s_ready = fullA + 14;  // the consumer warps have written S^T (and read D3)
  uint64_t* ofull = fullA + 15;    // [2] a chunk's -o^T is complete in its O buffer
  uint64_t* ofree = fullA + 17;    // [2] the o warps have read an O buffer
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::oTmem);

  // one-dimensional grid, sequence-rank major: all heads of the longest sequence first
  const int s = map.seq_order[chain_idx / H], h = chain_idx % H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int32_t j0 = map.seq_chunk0[s];
  const int32_t nch = map.seq_chunk0[s + 1] - j0;
  const int64_t seq_start = cu ? (int64_t)cu[s] : (int64_t)s * T_seq;
  const int64_t seq_end = cu ? (int64_t)cu[s + 1] : seq_start + T_seq;

  if (tid == 0) {
    for (int i = 0; i < 13; ++i) tc::mbar_init(fullA + i, 1);
    tc::mbar_init(vn_ready, kConsumerWarps);
    tc::mbar_init(s_ready, kConsumerWarps);
    tc::mbar_init(ofull, 1);
    tc::mbar_init(ofull + 1, 1);
    tc::mbar_init(ofree, kOWarps);
    tc::mbar_init(ofree + 1, kOWarps);
    tc::fence_mbar_init();
  }
  // the identity B operand of u^T I: row n holds 1 in column n
  for (int idx = tid; idx < C * 8; idx += (int)blockDim.x) {
    const int n = idx >> 3, ch = idx & 7;   // row, 16-byte chunk of 8 columns
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if ((n >> 3) == ch) {
      const uint32_t one = (n & 1) ? 0x3c000000u : 0x00003c00u;   // fp16 1.0 in the low or high half
      const int w = (n & 7) >> 1;
      v.x = w == 0 ? one : 0u;
      v.y = w == 1 ? one : 0u;
      v.z = w == 2 ? one : 0u;
      v.w = w == 3 ? one : 0u;
    }
    *reinterpret_cast<uint4*>(sm + L::oI + (uint32_t)n * 128u + ((uint32_t)(ch ^ (n & 7)) << 4)) = v;
  }
  if (warp == 0) {
    tc::tmem_alloc(tslot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_proxy_async_smem();   // the identity, written by the threads, read by the MMAs
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == kTmaWarp) {
    // ---------------- TMA producer: lane 0 ring A, lane 16 ring B (each slot refilled
    // once the products that read it have completed)
    const uint64_t pol = ready ? tc::l2_policy_evict_first() : tc::l2_policy_evict_normal();
    if (lane == 0) {
      tc::tma_prefetch_desc(&tmWQ);
      tc::tma_prefetch_desc(&tmU);
      int issued = 0;
      for (int i = 0; i < nch; ++i) {
        const int sl = i % kSlotsA;
        if (i >= kSlotsA && !tc::mbar_wait(emptyA + sl, ((i / kSlotsA) - 1) & 1, kWaitLimit)) {
          atomicExch(dev_err, (int32_t)kDevErrTimeout);
          break;
        }
        const int64_t rec = (int64_t)(j0 + i) * H + h;
        if (ready && !wait_record(ready + rec)) {
          atomicExch(dev_err, (int32_t)kDevErrTimeout);
          break;
        }
        uint8_t* slot = sm + sl * L::kSlotA;
        tc::mbar_arrive_expect_tx(fullA + sl, L::kTxA);
        tc::tma_load_2d_hint(slot, &tmWQ, 0, (int32_t)(rec * 128), fullA + sl, pol);
        tc::tma_load_2d_hint(slot + 16384, &tmWQ, 64, (int32_t)(rec * 128), fullA + sl, pol);
        tc::tma_load_2d_hint(slot + L::kAU, &tmU, 0, (int32_t)(rec * C), fullA + sl, pol);
        tc::tma_load_2d_hint(slot + L::kAU + 8192, &tmU, 64, (int32_t)(rec * C), fullA + sl, pol);
        ++issued;
      }
      // never leave loads in flight: wait (bounded) until the last ones landed
      for (int i = (issued > kSlotsA ? issued - kSlotsA : 0); i < issued; ++i)
        tc::mbar_wait(fullA + i % kSlotsA, (i / kSlotsA) & 1, kWaitLimit);
    } else if (lane == 16) {
      tc::tma_prefetch_desc(&tmKT);
      tc::tma_prefetch_desc(&tmP);
      tc::tma_prefetch_desc(&tmGam);
      int issued = 0;
      for (int i = 0; i < nch; ++i) {
        const int sl = i & 1;
        // the e^{G_last} slot of chunk i - 4 is free by then too: its state update
        // preceded the consumers' V_new of chunk i - 2, which group 2 of i - 2 waited for
        if (i >= kSlotsB && !tc::mbar_wait(emptyB + sl, ((i >> 1) - 1) & 1, kWaitLimit)) {
          atomicExch(dev_err, (int32_t)kDevErrTimeout);
          break;
        }
        const int64_t rec = (int64_t)(j0 + i) * H + h;
        if (ready && !wait_record(ready + rec)) {
          atomicExch(dev_err, (int32_t)kDevErrTimeout);
          break;
        }
        uint8_t* slot = sm + L::oB + sl * L::kSlotB;
        tc::mbar_arrive_expect_tx(fullB + sl, L::kTxB);
        tc::tma_load_2d_hint(slot, &tmKT, 0, (int32_t)(rec * DK), fullB + sl, pol);
        tc::tma_load_2d_hint(slot + L::kBP, &tmP, 0, (int32_t)(rec * C), fullB + sl, pol);
        tc::tma_load_2d_hint(sm + L::oGam + (i % kGamSlots) * DK * 4, &tmGam, 0, (int32_t)rec, fullB + sl, pol);
        ++issued;
      }
      for (int i = (issued > kSlotsB ? issued - kSlotsB : 0); i < issued; ++i)
        tc::mbar_wait(fullB + (i & 1), (i >> 1) & 1, kWaitLimit);
    }
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer (the whole warp runs the loop; one elected lane issues)
    const uint64_t dSm = tc::desc_kmajor_sw128(tc::smem_u32(sm));   // base for the K-major tiles
    const uint64_t dI = tc::desc_kmajor_sw128(tc::smem_u32(sm + L::oI));
    auto wait_all = [&](uint64_t* b, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, tc::mbar_wait(b, parity, kWaitLimit));
    };
    // u^T I of chunk j into VN (its V_new^T of chunk j - 1 was read before that
    // chunk's V_new hand-off), once chunk j's ring-A slot has landed: issued
    // after the previous chunk's o product, it runs while the state is updated
    auto issue_u = [&](int j) -> bool {
      const int sa = j % kSlotsA;
      if (!wait_all(fullA + sa, (j / kSlotsA) & 1)) return false;
      tc::tc_fence_after();
      const uint64_t dU = tc::desc_mnmajor_sw128_atoms(tc::smem_u32(sm + sa * L::kSlotA + L::kAU), 8192);
#pragma unroll
      for (int kk = 0; kk < C / 16; ++kk)
        tc::mma_16bit_w(tmem + kVN, dU + ((kk * 2048) >> 4), dI + ((kk * 32) >> 4), kIdU, kk > 0);
      return true;
    };
    bool ok = nch == 0 || issue_u(0), issued = nch > 0 && ok;
    for (int i = 0; i < nch && ok; ++i) {
      const int sa = i % kSlotsA, sb = i & 1;
      const uint32_t b = (uint32_t)(i & 1);
      const uint32_t sA = tmem + kSA + b * 64;   // this chunk's S^T
      const uint64_t dWQ = dSm + ((uint64_t)(sa * L::kSlotA) >> 4);
      ok = wait_all(s_ready, i & 1);
      if (!ok) break;
      tc::tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < DK / 16; ++kk)   // group 1: VN += -S^T w^T
        tc::mma_16bit_tw(tmem + kVN, sA + 8 * kk, dWQ + (((kk >> 2) * 16384 + (kk & 3) * 32) >> 4), kIdNeg64, 1u);
      tc::mma_commit_w(mma1);
      ok = wait_all(vn_ready, i & 1) && wait_all(fullB + sb, (i >> 1) & 1);
      if (!ok) break;
      tc::tc_fence_after();
      const uint64_t dKT = dSm + ((uint64_t)(L::oB + sb * L::kSlotB) >> 4);
#pragma unroll
      for (int kk = 0; kk < C / 16; ++kk)   // group 2: the state product first, it is on the chain's path
        tc::mma_16bit_tw(tmem + kD3, tmem + kVA + 8 * kk, dKT + ((kk * 32) >> 4), kIdN128, kk > 0);
      tc::mma_commit_w(mma2);
      // the o rows, once the o warps have read this buffer's previous chunk:
      // -S^T (q e^G)^T from this chunk's copy of S^T (the state update writes the
      // other one), then -V_new^T P^T
      ok = i < 2 || wait_all(ofree + b, ((i >> 1) - 1) & 1);
      if (!ok) break;
      tc::tc_fence_after();
      const uint32_t dO = tmem + kO + b * 64;
#pragma unroll
      for (int kk = 0; kk < DK / 16; ++kk)
        tc::mma_16bit_tw(dO, sA + 8 * kk, dWQ + ((8192 + (kk >> 2) * 16384 + (kk & 3) * 32) >> 4), kIdNeg64, kk > 0);
      tc::mma_commit_w(emptyA + sa);
#pragma unroll
      for (int kk = 0; kk < C / 16; ++kk)
        tc::mma_16bit_tw(dO, tmem + kVA + 8 * kk, dKT + ((L::kBP + kk * 32) >> 4), kIdNeg64, 1u);
      tc::mma_commit_w(ofull + b);
      tc::mma_commit_w(emptyB + sb);
      if (i + 1 < nch) ok = issue_u(i + 1);
    }
    if (!ok && lane == 0) atomicExch(dev_err, (int32_t)kDevErrTimeout);
    if (issued) {
      tc::mma_commit_w(drain);
      wait_all(drain, 0);
    }
  } else if (warp < kConsumerWarps) {
    // ---------------- consumers: V_new^T and the state
    constexpr int KPW = W::KPW, TPW = W::TPW;
    const int q = warp & 3, part = warp >> 2;
    const int c = 32 * q + lane;   // value column = TMEM lane
    const uint32_t tl = (uint32_t)(32 * q);
    float S[KPW];                  // S[key KPW part + j][value c]
    const int64_t sbase = ((int64_t)s * H + h) * DK * DV + (int64_t)(KPW * part) * DV + c;
#pragma unroll
    for (int j = 0; j < KPW; ++j) S[j] = s0 ? s0[sbase + (int64_t)j * DV] : 0.f;
    // S^T into TMEM buffer `buf` as the fp16 A operand (key pairs per column)
    auto write_sa = [&](uint32_t buf) {
#pragma unroll
      for (int h16 = 0; h16 < KPW / 32; ++h16) {
        uint32_t w[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) w[m] = pack_f16x2(S[32 * h16 + 2 * m], S[32 * h16 + 2 * m + 1]);
        tc::tmem_st16(tc::tmem_addr(tmem, tl, kSA + 64 * buf + (KPW / 2) * part + 16 * h16), w);
      }
    };
    write_sa(0);
    tc::tmem_st_wait();
    tc::tc_fence_before();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(s_ready);
    // state snapshots: chunks left until the next one, and its slot
    int snap_left = map.snap_every > 0 ? map.snap_every : 0x7fffffff;
    int64_t snap_slot = map.snap_every > 0 ? (int64_t)map.snap_slot0[s] : 0;
    const int32_t n_full = (int32_t)((seq_end - seq_start) / C);   // full chunks of the sequence
    bool bad = false;
    int i = 0;
    for (; i < nch; ++i) {
      const uint32_t b = (uint32_t)(i & 1);
      // e^{G_last} of this chunk is read in the state update; its copy is counted on
      // the ring-B barrier, whose phase for chunk i + 2 cannot start before this
      // warp's V_new hand-off below
      bad |= !tc::mbar_wait(fullB + (i & 1), (i >> 1) & 1, kWaitLimit);
      bad |= !tc::mbar_wait(mma1, i & 1, kWaitLimit);
      if (__any_sync(0xffffffffu, bad)) {   // warp-uniform, so that no lane is left at a __syncwarp
        bad = true;
        break;
      }
      tc::tc_fence_after();
      // V_new^T (fp32, tokens TPW part .. +TPW-1) to fp16 pairs, as the A operand of group 2
#pragma unroll
      for (int h16 = 0; h16 < TPW / 16; ++h16) {
        float d[16];
        tc::tmem_ld16(tc::tmem_addr(tmem, tl, kVN + TPW * part + 16 * h16), d);
        uint32_t vw[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) vw[m] = pack_f16x2(d[2 * m], d[2 * m + 1]);
        tc::tmem_st8(tc::tmem_addr(tmem, tl, kVA + (TPW / 2) * part + 8 * h16), vw);
      }
      tc::tmem_st_wait();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(vn_ready);
      bad |= !tc::mbar_wait(mma2, i & 1, kWaitLimit);
      if (__any_sync(0xffffffffu, bad)) {
        bad = true;
        break;
      }
      tc::tc_fence_after();
      // S^T = S^T Diag(e^{G_last}) + D3 for the warp's keys, then its fp16 copy
      // into the next chunk's buffer
      const float* gam = reinterpret_cast<const float*>(sm + L::oGam + (i % kGamSlots) * DK * 4) + KPW * part;
#pragma unroll
      for (int g = 0; g < KPW / 16; ++g) {
        float d[16];
        tc::tmem_ld16(tc::tmem_addr(tmem, tl, kD3 + KPW * part + 16 * g), d);
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4) {   // key pairs in packed fp32x2 fused multiply-adds
          const float4 gv = *reinterpret_cast<const float4*>(gam + 16 * g + 4 * e4);
          float* sp = S + 16 * g + 4 * e4;
          const float2 s01 = __ffma2_rn(make_float2(gv.x, gv.y), make_float2(sp[0], sp[1]),
                                        make_float2(d[4 * e4 + 0], d[4 * e4 + 1]));
          const float2 s23 = __ffma2_rn(make_float2(gv.z, gv.w), make_float2(sp[2], sp[3]),
                                        make_float2(d[4 * e4 + 2], d[4 * e4 + 3]));
          sp[0] = s01.x;
          sp[1] = s01.y;
          sp[2] = s23.x;
          sp[3] = s23.y;
        }
      }
      write_sa(b ^ 1u);
      tc::tmem_st_wait();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(s_ready);
      if (--snap_left == 0) {   // the slot rule of snapshot_slot(), counted down instead of divided
        snap_left = map.snap_every;
        if (i < n_full) {
          float* dst = map.snaps + ((snap_slot * H + h) * DK + KPW * part) * DV + c;
#pragma unroll
          for (int j = 0; j < KPW; ++j) dst[(int64_t)j * DV] = S[j];
          ++snap_slot;
        }
      }
    }
    if (i < nch || bad) {
      atomicExch(dev_err, (int32_t)kDevErrTimeout);
    } else {
      float nonfinite = 0.f;   // stays 0 unless a state value is inf or NaN (x * 0 is then NaN)
#pragma unroll
      for (int j = 0; j < KPW; ++j) nonfinite = fmaf(S[j], 0.f, nonfinite);
      report_nonfinite(nonfinite, dev_err);
      if (s_final) {
        float* dst = s_final + sbase;
#pragma unroll
        for (int j = 0; j < KPW; ++j) dst[(int64_t)j * DV] = S[j];
      }
    }
  } else if (warp < kOWarp0 + kOWarps) {
    // ---------------- o warps
    // Each chunk: o^T out of TMEM (this warp's 32 value lanes, 64 tokens, in 16 x 8
    // blocks) as bf16 into the two staging boxes (the layout of a TMA store, by
    // transposing 8 x 8 matrix stores), the O buffer released; then, after a
    // barrier of the four o warps, a full chunk leaves
    // by two TMA stores, and a sequence's last, partial chunk row by row (thread
    // ot writes the 8 values 8 (ot % 16) .. +7 of rows 8 j + ot / 16: 16 lanes
    // per 256-byte row).
    const int q = warp & 3;
    const int ot = tid - 32 * kOWarp0, g8 = ot & 15, r0 = ot >> 4;
    uint8_t* stile = sm + L::oO;
    // byte offset of (token t, value v) in the staging boxes: box v / 64, 16-byte chunk (v % 64) / 8 ^ t % 8
    auto soff = [](int t, int v) -> uint32_t {
      return (uint32_t)(v >> 6) * 8192u + (uint32_t)t * 128u + ((uint32_t)(((v & 63) >> 3) ^ (t & 7)) << 4) +
             (uint32_t)(v & 7) * 2u;
    };
    float nonfinite = 0.f;          // stays 0 unless an o value is inf or NaN
    bool bad = false, store_pending = false;   // store_pending: thread 0 has TMA stores reading the staging
    for (int i = 0; i < nch; ++i) {
      const uint32_t b = (uint32_t)(i & 1);
      const int64_t t0 = seq_start + (int64_t)i * C;
      const int len = (int)min((int64_t)C, seq_end - t0);
      const bool okw = tc::mbar_wait(ofull + b, (i >> 1) & 1, kWaitLimit);
      const bool wbad = __any_sync(0xffffffffu, !okw);
      if (store_pending) {   // thread 0: the previous chunk's stores have read the staging
        tc::bulk_wait_read0();
        store_pending = false;
      }
      // every o warp reaches both barriers once per chunk, also after a failed wait:
      // the first ends the previous chunk's use of the staging, the second this chunk's writes
      if (tc::bar_sync_or(1, 32 * kOWarps, wbad)) {
        bad = true;
        break;
      }
      tc::tc_fence_after();
      if (recs) {   // every product of this chunk has completed: its record's L2 lines are dead
        const int64_t rec = (int64_t)(j0 + i) * H + h;
        for (int l = ot; l < 256 + 128 + 128 + 64; l += 32 * kOWarps) {
          const __half* line = l < 256 ? recs->wq + rec * 128 * DK + l * 64
                               : l < 384 ? recs->u + rec * C * DV + (l - 256) * 64
                               : l < 512 ? recs->kt + rec * DK * C + (l - 384) * 64
                                         : recs->p + rec * C * C + (l - 512) * 64;
          tc::discard_l2_line(line);
        }
      }
#pragma unroll
      for (int hl = 0; hl < 2; ++hl) {   // value lanes 32 q + 16 hl .. +15
        float v[32];
        tc::tmem_ld_16x256b_x8(tc::tmem_addr(tmem, (uint32_t)(32 * q + 16 * hl), kO + b * 64), v);
        // o (the accumulator holds -o) as bf16 pairs of consecutive tokens: the 8 x 8
        // blocks [8 values][8 tokens] of token block tb, value half vh in pk[2 tb + vh]
        uint32_t pk[16];
#pragma unroll
        for (int tb = 0; tb < 8; ++tb) {
#pragma unroll
          for (int e = 0; e < 4; ++e) nonfinite = fmaf(v[4 * tb + e], 0.f, nonfinite);
          pk[2 * tb] = pack_bf16x2(-v[4 * tb], -v[4 * tb + 1]);
          pk[2 * tb + 1] = pack_bf16x2(-v[4 * tb + 2], -v[4 * tb + 3]);
        }
        // stored transposed (token rows of 8 values): call sc takes token blocks
        // 2 sc, 2 sc + 1; lane L gives the address of row L % 8 of block L / 8
        const int mL = lane >> 3, rL = lane & 7;
#pragma unroll
        for (int sc = 0; sc < 4; ++sc)
          tc::stmatrix_x4_trans(tc::smem_u32(stile + soff(8 * (2 * sc + (mL >> 1)) + rL, 32 * q + 16 * hl + 8 * (mL & 1))),
                                pk[4 * sc], pk[4 * sc + 1], pk[4 * sc + 2], pk[4 * sc + 3]);
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(ofree + b);
      tc::fence_proxy_async_smem();   // the staging, written by the threads, read by the TMA unit
      tc::bar_sync_or(1, 32 * kOWarps, false);
      if (len == C) {
        if (ot == 0) {
          tc::tma_store_3d(&tmO, 0, h, (int32_t)t0, stile);
          tc::tma_store_3d(&tmO, 64, h, (int32_t)t0, stile + 8192);
          tc::bulk_commit();
          store_pending = true;
        }
      } else {
        bf16* orow0 = o + (t0 * H + h) * DV + 8 * g8;   // value 8 g8 of the chunk's first row
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int r = 8 * j + r0;
          if (r < len)
            *reinterpret_cast<uint4*>(orow0 + (int64_t)r * H * DV) = *reinterpret_cast<const uint4*>(stile + soff(r, 8 * g8));
        }
      }
    }
    if (store_pending) tc::bulk_wait0();   // thread 0: every o store has completed
    if (bad) atomicExch(dev_err, (int32_t)kDevErrTimeout);
    else report_nonfinite(nonfinite, dev_err);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace vm
}  // namespace kda
