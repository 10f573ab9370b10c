// Tensor-core backward (fp16/bf16, D in {32, 64, 96, 128}): a dK/dV kernel and a dQ kernel, both
// TMA + tcgen05 + TMEM, recomputing P from the forward's logsumexp ("[Metal] Add Flash
// Attention VJP for training", sections "Implementation Notes" and "Limitations").
//
// dK/dV kernel: one block owns 128 rows of one KV head (KV-row ownership: every dK/dV
// row is written once by one block, so no atomics) and loops over the G query heads of
// its GQA group and their 128-row query blocks.  Per query block, with keys in TMEM lanes:
//   Sᵀ = K·Qᵀ, dPᵀ = V·dOᵀ                          (tcgen05, fp32 in TMEM)
//   Pᵀ = exp2(c·Sᵀ − log2e·lse), dSᵀ = Pᵀ∘(dPᵀ − δ)  (element warps; written back over
//                                                     Sᵀ and dPᵀ as 16-bit A operands)
//   dV += Pᵀ·dO, dK += dSᵀ·Q                         (tcgen05, accumulators stay in TMEM)
// and finally dK·scale and dV are rounded and stored.  The element warps publish Pᵀ in
// two halves (each warp's first 16 queries, then the rest), so dV starts over the first
// half while the second is computed and runs while dSᵀ is computed, and Sᵀ of the next
// block starts as soon as dV has consumed Pᵀ (the MMA order is dV(n), Sᵀ(n+1), dK(n),
// dPᵀ(n+1)).  dSᵀ is formed from Pᵀ in fp32 (dV uses Pᵀ rounded to the element type, as
// the A operand of a 16-bit MMA must be).  Q and dO tiles stream through separate rings:
// Q(n) is read until dK(n), late in the iteration, dO(n) only until dPᵀ(n) and dV(n), so
// Q has three slots (two in the masked instantiation, whose mask tile takes the third's
// place) and dO two.
//
// dQ kernel: one block owns 128 query rows of one head and loops over 128-row KV blocks:
//   S = Q·Kᵀ, dP = dO·Vᵀ, P = exp2(c·S − log2e·lse_i), dS = P∘(dP − δ_i), dQ += dS·K,
// then dQ·scale is stored.  S alternates between two TMEM buffers, so S of block n+1 is
// computed while block n's element work runs; S, dP and dQ have an issuer warp each, so
// that no issuer waits for an MMA it has just issued.
//
// All MMAs have M = 128, N = 128 (N = D for the accumulating ones): narrower N would make
// the shared-memory operand traffic exceed what one SM's shared memory can deliver.
// Warps 0-15 do the element work: warp e reads TMEM lane quarter e % 4 and owns the
// 32 columns [32c, 32c + 32) of each 128-column block of scores (c = e / 4), writing its
// packed 16-bit results over the first 16 of them; with four warps per SM sub-partition
// the exponential and dS passes hide each other's latencies.  Warp 16 is the TMA producer,
// warps 17 and 18 (and 19 in the dQ kernel) issue the MMAs and warp 17 owns the 512 TMEM
// columns.
//
// Attention masks: both kernels have a masked instantiation (kMasked) that adds log2e·M
// to the log2-domain scores before the exponential.  The dK/dV kernel's producer loads
// each query block's [128 x 128] mask tile by TMA into shared memory, from which each
// element warp reads its keys' column; the dQ kernel (no shared memory left at D = 128)
// reads its row's 32 mask values from global memory in 16-byte pieces before its barrier
// waits.  A row whose lse is −inf (it saw no key) gets P = 0.  Sinks need no change here:
// the forward's lse already includes them.
#include "launch.h"
#include "tc_common.cuh"

namespace sdpa {
namespace {
using namespace tc;

// dK/dV: warps 0-15 element work (four per TMEM lane quarter, each with 32 of the 128
// queries of a block), 16 producer, 17-18 MMA issuers.  65,536 / 608 threads leaves 104
// registers a thread, which the 32-query element work fits.
constexpr int kKvThreads = 608;
constexpr int kKvProducerWarp = 16;
constexpr int kKvMmaWarp = 17;
// dQ: warps 0-15 element work (four per TMEM lane quarter, each with 32 of the 128 keys of
// a block), 16 producer, 17-19 MMA issuers.  Register split (setmaxnreg): launched at 96
// registers a thread (65,536 / 640 rounded down to a multiple of 8, 61,440 in all);
// warpgroup 4 drops to 56 and the element warpgroups rise to 104: 128·56 + 512·104 = 60,416.
constexpr int kDqThreads = 640;
constexpr int kRegsLow = 56;
constexpr int kRegsHigh = 104;
static_assert(128 * kRegsLow + 512 * kRegsHigh <= kDqThreads * 96, "register split exceeds the launch");
constexpr int kProducerWarp = 16;
constexpr int kMmaWarp = 17;
constexpr int kRows = 128;  // rows owned by a block (keys for dK/dV, queries for dQ)
constexpr int kBlk = 128;   // rows of the streamed operand per iteration
constexpr int kStages = 2;  // dK/dV: depth of the dO ring and of the per-query vector ring

template <typename T>
struct IsBf16 { static constexpr bool value = false; };
template <>
struct IsBf16<__nv_bfloat16> { static constexpr bool value = true; };

__device__ __forceinline__ float pos_inf() { return __int_as_float(0x7f800000); }

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > limit_ns) return;
  }
}

// TMEM column of the packed 16-bit A operand for K-step kk (16 rows of the streamed
// operand) when the element warps own kSplit columns each and pack their results into the
// first kSplit / 2 of them: dQ (kSplit = 64) packs rows 0-63 into columns [0, 32) and rows
// 64-127 into [64, 96); dK/dV (kSplit = 32) packs rows [32c, 32c + 32) into columns
// [32c, 32c + 16).
template <int kSplit>
__device__ __forceinline__ uint32_t packed_col(int kk) {
  constexpr int kSteps = kSplit / 16;  // K-steps per owner
  return (kk / kSteps) * kSplit + (kk % kSteps) * 8;
}

// Shared-memory plan (offsets from a 1024-byte aligned base).
template <int D>
struct BwdLayout {
  static constexpr int kCB = (D + 63) / 64;            // 64-column blocks (D = 96 padded to 128)
  static constexpr int kTileBytes = kRows * kCB * 64 * 2;  // one [128 x D] tile
  static constexpr int kOwnA = 0;                      // K (dK/dV) or Q (dQ)
  static constexpr int kOwnB = kTileBytes;             // V (dK/dV) or dO (dQ)
  static constexpr int kCbStride = kRows * 128;        // one 64-column block of a tile
};

struct BwdBars {
  uint64_t own_full;
  uint64_t q_full[3];
  uint64_t q_empty[3];        // dK(n) has read the Q slot of query block n
  uint64_t do_full[kStages];
  uint64_t do_empty[kStages]; // dPᵀ(n) and dV(n) have read the dO slot of block n
  uint64_t vec_full[kStages];
  uint64_t vec_empty[kStages];  // every element thread is done with the slot's vectors
  uint64_t s_full[2];     // dK/dV: [0] only.  dQ: one per S buffer
  uint64_t dp_full;
  uint64_t p_half;        // dK/dV: Pᵀ of each warp's first 16 queries packed
  uint64_t p_ready;       // dK/dV: Pᵀ packed
  uint64_t ds_ready;      // dSᵀ / dS packed
  uint64_t x_free;        // dK/dV: dV consumed Pᵀ (Sᵀ region free)
  uint64_t y_free;        // dK/dV: dK consumed dSᵀ (dPᵀ region free)
  uint64_t dq_done[2];    // dQ: dQ MMA of the block in S buffer i has finished
  uint64_t acc_done;
  uint64_t mask_full;     // dK/dV, masked: the query block's mask tile has landed
  uint64_t mask_free;     // dK/dV, masked: every element warp has read it
  uint32_t tmem_base;
  int abort;
  alignas(16) float nlse2[kStages][kBlk];   // dK/dV: −log2e·lse per query (−inf past Lq)
  alignas(16) float ndelta[kStages][kBlk];  // dK/dV: −δ per query
};

__device__ __forceinline__ void init_bars(BwdBars& bars) {
  bars.abort = 0;
  mbar_init(&bars.own_full, 1);
  for (int s = 0; s < 3; ++s) {
    mbar_init(&bars.q_full[s], 1);
    mbar_init(&bars.q_empty[s], 1);
  }
  for (int s = 0; s < kStages; ++s) {
    mbar_init(&bars.do_full[s], 1);
    mbar_init(&bars.do_empty[s], 2);  // released by both MMA issuers
    mbar_init(&bars.vec_full[s], 32);
    mbar_init(&bars.vec_empty[s], 512);
  }
  mbar_init(&bars.s_full[0], 1);
  mbar_init(&bars.s_full[1], 1);
  mbar_init(&bars.dp_full, 1);
  mbar_init(&bars.p_half, 512);    // every element thread of the dK/dV kernel
  mbar_init(&bars.p_ready, 512);
  mbar_init(&bars.ds_ready, 512);
  mbar_init(&bars.x_free, 1);
  mbar_init(&bars.y_free, 1);
  mbar_init(&bars.dq_done[0], 1);
  mbar_init(&bars.dq_done[1], 1);
  mbar_init(&bars.acc_done, 2);  // one commit per MMA issuer
  mbar_init(&bars.mask_full, 1);
  mbar_init(&bars.mask_free, 16);  // one arrival per element warp
  fence_mbar_init();
}

// dK/dV shared memory: the K and V tiles, a ring of Q slots (three, or two in the masked
// instantiation: Q(n) is read until dK(n), late in the iteration), two dO slots (dO(n) is
// free once dPᵀ(n) and dV(n) have read it), then (masked instantiation) one [128 queries x
// 128 keys] mask tile, then the barriers and per-query vectors.  Everything is dynamic
// shared memory with no static part, whose base is the start of the block's shared window
// (1024-byte aligned), so the 224 KB of tiles, mask and barriers need no alignment padding.
template <int D, bool kMasked, bool kRowBc = false>
struct KvSmem {
  static constexpr bool kTileMask = kMasked && !kRowBc;  // a staged mask tile
  static constexpr int kQSlots = kTileMask ? 2 : 3;
  static constexpr int kQ = 2 * BwdLayout<D>::kTileBytes;
  static constexpr int kDo = kQ + kQSlots * BwdLayout<D>::kTileBytes;
  static constexpr int kMask = kDo + kStages * BwdLayout<D>::kTileBytes;
  static constexpr int kMaskBytes = kTileMask ? kBlk * kRows * 2 : 0;  // 16-bit or byte elements
  static constexpr int kBars = kMask + kMaskBytes;
  static constexpr int kBytes = kBars + (int)sizeof(BwdBars);
};
static_assert(KvSmem<128, true>::kBytes <= 227 * 1024, "dK/dV shared memory exceeds the per-block limit");
static_assert(KvSmem<128, false>::kBytes <= 227 * 1024, "dK/dV shared memory exceeds the per-block limit");
static_assert(KvSmem<128, true, true>::kBytes <= 227 * 1024, "dK/dV shared memory exceeds the per-block limit");

// Issues C[tmem] = A·Bᵀ for two [128 x D] K-major tiles in shared memory (N = 128).
// Called by all 32 lanes of the issuing warp; one elected lane issues.
template <int D>
__device__ __forceinline__ void mma_scores(uint32_t c_tmem, uint32_t a_s, uint32_t b_s, uint32_t idesc) {
  const uint64_t ad = sdesc_sw128(a_s, 16, 1024), bd = sdesc_sw128(b_s, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk / 4) * BwdLayout<D>::kCbStride + (kk % 4) * 32;
    mma_ss_w(c_tmem, sdesc_advance(ad, off), sdesc_advance(bd, off), idesc, kk > 0);
  }
}

// Issues Acc[tmem] (+)= A·B with A = packed 16-bit [128 x 128] in TMEM (see packed_col)
// and B = a [128 x D] tile in shared memory read MN-major (N = D, K = its 128 rows).
template <int D, int kSplit>
__device__ __forceinline__ void mma_accumulate(uint32_t acc_tmem, uint32_t a_tmem, uint32_t b_s,
                                               uint32_t idesc, bool first) {
  const uint64_t bd = sdesc_sw128(b_s, BwdLayout<D>::kCbStride, 1024);
#pragma unroll
  for (int kk = 0; kk < kBlk / 16; ++kk)
    mma_ts_w(acc_tmem, a_tmem + packed_col<kSplit>(kk), sdesc_advance(bd, kk * 2048), idesc,
             (!first || kk > 0) ? 1u : 0u);
}

// The K-steps kk = odd, odd + 2, ... of mma_accumulate (odd = 0: the even steps, which
// read each owner's first 16 rows of A; odd = 1: the others).
template <int D, int kSplit>
__device__ __forceinline__ void mma_accumulate_half(uint32_t acc_tmem, uint32_t a_tmem, uint32_t b_s,
                                                    uint32_t idesc, bool first, int odd) {
  const uint64_t bd = sdesc_sw128(b_s, BwdLayout<D>::kCbStride, 1024);
#pragma unroll
  for (int kk = odd; kk < kBlk / 16; kk += 2)
    mma_ts_w(acc_tmem, a_tmem + packed_col<kSplit>(kk), sdesc_advance(bd, kk * 2048), idesc,
             (!first || kk > 0) ? 1u : 0u);
}

// ================================================================== dK / dV
// kRowBc (with kMasked): the mask has one row for every query (row stride 0, the
// [B, 1, 1, Lkv] key-padding form); each element thread reads its key's value from global
// memory once per query block, so no mask tile is staged and Q keeps three slots.
template <typename T, int D, bool kMasked, bool kRowBc>
__global__ void __launch_bounds__(kKvThreads, 1)
    tc_dkdv_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                   const __grid_constant__ CUtensorMap tdk, const __grid_constant__ CUtensorMap tdv,
                   const __grid_constant__ CUtensorMap tm, Problem p) {
  using L = BwdLayout<D>;
  constexpr int kCB = L::kCB;
  constexpr bool kBf16 = IsBf16<T>::value;
  constexpr uint32_t kIdS = idesc_f16(kRows, kBlk, kBf16, false, false);
  constexpr uint32_t kIdAcc = idesc_f16(kRows, D, kBf16, false, true);
  // TMEM columns: dV, dK, Sᵀ (→ Pᵀ), dPᵀ (→ dSᵀ)
  constexpr uint32_t kColDv = 0, kColDk = 128, kColX = 256, kColY = 384;
  using SM = KvSmem<D, kMasked, kRowBc>;
  constexpr bool kTileMask = SM::kTileMask;
  extern __shared__ unsigned char smem_raw[];
  // The layout assumes a 1024-byte aligned base (TMA's 128-byte swizzle and the MMA
  // descriptors need it); should a launch ever place it elsewhere, the block reports an
  // error and leaves before touching shared memory.
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) report_error(p.err, kDevErrLayout, kKidTcDkdv);
    return;
  }
  uint8_t* sm = smem_raw;
  BwdBars& bars = *reinterpret_cast<BwdBars*>(sm + SM::kBars);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // Block order: all (batch, KV head) units of one key tile, then the next tile; under the
  // causal mask the first key tiles see the most queries, so the heavy blocks go first.
  const int units = p.B * p.Hkv;
  const int unit = blockIdx.x % units;
  const int b = unit / p.Hkv, g = unit % p.Hkv;
  const int j0 = (blockIdx.x / units) * kRows;  // first key of this block
  // Queries before j0 - coff see none of these keys.
  const int i_begin = p.causal ? max(0, j0 - p.coff) : 0;
  const int nqb = i_begin < p.Lq ? (p.Lq - i_begin + kBlk - 1) / kBlk : 0;
  const int total = p.G * nqb;

  if (threadIdx.x == 0) init_bars(bars);
  if (warp == kKvMmaWarp) {
    tmem_alloc(&bars.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars.tmem_base;
  const WaitCtx wc{&bars.abort, 0, p.wait_limit_ns, p.err, kKidTcDkdv};

  if (warp == kKvProducerWarp) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tdo);
      mbar_arrive_expect_tx(&bars.own_full, 2 * L::kTileBytes);
      for (int cb = 0; cb < kCB; ++cb) {
        tma_load_4d(sm + L::kOwnA + cb * L::kCbStride, &tk, &bars.own_full, cb * 64, j0, g, b);
        tma_load_4d(sm + L::kOwnB + cb * L::kCbStride, &tv, &bars.own_full, cb * 64, j0, g, b);
      }
    }
    // Per query block n: Q(n) into its slot once dK of the block that last used it has read
    // it, dO(n) into its slot once dPᵀ and dV of that block have, the mask tile (masked),
    // then the per-query vectors once the element threads are done with those of n - 2.
    int q_issued = 0, do_issued = 0, m_issued = 0;
    bool ok = true;
    for (int n = 0; ok && n < total; ++n) {
      const int s = n % kStages, qs = n % SM::kQSlots;
      const int h = g * p.G + n / nqb;
      const int i0 = i_begin + (n % nqb) * kBlk;
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.q_empty[qs], ((n / SM::kQSlots) & 1) ^ 1, wc));
      if (!ok) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars.q_full[qs], L::kTileBytes);
        for (int cb = 0; cb < kCB; ++cb)
          tma_load_4d(sm + SM::kQ + qs * L::kTileBytes + cb * L::kCbStride, &tq, &bars.q_full[qs], cb * 64, i0, h,
                      b);
      }
      q_issued = n + 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.do_empty[s], ((n / kStages) & 1) ^ 1, wc));
      if (!ok) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars.do_full[s], L::kTileBytes);
        for (int cb = 0; cb < kCB; ++cb)
          tma_load_4d(sm + SM::kDo + s * L::kTileBytes + cb * L::kCbStride, &tdo, &bars.do_full[s], cb * 64, i0,
                      h, b);
      }
      do_issued = n + 1;
      if (kTileMask) {
        // The query block's mask tile, once every element warp has read the previous one.
        if (n > 0) ok = __all_sync(0xffffffffu, mbar_wait(&bars.mask_free, (n - 1) & 1, wc));
        if (!ok) break;
        if (lane == 0) {
          const int es = p.mask_kind == kMaskBool ? 1 : 2;
          const bool row_bc = p.lm.sl == 0;  // one row serves every query
          mbar_arrive_expect_tx(&bars.mask_full, (row_bc ? 1 : kBlk) * kRows * es);
          tma_load_4d(sm + SM::kMask, &tm, &bars.mask_full, j0, row_bc ? 0 : i0, p.lm.sh == 0 ? 0 : h,
                      p.lm.sb == 0 ? 0 : b);
        }
        m_issued = n + 1;
      }
      // Per-query vectors, negated for the packed math of the element warps.
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.vec_empty[s], ((n / kStages) & 1) ^ 1, wc));
      if (!ok) break;
      const float* lsep = p.lse + q_row(p, b, h, 0);
      const float* dlp = p.delta + q_row(p, b, h, 0);
#pragma unroll
      for (int e = lane; e < kBlk; e += 32) {
        const int i = i0 + e;
        const float l = i < p.Lq ? lsep[i] : -pos_inf();  // −inf: the row sees no key, P = 0
        bars.nlse2[s][e] = l == -pos_inf() ? -pos_inf() : -l * kLog2e;
        bars.ndelta[s][e] = i < p.Lq ? -dlp[i] : 0.f;
      }
      mbar_arrive(&bars.vec_full[s]);
    }
    if (lane == 0 && (!ok || bars.abort)) {  // let copies still in flight land before the block exits
      for (int n = max(0, q_issued - SM::kQSlots); n < q_issued; ++n)
        drain_wait(&bars.q_full[n % SM::kQSlots], (n / SM::kQSlots) & 1, 100000000ull);
      for (int n = max(0, do_issued - kStages); n < do_issued; ++n)
        drain_wait(&bars.do_full[n % kStages], (n / kStages) & 1, 100000000ull);
      if (kTileMask && m_issued > 0) drain_wait(&bars.mask_full, (m_issued - 1) & 1, 100000000ull);
    }
  } else if (warp == kKvMmaWarp || warp == kKvMmaWarp + 1) {
    // ---------------------------------------------------------------- MMA issuers
    // Warp 17 issues Sᵀ, dV and dK in the order dV(n), Sᵀ(n+1), dK(n): Sᵀ(n+1) overwrites the
    // Pᵀ(n) that dV(n) reads, so it waits for dV(n) to finish, and issuing dK(n) only after
    // it keeps dK(n) from running ahead of Sᵀ(n+1) (the element warps need Sᵀ(n+1) next,
    // while dK(n) only gates dPᵀ(n+1), which they need a whole exponential pass later).
    // Warp 18 issues dPᵀ(n) once dK(n-1) has consumed dSᵀ(n-1).
    constexpr unsigned kAll = 0xffffffffu;
    const bool chain_x = __shfl_sync(kAll, warp, 0) == kKvMmaWarp;
    bool ok = __all_sync(kAll, mbar_wait(&bars.own_full, 0, wc));
    tc_fence_after();
    const uint32_t k_s = smem_u32(sm + L::kOwnA), v_s = smem_u32(sm + L::kOwnB);
    constexpr int kQs = SM::kQSlots;
    auto q_slot = [&](int n) { return smem_u32(sm + SM::kQ + (n % kQs) * L::kTileBytes); };
    auto do_slot = [&](int n) { return smem_u32(sm + SM::kDo + (n % kStages) * L::kTileBytes); };
    if (chain_x) {
      if (ok && total > 0) {
        ok = __all_sync(kAll, mbar_wait(&bars.q_full[0], 0, wc));
        if (ok) {
          tc_fence_after();
          mma_scores<D>(tbase + kColX, k_s, q_slot(0), kIdS);  // Sᵀ(0) = K·Q(0)ᵀ
          mma_commit_w(&bars.s_full[0]);
        }
      }
      for (int n = 0; ok && n < total; ++n) {
        const uint32_t q_s = q_slot(n), do_s = do_slot(n);
        // dV += Pᵀ·dO in two halves: the K-steps of the queries whose Pᵀ the element warps
        // write first, then the rest, so that dV(n) is half done when the Pᵀ pass ends.
        if (!(ok = __all_sync(kAll, mbar_wait(&bars.p_half, n & 1, wc) &&
                                        mbar_wait(&bars.do_full[n % kStages], (n / kStages) & 1, wc))))
          break;
        tc_fence_after();
        mma_accumulate_half<D, 32>(tbase + kColDv, tbase + kColX, do_s, kIdAcc, n == 0, 0);
        if (!(ok = __all_sync(kAll, mbar_wait(&bars.p_ready, n & 1, wc)))) break;
        tc_fence_after();
        mma_accumulate_half<D, 32>(tbase + kColDv, tbase + kColX, do_s, kIdAcc, n == 0, 1);
        mma_commit_w(&bars.x_free);
        mma_commit_w(&bars.do_empty[n % kStages]);  // one of the slot's two arrivals
        if (n + 1 < total) {
          if (!(ok = __all_sync(kAll, mbar_wait(&bars.q_full[(n + 1) % kQs], ((n + 1) / kQs) & 1, wc) &&
                                          mbar_wait(&bars.x_free, n & 1, wc))))
            break;
          tc_fence_after();
          mma_scores<D>(tbase + kColX, k_s, q_slot(n + 1), kIdS);  // Sᵀ(n+1)
          mma_commit_w(&bars.s_full[0]);
        }
        if (!(ok = __all_sync(kAll, mbar_wait(&bars.ds_ready, n & 1, wc)))) break;
        tc_fence_after();
        mma_accumulate<D, 32>(tbase + kColDk, tbase + kColY, q_s, kIdAcc, n == 0);  // dK += dSᵀ·Q
        mma_commit_w(&bars.y_free);
        mma_commit_w(&bars.q_empty[n % kQs]);
      }
    } else {
      for (int n = 0; ok && n < total; ++n) {
        const uint32_t do_s = do_slot(n);
        if (!(ok = __all_sync(kAll, mbar_wait(&bars.do_full[n % kStages], (n / kStages) & 1, wc)))) break;
        if (n > 0 && !(ok = __all_sync(kAll, mbar_wait(&bars.y_free, (n - 1) & 1, wc)))) break;
        tc_fence_after();
        mma_scores<D>(tbase + kColY, v_s, do_s, kIdS);  // dPᵀ = V·dOᵀ
        mma_commit_w(&bars.dp_full);
        mma_commit_w(&bars.do_empty[n % kStages]);  // one of the slot's two arrivals
      }
    }
    mma_commit_w(&bars.acc_done);
    drain_wait(&bars.acc_done, 0, 100000000ull);
  } else {
    // ---------------------------------------------------------------- element warps
    // Warp e: TMEM lane quarter e % 4 (keys), query columns [32c, 32c + 32) with c = e / 4.
    const int c = warp / 4, quarter = warp % 4;
    const int j = j0 + quarter * 32 + lane;  // this thread's key
    const uint32_t x_addr = tmem_addr(tbase, quarter * 32, kColX + 32 * c);
    const uint32_t y_addr = tmem_addr(tbase, quarter * 32, kColY + 32 * c);
    const uint64_t cc = f2pack(p.scale_log2, p.scale_log2);
    constexpr bool masked = kMasked;  // a separate instantiation carries the mask code
    bool ok = true;
    for (int n = 0; n < total; ++n) {
      const int s = n % kStages;
      const int i0 = i_begin + (n % nqb) * kBlk + 32 * c;  // first query of this warp's columns
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.s_full[0], n & 1, wc) &&
                                       mbar_wait(&bars.vec_full[s], (n / kStages) & 1, wc) &&
                                       (!kTileMask || mbar_wait(&bars.mask_full, n & 1, wc)));
      if (!ok) break;
      tc_fence_after();
      const int ic = i0 + p.coff;  // key j is hidden from query i0 + q when j > ic + q
      const bool diag = p.causal && j0 + kRows - 1 > ic;
      const uint64_t* nl2 = reinterpret_cast<const uint64_t*>(&bars.nlse2[s][32 * c]);
      const uint64_t* nd2 = reinterpret_cast<const uint64_t*>(&bars.ndelta[s][32 * c]);
      // Pᵀ for this warp's 32 queries from one TMEM load; the packed 16-bit values go over
      // the first 16 of its own Sᵀ columns for dV, and Pᵀ stays in registers in fp32 for dSᵀ.
      uint64_t pf[16];  // fp32 pairs
      uint64_t mrow = 0;  // one-row mask: log2e·M of this key, in both halves
      {
        uint32_t sr[32];
        tmem_ld32(x_addr, sr);
        tmem_ld_wait(sr);
        if constexpr (masked && kRowBc) {
          // The one mask value of this key for every query (0 past Lkv: those keys' rows
          // are clipped) goes into the per-query constant below: c·s + (−log2e·lse + log2e·M).
          const float mv = j < p.Lkv ? mask_log2<T>(p, row_off(p.lm, b, g * p.G + n / nqb, 0) + j) : 0.f;
          mrow = f2pack(mv, mv);
        } else if constexpr (masked) {
          // c·s + log2e·M for this key against the warp's queries, M read from the block's
          // mask tile in shared memory (row q, key k at element 128q + k; one row when the
          // mask is broadcast over queries).  Rows past Lq and keys past Lkv were filled with
          // zeros by the load: those P are zero or clipped anyway.  c·s is finite, so a
          // hidden key's −inf passes through the fma unchanged.
          const int k_local = quarter * 32 + lane;
          if (p.mask_kind == kMaskBool) {
            const uint8_t* m8 = sm + SM::kMask + k_local;
            if (p.lm.sl == 0) {
              const float mv = m8[0] ? 0.f : minus_inf();
#pragma unroll
              for (int e = 0; e < 32; ++e) sr[e] = __float_as_uint(fmaf(p.scale_log2, __uint_as_float(sr[e]), mv));
            } else {
              m8 += 32 * c * kRows;
#pragma unroll
              for (int e = 0; e < 32; ++e)
                sr[e] = __float_as_uint(fmaf(p.scale_log2, __uint_as_float(sr[e]), m8[e * kRows] ? 0.f : minus_inf()));
            }
          } else {
            const T* m16 = reinterpret_cast<const T*>(sm + SM::kMask) + k_local;
            if (p.lm.sl == 0) {
              const float mv = Elem<T>::to_f(m16[0]) * kLog2e;
#pragma unroll
              for (int e = 0; e < 32; ++e) sr[e] = __float_as_uint(fmaf(p.scale_log2, __uint_as_float(sr[e]), mv));
            } else {
              m16 += 32 * c * kRows;
#pragma unroll
              for (int e = 0; e < 32; ++e)
                sr[e] = __float_as_uint(fmaf(p.scale_log2, __uint_as_float(sr[e]), Elem<T>::to_f(m16[e * kRows]) * kLog2e));
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars.mask_free);  // this warp is done with the mask tile
        }
        const uint64_t ce = kTileMask ? f2pack(1.f, 1.f) : cc;
        // Two halves of 16 queries, each stored as soon as it is packed: the first half
        // lets the dV product start (p_half) while the second is computed.
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t pk[8];
#pragma unroll
          for (int e8 = 0; e8 < 8; ++e8) {
            const int e = 8 * hf + e8;
            float p0, p1;
            const uint64_t nle = kRowBc ? fadd2(nl2[e], mrow) : nl2[e];
            ex2_pair(ffma2(f2pack(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1])), ce, nle), p0, p1);
            if (diag) {
              if (j > ic + 2 * e) p0 = 0.f;
              if (j > ic + 2 * e + 1) p1 = 0.f;
            }
            pf[e] = f2pack(p0, p1);
            pk[e8] = pack2<T>(p0, p1);
          }
          tmem_st8(x_addr + 8 * hf, pk);
          if (hf == 0) {
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bars.p_half);
          }
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars.p_ready);
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.dp_full, n & 1, wc));
      if (!ok) break;
      tc_fence_after();
      // dSᵀ = Pᵀ∘(dPᵀ − δ), one TMEM load.
      {
        uint32_t dr[32];
        tmem_ld32(y_addr, dr);
        tmem_ld_wait(dr);
        uint32_t dk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float d0, d1;
          f2unpack(fmul2(pf[e], fadd2(f2pack(__uint_as_float(dr[2 * e]), __uint_as_float(dr[2 * e + 1])), nd2[e])), d0,
                   d1);
          dk[e] = pack2<T>(d0, d1);
        }
        tmem_st16(y_addr, dk);
      }
      mbar_arrive(&bars.vec_empty[s]);  // done with this block's lse and δ
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars.ds_ready);
    }
    // Epilogue: dV and dK·scale, each in D/32 chunks of 32 columns; warpgroup wg takes the
    // chunks whose index is wg modulo 4.  They are staged in the block's own V and K buffers
    // (no MMA reads them once acc_done has completed) in the swizzled tile layout and written
    // by bulk tensor stores (keys past Lkv are clipped) once all 16 warps have staged theirs.
    // The staging buffers are ones the block's own TMA load fills; with no MMA (total == 0)
    // nothing else has waited for that load, so wait for it here too.
    if (ok)
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.own_full, 0, wc) && (total == 0 || mbar_wait(&bars.acc_done, 0, wc)));
    const int r = quarter * 32 + lane;
    if (ok) {
      tc_fence_after();
      constexpr int kChunks = D / 32;
#pragma unroll 1
      for (int ch = c; ch < 2 * kChunks; ch += 4) {
        const bool is_dk = ch >= kChunks;
        const int c32 = is_dk ? ch - kChunks : ch;
        const float mul = is_dk ? p.scale : 1.f;
        uint32_t acc[32];
        if (total > 0) {
          tmem_ld32(tmem_addr(tbase, quarter * 32, (is_dk ? kColDk : kColDv) + 32 * c32), acc);
          tmem_ld_wait(acc);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) acc[e] = 0u;  // no query sees these keys
        }
        uint32_t packed[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          packed[e] = pack2<T>(__uint_as_float(acc[2 * e]) * mul, __uint_as_float(acc[2 * e + 1]) * mul);
        uint8_t* blk = sm + (is_dk ? L::kOwnA : L::kOwnB) + (c32 / 2) * L::kCbStride;
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4)
          *reinterpret_cast<uint4*>(blk + sw128_off(r, (c32 % 2) * 4 + v4)) =
              make_uint4(packed[4 * v4], packed[4 * v4 + 1], packed[4 * v4 + 2], packed[4 * v4 + 3]);
      }
      fence_async_smem();
    }
    if (named_sync_and(1, 512, ok) && warp == 0 && lane == 0) {
      for (int cb = 0; cb < kCB; ++cb) {
        tma_store_4d(&tdv, sm + L::kOwnB + cb * L::kCbStride, cb * 64, j0, g, b);
        tma_store_4d(&tdk, sm + L::kOwnA + cb * L::kCbStride, cb * 64, j0, g, b);
      }
      bulk_commit();
      bulk_wait_read();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kKvMmaWarp) {
    __syncwarp();
    tmem_dealloc(tbase, 512);
  }
}

// ================================================================== dQ
// K blocks live until dQ has used them, V blocks only until dP has, so they have rings of
// their own: three K stages let the next K block load while dQ still reads the current one.
constexpr int kKStages = 3;
constexpr int kVStages = 2;

template <int D>
struct DqLayout {
  static constexpr int kCB = (D + 63) / 64;  // 64-column blocks (D = 96 padded to 128)
  static constexpr int kTileBytes = kRows * kCB * 64 * 2;
  static constexpr int kQ = 0;
  static constexpr int kDo = kTileBytes;
  static constexpr int kK = 2 * kTileBytes;                       // kKStages K blocks
  static constexpr int kV = kK + kKStages * kTileBytes;           // kVStages V blocks
  static constexpr int kBytes = kV + kVStages * kTileBytes;
};

struct DqBars {
  uint64_t own_full;
  uint64_t k_full[kKStages];
  uint64_t k_empty[kKStages];
  uint64_t v_full[kVStages];
  uint64_t v_empty[kVStages];
  uint64_t s_full[2];   // one per S buffer
  uint64_t dp_full;
  uint64_t dp_free;     // the element warps have read dP (its buffer may be refilled)
  // dS of the block in S buffer i packed (one barrier per buffer: an element warp may start
  // block n+1 while another still packs dS(n), and one barrier could not tell their arrivals
  // apart; block n+2 starts only after dQ(n) has read buffer n % 2, so two suffice)
  uint64_t ds_ready[2];
  uint64_t dq_done[2];  // dQ MMA of the block in S buffer i has finished
  uint64_t acc_done;
  uint32_t tmem_base;
  int abort;
};

template <typename T, int D, bool kMasked>
__global__ void __launch_bounds__(kDqThreads, 1)
    tc_dq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                 const __grid_constant__ CUtensorMap tdq, Problem p) {
  using L = DqLayout<D>;
  constexpr int kCB = L::kCB;
  constexpr int kCbStride = kRows * 128;
  constexpr bool kBf16 = IsBf16<T>::value;
  constexpr uint32_t kIdS = idesc_f16(kRows, kBlk, kBf16, false, false);
  constexpr uint32_t kIdAcc = idesc_f16(kRows, D, kBf16, false, true);
  // TMEM columns: dQ, two S buffers (→ dS), dP
  constexpr uint32_t kColDq = 0, kColS0 = 128, kColDp = 384;
  extern __shared__ unsigned char smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ DqBars bars;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // Block order: all heads of one query tile, then the next; causal: heaviest tiles first.
  const int units = p.B * p.Hq;
  const int unit = blockIdx.x % units, rank = blockIdx.x / units;
  const int b = unit / p.Hq, h = unit % p.Hq, g = h / p.G;
  const int nqt = (p.Lq + kRows - 1) / kRows;
  const int qt = p.causal ? nqt - 1 - rank : rank;
  const int i0 = qt * kRows;
  const int kend = p.causal ? min(p.Lkv, min(p.Lq, i0 + kRows) + p.coff) : p.Lkv;
  const int total = (kend + kBlk - 1) / kBlk;  // KV blocks visited

  if (threadIdx.x == 0) {
    bars.abort = 0;
    mbar_init(&bars.own_full, 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&bars.k_full[s], 1);
      mbar_init(&bars.k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&bars.v_full[s], 1);
      mbar_init(&bars.v_empty[s], 1);
    }
    mbar_init(&bars.s_full[0], 1);
    mbar_init(&bars.s_full[1], 1);
    mbar_init(&bars.dp_full, 1);
    mbar_init(&bars.dp_free, 512);   // every element thread
    mbar_init(&bars.ds_ready[0], 512);
    mbar_init(&bars.ds_ready[1], 512);
    mbar_init(&bars.dq_done[0], 1);
    mbar_init(&bars.dq_done[1], 1);
    mbar_init(&bars.acc_done, 3);  // one commit per MMA issuer
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars.tmem_base;
  const WaitCtx wc{&bars.abort, 0, p.wait_limit_ns, p.err, kKidTcDq};
  if (warp >= 16) regs_dec<kRegsLow>();

  if (warp == kProducerWarp) {
    if (lane == 0) {
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      mbar_arrive_expect_tx(&bars.own_full, 2 * L::kTileBytes);
      for (int cb = 0; cb < kCB; ++cb) {
        tma_load_4d(sm + L::kQ + cb * kCbStride, &tq, &bars.own_full, cb * 64, i0, h, b);
        tma_load_4d(sm + L::kDo + cb * kCbStride, &tdo, &bars.own_full, cb * 64, i0, h, b);
      }
      // The block one wave later (about num_sms blocks on) starts when some block ends:
      // bring its Q and dO tiles into L2 now, so that its first loads come from L2, not HBM.
      if (p.num_sms > 0 && blockIdx.x + p.num_sms < gridDim.x) {
        const int nb = blockIdx.x + p.num_sms;
        const int nu = nb % units, nrank = nb / units;
        const int ni0 = (p.causal ? nqt - 1 - nrank : nrank) * kRows;
        for (int cb = 0; cb < kCB; ++cb) {
          tma_prefetch_l2_4d(&tq, cb * 64, ni0, nu % p.Hq, nu / p.Hq);
          tma_prefetch_l2_4d(&tdo, cb * 64, ni0, nu % p.Hq, nu / p.Hq);
        }
      }
      int k_issued = 0, v_issued = 0;
      bool ok = true;
      for (int n = 0; ok && n < total; ++n) {
        const int sk = n % kKStages, sv = n % kVStages;
        if (!(ok = mbar_wait(&bars.k_empty[sk], ((n / kKStages) & 1) ^ 1, wc))) break;
        mbar_arrive_expect_tx(&bars.k_full[sk], L::kTileBytes);
        for (int cb = 0; cb < kCB; ++cb)
          tma_load_4d(sm + L::kK + sk * L::kTileBytes + cb * kCbStride, &tk, &bars.k_full[sk], cb * 64,
                      n * kBlk, g, b);
        k_issued = n + 1;
        if (!(ok = mbar_wait(&bars.v_empty[sv], ((n / kVStages) & 1) ^ 1, wc))) break;
        mbar_arrive_expect_tx(&bars.v_full[sv], L::kTileBytes);
        for (int cb = 0; cb < kCB; ++cb)
          tma_load_4d(sm + L::kV + sv * L::kTileBytes + cb * kCbStride, &tv, &bars.v_full[sv], cb * 64,
                      n * kBlk, g, b);
        v_issued = n + 1;
      }
      if (!ok || bars.abort) {
        for (int n = max(0, k_issued - kKStages); n < k_issued; ++n)
          drain_wait(&bars.k_full[n % kKStages], (n / kKStages) & 1, 100000000ull);
        for (int n = max(0, v_issued - kVStages); n < v_issued; ++n)
          drain_wait(&bars.v_full[n % kVStages], (n / kVStages) & 1, 100000000ull);
      }
    }
  } else if (warp >= kMmaWarp) {
    // Three issuers, each at its own pace (all lanes of an issuer warp run its loop; one
    // elected lane issues): warp 17 issues S(n) = Q·K(n)ᵀ into S buffer n % 2 once dQ(n-2)
    // has read dS(n-2) from it, warp 18 issues dP(n) = dO·V(n)ᵀ once the element warps
    // have read dP(n-1), and warp 19 issues dQ += dS(n)·K(n) as soon as dS(n) is packed.
    // Keeping dQ apart from S means no issuer waits for an MMA it has just issued.
    constexpr unsigned kAll = 0xffffffffu;
    const int role = __shfl_sync(kAll, warp - kMmaWarp, 0);
    bool ok = __all_sync(kAll, mbar_wait(&bars.own_full, 0, wc));
    tc_fence_after();
    const uint32_t q_s = smem_u32(sm + L::kQ), do_s = smem_u32(sm + L::kDo);
    const uint32_t k_s = smem_u32(sm + L::kK), v_s = smem_u32(sm + L::kV);
    if (role == 0) {
      for (int n = 0; ok && n < total; ++n) {
        if (!(ok = __all_sync(kAll, mbar_wait(&bars.k_full[n % kKStages], (n / kKStages) & 1, wc)))) break;
        if (n >= 2 && !(ok = __all_sync(kAll, mbar_wait(&bars.dq_done[n % 2], ((n - 2) / 2) & 1, wc)))) break;
        tc_fence_after();
        mma_scores<D>(tbase + kColS0 + 128 * (n % 2), q_s, k_s + (n % kKStages) * L::kTileBytes, kIdS);
        mma_commit_w(&bars.s_full[n % 2]);
      }
    } else if (role == 1) {
      // dP(n) into the dP buffer (free once the element warps have read dP(n-1)).
      for (int n = 0; ok && n < total; ++n) {
        if (!(ok = __all_sync(kAll, mbar_wait(&bars.v_full[n % kVStages], (n / kVStages) & 1, wc)))) break;
        if (n >= 1 && !(ok = __all_sync(kAll, mbar_wait(&bars.dp_free, (n - 1) & 1, wc)))) break;
        tc_fence_after();
        mma_scores<D>(tbase + kColDp, do_s, v_s + (n % kVStages) * L::kTileBytes, kIdS);
        mma_commit_w(&bars.dp_full);
        mma_commit_w(&bars.v_empty[n % kVStages]);
      }
    } else {
      for (int n = 0; ok && n < total; ++n) {
        // K(n) is loaded (S(n) read it before dS(n) could exist); waiting on its barrier too
        // makes the TMA writes visible to this warp's MMA directly.
        if (!(ok = __all_sync(kAll, mbar_wait(&bars.ds_ready[n % 2], (n / 2) & 1, wc) &&
                                        mbar_wait(&bars.k_full[n % kKStages], (n / kKStages) & 1, wc))))
          break;
        tc_fence_after();
        // dQ += dS·K: B = the K block read MN-major.
        mma_accumulate<D, 32>(tbase + kColDq, tbase + kColS0 + 128 * (n % 2), k_s + (n % kKStages) * L::kTileBytes,
                          kIdAcc, n == 0);
        mma_commit_w(&bars.dq_done[n % 2]);
        mma_commit_w(&bars.k_empty[n % kKStages]);
      }
    }
    mma_commit_w(&bars.acc_done);
    drain_wait(&bars.acc_done, 0, 100000000ull);
  } else if (warp < 16) {
    regs_inc<kRegsHigh>();
    // Warp e: TMEM lane quarter e % 4 (queries), key columns [32c, 32c + 32) with c = e / 4.
    const int c = warp / 4, quarter = warp % 4;
    const int i = i0 + quarter * 32 + lane;  // this thread's query
    const bool valid = i < p.Lq;
    const int64_t row = q_row(p, b, h, valid ? i : 0);
    const float lse = valid ? p.lse[row] : -pos_inf();
    const float lse2 = lse == -pos_inf() ? pos_inf() : lse * kLog2e;  // no visible key: P = 0
    const float dl = valid ? p.delta[row] : 0.f;
    constexpr bool masked = kMasked;  // a separate instantiation carries the mask code
    const int64_t moff = masked && valid ? row_off(p.lm, b, h, i) : 0;
    const uint64_t cc = f2pack(p.scale_log2, p.scale_log2);
    const uint64_t nl = f2pack(-lse2, -lse2), nd = f2pack(-dl, -dl);
    bool ok = true;
    for (int n = 0; n < total; ++n) {
      const int k0 = n * kBlk + 32 * c;  // first key of this warp's columns
      // Mask terms of this warp's keys as 16-bit pairs (0 past the row's mask pieces: those
      // keys are past Lkv and hidden by lim), read before the waits so that the waits hide
      // their latency.
      uint32_t mk[kMasked ? 16 : 1];
      if constexpr (kMasked) mask_pairs<T, 32>(mk, p, moff + k0, valid && k0 < p.Lkv ? p.Lkv - k0 : 0);
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.s_full[n % 2], (n / 2) & 1, wc) &&
                                       mbar_wait(&bars.dp_full, n & 1, wc));
      if (!ok) break;
      tc_fence_after();
      const bool need_mask = (k0 + 32 > p.Lkv) || (p.causal && k0 + 31 > i0 + p.coff);
      // keys k0 + e with e < lim are visible to this query
      const int lim = min(p.Lkv - k0, p.causal ? i + p.coff - k0 + 1 : 32);
      const uint32_t s_addr = tmem_addr(tbase, quarter * 32, kColS0 + 128 * (n % 2) + 32 * c);
      const uint32_t dp_addr = tmem_addr(tbase, quarter * 32, kColDp + 32 * c);
      // dP and S of this warp's columns in one TMEM round trip; the dP buffer is released at
      // once so that the next block's dP can be computed during this block's math.
      uint32_t dr[32], sr[32];
      tmem_ld32(dp_addr, dr);
      tmem_ld32(s_addr, sr);
      tmem_ld_wait(dr);
      reg_fence(sr);
      tc_fence_before();
      mbar_arrive(&bars.dp_free);
      uint32_t dsk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        float p0, p1;
        uint64_t xx = ffma2(f2pack(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1])), cc, nl);
        if constexpr (kMasked) {
          float x0, x1, m0, m1;
          f2unpack(xx, x0, x1);
          unpack2<T>(mk[e], m0, m1);
          xx = f2pack(x0 + m0 * kLog2e, x1 + m1 * kLog2e);
        }
        ex2_pair(xx, p0, p1);
        if (need_mask) {
          if (2 * e >= lim) p0 = 0.f;
          if (2 * e + 1 >= lim) p1 = 0.f;
        }
        float d0, d1;
        f2unpack(fmul2(f2pack(p0, p1), fadd2(f2pack(__uint_as_float(dr[2 * e]), __uint_as_float(dr[2 * e + 1])), nd)),
                 d0, d1);
        dsk[e] = pack2<T>(d0, d1);
      }
      tmem_st16(s_addr, dsk);  // dS over the first 16 of this warp's columns (all of them read)
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars.ds_ready[n % 2]);
    }
    // Epilogue: dQ·scale in D/32 chunks of 32 columns, warpgroup wg taking the chunks whose
    // index is wg modulo 4, staged in the block's Q buffer (the last S MMA has read it) and
    // written by bulk tensor stores once all 16 warps have staged theirs.  The staging buffer
    // is one the block's own TMA load fills; with no MMA (total == 0) nothing else has
    // waited for that load, so wait for it here too.
    if (ok)
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.own_full, 0, wc) && (total == 0 || mbar_wait(&bars.acc_done, 0, wc)));
    const int r = quarter * 32 + lane;
    if (ok) {
      tc_fence_after();
#pragma unroll 1
      for (int c32 = c; c32 < D / 32; c32 += 4) {
        uint32_t acc[32];
        if (total > 0) {
          tmem_ld32(tmem_addr(tbase, quarter * 32, kColDq + 32 * c32), acc);
          tmem_ld_wait(acc);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) acc[e] = 0u;
        }
        uint32_t packed[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          packed[e] = pack2<T>(__uint_as_float(acc[2 * e]) * p.scale, __uint_as_float(acc[2 * e + 1]) * p.scale);
        uint8_t* blk = sm + L::kQ + (c32 / 2) * kCbStride;
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4)
          *reinterpret_cast<uint4*>(blk + sw128_off(r, (c32 % 2) * 4 + v4)) =
              make_uint4(packed[4 * v4], packed[4 * v4 + 1], packed[4 * v4 + 2], packed[4 * v4 + 3]);
      }
      fence_async_smem();
    }
    if (named_sync_and(1, 512, ok) && warp == 0 && lane == 0) {
      for (int cb = 0; cb < kCB; ++cb) tma_store_4d(&tdq, sm + L::kQ + cb * kCbStride, cb * 64, i0, h, b);
      bulk_commit();
      bulk_wait_read();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tmem_dealloc(tbase, 512);
  }
}

struct Maps {
  CUtensorMap q, k, v, dout, dq, dk, dv;
};

bool make_maps(const Problem& p, int D, Maps* m) {
  return make_tmap_4d(&m->q, p.q, D, p.Lq, p.Hq, p.B, p.lq, kRows) &&
         make_tmap_4d(&m->dq, p.dq, D, p.Lq, p.Hq, p.B, p.ldq, kRows) &&
         make_tmap_4d(&m->dk, p.dk, D, p.Lkv, p.Hkv, p.B, p.ldk, kRows) &&
         make_tmap_4d(&m->dv, p.dv, D, p.Lkv, p.Hkv, p.B, p.ldv, kRows) &&
         make_tmap_4d(&m->dout, p.dout, D, p.Lq, p.Hq, p.B, p.ldo, kRows) &&
         make_tmap_4d(&m->k, p.k, D, p.Lkv, p.Hkv, p.B, p.lk, kRows) &&
         make_tmap_4d(&m->v, p.v, D, p.Lkv, p.Hkv, p.B, p.lv, kRows);
}

template <typename T, int D>
cudaError_t dkdv_t(const Problem& p, cudaStream_t s) {
  Maps m;
  if (!make_maps(p, D, &m)) return cudaErrorInvalidValue;
  // A mask with one row for every query is read from global memory (no tile); any other
  // mask is staged in [128 x 128] tiles.
  const bool row_mask = p.mask && p.lm.sl == 0;
  CUtensorMap tm = m.k;  // unused without a staged mask
  if (p.mask && !row_mask && !make_tmap_mask(&tm, p, p.mask_kind == kMaskBool ? 1 : 2, kRows, kBlk, false))
    return cudaErrorInvalidValue;
  const int smem = row_mask ? KvSmem<D, true, true>::kBytes
                   : p.mask ? KvSmem<D, true>::kBytes
                            : KvSmem<D, false>::kBytes;
  auto kern = row_mask ? tc_dkdv_kernel<T, D, true, true>
              : p.mask ? tc_dkdv_kernel<T, D, true, false>
                       : tc_dkdv_kernel<T, D, false, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const unsigned nkt = (p.Lkv + kRows - 1) / kRows;
  kern<<<nkt * p.Hkv * p.B, kKvThreads, smem, s>>>(m.q, m.k, m.v, m.dout, m.dk, m.dv, tm, p);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t dq_t(const Problem& p, cudaStream_t s) {
  Maps m;
  if (!make_maps(p, D, &m)) return cudaErrorInvalidValue;
  const int smem = DqLayout<D>::kBytes + 1024;
  auto kern = p.mask ? tc_dq_kernel<T, D, true> : tc_dq_kernel<T, D, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const unsigned nqt = (p.Lq + kRows - 1) / kRows;
  kern<<<nqt * p.Hq * p.B, kDqThreads, smem, s>>>(m.q, m.k, m.v, m.dout, m.dq, p);
  return cudaGetLastError();
}

}  // namespace

// D = 256 has no tensor-core backward: dK and dV of 128 keys would take all 512 TMEM
// columns, and the block's own K and V plus one Q/dO stage would fill shared memory.
bool tensor_bwd_supported(const Problem& p, int dtype) { return tensor_supported(p, dtype) && p.D <= 128; }

cudaError_t launch_tc_dkdv(const Problem& p, int dtype, cudaStream_t s) {
  if (dtype == 2) {
    if (p.D == 128) return dkdv_t<__nv_bfloat16, 128>(p, s);
    if (p.D == 96) return dkdv_t<__nv_bfloat16, 96>(p, s);
    if (p.D == 32) return dkdv_t<__nv_bfloat16, 32>(p, s);
    return dkdv_t<__nv_bfloat16, 64>(p, s);
  }
  if (p.D == 128) return dkdv_t<__half, 128>(p, s);
  if (p.D == 96) return dkdv_t<__half, 96>(p, s);
  if (p.D == 32) return dkdv_t<__half, 32>(p, s);
  return dkdv_t<__half, 64>(p, s);
}

cudaError_t launch_tc_dq(const Problem& p, int dtype, cudaStream_t s) {
  if (dtype == 2) {
    if (p.D == 128) return dq_t<__nv_bfloat16, 128>(p, s);
    if (p.D == 96) return dq_t<__nv_bfloat16, 96>(p, s);
    if (p.D == 32) return dq_t<__nv_bfloat16, 32>(p, s);
    return dq_t<__nv_bfloat16, 64>(p, s);
  }
  if (p.D == 128) return dq_t<__half, 128>(p, s);
  if (p.D == 96) return dq_t<__half, 96>(p, s);
  if (p.D == 32) return dq_t<__half, 32>(p, s);
  return dq_t<__half, 64>(p, s);
}

}  // namespace sdpa
