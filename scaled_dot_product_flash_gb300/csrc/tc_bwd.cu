// Tensor-core backward (fp16/bf16, D in {64, 128}): a dK/dV kernel and a dQ kernel, both
// TMA + tcgen05 + TMEM, recomputing P from the forward's logsumexp ("[Metal] Add Flash
// Attention VJP for training", sections "Implementation Notes" and "Limitations").
//
// dK/dV kernel: one block owns 128 rows of one KV head (KV-row ownership: every dK/dV
// row is written once by one block, so no atomics) and loops over the G query heads of
// its GQA group and their 64-row query blocks.  Per query block, with keys in TMEM lanes:
//   Sᵀ = K·Qᵀ, dPᵀ = V·dOᵀ                      (tcgen05, fp32 in TMEM)
//   Pᵀ = exp2(c·Sᵀ − log2e·lse), dSᵀ = Pᵀ∘(dPᵀ − δ)  (element warps, written back to TMEM
//                                                   as 16-bit A operands)
//   dV += Pᵀ·dO, dK += dSᵀ·Q                     (tcgen05, accumulators stay in TMEM)
// and finally dK·scale and dV are rounded and stored.
//
// dQ kernel: one block owns 128 query rows of one head and loops over 64-row KV blocks:
//   S = Q·Kᵀ, dP = dO·Vᵀ, P = exp2(c·S − log2e·lse_i), dS = P∘(dP − δ_i), dQ += dS·K,
// then dQ·scale is stored.
//
// Both kernels: warps 0-3 and 4-7 are two element warpgroups that take alternate blocks
// (warpgroup w owns TMEM buffer w), warp 8 is the TMA producer, warp 9 issues the MMAs
// and owns the 512 TMEM columns.  The MMA issuer runs one block ahead, so the tensor core
// computes block n+1's scores while block n's elementwise work runs.
#include "launch.h"
#include "tc_common.cuh"

namespace sdpa {
namespace {
using namespace tc;

constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kRows = 128;  // rows owned by a block (keys for dK/dV, queries for dQ)
constexpr int kBlk = 64;    // rows of the streamed operand per iteration
constexpr int kStages = 3;  // ring depth of the streamed operand

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

// Element work of the dK/dV kernel for one key row and a 64-query block: Pᵀ and dSᵀ from
// Sᵀ and dPᵀ in TMEM, written back as packed 16-bit pairs over the first 32 columns of
// each (columns already read).  Per pair of queries: one packed FMA, two exponentials, one
// packed add and one packed multiply, two conversions.
template <typename T, bool kCausalMask>
__device__ __forceinline__ void dkdv_elements(uint32_t s_addr, float c, const float* nlse2,
                                              const float* ndelta, int j, int i0) {
  const uint32_t dp_addr = s_addr + 64;
  const uint64_t cc = f2pack(c, c);
#pragma unroll 1
  for (int half = 0; half < 2; ++half) {
    uint32_t sr[32], dr[32];
    tmem_ld32(s_addr + half * 32, sr);
    tmem_ld32(dp_addr + half * 32, dr);
    tmem_ld_wait();
    const uint64_t* nl2 = reinterpret_cast<const uint64_t*>(nlse2 + half * 32);
    const uint64_t* nd2 = reinterpret_cast<const uint64_t*>(ndelta + half * 32);
    uint32_t pk[16], dk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      float p0, p1;
      f2unpack(ffma2(f2pack(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1])), cc, nl2[e]), p0, p1);
      p0 = ex2(p0);
      p1 = ex2(p1);
      if constexpr (kCausalMask) {
        const int q0 = i0 + half * 32 + 2 * e;
        if (j > q0) p0 = 0.f;
        if (j > q0 + 1) p1 = 0.f;
      }
      const uint64_t pp = f2pack(p0, p1);
      const uint64_t t = fadd2(f2pack(__uint_as_float(dr[2 * e]), __uint_as_float(dr[2 * e + 1])), nd2[e]);
      float d0, d1;
      f2unpack(fmul2(pp, t), d0, d1);
      pk[e] = pack2<T>(p0, p1);
      dk[e] = pack2<T>(d0, d1);
    }
    tmem_st16(s_addr + half * 16, pk);
    tmem_st16(dp_addr + half * 16, dk);
  }
}

// Element work of the dQ kernel for one query row and a 64-key block: dS = P∘(dP − δ) with
// P = exp2(c·S − log2e·lse), packed into the first 32 columns of S (all of S read first).
template <typename T, bool kMask>
__device__ __forceinline__ void dq_elements(uint32_t s_addr, float c, float nlse2, float ndl, int k0,
                                            int i, const Problem& p) {
  const uint32_t dp_addr = s_addr + 64;
  const uint64_t cc = f2pack(c, c), nl = f2pack(nlse2, nlse2), nd = f2pack(ndl, ndl);
  uint32_t dsk[32];
#pragma unroll 1
  for (int half = 0; half < 2; ++half) {
    uint32_t sr[32], dr[32];
    tmem_ld32(s_addr + half * 32, sr);
    tmem_ld32(dp_addr + half * 32, dr);
    tmem_ld_wait();
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      float p0, p1;
      f2unpack(ffma2(f2pack(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1])), cc, nl), p0, p1);
      p0 = ex2(p0);
      p1 = ex2(p1);
      if constexpr (kMask) {
        const int key = k0 + half * 32 + 2 * e;
        if (key >= p.Lkv || (p.causal && key > i)) p0 = 0.f;
        if (key + 1 >= p.Lkv || (p.causal && key + 1 > i)) p1 = 0.f;
      }
      const uint64_t t = fadd2(f2pack(__uint_as_float(dr[2 * e]), __uint_as_float(dr[2 * e + 1])), nd);
      float d0, d1;
      f2unpack(fmul2(f2pack(p0, p1), t), d0, d1);
      const uint32_t v = pack2<T>(d0, d1);
      if (half == 0) dsk[e] = v;
      else dsk[16 + e] = v;
    }
  }
  tmem_st32(s_addr, dsk);
}

// Shared-memory plan (offsets from a 1024-byte aligned base).
template <int D>
struct BwdLayout {
  static constexpr int kOwnBytes = kRows * D * 2;     // one owned [128 x D] tile
  static constexpr int kBlkBytes = kBlk * D * 2;      // one streamed [64 x D] tile
  static constexpr int kOwnA = 0;                     // K (dK/dV) or Q (dQ)
  static constexpr int kOwnB = kOwnBytes;             // V (dK/dV) or dO (dQ)
  static constexpr int kRing = 2 * kOwnBytes;         // stages of {A block, B block}
  static constexpr int kStageBytes = 2 * kBlkBytes;
  static constexpr int kBytes = kRing + kStages * kStageBytes;
  // TMEM columns
  static constexpr int kAcc0 = 0;        // dV (dK/dV kernel) or dQ (dQ kernel)
  static constexpr int kAcc1 = D;        // dK (dK/dV kernel)
  static constexpr int kBuf = 2 * D;     // two buffers of {S (64 cols), dP (64 cols)}
};

struct BwdBars {
  uint64_t own_full;
  uint64_t ring_full[kStages];
  uint64_t ring_empty[kStages];
  uint64_t vec_full[kStages];   // per-row vectors of the streamed block (dK/dV kernel)
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t buf_free[2];
  uint64_t acc_done;
  uint32_t tmem_base;
  int abort;
  alignas(16) float nlse2[kStages][kBlk];   // −log2e·lse per query (−inf past Lq: P = 0 there)
  alignas(16) float ndelta[kStages][kBlk];  // −δ per query
};

// ================================================================== dK / dV
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
    tc_dkdv_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                   Problem p) {
  using L = BwdLayout<D>;
  constexpr int kCB = D / 64;
  constexpr bool kBf16 = IsBf16<T>::value;
  constexpr uint32_t kIdS = idesc_f16(kRows, kBlk, kBf16, false, false);  // N = 64 queries
  constexpr uint32_t kIdAcc = idesc_f16(kRows, D, kBf16, false, true);    // N = D, B MN-major
  extern __shared__ unsigned char smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ BwdBars bars;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int b = blockIdx.z, g = blockIdx.y;
  const int j0 = blockIdx.x * kRows;  // first key of this block
  // Query blocks visited: for each of the G heads, blocks from i_begin to Lq.
  const int i_begin = p.causal ? j0 : 0;  // queries before j0 see none of these keys
  const int nqb = i_begin < p.Lq ? (p.Lq - i_begin + kBlk - 1) / kBlk : 0;
  const int total = p.G * nqb;  // iterations

  if (threadIdx.x == 0) {
    bars.abort = 0;
    mbar_init(&bars.own_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars.ring_full[s], 1);
      mbar_init(&bars.ring_empty[s], 1);
      mbar_init(&bars.vec_full[s], 32);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(&bars.s_full[w], 1);
      mbar_init(&bars.p_full[w], 128);
      mbar_init(&bars.buf_free[w], 1);
    }
    mbar_init(&bars.acc_done, 1);
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
  const WaitCtx wc{&bars.abort, 0, p.wait_limit_ns, p.err, kKidTcDkdv};

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tdo);
      mbar_arrive_expect_tx(&bars.own_full, 2 * L::kOwnBytes);
      for (int cb = 0; cb < kCB; ++cb) {
        tma_load_3d(sm + L::kOwnA + cb * (kRows * 128), &tk, &bars.own_full, cb * 64, j0, b * p.Hkv + g);
        tma_load_3d(sm + L::kOwnB + cb * (kRows * 128), &tv, &bars.own_full, cb * 64, j0, b * p.Hkv + g);
      }
    }
    int issued = 0;
    bool ok = true;
    for (int n = 0; ok && n < total; ++n) {
      const int s = n % kStages;
      const uint32_t ph = (n / kStages) & 1;
      ok = mbar_wait(&bars.ring_empty[s], ph ^ 1, wc);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const int h = g * p.G + n / nqb;
      const int i0 = i_begin + (n % nqb) * kBlk;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars.ring_full[s], 2 * L::kBlkBytes);
        uint8_t* st = sm + L::kRing + s * L::kStageBytes;
        for (int cb = 0; cb < kCB; ++cb) {
          tma_load_3d(st + cb * (kBlk * 128), &tq, &bars.ring_full[s], cb * 64, i0, b * p.Hq + h);
          tma_load_3d(st + L::kBlkBytes + cb * (kBlk * 128), &tdo, &bars.ring_full[s], cb * 64, i0,
                      b * p.Hq + h);
        }
      }
      // Per-query vectors of the block, negated for the packed FMA/ADD of the element
      // warps: −log2e·lse (−inf past Lq, so P = 0 there) and −δ.
      const float* lsep = p.lse + q_row(p, b, h, 0);
      const float* dlp = p.delta + q_row(p, b, h, 0);
#pragma unroll
      for (int e = lane; e < kBlk; e += 32) {
        const int i = i0 + e;
        bars.nlse2[s][e] = i < p.Lq ? -lsep[i] * kLog2e : -pos_inf();
        bars.ndelta[s][e] = i < p.Lq ? -dlp[i] : 0.f;
      }
      mbar_arrive(&bars.vec_full[s]);
      issued = n + 1;
    }
    if (lane == 0 && (!ok || bars.abort)) {
      for (int n = max(0, issued - kStages); n < issued; ++n)
        drain_wait(&bars.ring_full[n % kStages], (n / kStages) & 1, 100000000ull);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(&bars.own_full, 0, wc);
      tc_fence_after();
      const uint32_t k_s = smem_u32(sm + L::kOwnA), v_s = smem_u32(sm + L::kOwnB);
      // Scores of block n into buffer n % 2: Sᵀ = K·Qᵀ and dPᵀ = V·dOᵀ.
      auto issue_scores = [&](int n) -> bool {
        const int s = n % kStages, w = n % 2;
        if (!mbar_wait(&bars.ring_full[s], (n / kStages) & 1, wc)) return false;
        if (n >= 2 && !mbar_wait(&bars.buf_free[w], ((n - 2) / 2) & 1, wc)) return false;
        tc_fence_after();
        const uint32_t qs = smem_u32(sm + L::kRing + s * L::kStageBytes);
        const uint32_t dos = qs + L::kBlkBytes;
        const uint32_t s_col = tbase + L::kBuf + w * 128, dp_col = s_col + 64;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t own = (kk / 4) * (kRows * 128) + (kk % 4) * 32;
          const uint32_t blk = (kk / 4) * (kBlk * 128) + (kk % 4) * 32;
          mma_ss(s_col, sdesc_sw128(k_s + own, 16, 1024), sdesc_sw128(qs + blk, 16, 1024), kIdS, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t own = (kk / 4) * (kRows * 128) + (kk % 4) * 32;
          const uint32_t blk = (kk / 4) * (kBlk * 128) + (kk % 4) * 32;
          mma_ss(dp_col, sdesc_sw128(v_s + own, 16, 1024), sdesc_sw128(dos + blk, 16, 1024), kIdS, kk > 0);
        }
        mma_commit(&bars.s_full[w]);
        return true;
      };
      if (ok && total > 0) ok = issue_scores(0);
      for (int n = 0; ok && n < total; ++n) {
        if (n + 1 < total && !(ok = issue_scores(n + 1))) break;
        const int s = n % kStages, w = n % 2;
        if (!(ok = mbar_wait(&bars.p_full[w], (n / 2) & 1, wc))) break;
        tc_fence_after();
        const uint32_t qs = smem_u32(sm + L::kRing + s * L::kStageBytes);
        const uint32_t dos = qs + L::kBlkBytes;
        const uint32_t p_col = tbase + L::kBuf + w * 128, ds_col = p_col + 64;
        // dV += Pᵀ·dO and dK += dSᵀ·Q: K = 64 queries, B operands MN-major [64 x D].
#pragma unroll
        for (int kk = 0; kk < kBlk / 16; ++kk) {
          const uint32_t acc = (n > 0 || kk > 0) ? 1u : 0u;
          mma_ts(tbase + L::kAcc0, p_col + kk * 8, sdesc_sw128(dos + kk * 2048, kBlk * 128, 1024), kIdAcc, acc);
          mma_ts(tbase + L::kAcc1, ds_col + kk * 8, sdesc_sw128(qs + kk * 2048, kBlk * 128, 1024), kIdAcc, acc);
        }
        mma_commit(&bars.buf_free[w]);
        mma_commit(&bars.ring_empty[s]);
      }
      mma_commit(&bars.acc_done);
      drain_wait(&bars.acc_done, 0, 100000000ull);
    }
  } else {
    // ---------------------------------------------------------------- element warps
    const int w = warp / 4, quarter = warp % 4;
    const int r = quarter * 32 + lane;
    const int j = j0 + r;  // this thread's key
    const float c = p.scale_log2;
    bool ok = true;
    for (int n = w; n < total; n += 2) {
      const int s = n % kStages;
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.s_full[w], (n / 2) & 1, wc) &&
                                       mbar_wait(&bars.vec_full[s], (n / kStages) & 1, wc));
      if (!ok) break;
      tc_fence_after();
      const int i0 = i_begin + (n % nqb) * kBlk;
      const bool diag = p.causal && j0 + kRows - 1 > i0;  // some key of this block is after some query
      const uint32_t s_addr = tmem_addr(tbase, quarter * 32, L::kBuf + w * 128);
      if (diag)
        dkdv_elements<T, true>(s_addr, c, bars.nlse2[s], bars.ndelta[s], j, i0);
      else
        dkdv_elements<T, false>(s_addr, c, bars.nlse2[s], bars.ndelta[s], j, i0);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars.p_full[w]);
    }
    // Epilogue: warpgroup 0 writes dV, warpgroup 1 writes dK·scale.
    if (ok) ok = __all_sync(0xffffffffu, total == 0 || mbar_wait(&bars.acc_done, 0, wc));
    if (ok) {
      tc_fence_after();
      const bool valid = j < p.Lkv;
      T* dst = static_cast<T*>(w == 0 ? p.dv : p.dk) + kv_row(p, b, g, valid ? j : 0) * D;
      const float mul = w == 0 ? 1.f : p.scale;
      const uint32_t a_addr = tmem_addr(tbase, quarter * 32, w == 0 ? L::kAcc0 : L::kAcc1);
#pragma unroll
      for (int c32 = 0; c32 < D / 32; ++c32) {
        uint32_t acc[32];
        if (total > 0) {
          tmem_ld32(a_addr + c32 * 32, acc);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) acc[e] = 0u;  // no query sees these keys
        }
        uint32_t packed[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          packed[e] = pack2<T>(__uint_as_float(acc[2 * e]) * mul, __uint_as_float(acc[2 * e + 1]) * mul);
        if (valid) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c32 * 32);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            d4[v4] = make_uint4(packed[4 * v4], packed[4 * v4 + 1], packed[4 * v4 + 2], packed[4 * v4 + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tmem_dealloc(tbase, 512);
  }
}

// ================================================================== dQ
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
    tc_dq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                 Problem p) {
  using L = BwdLayout<D>;
  constexpr int kCB = D / 64;
  constexpr bool kBf16 = IsBf16<T>::value;
  constexpr uint32_t kIdS = idesc_f16(kRows, kBlk, kBf16, false, false);  // N = 64 keys
  constexpr uint32_t kIdAcc = idesc_f16(kRows, D, kBf16, false, true);    // N = D, B MN-major
  extern __shared__ unsigned char smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ BwdBars bars;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int b = blockIdx.z, h = blockIdx.y, g = h / p.G;
  const int qt = p.causal ? (int)(gridDim.x - 1 - blockIdx.x) : (int)blockIdx.x;  // heavy first
  const int i0 = qt * kRows;
  const int kend = p.causal ? min(p.Lkv, min(p.Lq, i0 + kRows)) : p.Lkv;
  const int total = (kend + kBlk - 1) / kBlk;  // KV blocks visited

  if (threadIdx.x == 0) {
    bars.abort = 0;
    mbar_init(&bars.own_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars.ring_full[s], 1);
      mbar_init(&bars.ring_empty[s], 1);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(&bars.s_full[w], 1);
      mbar_init(&bars.p_full[w], 128);
      mbar_init(&bars.buf_free[w], 1);
    }
    mbar_init(&bars.acc_done, 1);
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

  if (warp == kProducerWarp) {
    if (lane == 0) {
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      mbar_arrive_expect_tx(&bars.own_full, 2 * L::kOwnBytes);
      for (int cb = 0; cb < kCB; ++cb) {
        tma_load_3d(sm + L::kOwnA + cb * (kRows * 128), &tq, &bars.own_full, cb * 64, i0, b * p.Hq + h);
        tma_load_3d(sm + L::kOwnB + cb * (kRows * 128), &tdo, &bars.own_full, cb * 64, i0, b * p.Hq + h);
      }
      int issued = 0;
      bool ok = true;
      for (int n = 0; ok && n < total; ++n) {
        const int s = n % kStages;
        if (!(ok = mbar_wait(&bars.ring_empty[s], ((n / kStages) & 1) ^ 1, wc))) break;
        mbar_arrive_expect_tx(&bars.ring_full[s], 2 * L::kBlkBytes);
        uint8_t* st = sm + L::kRing + s * L::kStageBytes;
        for (int cb = 0; cb < kCB; ++cb) {
          tma_load_3d(st + cb * (kBlk * 128), &tk, &bars.ring_full[s], cb * 64, n * kBlk, b * p.Hkv + g);
          tma_load_3d(st + L::kBlkBytes + cb * (kBlk * 128), &tv, &bars.ring_full[s], cb * 64, n * kBlk,
                      b * p.Hkv + g);
        }
        issued = n + 1;
      }
      if (!ok || bars.abort) {
        for (int n = max(0, issued - kStages); n < issued; ++n)
          drain_wait(&bars.ring_full[n % kStages], (n / kStages) & 1, 100000000ull);
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      bool ok = mbar_wait(&bars.own_full, 0, wc);
      tc_fence_after();
      const uint32_t q_s = smem_u32(sm + L::kOwnA), do_s = smem_u32(sm + L::kOwnB);
      auto issue_scores = [&](int n) -> bool {
        const int s = n % kStages, w = n % 2;
        if (!mbar_wait(&bars.ring_full[s], (n / kStages) & 1, wc)) return false;
        if (n >= 2 && !mbar_wait(&bars.buf_free[w], ((n - 2) / 2) & 1, wc)) return false;
        tc_fence_after();
        const uint32_t ks = smem_u32(sm + L::kRing + s * L::kStageBytes);
        const uint32_t vs = ks + L::kBlkBytes;
        const uint32_t s_col = tbase + L::kBuf + w * 128, dp_col = s_col + 64;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t own = (kk / 4) * (kRows * 128) + (kk % 4) * 32;
          const uint32_t blk = (kk / 4) * (kBlk * 128) + (kk % 4) * 32;
          mma_ss(s_col, sdesc_sw128(q_s + own, 16, 1024), sdesc_sw128(ks + blk, 16, 1024), kIdS, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t own = (kk / 4) * (kRows * 128) + (kk % 4) * 32;
          const uint32_t blk = (kk / 4) * (kBlk * 128) + (kk % 4) * 32;
          mma_ss(dp_col, sdesc_sw128(do_s + own, 16, 1024), sdesc_sw128(vs + blk, 16, 1024), kIdS, kk > 0);
        }
        mma_commit(&bars.s_full[w]);
        return true;
      };
      if (ok && total > 0) ok = issue_scores(0);
      for (int n = 0; ok && n < total; ++n) {
        if (n + 1 < total && !(ok = issue_scores(n + 1))) break;
        const int s = n % kStages, w = n % 2;
        if (!(ok = mbar_wait(&bars.p_full[w], (n / 2) & 1, wc))) break;
        tc_fence_after();
        const uint32_t ks = smem_u32(sm + L::kRing + s * L::kStageBytes);
        const uint32_t ds_col = tbase + L::kBuf + w * 128;
        // dQ += dS·K: K = 64 keys, B = K block MN-major [64 x D].
#pragma unroll
        for (int kk = 0; kk < kBlk / 16; ++kk)
          mma_ts(tbase + L::kAcc0, ds_col + kk * 8, sdesc_sw128(ks + kk * 2048, kBlk * 128, 1024), kIdAcc,
                 (n > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars.buf_free[w]);
        mma_commit(&bars.ring_empty[s]);
      }
      mma_commit(&bars.acc_done);
      drain_wait(&bars.acc_done, 0, 100000000ull);
    }
  } else {
    const int w = warp / 4, quarter = warp % 4;
    const int r = quarter * 32 + lane;
    const int i = i0 + r;  // this thread's query
    const bool valid = i < p.Lq;
    const int64_t row = q_row(p, b, h, valid ? i : 0);
    const float lse2 = valid ? p.lse[row] * kLog2e : pos_inf();
    const float dl = valid ? p.delta[row] : 0.f;
    const float c = p.scale_log2;
    bool ok = true;
    for (int n = w; n < total; n += 2) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.s_full[w], (n / 2) & 1, wc));
      if (!ok) break;
      tc_fence_after();
      const int k0 = n * kBlk;
      const bool need_mask = (k0 + kBlk > p.Lkv) || (p.causal && k0 + kBlk - 1 > i0);
      const uint32_t s_addr = tmem_addr(tbase, quarter * 32, L::kBuf + w * 128);
      if (need_mask)
        dq_elements<T, true>(s_addr, c, -lse2, -dl, k0, i, p);
      else
        dq_elements<T, false>(s_addr, c, -lse2, -dl, k0, i, p);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars.p_full[w]);
    }
    if (ok) ok = __all_sync(0xffffffffu, total == 0 || mbar_wait(&bars.acc_done, 0, wc));
    if (ok && w == 0) {
      tc_fence_after();
      T* dst = static_cast<T*>(p.dq) + row * D;
      const uint32_t a_addr = tmem_addr(tbase, quarter * 32, L::kAcc0);
#pragma unroll
      for (int c32 = 0; c32 < D / 32; ++c32) {
        uint32_t acc[32];
        if (total > 0) {
          tmem_ld32(a_addr + c32 * 32, acc);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) acc[e] = 0u;
        }
        uint32_t packed[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          packed[e] = pack2<T>(__uint_as_float(acc[2 * e]) * p.scale, __uint_as_float(acc[2 * e + 1]) * p.scale);
        if (valid) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c32 * 32);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            d4[v4] = make_uint4(packed[4 * v4], packed[4 * v4 + 1], packed[4 * v4 + 2], packed[4 * v4 + 3]);
        }
      }
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
  CUtensorMap q, k, v, dout;
};

bool make_maps(const Problem& p, int D, int q_box, int kv_box, Maps* m) {
  return make_tmap_3d(&m->q, p.q, D, p.Lq, p.B * p.Hq, q_box) &&
         make_tmap_3d(&m->dout, p.dout, D, p.Lq, p.B * p.Hq, q_box) &&
         make_tmap_3d(&m->k, p.k, D, p.Lkv, p.B * p.Hkv, kv_box) &&
         make_tmap_3d(&m->v, p.v, D, p.Lkv, p.B * p.Hkv, kv_box);
}

template <typename T, int D>
cudaError_t dkdv_t(const Problem& p, cudaStream_t s) {
  Maps m;
  if (!make_maps(p, D, kBlk, kRows, &m)) return cudaErrorInvalidValue;
  const int smem = BwdLayout<D>::kBytes + 1024;
  auto kern = tc_dkdv_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((p.Lkv + kRows - 1) / kRows, p.Hkv, p.B);
  kern<<<grid, kThreads, smem, s>>>(m.q, m.k, m.v, m.dout, p);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t dq_t(const Problem& p, cudaStream_t s) {
  Maps m;
  if (!make_maps(p, D, kRows, kBlk, &m)) return cudaErrorInvalidValue;
  const int smem = BwdLayout<D>::kBytes + 1024;
  auto kern = tc_dq_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((p.Lq + kRows - 1) / kRows, p.Hq, p.B);
  kern<<<grid, kThreads, smem, s>>>(m.q, m.k, m.v, m.dout, p);
  return cudaGetLastError();
}

}  // namespace

bool tensor_bwd_supported(const Problem& p, int dtype) { return tensor_supported(p, dtype); }

cudaError_t launch_tc_dkdv(const Problem& p, int dtype, cudaStream_t s) {
  if (dtype == 2) return p.D == 128 ? dkdv_t<__nv_bfloat16, 128>(p, s) : dkdv_t<__nv_bfloat16, 64>(p, s);
  return p.D == 128 ? dkdv_t<__half, 128>(p, s) : dkdv_t<__half, 64>(p, s);
}

cudaError_t launch_tc_dq(const Problem& p, int dtype, cudaStream_t s) {
  if (dtype == 2) return p.D == 128 ? dq_t<__nv_bfloat16, 128>(p, s) : dq_t<__nv_bfloat16, 64>(p, s);
  return p.D == 128 ? dq_t<__half, 128>(p, s) : dq_t<__half, 64>(p, s);
}

}  // namespace sdpa
