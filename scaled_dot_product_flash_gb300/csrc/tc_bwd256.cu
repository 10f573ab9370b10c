// Tensor-core backward at head dim 256 (fp16/bf16): a dQ kernel and a
// dK/dV kernel on TMA + tcgen05 + TMEM, recomputing P from the forward's logsumexp as the
// D <= 128 kernels do ("[Metal] Add Flash Attention VJP for training", sections
// "Implementation Notes" and "Limitations").  At D = 256 one SM's budgets (512 TMEM
// columns, 227 KB of shared memory) shape them differently:
//   dQ: a block owns 128 query rows of one head and streams 64-key blocks.  TMEM: dQ in
//       256 columns, Q in 128 (the A operand of S = Q·Kᵀ) and two 64-column buffers that
//       take S, then dP = dO·Vᵀ over it, then dS over that.  Shared memory: dO (64 KB),
//       three K stages and two V stages (32 KB each).  S and dP are M = 128, N = 64
//       products over 16 K-steps; dQ += dS·K is one M = 128, N = 256 product over 4.
//   dK/dV: a block owns 128 keys of one KV head and streams 64-row query blocks of the G
//       query heads of its group; one block of a neighbouring pair accumulates dK, the
//       other dV, each over the full D in 256 TMEM columns.  Both compute Sᵀ = K·Qᵀ; the dK
//       block also dPᵀ = V·dOᵀ (2.5F of MMA work in all against 3F for a split of D).
// Warp roles as in the D <= 128 kernels: warps 0-15 element work, warp 16 the TMA
// producer, warps 17-19 the MMA issuers; warp 17 owns the TMEM.  The element warps form two
// groups of 8 that take the even and the odd streamed blocks (TMEM buffer n % 2); warp e of
// a group takes TMEM lane quarter e % 4 and 32 streamed columns, and packs its 16-bit
// results over the first 8 of each 16.  Every wait is bounded, as everywhere in the library.
// Attention masks: each kernel has a masked instantiation (kMasked) that adds log2e·M to
// the log2-domain scores before the exponential, as the D <= 128 kernels do.  The dQ
// kernel has no shared memory left for a mask tile and reads its row's 32 mask values
// from global memory in 16-byte pieces before its barrier wait; the dK/dV kernel reads a
// mask with one row for every query once per key from global memory and stages any other
// mask's [64 x 128] tiles by TMA in the place of its third Q slot.
#include "launch.h"
#include "tc_common.cuh"

namespace sdpa {
namespace {
using namespace tc;

constexpr int kD = 256;
constexpr int kOwn = 128;                   // rows owned by a block
constexpr int kStr = 64;                    // rows of a streamed block
constexpr int kOwnBytes = kOwn * kD * 2;    // [128 x 256] 16-bit: 64 KB
constexpr int kOwnCb = kOwn * 128;          // one 64-column block of an own tile
constexpr int kStrBytes = kStr * kD * 2;    // [64 x 256] 16-bit: 32 KB
constexpr int kStrCb = kStr * 128;          // one 64-column block of a streamed tile
constexpr int kProducer = 16;
constexpr int kIssuer = 17;
// Both kernels: launched at 96 registers a thread (65,536 / 640 rounded down to a multiple
// of 8); warpgroup 4 (producer and issuers) drops to 56 and the element warpgroups rise to
// 104.
constexpr int kDqThreads = 640;
constexpr int kRegsLow = 56;
constexpr int kRegsHigh = 104;
static_assert(128 * kRegsLow + 512 * kRegsHigh <= kDqThreads * 96, "register split exceeds the launch");

template <typename T>
struct IsBf16 { static constexpr bool value = false; };
template <>
struct IsBf16<__nv_bfloat16> { static constexpr bool value = true; };

__device__ __forceinline__ float pos_inf() { return __int_as_float(0x7f800000); }

// Thread-block cluster helpers: rank of this block in its cluster, a barrier over every
// thread of the cluster (release / acquire at cluster scope), the address of a shared-memory
// location in the block of another rank, and a 16-byte store there.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > 100000000ull) return;
  }
}

// S (or Sᵀ) = A·Bᵀ over D = 256: A an own [128 x 256] tile and B a streamed [64 x 256]
// tile, both K-major in the 128-byte swizzle as four 64-column blocks; M = 128, N = 64,
// 16 K-steps.  Called by all 32 lanes of the issuing warp; one elected lane issues.
__device__ __forceinline__ void mma_scores256(uint32_t c_tmem, uint32_t a_s, uint32_t b_s, uint32_t idesc) {
  const uint64_t ad = sdesc_sw128(a_s, 16, 1024), bd = sdesc_sw128(b_s, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < kD / 16; ++kk) {
    const uint32_t ka = (kk / 4) * kOwnCb + (kk % 4) * 32, kb = (kk / 4) * kStrCb + (kk % 4) * 32;
    mma_ss_w(c_tmem, sdesc_advance(ad, ka), sdesc_advance(bd, kb), idesc, kk > 0);
  }
}

// The same product with A = the own tile held in TMEM (row r in lane r, elements (2i, 2i+1)
// of D in column a_tmem + i): only B is read from shared memory.
__device__ __forceinline__ void mma_scores256_ts(uint32_t c_tmem, uint32_t a_tmem, uint32_t b_s, uint32_t idesc) {
  const uint64_t bd = sdesc_sw128(b_s, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < kD / 16; ++kk)
    mma_ts_w(c_tmem, a_tmem + 8 * kk, sdesc_advance(bd, (kk / 4) * kStrCb + (kk % 4) * 32), idesc, kk > 0);
}

// Acc (+)= A·B: A the packed 16-bit [128 x 64] in TMEM (K-step kk, rows [16kk, 16kk + 16)
// of the streamed block, in columns [a_tmem + 16kk, a_tmem + 16kk + 8)) and B the columns
// of a streamed [64 x 256] tile from b_s on (as many 64-column blocks as the instruction's
// N), read MN-major with K = its 64 rows.
__device__ __forceinline__ void mma_acc256(uint32_t acc_tmem, uint32_t a_tmem, uint32_t b_s, uint32_t idesc,
                                           bool first) {
  const uint64_t bd = sdesc_sw128(b_s, kStrCb, 1024);
#pragma unroll
  for (int kk = 0; kk < kStr / 16; ++kk)
    mma_ts_w(acc_tmem, a_tmem + 16 * kk, sdesc_advance(bd, kk * 2048), idesc, (!first || kk > 0) ? 1u : 0u);
}

// ================================================================== dQ
// Shared memory: dO (64 KB, read by every dP), three K stages (K(n) is read by S(n) and by
// dQ += dS(n)·K(n), late in the iteration) and two V stages, 32 KB each (224 KB).  Q is
// loaded once into the V stages and copied into TMEM, where S = Q·Kᵀ reads it as the A
// operand; the V stages are filled only after the copy.
constexpr int kDqDo = 0;
constexpr int kDqK = kOwnBytes;                 // three K stages
constexpr int kDqV = kDqK + 3 * kStrBytes;      // two V stages (first holding Q)
constexpr int kDqBytes = kDqV + 2 * kStrBytes;  // 224 KB

struct Dq256Bars {
  uint64_t own_full;      // Q and dO
  uint64_t k_full[3];
  uint64_t k_empty[3];    // dQ(n) has read K stage n % 3
  uint64_t v_full[2];
  uint64_t v_empty[2];    // dP(n) has read V stage n % 2
  uint64_t opnd_ready;    // Q is in TMEM (512 element threads): the V stages are free
  uint64_t s_full[2];     // S(n) in buffer n % 2
  uint64_t s_read[2];     // every thread of the buffer's element group has read S(n)
  uint64_t dp_full[2];    // dP(n) over S(n) in buffer n % 2
  uint64_t ds_ready[2];   // dS(n) packed in buffer n % 2
  uint64_t dq_done[2];    // dQ(n) has read buffer n % 2
  uint64_t acc_done;
  uint32_t tmem_base;
  int abort;
};

template <typename T, bool kMasked>
__global__ void __launch_bounds__(kDqThreads, 1)
    tc_dq256_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                    const __grid_constant__ CUtensorMap tdq, Problem p) {
  constexpr bool kBf16 = IsBf16<T>::value;
  constexpr uint32_t kIdS = idesc_f16(kOwn, kStr, kBf16, false, false);  // M = 128, N = 64
  constexpr uint32_t kIdAcc = idesc_f16(kOwn, kD, kBf16, false, true);   // M = 128, N = 256, B MN-major
  // TMEM columns: dQ [0, 256), two buffers [256, 384) that take S(n), then dP(n) over it
  // once the element group has read S(n), then dS(n) over that; Q [384, 512).
  constexpr uint32_t kColDq = 0, kColX = 256, kColQ = 384;
  extern __shared__ unsigned char smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Dq256Bars bars;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // Block order: all heads of one query tile, then the next; causal: heaviest tiles first.
  const int units = p.B * p.Hq;
  const int unit = blockIdx.x % units, rank = blockIdx.x / units;
  const int b = unit / p.Hq, h = unit % p.Hq, g = h / p.G;
  const int nqt = (p.Lq + kOwn - 1) / kOwn;
  const int i0 = (p.causal ? nqt - 1 - rank : rank) * kOwn;
  const int kend = p.causal ? min(p.Lkv, min(p.Lq, i0 + kOwn) + p.coff) : p.Lkv;
  const int total = (kend + kStr - 1) / kStr;  // key blocks visited

  if (threadIdx.x == 0) {
    bars.abort = 0;
    mbar_init(&bars.own_full, 1);
    for (int s = 0; s < 3; ++s) {
      mbar_init(&bars.k_full[s], 1);
      mbar_init(&bars.k_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.v_full[s], 1);
      mbar_init(&bars.v_empty[s], 1);
      mbar_init(&bars.s_full[s], 1);
      mbar_init(&bars.s_read[s], 256);  // the element group of buffer s (8 warps)
      mbar_init(&bars.dp_full[s], 1);
      mbar_init(&bars.ds_ready[s], 256);
      mbar_init(&bars.dq_done[s], 1);
    }
    mbar_init(&bars.opnd_ready, 512);
    mbar_init(&bars.acc_done, 3);  // one commit per MMA issuer
    fence_mbar_init();
  }
  if (warp == kIssuer) {
    tmem_alloc(&bars.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars.tmem_base;
  const WaitCtx wc{&bars.abort, 0, p.wait_limit_ns, p.err, kKidTcDq};
  if (warp >= 16) regs_dec<kRegsLow>();

  if (warp == kProducer) {
    // Q (into the V stages) and dO once; then K(n) into stage n % 3 once dQ(n-3) has read
    // it, and V(n) into stage n % 2 once dP(n-2) has read it (the first two once Q is in
    // TMEM).
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      prefetch_tmap(&tdo);
      mbar_arrive_expect_tx(&bars.own_full, 2 * kOwnBytes);
      for (int cb = 0; cb < 4; ++cb) {
        tma_load_4d(sm + kDqV + cb * kOwnCb, &tq, &bars.own_full, cb * 64, i0, h, b);
        tma_load_4d(sm + kDqDo + cb * kOwnCb, &tdo, &bars.own_full, cb * 64, i0, h, b);
      }
      // The block one wave later (about num_sms blocks on) starts when some block ends:
      // bring its Q and dO tiles into L2 now, so that its first loads come from L2.
      if (p.num_sms > 0 && blockIdx.x + p.num_sms < gridDim.x) {
        const int nb = blockIdx.x + p.num_sms;
        const int nu = nb % units, nrank = nb / units;
        const int ni0 = (p.causal ? nqt - 1 - nrank : nrank) * kOwn;
        for (int cb = 0; cb < 4; ++cb) {
          tma_prefetch_l2_4d(&tq, cb * 64, ni0, nu % p.Hq, nu / p.Hq);
          tma_prefetch_l2_4d(&tdo, cb * 64, ni0, nu % p.Hq, nu / p.Hq);
        }
      }
      int k_issued = 0, v_issued = 0;
      bool ok = true;
      for (int n = 0; ok && n < total; ++n) {
        const int ks = n % 3, vs = n % 2;
        if (!(ok = mbar_wait(&bars.k_empty[ks], ((n / 3) & 1) ^ 1, wc))) break;
        mbar_arrive_expect_tx(&bars.k_full[ks], kStrBytes);
        for (int cb = 0; cb < 4; ++cb)
          tma_load_4d(sm + kDqK + ks * kStrBytes + cb * kStrCb, &tk, &bars.k_full[ks], cb * 64, n * kStr, g, b);
        k_issued = n + 1;
        if (!(ok = mbar_wait(&bars.v_empty[vs], ((n / 2) & 1) ^ 1, wc) &&
                   (n >= 2 || mbar_wait(&bars.opnd_ready, 0, wc))))
          break;
        mbar_arrive_expect_tx(&bars.v_full[vs], kStrBytes);
        for (int cb = 0; cb < 4; ++cb)
          tma_load_4d(sm + kDqV + vs * kStrBytes + cb * kStrCb, &tv, &bars.v_full[vs], cb * 64, n * kStr, g, b);
        v_issued = n + 1;
      }
      if (!ok || bars.abort) {  // let copies still in flight land before the block exits
        for (int n = max(0, k_issued - 3); n < k_issued; ++n) drain_wait(&bars.k_full[n % 3], (n / 3) & 1);
        for (int n = max(0, v_issued - 2); n < v_issued; ++n) drain_wait(&bars.v_full[n % 2], (n / 2) & 1);
      }
    }
  } else if (warp >= kIssuer) {
    // Warp 17: S(n) = Q·K(n)ᵀ into buffer n % 2 once dQ(n-2) has read it.
    // Warp 18: dP(n) = dO·V(n)ᵀ over S(n) once the element group has read S(n).
    // Warp 19: dQ += dS(n)·K(n) once dS(n) is packed.
    constexpr unsigned kAll = 0xffffffffu;
    const int role = __shfl_sync(kAll, warp - kIssuer, 0);
    bool ok = __all_sync(kAll, mbar_wait(&bars.own_full, 0, wc));
    if (role == 0 && ok) ok = __all_sync(kAll, mbar_wait(&bars.opnd_ready, 0, wc));
    tc_fence_after();
    const uint32_t do_s = smem_u32(sm + kDqDo);
    auto k_s = [&](int n) { return smem_u32(sm + kDqK + (n % 3) * kStrBytes); };
    auto v_s = [&](int n) { return smem_u32(sm + kDqV + (n % 2) * kStrBytes); };
    if (role == 0) {
      for (int n = 0; ok && n < total; ++n) {
        if (!(ok = __all_sync(kAll, mbar_wait(&bars.k_full[n % 3], (n / 3) & 1, wc) &&
                                        mbar_wait(&bars.dq_done[n % 2], ((n / 2) & 1) ^ 1, wc))))
          break;
        tc_fence_after();
        mma_scores256_ts(tbase + kColX + 64 * (n % 2), tbase + kColQ, k_s(n), kIdS);
        mma_commit_w(&bars.s_full[n % 2]);
      }
    } else if (role == 1) {
      for (int n = 0; ok && n < total; ++n) {
        if (!(ok = __all_sync(kAll, mbar_wait(&bars.v_full[n % 2], (n / 2) & 1, wc) &&
                                        mbar_wait(&bars.s_read[n % 2], (n / 2) & 1, wc))))
          break;
        tc_fence_after();
        mma_scores256(tbase + kColX + 64 * (n % 2), do_s, v_s(n), kIdS);
        mma_commit_w(&bars.dp_full[n % 2]);
        mma_commit_w(&bars.v_empty[n % 2]);
      }
    } else {
      for (int n = 0; ok && n < total; ++n) {
        // K(n) is loaded (S(n) read it before dS(n) could exist); waiting on its barrier too
        // makes the TMA writes visible to this warp's MMA directly.
        if (!(ok = __all_sync(kAll, mbar_wait(&bars.ds_ready[n % 2], (n / 2) & 1, wc) &&
                                        mbar_wait(&bars.k_full[n % 3], (n / 3) & 1, wc))))
          break;
        tc_fence_after();
        mma_acc256(tbase + kColDq, tbase + kColX + 64 * (n % 2), k_s(n), kIdAcc, n == 0);
        mma_commit_w(&bars.dq_done[n % 2]);
        mma_commit_w(&bars.k_empty[n % 3]);
      }
    }
    mma_commit_w(&bars.acc_done);
    drain_wait(&bars.acc_done, 0);
  } else {
    regs_inc<kRegsHigh>();
    const int c = warp / 4, quarter = warp % 4;
    const int i = i0 + quarter * 32 + lane;  // this thread's query
    const bool valid = i < p.Lq;
    const int64_t row = q_row(p, b, h, valid ? i : 0);
    const float lse = valid ? p.lse[row] : -pos_inf();
    const float lse2 = lse == -pos_inf() ? pos_inf() : lse * kLog2e;  // no visible key: P = 0
    const float dl = valid ? p.delta[row] : 0.f;
    const int64_t moff = kMasked && valid ? row_off(p.lm, b, h, i) : 0;
    const uint64_t cc = f2pack(p.scale_log2, p.scale_log2);
    const uint64_t nl = f2pack(-lse2, -lse2), nd = f2pack(-dl, -dl);
    // Q into TMEM columns [384, 512): row r in lane r, elements (2i, 2i+1) of D in column
    // 384 + i.  Warp e copies rows [32(e % 4), +32) of D columns [64c, 64c + 64); the 16-byte
    // pieces of a swizzled row hold consecutive element pairs, so they go over as they are.
    bool ok = __all_sync(0xffffffffu, mbar_wait(&bars.own_full, 0, wc));
    if (ok) {
      const uint8_t* src = sm + kDqV + c * kOwnCb;
      const int r = quarter * 32 + lane;
      uint32_t w[32];
#pragma unroll
      for (int pc = 0; pc < 8; ++pc) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + sw128_off(r, pc));
        w[4 * pc] = v.x;
        w[4 * pc + 1] = v.y;
        w[4 * pc + 2] = v.z;
        w[4 * pc + 3] = v.w;
      }
      tmem_st32(tmem_addr(tbase, quarter * 32, kColQ + 32 * c), w);
      tmem_st_wait();
      tc_fence_before();
    }
    mbar_arrive(&bars.opnd_ready);
    // The element warps form two groups of 8 that take turns: group gq = e / 8 takes the
    // key blocks n with n % 2 == gq (TMEM buffer n % 2).  Warp e of a group has lane quarter
    // e % 4 (queries) and key columns [32h, 32h + 32), h = (e / 4) % 2; it packs the 16-bit
    // dS of keys [32h, 32h + 16) over columns [32h, 32h + 8) and those of [32h + 16, 32h + 32)
    // over [32h + 16, 32h + 24), where the K-steps 2h and 2h + 1 of the dQ product read them.
    const int gq = warp / 8, h2 = (warp / 4) % 2;
    for (int n = gq; ok && n < total; n += 2) {
      const int s = n % 2;
      const int k0 = n * kStr + 32 * h2;  // first key of this warp's columns
      // Mask terms of this warp's keys as 16-bit pairs (0 past the row's mask pieces: those
      // keys are past Lkv and hidden by lim), read before the wait so that it hides the
      // loads' latency.
      uint32_t mk[kMasked ? 16 : 1];
      if constexpr (kMasked) mask_pairs<T, 32>(mk, p, moff + k0, valid && k0 < p.Lkv ? p.Lkv - k0 : 0);
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.s_full[s], (n / 2) & 1, wc));
      if (!ok) break;
      tc_fence_after();
      const bool need_mask = (k0 + 32 > p.Lkv) || (p.causal && k0 + 31 > i0 + p.coff);
      const int lim = min(p.Lkv - k0, p.causal ? i + p.coff - k0 + 1 : 32);  // keys k0 + e, e < lim
      const uint32_t x_addr = tmem_addr(tbase, quarter * 32, kColX + 64 * s + 32 * h2);
      // P of this warp's 32 keys, in fp32 pairs (one TMEM round trip for S).
      uint64_t pf[16];
      uint32_t sr[32];
      tmem_ld32(x_addr, sr);
      tmem_ld_wait(sr);
      tc_fence_before();  // dP(n) may now overwrite S(n)
      mbar_arrive(&bars.s_read[s]);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int x = 8 * hf + e;
          float p0, p1;
          uint64_t xx = ffma2(f2pack(__uint_as_float(sr[2 * x]), __uint_as_float(sr[2 * x + 1])), cc, nl);
          if constexpr (kMasked) {
            float x0, x1, m0, m1;
            f2unpack(xx, x0, x1);
            unpack2<T>(mk[x], m0, m1);
            xx = f2pack(x0 + m0 * kLog2e, x1 + m1 * kLog2e);
          }
          ex2_pair(xx, p0, p1);
          if (need_mask) {
            if (2 * x >= lim) p0 = 0.f;
            if (2 * x + 1 >= lim) p1 = 0.f;
          }
          pf[x] = f2pack(p0, p1);
        }
      }
      // dS = P∘(dP − δ) (one TMEM round trip for dP).
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.dp_full[s], (n / 2) & 1, wc));
      if (!ok) break;
      tc_fence_after();
      uint32_t dr[32];
      tmem_ld32(x_addr, dr);
      tmem_ld_wait(dr);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t pk[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int x = 8 * hf + e;
          float d0, d1;
          f2unpack(fmul2(pf[x], fadd2(f2pack(__uint_as_float(dr[2 * x]), __uint_as_float(dr[2 * x + 1])), nd)), d0, d1);
          pk[e] = pack2<T>(d0, d1);
        }
        tmem_st8(x_addr + 16 * hf, pk);  // dS over the first 8 of each 16 columns
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars.ds_ready[s]);
    }
    // Epilogue: dQ·scale in 8 chunks of 32 columns (warps of group c take chunks c and
    // c + 4), staged in the dO buffer (the last dP product has read it) and written by bulk
    // tensor stores once all 16 warps have staged theirs (rows past Lq are clipped).
    if (ok) ok = __all_sync(0xffffffffu, total == 0 || mbar_wait(&bars.acc_done, 0, wc));
    const int r = quarter * 32 + lane;
    if (ok) {
      tc_fence_after();
#pragma unroll 1
      for (int c32 = c; c32 < kD / 32; c32 += 4) {
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
        uint8_t* blk = sm + kDqDo + (c32 / 2) * kOwnCb;
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4)
          *reinterpret_cast<uint4*>(blk + sw128_off(r, (c32 % 2) * 4 + v4)) =
              make_uint4(packed[4 * v4], packed[4 * v4 + 1], packed[4 * v4 + 2], packed[4 * v4 + 3]);
      }
      fence_async_smem();
    }
    if (named_sync_and(1, 512, ok) && warp == 0 && lane == 0) {
      for (int cb = 0; cb < 4; ++cb) tma_store_4d(&tdq, sm + kDqDo + cb * kOwnCb, cb * 64, i0, h, b);
      bulk_commit();
      bulk_wait_read();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kIssuer) {
    __syncwarp();
    tmem_dealloc(tbase, 512);
  }
}

// ================================================================== dK / dV
// Two kinds of block: a dK block computes Sᵀ = K·Qᵀ, dPᵀ = V·dOᵀ and dK += dSᵀ·Q; a dV
// block computes Sᵀ and dV += Pᵀ·dO.  Each accumulates its gradient over the full D in 256
// TMEM columns; Sᵀ is computed by both (2.5F of MMA work in all where a split of D into
// halves would take 3F).  Each block copies one owned tile into TMEM columns [384, 512)
// (the dV block K, the dK block V) and runs that score product with A from TMEM.  Each
// runs as a cluster of two blocks that take the first and the second half of the query
// blocks: the heaviest causal key tile (every query of every head of the group) would
// otherwise set the kernel's time alone.  At the end the second block writes its fp32
// partial sum into the first block's shared memory, which adds it to its own and stores
// the result.
//   dK block: TMEM dK [0, 256), two 64-column buffers [256, 384) that take Sᵀ(n), then
//     dPᵀ(n) over it once the buffer's element group has read Sᵀ(n) (Pᵀ stays in
//     registers), then dSᵀ(n) over that; V [384, 512).  Shared memory: K, two dO slots in
//     the place of V once V is in TMEM, three Q slots (Q(n) is read until dK(n), late in
//     the iteration; two when mask tiles are staged).  Warp 17 issues Sᵀ(n) into buffer
//     n % 2 once dK(n-2) has read it, warp 18 dPᵀ(n), warp 19 dK += dSᵀ(n)·Q(n).
//   dV block: TMEM dV [0, 256), Sᵀ → Pᵀ in the two buffers [256, 384), K [384, 512).  Shared
//     memory: K (read once, into TMEM), two dO slots, three (or two) Q slots.  Warp 17
//     issues Sᵀ(n) into buffer n % 2 once dV(n-2) has read it, warp 18 dV += Pᵀ(n)·dO(n);
//     warp 19 has nothing to issue.
// The rings let a load be issued about two iterations before its data is needed: a TMA
// load of a 32 KB tile took 750-2000 cycles to land under this kernel's load.
struct Kv256Bars {
  uint64_t own_full;
  uint64_t q_full[3];
  uint64_t q_empty[3];    // the last MMA reading Q slot i has finished
  uint64_t do_full[2];
  uint64_t do_empty[2];   // the MMA reading dO slot i has finished
  uint64_t vec_full[2];   // per-query vectors of slot i written (32 producer lanes)
  uint64_t vec_empty[2];  // the element group of slot i is done with them
  uint64_t s_full[2];     // Sᵀ in buffer i
  uint64_t s_read[2];     // dK blocks: the element group of buffer i has read Sᵀ
  uint64_t p_ready[2];    // dV blocks: Pᵀ packed in buffer i
  uint64_t x_free[2];     // dV blocks: dV has read buffer i
  uint64_t dp_full[2];    // dK blocks: dPᵀ in buffer i
  uint64_t ds_ready[2];   // dK blocks: dSᵀ packed in buffer i
  uint64_t y_free[2];     // dK blocks: dK has read buffer i
  uint64_t opnd_ready;    // the TMEM copy of the owned operand is complete (512 threads)
  uint64_t mask_full[2];  // staged-mask variant: the mask tile of query block n in slot n % 2
  uint64_t mask_empty[2]; // the element group of slot i has read it
  uint64_t acc_done;
  uint32_t tmem_base;
  int abort;
  alignas(16) float nlse2[2][kStr];   // −log2e·lse per query of the block in Q slot i
  alignas(16) float ndelta[2][kStr];  // −δ per query
};
constexpr int kKvK = 0;
constexpr int kKvV = kOwnBytes;            // V (dK blocks, until it is in TMEM), then two dO slots
constexpr int kKvQ = 2 * kOwnBytes;        // three Q slots (two with a staged mask)
constexpr int kKvBars = kKvQ + 3 * kStrBytes;  // 224 KB of tiles, then the barriers
// Staged-mask variant: two mask tiles [64 queries x 128 keys] of at most 16-bit elements in
// the place of the third Q slot.
constexpr int kKvMaskTile = kStr * kOwn * 2;
constexpr int kKvMask = kKvQ + 2 * kStrBytes;
static_assert(kKvMask + 2 * kKvMaskTile <= kKvBars, "mask tiles overlap the barriers");
// The partner's fp32 partial sum [128 x 256] in the first block of a cluster, once no MMA
// reads V, dO or Q any more: 16-byte pieces ordered (32-column chunk, piece, row).
constexpr int kKvRed = kOwnBytes;
static_assert(kKvRed + kOwn * kD * 4 <= kKvBars, "partial sum overlaps the barriers");
constexpr int kKvBytes = kKvBars + (int)sizeof(Kv256Bars);
static_assert(kKvBytes <= 227 * 1024, "dK/dV shared memory exceeds the per-block limit");
constexpr int kKvThreads = 640;

// kRowBc: the mask has one row for every query (row stride 0, e.g. key padding), read once
// per key from global memory.  Any other mask is staged: the producer loads each query
// block's [64 x 128] mask tile by TMA (map tm) into one of two slots, from which each
// element thread reads its key's column; the third Q slot gives way to the two tiles.
template <typename T, bool kMasked, bool kRowBc>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kKvThreads, 1)
    tc_dkdv256_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                      const __grid_constant__ CUtensorMap tdk, const __grid_constant__ CUtensorMap tdv,
                      const __grid_constant__ CUtensorMap tm, Problem p) {
  constexpr bool kTileMask = kMasked && !kRowBc;
  constexpr int kQs = kTileMask ? 2 : 3;  // Q slots
  constexpr bool kBf16 = IsBf16<T>::value;
  constexpr uint32_t kIdS = idesc_f16(kOwn, kStr, kBf16, false, false);  // M = 128, N = 64
  constexpr uint32_t kIdAcc = idesc_f16(kOwn, kD, kBf16, false, true);   // M = 128, N = 256, B MN-major
  constexpr uint32_t kColAcc = 0, kColX = 256, kColOp = 384;
  extern __shared__ unsigned char smem_raw[];
  // The layout assumes a 1024-byte aligned base (TMA's 128-byte swizzle and the MMA
  // descriptors need it); should a launch place it elsewhere, the block reports an error
  // and leaves before touching shared memory.
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) report_error(p.err, kDevErrLayout, kKidTcDkdv);
    return;
  }
  uint8_t* sm = smem_raw;
  Kv256Bars& bars = *reinterpret_cast<Kv256Bars*>(sm + kKvBars);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // Block order: the two blocks of a cluster, then the dK and the dV cluster of one (batch,
  // KV head, key tile), all units of one key tile, then the next tile; under the causal mask
  // the first key tiles see the most queries, so the heavy blocks go first.
  const uint32_t rank = cluster_rank();
  const bool dv = ((blockIdx.x >> 1) & 1) != 0;
  const int rest = blockIdx.x >> 2;
  const int units = p.B * p.Hkv;
  const int unit = rest % units;
  const int b = unit / p.Hkv, g = unit % p.Hkv;
  const int j0 = (rest / units) * kOwn;  // first key of this block
  // Queries before j0 - coff see none of these keys.
  const int i_begin = p.causal ? max(0, j0 - p.coff) : 0;
  const int nqb = i_begin < p.Lq ? (p.Lq - i_begin + kStr - 1) / kStr : 0;
  // This block's share of the G·nqb query blocks: [n_begin, n_begin + total).
  const int n_half = (p.G * nqb + 1) / 2;
  const int n_begin = rank == 0 ? 0 : n_half;
  const int total = rank == 0 ? n_half : p.G * nqb - n_half;
  // Loops below count n from 0 (barrier phases and slots follow it); query block n of this
  // block is block n_begin + n of the key tile's list.
  // dO slot of query block n, the parity of its use and its place.
  auto do_slot = [&](int n) { return n & 1; };
  auto do_par = [&](int n) { return static_cast<uint32_t>((n >> 1) & 1); };
  auto do_off = [&](int n) { return kKvV + (n & 1) * kStrBytes; };

  if (threadIdx.x == 0) {
    bars.abort = 0;
    mbar_init(&bars.own_full, 1);
    for (int s = 0; s < 3; ++s) {
      mbar_init(&bars.q_full[s], 1);
      mbar_init(&bars.q_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.do_full[s], 1);
      mbar_init(&bars.do_empty[s], 1);
      mbar_init(&bars.vec_full[s], 32);  // every lane of the producer warp
      mbar_init(&bars.vec_empty[s], 256);  // the element group of buffer s (8 warps)
      mbar_init(&bars.s_full[s], 1);
      mbar_init(&bars.p_ready[s], 256);
      mbar_init(&bars.x_free[s], 1);
      mbar_init(&bars.s_read[s], 256);
      mbar_init(&bars.dp_full[s], 1);
      mbar_init(&bars.ds_ready[s], 256);
      mbar_init(&bars.y_free[s], 1);
      mbar_init(&bars.mask_full[s], 1);
      mbar_init(&bars.mask_empty[s], 256);
    }
    mbar_init(&bars.opnd_ready, 512);
    mbar_init(&bars.acc_done, 3);  // one commit per MMA issuer warp
    fence_mbar_init();
  }
  if (warp == kIssuer) {
    tmem_alloc(&bars.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars.tmem_base;
  const WaitCtx wc{&bars.abort, 0, p.wait_limit_ns, p.err, kKidTcDkdv};
  constexpr unsigned kAll = 0xffffffffu;
  if (warp >= 16) regs_dec<kRegsLow>();
  bool el_ok = true;  // element threads: every wait of the loop and of acc_done succeeded

  if (warp == kProducer) {
    // K (and V in dK blocks) once; per query block n: Q(n) into slot n % kQs once its last
    // reader of n-3 has finished, dO(n) into slot n % 2 once the reader of n-2 has finished
    // (in dK blocks the first dO load waits for V to be copied out of its place), then the
    // per-query vectors into slot n % 2 once the element threads are done with those of n-2.
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tdo);
      mbar_arrive_expect_tx(&bars.own_full, (dv ? 1 : 2) * kOwnBytes);
      for (int cb = 0; cb < 4; ++cb) {
        tma_load_4d(sm + kKvK + cb * kOwnCb, &tk, &bars.own_full, cb * 64, j0, g, b);
        if (!dv) tma_load_4d(sm + kKvV + cb * kOwnCb, &tv, &bars.own_full, cb * 64, j0, g, b);
      }
    }
    // The per-query lse and δ of query block n (lane e holds queries e and e + 32) are read
    // from global memory one block ahead, so their latency overlaps the loop's waits
    // instead of holding back the next TMA loads.
    float lv[2], dl[2];
    auto fetch = [&](int n) {
      const int h = g * p.G + (n_begin + n) / nqb;
      const int i0 = i_begin + ((n_begin + n) % nqb) * kStr;
      const float* lsep = p.lse + q_row(p, b, h, 0);
      const float* dlp = p.delta + q_row(p, b, h, 0);
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int i = i0 + lane + 32 * t;
        lv[t] = i < p.Lq ? lsep[i] : -pos_inf();  // −inf: the row sees no key, P = 0
        dl[t] = (!dv && i < p.Lq) ? dlp[i] : 0.f;
      }
    };
    if (total > 0) fetch(0);
    int q_issued = 0, do_issued = 0, mask_issued = 0;
    bool ok = true;
    for (int n = 0; ok && n < total; ++n) {
      const int s = n % 2;
      const int h = g * p.G + (n_begin + n) / nqb;
      const int i0 = i_begin + ((n_begin + n) % nqb) * kStr;
      const int qs = n % kQs;
      if (!(ok = __all_sync(kAll, mbar_wait(&bars.q_empty[qs], ((n / kQs) & 1) ^ 1, wc)))) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars.q_full[qs], kStrBytes);
        for (int cb = 0; cb < 4; ++cb)
          tma_load_4d(sm + kKvQ + qs * kStrBytes + cb * kStrCb, &tq, &bars.q_full[qs], cb * 64, i0, h, b);
      }
      q_issued = n + 1;
      if (!(ok = __all_sync(kAll, mbar_wait(&bars.do_empty[do_slot(n)], do_par(n) ^ 1, wc) &&
                                      (dv || n > 0 || mbar_wait(&bars.opnd_ready, 0, wc)))))
        break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars.do_full[do_slot(n)], kStrBytes);
        for (int cb = 0; cb < 4; ++cb)
          tma_load_4d(sm + do_off(n) + cb * kStrCb, &tdo, &bars.do_full[do_slot(n)], cb * 64, i0, h, b);
      }
      do_issued = n + 1;
      // Per-query vectors, negated for the packed math of the element warps.
      if (!(ok = __all_sync(kAll, mbar_wait(&bars.vec_empty[s], ((n / 2) & 1) ^ 1, wc)))) break;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        bars.nlse2[s][lane + 32 * t] = lv[t] == -pos_inf() ? -pos_inf() : -lv[t] * kLog2e;
        bars.ndelta[s][lane + 32 * t] = -dl[t];
      }
      mbar_arrive(&bars.vec_full[s]);
      if constexpr (kTileMask) {  // the query block's mask tile, once its slot's readers are done
        if (!(ok = __all_sync(kAll, mbar_wait(&bars.mask_empty[s], ((n / 2) & 1) ^ 1, wc)))) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars.mask_full[s], kStr * kOwn * (p.mask_kind == kMaskBool ? 1 : 2));
          tma_load_4d(sm + kKvMask + s * kKvMaskTile, &tm, &bars.mask_full[s], j0, i0, p.lm.sh == 0 ? 0 : h,
                      p.lm.sb == 0 ? 0 : b);
        }
        mask_issued = n + 1;
      }
      if (n + 1 < total) fetch(n + 1);
    }
    if (lane == 0 && (!ok || bars.abort)) {  // let copies still in flight land before the block exits
      for (int n = max(0, q_issued - kQs); n < q_issued; ++n) drain_wait(&bars.q_full[n % kQs], (n / kQs) & 1);
      for (int n = max(0, do_issued - 2); n < do_issued; ++n)
        drain_wait(&bars.do_full[do_slot(n)], do_par(n));
      for (int n = max(0, mask_issued - 2); n < mask_issued; ++n) drain_wait(&bars.mask_full[n % 2], (n / 2) & 1);
    }
  } else if (warp >= kIssuer) {
    const int role = __shfl_sync(kAll, warp - kIssuer, 0);
    bool ok = __all_sync(kAll, mbar_wait(&bars.own_full, 0, wc));
    tc_fence_after();
    const uint32_t k_s = smem_u32(sm + kKvK);
    auto q_s = [&](int n) { return smem_u32(sm + kKvQ + (n % kQs) * kStrBytes); };
    // The TS score product of the block (dV: Sᵀ; dK: dPᵀ) reads the TMEM copy of K or V.
    if (role < 2 && (role == 0) == dv && ok) ok = __all_sync(kAll, mbar_wait(&bars.opnd_ready, 0, wc));
    if (role == 0) {
      // Sᵀ(n) = K·Q(n)ᵀ into buffer n % 2 once dV(n-2) or dK(n-2) has read it.
      for (int n = 0; ok && n < total; ++n) {
        const int s = n % 2;
        if (!(ok = __all_sync(kAll, mbar_wait(&bars.q_full[n % kQs], (n / kQs) & 1, wc) &&
                                        mbar_wait(dv ? &bars.x_free[s] : &bars.y_free[s], ((n / 2) & 1) ^ 1, wc))))
          break;
        tc_fence_after();
        if (dv) mma_scores256_ts(tbase + kColX + 64 * s, tbase + kColOp, q_s(n), kIdS);
        else mma_scores256(tbase + kColX + 64 * s, k_s, q_s(n), kIdS);
        mma_commit_w(&bars.s_full[s]);
        if (dv) mma_commit_w(&bars.q_empty[n % kQs]);
      }
    } else if (role == 1 && dv) {
      // dV += Pᵀ(n)·dO(n).
      for (int n = 0; ok && n < total; ++n) {
        const int s = n % 2;
        if (!(ok = __all_sync(kAll, mbar_wait(&bars.p_ready[s], (n / 2) & 1, wc) &&
                                        mbar_wait(&bars.do_full[do_slot(n)], do_par(n), wc))))
          break;
        tc_fence_after();
        mma_acc256(tbase + kColAcc, tbase + kColX + 64 * s, smem_u32(sm + do_off(n)), kIdAcc, n == 0);
        mma_commit_w(&bars.x_free[s]);
        mma_commit_w(&bars.do_empty[do_slot(n)]);
      }
    } else if (role == 1) {
      // dPᵀ(n) = V·dO(n)ᵀ over Sᵀ(n) in buffer n % 2 once its element group has read it.
      for (int n = 0; ok && n < total; ++n) {
        const int s = n % 2;
        if (!(ok = __all_sync(kAll, mbar_wait(&bars.do_full[do_slot(n)], do_par(n), wc) &&
                                        mbar_wait(&bars.s_read[s], (n / 2) & 1, wc))))
          break;
        tc_fence_after();
        mma_scores256_ts(tbase + kColX + 64 * s, tbase + kColOp, smem_u32(sm + do_off(n)), kIdS);
        mma_commit_w(&bars.dp_full[s]);
        mma_commit_w(&bars.do_empty[do_slot(n)]);
      }
    } else if (!dv) {
      // dK += dSᵀ(n)·Q(n).  Q(n) is loaded (Sᵀ(n) read it before dSᵀ(n) could exist);
      // waiting on its barrier too makes the TMA writes visible to this warp's MMA directly.
      for (int n = 0; ok && n < total; ++n) {
        const int s = n % 2;
        if (!(ok = __all_sync(kAll, mbar_wait(&bars.ds_ready[s], (n / 2) & 1, wc) &&
                                        mbar_wait(&bars.q_full[n % kQs], (n / kQs) & 1, wc))))
          break;
        tc_fence_after();
        mma_acc256(tbase + kColAcc, tbase + kColX + 64 * s, q_s(n), kIdAcc, n == 0);
        mma_commit_w(&bars.y_free[s]);
        mma_commit_w(&bars.q_empty[n % kQs]);
      }
    }
    mma_commit_w(&bars.acc_done);
    drain_wait(&bars.acc_done, 0);
  } else {
    regs_inc<kRegsHigh>();
    const int c = warp / 4, quarter = warp % 4;
    const int j = j0 + quarter * 32 + lane;  // this thread's key
    const uint64_t cc = f2pack(p.scale_log2, p.scale_log2);
    // The owned tile the TS score product reads (dV blocks: K for Sᵀ; dK blocks: V for dPᵀ)
    // into TMEM columns [384, 512): row r in lane r, elements (2i, 2i+1) of D in column
    // 384 + i.  Warp e copies rows [32(e % 4), +32) of D columns [64c, 64c + 64); the 16-byte
    // pieces of a swizzled row hold consecutive element pairs, so they go over as they are.
    bool ok = __all_sync(kAll, mbar_wait(&bars.own_full, 0, wc));
    if (ok) {
      const uint8_t* src = sm + (dv ? kKvK : kKvV) + c * kOwnCb;
      const int r = quarter * 32 + lane;
      uint32_t w[32];
#pragma unroll
      for (int pc = 0; pc < 8; ++pc) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + sw128_off(r, pc));
        w[4 * pc] = v.x;
        w[4 * pc + 1] = v.y;
        w[4 * pc + 2] = v.z;
        w[4 * pc + 3] = v.w;
      }
      tmem_st32(tmem_addr(tbase, quarter * 32, kColOp + 32 * c), w);
      tmem_st_wait();
      tc_fence_before();
    }
    mbar_arrive(&bars.opnd_ready);
    // The element warps form two groups of 8 that take turns: group gq = e / 8 takes the
    // query blocks n with n % 2 == gq (TMEM buffer n % 2), so one group's TMEM round trips,
    // exponentials and barrier hand-offs overlap the other's block.  Warp e of a group has
    // lane quarter e % 4 (keys) and query columns [32h, 32h + 32), h = (e / 4) % 2; it packs
    // the 16-bit results of queries [32h, 32h + 16) over columns [32h, 32h + 8) and those of
    // [32h + 16, 32h + 32) over [32h + 16, 32h + 24), where the K-steps 2h and 2h + 1 of the
    // dV / dK products read them.
    const int gq = warp / 8, h2 = (warp / 4) % 2;
    for (int n = gq; ok && n < total; n += 2) {
      const int s = n % 2;
      const int i0 = i_begin + ((n_begin + n) % nqb) * kStr + 32 * h2;  // first query of this warp's columns
      ok = __all_sync(kAll, mbar_wait(&bars.s_full[s], (n / 2) & 1, wc) &&
                                mbar_wait(&bars.vec_full[s], (n / 2) & 1, wc) &&
                                (!kTileMask || mbar_wait(&bars.mask_full[s], (n / 2) & 1, wc)));
      if (!ok) break;
      tc_fence_after();
      const int ic = i0 + p.coff;  // key j is hidden from query i0 + q when j > ic + q
      const bool diag = p.causal && j0 + kOwn - 1 > ic;
      const uint64_t* nl2 = reinterpret_cast<const uint64_t*>(&bars.nlse2[s][32 * h2]);
      const uint64_t* nd2 = reinterpret_cast<const uint64_t*>(&bars.ndelta[s][32 * h2]);
      const uint32_t x_addr = tmem_addr(tbase, quarter * 32, kColX + 64 * s + 32 * h2);
      // Mask element (this block's head, query 0, key j); keys past Lkv are not read.
      const int64_t mcol = kRowBc ? row_off(p.lm, b, g * p.G + (n_begin + n) / nqb, 0) + j : 0;
      // Pᵀ of this warp's 32 queries, in fp32 pairs.
      uint64_t pf[16];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t sr[16];
        tmem_ld16(x_addr + 16 * hf, sr);
        float mv[kMasked ? 16 : 1];  // log2e·M of query i0 + 16hf + e
        if constexpr (kMasked) {
          if constexpr (kRowBc) {
            const float m = j < p.Lkv ? mask_log2<T>(p, mcol) : 0.f;
#pragma unroll
            for (int e = 0; e < 16; ++e) mv[e] = i0 + 16 * hf + e < p.Lq ? m : 0.f;
          } else {
            // Row q of the tile holds query i0 - 32h + q, key k at element 128q + k; rows
            // past Lq and keys past Lkv were filled with zeros by the load (those P are zero
            // or clipped anyway).
            const int kl = quarter * 32 + lane, q0 = 32 * h2 + 16 * hf;
            const uint8_t* tile = sm + kKvMask + s * kKvMaskTile;
            if (p.mask_kind == kMaskBool) {
#pragma unroll
              for (int e = 0; e < 16; ++e) mv[e] = tile[(q0 + e) * kOwn + kl] ? 0.f : minus_inf();
            } else {
              const T* t16 = reinterpret_cast<const T*>(tile);
#pragma unroll
              for (int e = 0; e < 16; ++e) mv[e] = Elem<T>::to_f(t16[(q0 + e) * kOwn + kl]) * kLog2e;
            }
          }
        }
        tmem_ld_wait(sr);
        if (!dv && hf == 1) {  // dPᵀ(n) may now overwrite Sᵀ(n)
          tc_fence_before();
          mbar_arrive(&bars.s_read[s]);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int x = 8 * hf + e;
          float p0, p1;
          if constexpr (kMasked) {  // c·s is finite, so a hidden key's −inf passes through the fma
            ex2_pair(fadd2(f2pack(fmaf(p.scale_log2, __uint_as_float(sr[2 * e]), mv[2 * e]),
                                  fmaf(p.scale_log2, __uint_as_float(sr[2 * e + 1]), mv[2 * e + 1])),
                           nl2[x]),
                     p0, p1);
          } else {
            ex2_pair(ffma2(f2pack(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1])), cc, nl2[x]), p0, p1);
          }
          if (diag) {
            if (j > ic + 2 * x) p0 = 0.f;
            if (j > ic + 2 * x + 1) p1 = 0.f;
          }
          pf[x] = f2pack(p0, p1);
        }
      }
      if constexpr (kTileMask) mbar_arrive(&bars.mask_empty[s]);  // done with the mask tile
      uint32_t pk[8];
      if (dv) {
        mbar_arrive(&bars.vec_empty[s]);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            float p0, p1;
            f2unpack(pf[8 * hf + e], p0, p1);
            pk[e] = pack2<T>(p0, p1);
          }
          tmem_st8(x_addr + 16 * hf, pk);  // Pᵀ over the first 8 of each 16 columns
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars.p_ready[s]);
      } else {
        // dSᵀ = Pᵀ∘(dPᵀ − δ).
        ok = __all_sync(kAll, mbar_wait(&bars.dp_full[s], (n / 2) & 1, wc));
        if (!ok) break;
        tc_fence_after();
        // In two halves of 16 columns (the half-0 store does not touch half 1's columns).
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t dr[16];
          tmem_ld16(x_addr + 16 * hf, dr);
          tmem_ld_wait(dr);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int x = 8 * hf + e;
            float d0, d1;
            f2unpack(fmul2(pf[x], fadd2(f2pack(__uint_as_float(dr[2 * e]), __uint_as_float(dr[2 * e + 1])), nd2[x])),
                     d0, d1);
            pk[e] = pack2<T>(d0, d1);
          }
          tmem_st8(x_addr + 16 * hf, pk);  // dSᵀ over the first 8 of each 16 columns
        }
        mbar_arrive(&bars.vec_empty[s]);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars.ds_ready[s]);
      }
    }
    // With no query block (total == 0) nothing else has waited for the K load; the
    // epilogue overwrites K, so wait for it here.
    if (ok)
      ok = __all_sync(kAll, mbar_wait(&bars.own_full, 0, wc) && (total == 0 || mbar_wait(&bars.acc_done, 0, wc)));
    el_ok = ok;
  }
  // Epilogue, every thread of both blocks.  After the first cluster barrier no MMA of
  // either block runs any more (the element threads waited for acc_done; the issuers
  // drained it), so the second block writes its partial sum into the first block's V/dO
  // and Q space; after the second the first block adds it to its own, scales (dK by the
  // softmax scale), packs the result in 8 chunks of 32 columns (warps of group c take
  // chunks c and c + 4), stages it in its K buffer and writes it by bulk tensor stores
  // once all 16 warps have staged theirs (keys past Lkv are clipped).
  cluster_sync();
  const bool elem = warp < 16;
  const int c = warp / 4, quarter = warp % 4, r = quarter * 32 + lane;
  if (elem && rank != 0 && el_ok) {
    tc_fence_after();
    const uint32_t red = map_to_rank(smem_u32(sm + kKvRed), 0);
#pragma unroll 1
    for (int c32 = c; c32 < kD / 32; c32 += 4) {
      uint32_t acc[32];
      if (total > 0) {
        tmem_ld32(tmem_addr(tbase, quarter * 32, kColAcc + 32 * c32), acc);
        tmem_ld_wait(acc);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) acc[e] = 0u;  // no query block in this half
      }
#pragma unroll
      for (int e4 = 0; e4 < 8; ++e4)
        st_cluster_v4(red + ((c32 * 8 + e4) * kOwn + r) * 16, acc[4 * e4], acc[4 * e4 + 1], acc[4 * e4 + 2],
                      acc[4 * e4 + 3]);
    }
  }
  cluster_sync();
  if (elem && rank == 0) {
    if (el_ok) {
      tc_fence_after();
      const float mul = dv ? 1.f : p.scale;
#pragma unroll 1
      for (int c32 = c; c32 < kD / 32; c32 += 4) {
        uint32_t acc[32];
        if (total > 0) {
          tmem_ld32(tmem_addr(tbase, quarter * 32, kColAcc + 32 * c32), acc);
          tmem_ld_wait(acc);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) acc[e] = 0u;  // no query sees these keys
        }
        uint32_t packed[16];
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const uint4 o = *reinterpret_cast<const uint4*>(sm + kKvRed + ((c32 * 8 + e4) * kOwn + r) * 16);
          const float a0 = (__uint_as_float(acc[4 * e4]) + __uint_as_float(o.x)) * mul;
          const float a1 = (__uint_as_float(acc[4 * e4 + 1]) + __uint_as_float(o.y)) * mul;
          const float a2 = (__uint_as_float(acc[4 * e4 + 2]) + __uint_as_float(o.z)) * mul;
          const float a3 = (__uint_as_float(acc[4 * e4 + 3]) + __uint_as_float(o.w)) * mul;
          packed[2 * e4] = pack2<T>(a0, a1);
          packed[2 * e4 + 1] = pack2<T>(a2, a3);
        }
        uint8_t* blk = sm + kKvK + (c32 / 2) * kOwnCb;
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4)
          *reinterpret_cast<uint4*>(blk + sw128_off(r, (c32 % 2) * 4 + v4)) =
              make_uint4(packed[4 * v4], packed[4 * v4 + 1], packed[4 * v4 + 2], packed[4 * v4 + 3]);
      }
      fence_async_smem();
    }
    if (named_sync_and(1, 512, el_ok) && warp == 0 && lane == 0) {
      for (int cb = 0; cb < 4; ++cb) tma_store_4d(dv ? &tdv : &tdk, sm + kKvK + cb * kOwnCb, cb * 64, j0, g, b);
      bulk_commit();
      bulk_wait_read();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kIssuer) {
    __syncwarp();
    tmem_dealloc(tbase, 512);
  }
}

template <typename T, bool kMasked>
cudaError_t dq256_t(const Problem& p, cudaStream_t s) {
  CUtensorMap tq, tk, tv, tdo, tdq;
  if (!make_tmap_4d(&tq, p.q, kD, p.Lq, p.Hq, p.B, p.lq, kOwn) ||
      !make_tmap_4d(&tdo, p.dout, kD, p.Lq, p.Hq, p.B, p.ldo, kOwn) ||
      !make_tmap_4d(&tdq, p.dq, kD, p.Lq, p.Hq, p.B, p.ldq, kOwn) ||
      !make_tmap_4d(&tk, p.k, kD, p.Lkv, p.Hkv, p.B, p.lk, kStr) ||
      !make_tmap_4d(&tv, p.v, kD, p.Lkv, p.Hkv, p.B, p.lv, kStr))
    return cudaErrorInvalidValue;
  const int smem = kDqBytes + 1024;
  auto kern = tc_dq256_kernel<T, kMasked>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const unsigned nqt = (p.Lq + kOwn - 1) / kOwn;
  kern<<<nqt * p.Hq * p.B, kDqThreads, smem, s>>>(tq, tk, tv, tdo, tdq, p);
  return cudaGetLastError();
}

template <typename T, bool kMasked, bool kRowBc>
cudaError_t dkdv256_t(const Problem& p, cudaStream_t s) {
  CUtensorMap tq, tk, tv, tdo, tdk, tdv, tm;
  memset(&tm, 0, sizeof(tm));  // not read unless the mask is staged
  if (kMasked && !kRowBc && !make_tmap_mask(&tm, p, p.mask_kind == kMaskBool ? 1 : 2, kOwn, kStr, false))
    return cudaErrorInvalidValue;
  if (!make_tmap_4d(&tk, p.k, kD, p.Lkv, p.Hkv, p.B, p.lk, kOwn) ||
      !make_tmap_4d(&tv, p.v, kD, p.Lkv, p.Hkv, p.B, p.lv, kOwn) ||
      !make_tmap_4d(&tdk, p.dk, kD, p.Lkv, p.Hkv, p.B, p.ldk, kOwn) ||
      !make_tmap_4d(&tdv, p.dv, kD, p.Lkv, p.Hkv, p.B, p.ldv, kOwn) ||
      !make_tmap_4d(&tq, p.q, kD, p.Lq, p.Hq, p.B, p.lq, kStr) ||
      !make_tmap_4d(&tdo, p.dout, kD, p.Lq, p.Hq, p.B, p.ldo, kStr))
    return cudaErrorInvalidValue;
  auto kern = tc_dkdv256_kernel<T, kMasked, kRowBc>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kKvBytes);
  if (e != cudaSuccess) return e;
  const unsigned nkt = (p.Lkv + kOwn - 1) / kOwn;
  kern<<<4 * nkt * p.Hkv * p.B, kKvThreads, kKvBytes, s>>>(tq, tk, tv, tdo, tdk, tdv, tm, p);
  return cudaGetLastError();
}

}  // namespace

bool tensor_bwd256_supported(const Problem& p, int dtype) { return tensor_supported(p, dtype) && p.D == kD; }

cudaError_t launch_tc_dq256(const Problem& p, int dtype, cudaStream_t s) {
  if (p.mask) return dtype == 2 ? dq256_t<__nv_bfloat16, true>(p, s) : dq256_t<__half, true>(p, s);
  return dtype == 2 ? dq256_t<__nv_bfloat16, false>(p, s) : dq256_t<__half, false>(p, s);
}

cudaError_t launch_tc_dkdv256(const Problem& p, int dtype, cudaStream_t s) {
  if (p.mask && p.lm.sl == 0)
    return dtype == 2 ? dkdv256_t<__nv_bfloat16, true, true>(p, s) : dkdv256_t<__half, true, true>(p, s);
  if (p.mask) return dtype == 2 ? dkdv256_t<__nv_bfloat16, true, false>(p, s) : dkdv256_t<__half, true, false>(p, s);
  return dtype == 2 ? dkdv256_t<__nv_bfloat16, false, false>(p, s) : dkdv256_t<__half, false, false>(p, s);
}

}  // namespace sdpa
