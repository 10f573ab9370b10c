// Tensor-core forward (fp16/bf16, D in {32, 64, 96, 128}): TMA + tcgen05 + TMEM.
//
// One block computes 256 query rows (two 128-row Q tiles) of one (batch, head) against
// the keys of its KV head (h / G).  Warp roles (384 threads):
//   warps 0-3 / 4-7  softmax warpgroup of Q tile 0 / 1: thread = one query row = one TMEM
//                    lane; online softmax in the log2 domain ("[Metal] Add Flash Attention
//                    VJP for training", section "Implementation Notes": log2 domain)
//   warp 8           TMA producer: Q tiles once, then K_j, V_j tiles into a 4-stage ring
//                    (3 stages with a mask, whose tiles take the room of the fourth)
//   warps 9 / 10     tcgen05 issuers for Q tile 0 / 1 (whole warp runs the loop, one
//                    elected lane issues); warp 9 owns TMEM
//   warp 11          mask tile producer with a mask; otherwise idle (it completes
//                    warpgroup 2 for the register split)
// setmaxnreg moves registers from warpgroup 2 to the softmax warpgroups, so a softmax
// thread holds its row's 128 scores in registers after one TMEM round trip and computes
// the row maximum and the exponentials from there.  The two softmax warpgroups take turns
// at the exponential pass, so one tile's pass overlaps the other tile's MMAs.
// Tensor memory (512 columns, fp32): S_w = Q_w·K_jᵀ at columns [128w, 128w+128); P_w is
// written back over the first 64 columns of S_w as packed 16-bit pairs and read from TMEM
// as the A operand of O_w += P_w·V_j, with O_w at columns [256 + 128w, 256 + 128w + D).
// Without a mask PV is issued in two halves of 64 keys, the first as soon as the softmax
// has written that half of P, so the next S waits only for the second half.
// The running maximum is raised lazily: O and l are rescaled only when a row's maximum
// grows by more than 2^8, so exponentials stay <= 256 while O and l use one consistent
// maximum, which keeps the result exact up to rounding.
// Rows with few visible keys (the first Q tile under the causal mask, or every row when
// Lkv <= 128) can have |O| near the largest inputs, where rounding P to 16 bits would
// add an error comparable to the output's own rounding.  For that one KV tile (under an
// attention mask, for every tile the softmax warps vote to split, see kSplitShare) P is
// split into a 16-bit head and a 16-bit remainder (written to S columns [64, 128)) and
// both are multiplied into O, so P enters O with ~16 extra bits.
// Epilogue: O / l rounded to the element type and staged in the tile's (now unused) Q
// buffer, then written by bulk tensor stores; lse = ln2·(m + log2 l) (natural log).
#include "launch.h"
#include "tc_common.cuh"

namespace sdpa {
namespace {
using namespace tc;

constexpr int kBM = 128;      // rows per Q tile
constexpr int kBN = 128;      // keys per KV tile
constexpr int kQTiles = 2;    // Q tiles per block
constexpr int kMaxStages = 4;  // K/V ring stages (each one [kBN x D] tile), unmasked kernel
constexpr int kThreads = 384;    // warps 0-7 softmax, 8 producer, 9-10 MMA issuers, 11 mask producer
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kMaskWarp = 11;
// Register split (setmaxnreg): the block launches with 168 registers a thread (65,536 / 384
// rounded down to a multiple of 8, 64,512 in all); warpgroup 2 (producer, issuers, idle
// warp) drops to 56 and the softmax warpgroups rise to 224: 128·56 + 256·224 = 64,512.
constexpr int kRegsLow = 56;
constexpr int kRegsHigh = 224;
static_assert(128 * kRegsLow + 256 * kRegsHigh <= kThreads * 168, "register split exceeds the launch");
constexpr float kRescale = 8.f;  // log2 of the largest exponential allowed before rescaling
// Under an attention mask a KV tile gets the split P when some row's largest P in it exceeds
// this share of the weight the row has gathered before it (always on its first visible
// tile).  On the other tiles no key holds more than a quarter of its row's weight when its
// tile arrives, so rounding P to 16 bits (relative 2^-9 per key) moves O by at most
// 2^-9·max|V| over all such keys together, the bound the unmasked kernel has on every tile
// after its first; a row resting on a few keys still gets the split on their tiles.
constexpr float kSplitShare = 1.f / 4.f;

template <int D, bool kMasked>
struct FwdLayout {
  // Tiles hold ceil(D/64) 64-column blocks (D = 96 is padded to 128 columns: TMA fills
  // the missing columns with zeros on loads and clips them on stores).
  static constexpr int kCB = (D + 63) / 64;
  static constexpr int kTileBytes = kBM * kCB * 64 * 2;
  static constexpr int kQOff = 0;
  static constexpr int kRingOff = kQTiles * kTileBytes;
  // The masked kernel keeps three ring stages (measured as fast as four) to make room for
  // one [128 x 128] mask tile per Q tile (16-bit values; a boolean tile uses half).
  static constexpr int kStages = kMasked ? 3 : kMaxStages;
  static constexpr int kMaskOff = kRingOff + kStages * kTileBytes;
  static constexpr int kMaskTile = kBM * kBN * 2;
  static constexpr int kBytes = kMaskOff + (kMasked ? kQTiles * kMaskTile : 0);
  static constexpr int kSCol = 0;    // S_w at column 128·w
  static constexpr int kOCol = 256;  // O_w at column 256 + 128·w
};

struct FwdBars {
  uint64_t q_full;
  uint64_t kv_full[kMaxStages];
  uint64_t kv_empty[kMaxStages];
  uint64_t s_full[kQTiles];
  uint64_t p_full[kQTiles];
  uint64_t o_done[kQTiles];
  uint64_t mma_done[kQTiles];
  uint64_t turn[kQTiles];  // exponential pass of Q tile w may start (alternates 0, 1, 0, ...)
  uint64_t p_half[kQTiles];  // unmasked: P_w of keys [0, 64) has been written
  uint64_t mask_full[kQTiles];  // masked: Q tile w's mask tile for its next KV tile has landed
  uint64_t mask_free[kQTiles];  // masked: the four warps of warpgroup w have read it
  uint64_t vote[kQTiles];       // masked: the four warps of warpgroup w have voted on the split
  int need[kQTiles][2][4];      // masked: warp q of warpgroup w wants the split P for tile j (at j % 2)
  uint32_t tmem_base;
  int abort;
};

template <typename T>
struct IsBf16 { static constexpr bool value = false; };
template <>
struct IsBf16<__nv_bfloat16> { static constexpr bool value = true; };

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// KV tile j of Q tile starting at tile_row0 gets the split (head + remainder) P: the first
// tile of rows that see few keys, and every tile under an attention mask, which can leave
// any row with few keys of non-negligible weight.
__device__ __forceinline__ bool split_tile(const Problem& p, int j, int tile_row0) {
  return j == 0 && (tile_row0 == 0 || p.Lkv <= kBN);
}

// The split vote of one KV tile under a mask: set when any warp of the warpgroup voted
// for it (the flags are written before the warps arrive on the vote and P barriers).
__device__ __forceinline__ bool split_voted(const int (&need)[4]) {
  const volatile int* v = need;
  return (v[0] | v[1] | v[2] | v[3]) != 0;
}

// One 16-byte piece of shared memory, read in program order with the other such reads
// (a volatile load: the scheduler may not hoist the whole row's pieces at once).
__device__ __forceinline__ uint4 lds_ordered(const uint8_t* ptr) {
  uint4 v;
  asm volatile("ld.volatile.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(ptr)));
  return v;
}

// Bit 7 of each byte of the result is set iff that byte of w is nonzero (the low seven
// bits plus 0x7f carry into bit 7 when any of them is set, without crossing into the next
// byte; or-ing w adds bit 7 itself); the other bits are zero.
__device__ __forceinline__ uint32_t nonzero_bytes(uint32_t w) {
  return (((w & 0x7f7f7f7fu) + 0x7f7f7f7fu) | w) & 0x80808080u;
}

// Replicates the top bit of byte t of x over a 32-bit word (prmt's sign-replicate mode).
__device__ __forceinline__ uint32_t byte_sign(uint32_t x, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(d) : "r"(x), "r"(sel));
  return d;
}

// Applies the Q tile's mask to one query row's raw scores sv (fp32 bits) and returns the
// factor the softmax then applies to them (log2-domain score = factor · sv[e]).  The mask
// tile in shared memory holds, for a full mask, the 128 rows in the 128-byte swizzle of its
// TMA load (16-bit values as two 64-key boxes, 16 KB apart) and, for a mask broadcast over
// queries, one plain row (128 bytes boolean, 256 bytes 16-bit) that every thread reads.
// Keys past Lkv and rows past Lq were filled with zeros; the callers hide such keys by
// their key limit and never store such rows.
//   - A broadcast row that keeps every key (boolean) or adds 0 to every key (additive) is
//     left as it is, with the factor c = scale·log2e; the warp checks it together (each
//     lane one slice of the row, then a vote).
//   - Boolean, c > 0: a hidden key's raw score becomes −inf (c·−inf = −inf), factor c.
//   - Boolean, c <= 0: c·s plus 0 or −inf, factor 1.
//   - Additive: scale·s + M (natural-log domain, −inf stays −inf), factor log2e.
// kOrdered reads the pieces with ordered (volatile) loads, which keeps the scheduler from
// hoisting them all at once where registers are short (the D = 256 kernel).
template <typename T, bool kOrdered>
__device__ __forceinline__ float mask_row(uint32_t (&sv)[kBN], const uint8_t* tile, int r, int lane, bool row_bc,
                                          bool is_bool, float c, float scale) {
  if (row_bc) {
    bool any;
    if (is_bool) {
      const uint32_t w = *reinterpret_cast<const volatile uint32_t*>(tile + 4 * lane);
      any = __any_sync(0xffffffffu, nonzero_bytes(w) != 0x80808080u);  // some key hidden
    } else {
      const volatile uint32_t* v = reinterpret_cast<const volatile uint32_t*>(tile + 8 * lane);
      any = __any_sync(0xffffffffu, ((v[0] | v[1]) & 0x7fff7fffu) != 0u);  // some value nonzero
    }
    if (!any) return c;
  }
  auto piece = [&](int q) {  // the q-th 16-byte piece of the row
    const int x = q / 8, qq = q % 8;
    const uint8_t* a = is_bool ? tile + (row_bc ? 16 * q : sw128_off(r, q))
                               : tile + (row_bc ? 128 * x + 16 * qq : 16384 * x + sw128_off(r, qq));
    return kOrdered ? lds_ordered(a) : *reinterpret_cast<const uint4*>(a);
  };
  if (is_bool && c > 0.f) {
#pragma unroll
    for (int q = 0; q < kBN / 16; ++q) {
      const uint4 w = piece(q);
      const uint32_t keep[4] = {nonzero_bytes(w.x), nonzero_bytes(w.y), nonzero_bytes(w.z), nonzero_bytes(w.w)};
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const uint32_t m = byte_sign(keep[t / 4], 0x8888u | (0x1111u * (t % 4)));
        sv[16 * q + t] = (sv[16 * q + t] & m) | (0xff800000u & ~m);
      }
    }
    return c;
  }
  if (is_bool) {
#pragma unroll
    for (int q = 0; q < kBN / 16; ++q) {
      const uint4 w = piece(q);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const bool keep = ((ws[t / 4] >> (8 * (t % 4))) & 0xffu) != 0u;
        sv[16 * q + t] = __float_as_uint(fmaf(c, __uint_as_float(sv[16 * q + t]), keep ? 0.f : neg_inf()));
      }
    }
    return 1.f;
  }
  const uint64_t sc = f2pack(scale, scale);
#pragma unroll
  for (int q = 0; q < kBN / 8; ++q) {
    union { uint4 u; T e[8]; } w;
    w.u = piece(q);
#pragma unroll
    for (int t = 0; t < 8; t += 2) {
      float a, b;
      f2unpack(ffma2(sc, f2pack(__uint_as_float(sv[8 * q + t]), __uint_as_float(sv[8 * q + t + 1])),
                     f2pack(Elem<T>::to_f(w.e[t]), Elem<T>::to_f(w.e[t + 1]))),
               a, b);
      sv[8 * q + t] = __float_as_uint(a);
      sv[8 * q + t + 1] = __float_as_uint(b);
    }
  }
  return kLog2e;
}

// The mask tile of rows [row, row + 128) (row 0 of a mask broadcast over queries) and keys
// [k0, k0 + 128) into dst (1024-byte aligned), completing on bar.  One 128-key box of a
// boolean mask, two 64-key boxes of a 16-bit one.
__device__ __forceinline__ void load_mask_tile(uint8_t* dst, const CUtensorMap* tm, uint64_t* bar, const Problem& p,
                                               int k0, int row, int h, int b) {
  const bool row_bc = p.lm.sl == 0;
  const int es = p.mask_kind == kMaskBool ? 1 : 2;
  mbar_arrive_expect_tx(bar, (row_bc ? 1 : kBM) * kBN * es);
  const int hh = p.lm.sh == 0 ? 0 : h, bb = p.lm.sb == 0 ? 0 : b, rr = row_bc ? 0 : row;
  if (es == 1) {
    tma_load_4d(dst, tm, bar, k0, rr, hh, bb);
  } else {
    tma_load_4d(dst, tm, bar, k0, rr, hh, bb);
    tma_load_4d(dst + (row_bc ? 128 : 16384), tm, bar, k0 + 64, rr, hh, bb);
  }
}

// The tensor map of the forward's mask tiles (box and swizzle as mask_row reads them).
bool make_fwd_mask_map(CUtensorMap* tm, const Problem& p) {
  const bool row_bc = p.lm.sl == 0;
  const int es = p.mask_kind == kMaskBool ? 1 : 2;
  return make_tmap_mask(tm, p, es, es == 1 ? 128 : 64, row_bc ? 1 : kBM, !row_bc);
}

// Number of leading keys of the tile starting at k0 that row i may see: key k0 + e is
// visible iff e < lim (keys past Lkv are padding; under the causal mask key <= i + coff).
__device__ __forceinline__ int visible_keys(const Problem& p, int k0, int i) {
  int lim = min(p.Lkv - k0, kBN);
  if (p.causal) lim = min(lim, i + p.coff - k0 + 1);
  return lim;
}

// Row maximum of the scaled scores of a 128-key tile held in registers (three-input max):
// the maximum raw score (the minimum for a negative scale) over the visible keys e < lim,
// scaled once.  A row that sees no key of the tile gets -inf.
template <bool kMask>
__device__ __forceinline__ float tile_max(const uint32_t (&sv)[kBN], float c, int lim) {
  constexpr int kH = kBN / 2;
  if (kMask && lim <= 0) return neg_inf();
  float acc[4];
  if (c >= 0.f) {
    acc[0] = acc[1] = acc[2] = acc[3] = neg_inf();
#pragma unroll
    for (int e = 0; e < kH; ++e) {
      const float xa = (!kMask || e < lim) ? __uint_as_float(sv[e]) : neg_inf();
      const float xb = (!kMask || kH + e < lim) ? __uint_as_float(sv[kH + e]) : neg_inf();
      acc[e % 4] = fmax3(acc[e % 4], xa, xb);
    }
    return fmaxf(fmaxf(acc[0], acc[1]), fmaxf(acc[2], acc[3])) * c;
  }
  acc[0] = acc[1] = acc[2] = acc[3] = -neg_inf();
#pragma unroll
  for (int e = 0; e < kH; ++e) {
    const float xa = (!kMask || e < lim) ? __uint_as_float(sv[e]) : -neg_inf();
    const float xb = (!kMask || kH + e < lim) ? __uint_as_float(sv[kH + e]) : -neg_inf();
    acc[e % 4] = fmin3(acc[e % 4], xa, xb);
  }
  return fminf(fminf(acc[0], acc[1]), fminf(acc[2], acc[3])) * c;
}

// Exponentials of a 128-key tile held in registers: returns their sum and writes P packed
// to 16 bits into TMEM columns [0, 64) of the S tile (column q holds keys 2q and 2q + 1).
// With `half`, arrives on it once P of keys [0, 64) is in TMEM, so that the PV product of
// those keys can start while the other half is computed.
template <typename T, bool kMask>
__device__ __forceinline__ float exp_pass(const uint32_t (&sv)[kBN], uint32_t s_addr, float c, float neg_m,
                                          int lim, uint64_t* half) {
  const uint64_t cc = f2pack(c, c), nm = f2pack(neg_m, neg_m);
  uint64_t acc0 = f2pack(0.f, 0.f), acc1 = acc0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t pk[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const int col = 64 * h + 2 * e;
      uint64_t xx = ffma2(f2pack(__uint_as_float(sv[col]), __uint_as_float(sv[col + 1])), cc, nm);
      if constexpr (kMask) {
        float x0, x1;
        f2unpack(xx, x0, x1);
        if (col >= lim) x0 = neg_inf();
        if (col + 1 >= lim) x1 = neg_inf();
        xx = f2pack(x0, x1);
      }
      float p0, p1;
      ex2_pair(xx, p0, p1);
      if (e % 2 == 0) acc0 = fadd2(acc0, f2pack(p0, p1));
      else acc1 = fadd2(acc1, f2pack(p0, p1));
      pk[e] = pack2<T>(p0, p1);
    }
    tmem_st32(s_addr + 32 * h, pk);
    if (h == 0 && half != nullptr) {
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(half);
    }
  }
  float a, b, c2, d;
  f2unpack(acc0, a, b);
  f2unpack(acc1, c2, d);
  return (a + b) + (c2 + d);
}

// As exp_pass, and also the remainder P − head(P), packed to 16 bits into columns
// [64, 128) (their scores are already in registers), so that P enters O with about 16
// more bits.  Written 16 keys at a time to keep few packed values live.
template <typename T>
__device__ __forceinline__ float exp_pass_split(const uint32_t (&sv)[kBN], uint32_t s_addr, float c, float neg_m,
                                                int lim) {
  const uint64_t cc = f2pack(c, c), nm = f2pack(neg_m, neg_m);
  uint64_t acc0 = f2pack(0.f, 0.f), acc1 = acc0;
#pragma unroll
  for (int q = 0; q < kBN / 16; ++q) {
    uint32_t pk[8], rk[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int col = 16 * q + 2 * e;
      uint64_t xx = ffma2(f2pack(__uint_as_float(sv[col]), __uint_as_float(sv[col + 1])), cc, nm);
      float x0, x1;
      f2unpack(xx, x0, x1);
      if (col >= lim) x0 = neg_inf();
      if (col + 1 >= lim) x1 = neg_inf();
      float p0, p1;
      ex2_pair(f2pack(x0, x1), p0, p1);
      if (e % 2 == 0) acc0 = fadd2(acc0, f2pack(p0, p1));
      else acc1 = fadd2(acc1, f2pack(p0, p1));
      pk[e] = pack2<T>(p0, p1);
      float h0, h1;
      unpack2<T>(pk[e], h0, h1);
      rk[e] = pack2<T>(p0 - h0, p1 - h1);
    }
    tmem_st8(s_addr + 8 * q, pk);
    tmem_st8(s_addr + 64 + 8 * q, rk);
  }
  float a, b, c2, d;
  f2unpack(acc0, a, b);
  f2unpack(acc1, c2, d);
  return (a + b) + (c2 + d);
}

// Bounded wait that ignores the abort flag (used to drain in-flight work at teardown).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > limit_ns) return;
  }
}

// kMasked: the call has an attention mask (a separate instantiation, so that the
// unmasked kernel carries none of the mask code).
template <typename T, int D, bool kMasked>
__global__ void __launch_bounds__(kThreads, 1)
    tc_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                  const __grid_constant__ CUtensorMap tm, Problem p) {
  using L = FwdLayout<D, kMasked>;
  constexpr int kCB = L::kCB;
  constexpr int kStages = L::kStages;
  constexpr bool kBf16 = IsBf16<T>::value;
  constexpr uint32_t kIdS = idesc_f16(kBM, kBN, kBf16, false, false);
  constexpr uint32_t kIdO = idesc_f16(kBM, D, kBf16, false, true);
  extern __shared__ unsigned char smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ FwdBars bars;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // Block order: all heads of one query block, then the next block; under the causal mask
  // the last (heaviest) query blocks go first so that the tail of the grid is light.
  const int units = p.B * p.Hq;
  const int unit = blockIdx.x % units, rank = blockIdx.x / units;
  const int b = unit / p.Hq, h = unit % p.Hq, g = h / p.G;
  const int nqb = (p.Lq + kBM * kQTiles - 1) / (kBM * kQTiles);
  const int qb = p.causal ? nqb - 1 - rank : rank;
  const int row0 = qb * kBM * kQTiles;
  int nkv[kQTiles];
#pragma unroll
  for (int w = 0; w < kQTiles; ++w) {
    const int r0 = row0 + w * kBM;
    if (r0 >= p.Lq) {
      nkv[w] = 0;
    } else {
      const int kend = p.causal ? min(p.Lkv, min(p.Lq, r0 + kBM) + p.coff) : p.Lkv;
      nkv[w] = (kend + kBN - 1) / kBN;
    }
  }
  const int nmax = max(nkv[0], nkv[1]);

  if (threadIdx.x == 0) {
    bars.abort = 0;
    mbar_init(&bars.q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars.kv_full[s], 1);
      mbar_init(&bars.kv_empty[s], kQTiles);  // released by both MMA issuers
    }
    for (int w = 0; w < kQTiles; ++w) {
      mbar_init(&bars.s_full[w], 1);
      mbar_init(&bars.p_full[w], kBM);
      mbar_init(&bars.o_done[w], 1);
      mbar_init(&bars.p_half[w], kBM);
    }
    mbar_init(&bars.mma_done[0], 1);
    mbar_init(&bars.mma_done[1], 1);
    mbar_init(&bars.turn[0], 4);  // one arrival per warp of the other warpgroup
    mbar_init(&bars.turn[1], 4);
    for (int w = 0; w < kQTiles; ++w) {
      mbar_init(&bars.mask_full[w], 1);
      mbar_init(&bars.mask_free[w], 4);  // one arrival per warp of warpgroup w
      mbar_init(&bars.vote[w], 4);
    }
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
  const WaitCtx wc{&bars.abort, 0, p.wait_limit_ns, p.err, kKidTcFwd};
  if (warp >= 8) regs_dec<kRegsLow>();

  if (warp == kProducerWarp) {
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      prefetch_tmap(&to);
      const int nq = nkv[1] > 0 ? 2 : 1;
      mbar_arrive_expect_tx(&bars.q_full, nq * L::kTileBytes);
      for (int w = 0; w < nq; ++w)
        for (int cb = 0; cb < kCB; ++cb)
          tma_load_4d(sm + L::kQOff + w * L::kTileBytes + cb * 16384, &tq, &bars.q_full, cb * 64,
                      row0 + w * kBM, h, b);
      // The block one wave later (about num_sms blocks on) starts when some block ends:
      // bring its Q tiles into L2 now, so that its first loads come from L2, not HBM.
      if (p.num_sms > 0 && blockIdx.x + p.num_sms < gridDim.x) {
        const int nb = blockIdx.x + p.num_sms;
        const int nu = nb % units, nrank = nb / units;
        const int nrow0 = (p.causal ? nqb - 1 - nrank : nrank) * kBM * kQTiles;
        for (int w = 0; w < kQTiles; ++w)
          if (nrow0 + w * kBM < p.Lq)
            for (int cb = 0; cb < kCB; ++cb) tma_prefetch_l2_4d(&tq, cb * 64, nrow0 + w * kBM, nu % p.Hq, nu / p.Hq);
      }
      int issued = 0;
      bool ok = true;
      for (int j = 0; ok && j < nmax; ++j) {
        for (int kv = 0; kv < 2; ++kv) {
          const int it = 2 * j + kv, s = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!(ok = mbar_wait(&bars.kv_empty[s], ph ^ 1, wc))) break;
          if (p.inject == 1 && it == 0) continue;  // test hook: never deliver the first K tile
          mbar_arrive_expect_tx(&bars.kv_full[s], L::kTileBytes);
          for (int cb = 0; cb < kCB; ++cb)
            tma_load_4d(sm + L::kRingOff + s * L::kTileBytes + cb * 16384, kv ? &tv : &tk,
                        &bars.kv_full[s], cb * 64, j * kBN, g, b);
          issued = it + 1;
        }
      }
      if (!ok || bars.abort) {  // let copies still in flight land before the block exits
        for (int it = max(0, issued - kStages); it < issued; ++it)
          drain_wait(&bars.kv_full[it % kStages], (it / kStages) & 1, 100000000ull);
      }
    }
  } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
    // One MMA issuer warp per Q tile, so that each tile's chain S → softmax → PV → S
    // advances at its own pace.  The whole warp runs the loop; one lane issues.
    constexpr unsigned kAll = 0xffffffffu;
    const int w = __shfl_sync(kAll, warp - kMmaWarp, 0);
    const int nkv_w = w == 0 ? nkv[0] : nkv[1];
    bool ok = __all_sync(kAll, mbar_wait(&bars.q_full, 0, wc));
    tc_fence_after();
    const uint64_t qd = sdesc_sw128(smem_u32(sm + L::kQOff) + w * L::kTileBytes, 16, 1024);
    const uint32_t ring_s = smem_u32(sm + L::kRingOff);
    const uint32_t s_tm = tbase + L::kSCol + w * 128, o_tm = tbase + L::kOCol + w * 128;
    const int tile_row0 = row0 + w * kBM;
    if constexpr (!kMasked) {
      // PV_w(j) in two K = 64 halves: the half over keys 0..63 starts once the softmax has
      // written that half of P(j), so it runs while the other half is computed and the chain
      // S → softmax → PV → S only waits for the second half.  (S(j+1) stays one N = 128
      // product: N = 64 halves issued early measured slower, the MMA count doubling.)  Every
      // ring stage still gets exactly one kv_empty arrival per use, in order.
      auto s_full_product = [&](int stage) {
        const uint64_t kd = sdesc_sw128(ring_s + stage * L::kTileBytes, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
          mma_ss_w(s_tm, sdesc_advance(qd, off), sdesc_advance(kd, off), kIdS, kk > 0);
        }
      };
      auto pv_half = [&](int stage, int hi, bool first) {  // keys [64·hi, 64·hi + 64) of P·V
        const uint64_t vd = sdesc_sw128(ring_s + stage * L::kTileBytes, 16384, 1024);
#pragma unroll
        for (int kk = 4 * hi; kk < 4 * hi + 4; ++kk)
          mma_ts_w(o_tm, s_tm + kk * 8, sdesc_advance(vd, kk * 2048), kIdO, (!first || kk > 0) ? 1u : 0u);
      };
      // K(0) and S(0).
      ok = __all_sync(kAll, mbar_wait(&bars.kv_full[0], 0, wc));
      if (ok && nkv_w > 0) {
        tc_fence_after();
        s_full_product(0);
        mma_commit_w(&bars.s_full[w]);
      }
      if (ok) mma_commit_w(&bars.kv_empty[0]);
      for (int j = 0; ok && j < nmax; ++j) {
        const int itv = 2 * j + 1, itk = 2 * j + 2;  // V(j), K(j+1)
        const int sv = itv % kStages, sk = itk % kStages;
        const uint32_t phv = (itv / kStages) & 1, phk = (itk / kStages) & 1;
        const bool act = j < nkv_w, act1 = j + 1 < nkv_w, nxt = j + 1 < nmax;
        const bool spl = act && split_tile(p, j, tile_row0);
        if (!(ok = __all_sync(kAll, mbar_wait(&bars.kv_full[sv], phv, wc)))) break;
        if (act) {
          if (!(ok = __all_sync(kAll, mbar_wait(spl ? &bars.p_full[w] : &bars.p_half[w], j & 1, wc)))) break;
          tc_fence_after();
          pv_half(sv, 0, j == 0);
          if (spl) {  // the whole P and its remainder (columns [64, 128))
            pv_half(sv, 1, false);
            const uint64_t vd = sdesc_sw128(ring_s + sv * L::kTileBytes, 16384, 1024);
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
              mma_ts_w(o_tm, s_tm + 64 + kk * 8, sdesc_advance(vd, kk * 2048), kIdO, 1u);
          }
        }
        if (act && !spl) {
          if (!(ok = __all_sync(kAll, mbar_wait(&bars.p_full[w], j & 1, wc)))) break;
          tc_fence_after();
          pv_half(sv, 1, false);
        }
        if (act) mma_commit_w(&bars.o_done[w]);
        mma_commit_w(&bars.kv_empty[sv]);
        if (nxt) {
          if (!(ok = __all_sync(kAll, mbar_wait(&bars.kv_full[sk], phk, wc)))) break;
          if (act1) {
            // P(j) consumed: S(j+1) may overwrite S_w.
            if (!(ok = __all_sync(kAll, mbar_wait(&bars.o_done[w], j & 1, wc)))) break;
            tc_fence_after();
            s_full_product(sk);
            mma_commit_w(&bars.s_full[w]);
          }
          mma_commit_w(&bars.kv_empty[sk]);
        }
      }
    } else {
      for (int j = 0; ok && j < nmax; ++j) {
        const int sk = (2 * j) % kStages, sv = (2 * j + 1) % kStages;
        const uint32_t phk = ((2 * j) / kStages) & 1, phv = ((2 * j + 1) / kStages) & 1;
        // Every stage use gets exactly one arrival from each issuer, made only after the
        // stage was filled for this use, even by an issuer whose tile needs no MMA here.
        if (!(ok = __all_sync(kAll, mbar_wait(&bars.kv_full[sk], phk, wc)))) break;
        if (j < nkv_w) {
          if (j > 0 && !(ok = __all_sync(kAll, mbar_wait(&bars.o_done[w], (j - 1) & 1, wc)))) break;
          tc_fence_after();  // P_w(j-1) consumed: S_w may be overwritten
          const uint64_t kd = sdesc_sw128(ring_s + sk * L::kTileBytes, 16, 1024);
  #pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
            mma_ss_w(s_tm, sdesc_advance(qd, off), sdesc_advance(kd, off), kIdS, kk > 0);
          }
          mma_commit_w(&bars.s_full[w]);
        }
        mma_commit_w(&bars.kv_empty[sk]);  // one of the stage's two arrivals
        if (!(ok = __all_sync(kAll, mbar_wait(&bars.kv_full[sv], phv, wc)))) break;
        if (j < nkv_w) {
          if (!(ok = __all_sync(kAll, mbar_wait(&bars.p_full[w], j & 1, wc)))) break;
          tc_fence_after();
          const uint64_t vd = sdesc_sw128(ring_s + sv * L::kTileBytes, 16384, 1024);
  #pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma_ts_w(o_tm, s_tm + kk * 8, sdesc_advance(vd, kk * 2048), kIdO, (j > 0 || kk > 0) ? 1u : 0u);
          if (kMasked ? split_voted(bars.need[w][j % 2]) : split_tile(p, j, tile_row0)) {  // remainder of P, columns [64, 128)
  #pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
              mma_ts_w(o_tm, s_tm + 64 + kk * 8, sdesc_advance(vd, kk * 2048), kIdO, 1u);
          }
          mma_commit_w(&bars.o_done[w]);
        }
        mma_commit_w(&bars.kv_empty[sv]);
      }
    }
    mma_commit_w(&bars.mma_done[w]);
    drain_wait(&bars.mma_done[w], 0, 100000000ull);
  } else if (kMasked && warp == kMaskWarp) {
    // Mask producer: Q tile w's mask tile for KV tile j once its four softmax warps have
    // read the one for KV tile j-1.
    if (lane == 0) {
      prefetch_tmap(&tm);
      int issued[kQTiles] = {0, 0};
      bool ok = true;
      for (int j = 0; ok && j < nmax; ++j)
        for (int w = 0; w < kQTiles; ++w) {
          if (j >= nkv[w]) continue;
          if (j > 0 && !(ok = mbar_wait(&bars.mask_free[w], (j - 1) & 1, wc))) break;
          load_mask_tile(sm + L::kMaskOff + w * L::kMaskTile, &tm, &bars.mask_full[w], p, j * kBN, row0 + w * kBM, h, b);
          issued[w] = j + 1;
        }
      if (!ok || bars.abort)  // let copies still in flight land before the block exits
        for (int w = 0; w < kQTiles; ++w)
          if (issued[w] > 0) drain_wait(&bars.mask_full[w], (issued[w] - 1) & 1, 100000000ull);
    }
  } else if (warp < 8) {
    // Softmax warpgroups.
    regs_inc<kRegsHigh>();
    const int w = warp / 4, quarter = warp % 4;
    const int r = quarter * 32 + lane;
    const int i = row0 + w * kBM + r;
    const uint32_t s_addr = tmem_addr(tbase, quarter * 32, L::kSCol + w * 128);
    const uint32_t o_addr = tmem_addr(tbase, quarter * 32, L::kOCol + w * 128);
    const float c = p.scale_log2;
    const int tile_row0 = row0 + w * kBM;
    float m = neg_inf(), l = 0.f;
    bool ok = true;
    // The two warpgroups take turns at the exponential pass (0, 1, 0, 1, ... while both
    // tiles have KV tiles left), so the pass of one tile has the multi-function units to
    // itself while the tensor core works on the other tile's PV and next S.
    const int nboth = min(nkv[0], nkv[1]);
    constexpr bool masked = kMasked;
    const uint8_t* mtile = sm + (masked ? L::kMaskOff + w * L::kMaskTile : 0);
    const bool row_bc = p.lm.sl == 0, mbool = p.mask_kind == kMaskBool;
    for (int j = 0; j < nkv[w]; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.s_full[w], j & 1, wc) &&
                                       (!masked || mbar_wait(&bars.mask_full[w], j & 1, wc)));
      if (!ok) break;
      tc_fence_after();
      const int k0 = j * kBN;
      const bool need_mask = (k0 + kBN > p.Lkv) || (p.causal && k0 + kBN - 1 > tile_row0 + p.coff);
      // The row's 128 scores in registers (one TMEM round trip), then its maximum.
      uint32_t sv[kBN];
#pragma unroll
      for (int q4 = 0; q4 < kBN / 32; ++q4)
        tmem_ld32(s_addr + 32 * q4, *reinterpret_cast<uint32_t(*)[32]>(&sv[32 * q4]));
      tmem_ld_wait(sv);
      const int lim = visible_keys(p, k0, i);
      // Under a mask, mask_row applies it and gives the factor the scores are used with.
      float cs = c;
      if constexpr (masked) {
        cs = mask_row<T, false>(sv, mtile, r, lane, row_bc, mbool, c, p.scale);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.mask_free[w]);  // this warp is done with the mask tile
      }
      const float mt = need_mask ? tile_max<true>(sv, cs, lim) : tile_max<false>(sv, cs, lim);
      const float m_new = fmaxf(m, mt);
      const bool resc = m_new > m + kRescale;  // always true on the first tile (m = -inf)
      const float alpha = resc ? ex2(m - m_new) : 1.f;  // 0 when m was −inf
      if (resc) {
        l *= alpha;
        m = m_new;
      }
      if constexpr (masked) {
        // Split vote: this tile's largest P against the weight the row has so far (0 before
        // its first visible key, so that tile always votes for the split).
        const float pmax = ex2(mt + (m == neg_inf() ? 0.f : -m));
        const bool wn = __any_sync(0xffffffffu, pmax > l * kSplitShare);
        if (lane == 0) {
          bars.need[w][j % 2][quarter] = wn;
          mbar_arrive(&bars.vote[w]);
        }
      }
      if (j > 0 && __any_sync(0xffffffffu, resc)) {
        // Some row of this warp raised its maximum: rescale O once PV(j-1) has landed.
        ok = __all_sync(0xffffffffu, mbar_wait(&bars.o_done[w], (j - 1) & 1, wc));
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int c32 = 0; c32 < D / 32; ++c32) {
          uint32_t orr[32];
          tmem_ld32(o_addr + c32 * 32, orr);
          tmem_ld_wait(orr);
#pragma unroll
          for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
          tmem_st32(o_addr + c32 * 32, orr);
        }
        tmem_st_wait();
      }
      if (j < nboth && (w == 1 || j > 0)) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bars.turn[w], (w == 1 ? j : j - 1) & 1, wc));
        if (!ok) break;
      }
      // Pass 2: P = exp2(c·s − m), row sum, P packed to 16 bits over S's first 64 columns.
      // m is −inf only while a mask has hidden every key so far; any finite shift then
      // gives P = 0 for those keys.
      const float neg_m = (kMasked && m == neg_inf()) ? 0.f : -m;
      bool split;
      if constexpr (masked) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bars.vote[w], j & 1, wc));
        if (!ok) break;
        split = split_voted(bars.need[w][j % 2]);
      } else {
        split = split_tile(p, j, tile_row0);
      }
      uint64_t* half = kMasked ? nullptr : &bars.p_half[w];
      if (split)
        l += exp_pass_split<T>(sv, s_addr, cs, neg_m, lim);
      else if (need_mask)
        l += exp_pass<T, true>(sv, s_addr, cs, neg_m, lim, half);
      else
        l += exp_pass<T, false>(sv, s_addr, cs, neg_m, lim, half);
      tmem_st_wait();
      tc_fence_before();
      if (!kMasked && split) mbar_arrive(&bars.p_half[w]);  // one p_half phase per tile
      // Hand the turn to the other tile before arriving on p_full: P(j) complete then implies
      // that every warp of this warpgroup has also arrived on the turn barrier for tile j, so
      // no warp's arrival for tile j+1 can count toward tile j.
      if (j < nboth - w) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.turn[1 - w]);
      }
      mbar_arrive(&bars.p_full[w]);
    }
    if (ok && nkv[w] > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.o_done[w], (nkv[w] - 1) & 1, wc));
    if (nkv[w] > 0) {  // the same for every thread of the warpgroup
      // O / l is staged in this tile's Q buffer (its last reader, S_w(nkv-1), has finished)
      // in the swizzled layout of the Q tile, then written by one bulk tensor store per
      // 64-column block; rows at or past Lq are clipped by the store.
      uint8_t* stage = sm + L::kQOff + w * L::kTileBytes;
      if (ok) {
        tc_fence_after();
        const float a = fold_sink(p, h, m, l);
        const float inv = (!kMasked || l > 0.f) ? a / l : 0.f;  // a row that sees no key: O = 0
#pragma unroll
        for (int c32 = 0; c32 < D / 32; ++c32) {
          uint32_t orr[32];
          tmem_ld32(o_addr + c32 * 32, orr);
          tmem_ld_wait(orr);
          uint32_t packed[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            packed[e] = pack2<T>(__uint_as_float(orr[2 * e]) * inv, __uint_as_float(orr[2 * e + 1]) * inv);
          uint8_t* blk = stage + (c32 / 2) * 16384;
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            *reinterpret_cast<uint4*>(blk + sw128_off(r, (c32 % 2) * 4 + v4)) =
                make_uint4(packed[4 * v4], packed[4 * v4 + 1], packed[4 * v4 + 2], packed[4 * v4 + 3]);
        }
        fence_async_smem();
        if (i < p.Lq && p.lse) p.lse[q_row(p, b, h, i)] = (!kMasked || l > 0.f) ? (m + __log2f(l)) * kLn2 : neg_inf();
      }
      if (named_sync_and(1 + w, kBM, ok) && r == 0) {
        for (int cb = 0; cb < kCB; ++cb) tma_store_4d(&to, stage + cb * 16384, cb * 64, tile_row0, h, b);
        bulk_commit();
        bulk_wait_read();
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

// ================================================================== head dim 256
// One block computes 128 query rows (one Q tile) of one (batch, head).  Tensor memory: two
// S buffers (columns [0, 128) and [128, 256)) and O (columns [256, 512), all 256 of D),
// so S of KV tile j+1 is computed into the other buffer while the softmax of tile j runs,
// and S never waits for a PV product that reads P from the same buffer except two tiles
// back.  Per KV tile: S = Q·Kᵀ (16 K-steps of M = N = 128) and O += P·V (8 K-steps of
// M = 128, N = 256).  Shared memory: Q (64 KB), one 64 KB stage for K tiles and one for V
// tiles, and under an attention mask one [128 x 128] mask tile.  The K stage is handed
// back in its four 64-column blocks (S reads block kk / 4 in K-step kk) and the V stage in
// its two 64-row halves (PV reads rows [16kk, 16kk + 16) in K-step kk), so the next tile's
// first pieces are on their way while the current product still reads the rest.
// Warp roles (256 threads): warps 0-3 softmax (one thread per query row, all 128 keys of
// a tile, as in the D <= 128 kernel), 4 and 7 TMA producers (Q and K; mask and V), 5 S
// issuer (owns TMEM), 6 PV issuer.
constexpr int k256Threads = 256;
constexpr int k256Stages = 2;
template <bool kMasked>
struct Fwd256Layout {
  static constexpr int kCB = 4;                       // 64-column blocks of D
  static constexpr int kTileBytes = kBM * kCB * 128;  // [128 rows x 256] 16-bit
  static constexpr int kQOff = 0;
  static constexpr int kRingOff = kTileBytes;
  static constexpr int kMaskOff = kRingOff + k256Stages * kTileBytes;
  static constexpr int kBytes = kMaskOff + (kMasked ? kBM * kBN * 2 : 0);
};
struct Fwd256Bars {
  uint64_t q_full;
  uint64_t k_full[4];   // column block cb of K(j) has landed
  uint64_t k_empty[4];  // S(j) has read column block cb
  uint64_t v_full[2];   // rows [64h, 64h + 64) of V(j) have landed
  uint64_t v_empty[2];  // PV(j) has read them
  uint64_t s_full[2];   // S buffer b holds S of KV tile j with j % 2 == b
  uint64_t p_full[2];   // its P has been written
  uint64_t pv_done[2];  // PV of that tile has finished (buffer free, O updated)
  uint64_t fin;
  uint64_t mask_full;   // masked: the mask tile of the next KV tile has landed
  uint64_t mask_free;   // masked: the four softmax warps have read it
  uint64_t vote;        // masked: the four softmax warps have voted on the split
  // masked: softmax warp q wants the split P for KV tile j (at j % 2: a warp may vote on
  // tile j+1 before another warp or the PV issuer has read the votes on tile j)
  int need[2][4];
  uint32_t tmem_base;
  int abort;
};

template <typename T, bool kMasked>
__global__ void __launch_bounds__(k256Threads, 1)
    tc_fwd256_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                     const __grid_constant__ CUtensorMap tm, Problem p) {
  using L = Fwd256Layout<kMasked>;
  constexpr int D = 256, kCB = L::kCB;
  constexpr bool kBf16 = IsBf16<T>::value;
  constexpr uint32_t kIdS = idesc_f16(kBM, kBN, kBf16, false, false);
  constexpr uint32_t kIdO = idesc_f16(kBM, D, kBf16, false, true);
  constexpr uint32_t kColO = 256;
  extern __shared__ unsigned char smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Fwd256Bars bars;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // Block order: all heads of one query tile, then the next; causal: heaviest first.
  const int units = p.B * p.Hq;
  const int unit = blockIdx.x % units, rank = blockIdx.x / units;
  const int b = unit / p.Hq, h = unit % p.Hq, g = h / p.G;
  const int nqt = (p.Lq + kBM - 1) / kBM;
  const int row0 = (p.causal ? nqt - 1 - rank : rank) * kBM;
  const int kend = p.causal ? min(p.Lkv, min(p.Lq, row0 + kBM) + p.coff) : p.Lkv;
  const int nkv = (kend + kBN - 1) / kBN;  // >= 1

  if (threadIdx.x == 0) {
    bars.abort = 0;
    mbar_init(&bars.q_full, 1);
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bars.k_full[s], 1);
      mbar_init(&bars.k_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.v_full[s], 1);
      mbar_init(&bars.v_empty[s], 1);
    }
    for (int c = 0; c < 2; ++c) {
      mbar_init(&bars.s_full[c], 1);
      mbar_init(&bars.p_full[c], kBM);
      mbar_init(&bars.pv_done[c], 1);
    }
    mbar_init(&bars.fin, 2);  // one commit per issuer
    mbar_init(&bars.mask_full, 1);
    mbar_init(&bars.mask_free, 4);  // one arrival per softmax warp
    mbar_init(&bars.vote, 4);
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&bars.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars.tmem_base;
  const WaitCtx wc{&bars.abort, 0, p.wait_limit_ns, p.err, kKidTcFwd};

  if (warp == 4 || warp == 7) {
    // ---------------------------------------------------------------- producers
    // Warp 4 loads Q, then each column block of K(j) into stage 0 as soon as S(j-1) has
    // read that block of K(j-1); warp 7 loads each 64-row half of V(j) into stage 1 as
    // soon as PV(j-1) has read that half of V(j-1), and before it (masked) the mask tile
    // of KV tile j once the softmax warps have read that of tile j-1.  Two producers, so
    // that neither kind of tile waits behind the other.
    if (lane == 0) {
      const int kv = warp == 4 ? 0 : 1;
      if (kv == 0) {
        prefetch_tmap(&tq);
        prefetch_tmap(&tk);
        prefetch_tmap(&to);
        mbar_arrive_expect_tx(&bars.q_full, L::kTileBytes);
        for (int cb = 0; cb < kCB; ++cb)
          tma_load_4d(sm + L::kQOff + cb * 16384, &tq, &bars.q_full, cb * 64, row0, h, b);
        // The block one wave later (about num_sms blocks on) starts when some block ends:
        // bring its Q tile into L2 now, so that its first load comes from L2, not HBM.
        if (p.num_sms > 0 && blockIdx.x + p.num_sms < gridDim.x) {
          const int nb = blockIdx.x + p.num_sms;
          const int nu = nb % units, nrank = nb / units;
          const int nrow0 = (p.causal ? nqt - 1 - nrank : nrank) * kBM;
          for (int cb = 0; cb < kCB; ++cb) tma_prefetch_l2_4d(&tq, cb * 64, nrow0, nu % p.Hq, nu / p.Hq);
        }
      } else {
        prefetch_tmap(&tv);
        if (kMasked) prefetch_tmap(&tm);
      }
      int piece_issued[kCB] = {0, 0, 0, 0}, m_issued = 0;  // tiles issued per K block / V half
      bool ok = true;
      for (int j = 0; ok && j < nkv; ++j) {
        if (kMasked && kv == 1) {
          if (j > 0 && !(ok = mbar_wait(&bars.mask_free, (j - 1) & 1, wc))) break;
          load_mask_tile(sm + L::kMaskOff, &tm, &bars.mask_full, p, j * kBN, row0, h, b);
          m_issued = j + 1;
        }
        if (p.inject == 1 && kv == 0 && j == 0) continue;  // test hook: never deliver the first K tile
        uint8_t* stage = sm + L::kRingOff + kv * L::kTileBytes;
        if (kv == 0) {
          for (int cb = 0; cb < kCB && ok; ++cb) {
            if (!(ok = mbar_wait(&bars.k_empty[cb], (j & 1) ^ 1, wc))) break;
            mbar_arrive_expect_tx(&bars.k_full[cb], L::kTileBytes / kCB);
            tma_load_4d(stage + cb * 16384, &tk, &bars.k_full[cb], cb * 64, j * kBN, g, b);
            piece_issued[cb] = j + 1;
          }
        } else {
          // rows [64h, 64h + 64) of every column block: a 64-row box at row offset 64h
          for (int hr = 0; hr < 2 && ok; ++hr) {
            if (!(ok = mbar_wait(&bars.v_empty[hr], (j & 1) ^ 1, wc))) break;
            mbar_arrive_expect_tx(&bars.v_full[hr], L::kTileBytes / 2);
            for (int cb = 0; cb < kCB; ++cb)
              tma_load_4d(stage + cb * 16384 + hr * 8192, &tv, &bars.v_full[hr], cb * 64, j * kBN + 64 * hr, g, b);
            piece_issued[hr] = j + 1;
          }
        }
      }
      if (!ok || bars.abort) {  // let copies still in flight land before the block exits
        for (int x = 0; x < (kv == 0 ? kCB : 2); ++x)
          if (piece_issued[x] > 0)
            drain_wait(kv == 0 ? &bars.k_full[x] : &bars.v_full[x], (piece_issued[x] - 1) & 1, 100000000ull);
      }
      if ((!ok || bars.abort) && m_issued > 0)
        drain_wait(&bars.mask_full, (m_issued - 1) & 1, 100000000ull);
    }
  } else if (warp == 5 || warp == 6) {
    // ---------------------------------------------------------------- MMA issuers
    // Warp 5: S(j) = Q·K(j)ᵀ into buffer j % 2 once PV(j-2) has read P(j-2) from it.
    // Warp 6: O += P(j)·V(j) once the softmax has written P(j).
    constexpr unsigned kAll = 0xffffffffu;
    const bool s_issuer = __shfl_sync(kAll, warp, 0) == 5;
    bool ok = __all_sync(kAll, mbar_wait(&bars.q_full, 0, wc));
    tc_fence_after();
    const uint64_t qd = sdesc_sw128(smem_u32(sm + L::kQOff), 16, 1024);
    const uint32_t ring_s = smem_u32(sm + L::kRingOff);
    for (int j = 0; ok && j < nkv; ++j) {
      const int buf = j % 2;
      if (s_issuer) {
        // K(j) in stage 0, one 64-column block at a time: K-steps 4cb .. 4cb + 3 read block
        // cb, which is handed back as soon as they are done.
        if (j >= 2 && !(ok = __all_sync(kAll, mbar_wait(&bars.pv_done[buf], ((j - 2) / 2) & 1, wc)))) break;
        const uint64_t kd = sdesc_sw128(ring_s, 16, 1024);
#pragma unroll
        for (int cb = 0; cb < kCB; ++cb) {
          if (!(ok = __all_sync(kAll, mbar_wait(&bars.k_full[cb], j & 1, wc)))) break;
          tc_fence_after();
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const uint32_t off = cb * 16384 + k4 * 32;
            mma_ss_w(tbase + 128 * buf, sdesc_advance(qd, off), sdesc_advance(kd, off), kIdS, cb + k4 > 0);
          }
          mma_commit_w(&bars.k_empty[cb]);
        }
        if (!ok) break;
        mma_commit_w(&bars.s_full[buf]);
      } else {
        // V(j) in stage 1, one 64-row half at a time: K-steps 4h .. 4h + 3 (and those of the
        // remainder of P, columns [64, 128), when the tile is split) read rows [64h, 64h + 64),
        // which are handed back as soon as they are done.
        if (!(ok = __all_sync(kAll, mbar_wait(&bars.p_full[buf], (j / 2) & 1, wc)))) break;
        const bool split = kMasked ? split_voted(bars.need[j % 2]) : split_tile(p, j, row0);
        const uint64_t vd = sdesc_sw128(ring_s + L::kTileBytes, 16384, 1024);
        const uint32_t s_tm = tbase + 128 * buf;
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          if (!(ok = __all_sync(kAll, mbar_wait(&bars.v_full[hr], j & 1, wc)))) break;
          tc_fence_after();
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const int kk = 4 * hr + k4;
            mma_ts_w(tbase + kColO, s_tm + kk * 8, sdesc_advance(vd, kk * 2048), kIdO, (j > 0 || kk > 0) ? 1u : 0u);
          }
          if (split) {
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
              const int kk = 4 * hr + k4;
              mma_ts_w(tbase + kColO, s_tm + 64 + kk * 8, sdesc_advance(vd, kk * 2048), kIdO, 1u);
            }
          }
          mma_commit_w(&bars.v_empty[hr]);
        }
        if (!ok) break;
        mma_commit_w(&bars.pv_done[buf]);
      }
    }
    mma_commit_w(&bars.fin);
    drain_wait(&bars.fin, 0, 100000000ull);
  } else if (warp < 4) {
    // ---------------------------------------------------------------- softmax
    const int r = warp * 32 + lane;
    const int i = row0 + r;
    const uint32_t o_addr = tmem_addr(tbase, warp * 32, kColO);
    const float c = p.scale_log2;
    float m = neg_inf(), l = 0.f;
    bool ok = true;
    constexpr bool masked = kMasked;
    const bool row_bc = p.lm.sl == 0, mbool = p.mask_kind == kMaskBool;
    for (int j = 0; j < nkv; ++j) {
      const int buf = j % 2;
      const int k0 = j * kBN;
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.s_full[buf], (j / 2) & 1, wc) &&
                                       (!masked || mbar_wait(&bars.mask_full, j & 1, wc)));
      if (!ok) break;
      tc_fence_after();
      const uint32_t s_addr = tmem_addr(tbase, warp * 32, 128 * buf);
      const bool need_mask = (k0 + kBN > p.Lkv) || (p.causal && k0 + kBN - 1 > row0 + p.coff);
      uint32_t sv[kBN];
#pragma unroll
      for (int q4 = 0; q4 < kBN / 32; ++q4)
        tmem_ld32(s_addr + 32 * q4, *reinterpret_cast<uint32_t(*)[32]>(&sv[32 * q4]));
      tmem_ld_wait(sv);
      int lim = min(p.Lkv - k0, kBN);
      if (p.causal) lim = min(lim, i + p.coff - k0 + 1);
      float cs = c;
      if constexpr (masked) {
        cs = mask_row<T, true>(sv, sm + L::kMaskOff, r, lane, row_bc, mbool, c, p.scale);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.mask_free);  // this warp is done with the mask tile
      }
      const float mt = need_mask ? tile_max<true>(sv, cs, lim) : tile_max<false>(sv, cs, lim);
      const float m_new = fmaxf(m, mt);
      const bool resc = m_new > m + kRescale;  // always true on the first tile (m = -inf)
      const float alpha = resc ? ex2(m - m_new) : 1.f;
      if (resc) {
        l *= alpha;
        m = m_new;
      }
      if constexpr (masked) {  // split vote, as in the D <= 128 kernel
        const float pmax = ex2(mt + (m == neg_inf() ? 0.f : -m));
        const bool wn = __any_sync(0xffffffffu, pmax > l * kSplitShare);
        if (lane == 0) {
          bars.need[j % 2][warp] = wn;
          mbar_arrive(&bars.vote);
        }
      }
      if (j > 0 && __any_sync(0xffffffffu, resc)) {
        // Rescale O once PV(j-1) has landed.
        ok = __all_sync(0xffffffffu, mbar_wait(&bars.pv_done[(j - 1) % 2], ((j - 1) / 2) & 1, wc));
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int c32 = 0; c32 < D / 32; ++c32) {
          uint32_t orr[32];
          tmem_ld32(o_addr + c32 * 32, orr);
          tmem_ld_wait(orr);
#pragma unroll
          for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
          tmem_st32(o_addr + c32 * 32, orr);
        }
        tmem_st_wait();
      }
      const float neg_m = (kMasked && m == neg_inf()) ? 0.f : -m;
      bool split;
      if constexpr (masked) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bars.vote, j & 1, wc));
        if (!ok) break;
        split = split_voted(bars.need[j % 2]);
      } else {
        split = split_tile(p, j, row0);
      }
      if (split)
        l += exp_pass_split<T>(sv, s_addr, cs, neg_m, lim);
      else if (need_mask)
        l += exp_pass<T, true>(sv, s_addr, cs, neg_m, lim, nullptr);
      else
        l += exp_pass<T, false>(sv, s_addr, cs, neg_m, lim, nullptr);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars.p_full[buf]);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars.pv_done[(nkv - 1) % 2], ((nkv - 1) / 2) & 1, wc));
    // O / l staged in the Q buffer (the last S MMA has read it), then bulk tensor stores.
    uint8_t* stage = sm + L::kQOff;
    if (ok) {
      tc_fence_after();
      const float a = fold_sink(p, h, m, l);
      const float inv = (!kMasked || l > 0.f) ? a / l : 0.f;
#pragma unroll 1
      for (int c32 = 0; c32 < D / 32; ++c32) {
        uint32_t orr[32];
        tmem_ld32(o_addr + c32 * 32, orr);
        tmem_ld_wait(orr);
        uint32_t packed[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          packed[e] = pack2<T>(__uint_as_float(orr[2 * e]) * inv, __uint_as_float(orr[2 * e + 1]) * inv);
        uint8_t* blk = stage + (c32 / 2) * 16384;
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4)
          *reinterpret_cast<uint4*>(blk + sw128_off(r, (c32 % 2) * 4 + v4)) =
              make_uint4(packed[4 * v4], packed[4 * v4 + 1], packed[4 * v4 + 2], packed[4 * v4 + 3]);
      }
      fence_async_smem();
      if (i < p.Lq && p.lse) p.lse[q_row(p, b, h, i)] = (!kMasked || l > 0.f) ? (m + __log2f(l)) * kLn2 : neg_inf();
    }
    if (named_sync_and(1, kBM, ok) && r == 0) {
      for (int cb = 0; cb < kCB; ++cb) tma_store_4d(&to, stage + cb * 16384, cb * 64, row0, h, b);
      bulk_commit();
      bulk_wait_read();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    tmem_dealloc(tbase, 512);
  }
}

template <typename T, bool kMasked>
cudaError_t tc_fwd256_m(const Problem& p, cudaStream_t s) {
  CUtensorMap tq, tk, tv, to;
  if (!make_tmap_4d(&tq, p.q, 256, p.Lq, p.Hq, p.B, p.lq, kBM) || !make_tmap_4d(&to, p.out, 256, p.Lq, p.Hq, p.B, p.lo, kBM) ||
      !make_tmap_4d(&tk, p.k, 256, p.Lkv, p.Hkv, p.B, p.lk, kBN) ||
      !make_tmap_4d(&tv, p.v, 256, p.Lkv, p.Hkv, p.B, p.lv, kBN / 2))  // V in 64-row halves
    return cudaErrorInvalidValue;
  CUtensorMap tm = tq;  // unused without a mask
  if (kMasked && !make_fwd_mask_map(&tm, p)) return cudaErrorInvalidValue;
  const int smem = Fwd256Layout<kMasked>::kBytes + 1024;
  auto kern = tc_fwd256_kernel<T, kMasked>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const unsigned nqt = (p.Lq + kBM - 1) / kBM;
  kern<<<nqt * p.Hq * p.B, k256Threads, smem, s>>>(tq, tk, tv, to, tm, p);
  return cudaGetLastError();
}

template <typename T, int D, bool kMasked>
cudaError_t tc_fwd_m(const Problem& p, cudaStream_t s) {
  CUtensorMap tq, tk, tv, to;
  if (!make_tmap_4d(&tq, p.q, D, p.Lq, p.Hq, p.B, p.lq, kBM) || !make_tmap_4d(&to, p.out, D, p.Lq, p.Hq, p.B, p.lo, kBM) ||
      !make_tmap_4d(&tk, p.k, D, p.Lkv, p.Hkv, p.B, p.lk, kBN) ||
      !make_tmap_4d(&tv, p.v, D, p.Lkv, p.Hkv, p.B, p.lv, kBN))
    return cudaErrorInvalidValue;
  CUtensorMap tm = tq;  // unused without a mask
  if (kMasked && !make_fwd_mask_map(&tm, p)) return cudaErrorInvalidValue;
  const int smem = FwdLayout<D, kMasked>::kBytes + 1024;
  auto kern = tc_fwd_kernel<T, D, kMasked>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const unsigned nqb = (p.Lq + kBM * kQTiles - 1) / (kBM * kQTiles);
  kern<<<nqb * p.Hq * p.B, kThreads, smem, s>>>(tq, tk, tv, to, tm, p);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t tc_fwd_t(const Problem& p, cudaStream_t s) {
  if constexpr (D == 256) return p.mask ? tc_fwd256_m<T, true>(p, s) : tc_fwd256_m<T, false>(p, s);
  else return p.mask ? tc_fwd_m<T, D, true>(p, s) : tc_fwd_m<T, D, false>(p, s);
}

}  // namespace

bool tensor_supported(const Problem& p, int dtype) {
  return (dtype == 1 || dtype == 2) && (p.D == 32 || p.D == 64 || p.D == 96 || p.D == 128 || p.D == 256);
}

cudaError_t launch_tc_fwd(const Problem& p, int dtype, cudaStream_t s) {
  if (dtype == 2) {
    if (p.D == 256) return tc_fwd_t<__nv_bfloat16, 256>(p, s);
    if (p.D == 128) return tc_fwd_t<__nv_bfloat16, 128>(p, s);
    if (p.D == 96) return tc_fwd_t<__nv_bfloat16, 96>(p, s);
    if (p.D == 32) return tc_fwd_t<__nv_bfloat16, 32>(p, s);
    return tc_fwd_t<__nv_bfloat16, 64>(p, s);
  }
  if (p.D == 256) return tc_fwd_t<__half, 256>(p, s);
  if (p.D == 128) return tc_fwd_t<__half, 128>(p, s);
  if (p.D == 96) return tc_fwd_t<__half, 96>(p, s);
  if (p.D == 32) return tc_fwd_t<__half, 32>(p, s);
  return tc_fwd_t<__half, 64>(p, s);
}

}  // namespace sdpa
