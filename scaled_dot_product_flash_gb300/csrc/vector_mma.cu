// Short-query ("vector") forward and backward for fp16/bf16 with D in {64, 128}, on
// warp-level MMAs.
//
// Lq <= 8 and G·Lq <= 32 rows per KV head: the work is a stream over the KV rows, and the
// kernel is meant to run at HBM speed.  The arithmetic per key byte (up to 32 rows × 2
// FLOP per element) is beyond what fp32 FMAs sustain at that speed, so both products use
// warp-level mma.sync (m16n8k16, fp32 accumulate); everything else is the short-sequence
// design of "[Metal] Add Flash Attention VJP for training" (section "Implementation Notes",
// item 3): per-row reductions by warp shuffles, fp32 accumulators, and shared-memory
// reductions to merge partial results.
//
// One cluster of 8 blocks per (batch, KV head); block c owns a contiguous chunk of keys,
// streamed by TMA in 64-key tiles through a 3-stage ring (each K/V byte read once).
// A forward block has four warps; with MT row blocks of 16 (MT = 1 or 2), warp (mt, kq)
// takes rows [16mt, 16mt+16) of the group and the 64/(4/MT)-key slice kq of every tile, in
// 16-key steps, keeping its own online-softmax state (row maximum, row sum, O).  (The
// backward's eight-warp layout is described above its kernel.)  At the end the
// key slices are merged in shared memory and the eight blocks of the cluster through
// distributed shared memory (log-sum-exp merge), so no workspace is needed.  Row r of the
// group is query r % Lq of head g·G + r / Lq.
#include <cooperative_groups.h>

#include "launch.h"
#include "tc_common.cuh"

namespace cg = cooperative_groups;

namespace sdpa {
namespace {
using namespace tc;

constexpr int kCs = 8;        // blocks per cluster
constexpr int kKeys = 64;     // keys per streamed tile
constexpr int kRing = 3;      // ring stages

__device__ __forceinline__ float ninf() { return __int_as_float(0xff800000); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <typename T>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1);
template <>
__device__ __forceinline__ void mma16816<__nv_bfloat16>(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma16816<__half>(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Shared-memory address of (row, 16-byte chunk) in a [64 rows x D] 16-bit tile stored by
// TMA with 128-byte swizzle as D/64 column blocks of [64 rows][64 elements].
template <int D>
__device__ __forceinline__ uint32_t swz(uint32_t tile, int row, int chunk) {
  return tile + (chunk >> 3) * (kKeys * 128) + row * 128 + (((chunk & 7) ^ (row & 7)) << 4);
}

template <int D, int MT>
struct VmLayout {
  static constexpr int kTileBytes = kKeys * D * 2;
  static constexpr int kStageBytes = 2 * kTileBytes;            // K tile, V tile
  static constexpr int kRingBytes = kRing * kStageBytes;
  static constexpr int kWarps = 4;
  static constexpr int kSlices = 4 / MT;           // key slices per tile (one per warp of a row block)
  static constexpr int kRows = 16 * MT;
  // after the loop the ring is reused for the merges:
  static constexpr int kPartO = 0;                               // [warps][16][D] fp32
  static constexpr int kPartM = kPartO + kWarps * 16 * D * 4;    // [warps][16]
  static constexpr int kPartL = kPartM + kWarps * 16 * 4;
  static constexpr int kCtaO = kPartL + kWarps * 16 * 4;         // [rows][D] fp32
  static constexpr int kCtaM = kCtaO + kRows * D * 4;            // [rows]
  static constexpr int kCtaL = kCtaM + kRows * 4;
  static constexpr int kMergeBytes = kCtaL + kRows * 4;
  static constexpr int kBytes = kRingBytes > kMergeBytes ? kRingBytes : kMergeBytes;
};

template <typename T, int D, int MT>
__global__ void __launch_bounds__(128) vec_mma_fwd_kernel(const __grid_constant__ CUtensorMap tk,
                                                              const __grid_constant__ CUtensorMap tv, Problem p,
                                                              int chunk) {
  using L = VmLayout<D, MT>;
  constexpr int kWarps = L::kWarps;
  extern __shared__ unsigned char smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full[kRing], empty[kRing];
  __shared__ int abort_flag;
  cg::cluster_group cluster = cg::this_cluster();
  const int c = (int)cluster.block_rank();
  const int b = blockIdx.z, g = blockIdx.y;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int mt = warp % MT, kq = warp / MT;  // row block, key slice
  constexpr int kSliceKeys = kKeys / L::kSlices;
  const int R = p.G * p.Lq;
  const int kv_end = p.causal ? min(p.Lkv, p.Lq + p.coff) : p.Lkv;  // query i sees keys 0..i+coff
  const int j_begin = c * chunk, j_end = min(kv_end, j_begin + chunk);
  const int ntiles = j_end > j_begin ? (j_end - j_begin + kKeys - 1) / kKeys : 0;
  const WaitCtx wc{&abort_flag, 0, p.wait_limit_ns, p.err, kKidVecFwd};

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const uint32_t ring = smem_u32(sm);
  auto issue = [&](int t) {
    const int s = t % kRing;
    mbar_arrive_expect_tx(&full[s], L::kStageBytes);
    for (int cb = 0; cb < D / 64; ++cb) {
      tma_load_4d(sm + s * L::kStageBytes + cb * (kKeys * 128), &tk, &full[s], cb * 64, j_begin + t * kKeys, g,
                  b);
      tma_load_4d(sm + s * L::kStageBytes + L::kTileBytes + cb * (kKeys * 128), &tv, &full[s], cb * 64,
                  j_begin + t * kKeys, g, b);
    }
  };
  int issued = 0;  // tiles whose loads thread 0 has issued
  if (threadIdx.x == 0)
    for (; issued < min(kRing, ntiles); ++issued) issue(issued);

  // Q fragments (rows r0 = 16mt + lane/4 and r1 = r0 + 8 of the group).
  const int r0 = 16 * mt + lane / 4, r1 = r0 + 8;
  uint32_t qf[D / 16][4];
  {
    const T* q0 = r0 < R ? row_ptr<T>(p.q, p.lq, b, g * p.G + r0 / p.Lq, r0 % p.Lq) : nullptr;
    const T* q1 = r1 < R ? row_ptr<T>(p.q, p.lq, b, g * p.G + r1 / p.Lq, r1 % p.Lq) : nullptr;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int col = 16 * kk + 2 * (lane % 4);
      qf[kk][0] = q0 ? *reinterpret_cast<const uint32_t*>(q0 + col) : 0u;
      qf[kk][1] = q1 ? *reinterpret_cast<const uint32_t*>(q1 + col) : 0u;
      qf[kk][2] = q0 ? *reinterpret_cast<const uint32_t*>(q0 + col + 8) : 0u;
      qf[kk][3] = q1 ? *reinterpret_cast<const uint32_t*>(q1 + col + 8) : 0u;
    }
  }
  const int i0 = r0 < R ? r0 % p.Lq : 0, i1 = r1 < R ? r1 % p.Lq : 0;
  const float c2 = p.scale_log2;
  const bool split = p.causal || p.Lkv <= 256;  // rows see few keys
  float m0 = ninf(), m1 = ninf(), l0 = 0.f, l1 = 0.f;
  float o[D / 8][4];
#pragma unroll
  for (int dn = 0; dn < D / 8; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;

  bool ok = true;
  for (int t = 0; t < ntiles; ++t) {
    const int s = t % kRing;
    ok = __all_sync(0xffffffffu, mbar_wait(&full[s], (t / kRing) & 1, wc));
    if (!ok) break;
    const uint32_t kt = ring + s * L::kStageBytes, vt = kt + L::kTileBytes;
#pragma unroll 1
    for (int ch = 0; ch < kSliceKeys / 16; ++ch) {
      const int koff = kq * kSliceKeys + 16 * ch;  // first key of this 16-key step within the tile
      // S = Q·Kᵀ for this warp's 16 keys (two n-tiles of 8).
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int mm = lane / 8;
        const int key = koff + (mm / 2) * 8 + (lane % 8);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(swz<D>(kt, key, 2 * kk + (mm % 2)), b0, b1, b2, b3);
        mma16816<T>(sc[0], qf[kk], b0, b1);
        mma16816<T>(sc[1], qf[kk], b2, b3);
      }
      // Scale, mask, online softmax (rows r0: elements 0,1; r1: elements 2,3).
      const int kbase = j_begin + t * kKeys + koff + 2 * (lane % 4);
      float x[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = kbase + 8 * nt + (e & 1);
          const int ir = e < 2 ? i0 : i1, rr = e < 2 ? r0 : r1;
          const bool vis = j < j_end && rr < R && (!p.causal || j <= ir + p.coff);
          x[nt][e] = vis ? sc[nt][e] * c2 : ninf();
          if (vis && p.mask) x[nt][e] += mask_log2<T>(p, row_off(p.lm, b, g * p.G + rr / p.Lq, ir) + j);
        }
      float mx0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
      float mx1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
#pragma unroll
      for (int off = 1; off <= 2; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float a0 = mn0 == ninf() ? 1.f : ex2(m0 - mn0), a1 = mn1 == ninf() ? 1.f : ex2(m1 - mn1);
      m0 = mn0;
      m1 = mn1;
      float pr[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        pr[nt][0] = mn0 == ninf() ? 0.f : ex2(x[nt][0] - mn0);
        pr[nt][1] = mn0 == ninf() ? 0.f : ex2(x[nt][1] - mn0);
        pr[nt][2] = mn1 == ninf() ? 0.f : ex2(x[nt][2] - mn1);
        pr[nt][3] = mn1 == ninf() ? 0.f : ex2(x[nt][3] - mn1);
      }
      l0 = l0 * a0 + (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]);
      l1 = l1 * a1 + (pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]);
      if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn) {
          o[dn][0] *= a0;
          o[dn][1] *= a0;
          o[dn][2] *= a1;
          o[dn][3] *= a1;
        }
      }
      // O += P·V (P as the A fragment: the C layout of S, repacked to 16 bits).  With few
      // visible keys per row |O| can be as large as |V|; then P also enters as its 16-bit
      // remainder P − head(P), so that rounding P adds nothing measurable to O's own rounding.
      const uint32_t pa[4] = {pack2<T>(pr[0][0], pr[0][1]), pack2<T>(pr[0][2], pr[0][3]),
                              pack2<T>(pr[1][0], pr[1][1]), pack2<T>(pr[1][2], pr[1][3])};
      uint32_t pl[4];
      if (split) {
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          float h0, h1;
          unpack2<T>(pa[a], h0, h1);
          pl[a] = pack2<T>(pr[a / 2][2 * (a % 2)] - h0, pr[a / 2][2 * (a % 2) + 1] - h1);
        }
      }
#pragma unroll
      for (int dn2 = 0; dn2 < D / 16; ++dn2) {
        const int mm = lane / 8;
        const int key = koff + (mm % 2) * 8 + (lane % 8);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(swz<D>(vt, key, 2 * dn2 + mm / 2), b0, b1, b2, b3);
        mma16816<T>(o[2 * dn2], pa, b0, b1);
        mma16816<T>(o[2 * dn2 + 1], pa, b2, b3);
        if (split) {
          mma16816<T>(o[2 * dn2], pl, b0, b1);
          mma16816<T>(o[2 * dn2 + 1], pl, b2, b3);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (threadIdx.x == 0 && t + kRing < ntiles) {
      if (!mbar_wait(&empty[s], (t / kRing) & 1, wc)) ok = false;
      else issue(issued++);
    }
  }
  if (threadIdx.x == 0 && (!ok || abort_flag)) {  // let copies still in flight land
    for (int t = max(0, issued - kRing); t < issued; ++t) {
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(&full[t % kRing], (t / kRing) & 1) && globaltimer() - t0 < 100000000ull) {
      }
    }
  }
  // Row sums were kept per lane: finish them across the quad.
#pragma unroll
  for (int off = 1; off <= 2; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  __syncthreads();  // every stage consumed: the ring is free for the merges
  float* part_o = reinterpret_cast<float*>(sm + L::kPartO);
  float* part_m = reinterpret_cast<float*>(sm + L::kPartM);
  float* part_l = reinterpret_cast<float*>(sm + L::kPartL);
  {
    const int lr = lane / 4;
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
      const int d = 8 * dn + 2 * (lane % 4);
      part_o[(warp * 16 + lr) * D + d] = o[dn][0];
      part_o[(warp * 16 + lr) * D + d + 1] = o[dn][1];
      part_o[(warp * 16 + lr + 8) * D + d] = o[dn][2];
      part_o[(warp * 16 + lr + 8) * D + d + 1] = o[dn][3];
    }
    if (lane % 4 == 0) {
      part_m[warp * 16 + lr] = m0;
      part_m[warp * 16 + lr + 8] = m1;
      part_l[warp * 16 + lr] = l0;
      part_l[warp * 16 + lr + 8] = l1;
    }
  }
  __syncthreads();
  // Merge the key slices of each row block: this block's partial (M, L, O).
  float* cta_o = reinterpret_cast<float*>(sm + L::kCtaO);
  float* cta_m = reinterpret_cast<float*>(sm + L::kCtaM);
  float* cta_l = reinterpret_cast<float*>(sm + L::kCtaL);
  for (int e = threadIdx.x; e < L::kRows * D; e += blockDim.x) {
    const int r = e / D, d = e % D, mtr = r / 16, lr = r % 16;
    float M = ninf();
#pragma unroll
    for (int q4 = 0; q4 < L::kSlices; ++q4) M = fmaxf(M, part_m[(mtr + MT * q4) * 16 + lr]);
    float Lsum = 0.f, O = 0.f;
#pragma unroll
    for (int q4 = 0; q4 < L::kSlices; ++q4) {
      const int w = mtr + MT * q4;
      const float mw = part_m[w * 16 + lr];
      const float wgt = mw == ninf() ? 0.f : ex2(mw - M);
      Lsum = fmaf(part_l[w * 16 + lr], wgt, Lsum);
      O = fmaf(part_o[(w * 16 + lr) * D + d], wgt, O);
    }
    cta_o[r * D + d] = O;
    if (d == 0) {
      cta_m[r] = M;
      cta_l[r] = Lsum;
    }
  }
  cluster.sync();
  // Merge the cluster's blocks; block c finalises head-dim slice [c·D/8, (c+1)·D/8).
  constexpr int kSlice = D / kCs;
  for (int e = threadIdx.x; e < R * kSlice; e += blockDim.x) {
    const int r = e / kSlice, d = c * kSlice + e % kSlice;
    float M = ninf();
    for (int cc = 0; cc < kCs; ++cc) M = fmaxf(M, cluster.map_shared_rank(cta_m, cc)[r]);
    float Lsum = 0.f, O = 0.f;
    for (int cc = 0; cc < kCs; ++cc) {
      const float mc = cluster.map_shared_rank(cta_m, cc)[r];
      const float wgt = mc == ninf() ? 0.f : ex2(mc - M);
      Lsum = fmaf(cluster.map_shared_rank(cta_l, cc)[r], wgt, Lsum);
      O = fmaf(cluster.map_shared_rank(cta_o, cc)[r * D + d], wgt, O);
    }
    const int64_t row = q_row(p, b, g * p.G + r / p.Lq, r % p.Lq);
    const float a = fold_sink(p, g * p.G + r / p.Lq, M, Lsum);
    // A row that sees no key (only a mask can do that): O = 0, lse = −inf.
    row_ptr<T>(p.out, p.lo, b, g * p.G + r / p.Lq, r % p.Lq)[d] = Elem<T>::from_f(Lsum > 0.f ? O * a / Lsum : 0.f);
    if (p.lse && d == 0) p.lse[row] = Lsum > 0.f ? (M + __log2f(Lsum)) * kLn2 : ninf();
  }
  cluster.sync();  // peers may still be reading this block's shared memory
  (void)ok;
}

template <typename T, int D, int MT>
cudaError_t vec_mma_fwd_t(const Problem& p, cudaStream_t s) {
  CUtensorMap tk, tv;
  if (!make_tmap_4d(&tk, p.k, D, p.Lkv, p.Hkv, p.B, p.lk, kKeys) || !make_tmap_4d(&tv, p.v, D, p.Lkv, p.Hkv, p.B, p.lv, kKeys))
    return cudaErrorInvalidValue;
  const int smem = VmLayout<D, MT>::kBytes + 1024;
  auto kern = vec_mma_fwd_kernel<T, D, MT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int chunk = ((p.Lkv + kCs - 1) / kCs + kKeys - 1) / kKeys * kKeys;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kCs, p.Hkv, p.B);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, p, chunk);
}

template <typename T>
cudaError_t vec_mma_fwd_any(const Problem& p, cudaStream_t s) {
  const bool two = p.G * p.Lq > 16;
  if (p.D == 128) return two ? vec_mma_fwd_t<T, 128, 2>(p, s) : vec_mma_fwd_t<T, 128, 1>(p, s);
  return two ? vec_mma_fwd_t<T, 64, 2>(p, s) : vec_mma_fwd_t<T, 64, 1>(p, s);
}


// ------------------------------------------------------------------ backward
// Eight warps; warp w takes key slice q = w % 4 (keys [16q, 16q+16) of every tile) and
// half h = w / 4.  Per 64-key tile (keys owned by this block; all G·Lq rows of the group):
//   phase A: warp (q, 1) computes dP = dO·Vᵀ and hands its fp32 fragments to warp (q, 0)
//            through shared memory (a 64-thread named barrier; the hand-off buffer lies
//            over the P and dS buffers, so the four (q, 0) warps meet at a 128-thread
//            barrier before they write P and dS); warp (q, 0) computes S = Q·Kᵀ and
//            P = exp2(c·S − log2e·lse) meanwhile, then dS = P∘(dP − δ), and writes P and
//            dS (16-bit) to shared memory;
//   phase C: warp (q, 0) computes dV = Pᵀ·dO and warp (q, 1) dK = scale·dSᵀ·Q for the
//            slice's keys, complete (every row of the group is here) and stored at once;
//            warp (q, h) adds dS·K over keys [32h, 32h+32) of the tile to its dQ partial
//            for dims [q·D/4, (q+1)·D/4), kept in registers across tiles.
// The two key halves' dQ partials and the cluster's blocks are summed through distributed
// shared memory, in a fixed order.  Splitting each slice over two warps doubles the warps
// that hide the shared-memory and MMA latencies of a tile.  The K/V ring has three stages
// with up to 16 rows and two with 32, the most that keeps two blocks on an SM.
constexpr int kBwdWarps = 8;

// Named barrier 1 + q (immediate ids, so the block reserves six barriers, not sixteen)
// between the two warps of key slice q: the dP warp arrives, the P warp waits.
template <bool kSync>
__device__ __forceinline__ void pair_bar(int q) {
#define SDPA_PAIR_BAR(ID)                                                  \
  if (kSync) asm volatile("bar.sync " #ID ", 64;" ::: "memory");           \
  else asm volatile("bar.arrive " #ID ", 64;" ::: "memory");
  switch (q) {
    case 0: SDPA_PAIR_BAR(1) break;
    case 1: SDPA_PAIR_BAR(2) break;
    case 2: SDPA_PAIR_BAR(3) break;
    default: SDPA_PAIR_BAR(4) break;
  }
#undef SDPA_PAIR_BAR
}
// Named barrier 5: the four P warps (w < 4).
__device__ __forceinline__ void p_warps_bar() { asm volatile("bar.sync 5, 128;" ::: "memory"); }

template <int D, int MT>
struct VbLayout {
  static constexpr int kRing = MT == 1 ? 3 : 2;           // K/V ring stages
  static constexpr int kTileBytes = kKeys * D * 2;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kRows = 16 * MT;
  static constexpr int kRowStride = (D + 8) * 2;          // padded: conflict-free ldmatrix
  static constexpr int kPStride = (kKeys + 8) * 2;
  static constexpr int kQ = kRing * kStageBytes;          // [rows][D+8] 16-bit
  static constexpr int kDo = kQ + kRows * kRowStride;
  static constexpr int kP = kDo + kRows * kRowStride;     // [rows][64+8] 16-bit
  static constexpr int kDs = kP + kRows * kPStride;
  static constexpr int kVec = kDs + kRows * kPStride;     // nlse2[rows], ndelta[rows]
  static constexpr int kBytes = kVec + 2 * kRows * 4;
  static constexpr int kDpFrag = MT * 2 * 4 * 32;         // fp32 dP fragments of one key slice
  static constexpr int kDp = kP;                          // [4 slices][MT][2][4][32 lanes] fp32, over P and dS
  static constexpr int kDq = 0;                           // after the loop: [2 halves][rows][D] fp32
  static_assert(4 * kDpFrag * 4 <= 2 * kRows * kPStride, "dP hand-off must fit over P and dS");
  static_assert(2 * kRows * D * 4 <= kRing * kStageBytes, "dQ merge buffer must fit in the ring");
  // dynamic bytes + alignment slack + the 1 KB the SM reserves per block + static barriers
  static_assert(2 * (kBytes + 1024 + 1024 + 64) <= 233472, "two blocks per SM");
};

template <typename T, int D, int MT>
__global__ void __launch_bounds__(256, 2) vec_mma_bwd_kernel(const __grid_constant__ CUtensorMap tk,
                                                         const __grid_constant__ CUtensorMap tv, Problem p,
                                                         int chunk) {
  using L = VbLayout<D, MT>;
  constexpr int kWarps = kBwdWarps;
  extern __shared__ unsigned char smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int kBwdRing = L::kRing;
  __shared__ uint64_t full[kBwdRing], empty[kBwdRing];
  __shared__ int abort_flag;
  cg::cluster_group cluster = cg::this_cluster();
  const int c = (int)cluster.block_rank();
  const int b = blockIdx.z, g = blockIdx.y;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int q4 = warp % 4, half = warp / 4;  // key slice, and S/P/dV (0) or dP/dK (1)
  const int R = p.G * p.Lq;
  const int kv_end = p.causal ? min(p.Lkv, p.Lq + p.coff) : p.Lkv;
  const int j_begin = c * chunk, j_own_end = min(p.Lkv, j_begin + chunk);
  const int j_end = min(kv_end, j_own_end);
  const int ntiles = j_end > j_begin ? (j_end - j_begin + kKeys - 1) / kKeys : 0;
  const WaitCtx wc{&abort_flag, 0, p.wait_limit_ns, p.err, kKidVecBwd};
  const uint32_t ring = smem_u32(sm);
  const uint32_t qs = smem_u32(sm + L::kQ), dos = smem_u32(sm + L::kDo);
  const uint32_t ps = smem_u32(sm + L::kP), dss = smem_u32(sm + L::kDs);
  float* nlse2 = reinterpret_cast<float*>(sm + L::kVec);
  float* ndelta = nlse2 + L::kRows;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < kBwdRing; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  auto issue = [&](int t) {
    const int s = t % kBwdRing;
    mbar_arrive_expect_tx(&full[s], L::kStageBytes);
    for (int cb = 0; cb < D / 64; ++cb) {
      tma_load_4d(sm + s * L::kStageBytes + cb * (kKeys * 128), &tk, &full[s], cb * 64, j_begin + t * kKeys, g,
                  b);
      tma_load_4d(sm + s * L::kStageBytes + L::kTileBytes + cb * (kKeys * 128), &tv, &full[s], cb * 64,
                  j_begin + t * kKeys, g, b);
    }
  };
  int issued = 0;
  if (threadIdx.x == 0)
    for (; issued < min(kBwdRing, ntiles); ++issued) issue(issued);

  // Stage Q and dO (zero rows past R); δ_r = Σ_d dO·O and −log2e·lse per row.
  {
    for (int e = threadIdx.x; e < L::kRows * (D / 2); e += blockDim.x) {
      const int r = e / (D / 2), d = 2 * (e % (D / 2));
      uint32_t qv = 0u, dv = 0u;
      if (r < R) {
        const int h2 = g * p.G + r / p.Lq, i2 = r % p.Lq;
        qv = *reinterpret_cast<const uint32_t*>(row_ptr<T>(p.q, p.lq, b, h2, i2) + d);
        dv = *reinterpret_cast<const uint32_t*>(row_ptr<T>(p.dout, p.ldo, b, h2, i2) + d);
      }
      *reinterpret_cast<uint32_t*>(sm + L::kQ + r * L::kRowStride + d * 2) = qv;
      *reinterpret_cast<uint32_t*>(sm + L::kDo + r * L::kRowStride + d * 2) = dv;
    }
    for (int r = warp; r < L::kRows; r += kWarps) {
      float acc = 0.f, nl = -__int_as_float(0x7f800000);
      if (r < R) {
        const int h2 = g * p.G + r / p.Lq, i2 = r % p.Lq;
        const int64_t row = q_row(p, b, h2, i2);
        const T* op = row_ptr<T>(p.o, p.lo, b, h2, i2);
        const T* dop = row_ptr<T>(p.dout, p.ldo, b, h2, i2);
        for (int d = lane; d < D; d += 32) acc = fmaf(Elem<T>::to_f(op[d]), Elem<T>::to_f(dop[d]), acc);
        const float l = p.lse[row];
        nl = l == ninf() ? ninf() : -l * kLog2e;  // no visible key: P = 0
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (lane == 0) {
        ndelta[r] = -acc;
        nlse2[r] = nl;
      }
    }
  }
  __syncthreads();

  const float c2 = p.scale_log2;
  constexpr int kDqTiles = D / 32;  // n-tiles of 8 dims in this warp's quarter of D
  float dq[MT][kDqTiles][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < kDqTiles; ++nt) dq[mt][nt][0] = dq[mt][nt][1] = dq[mt][nt][2] = dq[mt][nt][3] = 0.f;
  T* dkg = row_ptr<T>(p.dk, p.ldk, b, g, 0);
  T* dvg = row_ptr<T>(p.dv, p.ldv, b, g, 0);
  const int mm = lane / 8;

  bool ok = true;
  for (int t = 0; t < ntiles; ++t) {
    const int s = t % kBwdRing;
    ok = __all_sync(0xffffffffu, mbar_wait(&full[s], (t / kBwdRing) & 1, wc));
    // every warp leaves together: a warp of a key slice must not wait at the pair barrier
    // for a partner that gave up
    if (__syncthreads_or(!ok)) {
      ok = false;
      break;
    }
    const uint32_t kt = ring + s * L::kStageBytes, vt = kt + L::kTileBytes;
    const int tile_key0 = j_begin + t * kKeys;
    // ---- phase A: warp (q, 0) S and P, warp (q, 1) dP, for keys [16q, 16q+16), all rows
    float* dpf = reinterpret_cast<float*>(sm + L::kDp) + q4 * L::kDpFrag;
    float acc2[MT][2][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) acc2[mt][nt][0] = acc2[mt][nt][1] = acc2[mt][nt][2] = acc2[mt][nt][3] = 0.f;
      const uint32_t a_s = half == 0 ? qs : dos, b_t = half == 0 ? kt : vt;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int arow = 16 * mt + (mm % 2) * 8 + (lane % 8), acol = 16 * kk + (mm / 2) * 8;
        uint32_t a[4];
        ldsm_x4(a_s + arow * L::kRowStride + acol * 2, a[0], a[1], a[2], a[3]);
        const int key = 16 * q4 + (mm / 2) * 8 + (lane % 8);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(swz<D>(b_t, key, 2 * kk + (mm % 2)), b0, b1, b2, b3);
        mma16816<T>(acc2[mt][0], a, b0, b1);
        mma16816<T>(acc2[mt][1], a, b2, b3);
      }
    }
    if (half == 1) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) dpf[((mt * 2 + nt) * 4 + e) * 32 + lane] = acc2[mt][nt][e];
      pair_bar<false>(q4);
    } else {
      // P from S in place, while the partner warp finishes dP
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int ra = 16 * mt + lane / 4, rb = ra + 8;
        const float nla = nlse2[ra], nlb = nlse2[rb];
        const int ia = ra < R ? ra % p.Lq : 0, ib = rb < R ? rb % p.Lq : 0;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int kl = 16 * q4 + 8 * nt + 2 * (lane % 4);  // key within the tile
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = tile_key0 + kl + (e & 1);
            const bool first = e < 2;
            const bool vis = j < j_end && (!p.causal || j <= (first ? ia : ib) + p.coff);
            const float sc = acc2[mt][nt][e];
            float x = fmaf(sc, c2, first ? nla : nlb);
            if (vis && p.mask && (first ? ra : rb) < R) {
              const int rr = first ? ra : rb;
              const float mv = mask_log2<T>(p, row_off(p.lm, b, g * p.G + rr / p.Lq, rr % p.Lq) + j);
              x = fmaf(sc, c2, mv) + (first ? nla : nlb);
            }
            acc2[mt][nt][e] = vis ? ex2(x) : 0.f;
          }
        }
      }
      pair_bar<true>(q4);
      float dsv[MT][2][4];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int ra = 16 * mt + lane / 4, rb = ra + 8;
        const float nda = ndelta[ra], ndb = ndelta[rb];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dsv[mt][nt][e] =
                acc2[mt][nt][e] * (dpf[((mt * 2 + nt) * 4 + e) * 32 + lane] + (e < 2 ? nda : ndb));
      }
      p_warps_bar();  // every P warp has read its dP: P and dS may now overwrite the hand-off
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int ra = 16 * mt + lane / 4, rb = ra + 8;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int kl = 16 * q4 + 8 * nt + 2 * (lane % 4);
          const float* pv = acc2[mt][nt];
          const float* ds = dsv[mt][nt];
          *reinterpret_cast<uint32_t*>(sm + L::kP + ra * L::kPStride + kl * 2) = pack2<T>(pv[0], pv[1]);
          *reinterpret_cast<uint32_t*>(sm + L::kP + rb * L::kPStride + kl * 2) = pack2<T>(pv[2], pv[3]);
          *reinterpret_cast<uint32_t*>(sm + L::kDs + ra * L::kPStride + kl * 2) = pack2<T>(ds[0], ds[1]);
          *reinterpret_cast<uint32_t*>(sm + L::kDs + rb * L::kPStride + kl * 2) = pack2<T>(ds[2], ds[3]);
        }
      }
    }
    __syncthreads();
    // ---- phase C (i): warp (q, 0) dV = Pᵀ·dO, warp (q, 1) dK = scale·dSᵀ·Q, keys [16q, 16q+16)
    uint32_t pk[D / 8][2];  // the result as 16-bit pairs: [8-dim block][key row lane/4, +8]
    {
      const int which = half;
      const uint32_t a_s = which == 0 ? ps : dss;
      const uint32_t b_s = which == 0 ? dos : qs;
      float acc[D / 8][4];
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) acc[dn][0] = acc[dn][1] = acc[dn][2] = acc[dn][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < MT; ++ks) {
        uint32_t a[4];
        const int prow = 16 * ks + (mm / 2) * 8 + (lane % 8), pcol = 16 * q4 + (mm % 2) * 8;
        ldsm_x4_t(a_s + prow * L::kPStride + pcol * 2, a[0], a[1], a[2], a[3]);
#pragma unroll
        for (int dn2 = 0; dn2 < D / 16; ++dn2) {
          const int brow = 16 * ks + (mm % 2) * 8 + (lane % 8), bcol = 16 * dn2 + (mm / 2) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(b_s + brow * L::kRowStride + bcol * 2, b0, b1, b2, b3);
          mma16816<T>(acc[2 * dn2], a, b0, b1);
          mma16816<T>(acc[2 * dn2 + 1], a, b2, b3);
        }
      }
      const float mul = which == 0 ? 1.f : p.scale;
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) {
        pk[dn][0] = pack2<T>(acc[dn][0] * mul, acc[dn][1] * mul);
        pk[dn][1] = pack2<T>(acc[dn][2] * mul, acc[dn][3] * mul);
      }
    }
    // ---- phase C (ii): dQ[:, q·D/4 : (q+1)·D/4) += dS·K over keys [32h, 32h+32) of the tile
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
      for (int k2 = 0; k2 < kKeys / 32; ++k2) {
        const int kk = (kKeys / 32) * half + k2;
        uint32_t a[4];
        const int arow = 16 * mt + (mm % 2) * 8 + (lane % 8), acol = 16 * kk + (mm / 2) * 8;
        ldsm_x4(dss + arow * L::kPStride + acol * 2, a[0], a[1], a[2], a[3]);
#pragma unroll
        for (int np = 0; np < kDqTiles / 2; ++np) {
          const int key = 16 * kk + (mm % 2) * 8 + (lane % 8);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(swz<D>(kt, key, (q4 * D / 4) / 8 + 2 * np + mm / 2), b0, b1, b2, b3);
          mma16816<T>(dq[mt][2 * np], a, b0, b1);
          mma16816<T>(dq[mt][2 * np + 1], a, b2, b3);
        }
      }
    }
    // ---- phase C (iii): once every warp is done with this stage's K and V, each warp
    // stages its 16 rows of dV (over V) or dK (over K), 16-byte block c of row r at block
    // c ^ (r % 8) (conflict-free fragment writes), and stores whole rows with 16-byte stores.
    __syncthreads();
    {
      uint8_t* stg = sm + s * L::kStageBytes + (half == 0 ? L::kTileBytes : 0) + q4 * 16 * (D * 2);
      const int r0 = lane / 4, r1 = r0 + 8, cb = (lane % 4) * 4;
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) {
        *reinterpret_cast<uint32_t*>(stg + r0 * (D * 2) + ((dn ^ (r0 & 7)) * 16) + cb) = pk[dn][0];
        *reinterpret_cast<uint32_t*>(stg + r1 * (D * 2) + ((dn ^ (r1 & 7)) * 16) + cb) = pk[dn][1];
      }
      __syncwarp();
      T* dst = half == 0 ? dvg : dkg;
      const int64_t rs = half == 0 ? p.ldv.sl : p.ldk.sl;
      constexpr int kBlocks = D / 8;        // 16-byte blocks per row
      constexpr int kRowsPer = 32 / kBlocks;
      const int ch = lane % kBlocks;
#pragma unroll
      for (int r = lane / kBlocks; r < 16; r += kRowsPer) {
        const int j = tile_key0 + 16 * q4 + r;
        const uint4 v = *reinterpret_cast<const uint4*>(stg + r * (D * 2) + ((ch ^ (r & 7)) * 16));
        if (j < j_own_end) *reinterpret_cast<uint4*>(dst + (int64_t)j * rs + ch * 8) = v;
      }
      fence_async_smem();  // these generic-proxy writes come before the next tile's TMA write here
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (threadIdx.x == 0 && t + kBwdRing < ntiles) {
      if (!mbar_wait(&empty[s], (t / kBwdRing) & 1, wc)) ok = false;
      else issue(issued++);
    }
    // no barrier here: the last reads of P and dS came before the staging barrier, and the
    // next tile starts with a block-wide vote
  }
  if (threadIdx.x == 0 && (!ok || abort_flag)) {  // let copies still in flight land
    for (int t = max(0, issued - kBwdRing); t < issued; ++t) {
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(&full[t % kBwdRing], (t / kBwdRing) & 1) && globaltimer() - t0 < 100000000ull) {
      }
    }
  }
  // Keys this block owns that no query can see (causal, j >= Lq + coff) get zero gradients.
  for (int64_t e = (int64_t)max(j_begin + ntiles * kKeys, j_begin) * D + threadIdx.x; e < (int64_t)j_own_end * D;
       e += blockDim.x) {
    const int64_t jj = e / D, d = e % D;
    dkg[jj * p.ldk.sl + d] = Elem<T>::from_f(0.f);
    dvg[jj * p.ldv.sl + d] = Elem<T>::from_f(0.f);
  }
  __syncthreads();  // the ring is free: reuse it for the two dQ partials of this block
  float* cta_dq = reinterpret_cast<float*>(sm + L::kDq);
  float* my_dq = cta_dq + half * (L::kRows * D);
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < kDqTiles; ++nt) {
      const int r = 16 * mt + lane / 4, d = q4 * D / 4 + 8 * nt + 2 * (lane % 4);
      my_dq[r * D + d] = dq[mt][nt][0];
      my_dq[r * D + d + 1] = dq[mt][nt][1];
      my_dq[(r + 8) * D + d] = dq[mt][nt][2];
      my_dq[(r + 8) * D + d + 1] = dq[mt][nt][3];
    }
  cluster.sync();
  constexpr int kSlice = D / kCs;
  for (int e = threadIdx.x; e < R * kSlice; e += blockDim.x) {
    const int r = e / kSlice, d = c * kSlice + e % kSlice;
    float acc = 0.f;
    for (int cc = 0; cc < kCs; ++cc) {
      const float* src = cluster.map_shared_rank(cta_dq, cc);
      acc += src[r * D + d];
      acc += src[L::kRows * D + r * D + d];
    }
    row_ptr<T>(p.dq, p.ldq, b, g * p.G + r / p.Lq, r % p.Lq)[d] = Elem<T>::from_f(acc * p.scale);
  }
  cluster.sync();
}

template <typename T, int D, int MT>
cudaError_t vec_mma_bwd_t(const Problem& p, cudaStream_t s) {
  CUtensorMap tk, tv;
  if (!make_tmap_4d(&tk, p.k, D, p.Lkv, p.Hkv, p.B, p.lk, kKeys) || !make_tmap_4d(&tv, p.v, D, p.Lkv, p.Hkv, p.B, p.lv, kKeys))
    return cudaErrorInvalidValue;
  const int smem = VbLayout<D, MT>::kBytes + 1024;
  auto kern = vec_mma_bwd_kernel<T, D, MT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int chunk = ((p.Lkv + kCs - 1) / kCs + kKeys - 1) / kKeys * kKeys;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kCs, p.Hkv, p.B);
  cfg.blockDim = dim3(32 * kBwdWarps, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, p, chunk);
}

template <typename T>
cudaError_t vec_mma_bwd_any(const Problem& p, cudaStream_t s) {
  const bool two = p.G * p.Lq > 16;
  if (p.D == 128) return two ? vec_mma_bwd_t<T, 128, 2>(p, s) : vec_mma_bwd_t<T, 128, 1>(p, s);
  return two ? vec_mma_bwd_t<T, 64, 2>(p, s) : vec_mma_bwd_t<T, 64, 1>(p, s);
}

}  // namespace

bool vector_mma_supported(const Problem& p, int dtype) {
  return (dtype == 1 || dtype == 2) && (p.D == 64 || p.D == 128) && p.Lq <= 8 && p.G * p.Lq <= 32;
}

cudaError_t launch_vector_mma_fwd(const Problem& p, int dtype, cudaStream_t s) {
  return dtype == 2 ? vec_mma_fwd_any<__nv_bfloat16>(p, s) : vec_mma_fwd_any<__half>(p, s);
}

cudaError_t launch_vector_mma_bwd(const Problem& p, int dtype, cudaStream_t s) {
  return dtype == 2 ? vec_mma_bwd_any<__nv_bfloat16>(p, s) : vec_mma_bwd_any<__half>(p, s);
}

}  // namespace sdpa
