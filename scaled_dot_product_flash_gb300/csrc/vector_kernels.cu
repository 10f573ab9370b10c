// Short-query ("vector") path: Lq <= 8 and G·Lq <= 32, where G = Hq / Hkv.
//
// The query side is tiny (at most 32 rows per KV head: the G query heads of a GQA group
// times Lq), so the work is a stream over the KV rows.  One thread-block cluster of kCs
// blocks serves one (batch, KV head); block c of the cluster owns a contiguous chunk of
// the keys, so each K/V byte is read from HBM exactly once.  The design follows the
// short-sequence VJP of "[Metal] Add Flash Attention VJP for training" (section
// "Implementation Notes", item 3: fp32 accumulators, shared-memory reductions), re-cut for
// this GPU: partial results of the cluster's blocks are merged through distributed shared
// memory, so neither direction needs a global workspace or atomics.
//
// Row r of the group (r < R = G·Lq) is query i = r % Lq of query head g·G + r / Lq.
// Thread layout per block: 8 warps; warp w owns head-dim slice [w·D/8, (w+1)·D/8); inside
// a warp, lane = (row r, part u) with RP/32... rows padded to RP (a power of two) and
// LPR = 32/RP lanes sharing a row's slice.  Dot products are finished with xor-shuffles
// inside the LPR lanes and with a shared-memory sum over the 8 warps.
#include <cooperative_groups.h>

#include "launch.h"

namespace cg = cooperative_groups;

namespace sdpa {
namespace {

constexpr int kCs = 8;       // blocks per cluster (portable cluster size)
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

template <int LPR>
__device__ __forceinline__ float reduce_lanes(float x) {
#pragma unroll
  for (int off = LPR / 2; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// Copy rows [r0, r0 + n) (n <= NB) of a slab of rows `rs` elements apart into a float
// tile; rows past `nrows` are zero.
template <typename T, int D, int NB>
__device__ __forceinline__ void stage_rows(float (*dst)[D], const T* src, int64_t rs, int r0, int nrows) {
  for (int e = threadIdx.x; e < NB * D; e += kThreads) {
    const int rr = e / D, d = e % D;
    const int r = r0 + rr;
    dst[rr][d] = r < nrows ? Elem<T>::to_f(src[(int64_t)r * rs + d]) : 0.f;
  }
}

template <int D>
struct VecGeom {
  static constexpr int DW = D / kWarps;  // head-dim slice per warp
};

// ------------------------------------------------------------------------ forward
template <typename T, int D, int RP>
struct VecFwdSmem {
  static constexpr int NB = 32;
  float ks[NB][D];
  float vs[NB][D];
  float spart[kWarps][RP][NB];
  float pr[RP][NB + 1];
  float alpha[RP];
  float mrow[RP];
  float lrow[RP];
  float oacc[RP][D];  // this block's unnormalised output, read by the cluster merge
};

template <typename T, int D, int RP>
__global__ void __launch_bounds__(kThreads) vec_fwd_kernel(Problem p, int chunk) {
  using S = VecFwdSmem<T, D, RP>;
  constexpr int NB = S::NB;
  constexpr int DW = VecGeom<D>::DW;
  constexpr int LPR = 32 / RP;
  constexpr int DPL = DW / LPR;
  static_assert(DPL >= 1 && DW % LPR == 0, "bad vector geometry");
  extern __shared__ __align__(16) unsigned char smem_raw[];
  S& sm = *reinterpret_cast<S*>(smem_raw);
  cg::cluster_group cluster = cg::this_cluster();
  const int c = (int)cluster.block_rank();
  const int b = blockIdx.z, g = blockIdx.y;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int r = lane / LPR, u = lane % LPR;
  const int d0 = warp * DW + u * DPL;
  const int R = p.G * p.Lq;
  const bool row_ok = r < R;
  const int hh = row_ok ? r / p.Lq : 0, i = row_ok ? r % p.Lq : 0;
  const int h = g * p.G + hh;

  float qv[DPL], ov[DPL];
  {
    const T* qp = row_ptr<T>(p.q, p.lq, b, h, i) + d0;
#pragma unroll
    for (int t = 0; t < DPL; ++t) {
      qv[t] = row_ok ? Elem<T>::to_f(qp[t]) : 0.f;
      ov[t] = 0.f;
    }
  }
  if (threadIdx.x < RP) {
    sm.mrow[threadIdx.x] = neg_inf();
    sm.lrow[threadIdx.x] = 0.f;
  }
  int kv_end = p.Lkv;
  if (p.causal) kv_end = min(p.Lkv, p.Lq + p.coff);  // query i sees keys 0..i+coff only
  const int j_begin = c * chunk, j_end = min(kv_end, j_begin + chunk);
  const T* kp = row_ptr<T>(p.k, p.lk, b, g, 0);
  const T* vp = row_ptr<T>(p.v, p.lv, b, g, 0);

  for (int j0 = j_begin; j0 < j_end; j0 += NB) {
    __syncthreads();
    stage_rows<T, D, NB>(sm.ks, kp, p.lk.sl, j0, j_end);
    stage_rows<T, D, NB>(sm.vs, vp, p.lv.sl, j0, j_end);
    __syncthreads();
    // Phase 1: partial scores over this warp's head-dim slice.
#pragma unroll 4
    for (int jj = 0; jj < NB; ++jj) {
      float acc = 0.f;
#pragma unroll
      for (int t = 0; t < DPL; ++t) acc = fmaf(qv[t], sm.ks[jj][d0 + t], acc);
      acc = reduce_lanes<LPR>(acc);
      if (u == 0) sm.spart[warp][r][jj] = acc;
    }
    __syncthreads();
    // Phase 2: finish scores, online softmax per row (8 threads per row, 4 keys each).
    if (threadIdx.x < RP * 8) {
      const int r2 = threadIdx.x / 8, part = threadIdx.x % 8;
      const int i2 = r2 < R ? r2 % p.Lq : 0;
      float s[NB / 8];
      float bmax = neg_inf();
#pragma unroll
      for (int e = 0; e < NB / 8; ++e) {
        const int jj = part * (NB / 8) + e;
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) acc += sm.spart[w][r2][jj];
        const int j = j0 + jj;
        const bool vis = r2 < R && j < j_end && (!p.causal || j <= i2 + p.coff);
        s[e] = vis ? acc * p.scale_log2 : neg_inf();
        if (vis && p.mask) s[e] += mask_log2<T>(p, row_off(p.lm, b, g * p.G + r2 / p.Lq, i2) + j);
        bmax = fmaxf(bmax, s[e]);
      }
#pragma unroll
      for (int off = 4; off > 0; off >>= 1) bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, off));
      const float m_old = sm.mrow[r2];
      const float m_new = fmaxf(m_old, bmax);
      float sum = 0.f;
#pragma unroll
      for (int e = 0; e < NB / 8; ++e) {
        const float pe = m_new == neg_inf() ? 0.f : exp2f(s[e] - m_new);
        sm.pr[r2][part * (NB / 8) + e] = pe;
        sum += pe;
      }
#pragma unroll
      for (int off = 4; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      __syncwarp();
      if (part == 0) {
        const float a = m_new == neg_inf() ? 1.f : exp2f(m_old - m_new);
        sm.alpha[r2] = a;
        sm.lrow[r2] = sm.lrow[r2] * a + sum;
        sm.mrow[r2] = m_new;
      }
    }
    __syncthreads();
    // Phase 3: rescale and accumulate this lane's slice of the output row.
    {
      const float a = sm.alpha[r];
#pragma unroll
      for (int t = 0; t < DPL; ++t) ov[t] *= a;
#pragma unroll 4
      for (int jj = 0; jj < NB; ++jj) {
        const float pj = sm.pr[r][jj];
#pragma unroll
        for (int t = 0; t < DPL; ++t) ov[t] = fmaf(pj, sm.vs[jj][d0 + t], ov[t]);
      }
    }
  }
  // Publish this block's partial state, then merge across the cluster.
#pragma unroll
  for (int t = 0; t < DPL; ++t) sm.oacc[r][d0 + t] = ov[t];
  cluster.sync();
  constexpr int kSlice = D / kCs;  // head-dim slice this block finalises
  for (int e = threadIdx.x; e < RP * kSlice; e += kThreads) {
    const int r2 = e / kSlice, d = c * kSlice + e % kSlice;
    if (r2 >= R) continue;
    float M = neg_inf();
    for (int cc = 0; cc < kCs; ++cc) M = fmaxf(M, cluster.map_shared_rank(&sm, cc)->mrow[r2]);
    float L = 0.f, O = 0.f;
    for (int cc = 0; cc < kCs; ++cc) {
      const S* peer = cluster.map_shared_rank(&sm, cc);
      const float mc = peer->mrow[r2];
      const float wgt = mc == neg_inf() ? 0.f : exp2f(mc - M);
      L = fmaf(peer->lrow[r2], wgt, L);
      O = fmaf(peer->oacc[r2][d], wgt, O);
    }
    const int hh2 = r2 / p.Lq, i2 = r2 % p.Lq;
    const int64_t row = q_row(p, b, g * p.G + hh2, i2);
    const float a = fold_sink(p, g * p.G + hh2, M, L);
    // A row that sees no key (only a mask can do that): O = 0, lse = −inf.
    row_ptr<T>(p.out, p.lo, b, g * p.G + hh2, i2)[d] = Elem<T>::from_f(L > 0.f ? O * a / L : 0.f);
    if (p.lse && d == 0) p.lse[row] = L > 0.f ? (M + log2f(L)) * kLn2 : neg_inf();
  }
  cluster.sync();  // peers may still be reading this block's shared memory
}

// ------------------------------------------------------------------------ backward
template <typename T, int D, int RP>
struct VecBwdSmem {
  static constexpr int NB = 16;
  float ks[NB][D];
  float vs[NB][D];
  float qs[RP][D];
  float dos[RP][D];
  float spart[kWarps][RP][NB];
  float dppart[kWarps][RP][NB];
  float pr[RP][NB + 1];
  float dsr[RP][NB + 1];
  float lse2[RP];
  float delta[RP];
  float dqacc[RP][D];
};

template <typename T, int D, int RP>
__global__ void __launch_bounds__(kThreads) vec_bwd_kernel(Problem p, int chunk) {
  using S = VecBwdSmem<T, D, RP>;
  constexpr int NB = S::NB;
  constexpr int DW = VecGeom<D>::DW;
  constexpr int LPR = 32 / RP;
  constexpr int DPL = DW / LPR;
  static_assert(DPL >= 1 && DW % LPR == 0, "bad vector geometry");
  extern __shared__ __align__(16) unsigned char smem_raw[];
  S& sm = *reinterpret_cast<S*>(smem_raw);
  cg::cluster_group cluster = cg::this_cluster();
  const int c = (int)cluster.block_rank();
  const int b = blockIdx.z, g = blockIdx.y;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int r = lane / LPR, u = lane % LPR;
  const int d0 = warp * DW + u * DPL;
  const int R = p.G * p.Lq;

  // Stage this group's Q and dO rows (fp32), and compute lse2 and δ = rowsum(dO∘O).
  for (int e = threadIdx.x; e < RP * D; e += kThreads) {
    const int r2 = e / D, d = e % D;
    float qv = 0.f, dov = 0.f;
    if (r2 < R) {
      const int h2 = g * p.G + r2 / p.Lq, i2 = r2 % p.Lq;
      qv = Elem<T>::to_f(row_ptr<T>(p.q, p.lq, b, h2, i2)[d]);
      dov = Elem<T>::to_f(row_ptr<T>(p.dout, p.ldo, b, h2, i2)[d]);
    }
    sm.qs[r2][d] = qv;
    sm.dos[r2][d] = dov;
  }
  for (int r2 = warp; r2 < RP; r2 += kWarps) {
    float acc = 0.f, l2 = 0.f;
    if (r2 < R) {
      const int h2 = g * p.G + r2 / p.Lq, i2 = r2 % p.Lq;
      const int64_t row = q_row(p, b, h2, i2);
      const T* op = row_ptr<T>(p.o, p.lo, b, h2, i2);
      const T* dop = row_ptr<T>(p.dout, p.ldo, b, h2, i2);
      for (int d = lane; d < D; d += 32) acc = fmaf(Elem<T>::to_f(op[d]), Elem<T>::to_f(dop[d]), acc);
      const float l = p.lse[row];
      l2 = l == neg_inf() ? -neg_inf() : l * kLog2e;  // no visible key: +inf makes P = 0
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) {
      sm.delta[r2] = acc;
      sm.lse2[r2] = l2;
    }
  }
  __syncthreads();
  float qv[DPL], dov[DPL], dq[DPL];
#pragma unroll
  for (int t = 0; t < DPL; ++t) {
    qv[t] = sm.qs[r][d0 + t];
    dov[t] = sm.dos[r][d0 + t];
    dq[t] = 0.f;
  }
  int kv_end = p.Lkv;
  if (p.causal) kv_end = min(p.Lkv, p.Lq + p.coff);
  const int j_begin = c * chunk, j_own_end = min(p.Lkv, j_begin + chunk);
  const int j_end = min(kv_end, j_own_end);
  const T* kp = row_ptr<T>(p.k, p.lk, b, g, 0);
  const T* vp = row_ptr<T>(p.v, p.lv, b, g, 0);
  T* dkp = row_ptr<T>(p.dk, p.ldk, b, g, 0);
  T* dvp = row_ptr<T>(p.dv, p.ldv, b, g, 0);

  for (int j0 = j_begin; j0 < j_end; j0 += NB) {
    __syncthreads();
    stage_rows<T, D, NB>(sm.ks, kp, p.lk.sl, j0, j_end);
    stage_rows<T, D, NB>(sm.vs, vp, p.lv.sl, j0, j_end);
    __syncthreads();
    // Phase 1: partial S = Q·Kᵀ and dP = dO·Vᵀ over this warp's head-dim slice.
#pragma unroll 4
    for (int jj = 0; jj < NB; ++jj) {
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int t = 0; t < DPL; ++t) {
        s = fmaf(qv[t], sm.ks[jj][d0 + t], s);
        dp = fmaf(dov[t], sm.vs[jj][d0 + t], dp);
      }
      s = reduce_lanes<LPR>(s);
      dp = reduce_lanes<LPR>(dp);
      if (u == 0) {
        sm.spart[warp][r][jj] = s;
        sm.dppart[warp][r][jj] = dp;
      }
    }
    __syncthreads();
    // Phase 2: P = exp2(S·c − lse2) and dS = P ∘ (dP − δ) for every (row, key).
    for (int e = threadIdx.x; e < RP * NB; e += kThreads) {
      const int r2 = e / NB, jj = e % NB;
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        s += sm.spart[w][r2][jj];
        dp += sm.dppart[w][r2][jj];
      }
      const int j = j0 + jj;
      const bool vis = r2 < R && j < j_end && (!p.causal || j <= r2 % p.Lq + p.coff);
      const float mv = vis && p.mask ? mask_log2<T>(p, row_off(p.lm, b, g * p.G + r2 / p.Lq, r2 % p.Lq) + j) : 0.f;
      const float pe = vis ? exp2f(s * p.scale_log2 + mv - sm.lse2[r2]) : 0.f;
      sm.pr[r2][jj] = pe;
      sm.dsr[r2][jj] = pe * (dp - sm.delta[r2]);
    }
    __syncthreads();
    // Phase 3a: dQ (this lane's slice) += dS · K.
#pragma unroll 4
    for (int jj = 0; jj < NB; ++jj) {
      const float ds = sm.dsr[r][jj];
#pragma unroll
      for (int t = 0; t < DPL; ++t) dq[t] = fmaf(ds, sm.ks[jj][d0 + t], dq[t]);
    }
    // Phase 3b: this block owns keys j0..j0+NB-1 and sees every row of the group, so
    // dK_j = scale·Σ_r dS_rj q_r and dV_j = Σ_r P_rj dO_r are complete here.
    {
      constexpr int kParts = kThreads / NB;  // threads per key
      constexpr int kDims = D / kParts;
      const int jj = threadIdx.x / kParts, dd = (threadIdx.x % kParts) * kDims;
      const int j = j0 + jj;
      float dk[kDims], dv[kDims];
#pragma unroll
      for (int t = 0; t < kDims; ++t) dk[t] = dv[t] = 0.f;
      for (int r2 = 0; r2 < R; ++r2) {
        const float pe = sm.pr[r2][jj], ds = sm.dsr[r2][jj];
#pragma unroll
        for (int t = 0; t < kDims; ++t) {
          dv[t] = fmaf(pe, sm.dos[r2][dd + t], dv[t]);
          dk[t] = fmaf(ds, sm.qs[r2][dd + t], dk[t]);
        }
      }
      if (j < j_end) {
#pragma unroll
        for (int t = 0; t < kDims; ++t) {
          dkp[(int64_t)j * p.ldk.sl + dd + t] = Elem<T>::from_f(dk[t] * p.scale);
          dvp[(int64_t)j * p.ldv.sl + dd + t] = Elem<T>::from_f(dv[t]);
        }
      }
    }
  }
  // Keys this block owns but no query can see (causal, j >= Lq + coff) get zero gradients.
  for (int64_t e = (int64_t)max(j_end, j_begin) * D + threadIdx.x; e < (int64_t)j_own_end * D;
       e += kThreads) {
    const int64_t jj = e / D, d = e % D;
    dkp[jj * p.ldk.sl + d] = Elem<T>::from_f(0.f);
    dvp[jj * p.ldv.sl + d] = Elem<T>::from_f(0.f);
  }
  // Merge the dQ partials of the cluster's blocks.
#pragma unroll
  for (int t = 0; t < DPL; ++t) sm.dqacc[r][d0 + t] = dq[t];
  cluster.sync();
  constexpr int kSlice = D / kCs;
  for (int e = threadIdx.x; e < RP * kSlice; e += kThreads) {
    const int r2 = e / kSlice, d = c * kSlice + e % kSlice;
    if (r2 >= R) continue;
    float acc = 0.f;
    for (int cc = 0; cc < kCs; ++cc) acc += cluster.map_shared_rank(&sm, cc)->dqacc[r2][d];
    row_ptr<T>(p.dq, p.ldq, b, g * p.G + r2 / p.Lq, r2 % p.Lq)[d] = Elem<T>::from_f(acc * p.scale);
  }
  cluster.sync();
}

int rows_padded(const Problem& p) {
  const int R = p.G * p.Lq;
  int rp = 4;
  while (rp < R) rp *= 2;
  if ((p.D == 32 || p.D == 96) && rp < 8) rp = 8;
  return rp;
}

template <typename Kern>
cudaError_t launch_cluster(Kern kern, const Problem& p, int chunk, size_t smem, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kCs, p.Hkv, p.B);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p, chunk);
}

template <typename T, int D, int RP>
cudaError_t vec_fwd_t(const Problem& p, cudaStream_t s) {
  constexpr int NB = VecFwdSmem<T, D, RP>::NB;
  const int chunk = ((p.Lkv + kCs - 1) / kCs + NB - 1) / NB * NB;
  return launch_cluster(vec_fwd_kernel<T, D, RP>, p, chunk, sizeof(VecFwdSmem<T, D, RP>), s);
}

template <typename T, int D, int RP>
cudaError_t vec_bwd_t(const Problem& p, cudaStream_t s) {
  constexpr int NB = VecBwdSmem<T, D, RP>::NB;
  const int chunk = ((p.Lkv + kCs - 1) / kCs + NB - 1) / NB * NB;
  return launch_cluster(vec_bwd_kernel<T, D, RP>, p, chunk, sizeof(VecBwdSmem<T, D, RP>), s);
}

template <typename T, int D, bool kFwd>
cudaError_t vec_rp(const Problem& p, cudaStream_t s) {
  switch (rows_padded(p)) {
    case 4:
      if constexpr (D == 64 || D == 128) return kFwd ? vec_fwd_t<T, D, 4>(p, s) : vec_bwd_t<T, D, 4>(p, s);
      break;
    case 8: return kFwd ? vec_fwd_t<T, D, 8>(p, s) : vec_bwd_t<T, D, 8>(p, s);
    case 16: return kFwd ? vec_fwd_t<T, D, 16>(p, s) : vec_bwd_t<T, D, 16>(p, s);
    case 32: return kFwd ? vec_fwd_t<T, D, 32>(p, s) : vec_bwd_t<T, D, 32>(p, s);
  }
  return cudaErrorInvalidValue;
}

template <typename T, bool kFwd>
cudaError_t vec_d(const Problem& p, cudaStream_t s) {
  switch (p.D) {
    case 32: return vec_rp<T, 32, kFwd>(p, s);
    case 64: return vec_rp<T, 64, kFwd>(p, s);
    case 96: return vec_rp<T, 96, kFwd>(p, s);
    case 128: return vec_rp<T, 128, kFwd>(p, s);
  }
  return cudaErrorInvalidValue;
}

template <bool kFwd>
cudaError_t vec_any(const Problem& p, int dtype, cudaStream_t s) {
  switch (dtype) {
    case 0: return vec_d<float, kFwd>(p, s);
    case 1: return vec_d<__half, kFwd>(p, s);
    case 2: return vec_d<__nv_bfloat16, kFwd>(p, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

bool vector_supported(const Problem& p, int dtype) {
  (void)dtype;
  return p.Lq <= 8 && p.G * p.Lq <= 32 && p.D <= 128;  // D = 256 runs on the tiled CUDA-core path
}

cudaError_t launch_vector_fwd(const Problem& p, int dtype, cudaStream_t s) { return vec_any<true>(p, dtype, s); }
cudaError_t launch_vector_bwd(const Problem& p, int dtype, cudaStream_t s) { return vec_any<false>(p, dtype, s); }

}  // namespace sdpa
