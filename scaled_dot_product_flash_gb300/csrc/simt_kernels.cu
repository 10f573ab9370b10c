// CUDA-core (FFMA) tiled kernels: forward, dQ, dK/dV and the δ pre-pass.
//
// These serve fp32 inputs exactly (fp32 products and sums, no reduced-precision
// operands) and every head dim in {32, 64, 96, 128, 256}.  They follow the same algorithm as
// the tensor-core path: online softmax in the log2 domain for the forward, P recomputed
// from the cached logsumexp for the backward, a dQ kernel that loops over KV blocks, and
// a dK/dV kernel in which each thread block owns its KV rows and loops over the query
// heads of its GQA group, so no atomics are needed ("[Metal] Add Flash Attention VJP for
// training", section "Implementation Notes").
//
// Thread mapping: a block of 128 threads owns 32 rows; 4 neighbouring threads share a
// row, each holding every 4th element of it, and dot products are finished with two
// xor-shuffles.  K/V (or Q/dO) tiles of 32 rows (16 at D = 256) are staged in shared
// memory as fp32.
#include "launch.h"

namespace sdpa {
namespace {

constexpr int kRows = 32;
constexpr int kTpr = 4;
constexpr int kThreads = kRows * kTpr;
// Rows of K/V (or Q/dO) staged per step: 32, or 16 for D = 256 so that the two fp32 tiles
// stay within the 48 KB of static shared memory.
template <int D>
struct TileRows {
  static constexpr int value = D > 128 ? 16 : 32;
};
__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

__device__ __forceinline__ float reduce4(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  return x;
}

// Cooperative load of rows [r0, r0 + TileRows<D>) of a slab of rows `rs` elements apart
// into fp32 smem; rows at or beyond `nrows` are zero.
template <typename T, int D>
__device__ __forceinline__ void load_tile(float (*dst)[D], const T* src, int64_t rs, int r0, int nrows) {
  for (int e = threadIdx.x; e < TileRows<D>::value * D; e += kThreads) {
    const int rr = e / D, d = e % D;
    const int r = r0 + rr;
    dst[rr][d] = r < nrows ? Elem<T>::to_f(src[(int64_t)r * rs + d]) : 0.f;
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) simt_fwd_kernel(Problem p) {
  constexpr int DPT = D / kTpr;
  constexpr int kTile = TileRows<D>::value;
  __shared__ float ks[kTile][D];
  __shared__ float vs[kTile][D];
  const int r = threadIdx.x / kTpr, sub = threadIdx.x % kTpr;
  const int b = blockIdx.z, h = blockIdx.y, g = h / p.G;
  const int i = blockIdx.x * kRows + r;
  const bool valid = i < p.Lq;
  const T* qp = row_ptr<T>(p.q, p.lq, b, h, valid ? i : 0);
  const T* kp = row_ptr<T>(p.k, p.lk, b, g, 0);
  const T* vp = row_ptr<T>(p.v, p.lv, b, g, 0);

  float qr[DPT], o[DPT];
#pragma unroll
  for (int t = 0; t < DPT; ++t) {
    qr[t] = valid ? Elem<T>::to_f(qp[sub + kTpr * t]) : 0.f;
    o[t] = 0.f;
  }
  float m = neg_inf(), l = 0.f;
  int kv_end = p.Lkv;
  if (p.causal) kv_end = min(p.Lkv, (int)blockIdx.x * kRows + kRows + p.coff);
  const int64_t moff = p.mask && valid ? row_off(p.lm, b, h, i) : 0;

  for (int j0 = 0; j0 < kv_end; j0 += kTile) {
    __syncthreads();
    load_tile<T, D>(ks, kp, p.lk.sl, j0, p.Lkv);
    load_tile<T, D>(vs, vp, p.lv.sl, j0, p.Lkv);
    __syncthreads();
    float s[kTile];
    float tmax = neg_inf();
#pragma unroll
    for (int jj = 0; jj < kTile; ++jj) {
      float acc = 0.f;
#pragma unroll
      for (int t = 0; t < DPT; ++t) acc = fmaf(qr[t], ks[jj][sub + kTpr * t], acc);
      acc = reduce4(acc);
      const int j = j0 + jj;
      const bool vis = j < p.Lkv && (!p.causal || j <= i + p.coff);
      s[jj] = vis ? acc * p.scale_log2 : neg_inf();
      if (vis && p.mask && valid) s[jj] += mask_log2<T>(p, moff + j);
      tmax = fmaxf(tmax, s[jj]);
    }
    const float m_new = fmaxf(m, tmax);
    if (m_new == neg_inf()) continue;  // nothing visible yet (only a mask can do that)
    const float alpha = exp2f(m - m_new);
    l *= alpha;
#pragma unroll
    for (int t = 0; t < DPT; ++t) o[t] *= alpha;
#pragma unroll
    for (int jj = 0; jj < kTile; ++jj) {
      const float pj = exp2f(s[jj] - m_new);
      l += pj;
#pragma unroll
      for (int t = 0; t < DPT; ++t) o[t] = fmaf(pj, vs[jj][sub + kTpr * t], o[t]);
    }
    m = m_new;
  }
  if (!valid) return;
  const float a = fold_sink(p, h, m, l);
  const float inv = l > 0.f ? a / l : 0.f;  // a row that sees no key: O = 0, lse = −inf
  T* op = row_ptr<T>(p.out, p.lo, b, h, i);
#pragma unroll
  for (int t = 0; t < DPT; ++t) op[sub + kTpr * t] = Elem<T>::from_f(o[t] * inv);
  if (p.lse && sub == 0) p.lse[q_row(p, b, h, i)] = l > 0.f ? (m + log2f(l)) * kLn2 : neg_inf();
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) simt_dq_kernel(Problem p) {
  constexpr int DPT = D / kTpr;
  constexpr int kTile = TileRows<D>::value;
  __shared__ float ks[kTile][D];
  __shared__ float vs[kTile][D];
  const int r = threadIdx.x / kTpr, sub = threadIdx.x % kTpr;
  const int b = blockIdx.z, h = blockIdx.y, g = h / p.G;
  const int i = blockIdx.x * kRows + r;
  const bool valid = i < p.Lq;
  const int64_t row = q_row(p, b, h, valid ? i : 0);
  const T* qp = row_ptr<T>(p.q, p.lq, b, h, valid ? i : 0);
  const T* dop = row_ptr<T>(p.dout, p.ldo, b, h, valid ? i : 0);
  const T* kp = row_ptr<T>(p.k, p.lk, b, g, 0);
  const T* vp = row_ptr<T>(p.v, p.lv, b, g, 0);

  float qr[DPT], dor[DPT], dq[DPT];
#pragma unroll
  for (int t = 0; t < DPT; ++t) {
    qr[t] = valid ? Elem<T>::to_f(qp[sub + kTpr * t]) : 0.f;
    dor[t] = valid ? Elem<T>::to_f(dop[sub + kTpr * t]) : 0.f;
    dq[t] = 0.f;
  }
  const float lse = valid ? p.lse[row] : neg_inf();
  const bool live = lse != neg_inf();  // a valid row that sees some key
  const float lse2 = live ? lse * kLog2e : 0.f;
  const float dl = valid ? p.delta[row] : 0.f;
  const int64_t moff = p.mask && live ? row_off(p.lm, b, h, i) : 0;
  int kv_end = p.Lkv;
  if (p.causal) kv_end = min(p.Lkv, (int)blockIdx.x * kRows + kRows + p.coff);

  for (int j0 = 0; j0 < kv_end; j0 += kTile) {
    __syncthreads();
    load_tile<T, D>(ks, kp, p.lk.sl, j0, p.Lkv);
    load_tile<T, D>(vs, vp, p.lv.sl, j0, p.Lkv);
    __syncthreads();
#pragma unroll 4
    for (int jj = 0; jj < kTile; ++jj) {
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int t = 0; t < DPT; ++t) {
        s = fmaf(qr[t], ks[jj][sub + kTpr * t], s);
        dp = fmaf(dor[t], vs[jj][sub + kTpr * t], dp);
      }
      s = reduce4(s);
      dp = reduce4(dp);
      const int j = j0 + jj;
      const bool vis = live && j < p.Lkv && (!p.causal || j <= i + p.coff);
      const float mv = vis && p.mask ? mask_log2<T>(p, moff + j) : 0.f;
      const float pj = vis ? exp2f(s * p.scale_log2 + mv - lse2) : 0.f;
      const float ds = pj * (dp - dl);
#pragma unroll
      for (int t = 0; t < DPT; ++t) dq[t] = fmaf(ds, ks[jj][sub + kTpr * t], dq[t]);
    }
  }
  if (!valid) return;
  T* out = row_ptr<T>(p.dq, p.ldq, b, h, i);
#pragma unroll
  for (int t = 0; t < DPT; ++t) out[sub + kTpr * t] = Elem<T>::from_f(dq[t] * p.scale);
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) simt_dkdv_kernel(Problem p) {
  constexpr int DPT = D / kTpr;
  constexpr int kTile = TileRows<D>::value;
  __shared__ float qs[kTile][D];
  __shared__ float dos[kTile][D];
  __shared__ float lse2s[kTile];
  __shared__ float dls[kTile];
  const int r = threadIdx.x / kTpr, sub = threadIdx.x % kTpr;
  const int b = blockIdx.z, g = blockIdx.y;
  const int j = blockIdx.x * kRows + r;
  const bool valid = j < p.Lkv;
  const T* kp = row_ptr<T>(p.k, p.lk, b, g, valid ? j : 0);
  const T* vp = row_ptr<T>(p.v, p.lv, b, g, valid ? j : 0);

  float kr[DPT], vr[DPT], dk[DPT], dv[DPT];
#pragma unroll
  for (int t = 0; t < DPT; ++t) {
    kr[t] = valid ? Elem<T>::to_f(kp[sub + kTpr * t]) : 0.f;
    vr[t] = valid ? Elem<T>::to_f(vp[sub + kTpr * t]) : 0.f;
    dk[t] = 0.f;
    dv[t] = 0.f;
  }
  // Under the causal mask, queries before this block's first key see none of its keys.
  const int i_begin = p.causal ? max(0, (int)blockIdx.x * kRows - p.coff) : 0;

  for (int hh = 0; hh < p.G; ++hh) {
    const int h = g * p.G + hh;
    const T* qp = row_ptr<T>(p.q, p.lq, b, h, 0);
    const T* dop = row_ptr<T>(p.dout, p.ldo, b, h, 0);
    const float* lsep = p.lse + q_row(p, b, h, 0);
    const float* dlp = p.delta + q_row(p, b, h, 0);
    for (int i0 = i_begin; i0 < p.Lq; i0 += kTile) {
      __syncthreads();
      load_tile<T, D>(qs, qp, p.lq.sl, i0, p.Lq);
      load_tile<T, D>(dos, dop, p.ldo.sl, i0, p.Lq);
      if (threadIdx.x < kTile) {
        const int i = i0 + threadIdx.x;
        // +inf for rows that see no key (lse = −inf): their P is exp2(… − inf) = 0.
        const float l = i < p.Lq ? lsep[i] : 0.f;
        lse2s[threadIdx.x] = l == neg_inf() ? -neg_inf() : l * kLog2e;
        dls[threadIdx.x] = i < p.Lq ? dlp[i] : 0.f;
      }
      __syncthreads();
#pragma unroll 4
      for (int ii = 0; ii < kTile; ++ii) {
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int t = 0; t < DPT; ++t) {
          s = fmaf(kr[t], qs[ii][sub + kTpr * t], s);
          dp = fmaf(vr[t], dos[ii][sub + kTpr * t], dp);
        }
        s = reduce4(s);
        dp = reduce4(dp);
        const int i = i0 + ii;
        const bool vis = valid && i < p.Lq && (!p.causal || j <= i + p.coff);
        const float mv = vis && p.mask ? mask_log2<T>(p, row_off(p.lm, b, h, i) + j) : 0.f;
        const float pj = vis ? exp2f(s * p.scale_log2 + mv - lse2s[ii]) : 0.f;
        const float ds = pj * (dp - dls[ii]);
#pragma unroll
        for (int t = 0; t < DPT; ++t) {
          dv[t] = fmaf(pj, dos[ii][sub + kTpr * t], dv[t]);
          dk[t] = fmaf(ds, qs[ii][sub + kTpr * t], dk[t]);
        }
      }
    }
  }
  if (!valid) return;
  T* dkp = row_ptr<T>(p.dk, p.ldk, b, g, j);
  T* dvp = row_ptr<T>(p.dv, p.ldv, b, g, j);
#pragma unroll
  for (int t = 0; t < DPT; ++t) {
    dkp[sub + kTpr * t] = Elem<T>::from_f(dk[t] * p.scale);
    dvp[sub + kTpr * t] = Elem<T>::from_f(dv[t]);
  }
}

// δ_i = Σ_d dO_id · O_id.  16 threads per row, each reading D/16 contiguous elements,
// so a warp reads two whole rows of each tensor with coalesced loads.
constexpr int kDeltaTpr = 16;
constexpr int kDeltaThreads = 256;

template <typename T, int N>
__device__ __forceinline__ void load_elems(const T* src, float (&dst)[N]) {
  constexpr int kBytes = N * (int)sizeof(T);
  if constexpr (kBytes % 16 == 0) {
    union { uint4 u[kBytes / 16]; T e[N]; } buf;
#pragma unroll
    for (int c = 0; c < kBytes / 16; ++c) buf.u[c] = __ldg(reinterpret_cast<const uint4*>(src) + c);
#pragma unroll
    for (int n = 0; n < N; ++n) dst[n] = Elem<T>::to_f(buf.e[n]);
  } else if constexpr (kBytes % 8 == 0) {
    union { uint2 u[kBytes / 8]; T e[N]; } buf;
#pragma unroll
    for (int c = 0; c < kBytes / 8; ++c) buf.u[c] = __ldg(reinterpret_cast<const uint2*>(src) + c);
#pragma unroll
    for (int n = 0; n < N; ++n) dst[n] = Elem<T>::to_f(buf.e[n]);
  } else {
    union { unsigned u[kBytes / 4]; T e[N]; } buf;
#pragma unroll
    for (int c = 0; c < kBytes / 4; ++c) buf.u[c] = __ldg(reinterpret_cast<const unsigned*>(src) + c);
#pragma unroll
    for (int n = 0; n < N; ++n) dst[n] = Elem<T>::to_f(buf.e[n]);
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(kDeltaThreads) delta_kernel(Problem p) {
  // Grid (row blocks, Hq, B): rows i of head h of batch b, kDeltaThreads / kDeltaTpr per block.
  constexpr int EPT = D / kDeltaTpr;
  const int b = blockIdx.z, h = blockIdx.y;
  const int i = blockIdx.x * (kDeltaThreads / kDeltaTpr) + threadIdx.x / kDeltaTpr;
  const int sub = threadIdx.x % kDeltaTpr;
  float acc = 0.f;
  if (i < p.Lq) {
    float a[EPT], c[EPT];
    load_elems<T, EPT>(row_ptr<T>(p.o, p.lo, b, h, i) + sub * EPT, a);
    load_elems<T, EPT>(row_ptr<T>(p.dout, p.ldo, b, h, i) + sub * EPT, c);
#pragma unroll
    for (int n = 0; n < EPT; ++n) acc = fmaf(a[n], c[n], acc);
  }
#pragma unroll
  for (int off = kDeltaTpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (i < p.Lq && sub == 0) p.delta[q_row(p, b, h, i)] = acc;
}

// Gradient of each query head's sink logit.  The sink is one more entry of every row's
// softmax with a zero value vector, so its dP entry is zero and its dS entry is
// −p_sink·δ with p_sink = exp(sink − lse) (lse includes the sink).  Summed over the batch
// and the rows: dsink_h = −Σ_{b,i} exp(sink_h − lse_bhi)·δ_bhi.  One block per head; the
// rows are split over the threads in a fixed order and reduced by a fixed tree, so the
// result is the same bits on every run.  A sink of −inf is no sink: its gradient is 0
// (rows that saw no key have lse = −inf too, and exp(−inf − (−inf)) would be NaN).  Rows
// with lse = −inf contribute nothing.
constexpr int kSinkThreads = 256;

__device__ __forceinline__ float sink_share(float sk, float lse) {
  return lse == minus_inf() ? 0.f : expf(sk - lse);
}

__global__ void __launch_bounds__(kSinkThreads) sink_grad_kernel(Problem p) {
  const int h = blockIdx.x;
  const float sk = p.sinks[h];
  if (sk == minus_inf()) {
    if (threadIdx.x == 0) p.dsinks[h] = 0.f;
    return;
  }
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int b = 0; b < p.B; ++b) {
    const float* lse = p.lse + q_row(p, b, h, 0);
    const float* dl = p.delta + q_row(p, b, h, 0);
    int i = threadIdx.x;
    for (; i + 3 * kSinkThreads < p.Lq; i += 4 * kSinkThreads) {
#pragma unroll
      for (int u = 0; u < 4; ++u)
        acc[u] = fmaf(sink_share(sk, lse[i + u * kSinkThreads]), dl[i + u * kSinkThreads], acc[u]);
    }
    for (; i < p.Lq; i += kSinkThreads) acc[0] = fmaf(sink_share(sk, lse[i]), dl[i], acc[0]);
  }
  float t = (acc[0] + acc[1]) + (acc[2] + acc[3]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
  __shared__ float part[kSinkThreads / 32];
  if (threadIdx.x % 32 == 0) part[threadIdx.x / 32] = t;
  __syncthreads();
  if (threadIdx.x == 0) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kSinkThreads / 32; ++w) sum += part[w];
    p.dsinks[h] = -sum;
  }
}

template <typename T, int D>
cudaError_t simt_fwd_t(const Problem& p, cudaStream_t s) {
  dim3 grid((p.Lq + kRows - 1) / kRows, p.Hq, p.B);
  simt_fwd_kernel<T, D><<<grid, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t simt_dq_t(const Problem& p, cudaStream_t s) {
  dim3 gq((p.Lq + kRows - 1) / kRows, p.Hq, p.B);
  simt_dq_kernel<T, D><<<gq, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t simt_dkdv_t(const Problem& p, cudaStream_t s) {
  dim3 gk((p.Lkv + kRows - 1) / kRows, p.Hkv, p.B);
  simt_dkdv_kernel<T, D><<<gk, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t delta_t(const Problem& p, cudaStream_t s) {
  constexpr int rows_per_block = kDeltaThreads / kDeltaTpr;
  const dim3 grid((p.Lq + rows_per_block - 1) / rows_per_block, p.Hq, p.B);
  delta_kernel<T, D><<<grid, kDeltaThreads, 0, s>>>(p);
  return cudaGetLastError();
}

#define SDPA_DISPATCH(FN, p, dtype, s)                                              \
  do {                                                                              \
    switch (dtype) {                                                                \
      case 0:                                                                       \
        switch (p.D) {                                                              \
          case 32: return FN<float, 32>(p, s);                                      \
          case 64: return FN<float, 64>(p, s);                                      \
          case 96: return FN<float, 96>(p, s);                                      \
          case 128: return FN<float, 128>(p, s);                                    \
          case 256: return FN<float, 256>(p, s);                                    \
        }                                                                           \
        break;                                                                      \
      case 1:                                                                       \
        switch (p.D) {                                                              \
          case 32: return FN<__half, 32>(p, s);                                     \
          case 64: return FN<__half, 64>(p, s);                                     \
          case 96: return FN<__half, 96>(p, s);                                     \
          case 128: return FN<__half, 128>(p, s);                                   \
          case 256: return FN<__half, 256>(p, s);                                   \
        }                                                                           \
        break;                                                                      \
      case 2:                                                                       \
        switch (p.D) {                                                              \
          case 32: return FN<__nv_bfloat16, 32>(p, s);                              \
          case 64: return FN<__nv_bfloat16, 64>(p, s);                              \
          case 96: return FN<__nv_bfloat16, 96>(p, s);                              \
          case 128: return FN<__nv_bfloat16, 128>(p, s);                            \
          case 256: return FN<__nv_bfloat16, 256>(p, s);                            \
        }                                                                           \
        break;                                                                      \
    }                                                                               \
    return cudaErrorInvalidValue;                                                   \
  } while (0)

cudaError_t simt_fwd_any(const Problem& p, int dtype, cudaStream_t s) { SDPA_DISPATCH(simt_fwd_t, p, dtype, s); }
cudaError_t simt_dq_any(const Problem& p, int dtype, cudaStream_t s) { SDPA_DISPATCH(simt_dq_t, p, dtype, s); }
cudaError_t simt_dkdv_any(const Problem& p, int dtype, cudaStream_t s) { SDPA_DISPATCH(simt_dkdv_t, p, dtype, s); }
cudaError_t delta_any(const Problem& p, int dtype, cudaStream_t s) { SDPA_DISPATCH(delta_t, p, dtype, s); }

}  // namespace

cudaError_t launch_simt_fwd(const Problem& p, int dtype, cudaStream_t s) { return simt_fwd_any(p, dtype, s); }
cudaError_t launch_simt_dq(const Problem& p, int dtype, cudaStream_t s) { return simt_dq_any(p, dtype, s); }
cudaError_t launch_simt_dkdv(const Problem& p, int dtype, cudaStream_t s) { return simt_dkdv_any(p, dtype, s); }
cudaError_t launch_delta(const Problem& p, int dtype, cudaStream_t s) { return delta_any(p, dtype, s); }

cudaError_t launch_sink_grad(const Problem& p, cudaStream_t s) {
  sink_grad_kernel<<<p.Hq, kSinkThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace sdpa
