// Shared device helpers: element conversion, launch parameters, error reporting.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace sdpa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Error codes written into the device error word (low 16 bits: code, high: kernel id).
enum DeviceError : unsigned {
  kDevErrNone = 0,
  kDevErrTimeout = 1,
};

// Kernel ids for the error word.
enum KernelId : unsigned {
  kKidSimtFwd = 1,
  kKidSimtDq = 2,
  kKidSimtDkdv = 3,
  kKidDelta = 4,
  kKidVecFwd = 5,
  kKidVecBwd = 6,
  kKidTcFwd = 7,
  kKidTcDq = 8,
  kKidTcDkdv = 9,
};

__device__ __forceinline__ void report_error(unsigned* err, unsigned code, unsigned kid) {
  if (err) atomicCAS(err, 0u, (kid << 16) | code);
}

// Element <-> fp32 conversion (round-to-nearest-even on the way down).
template <typename T> struct Elem;
template <> struct Elem<float> {
  static __device__ __forceinline__ float to_f(float x) { return x; }
  static __device__ __forceinline__ float from_f(float x) { return x; }
};
template <> struct Elem<__half> {
  static __device__ __forceinline__ float to_f(__half x) { return __half2float(x); }
  static __device__ __forceinline__ __half from_f(float x) { return __float2half_rn(x); }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

// Element strides of a [B, H, L, D] tensor whose D elements are contiguous.
struct Layout {
  int64_t sb, sh, sl;  // batch, head, row
};

// Sizes and pointers of one call, passed by value to every kernel.
struct Problem {
  const void* q;
  const void* k;
  const void* v;
  const void* o;     // forward output (backward input)
  const void* dout;
  void* out;         // forward output
  float* lse;        // natural-log logsumexp [B,Hq,Lq] (nullable in the forward)
  void* dq;
  void* dk;
  void* dv;
  float* delta;      // δ = rowsum(dO∘O) [B,Hq,Lq]
  const float* sinks;  // per-query-head sink logits [Hq] (natural log), or null
  float* dsinks;       // their gradients [Hq] (backward), or null
  int B, Hq, Hkv, Lq, Lkv, D;
  int G;             // Hq / Hkv
  float scale;
  float scale_log2;  // scale · log2(e)
  int causal;
  int coff;          // causal: key j is hidden from query i when j > i + coff (0 top-left,
                     // Lkv - Lq bottom-right)
  unsigned* err;     // device error word
  uint64_t wait_limit_ns;  // time limit of any single bounded wait inside a kernel
  int inject;        // test hook: 1 = the tensor-core forward never delivers its first K tile
  // Layouts of q, k, v, o (forward output / backward input), dout, dq, dk, dv.
  Layout lq, lk, lv, lo, ldo, ldq, ldk, ldv;
};

// Index of query row (b, h, i) in the contiguous [B, Hq, Lq] arrays lse and δ.
__host__ __device__ __forceinline__ int64_t q_row(const Problem& p, int b, int h, int i) {
  return ((int64_t)b * p.Hq + h) * p.Lq + i;
}
// Element offset of row (b, h, i) of a tensor with layout l.
__host__ __device__ __forceinline__ int64_t row_off(const Layout& l, int b, int h, int64_t i) {
  return (int64_t)b * l.sb + (int64_t)h * l.sh + i * l.sl;
}
// Attention sink of query head h: one more softmax entry per row with logit sinks[h] and
// a zero value vector.  Folds it into a finished row whose running maximum m and sum l are
// in the log2 domain (P = exp2(c·s − m)) and returns the factor a by which the row's
// unnormalised output must be scaled before the division by the updated l (1 without a
// sink, so the no-sink arithmetic is unchanged).  m and l then describe the row with the
// sink, so lse = ln2·(m + log2 l) includes it.  A NaN sink gives NaN outputs.
__device__ __forceinline__ float fold_sink(const Problem& p, int h, float& m, float& l) {
  if (!p.sinks) return 1.f;
  const float s2 = p.sinks[h] * kLog2e;
  if (s2 <= m) {
    l += exp2f(s2 - m);
    return 1.f;
  }
  const float a = exp2f(m - s2);
  l = fmaf(l, a, 1.f);
  m = s2;
  return a;
}

template <typename T>
__host__ __device__ __forceinline__ const T* row_ptr(const void* base, const Layout& l, int b, int h, int64_t i) {
  return static_cast<const T*>(base) + row_off(l, b, h, i);
}
template <typename T>
__host__ __device__ __forceinline__ T* row_ptr(void* base, const Layout& l, int b, int h, int64_t i) {
  return static_cast<T*>(base) + row_off(l, b, h, i);
}

}  // namespace sdpa
