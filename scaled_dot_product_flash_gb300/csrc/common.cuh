// Shared device helpers: element conversion, launch parameters, error reporting.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <type_traits>

namespace sdpa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Error codes written into the device error word (low 16 bits: code, high: kernel id).
enum DeviceError : unsigned {
  kDevErrNone = 0,
  kDevErrTimeout = 1,  // a bounded wait ran out
  kDevErrLayout = 2,   // a block found its shared memory placed other than its layout assumes
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
  const void* mask;    // attention mask [B, Hq, Lq, Lkv] through layout lm, or null
  int mask_kind;       // MaskKind
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
  int num_sms;       // SMs of the device (blocks resident at once in the one-block-per-SM kernels)
  // Layouts of q, k, v, o (forward output / backward input), dout, dq, dk, dv.
  Layout lq, lk, lv, lo, ldo, ldq, ldk, ldv;
  Layout lm;           // mask strides (batch, query head, row; 0 broadcasts), keys contiguous
};

// Attention mask kinds: boolean bytes (nonzero keeps the key for that query) or additive
// values of the element type, added to scale·q·k (−inf hides the key).
enum MaskKind : int { kMaskNone = 0, kMaskBool = 1, kMaskAdd = 2 };

// Index of query row (b, h, i) in the contiguous [B, Hq, Lq] arrays lse and δ.
__host__ __device__ __forceinline__ int64_t q_row(const Problem& p, int b, int h, int i) {
  return ((int64_t)b * p.Hq + h) * p.Lq + i;
}
// Element offset of row (b, h, i) of a tensor with layout l.
__host__ __device__ __forceinline__ int64_t row_off(const Layout& l, int b, int h, int64_t i) {
  return (int64_t)b * l.sb + (int64_t)h * l.sh + i * l.sl;
}
__device__ __forceinline__ float minus_inf() { return __int_as_float(0xff800000); }


// Attention sink of query head h: one more softmax entry per row with logit sinks[h] and
// a zero value vector.  Folds it into a finished row whose running maximum m and sum l are
// in the log2 domain (P = exp2(c·s − m)) and returns the factor a by which the row's
// unnormalised output must be scaled before the division by the updated l (1 without a
// sink, so the no-sink arithmetic is unchanged).  m and l then describe the row with the
// sink, so lse = ln2·(m + log2 l) includes it.  A sink of −inf is no sink (also for a row
// that saw no key, where m = −inf too).  A NaN sink gives NaN outputs.
__device__ __forceinline__ float fold_sink(const Problem& p, int h, float& m, float& l) {
  if (!p.sinks) return 1.f;
  const float s2 = p.sinks[h] * kLog2e;
  if (s2 == minus_inf()) return 1.f;
  if (s2 <= m) {
    l += exp2f(s2 - m);
    return 1.f;
  }
  const float a = exp2f(m - s2);
  l = fmaf(l, a, 1.f);
  m = s2;
  return a;
}

// Mask term of one (query row, key) pair in the log2 domain: log2e·M, or −inf for a key a
// boolean mask hides.  `off` is the element offset of the pair in the mask.
template <typename T>
__device__ __forceinline__ float mask_log2(const Problem& p, int64_t off) {
  if (p.mask_kind == kMaskBool) return static_cast<const uint8_t*>(p.mask)[off] ? 0.f : minus_inf();
  return Elem<T>::to_f(static_cast<const T*>(p.mask)[off]) * kLog2e;
}

// Mask values of N consecutive keys of one query row as packed pairs of the 16-bit element
// type T (key 2e in the low half of word e): the additive values as stored, or 0 / −inf
// for a boolean mask.  `off` is the mask offset of the first key.  The row is read in
// 16-byte pieces, and only the pieces that hold the first n keys (the ABI requires 16-byte
// aligned rows readable up to the next multiple of 16 bytes past Lkv); the other words
// are 0.
template <typename T, int N>
__device__ __forceinline__ void mask_pairs(uint32_t (&mk)[N / 2], const Problem& p, int64_t off, int n) {
  static_assert(sizeof(T) == 2, "16-bit element types only");
#pragma unroll
  for (int e = 0; e < N / 2; ++e) mk[e] = 0u;
  if (p.mask_kind == kMaskBool) {
    constexpr uint32_t kHide = std::is_same<T, __nv_bfloat16>::value ? 0xff80u : 0xfc00u;  // −inf
    const uint4* m = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.mask) + off);
    const int pieces = (n + 15) / 16;
#pragma unroll
    for (int q = 0; q < N / 16; ++q) {
      if (q < pieces) {
        const uint4 w = __ldg(m + q);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const uint32_t word = ws[t / 2], sh = 16 * (t % 2);
          const uint32_t lo = ((word >> sh) & 0xffu) ? 0u : kHide;
          const uint32_t hi = ((word >> (sh + 8)) & 0xffu) ? 0u : kHide;
          mk[8 * q + t] = lo | (hi << 16);
        }
      }
    }
  } else {
    const uint4* m = reinterpret_cast<const uint4*>(static_cast<const T*>(p.mask) + off);
    const int pieces = (n + 7) / 8;
#pragma unroll
    for (int q = 0; q < N / 8; ++q) {
      if (q < pieces) {
        const uint4 w = __ldg(m + q);
        mk[4 * q] = w.x;
        mk[4 * q + 1] = w.y;
        mk[4 * q + 2] = w.z;
        mk[4 * q + 3] = w.w;
      }
    }
  }
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
