// Unit test of the tcgen05 building blocks (descriptors, TMA swizzle, TMEM layouts),
// compiled by tests/test_tc_selftest.py into its own small library.  One 128-thread block
// computes a 128x128 product three ways and writes the fp32 accumulator to global:
//   variant 0: C = A · Bᵀ, A [128 x 128] and B [128 x 128] both K-major in smem (S = Q Kᵀ)
//   variant 1: C = A · B,  A [128 x 128] K-major, B [128 x 128] MN-major in smem (O = P V)
//   variant 2: as 1, with A packed into tensor memory by tcgen05.st (P from TMEM)
#include "../scaled_dot_product_flash_gb300/csrc/tc_common.cuh"
#include "../scaled_dot_product_flash_gb300/csrc/tc_host.cu"

using namespace sdpa;
using namespace sdpa::tc;

__global__ void __launch_bounds__(128) selftest_kernel(const __grid_constant__ CUtensorMap map_a,
                                                       const __grid_constant__ CUtensorMap map_b,
                                                       const __nv_bfloat16* a_glob, float* out,
                                                       int variant, unsigned* err) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sa = base;           // 2 column blocks of [128][64] bf16 = 32 KB
  uint8_t* sb = base + 32768;   // 32 KB
  __shared__ uint64_t bar_load, bar_mma;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid / 32;
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&bar_load, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;
  WaitCtx w{&abort_flag, 0, 1000000000ull, err, 99};
  if (tid == 0) {
    mbar_arrive_expect_tx(&bar_load, 65536);
    for (int cb = 0; cb < 2; ++cb) {
      tma_load_4d(sa + cb * 16384, &map_a, &bar_load, cb * 64, 0, 0, 0);
      tma_load_4d(sb + cb * 16384, &map_b, &bar_load, cb * 64, 0, 0, 0);
    }
  }
  if (variant == 2) {
    // Row tid of A into TMEM columns [256, 320), two bf16 per 32-bit column.
    const __nv_bfloat16* row = a_glob + tid * 128;
    for (int c = 0; c < 4; ++c) {
      uint32_t r[16];
      for (int e = 0; e < 16; ++e) {
        float lo = __bfloat162float(row[c * 32 + 2 * e]);
        float hi = __bfloat162float(row[c * 32 + 2 * e + 1]);
        r[e] = pack2<__nv_bfloat16>(lo, hi);
      }
      tmem_st16(tmem_addr(tbase, warp * 32, 256 + c * 16), r);
    }
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  bool ok = mbar_wait(&bar_load, 0, w);
  if (ok && tid == 0) {
    tc_fence_after();
    const uint32_t a0 = smem_u32(sa), b0 = smem_u32(sb);
    if (variant == 0) {
      constexpr uint32_t id = idesc_f16(128, 128, true, false, false);
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
        mma_ss(tbase, sdesc_sw128(a0 + off, 16, 1024), sdesc_sw128(b0 + off, 16, 1024), id, kk > 0);
      }
    } else if (variant == 1) {
      constexpr uint32_t id = idesc_f16(128, 128, true, false, true);
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t aoff = (kk / 4) * 16384 + (kk % 4) * 32;
        mma_ss(tbase, sdesc_sw128(a0 + aoff, 16, 1024), sdesc_sw128(b0 + kk * 2048, 16384, 1024), id,
               kk > 0);
      }
    } else {
      constexpr uint32_t id = idesc_f16(128, 128, true, false, true);
      for (int kk = 0; kk < 8; ++kk)
        mma_ts(tbase, tbase + 256 + kk * 8, sdesc_sw128(b0 + kk * 2048, 16384, 1024), id, kk > 0);
    }
    mma_commit(&bar_mma);
  }
  __syncthreads();
  ok = ok && mbar_wait(&bar_mma, 0, w);
  tc_fence_after();
  if (ok) {
    for (int c = 0; c < 4; ++c) {
      uint32_t r[32];
      tmem_ld32(tmem_addr(tbase, warp * 32, c * 32), r);
      tmem_ld_wait();
      for (int e = 0; e < 32; ++e) out[tid * 128 + c * 32 + e] = __uint_as_float(r[e]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, 512);
}

// a, b: device bf16 [128 x 128] row-major.  out: device fp32 [128 x 128].  err: device word.
extern "C" int selftest_mma(int variant, const void* a, const void* b, float* out, unsigned* err) {
  CUtensorMap ma, mb;
  const Layout l{128 * 128, 128 * 128, 128};
  if (!make_tmap_4d(&ma, a, 128, 128, 1, 1, l, 128) || !make_tmap_4d(&mb, b, 128, 128, 1, 1, l, 128)) return 1;
  const int smem = 65536 + 1024;
  if (cudaFuncSetAttribute(selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return 2;
  selftest_kernel<<<1, 128, smem>>>(ma, mb, static_cast<const __nv_bfloat16*>(a), out, variant, err);
  if (cudaGetLastError() != cudaSuccess) return 3;
  if (cudaDeviceSynchronize() != cudaSuccess) return 4;
  return 0;
}
