// sdpa_bwd_noalloc: the backward with its scratch in a static device array, for callers
// that cannot hand the library a workspace (declared and documented in include/sdpa.h).
//
// The only scratch the backward needs is the fp32 vector δ = rowsum(dO∘O), one float per
// query row.  Here it lives in g_bwd_scratch, a file-scope __device__ array that every GPU
// loading this library holds until the process exits.  Host code cannot use the array's
// name as a device address, so its address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and passed to the existing backward
// as its workspace; the kernels then see an ordinary device pointer.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "../../include/sdpa.h"

namespace sdpa {
namespace {

constexpr size_t kScratchFloats = SDPA_BWD_NOALLOC_MAX_ROWS;  // 4 MiB of fp32

static __device__ __align__(256) float g_bwd_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of g_bwd_scratch on the current device; looked up on first use.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SDPA_ERR_CUDA;
  void* ptr = g_scratch_ptr[dev].load();
  if (!ptr) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ptr = g_scratch_ptr[dev].load();
    if (!ptr) {
      if (cudaGetSymbolAddress(&ptr, g_bwd_scratch) != cudaSuccess || !ptr) return SDPA_ERR_CUDA;
      g_scratch_ptr[dev].store(ptr);
    }
  }
  *out = ptr;
  return SDPA_OK;
}

}  // namespace
}  // namespace sdpa

extern "C" int sdpa_bwd_noalloc(const void* q, const void* k, const void* v, const void* out,
                                const void* dout, const float* lse, void* dq, void* dk, void* dv,
                                int B, int Hq, int Hkv, int Lq, int Lkv, int D, float scale,
                                int is_causal, int dtype, void* stream) {
  // Sizes the backward rejects: let it report its own status (nothing is launched).
  if (sdpa_bwd_workspace_size(B, Hq, Hkv, Lq, Lkv, D, dtype) == 0)
    return sdpa_bwd(q, k, v, out, dout, lse, dq, dk, dv, B, Hq, Hkv, Lq, Lkv, D, scale, is_causal,
                    dtype, nullptr, 0, stream);
  if ((double)B * Hq * Lq > (double)sdpa::kScratchFloats) return SDPA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int st = sdpa::scratch_address(&scratch);
  if (st != SDPA_OK) return st;
  return sdpa_bwd(q, k, v, out, dout, lse, dq, dk, dv, B, Hq, Hkv, Lq, Lkv, D, scale, is_causal,
                  dtype, scratch, sdpa::kScratchFloats * sizeof(float), stream);
}
