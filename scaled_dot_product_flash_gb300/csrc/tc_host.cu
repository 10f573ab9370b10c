// Host side of the tensor-core path: TMA tensor-map encoding through the driver entry
// point (no link-time dependency on libcuda).
#include <cudaTypedefs.h>

#include "tc_common.cuh"

namespace sdpa {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}
}  // namespace

bool make_tmap_4d(CUtensorMap* map, const void* base, int D, int rows, int heads, int batch, const Layout& l,
                  int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)heads, (cuuint64_t)batch};
  cuuint64_t strides[3] = {(cuuint64_t)l.sl * 2, (cuuint64_t)l.sh * 2, (cuuint64_t)l.sb * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_mask(CUtensorMap* map, const Problem& p, int elem_bytes, int box_keys, int box_rows, bool swizzle128) {
  auto fn = encode_fn();
  if (!fn) return false;
  // A dimension with stride 0 is broadcast: it gets extent 1 (coordinate 0 always) and a
  // nominal stride, since a tensor map wants every stride to be a positive multiple of 16.
  const int64_t st[3] = {p.lm.sl, p.lm.sh, p.lm.sb};
  const int64_t ext[3] = {p.Lq, p.Hq, p.B};
  cuuint64_t dims[4] = {(cuuint64_t)p.Lkv, 1, 1, 1};
  cuuint64_t strides[3];
  for (int a = 0; a < 3; ++a) {
    dims[a + 1] = st[a] == 0 ? 1 : (cuuint64_t)ext[a];
    strides[a] = st[a] == 0 ? 16 : (cuuint64_t)(st[a] * elem_bytes);
  }
  cuuint32_t box[4] = {(cuuint32_t)box_keys, (cuuint32_t)box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 4,
                  const_cast<void*>(p.mask), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace sdpa
