// TMA tensor-map encoding (through the driver entry point, so the library
// needs no link-time dependency on libcuda) and the SM count.
#include <cuda_runtime.h>

#include <mutex>

#include "tma_host.h"

namespace moe {

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

}  // namespace

// Tiled map over a row-major tensor of `rank` dims (dims[0] contiguous),
// rows of dims[0] * elem bytes unless row_stride_bytes says otherwise; the
// box is box0 x box1 (x 1), 128-byte swizzle unless asked otherwise.
static bool encode(CUtensorMap *m, const void *ptr, bool f32, int rank, const uint64_t *dims,
                   uint64_t row_stride_bytes, uint32_t box0, uint32_t box1,
                   CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn enc = get_encoder();
  if (!enc) return false;
  const uint64_t elem = f32 ? 4 : 2;
  cuuint64_t d[3], st[2];
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) d[i] = dims[i];
  st[0] = row_stride_bytes ? row_stride_bytes : dims[0] * elem;
  if (rank == 3) st[1] = st[0] * dims[1];
  return enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank,
             const_cast<void *>(ptr), d, st, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_2d(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
                 uint32_t box_outer) {
  const uint64_t dims[2] = {inner, outer};
  return encode(m, ptr, false, 2, dims, 0, box_inner, box_outer);
}

bool make_map_2d_strided(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                         uint32_t box_inner, uint32_t box_outer) {
  const uint64_t dims[2] = {inner, outer};
  return encode(m, ptr, false, 2, dims, row_stride_bytes, box_inner, box_outer);
}

bool make_map_2d_strided_sw64(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t outer,
                              uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
  const uint64_t dims[2] = {inner, outer};
  return encode(m, ptr, false, 2, dims, row_stride_bytes, box_inner, box_outer, CU_TENSOR_MAP_SWIZZLE_64B);
}

bool make_map_3d(CUtensorMap *m, const void *ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box0,
                 uint32_t box1) {
  const uint64_t dims[3] = {d0, d1, d2};
  return encode(m, ptr, false, 3, dims, 0, box0, box1);
}

bool make_map_3d_f32(CUtensorMap *m, const void *ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box0,
                     uint32_t box1) {
  const uint64_t dims[3] = {d0, d1, d2};
  return encode(m, ptr, true, 3, dims, 0, box0, box1);
}

bool make_map_2d_f32(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
                     uint32_t box_outer) {
  const uint64_t dims[2] = {inner, outer};
  return encode(m, ptr, true, 2, dims, 0, box_inner, box_outer);
}

int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0, v = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    n = v > 0 ? v : 148;
  }
  return n;
}

}  // namespace moe
