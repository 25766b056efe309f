// tensor_map.cu -- host-side TMA descriptors (cuTensorMapEncodeTiled, looked
// up through the runtime so the library needs no link against libcuda) and
// the per-device host state the launch paths cache.
#include <atomic>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "internal.h"

namespace mpfa {

// The CUDA driver's encoder, looked up once (function-local static: thread-safe
// initialization).
static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() {
    cudaDriverEntryPointQueryResult q;
    void* ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

// 2-D byte matrix [rows][inner_bytes] (row pitch = inner_bytes), loaded in
// boxes of box_rows full rows with the given shared-memory swizzle.
bool make_map_2d_u8(CUtensorMap* m, const void* base, uint64_t inner_bytes, uint64_t rows,
                    uint32_t box_rows, CUtensorMapSwizzle sw) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner_bytes, rows};
  cuuint64_t strides[1] = {inner_bytes};
  cuuint32_t box[2] = {(cuuint32_t)inner_bytes, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D byte matrix [rows][inner_bytes] with row pitch `pitch` bytes, moved in
// boxes of box_inner bytes x box_rows rows with the given swizzle.
bool make_map_2d_u8_box(CUtensorMap* m, const void* base, uint64_t inner_bytes, uint64_t pitch,
                        uint64_t rows, uint32_t box_inner, uint32_t box_rows,
                        CUtensorMapSwizzle sw) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner_bytes, rows};
  cuuint64_t strides[1] = {pitch};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace mpfa

// ---------------------------------------------------------------------------
// per-device host state
// ---------------------------------------------------------------------------
namespace mpfa {

namespace {
std::atomic<int> g_sm_count[kMaxDevices];
}

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

int sm_count(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return 0;
  int n = g_sm_count[dev].load(std::memory_order_acquire);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 0;
  g_sm_count[dev].store(n, std::memory_order_release);
  return n;
}

// The attribute applies per device; setting it twice (two threads racing on a
// first call) is harmless, so a flag per device is enough.
cudaError_t set_smem_once(const void* func, int bytes, int dev,
                          std::atomic<bool> (&done)[kMaxDevices]) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[dev].store(true, std::memory_order_release);
  return e;
}

}  // namespace mpfa
