// quantize_noalloc.cu -- mpfa_quantize_qkv_noalloc: the quantization entry
// point for callers that cannot allocate device memory.
//
// mpfa_quantize_qkv needs a small device workspace (three amax words and,
// with the rank-one smoothing, the fp32 block means of Q).  Some callers
// cannot provide one: a serving process whose device memory is owned by its
// own pool allocator and must not call cudaMalloc after start-up (cudaMalloc
// can also synchronize the device in the middle of a step), or an embedding
// host that hands the library only its input and output tensors.  For them
// this file keeps the workspace in a fixed, file-scope device array instead.
//
// The array is static storage of the library: every GPU that loads the
// library holds kScratchBytes of it until the process exits.  All calls on a
// device share it, and it keeps the previous call's contents; the launch
// path clears the amax words at the start of every call, and the block means
// are fully rewritten before they are read.  Two calls whose work overlaps
// on the GPU (different streams, no ordering between them) race on the
// array; order them on one stream or with events.
#include <atomic>
#include <cuda_runtime.h>

#include "mpfa.h"

namespace {

// 16 MiB of block means (32768 query blocks of 128 rows, e.g. 32 heads at
// 128K tokens) plus 256 bytes of amax words.
constexpr size_t kScratchBytes = 256 + (size_t(16) << 20);

__device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of the array for the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p) return p;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
  g_scratch_addr[dev].store(p, std::memory_order_release);
  return p;
}

}  // namespace

extern "C" mpfa_status mpfa_quantize_qkv_noalloc(
    const void* q_bf16, const void* k_bf16, const void* v_bf16, int B, int Nq, int Nk, int Hq,
    int Hkv, int d, int compensate, int T, mpfa_nvfp4* q_out, mpfa_rank1* qbar_out,
    mpfa_nvfp4* k_out, mpfa_fp8* v_out, mpfa_stream_t stream) {
  const int comp = (q_bf16 && compensate) ? 1 : 0;
  const size_t need = mpfa_quantize_workspace_size(B, q_bf16 ? Nq : 0, 0, Hq, 0, comp, 0);
  if (need == 0 || need > kScratchBytes) return MPFA_ERR_INVALID_ARG;
  void* ws = scratch_address();
  if (!ws) return MPFA_ERR_CUDA;
  return mpfa_quantize_qkv(q_bf16, k_bf16, v_bf16, B, Nq, Nk, Hq, Hkv, d, compensate, T, q_out,
                           qbar_out, k_out, v_out, nullptr, ws, kScratchBytes, stream);
}
