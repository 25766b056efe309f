// internal.h -- host-side launch interfaces between the C ABI (api.cu) and
// the kernel translation units.  Not part of the public ABI.
#pragma once

#include <atomic>
#include <utility>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace mpfa {

// ---------------------------------------------------------------------------
// per-device host state (keyed by device ordinal; safe for concurrent first
// calls from several host threads).  The cached values assume the device's
// primary context is not reset while the library is loaded.
// ---------------------------------------------------------------------------
constexpr int kMaxDevices = 64;

// Current device ordinal in [0, kMaxDevices), or -1.
int current_device();
// Multiprocessor count of `dev` (cached), or 0 on failure.
int sm_count(int dev);
// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) of `func` on `dev`, done
// once per device (`done` is the kernel's own per-device flag array).
cudaError_t set_smem_once(const void* func, int bytes, int dev, std::atomic<bool> (&done)[kMaxDevices]);

// Everything the two quantization passes need.  Pointers are device pointers;
// a tensor whose input pointer is null is skipped.
// Launch with programmatic stream serialization: the kernel may begin (up
// to its pdl_wait()) while the stream's previous kernel finishes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct QuantArgs {
  const void* q;  // bf16 [B][Nq][Hq][128]
  const void* k;  // bf16 [B][Nk][Hkv][128]
  const void* v;  // bf16 [B][Nk][Hkv][128]
  int B, Nq, Nk, Hq, Hkv;
  int compensate, T;
  uint8_t *qc, *qs;
  float* s_q;
  uint8_t *qbc, *qbs;
  uint8_t *kc, *ks;
  float* s_k;
  uint8_t* vc;
  float* s_v;
  // K-side smoothing (ksmooth != 0): the keys' channel means and the LSE
  // term of every query row
  int ksmooth;
  float* kbar;       // [B][Hkv][128] (output)
  float* lse_shift;  // [B][Hq][Nq] (output; null when q is null)
  // workspace
  unsigned* amax;  // [3] fp32 bit patterns of amax(Q or Q'/qbar), amax(K or K'), amax(V)
  float* qbar;     // [B][Hq][Nq/128][128] fp32 block means (compensate only)
  float* kstat;    // [B][Hkv][Nk/128][3][128]: block mean, max, min of K (ksmooth only)
  int* err;
  // full-FP4 PV ablation (launch_quantize_vt only): V^T in NVFP4 along the
  // keys, codes [B][Hkv][128][Nk/2], block scales one 1 KB tile per
  // (b, KV head, 128-key tile) in the tensor core's scale-copy order;
  // tensor scale into s_v
  uint8_t *vtc, *vts;
};

size_t quant_workspace_bytes(int B, int Nq, int Nk, int Hq, int Hkv, int compensate, int ksmooth);
cudaError_t launch_quantize(const QuantArgs& a, cudaStream_t stream);
cudaError_t launch_quantize_vt(const QuantArgs& a, cudaStream_t stream);

// Quantize-on-append into a decode cache: new rows of K and V, quantized with
// the cache's tensor scales, written at rows seqlens[b] + t.
struct AppendArgs {
  const void* k_new;  // bf16 [B][n_new][Hkv][128]
  const void* v_new;  // bf16 [B][n_new][Hkv][128]
  const int32_t* seqlens;
  int B, n_new, Hkv, Lmax;
  uint8_t *kc, *ks;
  const float* s_k;
  uint8_t* vc;
  const float* s_v;
  const float* kbar;  // [B][Hkv][128] channel means of a smoothed cache, or null
  // paged pool (see DecodeArgs), or null block_table
  const int32_t* block_table;
  int num_pages, max_pages;
  int* err;
};

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream);

struct PrefillArgs {
  const uint8_t *qc, *qs;
  const float* s_q;
  const uint8_t *qbc, *qbs;  // rank-one terms (null when compensate == 0)
  const uint8_t *kc, *ks;
  const float* s_k;
  // V codes: E4M3 [B][Hkv][N][128]; with pv4, NVFP4 V^T codes
  // [B][Hkv][128][N/2] and their block scales (vts, 1 KB per 128-key tile)
  const uint8_t* vc;
  const uint8_t* vts;
  const float* s_v;
  int B, N, Hq, Hkv, causal, compensate, T;
  int pv4;     // 1: P and V in NVFP4 (the full-FP4 PV kernel)
  void* o;     // bf16 [B][N][Hq][128]
  float* lse;  // [B][Hq][N] or null
  const float* lse_shift;  // [B][Hq][N] added to the LSE (K-side smoothing), or null
  int* err;
};

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream);

struct DecodeArgs {
  const void* q;  // bf16 [B][Hq][128]
  const uint8_t *kc, *ks;
  const float* s_k;
  const uint8_t* vc;
  const float* s_v;
  const int32_t* seqlens;
  const float* kbar;  // [B][Hkv][128] channel means of a smoothed cache, or null
  // paged pool (null block_table: contiguous [B][Hkv][Lmax] cache): cache
  // rows [num_pages][Hkv][128], block_table [B][max_pages], Lmax = 128 * max_pages
  const int32_t* block_table;
  int num_pages, max_pages;
  int B, Hq, Hkv, Lmax, compensate, T, chunk, nsplit;
  void* o;     // bf16 [B][Hq][128]
  float* lse;  // [B][Hq] or null
  // quantized query (workspace or caller buffers)
  uint8_t *qc, *qs;    // [B][Hq][64], [B][Hq][8]
  uint8_t *qbc, *qbs;  // [B][Hkv][T][64], [B][Hkv][T][8]
  float* s_q;
  unsigned* amax;      // [1]
  float* qbar;         // [B][Hkv][128]
  float* part_o;       // [B][Hq][nsplit][128]
  float* part_lse;     // [B][Hq][nsplit]
  float* q_kbar;       // [B][Hq + Hkv]: code-unit dot products with kbar (kbar only)
  int* work;           // split kernel's item counter (zeroed by the launch)
  int* err;
};

int decode_default_chunk(int B, int Hkv, int Lmax, int num_sms);
size_t decode_workspace_bytes(int B, int Hq, int Hkv, int nsplit);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

}  // namespace mpfa
