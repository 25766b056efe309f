// api.cu -- the C ABI declared in include/mpfa.h: argument validation, the
// device status word, workspace carving and kernel launches.
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "device.cuh"
#include "internal.h"
#include "mpfa.h"

namespace {

// Device status word: kernels record MPFA_ERR_TIMEOUT (an expired bounded
// on-chip wait) or MPFA_ERR_INVALID_ARG (a device-side argument check) here.
// One word per device (static storage, not an allocation); its address is
// looked up once per device and cached (atomically: concurrent first calls
// from several host threads are safe).
__device__ int g_status;

std::atomic<int*> g_status_ptr[mpfa::kMaxDevices];

int* status_ptr() {
  const int dev = mpfa::current_device();
  if (dev < 0) return nullptr;
  int* p = g_status_ptr[dev].load(std::memory_order_acquire);
  if (p) return p;
  void* v = nullptr;
  if (cudaGetSymbolAddress(&v, g_status) != cudaSuccess || !v) return nullptr;
  p = static_cast<int*>(v);
  g_status_ptr[dev].store(p, std::memory_order_release);
  return p;
}

// One thread waits on a shared-memory barrier that nothing arrives on; the
// bounded wait gives up after limit_ns and records MPFA_ERR_TIMEOUT.
__global__ void selftest_wait_kernel(int* err, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = mpfa::smem_u32(&bar);
  mpfa::mbar_init(b, 1);
  mpfa::fence_barrier_init();
  mpfa::mbar_wait(b, 0, err, nullptr, limit_ns);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool ok_ptr(const void* p) { return p != nullptr && aligned16(p); }

// The last CUDA runtime error this library met on the calling host thread
// (reported by mpfa_last_cuda_error).
thread_local cudaError_t g_last_cuda = cudaSuccess;

mpfa_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return MPFA_OK;
  g_last_cuda = e;
  return MPFA_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* mpfa_last_cuda_error(void) { return cudaGetErrorName(g_last_cuda); }

const char* mpfa_status_string(mpfa_status s) {
  switch (s) {
    case MPFA_OK: return "MPFA_OK";
    case MPFA_ERR_INVALID_ARG: return "MPFA_ERR_INVALID_ARG";
    case MPFA_ERR_UNSUPPORTED: return "MPFA_ERR_UNSUPPORTED";
    case MPFA_ERR_CUDA: return "MPFA_ERR_CUDA";
    case MPFA_ERR_TIMEOUT: return "MPFA_ERR_TIMEOUT";
  }
  return "MPFA_ERR_UNKNOWN";
}

size_t mpfa_quantize_workspace_size(int B, int Nq, int Nk, int Hq, int Hkv, int compensate,
                                    int ksmooth) {
  if (B < 0 || Nq < 0 || Nk < 0 || Hq < 0 || Hkv < 0) return 0;
  return mpfa::quant_workspace_bytes(B, Nq, Nk, Hq, Hkv, compensate, ksmooth);
}

mpfa_status mpfa_quantize_qkv(const void* q_bf16, const void* k_bf16, const void* v_bf16, int B,
                              int Nq, int Nk, int Hq, int Hkv, int d, int compensate, int T,
                              mpfa_nvfp4* q_out, mpfa_rank1* qbar_out, mpfa_nvfp4* k_out,
                              mpfa_fp8* v_out, const mpfa_ksmooth* ksmooth, void* workspace,
                              size_t ws_bytes, mpfa_stream_t stream) {
  if (d != 128) return MPFA_ERR_UNSUPPORTED;
  if (B <= 0) return MPFA_ERR_INVALID_ARG;
  if (!q_bf16 && !k_bf16 && !v_bf16) return MPFA_ERR_INVALID_ARG;
  mpfa::QuantArgs a = {};
  a.B = B;
  a.Nq = Nq;
  a.Nk = Nk;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.compensate = q_bf16 ? (compensate != 0) : 0;
  a.T = T;
  if (q_bf16) {
    if (Nq <= 0 || Nq % 128 || Hq <= 0 || !ok_ptr(q_bf16) || !q_out || !ok_ptr(q_out->codes) ||
        !ok_ptr(q_out->scales) || !q_out->tensor_scale)
      return MPFA_ERR_INVALID_ARG;
    if (a.compensate) {
      if (T != 1 && T != 2) return MPFA_ERR_UNSUPPORTED;
      if (!qbar_out || !ok_ptr(qbar_out->codes) || !qbar_out->scales)
        return MPFA_ERR_INVALID_ARG;
    }
    a.q = q_bf16;
    a.qc = q_out->codes;
    a.qs = q_out->scales;
    a.s_q = q_out->tensor_scale;
    if (a.compensate) {
      a.qbc = qbar_out->codes;
      a.qbs = qbar_out->scales;
    }
  } else if (q_out) {
    return MPFA_ERR_INVALID_ARG;
  }
  if (k_bf16) {
    if (Nk <= 0 || Nk % 128 || Hkv <= 0 || !ok_ptr(k_bf16) || !k_out ||
        !ok_ptr(k_out->codes) || !ok_ptr(k_out->scales) || !k_out->tensor_scale)
      return MPFA_ERR_INVALID_ARG;
    a.k = k_bf16;
    a.kc = k_out->codes;
    a.ks = k_out->scales;
    a.s_k = k_out->tensor_scale;
  } else if (k_out) {
    return MPFA_ERR_INVALID_ARG;
  }
  if (v_bf16) {
    if (Nk <= 0 || Nk % 128 || Hkv <= 0 || !ok_ptr(v_bf16) || !v_out ||
        !ok_ptr(v_out->codes) || !v_out->tensor_scale)
      return MPFA_ERR_INVALID_ARG;
    a.v = v_bf16;
    a.vc = v_out->codes;
    a.s_v = v_out->tensor_scale;
  } else if (v_out) {
    return MPFA_ERR_INVALID_ARG;
  }
  if ((q_bf16 && (uint64_t)B * Hq * Nq >= (1ull << 31)) ||
      ((k_bf16 || v_bf16) && (uint64_t)B * Hkv * Nk >= (1ull << 31)))
    return MPFA_ERR_INVALID_ARG;
  if (ksmooth) {
    // key-side smoothing needs the keys, and the LSE term needs the queries
    if (!k_bf16 || !ok_ptr(ksmooth->kbar) || (ksmooth->lse_shift && !q_bf16) ||
        (q_bf16 && Hq % Hkv))
      return MPFA_ERR_INVALID_ARG;
    a.ksmooth = 1;
    a.kbar = ksmooth->kbar;
    a.lse_shift = q_bf16 ? ksmooth->lse_shift : nullptr;
  }
  const size_t need = mpfa::quant_workspace_bytes(B, q_bf16 ? Nq : 0, k_bf16 ? Nk : 0, Hq, Hkv,
                                                  a.compensate, a.ksmooth);
  if (!ok_ptr(workspace) || ws_bytes < need) return MPFA_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.amax = reinterpret_cast<unsigned*>(ws);
  size_t off = 256;
  if (a.compensate) {
    a.qbar = reinterpret_cast<float*>(ws + off);
    off += (size_t)B * Hq * (Nq / 128) * 128 * sizeof(float);
  }
  if (a.ksmooth) a.kstat = reinterpret_cast<float*>(ws + off);
  a.err = status_ptr();
  if (!a.err) return MPFA_ERR_CUDA;
  return from_cuda(mpfa::launch_quantize(a, reinterpret_cast<cudaStream_t>(stream)));
}

mpfa_status mpfa_quantize_v_fp4(const void* v_bf16, int B, int Nk, int Hkv, int d,
                                mpfa_nvfp4* vt_out, void* workspace, size_t ws_bytes,
                                mpfa_stream_t stream) {
  if (d != 128) return MPFA_ERR_UNSUPPORTED;
  if (B <= 0 || Nk <= 0 || Nk % 128 || Hkv <= 0 || !ok_ptr(v_bf16) || !vt_out ||
      !ok_ptr(vt_out->codes) || !ok_ptr(vt_out->scales) || !vt_out->tensor_scale)
    return MPFA_ERR_INVALID_ARG;
  if ((uint64_t)B * Hkv * Nk >= (1ull << 31)) return MPFA_ERR_INVALID_ARG;
  if (!ok_ptr(workspace) || ws_bytes < 256) return MPFA_ERR_INVALID_ARG;
  mpfa::QuantArgs a = {};
  a.B = B;
  a.Nk = Nk;
  a.Hkv = Hkv;
  a.v = v_bf16;
  a.vtc = vt_out->codes;
  a.vts = vt_out->scales;
  a.s_v = vt_out->tensor_scale;
  a.amax = static_cast<unsigned*>(workspace);
  a.err = status_ptr();
  if (!a.err) return MPFA_ERR_CUDA;
  return from_cuda(mpfa::launch_quantize_vt(a, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// The checks and argument set both prefill entries share; vc/vts/s_v are
// the V operand of either kernel.
mpfa_status prefill_common(const mpfa_nvfp4* q, const mpfa_rank1* qbar, const mpfa_nvfp4* k,
                           const uint8_t* vc, const uint8_t* vts, const float* s_v, int pv4,
                           int B, int N, int Hq, int Hkv, int d, int causal, int compensate, int T,
                           void* o_bf16, float* lse, const float* lse_shift, mpfa_stream_t stream) {
  if (d != 128) return MPFA_ERR_UNSUPPORTED;
  if (compensate && T != 1 && T != 2) return MPFA_ERR_UNSUPPORTED;
  if (!q || !k || B <= 0 || N <= 0 || N % 128 || Hq <= 0 || Hkv <= 0 || Hq % Hkv)
    return MPFA_ERR_INVALID_ARG;
  if (!ok_ptr(q->codes) || !ok_ptr(q->scales) || !q->tensor_scale || !ok_ptr(k->codes) ||
      !ok_ptr(k->scales) || !k->tensor_scale || !ok_ptr(vc) || !s_v || !ok_ptr(o_bf16))
    return MPFA_ERR_INVALID_ARG;
  if (pv4 && !ok_ptr(vts)) return MPFA_ERR_INVALID_ARG;
  if (compensate && (!qbar || !ok_ptr(qbar->codes) || !qbar->scales))
    return MPFA_ERR_INVALID_ARG;
  if ((uint64_t)B * Hq * N >= (1ull << 31) || (uint64_t)B * Hkv * N >= (1ull << 31))
    return MPFA_ERR_INVALID_ARG;
  mpfa::PrefillArgs a = {};
  a.qc = q->codes;
  a.qs = q->scales;
  a.s_q = q->tensor_scale;
  a.qbc = compensate ? qbar->codes : nullptr;
  a.qbs = compensate ? qbar->scales : nullptr;
  a.kc = k->codes;
  a.ks = k->scales;
  a.s_k = k->tensor_scale;
  a.vc = vc;
  a.vts = pv4 ? vts : nullptr;
  a.s_v = s_v;
  a.pv4 = pv4;
  a.B = B;
  a.N = N;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.causal = causal != 0;
  a.compensate = compensate != 0;
  a.T = compensate ? T : 0;
  a.o = o_bf16;
  a.lse = lse;
  a.lse_shift = lse_shift;
  a.err = status_ptr();
  if (!a.err) return MPFA_ERR_CUDA;
  return from_cuda(mpfa::launch_prefill(a, reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

mpfa_status mpfa_prefill(const mpfa_nvfp4* q, const mpfa_rank1* qbar, const mpfa_nvfp4* k,
                         const mpfa_fp8* v, int B, int N, int Hq, int Hkv, int d, int causal,
                         int compensate, int T, void* o_bf16, float* lse,
                         const float* lse_shift, mpfa_stream_t stream) {
  return prefill_common(q, qbar, k, v ? v->codes : nullptr, nullptr,
                        v ? v->tensor_scale : nullptr, 0, B, N, Hq, Hkv, d, causal, compensate,
                        T, o_bf16, lse, lse_shift, stream);
}

mpfa_status mpfa_prefill_fp4pv(const mpfa_nvfp4* q, const mpfa_rank1* qbar, const mpfa_nvfp4* k,
                               const mpfa_nvfp4* vt, int B, int N, int Hq, int Hkv, int d,
                               int causal, int compensate, int T, void* o_bf16, float* lse,
                               mpfa_stream_t stream) {
  return prefill_common(q, qbar, k, vt ? vt->codes : nullptr, vt ? vt->scales : nullptr,
                        vt ? vt->tensor_scale : nullptr, 1, B, N, Hq, Hkv, d, causal,
                        compensate, T, o_bf16, lse, nullptr, stream);
}

size_t mpfa_decode_workspace_size(int B, int Hq, int Hkv, int d, int Lmax, int kv_chunk) {
  if (d != 128 || B <= 0 || Hq <= 0 || Hkv <= 0 || Lmax <= 0) return 0;
  int sms = mpfa::sm_count(mpfa::current_device());
  if (sms <= 0) sms = 148;
  int chunk = kv_chunk > 0 ? kv_chunk : mpfa::decode_default_chunk(B, Hkv, Lmax, sms);
  int nsplit = (Lmax + chunk - 1) / chunk;
  return mpfa::decode_workspace_bytes(B, Hq, Hkv, nsplit);
}

}  // extern "C"

// Shared by mpfa_decode (block_table null: contiguous [B][Hkv][Lmax] cache)
// and mpfa_decode_paged (pool rows [num_pages][Hkv][128], Lmax = 128 * max_pages).
static mpfa_status decode_impl(const void* q_bf16, const mpfa_nvfp4* k_cache,
                               const mpfa_fp8* v_cache, const float* kbar,
                               const int32_t* block_table, int num_pages, int max_pages,
                               const int32_t* seqlens, int B, int Hq, int Hkv, int d, int Lmax,
                               int compensate, int T, int kv_chunk, void* o_bf16, float* lse,
                               mpfa_nvfp4* q_quant_out, mpfa_rank1* qbar_quant_out,
                               int* used_chunk, void* workspace, size_t ws_bytes,
                               mpfa_stream_t stream) {
  if (d != 128) return MPFA_ERR_UNSUPPORTED;
  if (compensate && T != 1 && T != 2) return MPFA_ERR_UNSUPPORTED;
  if (!ok_ptr(q_bf16) || !k_cache || !v_cache || !seqlens || B <= 0 || Hq <= 0 || Hkv <= 0 ||
      Hq % Hkv || Lmax <= 0 || Lmax % 128 || kv_chunk < 0 || kv_chunk % 128 || !ok_ptr(o_bf16))
    return MPFA_ERR_INVALID_ARG;
  if (!ok_ptr(k_cache->codes) || !ok_ptr(k_cache->scales) || !k_cache->tensor_scale ||
      !ok_ptr(v_cache->codes) || !v_cache->tensor_scale)
    return MPFA_ERR_INVALID_ARG;
  if (Hq / Hkv > 16) return MPFA_ERR_UNSUPPORTED;
  if (!block_table && (uint64_t)B * Hkv * Lmax >= (1ull << 31)) return MPFA_ERR_INVALID_ARG;
  if (block_table && (num_pages <= 0 || max_pages <= 0 ||
                      (uint64_t)num_pages * Hkv * 128 >= (1ull << 31) ||
                      (uint64_t)B * max_pages >= (1ull << 31)))
    return MPFA_ERR_INVALID_ARG;
  int sms = mpfa::sm_count(mpfa::current_device());
  if (sms <= 0) sms = 148;
  const int chunk = kv_chunk > 0 ? kv_chunk : mpfa::decode_default_chunk(B, Hkv, Lmax, sms);
  const int nsplit = (Lmax + chunk - 1) / chunk;
  const size_t need = mpfa::decode_workspace_bytes(B, Hq, Hkv, nsplit);
  if (!ok_ptr(workspace) || ws_bytes < need) return MPFA_ERR_INVALID_ARG;
  mpfa::DecodeArgs a = {};
  a.q = q_bf16;
  a.kc = k_cache->codes;
  a.ks = k_cache->scales;
  a.s_k = k_cache->tensor_scale;
  a.vc = v_cache->codes;
  a.s_v = v_cache->tensor_scale;
  a.seqlens = seqlens;
  a.kbar = kbar;
  a.block_table = block_table;
  a.num_pages = num_pages;
  a.max_pages = max_pages;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Lmax = Lmax;
  a.compensate = compensate != 0;
  a.T = compensate ? T : 0;
  a.chunk = chunk;
  a.nsplit = nsplit;
  a.o = o_bf16;
  a.lse = lse;
  // workspace carve: [amax 256 B][s_q 256 B][qc][qs][qbc][qbs][qbar][part_o][part_lse]
  uint8_t* w = static_cast<uint8_t*>(workspace);
  auto take = [&](size_t bytes) {
    uint8_t* p = w;
    w += (bytes + 255) & ~size_t(255);
    return p;
  };
  a.amax = reinterpret_cast<unsigned*>(take(256));
  float* s_q_ws = reinterpret_cast<float*>(take(256));
  uint8_t* qc_ws = take((size_t)B * Hq * 64);
  uint8_t* qs_ws = take((size_t)B * Hq * 8);
  uint8_t* qbc_ws = take((size_t)B * Hkv * 2 * 64);
  uint8_t* qbs_ws = take((size_t)B * Hkv * 2 * 8);
  a.qbar = reinterpret_cast<float*>(take((size_t)B * Hkv * 128 * sizeof(float)));
  a.part_o = reinterpret_cast<float*>(take((size_t)B * Hq * nsplit * 128 * sizeof(float)));
  a.part_lse = reinterpret_cast<float*>(take((size_t)B * Hq * nsplit * sizeof(float)));
  a.q_kbar = reinterpret_cast<float*>(take((size_t)B * (Hq + Hkv) * sizeof(float)));
  const bool qout = q_quant_out && q_quant_out->codes && q_quant_out->scales &&
                    q_quant_out->tensor_scale;
  a.qc = qout ? q_quant_out->codes : qc_ws;
  a.qs = qout ? q_quant_out->scales : qs_ws;
  a.s_q = qout ? q_quant_out->tensor_scale : s_q_ws;
  const bool bout = qbar_quant_out && qbar_quant_out->codes && qbar_quant_out->scales;
  a.qbc = bout ? qbar_quant_out->codes : qbc_ws;
  a.qbs = bout ? qbar_quant_out->scales : qbs_ws;
  a.err = status_ptr();
  if (!a.err) return MPFA_ERR_CUDA;
  if (used_chunk) *used_chunk = chunk;
  return from_cuda(mpfa::launch_decode(a, reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" {

mpfa_status mpfa_decode(const void* q_bf16, const mpfa_nvfp4* k_cache, const mpfa_fp8* v_cache,
                        const float* kbar, const int32_t* seqlens, int B, int Hq, int Hkv, int d,
                        int Lmax, int compensate, int T, int kv_chunk, void* o_bf16, float* lse,
                        mpfa_nvfp4* q_quant_out, mpfa_rank1* qbar_quant_out, int* used_chunk,
                        void* workspace, size_t ws_bytes, mpfa_stream_t stream) {
  return decode_impl(q_bf16, k_cache, v_cache, kbar, nullptr, 0, 0, seqlens, B, Hq, Hkv, d, Lmax,
                     compensate, T, kv_chunk, o_bf16, lse, q_quant_out, qbar_quant_out,
                     used_chunk, workspace, ws_bytes, stream);
}

mpfa_status mpfa_decode_paged(const void* q_bf16, const mpfa_nvfp4* k_pool, const mpfa_fp8* v_pool,
                              const int32_t* block_table, int num_pages, int max_pages,
                              const int32_t* seqlens, int B, int Hq, int Hkv, int d,
                              int compensate, int T, int kv_chunk, void* o_bf16, float* lse,
                              mpfa_nvfp4* q_quant_out, mpfa_rank1* qbar_quant_out,
                              int* used_chunk, void* workspace, size_t ws_bytes,
                              mpfa_stream_t stream) {
  if (!block_table) return MPFA_ERR_INVALID_ARG;
  if (max_pages <= 0 || max_pages > (1 << 30) / 128) return MPFA_ERR_INVALID_ARG;
  return decode_impl(q_bf16, k_pool, v_pool, nullptr, block_table, num_pages, max_pages, seqlens,
                     B, Hq, Hkv, d, 128 * max_pages, compensate, T, kv_chunk, o_bf16, lse,
                     q_quant_out, qbar_quant_out, used_chunk, workspace, ws_bytes, stream);
}

}  // extern "C"

static mpfa_status append_impl(const void* k_new_bf16, const void* v_new_bf16,
                               const int32_t* seqlens, const int32_t* block_table, int num_pages,
                               int max_pages, int B, int n_new, int Hkv, int d, int Lmax,
                               mpfa_nvfp4* k_cache, mpfa_fp8* v_cache, const float* kbar,
                               mpfa_stream_t stream) {
  if (d != 128) return MPFA_ERR_UNSUPPORTED;
  if (!ok_ptr(k_new_bf16) || !ok_ptr(v_new_bf16) || !seqlens || !k_cache || !v_cache ||
      B <= 0 || n_new <= 0 || Hkv <= 0 || Lmax <= 0 || Lmax % 128 || n_new > Lmax)
    return MPFA_ERR_INVALID_ARG;
  if (!ok_ptr(k_cache->codes) || !ok_ptr(k_cache->scales) || !k_cache->tensor_scale ||
      !ok_ptr(v_cache->codes) || !v_cache->tensor_scale)
    return MPFA_ERR_INVALID_ARG;
  if ((!block_table && (uint64_t)B * Hkv * Lmax >= (1ull << 31)) ||
      (uint64_t)B * n_new * Hkv >= (1ull << 31))
    return MPFA_ERR_INVALID_ARG;
  if (block_table && (num_pages <= 0 || max_pages <= 0 ||
                      (uint64_t)num_pages * Hkv * 128 >= (1ull << 31)))
    return MPFA_ERR_INVALID_ARG;
  mpfa::AppendArgs a = {};
  a.k_new = k_new_bf16;
  a.v_new = v_new_bf16;
  a.seqlens = seqlens;
  a.B = B;
  a.n_new = n_new;
  a.Hkv = Hkv;
  a.Lmax = Lmax;
  a.kc = k_cache->codes;
  a.ks = k_cache->scales;
  a.s_k = k_cache->tensor_scale;
  a.vc = v_cache->codes;
  a.s_v = v_cache->tensor_scale;
  a.kbar = kbar;
  a.block_table = block_table;
  a.num_pages = num_pages;
  a.max_pages = max_pages;
  a.err = status_ptr();
  if (!a.err) return MPFA_ERR_CUDA;
  return from_cuda(mpfa::launch_append(a, reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" {

mpfa_status mpfa_append_kv(const void* k_new_bf16, const void* v_new_bf16, const int32_t* seqlens,
                           int B, int n_new, int Hkv, int d, int Lmax, mpfa_nvfp4* k_cache,
                           mpfa_fp8* v_cache, const float* kbar, mpfa_stream_t stream) {
  return append_impl(k_new_bf16, v_new_bf16, seqlens, nullptr, 0, 0, B, n_new, Hkv, d, Lmax,
                     k_cache, v_cache, kbar, stream);
}

mpfa_status mpfa_append_kv_paged(const void* k_new_bf16, const void* v_new_bf16,
                                 const int32_t* seqlens, const int32_t* block_table,
                                 int num_pages, int max_pages, int B, int n_new, int Hkv, int d,
                                 mpfa_nvfp4* k_pool, mpfa_fp8* v_pool, mpfa_stream_t stream) {
  if (!block_table) return MPFA_ERR_INVALID_ARG;
  if (max_pages <= 0 || max_pages > (1 << 30) / 128) return MPFA_ERR_INVALID_ARG;
  return append_impl(k_new_bf16, v_new_bf16, seqlens, block_table, num_pages, max_pages, B, n_new,
                     Hkv, d, 128 * max_pages, k_pool, v_pool, nullptr, stream);
}

mpfa_status mpfa_selftest_wait_timeout(unsigned long long limit_ns, mpfa_stream_t stream) {
  if (limit_ns == 0 || limit_ns > 2000000000ull) return MPFA_ERR_INVALID_ARG;
  int* err = status_ptr();
  if (!err) return MPFA_ERR_CUDA;
  selftest_wait_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(err, limit_ns);
  return from_cuda(cudaGetLastError());
}

mpfa_status mpfa_get_error(mpfa_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return from_cuda(e);
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return MPFA_ERR_CUDA;
  if (v != 0) {
    int zero = 0;
    cudaMemcpyToSymbol(g_status, &zero, sizeof(int));
  }
  return v == 0 ? MPFA_OK : static_cast<mpfa_status>(v);
}

}  // extern "C"
