// prefill.cu -- MpFA QK4PV8 prefill forward on sm_103a.
//
// Method (MpFA abstract): S = Q K^T on block-scaled NVFP4 tensor cores, the
// rank-one smoothing term (the T NVFP4 terms of the query-block mean, the
// same row for all 128 rows) issued as extra MMAs into the same score
// accumulator, an online softmax (FlashAttention-2 section of the
// "FlashAttention压到4位" explainer), P converted to FP8 E4M3 in place in
// tensor memory and multiplied by FP8 V on the tensor core.  The running sum
// l is itself a tensor-core product of the rounded P codes with a ones tile,
// so the denominator consumes exactly the codes the PV product consumes (the
// explainer's Direct-P section states that rule).
//
// One CTA computes one 128-row query tile of one (batch, head):
//   warp 4    TMA producer: Q tile once, then K / K-scale / V tiles through a
//             ring of kStages shared-memory stages.
//   warp 5    MMA issuer: block scales into TMEM (tcgen05.cp), QK^T and the
//             rank-one MMAs into score bank j % 2, then PV_{j-1} and the
//             row-sum MMA once the softmax has published P_{j-1}.
//   warps 0-3 softmax + correction + epilogue, one query row per thread
//             (TMEM lane = row): max, exp2, E4M3 P stored over the scores,
//             rescale of O when the running max moves, O / l and LSE.
// Tensor memory (512 columns): S0 [0,128) S1 [128,256) O [256,384)
// L [384,400) scale factors [400,448).
#include <cmath>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "device.cuh"
#include "internal.h"

namespace mpfa {

bool make_map_2d_u8(CUtensorMap* m, const void* base, uint64_t inner_bytes, uint64_t rows,
                    uint32_t box_rows, CUtensorMapSwizzle sw);

namespace {

constexpr int kStages = 3;
constexpr int kThreads = 192;
constexpr int kTmemCols = 512;

constexpr uint32_t kColS0 = 0, kColO = 256, kColL = 384, kColSfQ = 400, kColSfQb = 408,
                   kColSfK = 424;

// shared memory layout (offsets from a 1024-byte aligned base)
constexpr uint32_t kOffQ = 0;                           // 8 KB
constexpr uint32_t kOffQb = kOffQ + 8192;               // 2 x 8 KB
constexpr uint32_t kOffK = kOffQb + 2 * 8192;           // kStages x 8 KB
constexpr uint32_t kOffV = kOffK + kStages * 8192;      // kStages x 16 KB
constexpr uint32_t kOffQs = kOffV + kStages * 16384;    // 1 KB
constexpr uint32_t kOffQbs = kOffQs + 1024;             // 2 x 1 KB
constexpr uint32_t kOffKs = kOffQbs + 2048;             // kStages x 1 KB
constexpr uint32_t kOffOnes = kOffKs + kStages * 1024;  // 2 KB
constexpr uint32_t kOffBar = kOffOnes + 2048;
constexpr uint32_t kNumBars = 8 + 3 * kStages;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemUsed = kOffMisc + 64;
// Request more than half an SM's shared memory so a single CTA owns the
// SM and its 512 TMEM columns.
constexpr uint32_t kSmemBytes = 160 * 1024;
static_assert(kSmemUsed + 1024 <= kSmemBytes, "shared memory layout overflow");

// barrier indices
enum : int {
  kBarQFull = 0,
  kBarQbReady = 1,
  kBarSFull0 = 2,   // +bank
  kBarPReady0 = 4,  // +bank
  kBarODone = 6,
  kBarDrain = 7,
  kBarKFull0 = 8,                  // +stage
  kBarVFull0 = 8 + kStages,        // +stage
  kBarKvEmpty0 = 8 + 2 * kStages,  // +stage
};

struct Params {
  PrefillArgs a;
  float log2e_rsqrt_d;  // fp32(log2(e) / sqrt(128))
  int q_tiles;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap map_q,
                   const __grid_constant__ CUtensorMap map_k,
                   const __grid_constant__ CUtensorMap map_v, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const PrefillArgs& a = p.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // work unit: heavy causal tiles first
  const int bh_count = a.B * a.Hq;
  const int qt = p.q_tiles - 1 - (int)(blockIdx.x / bh_count);
  const int bh = (int)(blockIdx.x % bh_count);
  const int h = bh % a.Hq, b = bh / a.Hq;
  const int g = a.Hq / a.Hkv;
  const int hk = h / g;
  const int nkv = a.causal ? qt + 1 : a.N / 128;
  const int T = a.compensate ? a.T : 0;

  auto bar = [&](int i) { return sbase + kOffBar + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc + 8);

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(kBarQFull), 1);
    mbar_init(bar(kBarQbReady), 128);
    mbar_init(bar(kBarSFull0), 1);
    mbar_init(bar(kBarSFull0 + 1), 1);
    mbar_init(bar(kBarPReady0), 128);
    mbar_init(bar(kBarPReady0 + 1), 128);
    mbar_init(bar(kBarODone), 1);
    mbar_init(bar(kBarDrain), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarKFull0 + s), 1);
      mbar_init(bar(kBarVFull0 + s), 1);
      mbar_init(bar(kBarKvEmpty0 + s), 1);
    }
    fence_barrier_init();
  }
  if (warp == 5) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      prefetch_tensormap(&map_q);
      prefetch_tensormap(&map_k);
      prefetch_tensormap(&map_v);
      const int qrow = (b * a.Hq + h) * a.N + qt * 128;
      mbar_expect_tx(bar(kBarQFull), 8192 + 1024);
      tma_load_2d(sbase + kOffQ, &map_q, 0, qrow, bar(kBarQFull));
      bulk_load(sbase + kOffQs, a.qs + (size_t)qrow * 8, 1024, bar(kBarQFull));
      const int kvrow0 = (b * a.Hkv + hk) * a.N;
      int issued = 0;
      for (int j = 0; j < nkv; ++j) {
        const int s = j % kStages;
        if (j >= kStages &&
            !mbar_wait(bar(kBarKvEmpty0 + s), ((j / kStages) - 1) & 1, a.err, abort_flag))
          break;
        const int row = kvrow0 + j * 128;
        mbar_expect_tx(bar(kBarKFull0 + s), 8192 + 1024);
        tma_load_2d(sbase + kOffK + s * 8192, &map_k, 0, row, bar(kBarKFull0 + s));
        bulk_load(sbase + kOffKs + s * 1024, a.ks + (size_t)row * 8, 1024, bar(kBarKFull0 + s));
        mbar_expect_tx(bar(kBarVFull0 + s), 16384);
        tma_load_2d(sbase + kOffV + s * 16384, &map_v, 0, row, bar(kBarVFull0 + s));
        issued = j + 1;
      }
      // drain: every stage's last load must have landed before the CTA exits
      for (int j = issued - kStages > 0 ? issued - kStages : 0; j < issued; ++j) {
        const int s = j % kStages;
        mbar_wait(bar(kBarKFull0 + s), (j / kStages) & 1, a.err, nullptr);
        mbar_wait(bar(kBarVFull0 + s), (j / kStages) & 1, a.err, nullptr);
      }
    }
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t id_qk = idesc_nvfp4(128, 128);
      const uint32_t id_pv = idesc_fp8(128, 128, 0, 1);
      const uint32_t id_l = idesc_fp8(128, 16, 0, 0);
      bool ok = mbar_wait(bar(kBarQFull), 0, a.err, abort_flag) &&
                mbar_wait(bar(kBarQbReady), 0, a.err, abort_flag);
      if (ok) {
        tc_fence_after();
        for (int kc = 0; kc < 2; ++kc)
          tmem_cp_32x128b_x4(tmem + kColSfQ + 4 * kc,
                             smem_desc(sbase + kOffQs + 512 * kc, 128, 128, kSwizzleNone));
        for (int t = 0; t < T; ++t)
          for (int kc = 0; kc < 2; ++kc)
            tmem_cp_32x128b_x4(
                tmem + kColSfQb + 8 * t + 4 * kc,
                smem_desc(sbase + kOffQbs + 1024 * t + 512 * kc, 128, 128, kSwizzleNone));
      }
      const uint64_t ones = smem_desc(sbase + kOffOnes, 128, 256, kSwizzleNone);
      auto issue_pv = [&](int jp) -> bool {
        const int bp = jp & 1, sp = jp % kStages;
        if (!mbar_wait(bar(kBarPReady0 + bp), (jp >> 1) & 1, a.err, abort_flag)) return false;
        if (!mbar_wait(bar(kBarVFull0 + sp), (jp / kStages) & 1, a.err, abort_flag))
          return false;
        tc_fence_after();
        const uint32_t pcol = tmem + kColS0 + 128 * bp;
        const uint32_t vaddr = sbase + kOffV + sp * 16384;
        for (int kk = 0; kk < 4; ++kk)
          mma_fp8_ts(tmem + kColO, pcol + 8 * kk, smem_desc(vaddr + 4096 * kk, 16, 1024, kSwizzle128B),
                     id_pv, (jp > 0 || kk > 0) ? 1u : 0u);
        for (int kk = 0; kk < 4; ++kk)
          mma_fp8_ts(tmem + kColL, pcol + 8 * kk, ones, id_l, (jp > 0 || kk > 0) ? 1u : 0u);
        tc_commit(bar(kBarODone));
        if (jp + kStages < nkv) tc_commit(bar(kBarKvEmpty0 + sp));
        return true;
      };
      for (int j = 0; ok && j < nkv; ++j) {
        const int s = j % kStages, bk = j & 1;
        if (!mbar_wait(bar(kBarKFull0 + s), (j / kStages) & 1, a.err, abort_flag)) break;
        // bank bk was last read by PV_{j-2}
        if (j >= 2 && !mbar_wait(bar(kBarODone), (j - 2) & 1, a.err, abort_flag)) break;
        tc_fence_after();
        const uint32_t sfk = tmem + kColSfK + 8 * s;
        for (int kc = 0; kc < 2; ++kc)
          tmem_cp_32x128b_x4(sfk + 4 * kc,
                             smem_desc(sbase + kOffKs + 1024 * s + 512 * kc, 128, 128, kSwizzleNone));
        const uint32_t dS = tmem + kColS0 + 128 * bk;
        const uint32_t kaddr = sbase + kOffK + 8192 * s;
        for (int kc = 0; kc < 2; ++kc)
          mma_nvfp4_ss(dS, smem_desc(sbase + kOffQ + 32 * kc, 16, 512, kSwizzle64B),
                       smem_desc(kaddr + 32 * kc, 16, 512, kSwizzle64B), id_qk, tmem + kColSfQ + 4 * kc,
                       sfk + 4 * kc, kc > 0 ? 1u : 0u);
        for (int t = 0; t < T; ++t)
          for (int kc = 0; kc < 2; ++kc)
            mma_nvfp4_ss(dS, smem_desc(sbase + kOffQb + 8192 * t + 32 * kc, 16, 512, kSwizzle64B),
                         smem_desc(kaddr + 32 * kc, 16, 512, kSwizzle64B), id_qk,
                         tmem + kColSfQb + 8 * t + 4 * kc, sfk + 4 * kc, 1u);
        tc_commit(bar(kBarSFull0 + bk));
        if (j >= 1 && !issue_pv(j - 1)) {
          ok = false;
          break;
        }
      }
      if (ok && nkv > 0) issue_pv(nkv - 1);
      // drain the tensor pipe before the CTA releases TMEM
      tc_commit(bar(kBarDrain));
      mbar_wait(bar(kBarDrain), 0, a.err, nullptr);
    }
  } else {
    // ---------------- softmax / correction / epilogue ----------------
    const int row = threadIdx.x;  // 0..127, TMEM lane
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    // Rank-one operand tiles: every row holds the block's term t (same 64
    // bytes), written with the 64-byte swizzle the TMA applies to Q and K.
    const int nblk = a.N / 128;
    for (int t = 0; t < T; ++t) {
      const uint8_t* src = a.qbc + (((size_t)bh * nblk + qt) * a.T + t) * 64;
      uint4* dst = reinterpret_cast<uint4*>(smem + kOffQb + 8192 * t + 64 * row);
#pragma unroll
      for (int c = 0; c < 4; ++c) dst[c ^ ((row >> 1) & 3)] = reinterpret_cast<const uint4*>(src)[c];
      const uint8_t* ssrc = a.qbs + (((size_t)bh * nblk + qt) * a.T + t) * 8;
      uint32_t w0 = *reinterpret_cast<const uint32_t*>(ssrc);
      uint32_t w1 = *reinterpret_cast<const uint32_t*>(ssrc + 4);
      reinterpret_cast<uint32_t*>(smem + kOffQbs + 1024 * t)[row] = w0;
      reinterpret_cast<uint32_t*>(smem + kOffQbs + 1024 * t + 512)[row] = w1;
    }
    // ones tile (E4M3 1.0 = 0x38) for the row-sum MMA
    reinterpret_cast<uint4*>(smem + kOffOnes)[row] = make_uint4(0x38383838u, 0x38383838u,
                                                                 0x38383838u, 0x38383838u);
    fence_proxy_async_smem();
    mbar_arrive(bar(kBarQbReady));

    const float cs = __fmul_rn(__fmul_rn(*a.s_q, *a.s_k), p.log2e_rsqrt_d);
    float m = -INFINITY;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int bk = j & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarSFull0 + bk), (j >> 1) & 1, a.err, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sS = tmem + lane_off + kColS0 + 128 * bk;
      uint32_t sr[4][32];
      tmem_ld32(sS, sr[0]);
      tmem_ld32(sS + 32, sr[1]);
      tmem_ld32(sS + 64, sr[2]);
      tmem_ld32(sS + 96, sr[3]);
      tmem_ld_wait();
      if (a.causal && j == qt) {  // diagonal tile: key > row is masked
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * c + i > row) sr[c][i] = 0xFF800000u;  // -inf
      }
      // cs > 0, so max_i(S_i * cs) == (max_i S_i) * cs exactly
      float smax = __uint_as_float(sr[0][0]);
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) smax = fmaxf(smax, __uint_as_float(sr[c][i]));
      const float mn = fmaxf(m, __fmul_rn(smax, cs));
      const float alpha = (m == -INFINITY) ? 0.0f : ex2(m - mn);
      const float bias = 8.0f - mn;  // P8 = E4M3(2^(t - m) * 2^8)
      uint32_t pw[32];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int w = 0; w < 8; ++w)
          pw[8 * c + w] = e4m3x4(ex2(fmaf(__uint_as_float(sr[c][4 * w]), cs, bias)),
                                 ex2(fmaf(__uint_as_float(sr[c][4 * w + 1]), cs, bias)),
                                 ex2(fmaf(__uint_as_float(sr[c][4 * w + 2]), cs, bias)),
                                 ex2(fmaf(__uint_as_float(sr[c][4 * w + 3]), cs, bias)));
      tmem_st32(sS, pw);
      // correction: O and L scale by alpha once PV_{j-1} has landed
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarODone), (j - 1) & 1, a.err, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t oO = tmem + lane_off + kColO;
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(oO + 32 * c, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(oO + 32 * c, o);
        }
        uint32_t l4[4];
        tmem_ld4(tmem + lane_off + kColL, l4);
        tmem_ld_wait();
        l4[0] = __float_as_uint(__uint_as_float(l4[0]) * alpha);
        tmem_st4(tmem + lane_off + kColL, l4);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(kBarPReady0 + bk));
      m = mn;
    }
    if (ok && nkv > 0 &&
        __all_sync(0xffffffffu, mbar_wait(bar(kBarODone), (nkv - 1) & 1, a.err, abort_flag))) {
      tc_fence_after();
      uint32_t l4[4];
      tmem_ld4(tmem + lane_off + kColL, l4);
      tmem_ld_wait();
      const float l = __uint_as_float(l4[0]);
      const float sc = __fdiv_rn(*a.s_v, l);
      const size_t grow = (size_t)qt * 128 + row;
      uint4* out = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.o) +
                                            (((size_t)b * a.N + grow) * a.Hq + h) * 128);
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + kColO + 32 * c, o);
        tmem_ld_wait();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(o[8 * q4 + 2 * e]) * sc,
                                                     __uint_as_float(o[8 * q4 + 2 * e + 1]) * sc);
            w[e] = *reinterpret_cast<uint32_t*>(&v);
          }
          out[4 * c + q4] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      if (a.lse) a.lse[(size_t)bh * a.N + grow] = 0.69314718055994531f * (m + __log2f(l) - 8.0f);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  const uint64_t qrows = (uint64_t)a.B * a.Hq * a.N, kvrows = (uint64_t)a.B * a.Hkv * a.N;
  if (!make_map_2d_u8(&mq, a.qc, 64, qrows, 128, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_map_2d_u8(&mk, a.kc, 64, kvrows, 128, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_map_2d_u8(&mv, a.vc, 128, kvrows, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  Params p;
  p.a = a;
  p.log2e_rsqrt_d = (float)(1.4426950408889634 / std::sqrt(128.0));
  p.q_tiles = a.N / 128;
  const unsigned grid = (unsigned)(p.q_tiles * a.B * a.Hq);
  if (grid == 0) return cudaSuccess;
  prefill_kernel<<<grid, kThreads, kSmemBytes, stream>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace mpfa
