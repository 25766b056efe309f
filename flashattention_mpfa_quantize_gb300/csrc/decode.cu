// decode.cu -- MpFA split-KV decode on sm_103a.
//
// MpFA abstract: the kernel partitions work adaptively across prefill and
// decode.  Decode has one query token per sequence, so the g = Hq/Hkv query
// heads that share a KV head are the only rows that share keys; putting them
// on the MMA's M dimension would waste 124 of 128 rows.  The tile is swapped
// instead: 128 keys are the M rows and the query heads are N columns,
//     S^T[key][n] = K[key] . Q[n]        (block-scaled NVFP4, N = 16)
//     O^T[ch][n] += V^T[ch][key] P^T[key][n]   (FP8 E4M3, N = 16)
//     L[.][n]    += 1 . P^T[key][n]            (row sums of the rounded P)
// and each split of the cache keeps its own running max and sum (the online
// softmax of the FlashAttention-2 section of the "FlashAttention压到4位"
// explainer); a combine kernel merges splits by their LSE.
//
// Kernels (one stream, in order):
//   dq_stats   per (b, kv head): fp32 mean of the g query rows (exact fp64
//              sum) and amax of q - mean / mean (or of q).
//   dq_quant   NVFP4 codes of q (or q - mean) and T terms of the mean.
//   split      one CTA per (b, kv head, split); TMA ring of K / V tiles,
//              warp 5 issues MMAs, warps 0-3 (thread = key) run the softmax.
//   combine    per (b, query head): LSE-weighted merge of the splits.
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
constexpr int kTmemCols = 128;
constexpr int kMaxG = 16;  // query heads per KV head (N columns of the swapped tile)

// TMEM columns
constexpr uint32_t kColS0 = 0, kColO = 32, kColL = 48, kColSfK = 64, kColSfQ = 88;

// shared memory (offsets from a 1024-byte aligned base)
constexpr uint32_t kOffK = 0;                           // kStages x 8 KB
constexpr uint32_t kOffV = kOffK + kStages * 8192;      // kStages x 16 KB
constexpr uint32_t kOffKs = kOffV + kStages * 16384;    // kStages x 1 KB
constexpr uint32_t kOffQ = kOffKs + kStages * 1024;     // (1 + 2) x 1 KB: q', qbar terms (16 rows x 64 B)
constexpr uint32_t kOffQs = kOffQ + 3 * 1024;           // (1 + 2) x 1 KB scale atoms
constexpr uint32_t kOffP = kOffQs + 3 * 1024;           // 2 x 2 KB: P^T (16 rows x 128 B)
constexpr uint32_t kOffOnes = kOffP + 2 * 2048;         // 4 KB ones (128 rows x 32 B)
constexpr uint32_t kOffRed = kOffOnes + 4096;           // 4 warps x 16 floats, 4 vote words
constexpr uint32_t kOffBar = kOffRed + 4 * 16 * 4 + 16;   // + 4 vote words
constexpr uint32_t kNumBars = 8 + 3 * kStages + 2;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemUsed = kOffMisc + 64;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;

enum : int {
  kBarQReady = 0,
  kBarSFull0 = 1,   // +bank
  kBarPReady0 = 3,  // +bank
  kBarODone = 5,
  kBarDrain = 6,
  kBarPFree0 = 7 + 3 * kStages + 1,  // +bank: P^T buffer read by its PV MMAs
  kBarKFull0 = 8,
  kBarVFull0 = 8 + kStages,
  kBarKvEmpty0 = 8 + 2 * kStages,
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float tensor_scale(unsigned amax_bits, float qmax) {
  float a = __uint_as_float(amax_bits);
  return a == 0.0f ? 1.0f : __fdiv_rn(a, qmax);
}

__device__ __forceinline__ float e2m1_value(uint32_t c) {
  uint32_t e = (c >> 1) & 3u, m = c & 1u;
  float mag = (e == 0) ? 0.5f * (float)m : (1.0f + 0.5f * (float)m) * (float)(1u << (e - 1));
  return (c & 8u) ? -mag : mag;
}

// Same block rule as the prefill quantizer (include/mpfa.h).
__device__ __forceinline__ void nvfp4_block(const float (&x)[16], float s, uint2& codes,
                                            uint32_t& sb) {
  float bamax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) bamax = fmaxf(bamax, fabsf(x[i]));
  float t = __fdiv_rn(bamax, __fmul_rn(6.0f, s));
  sb = e4m3_pos(t);
  uint32_t w0 = 0, w1 = 0;
  if (sb != 0) {
    float denom = __fmul_rn(e4m3_value(sb), s);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t byte = e2m1x2(__fdiv_rn(x[2 * i], denom), __fdiv_rn(x[2 * i + 1], denom));
      if (i < 4)
        w0 |= byte << (8 * i);
      else
        w1 |= byte << (8 * (i - 4));
    }
  }
  codes = make_uint2(w0, w1);
}

// ---------------------------------------------------------------------------
// query quantization
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(128) dq_stats_kernel(DecodeArgs a) {
  __shared__ unsigned red[4];
  pdl_trigger();
  const int bk = blockIdx.x;  // b * Hkv + kv head
  const int g = a.Hq / a.Hkv;
  const int c = threadIdx.x;
  const __nv_bfloat16* q = reinterpret_cast<const __nv_bfloat16*>(a.q) + (size_t)bk * g * 128;
  unsigned m = 0;
  if (a.compensate) {
    double s = 0.0;
    for (int r = 0; r < g; ++r) s += (double)__bfloat162float(q[r * 128 + c]);
    const float mean = (float)(s / (double)g);
    a.qbar[(size_t)bk * 128 + c] = mean;
    m = __float_as_uint(fabsf(mean));
    for (int r = 0; r < g; ++r)
      m = max(m, __float_as_uint(fabsf(__fsub_rn(__bfloat162float(q[r * 128 + c]), mean))));
  } else {
    for (int r = 0; r < g; ++r) m = max(m, __float_as_uint(fabsf(__bfloat162float(q[r * 128 + c]))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((c & 31) == 0) red[c >> 5] = m;
  __syncthreads();
  if (c == 0) {
    m = max(max(red[0], red[1]), max(red[2], red[3]));
    if (m) atomicMax(a.amax, m);
  }
}

// sum_i e2m1(code_i) * w_i over the 16 codes of one NVFP4 block (fp32)
__device__ __forceinline__ float codes_dot(const uint2& codes, const float* w) {
  const uint32_t cw[2] = {codes.x, codes.y};
  float acc = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i)
    acc = __fmaf_rn(e2m1_value((cw[i >> 3] >> (4 * (i & 7))) & 15u), w[i], acc);
  return acc;
}

// 8 threads per row: rows [0, B*Hq) are query rows, then B*Hkv mean rows.
// With a smoothed cache (kbar) each row also gets its code-unit dot product
// with kbar: sum over its blocks of block scale * sum e2m1(code) * kbar
// (a mean row: over its T terms), which combine_kernel turns into the LSE
// term q_eff . kbar / sqrt(d).
__global__ void __launch_bounds__(128) dq_quant_kernel(DecodeArgs a) {
  pdl_wait();
  pdl_trigger();
  const int g = a.Hq / a.Hkv;
  const float s = tensor_scale(a.amax[0], 2688.0f);
  if (blockIdx.x == 0 && threadIdx.x == 0) *a.s_q = s;
  const int gt = blockIdx.x * blockDim.x + threadIdx.x;
  const int row = gt >> 3, j = gt & 7;
  const int nq = a.B * a.Hq;
  const int nb = a.compensate ? a.B * a.Hkv : 0;
  float part = 0.0f;
  if (row < nq) {
    const __nv_bfloat16* q = reinterpret_cast<const __nv_bfloat16*>(a.q) + (size_t)row * 128 + 16 * j;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = __bfloat162float(q[i]);
    if (a.compensate) {
      const float* mb = a.qbar + (size_t)(row / g) * 128 + 16 * j;
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = __fsub_rn(x[i], mb[i]);
    }
    uint2 codes;
    uint32_t sb;
    nvfp4_block(x, s, codes, sb);
    *reinterpret_cast<uint2*>(a.qc + (size_t)row * 64 + 8 * j) = codes;
    a.qs[(size_t)row * 8 + j] = (uint8_t)sb;
    if (a.kbar) part = e4m3_value(sb) * codes_dot(codes, a.kbar + (size_t)(row / g) * 128 + 16 * j);
  } else if (row < nq + nb) {
    const int r = row - nq;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = a.qbar[(size_t)r * 128 + 16 * j + i];
    for (int t = 0; t < a.T; ++t) {
      uint2 codes;
      uint32_t sb;
      nvfp4_block(x, s, codes, sb);
      *reinterpret_cast<uint2*>(a.qbc + ((size_t)r * a.T + t) * 64 + 8 * j) = codes;
      a.qbs[((size_t)r * a.T + t) * 8 + j] = (uint8_t)sb;
      const float sbv = e4m3_value(sb);
      if (a.kbar) part = __fmaf_rn(sbv, codes_dot(codes, a.kbar + (size_t)r * 128 + 16 * j), part);
      uint32_t w[2] = {codes.x, codes.y};
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        uint32_t cc = (w[i >> 3] >> (4 * (i & 7))) & 15u;
        x[i] = __fsub_rn(x[i], __fmul_rn(__fmul_rn(e2m1_value(cc), sbv), s));
      }
    }
  }
  if (a.kbar) {
    // the 8 threads of a row are 8 consecutive lanes
    part += __shfl_xor_sync(0xffffffffu, part, 1);
    part += __shfl_xor_sync(0xffffffffu, part, 2);
    part += __shfl_xor_sync(0xffffffffu, part, 4);
    if (j == 0 && row < nq + nb) a.q_kbar[row] = part;
  }
}

// ---------------------------------------------------------------------------
// split kernel
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(kThreads) split_kernel(const __grid_constant__ CUtensorMap map_k,
                                                         const __grid_constant__ CUtensorMap map_v,
                                                         const DecodeArgs a, float log2e_rsqrt_d) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int units = a.B * a.Hkv;
  const int items = units * a.nsplit;
  const int g = a.Hq / a.Hkv;
  const int T = a.compensate ? a.T : 0;
  auto bar = [&](int i) { return sbase + kOffBar + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc + 8);
  volatile int* item_slot = reinterpret_cast<volatile int*>(smem + kOffMisc + 16);
  float* red = reinterpret_cast<float*>(smem + kOffRed);

  // Persistent: the CTA takes (KV unit, split) items from a global counter
  // until they run out, so a slot freed by a short split takes the next item
  // at once.  Items are numbered split-major (every unit's first split
  // before any second split), so the shorter tail splits of variable-length
  // sequences and the empty splits past a sequence's end come last.  Between
  // items the whole CTA synchronises: every asynchronous copy and product of
  // the item has been waited for by then, so the barriers are re-initialised
  // for the next item and the tensor memory is reused.
  if (threadIdx.x == 0) *abort_flag = 0;
  if (warp == 5) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  if (warp == 4 && lane == 0) {
    prefetch_tensormap(&map_k);
    prefetch_tensormap(&map_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the query codes and the item counter come from the kernels before
  pdl_wait();
  pdl_trigger();

  for (;;) {
  if (threadIdx.x == 0) {
    *item_slot = atomicAdd(a.work, 1);
    mbar_init(bar(kBarQReady), 128);
    mbar_init(bar(kBarSFull0), 1);
    mbar_init(bar(kBarSFull0 + 1), 1);
    mbar_init(bar(kBarPReady0), 128);
    mbar_init(bar(kBarPReady0 + 1), 128);
    mbar_init(bar(kBarODone), 1);
    mbar_init(bar(kBarDrain), 1);
    mbar_init(bar(kBarPFree0), 1);
    mbar_init(bar(kBarPFree0 + 1), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarKFull0 + s), 1);
      mbar_init(bar(kBarVFull0 + s), 1);
      mbar_init(bar(kBarKvEmpty0 + s), 1);
    }
    fence_barrier_init();
  }
  __syncthreads();
  const int item = *item_slot;
  if (item >= items || *abort_flag) break;
  const int split = item / units;
  const int bk = item % units;  // b * Hkv + kv head
  const int b = bk / a.Hkv;
  // 0 <= seqlens[b] <= Lmax is the caller's contract; a length outside it is
  // clamped (so no split reads past its own cache rows) and recorded as
  // MPFA_ERR_INVALID_ARG in the status word
  const int L_in = a.seqlens[b];
  const int L = L_in < 0 ? 0 : (L_in > a.Lmax ? a.Lmax : L_in);
  if (L != L_in && threadIdx.x == 0 && split == 0) record_error(a.err, kErrInvalidArg);
  const int k0 = split * a.chunk;
  const int k1 = min(L, k0 + a.chunk);
  const int ntiles = k1 > k0 ? (k1 - k0 + 127) / 128 : 0;

  if (ntiles == 0) {  // nothing to attend in this split
    if (threadIdx.x < 128)
      for (int n = 0; n < g; ++n) {
        const size_t row = (size_t)bk * g + n;
        a.part_o[(row * a.nsplit + split) * 128 + threadIdx.x] = 0.0f;
        if (threadIdx.x == 0) a.part_lse[row * a.nsplit + split] = -INFINITY;
      }
  } else if (warp == 4) {
    if (lane == 0) {
      const int row0 = bk * a.Lmax + k0;
      int issued = 0;
      for (int j = 0; j < ntiles; ++j) {
        const int s = j % kStages;
        if (j >= kStages &&
            !mbar_wait_tf(bar(kBarKvEmpty0 + s), ((j / kStages) - 1) & 1, a.err, abort_flag))
          break;
        // contiguous cache: rows of (b, KV head) at bk * Lmax; paged pool:
        // key tile k0/128 + j of sequence b lives in page block_table[b][.],
        // whose KV head's 128 rows start at (page * Hkv + head) * 128
        int row = row0 + j * 128;
        if (a.block_table) {
          int page = a.block_table[(size_t)b * a.max_pages + k0 / 128 + j];
          if (page < 0 || page >= a.num_pages) {  // a bad entry reads page 0, and is reported
            record_error(a.err, kErrInvalidArg);
            page = 0;
          }
          row = (page * a.Hkv + bk % a.Hkv) * 128;
        }
        mbar_expect_tx(bar(kBarKFull0 + s), 8192 + 1024);
        tma_load_2d(sbase + kOffK + s * 8192, &map_k, 0, row, bar(kBarKFull0 + s));
        bulk_load(sbase + kOffKs + s * 1024, a.ks + (size_t)row * 8, 1024, bar(kBarKFull0 + s));
        mbar_expect_tx(bar(kBarVFull0 + s), 16384);
        tma_load_2d(sbase + kOffV + s * 16384, &map_v, 0, row, bar(kBarVFull0 + s));
        issued = j + 1;
      }
      for (int j = issued - kStages > 0 ? issued - kStages : 0; j < issued; ++j) {
        const int s = j % kStages;
        mbar_wait_tf(bar(kBarKFull0 + s), (j / kStages) & 1, a.err, nullptr);
        mbar_wait_tf(bar(kBarVFull0 + s), (j / kStages) & 1, a.err, nullptr);
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      const uint32_t id_qk = idesc_nvfp4(128, 16);
      const uint32_t id_pv = idesc_fp8(128, 16, 1, 0);
      const uint32_t id_l = idesc_fp8(128, 16, 0, 0);
      bool ok = mbar_wait_tf(bar(kBarQReady), 0, a.err, abort_flag);
      if (ok) {
        tc_fence_after();
        for (int o = 0; o < 1 + T; ++o)
          for (int kc = 0; kc < 2; ++kc)
            tmem_cp_32x128b_x4(tmem + kColSfQ + 8 * o + 4 * kc,
                               smem_desc(sbase + kOffQs + 1024 * o + 512 * kc, 128, 128, kSwizzleNone));
      }
      auto issue_pv = [&](int jp) -> bool {
        const int bp = jp & 1, sp = jp % kStages;
        if (!mbar_wait_tf(bar(kBarPReady0 + bp), (jp >> 1) & 1, a.err, abort_flag)) return false;
        if (!mbar_wait_tf(bar(kBarVFull0 + sp), (jp / kStages) & 1, a.err, abort_flag)) return false;
        tc_fence_after();
        const uint32_t paddr = sbase + kOffP + 2048 * bp;
        const uint32_t vaddr = sbase + kOffV + 16384 * sp;
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t pdesc = smem_desc(paddr + 32 * kk, 16, 1024, kSwizzle128B);
          mma_fp8_ss(tmem + kColO, smem_desc(vaddr + 4096 * kk, 16, 1024, kSwizzle128B), pdesc,
                     id_pv, (jp > 0 || kk > 0) ? 1u : 0u);
          mma_fp8_ss(tmem + kColL, smem_desc(sbase + kOffOnes, 128, 256, kSwizzleNone), pdesc,
                     id_l, (jp > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(bar(kBarODone));
        if (jp + 2 < ntiles) tc_commit(bar(kBarPFree0 + bp));
        if (jp + kStages < ntiles) tc_commit(bar(kBarKvEmpty0 + sp));
        return true;
      };
      for (int j = 0; ok && j < ntiles; ++j) {
        const int s = j % kStages, bkk = j & 1;
        // bank j % 2 was last read by the softmax of tile j-2, which published
        // P_{j-2} before this thread issued PV_{j-2} (previous iteration)
        if (!mbar_wait_tf(bar(kBarKFull0 + s), (j / kStages) & 1, a.err, abort_flag)) break;
        tc_fence_after();
        const uint32_t sfk = tmem + kColSfK + 8 * s;
        for (int kc = 0; kc < 2; ++kc)
          tmem_cp_32x128b_x4(sfk + 4 * kc,
                             smem_desc(sbase + kOffKs + 1024 * s + 512 * kc, 128, 128, kSwizzleNone));
        const uint32_t dS = tmem + kColS0 + 16 * bkk;
        const uint32_t kaddr = sbase + kOffK + 8192 * s;
        for (int o = 0; o < 1 + T; ++o)
          for (int kc = 0; kc < 2; ++kc)
            mma_nvfp4_ss(dS, smem_desc(kaddr + 32 * kc, 16, 512, kSwizzle64B),
                         smem_desc(sbase + kOffQ + 1024 * o + 32 * kc, 16, 512, kSwizzle64B), id_qk,
                         sfk + 4 * kc, tmem + kColSfQ + 8 * o + 4 * kc, (o > 0 || kc > 0) ? 1u : 0u);
        tc_commit(bar(kBarSFull0 + bkk));
        if (j >= 1 && !issue_pv(j - 1)) {
          ok = false;
          break;
        }
      }
      if (ok) issue_pv(ntiles - 1);
      tc_commit(bar(kBarDrain));
      mbar_wait_tf(bar(kBarDrain), 0, a.err, nullptr);
    }
  } else {
    // ---------------- softmax: thread = key (TMEM lane) ----------------
    const int t = threadIdx.x;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    // B operands: q' rows (n < g) and the rank-one terms broadcast to rows n < g,
    // 16 rows x 64 B, 64-byte swizzle; scale atoms (32 rows x 16 B per chunk).
    if (t < 16 * (1 + T)) {
      const int o = t / 16, n = t % 16;
      uint4 src[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                      make_uint4(0, 0, 0, 0)};
      uint32_t s0 = 0, s1 = 0;
      if (n < g) {
        const uint8_t* cp;
        const uint8_t* sp;
        if (o == 0) {
          cp = a.qc + ((size_t)bk * g + n) * 64;
          sp = a.qs + ((size_t)bk * g + n) * 8;
        } else {
          cp = a.qbc + ((size_t)bk * a.T + (o - 1)) * 64;
          sp = a.qbs + ((size_t)bk * a.T + (o - 1)) * 8;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) src[c] = reinterpret_cast<const uint4*>(cp)[c];
        s0 = sp[0] | (sp[1] << 8) | (sp[2] << 16) | ((uint32_t)sp[3] << 24);
        s1 = sp[4] | (sp[5] << 8) | (sp[6] << 16) | ((uint32_t)sp[7] << 24);
      }
      uint4* dst = reinterpret_cast<uint4*>(smem + kOffQ + 1024 * o + 64 * n);
#pragma unroll
      for (int c = 0; c < 4; ++c) dst[c ^ ((n >> 1) & 3)] = src[c];
      // scale atom: row r holds rows r, r+32, r+64, r+96 -> only r = n < 16 used
      uint32_t* atom = reinterpret_cast<uint32_t*>(smem + kOffQs + 1024 * o);
      atom[n * 4 + 0] = s0;
      atom[128 + n * 4 + 0] = s1;
#pragma unroll
      for (int q = 1; q < 4; ++q) {
        atom[n * 4 + q] = 0;
        atom[128 + n * 4 + q] = 0;
      }
      // rows 16..31 of each atom
      for (int q = 0; q < 4; ++q) {
        atom[(16 + n) * 4 + q] = 0;
        atom[128 + (16 + n) * 4 + q] = 0;
      }
    }
    // ones tile (128 rows x 32 B, E4M3 1.0) and zeroed P^T buffers
    reinterpret_cast<uint4*>(smem + kOffOnes)[2 * t] = make_uint4(0x38383838u, 0x38383838u, 0x38383838u, 0x38383838u);
    reinterpret_cast<uint4*>(smem + kOffOnes)[2 * t + 1] = make_uint4(0x38383838u, 0x38383838u, 0x38383838u, 0x38383838u);
    reinterpret_cast<uint4*>(smem + kOffP)[2 * t] = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(smem + kOffP)[2 * t + 1] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    mbar_arrive(bar(kBarQReady));

    const float cs = __fmul_rn(__fmul_rn(*a.s_q, *a.s_k), log2e_rsqrt_d);
    float m[kMaxG];
#pragma unroll
    for (int n = 0; n < kMaxG; ++n) m[n] = -INFINITY;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int bkk = j & 1;
      if (!named_bar_and(2, 128, mbar_wait_tf(bar(kBarSFull0 + bkk), (j >> 1) & 1, a.err, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[16];
      {
        uint32_t (&s4)[4] = *reinterpret_cast<uint32_t(*)[4]>(&sr[0]);
        uint32_t (&s4b)[4] = *reinterpret_cast<uint32_t(*)[4]>(&sr[4]);
        uint32_t (&s4c)[4] = *reinterpret_cast<uint32_t(*)[4]>(&sr[8]);
        uint32_t (&s4d)[4] = *reinterpret_cast<uint32_t(*)[4]>(&sr[12]);
        const uint32_t sS = tmem + lane_off + kColS0 + 16 * bkk;
        tmem_ld4(sS, s4);
        tmem_ld4(sS + 4, s4b);
        tmem_ld4(sS + 8, s4c);
        tmem_ld4(sS + 12, s4d);
        tmem_ld_wait();
      }
      const int key = k0 + j * 128 + t;
      const bool valid = key < k1;
      float v[kMaxG];
#pragma unroll
      for (int n = 0; n < kMaxG; ++n) v[n] = valid ? __uint_as_float(sr[n]) : -INFINITY;
      // The reference max of head n moves only if some key of this tile has
      // S * cs > m + kRescaleTau; the tile max over the 128 keys (shuffles and
      // shared memory) is needed only then.  Vote first: bit n set if any key
      // of the CTA moves head n.
      uint32_t move = 0;
#pragma unroll
      for (int n = 0; n < kMaxG; ++n)
        if (n < g && (m[n] == -INFINITY ? v[n] != -INFINITY : __fmul_rn(v[n], cs) > m[n] + kRescaleTau))
          move |= 1u << n;
      move = __reduce_or_sync(0xffffffffu, move);
      if (lane == 0) reinterpret_cast<uint32_t*>(red)[64 + warp] = move;
      named_bar_sync(1, 128);
      move = reinterpret_cast<uint32_t*>(red)[64] | reinterpret_cast<uint32_t*>(red)[65] |
             reinterpret_cast<uint32_t*>(red)[66] | reinterpret_cast<uint32_t*>(red)[67];
      float alpha[kMaxG];
#pragma unroll
      for (int n = 0; n < kMaxG; ++n) alpha[n] = 1.0f;
      bool any_change = false;
      if (move) {
        // block max per query row over the 128 keys
#pragma unroll
        for (int n = 0; n < kMaxG; ++n) {
          float mx = v[n];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          if (lane == 0) red[warp * 16 + n] = mx;
        }
        named_bar_sync(1, 128);
#pragma unroll
        for (int n = 0; n < kMaxG; ++n) {
          const float smax = fmaxf(fmaxf(red[n], red[16 + n]), fmaxf(red[32 + n], red[48 + n]));
          const float tmax = __fmul_rn(smax, cs);
          const float mn = (m[n] == -INFINITY || tmax > m[n] + kRescaleTau) ? tmax : m[n];
          alpha[n] = (m[n] == -INFINITY) ? 0.0f : (mn == m[n] ? 1.0f : ex2(m[n] - mn));
          any_change |= (n < g) && (alpha[n] != 1.0f);
          m[n] = mn;
        }
      }
      // P^T: row n, column key (128-byte rows, 128-byte swizzle).  Buffer
      // j % 2 was last read by PV_{j-2}; its own barrier completes once per
      // two tiles, so the parity cannot run two phases ahead of this wait.
      if (j >= 2 && !named_bar_and(2, 128, mbar_wait_tf(bar(kBarPFree0 + bkk), ((j >> 1) - 1) & 1,
                                                     a.err, abort_flag))) {
        ok = false;
        break;
      }
      uint8_t* pt = smem + kOffP + 2048 * bkk;
#pragma unroll
      for (int n = 0; n < kMaxG; ++n) {
        if (n < g) {
          const float pv = (m[n] == -INFINITY) ? 0.0f : ex2(fmaf(v[n], cs, kPShift - m[n]));
          pt[n * 128 + ((((t >> 4) ^ (n & 7))) << 4) + (t & 15)] = (uint8_t)e4m3_pos(pv);
        }
      }
      fence_proxy_async_smem();
      // correction of O^T and L (columns n < g) once PV_{j-1} has landed
      if (j > 0 && any_change) {
        if (!named_bar_and(2, 128, mbar_wait_tf(bar(kBarODone), (j - 1) & 1, a.err, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t o16[16], l16[16];
        {
          uint32_t (&oa)[4] = *reinterpret_cast<uint32_t(*)[4]>(&o16[0]);
          uint32_t (&ob)[4] = *reinterpret_cast<uint32_t(*)[4]>(&o16[4]);
          uint32_t (&oc)[4] = *reinterpret_cast<uint32_t(*)[4]>(&o16[8]);
          uint32_t (&od)[4] = *reinterpret_cast<uint32_t(*)[4]>(&o16[12]);
          uint32_t (&la)[4] = *reinterpret_cast<uint32_t(*)[4]>(&l16[0]);
          uint32_t (&lb)[4] = *reinterpret_cast<uint32_t(*)[4]>(&l16[4]);
          uint32_t (&lc)[4] = *reinterpret_cast<uint32_t(*)[4]>(&l16[8]);
          uint32_t (&ld)[4] = *reinterpret_cast<uint32_t(*)[4]>(&l16[12]);
          const uint32_t oO = tmem + lane_off + kColO, oL = tmem + lane_off + kColL;
          tmem_ld4(oO, oa);
          tmem_ld4(oO + 4, ob);
          tmem_ld4(oO + 8, oc);
          tmem_ld4(oO + 12, od);
          tmem_ld4(oL, la);
          tmem_ld4(oL + 4, lb);
          tmem_ld4(oL + 8, lc);
          tmem_ld4(oL + 12, ld);
          tmem_ld_wait();
#pragma unroll
          for (int n = 0; n < kMaxG; ++n) {
            o16[n] = __float_as_uint(__uint_as_float(o16[n]) * alpha[n]);
            l16[n] = __float_as_uint(__uint_as_float(l16[n]) * alpha[n]);
          }
          tmem_st4(oO, oa);
          tmem_st4(oO + 4, ob);
          tmem_st4(oO + 8, oc);
          tmem_st4(oO + 12, od);
          tmem_st4(oL, la);
          tmem_st4(oL + 4, lb);
          tmem_st4(oL + 8, lc);
          tmem_st4(oL + 12, ld);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(kBarPReady0 + bkk));
      named_bar_sync(1, 128);  // red[] is reused by the next tile
    }
    if (ok && named_bar_and(2, 128, mbar_wait_tf(bar(kBarODone), (ntiles - 1) & 1, a.err, abort_flag))) {
      tc_fence_after();
      uint32_t o16[16], l16[16];
      {
        uint32_t (&oa)[4] = *reinterpret_cast<uint32_t(*)[4]>(&o16[0]);
        uint32_t (&ob)[4] = *reinterpret_cast<uint32_t(*)[4]>(&o16[4]);
        uint32_t (&oc)[4] = *reinterpret_cast<uint32_t(*)[4]>(&o16[8]);
        uint32_t (&od)[4] = *reinterpret_cast<uint32_t(*)[4]>(&o16[12]);
        uint32_t (&la)[4] = *reinterpret_cast<uint32_t(*)[4]>(&l16[0]);
        uint32_t (&lb)[4] = *reinterpret_cast<uint32_t(*)[4]>(&l16[4]);
        uint32_t (&lc)[4] = *reinterpret_cast<uint32_t(*)[4]>(&l16[8]);
        uint32_t (&ld)[4] = *reinterpret_cast<uint32_t(*)[4]>(&l16[12]);
        const uint32_t oO = tmem + lane_off + kColO, oL = tmem + lane_off + kColL;
        tmem_ld4(oO, oa);
        tmem_ld4(oO + 4, ob);
        tmem_ld4(oO + 8, oc);
        tmem_ld4(oO + 12, od);
        tmem_ld4(oL, la);
        tmem_ld4(oL + 4, lb);
        tmem_ld4(oL + 8, lc);
        tmem_ld4(oL + 12, ld);
        tmem_ld_wait();
      }
      const float sv = *a.s_v;
#pragma unroll
      for (int n = 0; n < kMaxG; ++n) {
        if (n >= g) break;
        const float l = __uint_as_float(l16[n]);
        const size_t row = (size_t)bk * g + n;
        a.part_o[(row * a.nsplit + split) * 128 + t] = __uint_as_float(o16[n]) * __fdiv_rn(sv, l);
        if (t == 0)
          a.part_lse[row * a.nsplit + split] =
              0.69314718055994531f * (m[n] + __log2f(l) - kPShift);
      }
    }
  }
  // the item is done in every role; item_slot and the barriers are rewritten next
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// combine
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(128) combine_kernel(DecodeArgs a) {
  pdl_wait();
  const size_t row = blockIdx.x;  // b * Hq + h
  const int c = threadIdx.x;
  float lmax = -INFINITY;
  for (int s = 0; s < a.nsplit; ++s) lmax = fmaxf(lmax, a.part_lse[row * a.nsplit + s]);
  float acc = 0.0f, wsum = 0.0f;
  if (lmax != -INFINITY) {
    for (int s = 0; s < a.nsplit; ++s) {
      const float ls = a.part_lse[row * a.nsplit + s];
      if (ls == -INFINITY) continue;
      const float w = __expf(ls - lmax);
      wsum += w;
      acc = fmaf(w, a.part_o[(row * a.nsplit + s) * 128 + c], acc);
    }
  }
  const float o = wsum > 0.0f ? acc / wsum : 0.0f;
  reinterpret_cast<__nv_bfloat16*>(a.o)[row * 128 + c] = __float2bfloat16_rn(o);
  if (a.lse && c == 0) {
    float lse = wsum > 0.0f ? lmax + __logf(wsum) : -INFINITY;
    if (a.kbar && wsum > 0.0f) {
      // key-side smoothing: the dropped logit part s_q * (q codes + the
      // group's rank-one terms) . kbar / sqrt(d)
      const int g = a.Hq / a.Hkv;
      float dq = a.q_kbar[row];
      if (a.compensate) dq += a.q_kbar[(size_t)a.B * a.Hq + row / g];
      lse += __fmul_rn(__fmul_rn(dq, *a.s_q), 0.08838834764831845f);
    }
    a.lse[row] = lse;
  }
}

}  // namespace

// Resident split CTAs per SM, from the kernel's registers and shared memory
// against the SM's register file and shared-memory capacity (1 KB of each
// CTA's shared memory is reserved by the system).
static int split_ctas_per_sm(int dev) {
  static std::atomic<int> occ_of[kMaxDevices];
  if (dev < 0 || dev >= kMaxDevices) return 1;
  int occ = occ_of[dev].load(std::memory_order_acquire);
  if (occ > 0) return occ;
  int smem_sm = 0, regs_sm = 0;
  cudaFuncAttributes fa{};
  if (cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) ==
          cudaSuccess &&
      cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) ==
          cudaSuccess &&
      cudaFuncGetAttributes(&fa, split_kernel) == cudaSuccess && fa.numRegs > 0) {
    const int by_smem = smem_sm / (int)(kSmemBytes + fa.sharedSizeBytes + 1024);
    const int regs_warp = ((fa.numRegs * 32 + 255) / 256) * 256;
    const int by_regs = regs_sm / (regs_warp * (kThreads / 32));
    occ = by_smem < by_regs ? by_smem : by_regs;
  }
  if (occ < 1) occ = 1;
  occ_of[dev].store(occ, std::memory_order_release);
  return occ;
}

// Chunk (keys per split) for B x Hkv units of Lmax keys.  The split kernel
// is persistent with a dynamic item queue, so its time is about
//   (all tiles + a fixed cost per item) / resident slots  +  one item
// (the last item taken finishes alone).  The fixed cost (query codes,
// barrier set-up, pipeline fill and drain, partial results) is taken as
// 8 tiles' time; lengths are assumed to be Lmax.  The split count that
// minimises this is used.
int decode_default_chunk(int B, int Hkv, int Lmax, int num_sms) {
  constexpr double kItemCostTiles = 8.0;
  const double units = (double)B * Hkv;
  const double slots = (double)split_ctas_per_sm(current_device()) * num_sms;
  const long long tiles = (Lmax + 127) / 128;
  long long best_n = 1;
  double best_cost = -1.0;
  for (long long n = 1; n <= tiles; ++n) {
    const long long per_item = (tiles + n - 1) / n;
    if (n > 1 && (tiles + per_item - 1) / per_item < n) continue;  // same chunk as a smaller n
    const double cost = units * ((double)tiles + n * kItemCostTiles) / slots + (double)per_item;
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_n = n;
    }
  }
  return (int)(((tiles + best_n - 1) / best_n) * 128);
}

size_t decode_workspace_bytes(int B, int Hq, int Hkv, int nsplit) {
  auto r = [](size_t x) { return (x + 255) & ~size_t(255); };
  return r(256) + r(256) + r((size_t)B * Hq * 64) + r((size_t)B * Hq * 8) +
         r((size_t)B * Hkv * 2 * 64) + r((size_t)B * Hkv * 2 * 8) +
         r((size_t)B * Hkv * 128 * 4) + r((size_t)B * Hq * nsplit * 128 * 4) +
         r((size_t)B * Hq * nsplit * 4) + r((size_t)B * (Hq + Hkv) * 4);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  CUtensorMap mk, mv;
  const uint64_t rows = a.block_table ? (uint64_t)a.num_pages * a.Hkv * 128
                                      : (uint64_t)a.B * a.Hkv * a.Lmax;
  if (!make_map_2d_u8(&mk, a.kc, 64, rows, 128, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_map_2d_u8(&mv, a.vc, 128, rows, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  static std::atomic<bool> attr_set[kMaxDevices];
  {
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(split_kernel), kSmemBytes,
                                  current_device(), attr_set);
    if (e != cudaSuccess) return e;
  }
  // the amax word and the split kernel's item counter (same 256-byte slot)
  cudaError_t e = cudaMemsetAsync(a.amax, 0, 256, stream);
  if (e != cudaSuccess) return e;
  dq_stats_kernel<<<a.B * a.Hkv, 128, 0, stream>>>(a);
  const int rows_q = a.B * a.Hq + (a.compensate ? a.B * a.Hkv : 0);
  // the kernels after the statistics may start while their predecessor
  // finishes (each waits for it before reading its results)
  e = launch_pdl(dq_quant_kernel, dim3((rows_q * 8 + 127) / 128), dim3(128), 0, stream, a);
  if (e != cudaSuccess) return e;
  // persistent: one CTA per resident slot (or fewer if there are fewer items)
  const int items = a.B * a.Hkv * a.nsplit;
  const int sms = sm_count(current_device());
  const int slots = split_ctas_per_sm(current_device()) * (sms > 0 ? sms : 1);
  DecodeArgs ka = a;
  ka.work = reinterpret_cast<int*>(a.amax + 32);
  e = launch_pdl(split_kernel, dim3(items < slots ? items : slots), dim3(kThreads), kSmemBytes,
                 stream, mk, mv, ka, (float)(1.4426950408889634 / std::sqrt(128.0)));
  if (e != cudaSuccess) return e;
  e = launch_pdl(combine_kernel, dim3(a.B * a.Hq), dim3(128), 0, stream, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mpfa
