// prefill.cu -- MpFA QK4PV8 prefill forward on sm_103a.
//
// Method (MpFA abstract): S = Q K^T on block-scaled NVFP4 tensor cores, the
// rank-one smoothing term (the T NVFP4 terms of the query-block mean, the
// same row for all 128 rows) issued as extra MMAs into the same score
// accumulator, an online softmax (FlashAttention-2 section of the
// "FlashAttention压到4位" explainer), P converted to FP8 E4M3 in tensor
// memory and multiplied by FP8 V on the tensor core.  The running sum l comes
// out of the same MMA: each V stage is followed in shared memory by a tile of
// E4M3 ones that the PV product reads as 16 extra columns (N = 144), so the
// denominator consumes exactly the codes the numerator consumes (the
// explainer's Direct-P section states that rule) at no extra instruction.
//
// One CTA computes one 128-row query tile of one (batch, head):
//   warp 8    TMA producer: Q tile once, then K / K-scale tiles through a
//             ring of kKStages stages and V tiles through kVStages stages.
//   warps 9, 11  QK issuers, one per score bank (warp 9 the even tiles,
//             warp 11 the odd ones), each with its own TMEM slot for K's
//             block scales: tcgen05.cp of the scales, QK^T and the rank-one
//             MMAs into bank j % 2, QK_{j+2} as soon as the softmax has
//             loaded S_j into registers.  Neither thread's tiles wait behind
//             the other's.
//   warp 10   PV issuer: once the softmax has published P_j, PV_j (with the
//             row sum).  Each tcgen05 instruction costs its issuing thread on
//             the order of a hundred cycles while the softmax warps load the
//             scheduler it shares, hence three issuing threads on three
//             schedulers.
//   warps 0-7 softmax + correction + epilogue.  Warp w owns TMEM lanes
//             32(w%4)..32(w%4)+31 (query rows) for the KV tiles of parity
//             w/4: thread = one query row, all 128 keys of its tiles.  The two
//             warps on a scheduler thus alternate tiles, so one's
//             exponentials overlap the other's loads, maxima and stores; the
//             only exchange is the row's reference max, handed from the
//             owner of tile j to the owner of tile j+1 through shared memory.
// Tensor memory (512 columns): S0 [0,128) S1 [128,256) O [256,384) and the
// row sum l at 384 (columns [384,400) all hold l), P0 [416,448) P1 [448,480),
// block scales: Q [400,408), K slot 0 [408,416), rank-one terms
// [480,480+8T), K slot 1 [496,504).  P has its own columns so the scores
// of tile j+2 can be computed into bank j % 2 as soon as the softmax has read
// tile j, while PV_j still reads P_j.
#include <cmath>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "device.cuh"
#include "internal.h"

namespace mpfa {

bool make_map_2d_u8(CUtensorMap* m, const void* base, uint64_t inner_bytes, uint64_t rows,
                    uint32_t box_rows, CUtensorMapSwizzle sw);

namespace {

constexpr int kKStages = 4;   // K tiles: released once the softmax has loaded S
constexpr int kVStages = 3;   // V tiles: released once PV has read them
constexpr int kSfSlots = 2;   // TMEM block-scale slots for K: slot j % 2, one per QK issuer
constexpr int kThreads = 384;
// QK issuers: warp 9 for the even tiles (score bank 0, scale slot 0), warp 11
// for the odd ones (bank 1, slot 1)
constexpr int kWarpTma = 8, kWarpMma = 9, kWarpPv = 10, kWarpMma2 = 11;
constexpr int kSoftmaxThreads = 256;
constexpr int kTileThreads = 128;   // softmax threads that own one KV tile
constexpr int kTmemCols = 512;

constexpr uint32_t kColS0 = 0, kColO = 256, kColL = 384, kColP0 = 416, kColSfQ = 400,
                   kColSfQb = 480;
// K block-scale slot i of QK issuer i (8 columns each, 4-aligned as the MMA
// requires)
__device__ __forceinline__ uint32_t col_sf_k(int i) { return i == 0 ? 408u : 496u; }

// barrier indices
enum : int {
  kBarQFull = 0,
  kBarQbReady = 1,
  kBarSFull0 = 2,                      // +bank: scores of tile j in bank j % 2
  kBarPReady0 = 4,                     // +bank: P_j published in P bank j % 2
  kBarDrain = 6,
  kBarSRead0 = 7,                      // +K stage: S_j (K stage j % 4) loaded by the softmax
  kBarKFull0 = kBarSRead0 + kKStages,  // +K stage
  kBarVFull0 = kBarKFull0 + kKStages,  // +V stage
  kBarODone0 = kBarVFull0 + kVStages,  // +V stage: PV_j (V stage j % 3) completed
  kBarMax0 = kBarODone0 + kVStages,    // +2*quadrant+parity: reference max handed to that parity
  kBarQSf = kBarMax0 + 8,              // Q and rank-one block scales copied into TMEM
  kNumBars = kBarQSf + 1,
};

// shared memory layout (offsets from a 1024-byte aligned base)
constexpr uint32_t kOffQ = 0;                           // 8 KB
constexpr uint32_t kOffQb = kOffQ + 8192;               // 2 x 8 KB
constexpr uint32_t kOffK = kOffQb + 2 * 8192;            // kKStages x 8 KB
// V stage s: 16 KB of V at kOffV + 32 KB * s, then 16 KB of E4M3 ones (the
// second 128-byte atom of the N = 144 operand, kVOnesLbo bytes further on)
constexpr uint32_t kVStageBytes = 32768, kVOnesLbo = 16384;
constexpr uint32_t kOffV = kOffK + kKStages * 8192;           // kVStages x 32 KB
constexpr uint32_t kOffQs = kOffV + kVStages * kVStageBytes;  // 1 KB
constexpr uint32_t kOffQbs = kOffQs + 1024;                   // 2 x 1 KB
constexpr uint32_t kOffKs = kOffQbs + 2048;                   // kKStages x 1 KB
constexpr uint32_t kOffMax = kOffKs + kKStages * 1024;        // 128 floats: reference max per row
constexpr uint32_t kOffBar = kOffMax + 512;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemUsed = kOffMisc + 64;
// More than half an SM's shared memory, so a single CTA owns the SM and its
// 512 TMEM columns.
constexpr uint32_t kSmemBytes = 168 * 1024;
static_assert(kSmemUsed + 1024 <= kSmemBytes, "shared memory layout overflow");

struct Params {
  PrefillArgs a;
  float log2e_rsqrt_d;  // fp32(log2(e) / sqrt(128))
  int q_tiles;
  int wave;             // CTAs resident at once (one per SM)
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
    mbar_init(bar(kBarQbReady), kSoftmaxThreads);
    for (int b2 = 0; b2 < 2; ++b2) {
      mbar_init(bar(kBarSFull0 + b2), 1);
      mbar_init(bar(kBarPReady0 + b2), kTileThreads);
    }
    mbar_init(bar(kBarDrain), 3);   // one commit from each issuing thread
    mbar_init(bar(kBarQSf), 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(bar(kBarSRead0 + s), kTileThreads);
      mbar_init(bar(kBarKFull0 + s), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(bar(kBarVFull0 + s), 1);
      mbar_init(bar(kBarODone0 + s), 1);
    }
    for (int i = 0; i < 8; ++i) mbar_init(bar(kBarMax0 + i), 32);
    fence_barrier_init();
  }
  if (warp == kWarpMma) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpTma) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      prefetch_tensormap(&map_q);
      prefetch_tensormap(&map_k);
      prefetch_tensormap(&map_v);
      // L2 prefetch of the query-side inputs of the CTA one wave later (one
      // CTA per SM): its Q tile is otherwise a DRAM miss on its critical path
      {
        const unsigned nxt = blockIdx.x + (unsigned)p.wave;
        if (nxt < gridDim.x) {
          const int qt2 = p.q_tiles - 1 - (int)(nxt / bh_count);
          const int bh2 = (int)(nxt % bh_count);
          const size_t qrow2 = (size_t)bh2 * a.N + (size_t)qt2 * 128;
          prefetch_l2_bulk(a.qc + qrow2 * 64, 8192);
          prefetch_l2_bulk(a.qs + qrow2 * 8, 1024);
          if (T > 0) {
            const size_t qb2 = ((size_t)bh2 * (a.N / 128) + qt2) * a.T;
            prefetch_l2_bulk(a.qbc + qb2 * 64, 64u * a.T);
            prefetch_l2_line(a.qbs + qb2 * 8);
          }
        }
      }
      const int qrow = (b * a.Hq + h) * a.N + qt * 128;
      mbar_expect_tx(bar(kBarQFull), 8192 + 1024);
      tma_load_2d(sbase + kOffQ, &map_q, 0, qrow, bar(kBarQFull));
      bulk_load(sbase + kOffQs, a.qs + (size_t)qrow * 8, 1024, bar(kBarQFull));
      const int kvrow0 = (b * a.Hkv + hk) * a.N;
      // loads in the order the MMA warp consumes them: K_0, K_1, then
      // V_j and K_{j+2} for j = 0, 1, ...
      int k_issued = 0, v_issued = 0;
      auto load_k = [&](int j) -> bool {
        const int s = j % kKStages;
        // stage s held K_{j-4}: free once the softmax has loaded S_{j-4}
        if (j >= kKStages &&
            !mbar_wait(bar(kBarSRead0 + s), ((j / kKStages) - 1) & 1, a.err, abort_flag))
          return false;
        const int row = kvrow0 + j * 128;
        mbar_expect_tx(bar(kBarKFull0 + s), 8192 + 1024);
        tma_load_2d(sbase + kOffK + s * 8192, &map_k, 0, row, bar(kBarKFull0 + s));
        bulk_load(sbase + kOffKs + s * 1024, a.ks + (size_t)row * 8, 1024, bar(kBarKFull0 + s));
        k_issued = j + 1;
        return true;
      };
      auto load_v = [&](int j) -> bool {
        const int s = j % kVStages;
        // stage s held V_{j-3}: free once PV_{j-3} has completed
        if (j >= kVStages &&
            !mbar_wait(bar(kBarODone0 + s), ((j / kVStages) - 1) & 1, a.err, abort_flag))
          return false;
        mbar_expect_tx(bar(kBarVFull0 + s), 16384);
        tma_load_2d(sbase + kOffV + s * kVStageBytes, &map_v, 0, kvrow0 + j * 128,
                    bar(kBarVFull0 + s));
        v_issued = j + 1;
        return true;
      };
      bool lok = load_k(0) && (nkv < 2 || load_k(1));
      for (int j = 0; lok && j < nkv; ++j) {
        if (!load_v(j)) break;
        if (j + 2 < nkv && !load_k(j + 2)) break;
      }
      // drain: every stage's last load must have landed before the CTA exits
      for (int j = k_issued - kKStages > 0 ? k_issued - kKStages : 0; j < k_issued; ++j)
        mbar_wait(bar(kBarKFull0 + j % kKStages), (j / kKStages) & 1, a.err, nullptr);
      for (int j = v_issued - kVStages > 0 ? v_issued - kVStages : 0; j < v_issued; ++j)
        mbar_wait(bar(kBarVFull0 + j % kVStages), (j / kVStages) & 1, a.err, nullptr);
    }
  } else if (warp == kWarpMma || warp == kWarpMma2) {
    // ---------------- QK issuers ----------------
    // One thread per score bank, each issuing every other tile with its own
    // K scale slot: each accumulator and slot has a single issuing thread,
    // and neither thread's tiles wait behind the other's.
    if (lane == 0) {
      const int par = warp == kWarpMma ? 0 : 1;
      const uint32_t id_qk = idesc_nvfp4(128, 128);
      bool ok;
      if (par == 0) {
        ok = mbar_wait(bar(kBarQFull), 0, a.err, abort_flag) &&
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
          tc_commit(bar(kBarQSf));
        }
      } else {
        // the other issuer has copied the Q and rank-one scales into TMEM
        // (its commit also says Q and the rank-one operand are in shared
        // memory)
        ok = mbar_wait(bar(kBarQSf), 0, a.err, abort_flag);
        if (ok) tc_fence_after();
      }
      // shared-memory descriptors built once: the start address sits in the
      // low field in 16-byte units, so a K stage or a rank-one term (8 KB)
      // is +512 and the second 64-element K chunk (32 B) +2; every address
      // stays below 2^18, inside that field
      const uint64_t dq0 = smem_desc(sbase + kOffQ, 16, 512, kSwizzle64B);
      const uint64_t dk0 = smem_desc(sbase + kOffK, 16, 512, kSwizzle64B);
      const uint64_t dqb0 = smem_desc(sbase + kOffQb, 16, 512, kSwizzle64B);
      // QK_j (and the rank-one MMAs) into score bank j % 2
      auto issue_qk = [&](int j) -> bool {
        const int s = j % kKStages, bk = j & 1;
        if (!mbar_wait(bar(kBarKFull0 + s), (j / kKStages) & 1, a.err, abort_flag)) return false;
        tc_fence_after();
        // K_j's scales into this issuer's slot j % 2; its last reader,
        // QK_{j-2}, completed before the softmax loaded S_{j-2} (waited for)
        const uint32_t sfk = tmem + col_sf_k(j % kSfSlots);
        for (int kc = 0; kc < 2; ++kc)
          tmem_cp_32x128b_x4(sfk + 4 * kc,
                             smem_desc(sbase + kOffKs + 1024 * s + 512 * kc, 128, 128, kSwizzleNone));
        const uint32_t dS = tmem + kColS0 + 128 * bk;
        const uint64_t dk = dk0 + 512u * (uint32_t)s;
        mma_nvfp4_ss(dS, dq0, dk, id_qk, tmem + kColSfQ, sfk, 0u);
        mma_nvfp4_ss(dS, dq0 + 2u, dk + 2u, id_qk, tmem + kColSfQ + 4, sfk + 4, 1u);
        if (T > 0) {
          mma_nvfp4_ss(dS, dqb0, dk, id_qk, tmem + kColSfQb, sfk, 1u);
          mma_nvfp4_ss(dS, dqb0 + 2u, dk + 2u, id_qk, tmem + kColSfQb + 4, sfk + 4, 1u);
        }
        if (T > 1) {
          mma_nvfp4_ss(dS, dqb0 + 512u, dk, id_qk, tmem + kColSfQb + 8, sfk, 1u);
          mma_nvfp4_ss(dS, dqb0 + 514u, dk + 2u, id_qk, tmem + kColSfQb + 12, sfk + 4, 1u);
        }
        tc_commit(bar(kBarSFull0 + bk));
        return true;
      };
      for (int j = par; ok && j < nkv; j += 2) {
        // the softmax has loaded S_{j-2}: bank j % 2 and slot j % 2 are free.
        // SRead for stage (j-2) % 4 cannot be a phase further on: that needs
        // S_{j+2}.
        if (j >= 2 && !mbar_wait(bar(kBarSRead0 + (j - 2) % kKStages), ((j - 2) / kKStages) & 1,
                                 a.err, abort_flag))
          break;
        if (!issue_qk(j)) break;
      }
      // drain this thread's tensor-core work before the CTA releases TMEM
      tc_commit(bar(kBarDrain));
      mbar_wait(bar(kBarDrain), 0, a.err, nullptr);
    }
  } else if (warp == kWarpPv) {
    // ---------------- PV issuer ----------------
    if (lane == 0) {
      const uint32_t id_pv = idesc_fp8(128, 144, 0, 1);   // 128 V columns + 16 ones
      for (int j = 0; j < nkv; ++j) {
        const int bp = j & 1, sp = j % kVStages;
        // the softmax has published P_j in P bank j % 2
        if (!mbar_wait(bar(kBarPReady0 + bp), (j >> 1) & 1, a.err, abort_flag)) break;
        if (!mbar_wait(bar(kBarVFull0 + sp), (j / kVStages) & 1, a.err, abort_flag)) break;
        tc_fence_after();
        const uint32_t pcol = tmem + kColP0 + 32 * bp;
        const uint32_t vaddr = sbase + kOffV + sp * kVStageBytes;
        for (int kk = 0; kk < 4; ++kk)
          mma_fp8_ts(tmem + kColO, pcol + 8 * kk,
                     smem_desc(vaddr + 4096 * kk, kVOnesLbo, 1024, kSwizzle128B), id_pv,
                     (j > 0 || kk > 0) ? 1u : 0u);
        tc_commit(bar(kBarODone0 + sp));
      }
      tc_commit(bar(kBarDrain));
      mbar_wait(bar(kBarDrain), 0, a.err, nullptr);
    }
  } else {
    // ---------------- softmax / correction / epilogue ----------------
    const int half = warp >> 2;              // prologue split; afterwards the tile parity
    const int row = threadIdx.x & 127;       // query row = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    // Rank-one operand tiles: every row holds the block's term t (same 64
    // bytes), written with the 64-byte swizzle the TMA applies to Q and K.
    const int nblk = a.N / 128;
    if (half == 0) {
      for (int t = 0; t < T; ++t) {
        const uint8_t* src = a.qbc + (((size_t)bh * nblk + qt) * a.T + t) * 64;
        uint4* dst = reinterpret_cast<uint4*>(smem + kOffQb + 8192 * t + 64 * row);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          dst[c ^ ((row >> 1) & 3)] = reinterpret_cast<const uint4*>(src)[c];
      }
    } else {
      for (int t = 0; t < T; ++t) {
        const uint8_t* ssrc = a.qbs + (((size_t)bh * nblk + qt) * a.T + t) * 8;
        uint32_t w0 = *reinterpret_cast<const uint32_t*>(ssrc);
        uint32_t w1 = *reinterpret_cast<const uint32_t*>(ssrc + 4);
        reinterpret_cast<uint32_t*>(smem + kOffQbs + 1024 * t)[row] = w0;
        reinterpret_cast<uint32_t*>(smem + kOffQbs + 1024 * t + 512)[row] = w1;
      }
    }
    // the ones atoms beside the V stages (E4M3 1.0 = 0x38; every byte equal,
    // so the 128-byte swizzle leaves them unchanged)
    for (int s = 0; s < kVStages; ++s) {
      uint4* ones = reinterpret_cast<uint4*>(smem + kOffV + s * kVStageBytes + kVOnesLbo);
      for (int i = threadIdx.x; i < (int)(kVOnesLbo / 16); i += kSoftmaxThreads)
        ones[i] = make_uint4(0x38383838u, 0x38383838u, 0x38383838u, 0x38383838u);
    }
    fence_proxy_async_smem();
    mbar_arrive(bar(kBarQbReady));

    // Tiles j = par, par + 2, ... of this warp; the owner of tile j hands
    // the row's reference max m_j to the owner of tile j+1 (bar kBarMax0 +
    // 2*quadrant + receiving parity; one hand-over per phase, and a phase
    // cannot run ahead because the next hand-over needs the reply).
    const int par = half, quad = warp & 3;
    float* mrow = reinterpret_cast<float*>(smem + kOffMax);
    const uint32_t bar_in = bar(kBarMax0 + 2 * quad + par);
    const uint32_t bar_out = bar(kBarMax0 + 2 * quad + (par ^ 1));
    const float cs = __fmul_rn(__fmul_rn(*a.s_q, *a.s_k), p.log2e_rsqrt_d);
    float m = -INFINITY;
    bool ok = true;
    for (int j = par; j < nkv; j += 2) {
      const int bk = par;   // == j & 1
      const int it = j >> 1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarSFull0 + bk), it & 1, a.err, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sS = tmem + lane_off + kColS0 + 128 * bk;
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(sS + 32 * c, sr[c]);
      tmem_ld_wait();
      // S_j is in registers: bank j % 2 and K stage j % 4 may be reused
      tc_fence_before();
      mbar_arrive(bar(kBarSRead0 + j % kKStages));
      if (a.causal && j == qt) {  // diagonal tile: key > row is masked
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * c + i > row) sr[c][i] = 0xFF800000u;  // -inf
      }
      // tile max over the row's 128 keys (3-input max tree)
      float pm[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int e = 8 * k;
        pm[k] = fmax3(fmax3(__uint_as_float(sr[e >> 5][e & 31]),
                            __uint_as_float(sr[e >> 5][(e + 1) & 31]),
                            __uint_as_float(sr[e >> 5][(e + 2) & 31])),
                      fmax3(__uint_as_float(sr[e >> 5][(e + 3) & 31]),
                            __uint_as_float(sr[e >> 5][(e + 4) & 31]),
                            __uint_as_float(sr[e >> 5][(e + 5) & 31])),
                      fmaxf(__uint_as_float(sr[e >> 5][(e + 6) & 31]),
                            __uint_as_float(sr[e >> 5][(e + 7) & 31])));
      }
      const float smax = fmax3(fmax3(fmax3(pm[0], pm[1], pm[2]), fmax3(pm[3], pm[4], pm[5]),
                                     fmax3(pm[6], pm[7], pm[8])),
                               fmax3(pm[9], pm[10], pm[11]),
                               fmax3(fmax3(pm[12], pm[13], pm[14]), pm[15], -INFINITY));
      // reference max of the row after tile j-1, from that tile's owner
      if (j > 0) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar_in, ((j - 1) >> 1) & 1, a.err, abort_flag))) {
          ok = false;
          break;
        }
        m = mrow[row];
      }
      // cs > 0, so max_i(S_i * cs) == (max_i S_i) * cs exactly.  The reference
      // max moves only when the tile max exceeds it by more than kRescaleTau,
      // so O and L rarely need a rescale once the first tiles are done.
      const float tmax = __fmul_rn(smax, cs);
      const float mn = (m == -INFINITY || tmax > m + kRescaleTau) ? tmax : m;
      if (j + 1 < nkv) {
        mrow[row] = mn;
        mbar_arrive(bar_out);
      }
      const float alpha = (m == -INFINITY) ? 0.0f : (mn == m ? 1.0f : ex2(m - mn));
      const float bias = kPShift - mn;  // P8 = E4M3(2^(t - m) * 2^kPShift)
      uint32_t pw[32];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int w = 0; w < 8; ++w)
          pw[8 * c + w] = e4m3x4(ex2(fmaf(__uint_as_float(sr[c][4 * w]), cs, bias)),
                                 ex2(fmaf(__uint_as_float(sr[c][4 * w + 1]), cs, bias)),
                                 ex2(fmaf(__uint_as_float(sr[c][4 * w + 2]), cs, bias)),
                                 ex2(fmaf(__uint_as_float(sr[c][4 * w + 3]), cs, bias)));
      // correction: O and L scale by alpha once PV_{j-1} has landed (PV_j is
      // issued only after this tile's P is published)
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarODone0 + (j - 1) % kVStages),
                                               ((j - 1) / kVStages) & 1, a.err, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t oO = tmem + lane_off + kColO;
#pragma unroll 1
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
      // P bank j % 2 was last read by PV_{j-2}: wait for it to complete
      // (its ODone phase cannot be overtaken: PV_{j+1} needs this P first).
      if (j >= 2 && !__all_sync(0xffffffffu, mbar_wait(bar(kBarODone0 + (j - 2) % kVStages),
                                                        ((j - 2) / kVStages) & 1, a.err,
                                                        abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      tmem_st32(tmem + lane_off + kColP0 + 32 * bk, pw);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(kBarPReady0 + bk));
      m = mn;
    }
    // epilogue: the owner of the last tile holds the final reference max
    if (ok && nkv > 0 && par == ((nkv - 1) & 1) &&
        __all_sync(0xffffffffu, mbar_wait(bar(kBarODone0 + (nkv - 1) % kVStages),
                                          ((nkv - 1) / kVStages) & 1, a.err, abort_flag))) {
      tc_fence_after();
      uint32_t l4[4];
      tmem_ld4(tmem + lane_off + kColL, l4);
      tmem_ld_wait();
      const float l = __uint_as_float(l4[0]);
      const float sc = __fdiv_rn(*a.s_v, l);
      const size_t grow = (size_t)qt * 128 + row;
      uint4* out = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.o) +
                                            (((size_t)b * a.N + grow) * a.Hq + h) * 128);
#pragma unroll 1
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
      if (a.lse)
        a.lse[(size_t)bh * a.N + grow] = 0.69314718055994531f * (m + __log2f(l) - kPShift);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
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
  {
    static int sms = 0;
    if (!sms) {
      int dev = 0;
      cudaGetDevice(&dev);
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (sms <= 0) sms = 148;
    }
    p.wave = sms;
  }
  const unsigned grid = (unsigned)(p.q_tiles * a.B * a.Hq);
  if (grid == 0) return cudaSuccess;
  prefill_kernel<<<grid, kThreads, kSmemBytes, stream>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace mpfa
