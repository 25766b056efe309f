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
// Persistent: one CTA per SM walks a fixed list of work items (128-row query
// tile of one (batch, head)), heaviest causal items first, dealt to the CTAs
// in a snake order so every CTA gets a near-equal share of KV tiles.  All
// roles see the CTA's KV tiles as one stream g = 0, 1, ... across items, and
// every ring, bank and barrier phase is indexed by g, so the next item's Q,
// K and scores are in flight while the previous item's last tiles and its
// epilogue finish.
//   warp 8    TMA producer (whole warp): per item the Q tile and scales into
//             one of two Q buffers, the rank-one operand tile built by all 32
//             lanes; K / K-scale tiles through kKStages stages and V tiles
//             through kVStages stages, each ring refilled as soon as its own
//             stage frees up (polled, so a late V stage never holds back K).
//   warps 9, 11  QK issuers, one per score bank (warp 9 the even tiles of
//             the stream, warp 11 the odd ones), each with its own TMEM slot
//             for K's block scales: tcgen05.cp of the scales, QK^T and the
//             rank-one MMAs into bank g % 2, QK_{g+2} as soon as the softmax
//             has loaded S_g into registers.  The issuer of an item's first
//             tile also copies that item's Q scales into TMEM, once every
//             score product of the previous item has completed.
//   warp 10   PV issuer: once the softmax has published P_g, PV_g (with the
//             row sum); an item's first PV (which overwrites O) waits until
//             the previous item's O has been read out.  Each tcgen05
//             instruction costs its issuing thread on the order of a hundred
//             cycles while the softmax warps load the scheduler it shares,
//             hence three issuing threads on three schedulers.
//   warps 0-7 softmax + correction + epilogue.  Warp w owns TMEM lanes
//             32(w%4)..32(w%4)+31 (query rows) for the KV tiles of stream
//             parity w/4: thread = one query row, all 128 keys of its tiles.
//             The two warps on a scheduler thus alternate tiles, so one's
//             exponentials overlap the other's loads, maxima and stores; the
//             only exchange is the row's reference max, handed from the
//             owner of tile g to the owner of tile g+1 through shared memory
//             (also across items, where the value is not used, to keep the
//             hand-overs strictly alternating).  The owner of an item's last
//             tile reads O and l out of TMEM, frees them for the next item,
//             and writes O (bf16) and LSE while the other warps go on.
// Tensor memory (512 columns): S0 [0,128) S1 [128,256) O [256,384) and the
// row sum l at 384 (columns [384,400) all hold l), P0 [416,448) P1 [448,480),
// block scales: Q [400,408), K slot 0 [408,416), rank-one terms
// [480,480+8T), K slot 1 [496,504).  P has its own columns so the scores
// of tile g+2 can be computed into bank g % 2 as soon as the softmax has read
// tile g, while PV_g still reads P_g.
#include <cmath>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "device.cuh"
#include "internal.h"

namespace mpfa {

bool make_map_2d_u8(CUtensorMap* m, const void* base, uint64_t inner_bytes, uint64_t rows,
                    uint32_t box_rows, CUtensorMapSwizzle sw);
bool make_map_2d_u8_box(CUtensorMap* m, const void* base, uint64_t inner_bytes, uint64_t pitch,
                        uint64_t rows, uint32_t box_inner, uint32_t box_rows,
                        CUtensorMapSwizzle sw);

namespace {

constexpr int kKStages = 4;   // K tiles: released once the softmax has loaded S
constexpr int kVStages = 3;   // V tiles: released once PV has read them
constexpr int kThreads = 384;
// QK issuers: warp 9 for the even tiles of the stream (score bank 0, scale
// slot 0), warp 11 for the odd ones (bank 1, slot 1)
constexpr int kWarpTma = 8, kWarpMma = 9, kWarpPv = 10, kWarpMma2 = 11;
constexpr int kSoftmaxThreads = 256;
constexpr int kTileThreads = 128;   // softmax threads that own one KV tile
constexpr int kTmemCols = 512;

constexpr uint32_t kColS0 = 0, kColO = 256, kColL = 384, kColP0 = 416, kColSfQ = 400,
                   kColSfQb = 480;
// K block-scale slot i of QK issuer i (8 columns each, 4-aligned as the MMA
// requires)
__device__ __forceinline__ uint32_t col_sf_k(int i) { return i == 0 ? 408u : 496u; }

// Full-FP4 PV ablation (the kPv4 kernel): P codes in shared memory (two
// banks of 128 rows x 64 bytes, 64-byte swizzle, over the ones atom's region),
// P block scales in V stage 0's unused tail, the all-ones operand of the row
// sum (16 rows of E2M1 1.0 and their E4M3 1.0 scales) in V stage 1's tail
// (a V^T stage uses only its first 9 KB); TMEM: the P scales of bank b at
// 416 + 8b, the V^T scales of slot b at 432 + 8b, the ones' scales at 448
// (the FP8 kernel's P banks).  P = NVFP4 of x = 2^(t - m + 4) with the fixed
// tensor scale fp32(2^8 / 2688): the largest x a tile can produce, 2^(4+tau),
// maps to 6 * 448.
constexpr float kLog2SP4 = -3.3923173959064714f;   // log2(fp32(256 / 2688))
constexpr uint32_t kColSfP4 = 416, kColSfV4 = 432, kColSfOnes4 = 448;

// barrier indices
enum : int {
  kBarQFull0 = 0,                      // +Q buffer: Q tile, scales and rank-one operand in smem
  kBarQEmpty0 = 2,                     // +Q buffer: both QK issuers done with that buffer's item
  kBarQSf = 4,                         // the current item's Q block scales copied into TMEM
  kBarOnes = 5,                        // E4M3 ones beside the V stages written
  kBarOFree = 6,                       // the previous item's O and l read out of TMEM
  kBarDrain = 7,
  kBarSFull0 = 8,                      // +bank: scores of tile g in bank g % 2
  kBarPReady0 = 10,                    // +bank: P_g published in P bank g % 2
  kBarSRead0 = 12,                     // +K stage: S_g (K stage g % 4) loaded by the softmax
  kBarKFull0 = kBarSRead0 + kKStages,  // +K stage
  kBarVFull0 = kBarKFull0 + kKStages,  // +V stage
  kBarODone0 = kBarVFull0 + kVStages,  // +V stage: PV_g (V stage g % 3) completed
  kNumBars = kBarODone0 + kVStages,
};

// shared memory layout (offsets from a 1024-byte aligned base)
constexpr uint32_t kOffQ = 0;                            // 2 Q buffers x 8 KB
constexpr uint32_t kOffQb = kOffQ + 2 * 8192;            // 2 Q buffers x 2 terms x 8 KB
constexpr uint32_t kOffK = kOffQb + 2 * 2 * 8192;        // kKStages x 8 KB
constexpr uint32_t kVStageBytes = 16384;
constexpr uint32_t kOffV = kOffK + kKStages * 8192;      // kVStages x 16 KB
// 16 KB of E4M3 ones: the second 128-byte atom of every V stage's N = 144
// operand (each stage's descriptor reaches it with its own leading offset)
constexpr uint32_t kOffOnes = kOffV + kVStages * kVStageBytes;
// O staging, one 32 KB tile per softmax parity: two 64-column halves of
// 128 rows x 128 bytes in the 128-byte swizzle of the TMA store, each warp
// storing its own 32 rows
constexpr uint32_t kOffOst = kOffOnes + 16384;
constexpr uint32_t kOffQs = kOffOst + 2 * 32768;         // 2 Q buffers x 1 KB
constexpr uint32_t kOffQbs = kOffQs + 2 * 1024;               // 2 Q buffers x 2 terms x 1 KB
constexpr uint32_t kOffKs = kOffQbs + 2 * 2048;               // kKStages x 1 KB
// per row the reference max and the stream index of the tile it follows,
// one 64-bit word (bits 0-31 the fp32 max, 32-63 the tile index)
constexpr uint32_t kOffMax = kOffKs + kKStages * 1024;
// per QK issuer, the last stream tile of an item whose products it has seen
// complete (a counter: the copier of the next item polls it instead of a
// barrier phase that could be two completions behind)
constexpr uint32_t kOffQkDone = kOffMax + 1024;
constexpr uint32_t kOffBar = kOffQkDone + 64;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemUsed = kOffMisc + 64;
// More than half an SM's shared memory, so a single CTA owns the SM and its
// 512 TMEM columns.
constexpr uint32_t kSmemBytes = 224 * 1024;
static_assert(kSmemUsed + 1024 <= kSmemBytes, "shared memory layout overflow");
// every address a tcgen05 descriptor holds fits its 14-bit field (16-byte
// units) even after the 1 KB alignment of the dynamic shared base
static_assert(kOffMax + 2048 <= (1u << 18), "descriptor address field overflow");
constexpr uint32_t kOffP4 = kOffOnes;                          // 2 x 8 KB P codes
constexpr uint32_t kOffP4s = kOffV + 9216;                     // 2 x 1 KB P scales
constexpr uint32_t kOffOnes4 = kOffV + kVStageBytes + 9216;    // 1 KB of E2M1 1.0
constexpr uint32_t kOffOnes4s = kOffOnes4 + 1024;              // 1 KB of E4M3 1.0
static_assert(kOffP4s + 2048 <= kOffV + kVStageBytes && kOffOnes4s + 1024 <= kOffV + 2 * kVStageBytes,
              "FP4 PV operands overflow their V stage tails");

struct Params {
  PrefillArgs a;
  float log2e_rsqrt_d;  // fp32(log2(e) / sqrt(128))
  int q_tiles;
  int items;            // q_tiles * B * Hq work items
};

// One work item: query tile qt of (batch, head) bh, nkv KV tiles.
struct Item {
  int qt, bh, nkv;
};

// Item k of this CTA, or false past the end.  Items are numbered heaviest
// causal query tile first; round k deals items [kG, kG + G) to the G CTAs,
// in reverse on odd rounds, so the per-CTA sums of KV tiles stay within one
// round's spread.
__device__ __forceinline__ bool item_of(const Params& p, int k, Item& it) {
  const int G = (int)gridDim.x, c = (int)blockIdx.x;
  const int i = k * G + ((k & 1) ? G - 1 - c : c);
  if (i >= p.items) return false;
  const int bh_count = p.a.B * p.a.Hq;
  it.qt = p.q_tiles - 1 - i / bh_count;
  it.bh = i % bh_count;
  it.nkv = p.a.causal ? it.qt + 1 : p.q_tiles;
  return true;
}

__device__ __forceinline__ int ld_acquire_s32(const int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_s32(int* p, int v) {
  asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
// Bounded per-thread poll until *p >= want (false on timeout or abort).
__device__ __forceinline__ bool poll_ge(const int* p, int want, int* err, volatile int* abort) {
  if (ld_acquire_s32(p) >= want) return true;
  const unsigned long long t0 = globaltimer();
  for (int it = 0;; ++it) {
    if (ld_acquire_s32(p) >= want) return true;
    if ((it & 63) == 63) {
      if (*abort) return false;
      if (globaltimer() - t0 > kWaitLimitNs) {
        record_error(err, kErrTimeout);
        *abort = 1;
        return false;
      }
    }
  }
}

// Eight E2M1 codes (element 2i in the low nibble of byte i).
__device__ __forceinline__ uint32_t e2m1x8(const float* q) {
  uint32_t r;
  asm("{\n.reg .b8 t0, t1, t2, t3;\n"
      "cvt.rn.satfinite.e2m1x2.f32 t0, %2, %1;\n"
      "cvt.rn.satfinite.e2m1x2.f32 t1, %4, %3;\n"
      "cvt.rn.satfinite.e2m1x2.f32 t2, %6, %5;\n"
      "cvt.rn.satfinite.e2m1x2.f32 t3, %8, %7;\n"
      "mov.b32 %0, {t0, t1, t2, t3};\n}"
      : "=r"(r)
      : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
  return r;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <bool kPv4>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap map_q,
                   const __grid_constant__ CUtensorMap map_k,
                   const __grid_constant__ CUtensorMap map_v,
                   const __grid_constant__ CUtensorMap map_o, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const PrefillArgs& a = p.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g_kv = a.Hq / a.Hkv;
  const int T = a.compensate ? a.T : 0;

  auto bar = [&](int i) { return sbase + kOffBar + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc + 8);

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int b2 = 0; b2 < 2; ++b2) {
      mbar_init(bar(kBarQFull0 + b2), 2);    // TMA arrive.expect_tx + rank-one operand built
      mbar_init(bar(kBarQEmpty0 + b2), 2);   // one commit from each QK issuer
      mbar_init(bar(kBarSFull0 + b2), 1);
      // softmax-side barriers count warps: each warp arrives once, from one
      // lane, after a __syncwarp that orders its lanes' stores before it
      mbar_init(bar(kBarPReady0 + b2), kTileThreads / 32);
    }
    mbar_init(bar(kBarQSf), 1);
    mbar_init(bar(kBarOnes), kSoftmaxThreads);
    mbar_init(bar(kBarOFree), kTileThreads / 32);
    mbar_init(bar(kBarDrain), 3);   // one commit from each issuing thread
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(bar(kBarSRead0 + s), kTileThreads / 32);
      mbar_init(bar(kBarKFull0 + s), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(bar(kBarVFull0 + s), 1);
      mbar_init(bar(kBarODone0 + s), 1);
    }
    fence_barrier_init();
  }
  if (warp == kWarpMma) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  if (threadIdx.x < 128)   // no tile index yet
    reinterpret_cast<volatile unsigned long long*>(smem + kOffMax)[threadIdx.x] = ~0ull;
  int* qk_done = reinterpret_cast<int*>(smem + kOffQkDone);
  if (threadIdx.x < 2) qk_done[threadIdx.x] = -1;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the codes and tensor scales come from the quantization kernels before
  pdl_wait();
  pdl_trigger();

  if (warp == kWarpTma) {
    // ---------------- TMA producer (whole warp) ----------------
    // every lane polls the same barriers (so the warp stays converged), lane
    // 0 issues the copies, all lanes build the rank-one operand tile
    auto wait_all = [&](int b2, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar(b2), parity, a.err, abort_flag));
    };
    if (lane == 0) {
      prefetch_tensormap(&map_q);
      prefetch_tensormap(&map_k);
      prefetch_tensormap(&map_v);
      prefetch_tensormap(&map_o);
    }
    const int nblk = a.N / 128;
    // Q tile, its scales and the rank-one operand of item k into buffer k % 2
    auto load_q = [&](int k, const Item& it) -> bool {
      const int buf = k & 1;
      // the buffer held item k-2: both QK issuers are done with it
      if (k >= 2 && !wait_all(kBarQEmpty0 + buf, ((k - 2) >> 1) & 1)) return false;
      const size_t qrow = (size_t)it.bh * a.N + (size_t)it.qt * 128;
      if (lane == 0) {
        mbar_expect_tx(bar(kBarQFull0 + buf), 8192 + 1024);
        tma_load_2d(sbase + kOffQ + 8192 * buf, &map_q, 0, (int)qrow, bar(kBarQFull0 + buf));
        bulk_load(sbase + kOffQs + 1024 * buf, a.qs + qrow * 8, 1024, bar(kBarQFull0 + buf));
        // L2 prefetch of the next item's query-side inputs: its Q tile is
        // otherwise a DRAM miss when its turn comes
        Item nx;
        if (item_of(p, k + 1, nx)) {
          const size_t qrow2 = (size_t)nx.bh * a.N + (size_t)nx.qt * 128;
          prefetch_l2_bulk(a.qc + qrow2 * 64, 8192);
          prefetch_l2_bulk(a.qs + qrow2 * 8, 1024);
          if (T > 0) {
            const size_t qb2 = ((size_t)nx.bh * nblk + nx.qt) * a.T;
            prefetch_l2_bulk(a.qbc + qb2 * 64, 64u * a.T);
            prefetch_l2_line(a.qbs + qb2 * 8);
          }
        }
      }
      // rank-one operand: every row holds the block's term t (same 64
      // bytes), written with the 64-byte swizzle the TMA applies to Q and K;
      // its block scales likewise, one 8-byte row per query row
      for (int t = 0; t < T; ++t) {
        const size_t qb = ((size_t)it.bh * nblk + it.qt) * a.T + t;
        const uint4* src = reinterpret_cast<const uint4*>(a.qbc + qb * 64);
        const uint4 v0 = src[0], v1 = src[1], v2 = src[2], v3 = src[3];
        const uint32_t w0 = *reinterpret_cast<const uint32_t*>(a.qbs + qb * 8);
        const uint32_t w1 = *reinterpret_cast<const uint32_t*>(a.qbs + qb * 8 + 4);
        uint8_t* qbt = smem + kOffQb + 16384 * buf + 8192 * t;
        uint32_t* qbst = reinterpret_cast<uint32_t*>(smem + kOffQbs + 2048 * buf + 1024 * t);
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
          const int r = lane + 32 * rr, sw = (r >> 1) & 3;
          uint4* dst = reinterpret_cast<uint4*>(qbt + 64 * r);
          dst[0 ^ sw] = v0;
          dst[1 ^ sw] = v1;
          dst[2 ^ sw] = v2;
          dst[3 ^ sw] = v3;
          qbst[r] = w0;
          qbst[128 + r] = w1;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarQFull0 + buf));
      return true;
    };
    // K and V cursors over this CTA's items: tile g of the stream is tile
    // g - g0 of the cursor's item, whose K/V rows start at row0
    struct Cur {
      int k, g0, n, row0;
    };
    auto enter = [&](Cur& c, int k) -> bool {
      Item it;
      if (!item_of(p, k, it)) return false;
      const int b = it.bh / a.Hq, hk = (it.bh % a.Hq) / g_kv;
      c.k = k;
      c.n = it.nkv;
      c.row0 = (b * a.Hkv + hk) * a.N;
      return true;
    };
    Cur ck{0, 0, 0, 0}, cv{0, 0, 0, 0};
    int k_issued = 0, v_issued = 0, q_issued = 0;
    bool lok = enter(ck, 0) && enter(cv, 0);
    {
      Item it0;
      lok = lok && item_of(p, 0, it0) && load_q(0, it0);
    }
    if (lok) q_issued = 1;
    // lane 0's test of a phase, the same answer in every lane
    auto test_all = [&](int b2, uint32_t parity) -> bool {
      return __shfl_sync(0xffffffffu, mbar_test_wait(bar(b2), parity) ? 1 : 0, 0) != 0;
    };
    auto issue_k = [&](int g) {
      const int s = g % kKStages;
      if (lane == 0) {
        const int row = ck.row0 + (g - ck.g0) * 128;
        mbar_expect_tx(bar(kBarKFull0 + s), 8192 + 1024);
        tma_load_2d(sbase + kOffK + s * 8192, &map_k, 0, row, bar(kBarKFull0 + s));
        bulk_load(sbase + kOffKs + s * 1024, a.ks + (size_t)row * 8, 1024, bar(kBarKFull0 + s));
      }
      k_issued = g + 1;
    };
    auto issue_v = [&](int g) {
      const int s = g % kVStages;
      if (lane == 0) {
        if constexpr (kPv4) {
          // V^T tile: 128 channel rows x 128 keys (64 bytes) and its 1 KB
          // of block scales
          const int bhk = cv.row0 / a.N, t = g - cv.g0;
          mbar_expect_tx(bar(kBarVFull0 + s), 8192 + 1024);
          tma_load_2d(sbase + kOffV + s * kVStageBytes, &map_v, 64 * t, bhk * 128,
                      bar(kBarVFull0 + s));
          bulk_load(sbase + kOffV + s * kVStageBytes + 8192,
                    a.vts + ((size_t)bhk * (a.N / 128) + t) * 1024, 1024, bar(kBarVFull0 + s));
        } else {
          mbar_expect_tx(bar(kBarVFull0 + s), 16384);
          tma_load_2d(sbase + kOffV + s * kVStageBytes, &map_v, 0, cv.row0 + (g - cv.g0) * 128,
                      bar(kBarVFull0 + s));
        }
      }
      v_issued = g + 1;
    };
    // total tiles of this CTA's stream
    int gtot = 0;
    {
      Item it;
      for (int k = 0; item_of(p, k, it); ++k) gtot += it.nkv;
    }
    // K and V tiles are loaded as soon as their own stages free up, polled
    // without blocking, so neither ring waits behind the other: K stage
    // g % 4 held K_{g-4} (free once the softmax has loaded S_{g-4}), V stage
    // g % 3 held V_{g-3} (free once PV_{g-3} has completed); an item's Q
    // goes into its buffer before the item's first K tile, once both QK
    // issuers are done with the item two back.  Idle polls sleep briefly;
    // the polling gives up (timeout) when nothing has moved for the wait
    // limit.
    int gk = 0, gv = 0;
    unsigned long long idle_since = 0;
    unsigned spins = 0;
    while (lok && (gk < gtot || gv < gtot)) {
      bool did = false;
      if (gk < gtot) {
        if (gk >= ck.g0 + ck.n) {
          // the K cursor enters the next item: its Q first
          const int kn = ck.k + 1;
          if (kn < 2 || test_all(kBarQEmpty0 + (kn & 1), ((kn - 2) >> 1) & 1)) {
            const int g0n = ck.g0 + ck.n;
            Item it;
            if (!enter(ck, kn) || !item_of(p, kn, it)) {
              lok = false;
              break;
            }
            ck.g0 = g0n;
            if (!load_q(kn, it)) {
              lok = false;
              break;
            }
            q_issued = kn + 1;
            did = true;
          }
        } else if (gk < kKStages ||
                   test_all(kBarSRead0 + gk % kKStages, ((gk / kKStages) - 1) & 1)) {
          issue_k(gk);
          ++gk;
          did = true;
        }
      }
      if (gv < gtot) {
        if (gv >= cv.g0 + cv.n) {
          const int g0n = cv.g0 + cv.n;
          if (!enter(cv, cv.k + 1)) {
            lok = false;
            break;
          }
          cv.g0 = g0n;
        }
        if (gv < kVStages || test_all(kBarODone0 + gv % kVStages, ((gv / kVStages) - 1) & 1)) {
          issue_v(gv);
          ++gv;
          did = true;
        }
      }
      if (did) {
        idle_since = 0;
        continue;
      }
      if (*abort_flag) break;
      if (idle_since == 0) {
        idle_since = globaltimer();
      } else if ((++spins & 63u) == 0 && globaltimer() - idle_since > kWaitLimitNs) {
        if (lane == 0) {
          record_error(a.err, kErrTimeout);
          *abort_flag = 1;
        }
        break;
      }
      __nanosleep(40);
    }
    // drain: every buffer's last load must have landed before the CTA exits
    if (lane == 0) {
      for (int g = k_issued - kKStages > 0 ? k_issued - kKStages : 0; g < k_issued; ++g)
        mbar_wait(bar(kBarKFull0 + g % kKStages), (g / kKStages) & 1, a.err, nullptr);
      for (int g = v_issued - kVStages > 0 ? v_issued - kVStages : 0; g < v_issued; ++g)
        mbar_wait(bar(kBarVFull0 + g % kVStages), (g / kVStages) & 1, a.err, nullptr);
      for (int k = q_issued - 2 > 0 ? q_issued - 2 : 0; k < q_issued; ++k)
        mbar_wait(bar(kBarQFull0 + (k & 1)), (k >> 1) & 1, a.err, nullptr);
    }
  } else if (warp == kWarpMma || warp == kWarpMma2) {
    // ---------------- QK issuers (whole warps, converged) ----------------
    // One warp per score bank, each issuing every other tile of the stream
    // with its own K scale slot: each accumulator and slot has a single
    // issuing warp, and neither warp's tiles wait behind the other's.  Every
    // lane computes the warp-uniform operands; one lane, elected inside each
    // tcgen05 instruction block, issues it.
    {
      const uint32_t tmem_w = __shfl_sync(0xffffffffu, tmem, 0);
      auto mbar_wait_w = [&](uint32_t b, uint32_t parity, volatile int* ab) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(b, parity, a.err, ab));
      };
      const int par = warp == kWarpMma ? 0 : 1;
      const uint32_t id_qk = idesc_nvfp4(128, 128);
      // shared-memory descriptors built once: the start address sits in the
      // low field in 16-byte units, so a K stage, a Q buffer or a rank-one
      // term (8 KB) is +512 and the second 64-element K chunk (32 B) +2;
      // every address stays below 2^18, inside that field
      const uint64_t dq0 = smem_desc(sbase + kOffQ, 16, 512, kSwizzle64B);
      const uint64_t dk0 = smem_desc(sbase + kOffK, 16, 512, kSwizzle64B);
      const uint64_t dqb0 = smem_desc(sbase + kOffQb, 16, 512, kSwizzle64B);
      // QK_g (and the rank-one MMAs) into score bank g % 2, Q from buffer buf
      auto issue_qk = [&](int g, int buf) -> bool {
        const int s = g % kKStages, bk = g & 1;
        if (!mbar_wait_w(bar(kBarKFull0 + s), (g / kKStages) & 1, abort_flag)) return false;
        tc_fence_after();
        // K_g's scales into this issuer's slot; its last reader, QK_{g-2},
        // completed before the softmax loaded S_{g-2} (waited for)
        const uint32_t sfk = tmem_w + col_sf_k(bk);
        for (int kc = 0; kc < 2; ++kc)
          tmem_cp_32x128b_x4_w(sfk + 4 * kc,
                             smem_desc(sbase + kOffKs + 1024 * s + 512 * kc, 128, 128, kSwizzleNone));
        const uint32_t dS = tmem_w + kColS0 + 128 * bk;
        const uint64_t dk = dk0 + 512u * (uint32_t)s;
        const uint64_t dq = dq0 + 512u * (uint32_t)buf, dqb = dqb0 + 1024u * (uint32_t)buf;
        mma_nvfp4_ss_w(dS, dq, dk, id_qk, tmem_w + kColSfQ, sfk, 0u);
        mma_nvfp4_ss_w(dS, dq + 2u, dk + 2u, id_qk, tmem_w + kColSfQ + 4, sfk + 4, 1u);
        if (T > 0) {
          mma_nvfp4_ss_w(dS, dqb, dk, id_qk, tmem_w + kColSfQb, sfk, 1u);
          mma_nvfp4_ss_w(dS, dqb + 2u, dk + 2u, id_qk, tmem_w + kColSfQb + 4, sfk + 4, 1u);
        }
        if (T > 1) {
          mma_nvfp4_ss_w(dS, dqb + 512u, dk, id_qk, tmem_w + kColSfQb + 8, sfk, 1u);
          mma_nvfp4_ss_w(dS, dqb + 514u, dk + 2u, id_qk, tmem_w + kColSfQb + 12, sfk + 4, 1u);
        }
        tc_commit_w(bar(kBarSFull0 + bk));
        return true;
      };
      // the softmax has loaded S_{g-2}: bank g % 2 and slot g % 2 are free.
      // SRead for stage (g-2) % 4 cannot be a phase further on: that needs
      // S_{g+2}.
      auto wait_sread = [&](int g) -> bool {
        return g < 2 || mbar_wait_w(bar(kBarSRead0 + (g - 2) % kKStages),
                                  ((g - 2) / kKStages) & 1, abort_flag);
      };
      bool ok = true;
      int g0 = 0;
      Item it;
      for (int k = 0; ok && item_of(p, k, it); ++k) {
        const int buf = k & 1, n = it.nkv;
        const bool copier = (g0 & 1) == par;   // this thread issues the item's first tile
        if (copier) {
          // the item's Q is in buffer buf, and every score product reading
          // the TMEM Q scales of the previous item has completed: the other
          // thread's QK_{g0-1} (its bank's next commit needs these scales;
          // the other thread says so through its counter) and this thread's
          // QK_{g0-2} (waited for through S_{g0-2})
          ok = mbar_wait_w(bar(kBarQFull0 + buf), (k >> 1) & 1, abort_flag) &&
               (g0 < 1 ||
                __all_sync(0xffffffffu, poll_ge(qk_done + (par ^ 1), g0 - 1, a.err, abort_flag))) &&
               wait_sread(g0);
          if (!ok) break;
          tc_fence_after();
          for (int kc = 0; kc < 2; ++kc)
            tmem_cp_32x128b_x4_w(tmem_w + kColSfQ + 4 * kc,
                               smem_desc(sbase + kOffQs + 1024 * buf + 512 * kc, 128, 128,
                                         kSwizzleNone));
          for (int t = 0; t < T; ++t)
            for (int kc = 0; kc < 2; ++kc)
              tmem_cp_32x128b_x4_w(tmem_w + kColSfQb + 8 * t + 4 * kc,
                                 smem_desc(sbase + kOffQbs + 2048 * buf + 1024 * t + 512 * kc,
                                           128, 128, kSwizzleNone));
          // also says (to the other thread) that Q and the rank-one operand
          // are in shared memory
          tc_commit_w(bar(kBarQSf));
          ok = issue_qk(g0, buf);
        } else if (n > 1) {
          ok = mbar_wait_w(bar(kBarQSf), k & 1, abort_flag);
          if (ok) tc_fence_after();
        }
        for (int g = g0 + (copier ? 2 : 1); ok && g < g0 + n; g += 2) {
          if (!wait_sread(g) || !issue_qk(g, buf)) ok = false;
        }
        // the last tile this thread issued in the item: once its products
        // have landed, say so to the other thread.  Its own latest phase
        // cannot be two behind: that tile was issued after S of its tile
        // two back had been read.
        const int last = ((g0 + n - 1) & 1) == par ? g0 + n - 1 : g0 + n - 2;
        if (ok && last >= g0) {
          ok = mbar_wait_w(bar(kBarSFull0 + par), (last >> 1) & 1, abort_flag);
          if (ok && lane == 0) st_release_s32(qk_done + par, last);
          __syncwarp();
        }
        // this thread's products of item k done with Q buffer buf
        tc_commit_w(bar(kBarQEmpty0 + buf));
        g0 += n;
      }
      // drain this thread's tensor-core work before the CTA releases TMEM
      tc_commit_w(bar(kBarDrain));
      mbar_wait_w(bar(kBarDrain), 0, nullptr);
    }
  } else if (warp == kWarpPv) {
    // ---------------- PV issuer (whole warp, converged) ----------------
    {
      const uint32_t tmem_w = __shfl_sync(0xffffffffu, tmem, 0);
      auto mbar_wait_w = [&](uint32_t b, uint32_t parity, volatile int* ab) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(b, parity, a.err, ab));
      };
      const uint32_t id_pv = idesc_fp8(128, 144, 0, 1);   // 128 V columns + 16 ones
      const uint32_t id_pv4 = idesc_nvfp4(128, 128), id_l4 = idesc_nvfp4(128, 16);
      bool ok = mbar_wait_w(bar(kBarOnes), 0, abort_flag);
      if constexpr (kPv4) {
        // the ones operand's block scales (all E4M3 1.0), copied once
        if (ok) {
          tc_fence_after();
          for (int kc = 0; kc < 2; ++kc)
            tmem_cp_32x128b_x4_w(tmem_w + kColSfOnes4 + 4 * kc,
                                 smem_desc(sbase + kOffOnes4s + 512 * kc, 128, 128, kSwizzleNone));
        }
      }
      int g0 = 0;
      Item it;
      for (int k = 0; ok && item_of(p, k, it); ++k) {
        // the item's first PV overwrites O and l: the previous item's
        // epilogue must have read them out
        if (k >= 1 && !mbar_wait_w(bar(kBarOFree), (k - 1) & 1, abort_flag)) break;
        for (int j = 0; j < it.nkv; ++j) {
          const int g = g0 + j, bp = g & 1, sp = g % kVStages;
          // the softmax has published P_g in P bank g % 2
          if (!mbar_wait_w(bar(kBarPReady0 + bp), (g >> 1) & 1, abort_flag) ||
              !mbar_wait_w(bar(kBarVFull0 + sp), (g / kVStages) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t voff = kOffV + sp * kVStageBytes;
          if constexpr (kPv4) {
            // P_g's and V_g^T's block scales into TMEM (their slots' last
            // reader, PV_{g-2}, completed before the softmax published P_g);
            // then O += P V^T and l += P 1 in block-scaled FP4, K = 64 keys
            // per product
            const uint32_t sfa = tmem_w + kColSfP4 + 8 * bp, sfb = tmem_w + kColSfV4 + 8 * bp;
            for (int kc = 0; kc < 2; ++kc) {
              tmem_cp_32x128b_x4_w(sfa + 4 * kc, smem_desc(sbase + kOffP4s + 1024 * bp + 512 * kc,
                                                           128, 128, kSwizzleNone));
              tmem_cp_32x128b_x4_w(sfb + 4 * kc, smem_desc(sbase + voff + 8192 + 512 * kc, 128, 128,
                                                           kSwizzleNone));
            }
            const uint64_t da = smem_desc(sbase + kOffP4 + 8192 * bp, 16, 512, kSwizzle64B);
            const uint64_t db = smem_desc(sbase + voff, 16, 512, kSwizzle64B);
            const uint64_t d1 = smem_desc(sbase + kOffOnes4, 16, 512, kSwizzle64B);
            mma_nvfp4_ss_w(tmem_w + kColO, da, db, id_pv4, sfa, sfb, j > 0 ? 1u : 0u);
            mma_nvfp4_ss_w(tmem_w + kColO, da + 2u, db + 2u, id_pv4, sfa + 4, sfb + 4, 1u);
            mma_nvfp4_ss_w(tmem_w + kColL, da, d1, id_l4, sfa, tmem_w + kColSfOnes4,
                           j > 0 ? 1u : 0u);
            mma_nvfp4_ss_w(tmem_w + kColL, da + 2u, d1 + 2u, id_l4, sfa + 4,
                           tmem_w + kColSfOnes4 + 4, 1u);
          } else {
            const uint32_t pcol = tmem_w + kColP0 + 32 * bp;
            // the N = 144 operand: V's 128-byte atom, then the ones atom at a
            // leading offset of kOffOnes - voff bytes (the same 32-key
            // sub-tile offset in both)
            for (int kk = 0; kk < 4; ++kk)
              mma_fp8_ts_w(tmem_w + kColO, pcol + 8 * kk,
                           smem_desc(sbase + voff + 4096 * kk, kOffOnes - voff, 1024, kSwizzle128B),
                           id_pv, (j > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit_w(bar(kBarODone0 + sp));
        }
        g0 += it.nkv;
      }
      tc_commit_w(bar(kBarDrain));
      mbar_wait_w(bar(kBarDrain), 0, nullptr);
    }
  } else {
    // ---------------- softmax / correction / epilogue ----------------
    const int par = warp >> 2, quad = warp & 3;   // tile parity, TMEM lane quadrant
    const int row = threadIdx.x & 127;            // query row = TMEM lane
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    // the ones atom of the PV operand (E4M3 1.0 = 0x38; every byte equal,
    // so the 128-byte swizzle leaves it unchanged), written once
    if constexpr (kPv4) {
      // the row sum's operand: 16 rows of E2M1 1.0 (code 2) and their E4M3
      // 1.0 block scales (every byte equal, so any layout reads the same)
      uint4* ones = reinterpret_cast<uint4*>(smem + kOffOnes4);
      uint4* ones_s = reinterpret_cast<uint4*>(smem + kOffOnes4s);
      for (int i = threadIdx.x; i < 1024 / 16; i += kSoftmaxThreads) {
        ones[i] = make_uint4(0x22222222u, 0x22222222u, 0x22222222u, 0x22222222u);
        ones_s[i] = make_uint4(0x38383838u, 0x38383838u, 0x38383838u, 0x38383838u);
      }
    } else {
      uint4* ones = reinterpret_cast<uint4*>(smem + kOffOnes);
      for (int i = threadIdx.x; i < 16384 / 16; i += kSoftmaxThreads)
        ones[i] = make_uint4(0x38383838u, 0x38383838u, 0x38383838u, 0x38383838u);
    }
    fence_proxy_async_smem();
    mbar_arrive(bar(kBarOnes));

    int gtot = 0;
    {
      Item it;
      for (int k = 0; item_of(p, k, it); ++k) gtot += it.nkv;
    }
    // Tiles g = par, par + 2, ... of the stream; the owner of tile g hands
    // the row's reference max to the owner of tile g+1 through the row's
    // shared slot, tagged with g (the receiver polls for the tag; a slot
    // cannot be overwritten before it is read, since the next value needs
    // the reply).  No barrier: the value is the only thing passed, so
    // relaxed 64-bit accesses suffice.  At an item's first tile the value
    // handed over is ignored.
    volatile unsigned long long* mslot =
        reinterpret_cast<volatile unsigned long long*>(smem + kOffMax) + row;
    const float cs = __fmul_rn(__fmul_rn(*a.s_q, *a.s_k), p.log2e_rsqrt_d);
    bool ok = true;
    int g0 = 0;
    Item it;
    for (int k = 0; ok && item_of(p, k, it); ++k) {
      const int nkv = it.nkv, qt = it.qt;
      float m = -INFINITY;
      for (int j = (g0 & 1) == par ? 0 : 1; j < nkv; j += 2) {
        const int g = g0 + j, bk = par;   // bk == g & 1
        if (!__all_sync(0xffffffffu,
                        mbar_wait(bar(kBarSFull0 + bk), (g >> 1) & 1, a.err, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sS = tmem + lane_off + kColS0 + 128 * bk;
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(sS + 32 * c, sr[c]);
        tmem_ld_wait();
        // S_g is in registers: bank g % 2 and K stage g % 4 may be reused
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarSRead0 + g % kKStages));
        if (a.causal && j == qt) {  // diagonal tile: key > row is masked
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (32 * c + i > row) sr[c][i] = 0xFF800000u;  // -inf
        }
        // the partner's value, read before the max tree so the load's latency
        // is hidden (polled again below if it was not there yet)
        const unsigned long long v_early = *mslot;
        // tile max over the row's 128 keys (3-input max tree)
        float pm[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const int e = 8 * q;
          pm[q] = fmax3(fmax3(__uint_as_float(sr[e >> 5][e & 31]),
                              __uint_as_float(sr[e >> 5][(e + 1) & 31]),
                              __uint_as_float(sr[e >> 5][(e + 2) & 31])),
                        fmax3(__uint_as_float(sr[e >> 5][(e + 3) & 31]),
                              __uint_as_float(sr[e >> 5][(e + 4) & 31]),
                              __uint_as_float(sr[e >> 5][(e + 5) & 31])),
                        fmaxf(__uint_as_float(sr[e >> 5][(e + 6) & 31]),
                              __uint_as_float(sr[e >> 5][(e + 7) & 31])));
        }
        // (FP4 P keeps the eight 16-key block maxima for its block scales)
        float bmx[8];
        float smax;
        if constexpr (kPv4) {
#pragma unroll
          for (int kb = 0; kb < 8; ++kb) bmx[kb] = fmaxf(pm[2 * kb], pm[2 * kb + 1]);
          smax = fmax3(fmax3(bmx[0], bmx[1], bmx[2]), fmax3(bmx[3], bmx[4], bmx[5]),
                       fmaxf(bmx[6], bmx[7]));
        } else {
          smax = fmax3(fmax3(fmax3(pm[0], pm[1], pm[2]), fmax3(pm[3], pm[4], pm[5]),
                             fmax3(pm[6], pm[7], pm[8])),
                       fmax3(pm[9], pm[10], pm[11]),
                       fmax3(fmax3(pm[12], pm[13], pm[14]), pm[15], -INFINITY));
        }
        // reference max of the row after tile g-1, from that tile's owner
        if (g > 0) {
          // the row's slot holds tile g-1's value once its index reads g-1
          // (one aligned 64-bit word: value and index arrive together)
          unsigned long long v = v_early;
          bool got = (uint32_t)(v >> 32) == (uint32_t)(g - 1);
          if (!__all_sync(0xffffffffu, got)) {
            const unsigned long long t0 = globaltimer();
            for (int it = 0; !got; ++it) {
              v = *mslot;
              got = (uint32_t)(v >> 32) == (uint32_t)(g - 1);
              if (!got && (it & 63) == 63) {
                if (*abort_flag) break;
                if (globaltimer() - t0 > kWaitLimitNs) {
                  record_error(a.err, kErrTimeout);
                  *abort_flag = 1;
                  break;
                }
              }
            }
            if (!__all_sync(0xffffffffu, got)) {
              ok = false;
              break;
            }
          }
          const float mi = __uint_as_float((uint32_t)v);
          if (j > 0) m = mi;
        }
        // cs > 0, so max_i(S_i * cs) == (max_i S_i) * cs exactly.  The
        // reference max moves only when the tile max exceeds it by more than
        // kRescaleTau, so O and L rarely need a rescale once the first tiles
        // are done.
        const float tmax = __fmul_rn(smax, cs);
        const float mn = (m == -INFINITY || tmax > m + kRescaleTau) ? tmax : m;
        if (g + 1 < gtot)
          *mslot = ((unsigned long long)(uint32_t)g << 32) | __float_as_uint(mn);
        const float alpha = (m == -INFINITY) ? 0.0f : (mn == m ? 1.0f : ex2(m - mn));
        const float bias = kPShift - mn;  // P8 = E4M3(2^(t - m) * 2^kPShift)
        const float2 cs2 = make_float2(cs, cs), bias2 = make_float2(bias, bias);
        uint32_t pw[kPv4 ? 18 : 32];
        if constexpr (!kPv4) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int w = 0; w < 8; ++w) {
              // two scores per packed fp32 FMA
              const float2 t0 = __ffma2_rn(
                  make_float2(__uint_as_float(sr[c][4 * w]), __uint_as_float(sr[c][4 * w + 1])),
                  cs2, bias2);
              const float2 t1 = __ffma2_rn(
                  make_float2(__uint_as_float(sr[c][4 * w + 2]), __uint_as_float(sr[c][4 * w + 3])),
                  cs2, bias2);
              pw[8 * c + w] = e4m3x4(ex2(t0.x), ex2(t0.y), ex2(t1.x), ex2(t1.y));
            }
        } else {
          // x = 2^(t - m + 4) in NVFP4 per 16 keys with the fixed tensor
          // scale s_p = fp32(2^8 / 2688): block scale sb = E4M3(max x /
          // (6 s_p)), 1 / (6 s_p) = 1.75, with max x = x at the block's
          // largest score (x grows with the score; the block maxima come
          // from the tile's max tree); code = E2M1(x / (value(sb) s_p)), the
          // quotient taken in the exponent, 2^(t - m + 4 - log2(value(sb)
          // s_p)), so a key costs what it costs the FP8 path: half a packed
          // FMA, one exponential, half an E2M1 pair conversion.
          // pw[0..15]: 8 codes per word in key order; pw[16..17]: the block
          // scales of keys 0-63 and 64-127, four per word
          pw[16] = pw[17] = 0u;
#pragma unroll
          for (int kb = 0; kb < 8; ++kb) {
            const uint32_t sb =
                e4m3_pos(__fmul_rn(ex2(__fmaf_rn(bmx[kb], cs, bias)), 1.75f));
            // a block with no code above zero gets the exponent -inf (code 0)
            const float qb = sb != 0u ? bias - (lg2(e4m3_value(sb)) + kLog2SP4) : -INFINITY;
            const float2 qb2 = make_float2(qb, qb);
            float q[16];
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
              const uint32_t* sv = &sr[kb >> 1][16 * (kb & 1) + i];
              const float2 t2 = __ffma2_rn(
                  make_float2(__uint_as_float(sv[0]), __uint_as_float(sv[1])), cs2, qb2);
              q[i] = ex2(t2.x);
              q[i + 1] = ex2(t2.y);
            }
            pw[2 * kb] = e2m1x8(q);
            pw[2 * kb + 1] = e2m1x8(q + 8);
            pw[16 + (kb >> 2)] |= sb << (8 * (kb & 3));
          }
        }
        // correction: O and L scale by alpha once PV_{g-1} has landed (PV_g is
        // issued only after this tile's P is published)
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
          if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarODone0 + (g - 1) % kVStages),
                                                 ((g - 1) / kVStages) & 1, a.err, abort_flag))) {
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
        // P bank g % 2 was last read by PV_{g-2}: wait for it to complete
        // (its ODone phase cannot be overtaken: PV_{g+1} needs this P first).
        if (g >= 2 && !__all_sync(0xffffffffu, mbar_wait(bar(kBarODone0 + (g - 2) % kVStages),
                                                          ((g - 2) / kVStages) & 1, a.err,
                                                          abort_flag))) {
          ok = false;
          break;
        }
        if constexpr (kPv4) {
          // the row's 64 code bytes into P bank g % 2 in the 64-byte swizzle
          // of the MMA operand, its block-scale words in the scale-copy order
          uint8_t* prow = smem + kOffP4 + 8192 * bk + 64 * row;
          const int swz = (row >> 1) & 3;
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4)
            *reinterpret_cast<uint4*>(prow + 16 * (c4 ^ swz)) =
                make_uint4(pw[4 * c4], pw[4 * c4 + 1], pw[4 * c4 + 2], pw[4 * c4 + 3]);
#pragma unroll
          for (int kc = 0; kc < 2; ++kc)
            *reinterpret_cast<uint32_t*>(smem + kOffP4s + 1024 * bk + 512 * kc + (row & 31) * 16 +
                                         ((row >> 5) & 3) * 4) = pw[16 + kc];
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kBarPReady0 + bk));
        } else {
          tc_fence_after();
          tmem_st32(tmem + lane_off + kColP0 + 32 * bk, pw);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kBarPReady0 + bk));
        }
        m = mn;
      }
      if (!ok) break;
      if (((g0 + nkv - 1) & 1) == par) {
        const int g = g0 + nkv - 1;
        // epilogue of the item, by the owner of its last tile: once PV_g
        // has completed, O and l into registers, TMEM freed for the next
        // item's first PV, then the normalised O and the LSE out.  ODone
        // for stage g % 3 cannot move on before this: PV_{g+3} needs the
        // O freed here first.
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarODone0 + g % kVStages),
                                               (g / kVStages) & 1, a.err, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t l4[4], o[4][32];
        tmem_ld4(tmem + lane_off + kColL, l4);
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_off + kColO + 32 * c, o[c]);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarOFree));
        const float l = __uint_as_float(l4[0]);
        const float sc = __fdiv_rn(*a.s_v, l);
        const int h = it.bh % a.Hq, b = it.bh / a.Hq;
        const size_t grow = (size_t)qt * 128 + row;
        // O through this warp's 32 rows of its parity's staging tile and two
        // TMA stores issued by the warp's lane 0, whose previous stores must
        // have read those rows before they are rewritten
        const uint32_t ost = kOffOst + 32768u * (uint32_t)par + 4096u * (uint32_t)quad;
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              __nv_bfloat162 v =
                  __floats2bfloat162_rn(__uint_as_float(o[c][8 * q4 + 2 * e]) * sc,
                                        __uint_as_float(o[c][8 * q4 + 2 * e + 1]) * sc);
              w[e] = *reinterpret_cast<uint32_t*>(&v);
            }
            // columns 32c + 8q4 .. +7: half c / 2, 16-byte chunk 4(c % 2) + q4
            // of the row, at chunk position chunk ^ (row % 8)
            const int chunk = 4 * (c & 1) + q4;
            *reinterpret_cast<uint4*>(smem + ost + 16384u * (uint32_t)(c >> 1) + 128u * lane +
                                      16u * (uint32_t)(chunk ^ (lane & 7))) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          // O viewed as bytes [B*N rows][Hq*256]: head h at byte 256h
          const int y = b * a.N + qt * 128 + 32 * quad;
          tma_store_2d(&map_o, sbase + ost, 256 * h, y);
          tma_store_2d(&map_o, sbase + ost + 16384u, 256 * h + 128, y);
          bulk_commit_group();
        }
        if (a.lse) {
          // natural-log LSE of the scaled logits; with key-side smoothing
          // plus the row's dropped logit part q_eff . kbar / sqrt(d)
          const size_t li = (size_t)it.bh * a.N + grow;
          // (with FP4 P the row sum counts code * block scale: times s_p)
          const float lse = 0.69314718055994531f *
                            (m + __log2f(l) + (kPv4 ? kLog2SP4 : 0.0f) - kPShift);
          a.lse[li] = a.lse_shift ? lse + a.lse_shift[li] : lse;
        }
      }
      g0 += nkv;
    }
  }

  // the O stores issued by this thread (lane 0 of a softmax warp) have completed
  if (warp < 8 && lane == 0) bulk_wait_all();
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
  CUtensorMap mq, mk, mv, mo;
  const uint64_t qrows = (uint64_t)a.B * a.Hq * a.N, kvrows = (uint64_t)a.B * a.Hkv * a.N;
  // V: E4M3 rows of 128 channels, 128-key boxes; or (pv4) V^T rows of N/2
  // code bytes per channel, boxes of 128 keys (64 bytes) x 128 channels
  const bool mv_ok =
      a.pv4 ? make_map_2d_u8_box(&mv, a.vc, (uint64_t)a.N / 2, (uint64_t)a.N / 2,
                                 (uint64_t)a.B * a.Hkv * 128, 64, 128, CU_TENSOR_MAP_SWIZZLE_64B)
            : make_map_2d_u8(&mv, a.vc, 128, kvrows, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!make_map_2d_u8(&mq, a.qc, 64, qrows, 128, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_map_2d_u8(&mk, a.kc, 64, kvrows, 128, CU_TENSOR_MAP_SWIZZLE_64B) || !mv_ok ||
      !make_map_2d_u8_box(&mo, a.o, (uint64_t)a.Hq * 256, (uint64_t)a.Hq * 256,
                          (uint64_t)a.B * a.N, 128, 32, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  static std::atomic<bool> attr_set[2][kMaxDevices];
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  auto* kernel = a.pv4 ? prefill_kernel<true> : prefill_kernel<false>;
  {
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kernel), kSmemBytes, dev,
                                  attr_set[a.pv4 ? 1 : 0]);
    if (e != cudaSuccess) return e;
  }
  Params p;
  p.a = a;
  p.log2e_rsqrt_d = (float)(1.4426950408889634 / std::sqrt(128.0));
  p.q_tiles = a.N / 128;
  p.items = p.q_tiles * a.B * a.Hq;
  if (p.items == 0) return cudaSuccess;
  const int sms = sm_count(dev);
  if (sms <= 0) return cudaErrorInvalidDevice;
  // persistent: one CTA per SM (shared memory and TMEM admit one), each
  // walking its share of the work items
  const unsigned grid = (unsigned)(p.items < sms ? p.items : sms);
  // may start (barriers, tensor memory) while the quantization finishes
  return launch_pdl(kernel, dim3(grid), dim3(kThreads), kSmemBytes, stream, mq, mk, mv, mo, p);
}

}  // namespace mpfa
