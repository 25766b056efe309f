// quantize.cu -- online NVFP4 quantization of Q and K and FP8 quantization
// of V (MpFA abstract: the QK operands in NVFP4, the PV operands in FP8;
// formats per the FP4 section of the "FlashAttention压到4位" explainer: E2M1
// codes, one E4M3 scale per 16 elements, one FP32 tensor scale), plus the
// rank-one smoothing of Q
// (block mean removed before quantization, the mean kept as T NVFP4 terms).
//
// Two HBM-streaming passes, because every tensor scale depends on the whole
// tensor:
//   stats_kernel : amax of K and V; for Q either amax(Q) or, with the
//                  smoothing, the fp32 block means qbar (exact column sums) and
//                  max(amax(Q - qbar), amax(qbar)).
//   quant_kernel : codes and scales of Q (or Q - qbar), of the qbar terms,
//                  of K and of V; the tensor scales.
// All rounding follows the rules in include/mpfa.h, one IEEE operation at a
// time (no fast math), so the codes are bit-identical to a plain
// sequential implementation of those rules.
#include <cuda_runtime.h>

#include "device.cuh"
#include "internal.h"

namespace mpfa {
namespace {

constexpr int kThreads = 128;        // quant_kernel
constexpr int kStatsThreads = 256;   // stats_kernel: 8 warps, one 16-column slice each
constexpr int kStatsCtasPerSm = 2;
constexpr float kNvfp4Max = 2688.0f;  // 6 * 448
constexpr float kFp8Max = 448.0f;

__device__ __forceinline__ float tensor_scale(unsigned amax_bits, float qmax) {
  float a = __uint_as_float(amax_bits);
  return a == 0.0f ? 1.0f : __fdiv_rn(a, qmax);
}

// Byte offset of block scale (row, j) in the 128-row tile layout.
__device__ __forceinline__ size_t sf_offset(size_t row, int j) {
  return (row >> 7) * 1024 + (size_t)(j >> 2) * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4;
}

// E2M1 value of a 4-bit code.
__device__ __forceinline__ float e2m1_value(uint32_t c) {
  uint32_t e = (c >> 1) & 3u, m = c & 1u;
  float mag = (e == 0) ? 0.5f * (float)m : (1.0f + 0.5f * (float)m) * (float)(1u << (e - 1));
  return (c & 8u) ? -mag : mag;
}

// x / d rounded to nearest even, for many x sharing one divisor d with
// y = RN(1/d) (Markstein's one-step correction, IBM J. Res. Dev. 34(1),
// 1990: q0 = RN(x y) is within an ulp of x / d, the residual x - d q0 comes
// from one fma, and RN(q0 + r y) is the correctly rounded quotient in
// binary32 when no intermediate leaves the normal range).  Callers keep d in
// [2^-90, 2^100]: then every quotient a code depends on (|x / d| >= 2^-10
// for E4M3, >= 1/4 for E2M1) has normal intermediates, and smaller ones
// keep their sign and stay below the first decision point.
constexpr float kDivLo = 0x1p-90f;
constexpr float kDivHi = 0x1p100f;
__device__ __forceinline__ float div_rn(float x, float d, float y) {
  const float q0 = __fmul_rn(x, y);
  return __fmaf_rn(__fmaf_rn(-d, q0, x), y, q0);
}

// Two quotients of div_rn at once (packed fp32; nd = -d, y = RN(1/d)).
__device__ __forceinline__ float2 div_rn2(float2 x, float2 nd, float2 y) {
  const float2 q0 = __fmul2_rn(x, y);
  return __ffma2_rn(__ffma2_rn(nd, q0, x), y, q0);
}

// Eight E2M1 codes (element 2i in the low nibble of byte i) of four pairs.
__device__ __forceinline__ uint32_t e2m1x8(float2 a, float2 b, float2 c, float2 d) {
  uint32_t r;
  asm("{\n.reg .b8 t0, t1, t2, t3;\n"
      "cvt.rn.satfinite.e2m1x2.f32 t0, %2, %1;\n"
      "cvt.rn.satfinite.e2m1x2.f32 t1, %4, %3;\n"
      "cvt.rn.satfinite.e2m1x2.f32 t2, %6, %5;\n"
      "cvt.rn.satfinite.e2m1x2.f32 t3, %8, %7;\n"
      "mov.b32 %0, {t0, t1, t2, t3};\n}"
      : "=r"(r)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y), "f"(d.x), "f"(d.y));
  return r;
}

// One NVFP4 block of 16 fp32 values with tensor scale s: eight code bytes
// (element 2i in the low nibble of byte i) and the E4M3 block scale.  The
// quotients are computed two at a time in packed fp32 operations (each half
// rounds on its own, so every quotient is the scalar one).
__device__ __forceinline__ void nvfp4_block(const float (&x)[16], float s, uint2& codes,
                                            uint32_t& sb) {
  float bamax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; i += 2) bamax = fmax3(bamax, fabsf(x[i]), fabsf(x[i + 1]));
  float t = __fdiv_rn(bamax, __fmul_rn(6.0f, s));
  sb = e4m3_pos(t);
  uint32_t w0 = 0, w1 = 0;
  if (sb != 0) {
    const float denom = __fmul_rn(e4m3_value(sb), s);
    float2 q[8];
    if (denom >= kDivLo && denom <= kDivHi && bamax <= 3.40282347e38f) {
      const float y = __frcp_rn(denom);
      const float2 y2 = make_float2(y, y), nd2 = make_float2(-denom, -denom);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        q[i] = div_rn2(make_float2(x[2 * i], x[2 * i + 1]), nd2, y2);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        q[i] = make_float2(__fdiv_rn(x[2 * i], denom), __fdiv_rn(x[2 * i + 1], denom));
    }
    w0 = e2m1x8(q[0], q[1], q[2], q[3]);
    w1 = e2m1x8(q[4], q[5], q[6], q[7]);
  }
  codes = make_uint2(w0, w1);
}

// Warp-cooperative write of one scale byte per lane (lane = 8 * row_in_warp
// + block j) into the tile layout: lanes with j % 4 == 0 store 4 bytes.
__device__ __forceinline__ void store_scales_tiled(uint8_t* scales, size_t row, int j,
                                                   uint32_t sb) {
  uint32_t b1 = __shfl_down_sync(0xffffffffu, sb, 1);
  uint32_t b2 = __shfl_down_sync(0xffffffffu, sb, 2);
  uint32_t b3 = __shfl_down_sync(0xffffffffu, sb, 3);
  if ((j & 3) == 0) {
    uint32_t word = sb | (b1 << 8) | (b2 << 16) | (b3 << 24);
    *reinterpret_cast<uint32_t*>(scales + sf_offset(row, j)) = word;
  }
}

__device__ __forceinline__ unsigned block_max_u32(unsigned v, unsigned* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) v = max(v, red[i]);
  }
  __syncthreads();
  return v;
}

// amax of a bf16 tensor of n8 groups of 8 values (grid-stride over `nblk`
// CTAs starting at block b0) -> atomicMax on the fp32 bit pattern.
__device__ void amax_bf16(const uint4* p, size_t n8, int b0, int nblk, unsigned* out,
                          unsigned* red) {
  unsigned m = 0;
  const size_t stride = (size_t)nblk * blockDim.x;
  size_t i = (size_t)(blockIdx.x - b0) * blockDim.x + threadIdx.x;
  // four independent loads in flight per thread
  for (; i + 3 * stride < n8; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = __ldg(p + i + u * stride);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      m = __vmaxu2(m, v[u].x & 0x7FFF7FFFu);
      m = __vmaxu2(m, v[u].y & 0x7FFF7FFFu);
      m = __vmaxu2(m, v[u].z & 0x7FFF7FFFu);
      m = __vmaxu2(m, v[u].w & 0x7FFF7FFFu);
    }
  }
  for (; i < n8; i += stride) {
    uint4 v = __ldg(p + i);
    m = __vmaxu2(m, v.x & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.y & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.z & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.w & 0x7FFF7FFFu);
  }
  m = max(m & 0xFFFFu, m >> 16);
  m = block_max_u32(m, red);
  if (threadIdx.x == 0 && m) atomicMax(out, m << 16);
}

// ---------------------------------------------------------------------------
// pass 1
// ---------------------------------------------------------------------------

// Exact fp32 means of the 128-row blocks of one (b, h) of a bf16 tensor
// x [B][N][H][128], persistent over the B*H*N/128 blocks (this CTA: blocks
// bid, bid + nblocks, ...), the next block's rows loaded while the current
// one is reduced.  Queries (kKeys false): the block means into out
// [B][H][N/128][128] and max(|qbar|, |x - qbar|) into *amax_out.  Keys
// (kKeys true): per block its means, column maxima and column minima into
// out [block][3][128] (the key-side smoothing's statistics).
template <bool kKeys>
__device__ __forceinline__ void block_stats(const __nv_bfloat16* x, int B, int N, int H, int bid,
                                            int nblocks, float* out, unsigned* amax_out,
                                            unsigned* red, float (*xpose)[32][33]) {
  // Warp w owns columns
  // 16w..16w+15 of the unit for all 128 rows (lane: 16-byte column group
  // 2w + (lane & 1), rows lane/2 + 16k), so every column reduction stays
  // inside the warp.
  //
  // Each column sum is exact, in two fp32 sums.  With E the largest
  // biased exponent of the column (at least 1) and u = 2^(E - 143) (the
  // bf16 spacing 9 binades below the largest value), every x splits
  // exactly into hi = x rounded to a multiple of u (adding and subtracting
  // C = 1.5 * 2^23 * u) and lo = x - hi, |lo| <= u / 2.  Any partial sum
  // of the his is a multiple of u below 2^24 u, and, when no nonzero value
  // lies more than 26 binades below E, any partial sum of the los is a
  // multiple of 2^(E - 160) below 2^24 times that: both are exact in fp32
  // in any order, and one fp32 addition rounds hi + lo correctly.  The
  // mean is that sum times 2^-7 (computed in fp64 if it is subnormal).  A
  // column with a wider spread, or with E > 247, takes an fp64 path with a
  // compensation term instead.  max |x - qbar| over a column is reached at
  // its largest or smallest x, since fp32(x - qbar) is monotonic in x.
  const int nblk = N / 128;
  const int units = B * H * nblk;
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cg = 2 * wid + (lane & 1);      // 16-byte column group (8 columns)
  const int rr = lane >> 1;                 // row within each group of 16
  auto load_unit = [&](int unit, uint4 (&w)[8]) {
    const int blk = unit % nblk, bh = unit / nblk;
    const int h = bh % H, b = bh / H;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const size_t n = (size_t)blk * 128 + rr + 16 * k;
      w[k] = __ldg(reinterpret_cast<const uint4*>(
          x + (((size_t)b * N + n) * H + h) * 128 + 8 * cg));
    }
  };
  auto word = [](const uint4& v, int j) -> uint32_t {
    return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
  };
  float (*xp)[33] = xpose[wid];
  unsigned m = 0;
  uint4 wn[8];
  if (bid < units) load_unit(bid, wn);
  for (int unit = bid; unit < units; unit += nblocks) {
    uint4 w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = wn[k];
    if (unit + nblocks < units) load_unit(unit + nblocks, wn);
    const int blk = unit % nblk, bh = unit / nblk;
    const int h = bh % H, b = bh / H;
    // per column over the 16 lanes of the column group: the largest and
    // smallest value (bf16 pairs, two columns per 32-bit word; a NaN makes
    // both NaN, which sends the column to the fp64 path) and the smallest
    // nonzero magnitude minus one (zero -> 0xFFFF)
    uint32_t hx[4], hn[4];
    float C[8];
    bool bad[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t mn = 0xFFFFFFFFu;
      __nv_bfloat162 vx = __halves2bfloat162(__ushort_as_bfloat16(0xFF80), __ushort_as_bfloat16(0xFF80));
      __nv_bfloat162 vn = __halves2bfloat162(__ushort_as_bfloat16(0x7F80), __ushort_as_bfloat16(0x7F80));
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t wv = word(w[k], j);
        const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&wv);
        vx = __hmax2_nan(vx, v);
        vn = __hmin2_nan(vn, v);
        mn = __vminu2(mn, __vsub2(wv & 0x7FFF7FFFu, 0x00010001u));
      }
      uint32_t ux = *reinterpret_cast<uint32_t*>(&vx), un = *reinterpret_cast<uint32_t*>(&vn);
#pragma unroll
      for (int o = 2; o < 32; o <<= 1) {
        const uint32_t ox = __shfl_xor_sync(0xffffffffu, ux, o);
        const uint32_t on = __shfl_xor_sync(0xffffffffu, un, o);
        mn = __vminu2(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        vx = __hmax2_nan(*reinterpret_cast<const __nv_bfloat162*>(&ux),
                         *reinterpret_cast<const __nv_bfloat162*>(&ox));
        vn = __hmin2_nan(*reinterpret_cast<const __nv_bfloat162*>(&un),
                         *reinterpret_cast<const __nv_bfloat162*>(&on));
        ux = *reinterpret_cast<uint32_t*>(&vx);
        un = *reinterpret_cast<uint32_t*>(&vn);
      }
      hx[j] = ux;
      hn[j] = un;
      // largest magnitude of each column: max(|largest|, |smallest|)
      const uint32_t mx = __vmaxu2(ux & 0x7FFF7FFFu, un & 0x7FFF7FFFu);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const uint32_t cmx = e ? mx >> 16 : mx & 0xFFFFu, cmn = e ? mn >> 16 : mn & 0xFFFFu;
        const int E = max((int)(cmx >> 7), 1);
        const int Emin = max((int)((cmn + 1) >> 7), 1);
        bad[2 * j + e] = E > 247 || (cmn != 0xFFFFu && Emin < E - 26);
        C[2 * j + e] = bad[2 * j + e] ? 0.0f : __uint_as_float(((uint32_t)(E + 7) << 23) | 0x400000u);
      }
    }
    // per column: the two sums over the lane's 8 rows, rows paired in the
    // two halves of packed fp32 operations (each half rounds on its own, so
    // every sum is the same exact value), stored lane-major [lane][column]
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const float2 cp = make_float2(C[t], C[t]), cn = make_float2(-C[t], -C[t]);
      const float2 m1 = make_float2(-1.0f, -1.0f);
      float2 s0 = make_float2(0.0f, 0.0f), s1 = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int k = 0; k < 8; k += 2) {
        const uint32_t wa = word(w[k], t >> 1), wb = word(w[k + 1], t >> 1);
        const float2 x = (t & 1) ? make_float2(bf16_hi(wa), bf16_hi(wb))
                                 : make_float2(bf16_lo(wa), bf16_lo(wb));
        const float2 hi = __fadd2_rn(__fadd2_rn(x, cp), cn);
        s0 = __fadd2_rn(s0, hi);
        s1 = __fadd2_rn(s1, __ffma2_rn(hi, m1, x));
      }
      xp[lane][t] = __fadd_rn(s0.x, s0.y);
      xp[lane][8 + t] = __fadd_rn(s1.x, s1.y);
    }
    __syncwarp();
    // lane L < 16 finishes column group 2w + (L & 1), column t = L >> 1:
    // sums over the 16 lanes of that group
    float s0 = 0.0f, s1 = 0.0f;
    const int gsel = lane & 1, tc = (lane >> 1) & 7;
    if (lane < 16) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float* row = xp[2 * i + gsel];
        s0 = __fadd_rn(s0, row[tc]);
        s1 = __fadd_rn(s1, row[8 + tc]);
      }
    }
    __syncwarp();   // xpose is rewritten by the next unit
    // the column's extremes (every lane of the group holds them)
    float xmx = 0.0f, xmn = 0.0f;
#pragma unroll
    for (int t = 0; t < 8; ++t)
      if (t == tc) {
        xmx = (t & 1) ? bf16_hi(hx[t >> 1]) : bf16_lo(hx[t >> 1]);
        xmn = (t & 1) ? bf16_hi(hn[t >> 1]) : bf16_lo(hn[t >> 1]);
      }
    // the column's flag (lane L belongs to column group 2w + (L & 1) itself)
    bool cbad = false;
#pragma unroll
    for (int t = 0; t < 8; ++t)
      if (t == tc) cbad = bad[t];
    if (lane < 16) {
      const int c = 8 * (2 * wid + gsel) + tc;
      float mean;
      if (!cbad) {
        mean = __fmul_rn(__fadd_rn(s0, s1), 0.0078125f);
        if (mean != 0.0f && fabsf(mean) < 1.17549435e-38f)
          mean = __double2float_rn(((double)s0 + (double)s1) * 0.0078125);
      } else {
        // fp64 sum with a compensation term (same rounding as a correctly
        // rounded sum whenever the correction captures the error)
        double sd = 0.0, comp = 0.0;
        for (int r = 0; r < 128; ++r) {
          const double v = (double)__bfloat162float(
              x[(((size_t)b * N + (size_t)blk * 128 + r) * H + h) * 128 + c]);
          const double t2 = sd + v;
          comp += (fabs(sd) >= fabs(v)) ? ((sd - t2) + v) : ((v - t2) + sd);
          sd = t2;
        }
        mean = (float)((sd + comp) * (1.0 / 128.0));
      }
      if (kKeys) {
        float* st = out + (size_t)unit * 384;
        st[c] = mean;
        st[128 + c] = xmx;
        st[256 + c] = xmn;
      } else {
        out[((size_t)bh * nblk + blk) * 128 + c] = mean;
        m = max(m, __float_as_uint(fabsf(mean)));
        m = max(m, __float_as_uint(fabsf(__fsub_rn(xmx, mean))));
        m = max(m, __float_as_uint(fabsf(__fsub_rn(xmn, mean))));
      }
    }
  }
  if (!kKeys) {
    m = block_max_u32(m, red);
    if (threadIdx.x == 0 && m) atomicMax(amax_out, m);
  }
}


__global__ void __launch_bounds__(kStatsThreads, kStatsCtasPerSm)
    stats_kernel(QuantArgs a, int nq_blocks, int nk_blocks, int nv_blocks) {
  __shared__ unsigned red[kStatsThreads / 32];
  pdl_trigger();
  // per warp: the 32 lanes' column partials, transposed through shared memory
  __shared__ float xpose[kStatsThreads / 32][32][33];
  int bid = blockIdx.x;
  if (bid < nq_blocks) {
    if (!a.compensate) {
      size_t n8 = (size_t)a.B * a.Nq * a.Hq * 16;
      amax_bf16(reinterpret_cast<const uint4*>(a.q), n8, 0, nq_blocks, &a.amax[0], red);
      return;
    }
    block_stats<false>(reinterpret_cast<const __nv_bfloat16*>(a.q), a.B, a.Nq, a.Hq, bid,
                       nq_blocks, a.qbar, &a.amax[0], red, xpose);
    return;
  }
  bid -= nq_blocks;
  if (bid < nk_blocks) {
    if (a.ksmooth) {
      // key-side smoothing: block statistics now, the channel means and
      // amax(K - kbar) in kbar_kernel
      block_stats<true>(reinterpret_cast<const __nv_bfloat16*>(a.k), a.B, a.Nk, a.Hkv, bid,
                        nk_blocks, a.kstat, nullptr, red, xpose);
      return;
    }
    size_t n8 = (size_t)a.B * a.Nk * a.Hkv * 16;
    amax_bf16(reinterpret_cast<const uint4*>(a.k), n8, nq_blocks, nk_blocks, &a.amax[1], red);
    return;
  }
  size_t n8 = (size_t)a.B * a.Nk * a.Hkv * 16;
  amax_bf16(reinterpret_cast<const uint4*>(a.v), n8, nq_blocks + nk_blocks, nv_blocks,
            &a.amax[2], red);
}

// Key-side smoothing: per (b, KV head) and channel, kbar = fp32(fp64 sum of
// the block means in block order / number of blocks), and amax(K - kbar)
// from the blocks' column extremes (fp32(x - kbar) is monotonic in x, so a
// column's largest |x - kbar| is at its largest or smallest x).
__global__ void __launch_bounds__(128) kbar_kernel(QuantArgs a) {
  __shared__ unsigned red[4];
  pdl_wait();
  pdl_trigger();
  const int bh = blockIdx.x, c = threadIdx.x;
  const int nblk = a.Nk / 128;
  const float* st = a.kstat + (size_t)bh * nblk * 384;
  double acc = 0.0;
  float mx = -INFINITY, mn = INFINITY;
  for (int blk = 0; blk < nblk; ++blk) {
    acc = __dadd_rn(acc, (double)st[(size_t)blk * 384 + c]);
    mx = fmaxf(mx, st[(size_t)blk * 384 + 128 + c]);
    mn = fminf(mn, st[(size_t)blk * 384 + 256 + c]);
  }
  const float kb = __double2float_rn(__ddiv_rn(acc, (double)nblk));
  a.kbar[(size_t)bh * 128 + c] = kb;
  unsigned m = max(__float_as_uint(fabsf(__fsub_rn(mx, kb))),
                   __float_as_uint(fabsf(__fsub_rn(mn, kb))));
  m = block_max_u32(m, red);
  if (threadIdx.x == 0 && m) atomicMax(&a.amax[1], m);
}

// ---------------------------------------------------------------------------
// pass 2
// ---------------------------------------------------------------------------

constexpr float kInvSqrtD = 0.08838834764831845f;  // fp32(1 / sqrt(128))

// sum_i e2m1(code_i) * w_i over the 16 codes of one NVFP4 block (fp32)
__device__ __forceinline__ float codes_dot(const uint2& codes, const float (&w)[16]) {
  const uint32_t cw[2] = {codes.x, codes.y};
  float acc = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i)
    acc = __fmaf_rn(e2m1_value((cw[i >> 3] >> (4 * (i & 7))) & 15u), w[i], acc);
  return acc;
}

// blockIdx.y: 0 = Q rows, 1 = qbar terms, 2 = K rows, 3 = V elements.
// kSmooth: the key-side smoothing variant (K' codes, the LSE term of every
// query row), with a register budget of its own.
template <bool kSmooth>
__global__ void __launch_bounds__(kThreads, kSmooth ? 5 : 6) quant_kernel(QuantArgs a) {
  pdl_wait();   // the statistics (and key means) of the kernels before
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int warps_total = gridDim.x * (kThreads / 32);
  const int gwarp = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  const int j = lane & 7;     // 16-element block within the row
  const int ri = lane >> 3;   // row within the warp's 4 rows
  const int part = blockIdx.y;

  if (part == 0 && a.q) {
    // One warp per (b, h, 128-row block): 8 rows per step (8 lanes per row,
    // one 16-element NVFP4 block per lane, two rows per lane), the block
    // means of the lane's 16 columns held in registers, the next step's rows
    // loaded before the current ones are coded.
    float s = tensor_scale(a.amax[0], kNvfp4Max);
    if (blockIdx.x == 0 && threadIdx.x == 0) *a.s_q = s;
    const __nv_bfloat16* q = reinterpret_cast<const __nv_bfloat16*>(a.q);
    const int nblk = a.Nq / 128;
    const size_t units = (size_t)a.B * a.Hq * nblk;
    // last units first: the stats pass read them last, so they may still be in L2
    for (size_t it = gwarp; it < units; it += warps_total) {
      const size_t unit = units - 1 - it;
      const size_t bh = unit / nblk, blk = unit % nblk;
      const size_t h = bh % a.Hq, b = bh / a.Hq;
      float m[16];
      if (a.compensate) {
        const float4* qb = reinterpret_cast<const float4*>(a.qbar + unit * 128 + 16 * j);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float4 v = qb[t];
          m[4 * t] = v.x;
          m[4 * t + 1] = v.y;
          m[4 * t + 2] = v.z;
          m[4 * t + 3] = v.w;
        }
      }
      // key-side smoothing: the lane's 16 channels of kbar and, with the
      // rank-one terms, their part of every row's q_eff . kbar (the terms
      // are re-derived here as the rank-one pass codes them)
      float kb[16];
      float rq = 0.0f;
      if (kSmooth && a.lse_shift) {
        const float4* kp = reinterpret_cast<const float4*>(
            a.kbar + (b * a.Hkv + h / (a.Hq / a.Hkv)) * 128 + 16 * j);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float4 v = kp[t];
          kb[4 * t] = v.x;
          kb[4 * t + 1] = v.y;
          kb[4 * t + 2] = v.z;
          kb[4 * t + 3] = v.w;
        }
        if (a.compensate) {
          float y[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) y[i] = m[i];
          for (int term = 0; term < a.T; ++term) {
            uint2 codes;
            uint32_t sb;
            nvfp4_block(y, s, codes, sb);
            const float sbv = e4m3_value(sb);
            rq = __fmaf_rn(sbv, codes_dot(codes, kb), rq);
            const uint32_t cw[2] = {codes.x, codes.y};
#pragma unroll
            for (int i = 0; i < 16; ++i)
              y[i] = __fsub_rn(y[i], __fmul_rn(__fmul_rn(e2m1_value((cw[i >> 3] >> (4 * (i & 7))) & 15u),
                                                         sbv), s));
          }
        }
      }
      // rows 8 step + ri and 8 step + 4 + ri of the block (lane group ri)
      auto src = [&](int row) {
        const size_t n = blk * 128 + row;
        return reinterpret_cast<const uint4*>(q + ((b * a.Nq + n) * a.Hq + h) * 128 + 16 * j);
      };
      uint4 nx[4];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        nx[2 * h2] = __ldg(src(4 * h2 + ri));
        nx[2 * h2 + 1] = __ldg(src(4 * h2 + ri) + 1);
      }
#pragma unroll 1
      for (int step = 0; step < 16; ++step) {
        uint4 cx[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) cx[i] = nx[i];
        if (step + 1 < 16) {
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            nx[2 * h2] = __ldg(src(8 * (step + 1) + 4 * h2 + ri));
            nx[2 * h2 + 1] = __ldg(src(8 * (step + 1) + 4 * h2 + ri) + 1);
          }
        }
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const uint32_t w[8] = {cx[2 * h2].x,     cx[2 * h2].y,     cx[2 * h2].z,
                                 cx[2 * h2].w,     cx[2 * h2 + 1].x, cx[2 * h2 + 1].y,
                                 cx[2 * h2 + 1].z, cx[2 * h2 + 1].w};
          float x[16];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            x[2 * i] = bf16_lo(w[i]);
            x[2 * i + 1] = bf16_hi(w[i]);
          }
          if (a.compensate) {
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
              const float2 d2 = __fadd2_rn(make_float2(x[i], x[i + 1]), make_float2(-m[i], -m[i + 1]));
              x[i] = d2.x;
              x[i + 1] = d2.y;
            }
          }
          const size_t r = bh * a.Nq + blk * 128 + 8 * step + 4 * h2 + ri;  // output row
          uint2 codes;
          uint32_t sb;
          nvfp4_block(x, s, codes, sb);
          *reinterpret_cast<uint2*>(a.qc + r * 64 + 8 * j) = codes;
          store_scales_tiled(a.qs, r, j, sb);
          if (kSmooth && a.lse_shift) {
            // s_q * (code * block scale + rank-one terms) . kbar / sqrt(d)
            float part = __fmaf_rn(e4m3_value(sb), codes_dot(codes, kb), rq);
            part += __shfl_xor_sync(0xffffffffu, part, 1);
            part += __shfl_xor_sync(0xffffffffu, part, 2);
            part += __shfl_xor_sync(0xffffffffu, part, 4);
            if (j == 0) a.lse_shift[r] = __fmul_rn(__fmul_rn(part, s), kInvSqrtD);
          }
        }
      }
    }
    return;
  }
  if (part == 1 && a.q && a.compensate) {
    float s = tensor_scale(a.amax[0], kNvfp4Max);
    size_t rows = (size_t)a.B * a.Hq * (a.Nq / 128);
    for (size_t u = gwarp; u < rows / 4 + 1; u += warps_total) {
      size_t r = u * 4 + ri;
      if (r >= rows) continue;
      float x[16];
      const float4* src = reinterpret_cast<const float4*>(a.qbar + r * 128 + 16 * j);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        float4 m = src[t];
        x[4 * t] = m.x;
        x[4 * t + 1] = m.y;
        x[4 * t + 2] = m.z;
        x[4 * t + 3] = m.w;
      }
      for (int term = 0; term < a.T; ++term) {
        uint2 codes;
        uint32_t sb;
        nvfp4_block(x, s, codes, sb);
        *reinterpret_cast<uint2*>(a.qbc + (r * a.T + term) * 64 + 8 * j) = codes;
        a.qbs[(r * a.T + term) * 8 + j] = (uint8_t)sb;
        // residual for the next term: x - fp32(fp32(code * sb) * s)
        float sbv = e4m3_value(sb);
        uint32_t w[2] = {codes.x, codes.y};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          uint32_t c = (w[i >> 3] >> (4 * (i & 7))) & 15u;
          float deq = __fmul_rn(__fmul_rn(e2m1_value(c), sbv), s);
          x[i] = __fsub_rn(x[i], deq);
        }
      }
    }
    return;
  }
  if (part == 2 && a.k) {
    float s = tensor_scale(a.amax[1], kNvfp4Max);
    if (blockIdx.x == 0 && threadIdx.x == 0) *a.s_k = s;
    const __nv_bfloat16* k = reinterpret_cast<const __nv_bfloat16*>(a.k);
    // 8 rows per warp step (two per lane), the next step's rows loaded
    // before the current ones are coded; rows is a multiple of 128
    const size_t nu = (size_t)a.B * a.Hkv * a.Nk / 8;
    auto src = [&](size_t r) {
      const size_t n = r % a.Nk, bh = r / a.Nk;
      const size_t h = bh % a.Hkv, b = bh / a.Hkv;
      return reinterpret_cast<const uint4*>(k + ((b * a.Nk + n) * a.Hkv + h) * 128 + 16 * j);
    };
    uint4 nx[4];
    size_t u = gwarp;
    if (u < nu) {
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        nx[2 * h2] = __ldg(src(8 * u + 4 * h2 + ri));
        nx[2 * h2 + 1] = __ldg(src(8 * u + 4 * h2 + ri) + 1);
      }
    }
    for (; u < nu; u += warps_total) {
      uint4 cx[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) cx[i] = nx[i];
      if (u + warps_total < nu) {
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          nx[2 * h2] = __ldg(src(8 * (u + warps_total) + 4 * h2 + ri));
          nx[2 * h2 + 1] = __ldg(src(8 * (u + warps_total) + 4 * h2 + ri) + 1);
        }
      }
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const uint32_t w[8] = {cx[2 * h2].x,     cx[2 * h2].y,     cx[2 * h2].z,
                               cx[2 * h2].w,     cx[2 * h2 + 1].x, cx[2 * h2 + 1].y,
                               cx[2 * h2 + 1].z, cx[2 * h2 + 1].w};
        float x[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          x[2 * i] = bf16_lo(w[i]);
          x[2 * i + 1] = bf16_hi(w[i]);
        }
        const size_t r = 8 * u + 4 * h2 + ri;
        if (kSmooth) {  // K' = fp32(K - kbar)
          const float4* kp = reinterpret_cast<const float4*>(a.kbar + (r / a.Nk) * 128 + 16 * j);
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const float4 v = kp[t];
            x[4 * t] = __fsub_rn(x[4 * t], v.x);
            x[4 * t + 1] = __fsub_rn(x[4 * t + 1], v.y);
            x[4 * t + 2] = __fsub_rn(x[4 * t + 2], v.z);
            x[4 * t + 3] = __fsub_rn(x[4 * t + 3], v.w);
          }
        }
        uint2 codes;
        uint32_t sb;
        nvfp4_block(x, s, codes, sb);
        *reinterpret_cast<uint2*>(a.kc + r * 64 + 8 * j) = codes;
        store_scales_tiled(a.ks, r, j, sb);
      }
    }
    return;
  }
  if (part == 3 && a.v) {
    float s = tensor_scale(a.amax[2], kFp8Max);
    if (blockIdx.x == 0 && threadIdx.x == 0) *a.s_v = s;
    const bool fast = s >= kDivLo && s <= kDivHi;
    const float ys = __frcp_rn(s);
    const __nv_bfloat16* v = reinterpret_cast<const __nv_bfloat16*>(a.v);
    // 16-element units, two per thread per step (e and e + stride), the
    // next step's loaded before the current ones are coded
    const size_t units = (size_t)a.B * a.Hkv * a.Nk * 8;
    const size_t stride = (size_t)gridDim.x * kThreads;
    auto src = [&](size_t e) {
      const size_t r = e >> 3;  // output row (b, h, n)
      const size_t n = r % a.Nk, bh = r / a.Nk;
      const size_t h = bh % a.Hkv, b = bh / a.Hkv;
      return reinterpret_cast<const uint4*>(v + ((b * a.Nk + n) * a.Hkv + h) * 128 +
                                            16 * (int)(e & 7));
    };
    auto code = [&](const uint4& c0, const uint4& c1, size_t e) {
      const uint32_t w8[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      float x[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        x[2 * i] = bf16_lo(w8[i]);
        x[2 * i + 1] = bf16_hi(w8[i]);
      }
      uint32_t w[4];
      float xm = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; i += 2) xm = fmax3(xm, fabsf(x[i]), fabsf(x[i + 1]));
      if (fast && xm <= 3.40282347e38f) {
        const float2 y2 = make_float2(ys, ys), nd2 = make_float2(-s, -s);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float2 u0 = div_rn2(make_float2(x[4 * t], x[4 * t + 1]), nd2, y2);
          const float2 u1 = div_rn2(make_float2(x[4 * t + 2], x[4 * t + 3]), nd2, y2);
          w[t] = e4m3x4(u0.x, u0.y, u1.x, u1.y);
        }
      } else {
#pragma unroll
        for (int t = 0; t < 4; ++t)
          w[t] = e4m3x4(__fdiv_rn(x[4 * t], s), __fdiv_rn(x[4 * t + 1], s),
                        __fdiv_rn(x[4 * t + 2], s), __fdiv_rn(x[4 * t + 3], s));
      }
      *reinterpret_cast<uint4*>(a.vc + (e >> 3) * 128 + 16 * (int)(e & 7)) =
          make_uint4(w[0], w[1], w[2], w[3]);
    };
    uint4 nx[4];
    size_t e = (size_t)blockIdx.x * kThreads + threadIdx.x;
    auto load2 = [&](size_t e0) {
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        if (e0 + h2 * stride < units) {
          nx[2 * h2] = __ldg(src(e0 + h2 * stride));
          nx[2 * h2 + 1] = __ldg(src(e0 + h2 * stride) + 1);
        }
      }
    };
    load2(e);
    for (; e < units; e += 2 * stride) {
      uint4 cx[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) cx[i] = nx[i];
      load2(e + 2 * stride);
      code(cx[0], cx[1], e);
      if (e + stride < units) code(cx[2], cx[3], e + stride);
    }
  }
}

// ---------------------------------------------------------------------------
// quantize-on-append into a decode cache
// ---------------------------------------------------------------------------


// New K and V rows, quantized with the cache's tensor scales exactly as the
// quant pass codes them (the same block and element arithmetic), written at
// cache rows seqlens[b] + t.  One thread per 16-element block, eight per row,
// four rows per warp: the tiled scale store gathers a row's neighbouring
// blocks by shuffles, so every lane takes part in every step and the
// out-of-range and overrunning rows are masked, not skipped.
__global__ void __launch_bounds__(kThreads) append_kernel(AppendArgs a) {
  pdl_wait();   // the cache and its tensor scales may come from the kernel before
  pdl_trigger();
  const float sk = *a.s_k, sv = *a.s_v;
  const bool vfast = sv >= kDivLo && sv <= kDivHi;
  const float ysv = __frcp_rn(sv);
  const __nv_bfloat16* kn = reinterpret_cast<const __nv_bfloat16*>(a.k_new);
  const __nv_bfloat16* vn = reinterpret_cast<const __nv_bfloat16*>(a.v_new);
  const size_t units = (size_t)a.B * a.n_new * a.Hkv * 8;
  const size_t stride = (size_t)gridDim.x * kThreads;
  const int lane = threadIdx.x & 31;
  for (size_t base = (size_t)blockIdx.x * kThreads + (threadIdx.x & ~31u); base < units;
       base += stride) {
    const size_t u = base + lane;
    const int j = (int)(u & 7);
    const size_t rr = u >> 3;  // new row in the input's order (b, t, h)
    const bool in = u < units;
    int b = 0, t = 0, h = 0;
    if (in) {
      h = (int)(rr % a.Hkv);
      const size_t bt = rr / a.Hkv;
      t = (int)(bt % a.n_new);
      b = (int)(bt / a.n_new);
    }
    const int pos0 = in ? a.seqlens[b] : 0;
    const bool fits = pos0 >= 0 && pos0 <= a.Lmax - a.n_new;
    if (in && !fits && t == 0 && h == 0 && j == 0) record_error(a.err, kErrInvalidArg);
    bool store = in && fits;
    size_t r = ((size_t)b * a.Hkv + h) * a.Lmax + (size_t)(store ? pos0 + t : 0);
    if (a.block_table && store) {
      // paged pool: row pos of sequence b is row pos % 128 of page
      // block_table[b][pos / 128], whose KV head h rows start at (page * Hkv + h) * 128
      const int pos = pos0 + t;
      const int page = a.block_table[(size_t)b * a.max_pages + pos / 128];
      if (page < 0 || page >= a.num_pages) {
        if (j == 0) record_error(a.err, kErrInvalidArg);
        store = false;
        r = 0;
      } else {
        r = ((size_t)page * a.Hkv + h) * 128 + (size_t)(pos % 128);
      }
    }
    float x[16];
    {
      uint4 c0 = make_uint4(0u, 0u, 0u, 0u), c1 = c0;
      if (in) {
        const uint4* src = reinterpret_cast<const uint4*>(kn + rr * 128 + 16 * j);
        c0 = __ldg(src);
        c1 = __ldg(src + 1);
      }
      const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        x[2 * i] = bf16_lo(w[i]);
        x[2 * i + 1] = bf16_hi(w[i]);
      }
    }
    if (a.kbar) {  // a smoothed cache holds K' = fp32(K - kbar)
      const float* kb = a.kbar + ((size_t)b * a.Hkv + h) * 128 + 16 * j;
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = __fsub_rn(x[i], kb[i]);
    }
    uint2 codes;
    uint32_t sb;
    nvfp4_block(x, sk, codes, sb);
    if (store) *reinterpret_cast<uint2*>(a.kc + r * 64 + 8 * j) = codes;
    {
      const uint32_t b1 = __shfl_down_sync(0xffffffffu, sb, 1);
      const uint32_t b2 = __shfl_down_sync(0xffffffffu, sb, 2);
      const uint32_t b3 = __shfl_down_sync(0xffffffffu, sb, 3);
      if (store && (j & 3) == 0)
        *reinterpret_cast<uint32_t*>(a.ks + sf_offset(r, j)) =
            sb | (b1 << 8) | (b2 << 16) | (b3 << 24);
    }
    if (in) {
      const uint4* src = reinterpret_cast<const uint4*>(vn + rr * 128 + 16 * j);
      const uint4 c0 = __ldg(src), c1 = __ldg(src + 1);
      const uint32_t w8[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        x[2 * i] = bf16_lo(w8[i]);
        x[2 * i + 1] = bf16_hi(w8[i]);
      }
      float xm = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) xm = fmaxf(xm, fabsf(x[i]));
      uint32_t w[4];
      if (vfast && xm <= 3.40282347e38f) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          w[q] = e4m3x4(div_rn(x[4 * q], sv, ysv), div_rn(x[4 * q + 1], sv, ysv),
                        div_rn(x[4 * q + 2], sv, ysv), div_rn(x[4 * q + 3], sv, ysv));
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          w[q] = e4m3x4(__fdiv_rn(x[4 * q], sv), __fdiv_rn(x[4 * q + 1], sv),
                        __fdiv_rn(x[4 * q + 2], sv), __fdiv_rn(x[4 * q + 3], sv));
      }
      if (store)
        *reinterpret_cast<uint4*>(a.vc + r * 128 + 16 * j) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// Full-FP4 PV ablation: V^T in NVFP4 along the keys (the reduction
// dimension of P V), one CTA per (b, KV head, 128-key tile).  The tile's
// 128 keys x 128 channels come into shared memory row by row (coalesced),
// then thread t codes channel t % 128 over the 64 keys of half t / 128: four
// 16-key blocks with the same block routine (and so the same codes) as K,
// 32 code bytes and one word of four block scales.
__global__ void __launch_bounds__(256) vt_quant_kernel(QuantArgs a) {
  __shared__ uint4 tile[128][16];   // [key][16-byte chunk of 8 channels]
  pdl_wait();   // amax(V) from the statistics kernel
  pdl_trigger();
  const int ntiles = a.Nk / 128;
  const int u = blockIdx.x, j = u % ntiles, bh = u / ntiles;
  const int h = bh % a.Hkv, b = bh / a.Hkv;
  const float s = tensor_scale(a.amax[2], kNvfp4Max);
  if (u == 0 && threadIdx.x == 0) *a.s_v = s;
  const __nv_bfloat16* v = reinterpret_cast<const __nv_bfloat16*>(a.v);
  for (int i = threadIdx.x; i < 128 * 16; i += blockDim.x) {
    const int key = i >> 4, ch = i & 15;
    tile[key][ch] = __ldg(reinterpret_cast<const uint4*>(
        v + (((size_t)b * a.Nk + (size_t)j * 128 + key) * a.Hkv + h) * 128 + 8 * ch));
  }
  __syncthreads();
  const int c = threadIdx.x & 127, half = threadIdx.x >> 7;
  const __nv_bfloat16* tb = reinterpret_cast<const __nv_bfloat16*>(&tile[0][0]);
  uint32_t cw[8];
  uint32_t sbw = 0;
#pragma unroll
  for (int kb = 0; kb < 4; ++kb) {
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = __bfloat162float(tb[(64 * half + 16 * kb + i) * 128 + c]);
    uint2 codes;
    uint32_t sb;
    nvfp4_block(x, s, codes, sb);
    cw[2 * kb] = codes.x;
    cw[2 * kb + 1] = codes.y;
    sbw |= sb << (8 * kb);
  }
  uint4* dst = reinterpret_cast<uint4*>(a.vtc + ((size_t)bh * 128 + c) * (a.Nk / 2) +
                                        (size_t)j * 64 + 32 * half);
  dst[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
  dst[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
  *reinterpret_cast<uint32_t*>(a.vts + ((size_t)bh * ntiles + j) * 1024 + 512 * half +
                               (c & 31) * 16 + ((c >> 5) & 3) * 4) = sbw;
}

int num_sms() {
  const int n = sm_count(current_device());
  return n > 0 ? n : 148;
}

}  // namespace

size_t quant_workspace_bytes(int B, int Nq, int Nk, int Hq, int Hkv, int compensate,
                             int ksmooth) {
  size_t bytes = 256;  // amax words
  if (compensate) bytes += (size_t)B * Hq * (Nq / 128) * 128 * sizeof(float);
  if (ksmooth) bytes += (size_t)B * Hkv * (Nk / 128) * 384 * sizeof(float);
  return bytes;
}

cudaError_t launch_quantize(const QuantArgs& a, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(a.amax, 0, 3 * sizeof(unsigned), stream);
  if (e != cudaSuccess) return e;
  const int sms = num_sms();
  auto amax_blocks = [&](size_t elems) {
    size_t need = (elems / 8 + kStatsThreads - 1) / kStatsThreads;
    size_t cap = (size_t)sms * kStatsCtasPerSm;   // one resident wave
    return (int)(need < cap ? (need ? need : 1) : cap);
  };
  int nq = 0, nk = 0, nv = 0;
  if (a.q) {
    const int units = a.B * a.Hq * (a.Nq / 128);
    nq = a.compensate ? (units < kStatsCtasPerSm * sms ? units : kStatsCtasPerSm * sms)  // persistent
                      : amax_blocks((size_t)a.B * a.Nq * a.Hq * 128);
  }
  if (a.k) {
    const int units = a.B * a.Hkv * (a.Nk / 128);
    nk = a.ksmooth ? (units < kStatsCtasPerSm * sms ? units : kStatsCtasPerSm * sms)  // persistent
                   : amax_blocks((size_t)a.B * a.Nk * a.Hkv * 128);
  }
  if (a.v) nv = amax_blocks((size_t)a.B * a.Nk * a.Hkv * 128);
  if (nq + nk + nv > 0) {
    stats_kernel<<<nq + nk + nv, kStatsThreads, 0, stream>>>(a, nq, nk, nv);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (a.k && a.ksmooth) {
    e = launch_pdl(kbar_kernel, dim3(a.B * a.Hkv), dim3(128), 0, stream, a);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(sms * 8, 4);
  // the coding pass may start while the statistics finish (it waits for them)
  if (a.ksmooth)
    e = launch_pdl(quant_kernel<true>, grid, dim3(kThreads), 0, stream, a);
  else
    e = launch_pdl(quant_kernel<false>, grid, dim3(kThreads), 0, stream, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_quantize_vt(const QuantArgs& a, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(a.amax, 0, 3 * sizeof(unsigned), stream);
  if (e != cudaSuccess) return e;
  const int sms = num_sms();
  const size_t n8 = (size_t)a.B * a.Nk * a.Hkv * 16;
  size_t need = (n8 + kStatsThreads - 1) / kStatsThreads;
  const size_t cap = (size_t)sms * kStatsCtasPerSm;
  const int nv = (int)(need < cap ? (need ? need : 1) : cap);
  stats_kernel<<<nv, kStatsThreads, 0, stream>>>(a, 0, 0, nv);   // amax(V) only
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_pdl(vt_quant_kernel, dim3(a.B * a.Hkv * (a.Nk / 128)), dim3(256), 0, stream, a);
}

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream) {
  const size_t units = (size_t)a.B * a.n_new * a.Hkv * 8;
  if (units == 0) return cudaSuccess;
  const size_t need = (units + kThreads - 1) / kThreads;
  const size_t cap = (size_t)num_sms() * 8;
  cudaError_t e = launch_pdl(append_kernel, dim3((unsigned)(need < cap ? need : cap)),
                             dim3(kThreads), 0, stream, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mpfa
