/*
 * mpfa.h -- C ABI of the MpFA QK4PV8 attention forward for GB300 (sm_103a).
 *
 * The method: "MpFA: Hardware-Efficient Train-Free QK4V8 FlashAttention
 * Kernels on Blackwell GPUs" (abstract).  Q and K are quantized online to
 * NVFP4 and multiplied on block-scaled FP4 tensor cores; P and V are FP8
 * E4M3 and multiplied on FP8 tensor cores ("QK4PV8"); a rank-one smoothing
 * compensation is one extra tensor-core MMA into the score accumulator; work
 * is partitioned differently for prefill and decode.  The number formats
 * follow the FP4 section ("FP4 只有约 15 个可表示的数") of the
 * "FlashAttention压到4位" explainer: E2M1 codes, one E4M3 scale per 16
 * elements, one FP32 tensor scale.  The online softmax follows that
 * explainer's FlashAttention-2 section ("注意力慢在哪儿").
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - All pointers are DEVICE pointers unless stated otherwise, owned by the
 *    caller, 16-byte aligned.  The library allocates and frees nothing and
 *    never synchronizes (except mpfa_get_error).  Work is enqueued on the
 *    caller's stream and runs asynchronously.
 *  - Head dimension d must be 128.  Query head h uses KV head h / (Hq/Hkv).
 *  - Host-checkable faults return synchronously with nothing enqueued:
 *    MPFA_ERR_INVALID_ARG (null pointer, misaligned pointer, bad size,
 *    workspace too small) or MPFA_ERR_UNSUPPORTED (d != 128, a T other than
 *    1 or 2).  A failed launch returns MPFA_ERR_CUDA.  A kernel whose bounded
 *    wait on an on-chip barrier expires records MPFA_ERR_TIMEOUT in a device
 *    status word and exits; mpfa_get_error reports it.
 *  - Per-device state (the status word's address, kernel attributes, SM
 *    counts) is looked up on a device's first call and cached; the cache
 *    assumes the device's primary context is not reset while the library is
 *    loaded.
 *
 * Quantized layouts
 * -----------------
 *  NVFP4 codes: [rows][64] bytes, two E2M1 codes per byte, the element with
 *  the lower index in the low nibble.  E2M1 code: bit 3 sign, bits 2..1
 *  exponent, bit 0 mantissa (magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6).
 *
 *  NVFP4 block scales ("128-row tile layout"): rows*8 bytes of unsigned E4M3
 *  (OCP E4M3, bias 7, max 448).  The scale of row r, block j (elements
 *  16j..16j+15, j = 0..7) is at byte
 *      (r / 128) * 1024 + (j / 4) * 512 + (r % 32) * 16 + ((r / 32) % 4) * 4 + (j % 4)
 *  so that each 128-row tile holds, per 64-element chunk, one 512-byte block
 *  the tensor core reads directly.  Row counts must be multiples of 128.
 *
 *  FP8 codes: OCP E4M3 bytes.
 *
 *  Quantization rules (FP32 arithmetic, each operation rounded once):
 *      s   = amax / 2688 (1 if amax == 0)        tensor scale, NVFP4
 *      sb  = E4M3_rne_sat(bamax / (6 * s))        per 16 elements
 *      code= E2M1_rne_sat(x / (sb * s)), all zero if sb == 0; sign bit = sign of x
 *      V:   s_v = amax / 448, code = E4M3_rne_sat(v / s_v)
 *  Rank-one smoothing (compensate != 0): per query block (128 rows of one
 *  (b, h) in prefill; the Hq/Hkv query heads of one KV head in decode)
 *      qbar = fp32 mean of the block's rows, Q' = Q - qbar,
 *      s_q from max(amax(Q'), amax(qbar)), codes of Q' and T NVFP4 terms of
 *      qbar (term 1 of qbar, term 2 of the fp32 residual qbar - deq(term 1)),
 *      all sharing s_q.  The score is s_q s_k (Q'K^T + 1 * (sum_t term_t) K^T).
 */
#ifndef MPFA_H
#define MPFA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (the CUDA runtime's stream handle). */
typedef struct CUstream_st *mpfa_stream_t;

typedef enum {
    MPFA_OK = 0,
    MPFA_ERR_INVALID_ARG = 1,
    MPFA_ERR_UNSUPPORTED = 2,
    MPFA_ERR_CUDA = 3,
    MPFA_ERR_TIMEOUT = 4
} mpfa_status;

/* NVFP4 tensor: codes [rows][64], scales in the 128-row tile layout,
 * tensor_scale points at one device float. */
typedef struct {
    uint8_t *codes;
    uint8_t *scales;
    float *tensor_scale;
} mpfa_nvfp4;

/* FP8 E4M3 tensor with one device float tensor scale. */
typedef struct {
    uint8_t *codes;
    float *tensor_scale;
} mpfa_fp8;

/* Rank-one smoothing terms: codes [nblocks][T][64], scales [nblocks][T][8]
 * (row-major E4M3), sharing the query tensor scale. */
typedef struct {
    uint8_t *codes;
    uint8_t *scales;
} mpfa_rank1;

/* Key-side smoothing outputs (an addition to the MpFA method, resting on the
 * softmax's invariance to one shift of all logits of a row, the explainer's
 * attention section).  kbar [B][Hkv][d] fp32: per (batch, KV head) and
 * channel, the fp32 rounding of the fp64 mean (block order, sequential) of
 * the keys' 128-row block means, each the correctly rounded fp32 mean of
 * its block.  The keys are coded as K' = fp32(K - kbar) with s_k from
 * amax(K').  lse_shift [B][Hq][Nq] fp32 (may be NULL): for every query row
 * the logit part the smoothed keys leave out, q_eff . kbar / sqrt(d), where
 * q_eff = s_q * (code * block scale of the row + the rank-one terms of its
 * block); mpfa_prefill adds it to the LSE.  O does not depend on it.  Both
 * device pointers, caller-owned. */
typedef struct {
    float *kbar;
    float *lse_shift;
} mpfa_ksmooth;

/* Human-readable name of a status. */
const char *mpfa_status_string(mpfa_status s);

/* Name of the last CUDA runtime error (cudaGetErrorName) behind an
 * MPFA_ERR_CUDA returned to the calling host thread; "cudaSuccess" if there
 * was none.  Diagnostic only: the library's own state, not the caller's CUDA
 * error state. */
const char *mpfa_last_cuda_error(void);

/* Bytes of device workspace mpfa_quantize_qkv needs (amax words, the fp32
 * block means of Q when compensate != 0, the keys' block statistics when
 * ksmooth != 0).  Nq = 0 / Nk = 0 for a call without queries / keys. */
size_t mpfa_quantize_workspace_size(int B, int Nq, int Nk, int Hq, int Hkv, int compensate,
                                    int ksmooth);

/*
 * Online quantization of one attention layer's inputs (MpFA abstract: the QK
 * operands in NVFP4, the PV operands in FP8; formats per the FP4 explainer
 * section).
 *
 *   q_bf16 [B][Nq][Hq][d], k_bf16 / v_bf16 [B][Nk][Hkv][d]  bf16, device.
 *   Any of q/k/v may be NULL to skip it (its output must then be NULL too);
 *   e.g. q = NULL builds a decode KV cache.
 *   q_out:  codes [B][Hq][Nq][64], scales tiled over the B*Hq*Nq rows.
 *   qbar_out (compensate != 0): codes [B][Hq][Nq/128][T][64], scales [..][T][8].
 *   k_out:  codes [B][Hkv][Nk][64], scales tiled over B*Hkv*Nk rows.
 *   v_out:  codes [B][Hkv][Nk][128].
 *   Nq, Nk multiples of 128 (when the tensor is given), T in {1, 2};
 *   B*Hq*Nq and B*Hkv*Nk below 2^31 rows (the row index the kernels and the
 *   tensor-memory-access coordinates use is 32-bit).
 *   Tensor scales are computed over each whole tensor argument.
 *   ksmooth: NULL, or key-side smoothing (see mpfa_ksmooth): needs k_bf16;
 *   lse_shift, if given, needs q_bf16 and Hq % Hkv == 0.
 *   workspace: device buffer of at least mpfa_quantize_workspace_size bytes.
 */
mpfa_status mpfa_quantize_qkv(const void *q_bf16, const void *k_bf16, const void *v_bf16,
                              int B, int Nq, int Nk, int Hq, int Hkv, int d, int compensate,
                              int T, mpfa_nvfp4 *q_out, mpfa_rank1 *qbar_out, mpfa_nvfp4 *k_out,
                              mpfa_fp8 *v_out, const mpfa_ksmooth *ksmooth, void *workspace,
                              size_t ws_bytes, mpfa_stream_t stream);

/*
 * mpfa_quantize_qkv without a caller workspace.  The paper has no
 * counterpart: this entry point exists for callers that cannot allocate
 * device memory (a serving process whose HBM is owned by its own pool and
 * must not call cudaMalloc after start-up; a host that hands the library only
 * its input and output tensors).  It allocates nothing; its scratch is a
 * fixed device array inside the library of 256 + 16 MiB bytes, which every
 * GPU that loads the library holds until the process exits.
 *   Arguments, layouts and results are those of mpfa_quantize_qkv without
 *   key-side smoothing.
 *   Limit: with compensate != 0 the block means of Q must fit, i.e.
 *   B * Hq * Nq / 128 <= 32768 query blocks; larger problems return
 *   MPFA_ERR_INVALID_ARG with nothing enqueued (use mpfa_quantize_qkv).
 *   The first call on each device looks up the array's device address (with
 *   that device current) and caches it; make that first call before any
 *   stream capture.  All calls on a device share the array: calls whose work
 *   overlaps on the GPU race, so order them (one stream, or events).
 */
mpfa_status mpfa_quantize_qkv_noalloc(const void *q_bf16, const void *k_bf16,
                                      const void *v_bf16, int B, int Nq, int Nk, int Hq, int Hkv,
                                      int d, int compensate, int T, mpfa_nvfp4 *q_out,
                                      mpfa_rank1 *qbar_out, mpfa_nvfp4 *k_out, mpfa_fp8 *v_out,
                                      mpfa_stream_t stream);

/*
 * Prefill forward (MpFA abstract; FlashAttention-2 tiling and online softmax
 * per the explainer): O = softmax(s_q s_k S / sqrt(d)) V with S from the
 * block-scaled FP4 product plus the rank-one term, P stored as E4M3(2^4 p)
 * with p = 2^(t - m) against the row's reference max m (set by the first
 * KV tile, moved to a tile's max only when that max exceeds m by more than
 * 4 in log2 units), KV tiles of 128 keys in ascending order, N_q = N_k = N (causal: key j
 * visible to query i iff j <= i).
 *   q/k/v from mpfa_quantize_qkv; qbar NULL iff compensate == 0.
 *   o_bf16 [B][N][Hq][d]; lse [B][Hq][N] natural-log sum-exp of the scaled
 *   logits (may be NULL).  N multiple of 128, Hq % Hkv == 0.
 *   lse_shift: NULL, or mpfa_ksmooth.lse_shift of keys quantized with
 *   key-side smoothing, added to the LSE.
 */
mpfa_status mpfa_prefill(const mpfa_nvfp4 *q, const mpfa_rank1 *qbar, const mpfa_nvfp4 *k,
                         const mpfa_fp8 *v, int B, int N, int Hq, int Hkv, int d, int causal,
                         int compensate, int T, void *o_bf16, float *lse,
                         const float *lse_shift, mpfa_stream_t stream);

/*
 * Full-FP4 PV ablation (the MpFA abstract weighs QK4PV8 against full FP4):
 * V^T quantized to NVFP4 along the keys, the reduction dimension of P V.
 * Per (b, KV head, channel) row of V^T, 16-key blocks with E4M3 block scales
 * and one fp32 tensor scale fp32(amax(V) / 2688), the same quantizer rules
 * as K.
 *   v_bf16 [B][Nk][Hkv][d], Nk a multiple of 128, d == 128.
 *   vt_out->codes [B][Hkv][d][Nk/2] (key 2i in the low nibble of byte i);
 *   vt_out->scales one 1 KB tile per (b, KV head, 128-key tile) in the
 *   tensor core's scale-copy order (byte (c%32)*16 + ((c/32)%4)*4 + j%4 of
 *   the 512-byte block j/4 for channel c, 16-key block j);
 *   vt_out->tensor_scale: one float.
 *   workspace: device, 16-byte aligned, >= 256 bytes (the amax words).
 * Caller-owned buffers; asynchronous on `stream`.
 */
mpfa_status mpfa_quantize_v_fp4(const void *v_bf16, int B, int Nk, int Hkv, int d,
                                mpfa_nvfp4 *vt_out, void *workspace, size_t ws_bytes,
                                mpfa_stream_t stream);

/*
 * Prefill forward with the full-FP4 PV of the ablation: as mpfa_prefill up
 * to p = 2^(t - m) under the same reference-max rule; then x = 2^4 p coded in
 * NVFP4 per 16 keys of a row with the fixed tensor scale
 * fp32(2^8 / 2688), multiplied in block-scaled FP4 with vt from
 * mpfa_quantize_v_fp4; the row sum l adds the same rounded values.
 *   Arguments as mpfa_prefill, vt in place of v; no lse_shift (the key-side
 *   smoothing is not part of the ablation).
 */
mpfa_status mpfa_prefill_fp4pv(const mpfa_nvfp4 *q, const mpfa_rank1 *qbar,
                               const mpfa_nvfp4 *k, const mpfa_nvfp4 *vt, int B, int N, int Hq,
                               int Hkv, int d, int causal, int compensate, int T, void *o_bf16,
                               float *lse, mpfa_stream_t stream);

/* Bytes of device workspace mpfa_decode needs for kv_chunk (0 = the chunk
 * the library would choose). */
size_t mpfa_decode_workspace_size(int B, int Hq, int Hkv, int d, int Lmax, int kv_chunk);

/*
 * Split-KV decode (MpFA abstract: "adaptive parallel partitioning across
 * prefill and decode"): one new query token per sequence against a
 * quantized KV cache.
 *   q_bf16 [B][Hq][d]; k_cache codes [B][Hkv][Lmax][64] + tiled scales,
 *   v_cache codes [B][Hkv][Lmax][128]; seqlens int32 [B] (device) with
 *   0 <= seqlens[b] <= Lmax.  A length outside that range is clamped to it
 *   on the device (no read leaves the sequence's own cache rows) and
 *   MPFA_ERR_INVALID_ARG is recorded in the device status word
 *   (mpfa_get_error).  Lmax multiple of 128; B*Hkv*Lmax below 2^31 rows.
 *   The query is quantized inside the call (rank-one block = the Hq/Hkv
 *   heads of one KV head).  Keys [s*C, min(L, (s+1)*C)) form split s
 *   (C = kv_chunk, a multiple of 128; 0 = chosen by the library, returned in
 *   *used_chunk, a host int).  Splits combine by their LSE.
 *   o_bf16 [B][Hq][d]; lse [B][Hq] or NULL.  A sequence of length 0 gets
 *   O = 0 and LSE = -inf.
 *   q_quant_out (optional, may be NULL): codes [B][Hq][64], scales
 *   [B][Hq][8] row-major, tensor scale; qbar_quant_out (optional):
 *   codes [B][Hkv][T][64], scales [B][Hkv][T][8].
 *   kbar: NULL, or the mpfa_ksmooth.kbar [B][Hkv][d] the cache's keys were
 *   smoothed with: the LSE then gets q_eff . kbar / sqrt(d) added (O is the
 *   same either way).
 */
mpfa_status mpfa_decode(const void *q_bf16, const mpfa_nvfp4 *k_cache, const mpfa_fp8 *v_cache,
                        const float *kbar, const int32_t *seqlens, int B, int Hq, int Hkv, int d, int Lmax,
                        int compensate, int T, int kv_chunk, void *o_bf16, float *lse,
                        mpfa_nvfp4 *q_quant_out, mpfa_rank1 *qbar_quant_out, int *used_chunk,
                        void *workspace, size_t ws_bytes, mpfa_stream_t stream);

/*
 * Quantize-on-append into a decode KV cache (the decode workload's producer:
 * the MpFA abstract's KV operands quantized when they are written; NVFP4 K
 * and FP8 V formats per the FP4 explainer section).  The n_new new tokens of
 * every sequence are quantized with the cache's existing tensor scales
 * (*k_cache->tensor_scale, *v_cache->tensor_scale, as mpfa_quantize_qkv set
 * them when it built the cache; the scales do not change, so values beyond
 * the cache's range saturate at the largest block scale and code) and
 * written to cache rows seqlens[b] .. seqlens[b] + n_new - 1 of each
 * (b, KV head), codes and tiled scales exactly as mpfa_quantize_qkv writes a
 * row with those tensor scales.
 *   k_new_bf16, v_new_bf16 [B][n_new][Hkv][d] bf16, device.
 *   seqlens int32 [B], device: read, not advanced (pass seqlens + n_new to
 *   the next mpfa_decode).  A sequence with seqlens[b] < 0 or
 *   seqlens[b] + n_new > Lmax is left untouched and MPFA_ERR_INVALID_ARG is
 *   recorded in the device status word (mpfa_get_error); the others are
 *   appended.
 *   k_cache / v_cache: as mpfa_quantize_qkv returned them for a [B][Lmax]
 *   cache; Lmax multiple of 128, 1 <= n_new <= Lmax, B*Hkv*Lmax below 2^31
 *   rows, d = 128 (else MPFA_ERR_UNSUPPORTED).  Host-checkable errors return
 *   MPFA_ERR_INVALID_ARG with nothing enqueued.
 *   kbar: NULL, or the kbar of a cache built with key-side smoothing: the
 *   new keys are then coded as fp32(K - kbar) like the cache's own rows.
 */
mpfa_status mpfa_append_kv(const void *k_new_bf16, const void *v_new_bf16, const int32_t *seqlens,
                           int B, int n_new, int Hkv, int d, int Lmax, mpfa_nvfp4 *k_cache,
                           mpfa_fp8 *v_cache, const float *kbar, mpfa_stream_t stream);

/*
 * Paged KV pool (the MXAttention blog's section on quantized KV caches: KV
 * quantized when written, its block scales in a pool of their own; the MpFA
 * abstract's decode partitioning).  The pool holds num_pages pages of 128
 * tokens; page p holds, for every KV head h, 128 rows of codes at pool rows
 * (p * Hkv + h) * 128 .. +127:
 *   k_pool: codes [num_pages][Hkv][128][64], block scales in the 128-row
 *   tile layout over those rows (one 1 KB tile per page and head, a pool of
 *   its own), tensor scale; v_pool: codes [num_pages][Hkv][128][128],
 *   tensor scale.  mpfa_quantize_qkv(NULL, K, V, B = num_pages, Nk = 128,
 *   ...) on bf16 K, V [num_pages][128][Hkv][d] writes exactly this layout.
 *   block_table [B][max_pages] int32 (device): page of each sequence's
 *   128-token block; sequence b's token t is row t % 128 of page
 *   block_table[b][t / 128].  Entries past a sequence's length are not
 *   read.  An entry outside [0, num_pages) is reported as
 *   MPFA_ERR_INVALID_ARG in the device status word (the decode reads page 0
 *   in its place, the append writes nothing for it).
 * Key-side smoothing is not offered for a pool: its kbar is one vector per
 * sequence and KV head, while the pool's codes have no sequence.
 */

/* Split-KV decode over a paged pool: as mpfa_decode with Lmax =
 * 128 * max_pages and the cache rows looked up through block_table.
 * Workspace: mpfa_decode_workspace_size(B, Hq, Hkv, d, 128 * max_pages,
 * kv_chunk). */
mpfa_status mpfa_decode_paged(const void *q_bf16, const mpfa_nvfp4 *k_pool, const mpfa_fp8 *v_pool,
                              const int32_t *block_table, int num_pages, int max_pages,
                              const int32_t *seqlens, int B, int Hq, int Hkv, int d,
                              int compensate, int T, int kv_chunk, void *o_bf16, float *lse,
                              mpfa_nvfp4 *q_quant_out, mpfa_rank1 *qbar_quant_out,
                              int *used_chunk, void *workspace, size_t ws_bytes,
                              mpfa_stream_t stream);

/* Quantize-on-append into a paged pool: as mpfa_append_kv with Lmax =
 * 128 * max_pages and token t of sequence b written to row t % 128 of page
 * block_table[b][t / 128] (the caller assigns the pages first). */
mpfa_status mpfa_append_kv_paged(const void *k_new_bf16, const void *v_new_bf16,
                                 const int32_t *seqlens, const int32_t *block_table,
                                 int num_pages, int max_pages, int B, int n_new, int Hkv, int d,
                                 mpfa_nvfp4 *k_pool, mpfa_fp8 *v_pool, mpfa_stream_t stream);

/* Failure-path self-test: enqueues a one-thread kernel that waits, with the
 * same bounded barrier wait every kernel uses, on an on-chip barrier that
 * nothing arrives on.  After limit_ns nanoseconds (1 .. 2e9) the wait gives up
 * and records MPFA_ERR_TIMEOUT in the device status word, which
 * mpfa_get_error then reports; the CUDA context stays usable.  No fault, no
 * hang. */
mpfa_status mpfa_selftest_wait_timeout(unsigned long long limit_ns, mpfa_stream_t stream);

/* Synchronizes the stream, then returns and clears the device status word
 * (MPFA_ERR_TIMEOUT after an expired on-chip wait), or MPFA_ERR_CUDA if the
 * stream reports a CUDA error. */
mpfa_status mpfa_get_error(mpfa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MPFA_H */
