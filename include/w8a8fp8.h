/*
 * w8a8fp8.h -- C ABI of the GB300 (sm_103a) FP8 W8A8 hot path.
 *
 * What the calls compute is fixed by these pages (title, then section/table):
 *   [FP8-RL] "FP8-RL: A Practical and Stable Low-Precision Stack for LLM
 *            Reinforcement Learning" (dcwnkz.com write-up), section 1 "dynamic
 *            weight sync" (E4M3 over [-448, 448]; weights re-quantized in
 *            128x128 blocks after every trainer update; activations quantized
 *            dynamically) and section 4 "KV cache" (per-step scale
 *            recalibration); the arXiv abstract on shd-paper.top, items (i)
 *            and (ii).
 *   [UFP8]   "Unified FP8: Moving Beyond Mixed Precision for Stable and
 *            Accelerated MoE RL" (papercache.org notes), quick-read section:
 *            S = max|X| / V_max and Q(x) = round(x / S); section "FP8 scale
 *            choice": FP32 scales rather than E8M0.
 *   [NeMo]   NeMo RL FP8 blog (nvidia.csdn.net), Table 1 (weights [128,128],
 *            input activations [1,128], FP32 block scales) and Table 3
 *            (per-tensor FP32 scales for QKV activations and the KV cache).
 *
 * Conventions for every call:
 *   - Pointers are DEVICE pointers unless marked "host".  The library never
 *     allocates, frees or retains memory: every buffer belongs to the caller
 *     and must stay valid until the work queued on `stream` has finished.
 *   - Matrices are contiguous and row-major.  BF16 data is passed as raw
 *     16-bit words (uint16_t), E4M3 codes as bytes (uint8_t).
 *   - Every call is asynchronous on `stream` (0 = the legacy default stream)
 *     and never synchronizes the host.
 *   - Arguments are validated on the host before anything is queued; a
 *     failed check returns a nonzero status and queues nothing.  A launch
 *     failure is reported as W8A8_ERR_CUDA (from cudaGetLastError).
 *   - Non-finite inputs are outside the contract.
 *   - Quantization: S = RN32(amax / 448) (S = 1 when amax = 0), and
 *     q = E4M3(RN32(x / S)) with round-to-nearest-even and saturation to
 *     +-448; signed zero keeps its sign.  Results are bit-exact with this
 *     definition.
 */
#ifndef W8A8FP8_H
#define W8A8FP8_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA runtime stream handle (same type as cudaStream_t). */
typedef struct CUstream_st *w8a8_stream_t;

typedef enum {
    W8A8_OK = 0,
    W8A8_ERR_NULL = 1,        /* a required pointer is NULL */
    W8A8_ERR_SHAPE = 2,       /* a size is negative or breaks a stated rule */
    W8A8_ERR_ALIGN = 3,       /* a pointer is not aligned as stated */
    W8A8_ERR_UNSUPPORTED = 4, /* valid request the library does not serve */
    W8A8_ERR_CUDA = 5         /* the CUDA runtime reported an error */
} w8a8_status;

/* Static, NUL-terminated description of a status code (host). */
const char *w8a8_status_string(w8a8_status status);

/* Library version as major*10000 + minor*100 + patch. */
int w8a8_version(void);

/* Text of the last CUDA runtime error seen by any call in this process
 * (host, static storage; "" if none).  Diagnostic only. */
const char *w8a8_last_cuda_error(void);

/* Reads and clears the device-side error code that a kernel sets when a
 * bounded wait inside it gives up (0 = none; nonzero identifies the wait:
 * 1..10 the GEMMs of more than 256 rows and the grouped GEMM, 31..37 the
 * GEMM of at most 256 rows, 51..58 the power-of-two GEMM (59: a scale it
 * cannot hold), 11..13 the weight quantizer, 21..23 the decode and prefill
 * attention,
 * 41..43 the batched dequantizer and error report).  When several are set,
 * the GEMMs' code is reported first, then the quantizer's, and all are
 * cleared.  Such a kernel stops early
 * and leaves its output incomplete.  Synchronous: blocks until the device
 * has finished prior work on the legacy stream. */
w8a8_status w8a8_consume_device_error(int *code);

/* Test hook for the abort paths: while `on` is nonzero, every later launch
 * of the GEMMs, of the weight quantizer and of the attention kernels
 * behaves as if one of its bounded waits had run out of time at once (the
 * GEMMs' MMA issuer before its first slab: code 5, 35 for m <= 256, 55 for
 * fp8_block_gemm_pow2; the weight quantizer's consumers on their first
 * block: code 13; each warp of fp8_decode_attention on its first chunk:
 * code 21; the MMA issuer of fp8_prefill_attention before its first MMA:
 * code 23).  The kernel then stops as it would after a
 * real time-out -- the other roles stop, copies and MMAs in flight are
 * drained, tensor memory is freed -- and its output is incomplete.  Nothing
 * faults or hangs.  Synchronous; call with 0 to return to normal. */
w8a8_status w8a8_debug_force_wait_timeout(int on);

/* ------------------------------------------------------------------------
 * E4M3 codec ([UFP8] "FP8 data formats", referring to the OCP FP8 spec;
 * [FP8-RL] section 1 range +-448).
 *
 * e4m3_encode_f32: q[i] = E4M3(x[i]), round to nearest even, |x| > 448
 *   saturates to +-448.  x: n floats; q: n bytes.
 * e4m3_decode_f32: x[i] = exact value of code q[i] (0x7F/0xFF give NaN).
 * Both: n >= 0; x and q 16-byte aligned.
 * ---------------------------------------------------------------------- */
w8a8_status e4m3_encode_f32(const float *x, int64_t n, uint8_t *q,
                            w8a8_stream_t stream);
w8a8_status e4m3_decode_f32(const uint8_t *q, int64_t n, float *x,
                            w8a8_stream_t stream);

/* ------------------------------------------------------------------------
 * quantize_weight_blockwise -- [FP8-RL] section 1 (128x128 blocks, each with
 * its own scale); [NeMo] Table 1 row "weights"; [UFP8] scale and
 * quantization equations.
 *
 *   w_bf16  [n, k] BF16 weights.
 *   wq      [n, k] E4M3 codes (out).
 *   ws      [ceil(n/128), ceil(k/128)] FP32 block scales (out), row-major.
 * Edge blocks that overhang the matrix use their in-bounds elements only.
 * n, k >= 0.  w_bf16 and wq 16-byte aligned, ws 4-byte aligned.
 * ---------------------------------------------------------------------- */
w8a8_status quantize_weight_blockwise(const uint16_t *w_bf16, int64_t n,
                                      int64_t k, uint8_t *wq, float *ws,
                                      w8a8_stream_t stream);

/* One matrix of a batched weight quantization (all pointers device). */
typedef struct {
    const uint16_t *w_bf16; /* [n, k] */
    uint8_t *wq;            /* [n, k] */
    float *ws;              /* [ceil(n/128), ceil(k/128)] */
    int64_t n;
    int64_t k;
} w8a8_weight_desc;

/* quantize_weight_blockwise over `count` matrices in as few launches as the
 * kernel-parameter space allows (the whole-model weight sync of [FP8-RL]
 * section 1 is one call).  descs is a HOST array, read before the call
 * returns.  Each entry obeys the rules of quantize_weight_blockwise.
 * count >= 0. */
w8a8_status quantize_weight_blockwise_batched(const w8a8_weight_desc *descs,
                                              int32_t count,
                                              w8a8_stream_t stream);

/* ------------------------------------------------------------------------
 * quantize_act_per_token_group -- [NeMo] Table 1 row "input activations"
 * ([1,128] groups, FP32 scales); [UFP8] quick-read section (per-token
 * activation quantization) and its scale/quantization equations; [FP8-RL]
 * section 1 (activations quantized dynamically at inference).
 *
 *   x_bf16  [m, k] BF16 activations.
 *   xq      [m, k] E4M3 codes (out).
 *   xs      [m, ceil(k/128)] FP32 group scales (out), row-major.
 * The last group of a row may be shorter than 128.  m, k >= 0.  x_bf16 and
 * xq 16-byte aligned, xs 4-byte aligned.
 * ---------------------------------------------------------------------- */
w8a8_status quantize_act_per_token_group(const uint16_t *x_bf16, int64_t m,
                                         int64_t k, uint8_t *xq, float *xs,
                                         w8a8_stream_t stream);

/* ------------------------------------------------------------------------
 * quantize_weight_blockwise_pow2, quantize_act_per_token_group_pow2 -- the
 * same quantizers with power-of-two scales, the "Power-of-2 Scaling Factor"
 * recipe option of the [NeMo] blog (section on recipe variants; [UFP8]
 * "FP8 scale choice" weighs it against FP32 scales):
 *
 *   S = the smallest 2^e with 448 * 2^e >= amax   (S = 1 when amax == 0)
 *   q = E4M3_RNE(x / S)                           (x / S is exact)
 *
 * so no code saturates and every scale is a UE8M0-representable power of
 * two.  Arguments, layouts and rules as the FP32-scale versions (the
 * batched one as quantize_weight_blockwise_batched); the GEMMs take these
 * scales unchanged.
 * ---------------------------------------------------------------------- */
w8a8_status quantize_weight_blockwise_pow2(const uint16_t *w_bf16, int64_t n,
                                           int64_t k, uint8_t *wq, float *ws,
                                           w8a8_stream_t stream);
w8a8_status quantize_act_per_token_group_pow2(const uint16_t *x_bf16, int64_t m,
                                              int64_t k, uint8_t *xq, float *xs,
                                              w8a8_stream_t stream);
w8a8_status quantize_weight_blockwise_batched_pow2(const w8a8_weight_desc *descs,
                                                   int32_t count,
                                                   w8a8_stream_t stream);

/* ------------------------------------------------------------------------
 * quantize_act_per_token_group_gather -- the activation quantizer above
 * applied to the routed rows of an MoE layer ([FP8-RL] section 1 expert
 * layers, [NeMo] Table 1 [1,128] groups): output row r is the per-token
 * group quantization of x row row_idx[r].  Quantization works per row, so
 * this equals quantizing x and then gathering its rows; the routed, expert-
 * sorted copy lets fp8_grouped_gemm read contiguous rows (row_idx = NULL).
 *
 *   x_bf16   [rows_x, k] BF16 activations (may be NULL when rows_x == 0).
 *   row_idx  [total_rows] int32 source row of each routed row; an index
 *            outside [0, rows_x) gives a zero row (codes 0, scales 1).
 *   xq       [total_rows, k] E4M3 codes (out).
 *   xs       [total_rows, ceil(k/128)] FP32 group scales (out), row-major.
 * Rules: rows_x, k, total_rows >= 0; k % 8 == 0 (else W8A8_ERR_UNSUPPORTED);
 * x_bf16 and xq 16-byte aligned; xs and row_idx 4-byte aligned.
 * ---------------------------------------------------------------------- */
w8a8_status quantize_act_per_token_group_gather(const uint16_t *x_bf16,
                                                int64_t rows_x, int64_t k,
                                                const int32_t *row_idx,
                                                int64_t total_rows, uint8_t *xq,
                                                float *xs, w8a8_stream_t stream);

/* ------------------------------------------------------------------------
 * dequantize_blockwise -- the inverse of the quantizers, "fake quant" in
 * the [UFP8] notes' error analysis (quantize-dequantize against the real
 * FP8 path):
 *
 *   y[r,c] = BF16_RN( RN32( dec(q[r,c]) * s[r/block_rows, c/block_cols] ) )
 *
 *   q       [rows, cols] E4M3 codes.
 *   s       [ceil(rows/block_rows), ceil(cols/block_cols)] FP32 scales,
 *           row-major: 128 x 128 for weights, 1 x 128 for activations,
 *           rows x cols (one scale) for a per-tensor KV cache.
 *   y_bf16  [rows, cols] BF16 (out).
 * Rules: rows, cols >= 0; block sizes > 0; q and y_bf16 16-byte aligned, s
 * 4-byte aligned.
 * ---------------------------------------------------------------------- */
w8a8_status dequantize_blockwise(const uint8_t *q, const float *s, int64_t rows,
                                 int64_t cols, int64_t block_rows,
                                 int64_t block_cols, uint16_t *y_bf16,
                                 w8a8_stream_t stream);

/* ------------------------------------------------------------------------
 * quant_error_report -- the quantization error the [UFP8] notes attribute
 * the train/rollout mismatch to, measured per report block: with
 * x_hat = RN32(dec(q) * s) as above,
 *
 *   stats[b] = { max |x - x_hat|,  sum (x - x_hat)^2,  sum x^2 }   (FP64)
 *
 * over report block b of report_block_rows x report_block_cols elements
 * (row-major block index, ragged edge blocks hold the in-bounds elements).
 * The quantization blocks (scale_block_rows x scale_block_cols) and the
 * report blocks are independent: a per-tensor KV scale can be reported per
 * row, for instance.  SQNR of any union of blocks is
 * 10 log10(sum x^2 / sum e^2).
 *   stats [ceil(rows/rbr), ceil(cols/rbc), 3] doubles (out).
 * Accuracy: the maximum is exact for pairs the quantizers produce (x_hat
 * within a factor 2 of x); the sums are within 1e-5 relative of FP64
 * (binary32 squares summed over 8 elements), for |x| and |e| in
 * [2^-63, 2^63].
 * Rules: as dequantize_blockwise, x_bf16 16-byte aligned, stats 8-byte
 * aligned; a report block holds at most 2^20 elements, else
 * W8A8_ERR_UNSUPPORTED.
 * ---------------------------------------------------------------------- */
w8a8_status quant_error_report(const uint16_t *x_bf16, const uint8_t *q,
                               const float *s, int64_t rows, int64_t cols,
                               int64_t scale_block_rows, int64_t scale_block_cols,
                               int64_t report_block_rows,
                               int64_t report_block_cols, double *stats,
                               w8a8_stream_t stream);

/* dequantize_blockwise and quant_error_report over `count` weight matrices
 * with 128 x 128 scale blocks (and, for the report, 128 x 128 report
 * blocks) in as few launches as the kernel-parameter space allows: every
 * matrix of a whole-model weight sync in one call each.  The same
 * arithmetic as the one-matrix calls: y bit-identical; the report's maxima
 * identical and its sums within a few binary32 roundings (the order of
 * summation differs).  descs is a HOST array, read before the call
 * returns.  Rules: n, k >= 0 and k % 16 == 0 for the dequantizer, k % 8 == 0
 * for the report; q, y_bf16 and x_bf16 16-byte aligned, s 4-byte aligned,
 * stats 8-byte aligned; count >= 0.  A bounded wait that gives up records
 * code 41..43 (w8a8_consume_device_error). */
typedef struct {
    const uint8_t *q;       /* [n, k] E4M3 codes */
    const float *s;         /* [ceil(n/128), ceil(k/128)] scales */
    uint16_t *y_bf16;       /* [n, k] (out) */
    int64_t n;
    int64_t k;
} w8a8_dequant_desc;
w8a8_status dequantize_blockwise_batched(const w8a8_dequant_desc *descs,
                                         int32_t count, w8a8_stream_t stream);

typedef struct {
    const uint16_t *x_bf16; /* [n, k] the BF16 matrix that was quantized */
    const uint8_t *q;       /* [n, k] its E4M3 codes */
    const float *s;         /* [ceil(n/128), ceil(k/128)] its scales */
    double *stats;          /* [ceil(n/128), ceil(k/128), 3] (out) */
    int64_t n;
    int64_t k;
} w8a8_error_desc;
w8a8_status quant_error_report_batched(const w8a8_error_desc *descs,
                                       int32_t count, w8a8_stream_t stream);

/* ------------------------------------------------------------------------
 * fp8_decode_attention -- attention of one new query token per sequence
 * over the FP8 KV cache, with the per-tensor FP32 scales of [NeMo] Table 3
 * (QKV activations and the stored KV cache) and [FP8-RL] section 4:
 *
 *   score_t = softmax_scale * sq * sk * sum_d dec(q[b,h,d]) dec(k[b,t,kh,d])
 *   out[b,h,d] = BF16( sv * sum_{t < len_b} softmax_t(score) dec(v[b,t,kh,d]) )
 *
 * with kh = h / (num_q_heads / num_kv_heads) (grouped-query heads).
 *   q        [batch, num_q_heads, head_dim] E4M3; q_scale one FP32 (device).
 *   k_cache, v_cache [batch, max_seq, num_kv_heads, head_dim] E4M3, as
 *            written by kv_amax_quantize; k_scale, v_scale one FP32 each.
 *   seq_lens [batch] int32 (device), each in [0, max_seq]; an empty
 *            sequence gives zeros.
 *   out_bf16 [batch, num_q_heads, head_dim] (out).
 * Accuracy: FP32 accumulation throughout (the E4M3 products of Q K^T are
 * exact; the softmax weights enter P V as two f16 parts, about 22 bits)
 * with an online softmax whose exponentials use the hardware's approximate
 * base-2 exponential (ex2.approx.ftz.f32, flushing subnormal results to
 * zero); |out - exact| <= 1e-3 * sv * sum_t p_t |dec(v_t,d)| + half a BF16
 * ulp + 2^-39 * sv * sum_t |dec(v_t,d)| (the tests also hold 2^-14 of the
 * first sum, which covers the error of the approximate exponential; the
 * last term is the weights below 2^-39 of the largest, which f16 cannot
 * hold and which are left out).
 * Lengths are read on the device and clamped to [0, max_seq].
 * Rules: head_dim == 128 and num_q_heads / num_kv_heads in {1, 2} or a
 * multiple of 4 (else W8A8_ERR_UNSUPPORTED); batch, max_seq and
 * batch * max_seq below 2^31 - 32 (TMA row coordinates; every over-size
 * input gives W8A8_ERR_UNSUPPORTED); q and the
 * caches 16-byte aligned, the rest 4-byte aligned.  Each (sequence, KV
 * head) slice of the cache is read once per 8 query heads (4 when the
 * group is not a multiple of 8), through TMA tile loads of 32 tokens; the
 * products run on the tensor cores (E4M3 codes for Q K^T, f16 for P V with
 * the weights split in two f16 parts).
 * ---------------------------------------------------------------------- */
w8a8_status fp8_decode_attention(const uint8_t *q, const float *q_scale,
                                 const uint8_t *k_cache, const float *k_scale,
                                 const uint8_t *v_cache, const float *v_scale,
                                 const int32_t *seq_lens, int64_t batch,
                                 int64_t max_seq, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_dim,
                                 float softmax_scale, uint16_t *out_bf16,
                                 w8a8_stream_t stream);

/* ------------------------------------------------------------------------
 * fp8_prefill_attention -- causal attention of a prompt's tokens over FP8
 * Q, K and V, with the per-tensor FP32 scales of [NeMo] Table 3:
 *
 *   score_j = softmax_scale * sq * sk * sum_d dec(q[b,i,h,d]) dec(k[b,j,kh,d])
 *   out[b,i,h,d] = BF16( sv * sum_{j <= i} softmax_j(score) dec(v[b,j,kh,d]) )
 *
 * query token i of sequence b reading tokens 0..i of the same sequence, with
 * kh = h / (num_q_heads / num_kv_heads) (grouped-query heads).
 *   q        [batch, seq, num_q_heads, head_dim] E4M3; q_scale one FP32 (device).
 *   k, v     [batch, seq, num_kv_heads, head_dim] E4M3 (the KV cache's
 *            layout, as written by kv_amax_quantize); k_scale, v_scale one
 *            FP32 each (device).
 *   out_bf16 [batch, seq, num_q_heads, head_dim] (out).
 * Accuracy: as fp8_decode_attention (FP32 accumulation, exact E4M3
 * products for Q K^T, the weights in two f16 parts for P V, the hardware's
 * approximate base-2 exponential): |out - exact| <= 1e-3 * sv * sum_j p_j
 * |dec(v_j,d)| + half a BF16 ulp + 2^-39 * sv * sum_{j <= i} |dec(v_j,d)|
 * (weights below 2^-39 of the row's largest, which f16 cannot hold, are
 * left out).
 * Rules: head_dim == 128 (else W8A8_ERR_UNSUPPORTED); num_q_heads and
 * batch at most 65535, seq and batch * seq below 2^31 - 128 (grid and TMA
 * coordinate limits; over-size inputs give W8A8_ERR_UNSUPPORTED); q, k, v
 * and out_bf16 16-byte aligned, the scales 4-byte aligned.  One persistent
 * CTA per SM takes blocks of 128 query tokens of one (sequence, query head)
 * in turn and streams the keys and values up to each block in chunks of
 * 128 tokens (TMA tiles); both products run on the tcgen05 tensor cores
 * with the accumulators in tensor memory (E4M3 for Q K^T, f16 for P V).  A
 * bounded wait that gives up records device error 23.
 * ---------------------------------------------------------------------- */
w8a8_status fp8_prefill_attention(const uint8_t *q, const float *q_scale,
                                  const uint8_t *k, const float *k_scale,
                                  const uint8_t *v, const float *v_scale, int64_t batch,
                                  int64_t seq, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, float softmax_scale, uint16_t *out_bf16,
                                  w8a8_stream_t stream);

/* ------------------------------------------------------------------------
 * fp8_block_gemm -- the W8A8 linear of [FP8-RL] section 1 / arXiv abstract
 * item (i) with the [NeMo] Table 1 granularities:
 *
 *   y[i,j] = BF16( sum_kb xs[i,kb] * ws[j/128,kb]
 *                        * sum_{k in slab kb} dec(xq[i,k]) * dec(wq[j,k]) )
 *
 * with FP32 accumulation and the scales applied once per 128-wide K slab.
 *   xq [m, k], xs [m, ceil(k/128)]     (from quantize_act_per_token_group)
 *   wq [n, k], ws [ceil(n/128), ceil(k/128)] (from quantize_weight_blockwise)
 *   y_bf16 [m, n] (out), round to nearest even.
 * Rules: m, n >= 0; k >= 0 and k % 16 == 0; n % 8 == 0; xq, wq, y_bf16
 * 16-byte aligned; xs, ws 4-byte aligned.  k == 0 writes zeros.
 * Accuracy: |y - exact| <= 1e-3 * sum_k |a_ik b_jk| + half a BF16 ulp.
 * ---------------------------------------------------------------------- */
w8a8_status fp8_block_gemm(const uint8_t *xq, const float *xs,
                           const uint8_t *wq, const float *ws,
                           uint16_t *y_bf16, int64_t m, int64_t n, int64_t k,
                           w8a8_stream_t stream);

/* ------------------------------------------------------------------------
 * fp8_block_gemm_ex -- fp8_block_gemm with option flags; the same result
 * (bit for bit) for every flag value.  flags = 0 is fp8_block_gemm.
 *
 *   W8A8_GEMM_STATIC_WEIGHTS: the caller states that wq and ws are not
 *     written by the kernel enqueued just before this call on `stream`
 *     (nor by anything that kernel may still overlap) -- as holds for a
 *     rollout's decode linears, whose weights change only at weight sync.
 *     For m <= 256 the GEMM then starts reading its first weight slabs
 *     while that previous kernel is finishing (programmatic dependent
 *     launch); activations and scales of the tokens are read only after it
 *     has completed.  Ignored for m > 256.
 * Other flag bits give W8A8_ERR_UNSUPPORTED.
 *
 * Every call with m <= 256 (and k <= 32768) is launched as a programmatic
 * dependent of the previous kernel on the stream: its prologue (barrier
 * set-up, tensor-memory allocation) may overlap that kernel's end, and, with
 * the flag, so may its first weight reads.
 * ---------------------------------------------------------------------- */
#define W8A8_GEMM_STATIC_WEIGHTS 1u
w8a8_status fp8_block_gemm_ex(const uint8_t *xq, const float *xs,
                              const uint8_t *wq, const float *ws,
                              uint16_t *y_bf16, int64_t m, int64_t n,
                              int64_t k, uint32_t flags, w8a8_stream_t stream);

/* ------------------------------------------------------------------------
 * fp8_block_gemm_pow2 -- fp8_block_gemm for power-of-two scales (the
 * "Power-of-2 Scaling Factor" recipe option of the [NeMo] blog, as made by
 * the *_pow2 quantizers), with the scaling done inside the tensor cores:
 * every scale is a UE8M0 factor of a block-scaled MMA ([UFP8] "FP8 scale
 * choice" names E8M0 as the alternative to FP32 scales), and the FP32
 * accumulator spans the whole K extent instead of being promoted through
 * registers once per 128-wide slab.
 *
 *   y[i,j] = BF16( sum_kb xs[i,kb] * ws[j/128,kb]
 *                        * sum_{k in slab kb} dec(xq[i,k]) * dec(wq[j,k]) )
 *
 * Arguments, layouts, rules and accuracy bound as fp8_block_gemm, plus:
 * every xs and ws value must be +2^e with -127 <= e <= 127.  The *_pow2
 * quantizers give such scales except for a block whose amax is below
 * 448 * 2^-127 (nonzero); a scale outside the rule makes that tile's rows
 * of y_bf16 wrong and records device error 59 (w8a8_consume_device_error),
 * nothing else.  Results differ from fp8_block_gemm's only in rounding
 * order (both within the bound).  Any m is served; for m <= 256 the weight
 * stream bounds both GEMMs and fp8_block_gemm is the faster.
 * ---------------------------------------------------------------------- */
w8a8_status fp8_block_gemm_pow2(const uint8_t *xq, const float *xs,
                                const uint8_t *wq, const float *ws,
                                uint16_t *y_bf16, int64_t m, int64_t n,
                                int64_t k, w8a8_stream_t stream);

/* ------------------------------------------------------------------------
 * w8a8_linear -- the whole W8A8 linear of [FP8-RL] section 1 from BF16
 * activations: 1 x 128 per-token activation quantization ([NeMo] Table 1,
 * as quantize_act_per_token_group) followed by fp8_block_gemm.
 *
 *   x_bf16 [m, k] BF16 activations; wq [n, k], ws [ceil(n/128),
 *   ceil(k/128)] the quantized weights; y_bf16 [m, n] (out).
 *   xq [m, k], xs [m, ceil(k/128)]: the activations' codes and scales (out),
 *   bit-exact with quantize_act_per_token_group.  Both NULL, or both not.
 *   flags: W8A8_GEMM_STATIC_WEIGHTS (as fp8_block_gemm_ex) and/or
 *   W8A8_LINEAR_SINGLE_KERNEL.
 *
 * Two ways to run it:
 *  - one kernel (m <= 128, k <= 32768): the GEMM's token loaders read the
 *    BF16 rows and quantize them on the way into shared memory, so the codes
 *    make no round trip through HBM and xq, xs may be NULL.  Every 128
 *    output columns repeat that quantization, so it is chosen by default
 *    only for n <= 1024; W8A8_LINEAR_SINGLE_KERNEL asks for it wherever it
 *    can run.
 *  - otherwise the activation quantizer, then the GEMM (xq and xs are
 *    required: the library allocates nothing).  Both are launched as
 *    programmatic dependents, so the GEMM's set-up (and, with static
 *    weights, its first weight reads) overlaps the quantizer.
 * y is within fp8_block_gemm's accuracy of the exact product of the codes.
 * Rules: as fp8_block_gemm (k % 16 == 0, n % 8 == 0); x_bf16, wq, y_bf16
 * and xq 16-byte aligned, ws and xs 4-byte aligned; xq and xs both NULL or
 * both not, and not NULL for the two-kernel way (else W8A8_ERR_NULL).
 * m == 0 or n == 0 does nothing; k == 0 writes zeros to y.
 * ---------------------------------------------------------------------- */
#define W8A8_LINEAR_SINGLE_KERNEL 2u
w8a8_status w8a8_linear(const uint16_t *x_bf16, int64_t m, int64_t k,
                        const uint8_t *wq, const float *ws, int64_t n,
                        uint16_t *y_bf16, uint8_t *xq, float *xs,
                        uint32_t flags, w8a8_stream_t stream);

/* ------------------------------------------------------------------------
 * fp8_grouped_gemm -- the MoE expert layers of [FP8-RL] section 1 (expert
 * layers are quantized) and section 3 (30B-A3B MoE): fp8_block_gemm per
 * expert over that expert's routed rows.
 *
 *   xq [rows_x, k], xs [rows_x, ceil(k/128)]  quantized activations.
 *   row_idx [total_rows] int32 source row of each routed row, or NULL for
 *           the identity (row r reads xq row r).
 *   group_offsets [g+1] int32, non-decreasing, group_offsets[0] = 0 and
 *           group_offsets[g] = total_rows: rows [off[e], off[e+1]) use
 *           expert e.  (device)
 *   total_rows   host copy of group_offsets[g].
 *   wq [g, n, k], ws [g, ceil(n/128), ceil(k/128)] expert weights.
 *   y_bf16 [total_rows, n] (out), in routed-row order.
 * Rules as fp8_block_gemm, plus g >= 0 and total_rows >= 0.  Device data is
 * range-checked in the kernel: a row_idx outside [0, rows_x) yields a zero
 * output row, and offsets are clamped to [0, total_rows].
 * ---------------------------------------------------------------------- */
w8a8_status fp8_grouped_gemm(const uint8_t *xq, const float *xs,
                             int64_t rows_x, const int32_t *row_idx,
                             const int32_t *group_offsets, int32_t g,
                             int64_t total_rows, const uint8_t *wq,
                             const float *ws, uint16_t *y_bf16, int64_t n,
                             int64_t k, w8a8_stream_t stream);

/* ------------------------------------------------------------------------
 * kv_amax_quantize -- the FP8 KV cache of [NeMo] "FP8 for KV cache and
 * attention" with Table 3 (per-tensor FP32 scale for the stored KV cache)
 * and the per-step recalibration of [FP8-RL] section 4 / arXiv abstract item
 * (ii): amax over the whole tensor, S = amax / 448, every element coded with
 * S.  Call once for K and once for V.
 *
 *   x_bf16 [numel] BF16 tensor (any shape, contiguous).
 *   q      [numel] E4M3 codes (out; unused in AMAX_ONLY).
 *   scale  1 float: out in AMAX_AND_QUANT and AMAX_ONLY, in for QUANT_ONLY.
 *   amax   1 float: out in AMAX_AND_QUANT and AMAX_ONLY (may be NULL in
 *          QUANT_ONLY).
 *   mode   W8A8_KV_AMAX_AND_QUANT, W8A8_KV_AMAX_ONLY or W8A8_KV_QUANT_ONLY.
 * numel >= 0 (numel == 0 gives amax 0 and scale 1).  x_bf16 and q 16-byte
 * aligned; scale and amax 4-byte aligned.  In QUANT_ONLY a stale scale may
 * push |x/S| past 448; those elements saturate.
 * ---------------------------------------------------------------------- */
enum {
    W8A8_KV_AMAX_AND_QUANT = 0,
    W8A8_KV_AMAX_ONLY = 1,
    W8A8_KV_QUANT_ONLY = 2
};
w8a8_status kv_amax_quantize(const uint16_t *x_bf16, int64_t numel,
                             uint8_t *q, float *scale, float *amax, int mode,
                             w8a8_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* W8A8FP8_H */
