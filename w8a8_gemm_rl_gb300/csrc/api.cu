// api.cu -- the C ABI declared in include/w8a8fp8.h.  Host-side argument
// checks happen here, before anything is queued; the kernels live in
// quant.cu and gemm.cu.
#include <stdint.h>
#include <string.h>

#include "../../include/w8a8fp8.h"
#include "kernels.h"

#define W8A8_API extern "C" __attribute__((visibility("default")))

namespace w8a8 {
cudaError_t consume_device_error(int* code);
cudaError_t consume_small_gemm_error(int* code);
cudaError_t consume_pow2_gemm_error(int* code);
cudaError_t set_pow2_gemm_force_timeout(int on);
cudaError_t set_gemm_force_timeout(int on);
cudaError_t set_small_gemm_force_timeout(int on);
cudaError_t set_quant_force_timeout(int on);
cudaError_t set_attn_force_timeout(int on);
cudaError_t consume_batch_error(int* code);
cudaError_t consume_quant_error(int* code);
cudaError_t consume_attention_error(int* code);
int grouped_gemm_max_groups();
}  // namespace w8a8

namespace {

char g_last_cuda_error[256] = "";

w8a8_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return W8A8_OK;
  const char* s = cudaGetErrorString(e);
  strncpy(g_last_cuda_error, s ? s : "unknown", sizeof(g_last_cuda_error) - 1);
  g_last_cuda_error[sizeof(g_last_cuda_error) - 1] = '\0';
  return W8A8_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr int64_t kMaxDim = (int64_t)1 << 31;  // TMA coordinates and tile math are 32-bit

cudaStream_t cs(w8a8_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace

W8A8_API const char* w8a8_status_string(w8a8_status status) {
  switch (status) {
    case W8A8_OK: return "ok";
    case W8A8_ERR_NULL: return "a required pointer is NULL";
    case W8A8_ERR_SHAPE: return "invalid size or shape";
    case W8A8_ERR_ALIGN: return "pointer not aligned as required";
    case W8A8_ERR_UNSUPPORTED: return "request not supported by this build";
    case W8A8_ERR_CUDA: return "CUDA runtime error";
  }
  return "unknown status";
}

W8A8_API int w8a8_version(void) { return 200; }

W8A8_API const char* w8a8_last_cuda_error(void) { return g_last_cuda_error; }

// ------------------------------------------------------------- E4M3 codec

W8A8_API w8a8_status e4m3_encode_f32(const float* x, int64_t n, uint8_t* q, w8a8_stream_t stream) {
  if (n < 0) return W8A8_ERR_SHAPE;
  if (n == 0) return W8A8_OK;
  if (!x || !q) return W8A8_ERR_NULL;
  if (!aligned(x, 16) || !aligned(q, 16)) return W8A8_ERR_ALIGN;
  return from_cuda(w8a8::launch_e4m3_encode(x, n, q, cs(stream)));
}

W8A8_API w8a8_status e4m3_decode_f32(const uint8_t* q, int64_t n, float* x, w8a8_stream_t stream) {
  if (n < 0) return W8A8_ERR_SHAPE;
  if (n == 0) return W8A8_OK;
  if (!x || !q) return W8A8_ERR_NULL;
  if (!aligned(x, 16) || !aligned(q, 16)) return W8A8_ERR_ALIGN;
  return from_cuda(w8a8::launch_e4m3_decode(q, n, x, cs(stream)));
}

// ------------------------------------------------------------- quantizers

static w8a8_status check_quant_matrix(const uint16_t* x, int64_t rows, int64_t cols,
                                      const uint8_t* q, const float* s) {
  if (rows < 0 || cols < 0) return W8A8_ERR_SHAPE;
  if (rows == 0 || cols == 0) return W8A8_OK;
  if (!x || !q || !s) return W8A8_ERR_NULL;
  if (!aligned(x, 16) || !aligned(q, 16) || !aligned(s, 4)) return W8A8_ERR_ALIGN;
  return W8A8_OK;
}

W8A8_API w8a8_status quantize_weight_blockwise(const uint16_t* w_bf16, int64_t n, int64_t k,
                                               uint8_t* wq, float* ws, w8a8_stream_t stream) {
  w8a8_status st = check_quant_matrix(w_bf16, n, k, wq, ws);
  if (st != W8A8_OK || n == 0 || k == 0) return st;
  w8a8::WeightJob j{w_bf16, wq, ws, n, k};
  return from_cuda(w8a8::launch_weight_quant(&j, 1, cs(stream)));
}

static w8a8_status weight_batch(const w8a8_weight_desc* descs, int32_t count, bool pow2,
                                w8a8_stream_t stream) {
  if (count < 0) return W8A8_ERR_SHAPE;
  if (count == 0) return W8A8_OK;
  if (!descs) return W8A8_ERR_NULL;
  for (int32_t i = 0; i < count; ++i) {
    w8a8_status st = check_quant_matrix(descs[i].w_bf16, descs[i].n, descs[i].k, descs[i].wq,
                                        descs[i].ws);
    if (st != W8A8_OK) return st;
  }
  // Jobs go to the launcher in groups of up to 256 (host stack bound).
  constexpr int kChunk = 256;
  w8a8::WeightJob jobs[kChunk];
  int nj = 0;
  for (int32_t i = 0; i < count; ++i) {
    jobs[nj++] = w8a8::WeightJob{descs[i].w_bf16, descs[i].wq, descs[i].ws, descs[i].n, descs[i].k};
    if (nj == kChunk || i == count - 1) {
      w8a8_status st = from_cuda(w8a8::launch_weight_quant(jobs, nj, cs(stream), pow2));
      if (st != W8A8_OK) return st;
      nj = 0;
    }
  }
  return W8A8_OK;
}

W8A8_API w8a8_status quantize_weight_blockwise_batched(const w8a8_weight_desc* descs,
                                                       int32_t count, w8a8_stream_t stream) {
  return weight_batch(descs, count, false, stream);
}

W8A8_API w8a8_status quantize_weight_blockwise_batched_pow2(const w8a8_weight_desc* descs,
                                                            int32_t count, w8a8_stream_t stream) {
  return weight_batch(descs, count, true, stream);
}

W8A8_API w8a8_status quantize_weight_blockwise_pow2(const uint16_t* w_bf16, int64_t n, int64_t k,
                                                    uint8_t* wq, float* ws, w8a8_stream_t stream) {
  w8a8_status st = check_quant_matrix(w_bf16, n, k, wq, ws);
  if (st != W8A8_OK || n == 0 || k == 0) return st;
  w8a8::WeightJob j{w_bf16, wq, ws, n, k};
  return from_cuda(w8a8::launch_weight_quant(&j, 1, cs(stream), true));
}

W8A8_API w8a8_status quantize_act_per_token_group_pow2(const uint16_t* x_bf16, int64_t m,
                                                       int64_t k, uint8_t* xq, float* xs,
                                                       w8a8_stream_t stream) {
  w8a8_status st = check_quant_matrix(x_bf16, m, k, xq, xs);
  if (st != W8A8_OK || m == 0 || k == 0) return st;
  return from_cuda(w8a8::launch_act_quant(x_bf16, m, k, xq, xs, cs(stream), true));
}

W8A8_API w8a8_status quantize_act_per_token_group(const uint16_t* x_bf16, int64_t m, int64_t k,
                                                  uint8_t* xq, float* xs, w8a8_stream_t stream) {
  w8a8_status st = check_quant_matrix(x_bf16, m, k, xq, xs);
  if (st != W8A8_OK || m == 0 || k == 0) return st;
  return from_cuda(w8a8::launch_act_quant(x_bf16, m, k, xq, xs, cs(stream)));
}

W8A8_API w8a8_status quantize_act_per_token_group_gather(const uint16_t* x_bf16, int64_t rows_x,
                                                         int64_t k, const int32_t* row_idx,
                                                         int64_t total_rows, uint8_t* xq, float* xs,
                                                         w8a8_stream_t stream) {
  if (rows_x < 0 || k < 0 || total_rows < 0) return W8A8_ERR_SHAPE;
  if (total_rows == 0 || k == 0) return W8A8_OK;
  if (!row_idx || !xq || !xs || (rows_x > 0 && !x_bf16)) return W8A8_ERR_NULL;
  if (!aligned(x_bf16, 16) || !aligned(xq, 16) || !aligned(xs, 4) || !aligned(row_idx, 4))
    return W8A8_ERR_ALIGN;
  if (k % 8 != 0) return W8A8_ERR_UNSUPPORTED;
  return from_cuda(w8a8::launch_act_quant_gather(x_bf16, rows_x, k, row_idx, total_rows, xq, xs,
                                                 cs(stream)));
}

// ----------------------------------------------- dequantization and report

W8A8_API w8a8_status dequantize_blockwise(const uint8_t* q, const float* s, int64_t rows,
                                          int64_t cols, int64_t block_rows, int64_t block_cols,
                                          uint16_t* y_bf16, w8a8_stream_t stream) {
  if (rows < 0 || cols < 0 || block_rows <= 0 || block_cols <= 0) return W8A8_ERR_SHAPE;
  if (rows == 0 || cols == 0) return W8A8_OK;
  if (!q || !s || !y_bf16) return W8A8_ERR_NULL;
  if (!aligned(q, 16) || !aligned(y_bf16, 16) || !aligned(s, 4)) return W8A8_ERR_ALIGN;
  return from_cuda(w8a8::launch_dequant(q, s, rows, cols, block_rows, block_cols, y_bf16,
                                        cs(stream)));
}

W8A8_API w8a8_status quant_error_report(const uint16_t* x_bf16, const uint8_t* q, const float* s,
                                        int64_t rows, int64_t cols, int64_t scale_block_rows,
                                        int64_t scale_block_cols, int64_t report_block_rows,
                                        int64_t report_block_cols, double* stats,
                                        w8a8_stream_t stream) {
  if (rows < 0 || cols < 0 || scale_block_rows <= 0 || scale_block_cols <= 0 ||
      report_block_rows <= 0 || report_block_cols <= 0)
    return W8A8_ERR_SHAPE;
  if (rows == 0 || cols == 0) return W8A8_OK;
  if (!x_bf16 || !q || !s || !stats) return W8A8_ERR_NULL;
  if (!aligned(x_bf16, 16) || !aligned(q, 16) || !aligned(s, 4) || !aligned(stats, 8))
    return W8A8_ERR_ALIGN;
  // one warp walks a report block: keep blocks to at most 2^20 elements
  if (report_block_rows > (1 << 20) || report_block_cols > (1 << 20) ||
      report_block_rows * report_block_cols > (1 << 20))
    return W8A8_ERR_UNSUPPORTED;
  return from_cuda(w8a8::launch_quant_error(x_bf16, q, s, rows, cols, scale_block_rows,
                                            scale_block_cols, report_block_rows,
                                            report_block_cols, stats, cs(stream)));
}

template <typename Desc, typename Fill>
static w8a8_status block_batch(const Desc* descs, int32_t count, Fill fill, bool report,
                               w8a8_stream_t stream) {
  if (count < 0) return W8A8_ERR_SHAPE;
  if (count == 0) return W8A8_OK;
  if (!descs) return W8A8_ERR_NULL;
  constexpr int kChunk = 256;
  w8a8::BlockJob jobs[kChunk];
  int nj = 0;
  for (int32_t i = 0; i < count; ++i) {
    w8a8::BlockJob j{};
    w8a8_status st = fill(descs[i], j);
    if (st != W8A8_OK) return st;
    if (j.n == 0 || j.k == 0) continue;
    jobs[nj++] = j;
    if (nj == kChunk || i == count - 1) {
      st = from_cuda(report ? w8a8::launch_quant_error_batch(jobs, nj, cs(stream))
                            : w8a8::launch_dequant_batch(jobs, nj, cs(stream)));
      if (st != W8A8_OK) return st;
      nj = 0;
    }
  }
  if (nj > 0)
    return from_cuda(report ? w8a8::launch_quant_error_batch(jobs, nj, cs(stream))
                            : w8a8::launch_dequant_batch(jobs, nj, cs(stream)));
  return W8A8_OK;
}

W8A8_API w8a8_status dequantize_blockwise_batched(const w8a8_dequant_desc* descs, int32_t count,
                                                  w8a8_stream_t stream) {
  // every entry is checked before anything is queued
  for (int32_t i = 0; descs && i < count; ++i) {
    const w8a8_dequant_desc& d = descs[i];
    if (d.n < 0 || d.k < 0 || d.n >= kMaxDim || d.k >= kMaxDim) return W8A8_ERR_SHAPE;
    if (d.n == 0 || d.k == 0) continue;
    if (d.k % 16 != 0) return W8A8_ERR_SHAPE;
    if (!d.q || !d.s || !d.y_bf16) return W8A8_ERR_NULL;
    if (!aligned(d.q, 16) || !aligned(d.y_bf16, 16) || !aligned(d.s, 4)) return W8A8_ERR_ALIGN;
  }
  return block_batch(descs, count, [](const w8a8_dequant_desc& d, w8a8::BlockJob& j) {
    j.q = d.q; j.s = d.s; j.y = d.y_bf16; j.n = d.n; j.k = d.k;
    return W8A8_OK;
  }, false, stream);
}

W8A8_API w8a8_status quant_error_report_batched(const w8a8_error_desc* descs, int32_t count,
                                                w8a8_stream_t stream) {
  for (int32_t i = 0; descs && i < count; ++i) {
    const w8a8_error_desc& d = descs[i];
    if (d.n < 0 || d.k < 0 || d.n >= kMaxDim || d.k >= kMaxDim) return W8A8_ERR_SHAPE;
    if (d.n == 0 || d.k == 0) continue;
    if (d.k % 8 != 0) return W8A8_ERR_SHAPE;
    if (!d.x_bf16 || !d.q || !d.s || !d.stats) return W8A8_ERR_NULL;
    if (!aligned(d.x_bf16, 16) || !aligned(d.q, 16) || !aligned(d.s, 4) || !aligned(d.stats, 8))
      return W8A8_ERR_ALIGN;
  }
  return block_batch(descs, count, [](const w8a8_error_desc& d, w8a8::BlockJob& j) {
    j.x = d.x_bf16; j.q = d.q; j.s = d.s; j.stats = d.stats; j.n = d.n; j.k = d.k;
    return W8A8_OK;
  }, true, stream);
}

// --------------------------------------------------------------- attention

W8A8_API w8a8_status fp8_decode_attention(const uint8_t* q, const float* q_scale,
                                          const uint8_t* k_cache, const float* k_scale,
                                          const uint8_t* v_cache, const float* v_scale,
                                          const int32_t* seq_lens, int64_t batch,
                                          int64_t max_seq, int32_t num_q_heads,
                                          int32_t num_kv_heads, int32_t head_dim,
                                          float softmax_scale, uint16_t* out_bf16,
                                          w8a8_stream_t stream) {
  if (batch < 0 || max_seq < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return W8A8_ERR_SHAPE;
  if (num_q_heads % num_kv_heads != 0) return W8A8_ERR_SHAPE;
  const int32_t g = num_q_heads / num_kv_heads;
  if (head_dim != 128 || !(g == 1 || g == 2 || g % 4 == 0)) return W8A8_ERR_UNSUPPORTED;
  // over-size inputs (TMA row coordinates are 32-bit) share one status
  if (max_seq >= kMaxDim || batch >= kMaxDim) return W8A8_ERR_UNSUPPORTED;
  if (batch == 0) return W8A8_OK;
  if (batch * max_seq > kMaxDim - 1 - 32) return W8A8_ERR_UNSUPPORTED;
  if (!q || !q_scale || !k_cache || !k_scale || !v_cache || !v_scale || !seq_lens || !out_bf16)
    return W8A8_ERR_NULL;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out_bf16, 4) ||
      !aligned(seq_lens, 4) || !aligned(q_scale, 4) || !aligned(k_scale, 4) || !aligned(v_scale, 4))
    return W8A8_ERR_ALIGN;
  return from_cuda(w8a8::launch_decode_attention(q, q_scale, k_cache, k_scale, v_cache, v_scale,
                                                 seq_lens, batch, max_seq, num_q_heads,
                                                 num_kv_heads, softmax_scale, out_bf16,
                                                 cs(stream)));
}

W8A8_API w8a8_status fp8_prefill_attention(const uint8_t* q, const float* q_scale,
                                           const uint8_t* k, const float* k_scale,
                                           const uint8_t* v, const float* v_scale, int64_t batch,
                                           int64_t seq, int32_t num_q_heads, int32_t num_kv_heads,
                                           int32_t head_dim, float softmax_scale,
                                           uint16_t* out_bf16, w8a8_stream_t stream) {
  if (batch < 0 || seq < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return W8A8_ERR_SHAPE;
  if (num_q_heads % num_kv_heads != 0) return W8A8_ERR_SHAPE;
  if (head_dim != 128) return W8A8_ERR_UNSUPPORTED;
  // over-size inputs (grid dimensions; TMA row coordinates are 32-bit) share one status
  if (num_q_heads > 65535 || batch > 65535 || seq >= kMaxDim) return W8A8_ERR_UNSUPPORTED;
  if (batch == 0 || seq == 0) return W8A8_OK;
  if (batch * seq > kMaxDim - 1 - 128) return W8A8_ERR_UNSUPPORTED;
  if (!q || !q_scale || !k || !k_scale || !v || !v_scale || !out_bf16) return W8A8_ERR_NULL;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out_bf16, 16) ||
      !aligned(q_scale, 4) || !aligned(k_scale, 4) || !aligned(v_scale, 4))
    return W8A8_ERR_ALIGN;
  return from_cuda(w8a8::launch_prefill_attention(q, q_scale, k, k_scale, v, v_scale, batch,
                                                  seq, num_q_heads, num_kv_heads, softmax_scale,
                                                  out_bf16, cs(stream)));
}

// ------------------------------------------------------------------ GEMMs

static w8a8_status check_gemm_common(const uint8_t* xq, const float* xs, const uint8_t* wq,
                                     const float* ws, const uint16_t* y, int64_t n, int64_t k) {
  if (n < 0 || k < 0 || n >= kMaxDim || k >= kMaxDim) return W8A8_ERR_SHAPE;
  if (k % 16 != 0 || n % 8 != 0) return W8A8_ERR_SHAPE;
  if (!y) return W8A8_ERR_NULL;
  if (k > 0 && (!xq || !xs || !wq || !ws)) return W8A8_ERR_NULL;
  if (!aligned(y, 16)) return W8A8_ERR_ALIGN;
  if (k > 0 && (!aligned(xq, 16) || !aligned(wq, 16) || !aligned(xs, 4) || !aligned(ws, 4)))
    return W8A8_ERR_ALIGN;
  return W8A8_OK;
}

W8A8_API w8a8_status fp8_block_gemm_ex(const uint8_t* xq, const float* xs, const uint8_t* wq,
                                       const float* ws, uint16_t* y_bf16, int64_t m, int64_t n,
                                       int64_t k, uint32_t flags, w8a8_stream_t stream) {
  if (m < 0 || n < 0 || k < 0 || m >= kMaxDim) return W8A8_ERR_SHAPE;
  if ((flags & ~(uint32_t)W8A8_GEMM_STATIC_WEIGHTS) != 0) return W8A8_ERR_UNSUPPORTED;
  if (m == 0 || n == 0) return (k % 16 == 0 && n % 8 == 0) ? W8A8_OK : W8A8_ERR_SHAPE;
  w8a8_status st = check_gemm_common(xq, xs, wq, ws, y_bf16, n, k);
  if (st != W8A8_OK) return st;
  // few rows (decode-sized batches): the weight-streaming kernel
  if (w8a8::block_gemm_small_m_serves(m, n, k))
    return from_cuda(w8a8::launch_block_gemm_small_m(
        xq, xs, wq, ws, y_bf16, m, n, k, (flags & W8A8_GEMM_STATIC_WEIGHTS) != 0, cs(stream)));
  return from_cuda(w8a8::launch_block_gemm(xq, xs, wq, ws, y_bf16, m, n, k, cs(stream)));
}

W8A8_API w8a8_status fp8_block_gemm(const uint8_t* xq, const float* xs, const uint8_t* wq,
                                    const float* ws, uint16_t* y_bf16, int64_t m, int64_t n,
                                    int64_t k, w8a8_stream_t stream) {
  return fp8_block_gemm_ex(xq, xs, wq, ws, y_bf16, m, n, k, 0u, stream);
}

W8A8_API w8a8_status fp8_block_gemm_pow2(const uint8_t* xq, const float* xs, const uint8_t* wq,
                                         const float* ws, uint16_t* y_bf16, int64_t m, int64_t n,
                                         int64_t k, w8a8_stream_t stream) {
  if (m < 0 || n < 0 || k < 0 || m >= kMaxDim) return W8A8_ERR_SHAPE;
  if (m == 0 || n == 0) return (k % 16 == 0 && n % 8 == 0) ? W8A8_OK : W8A8_ERR_SHAPE;
  w8a8_status st = check_gemm_common(xq, xs, wq, ws, y_bf16, n, k);
  if (st != W8A8_OK) return st;
  return from_cuda(w8a8::launch_block_gemm_pow2(xq, xs, wq, ws, y_bf16, m, n, k, cs(stream)));
}

W8A8_API w8a8_status w8a8_linear(const uint16_t* x_bf16, int64_t m, int64_t k, const uint8_t* wq,
                                 const float* ws, int64_t n, uint16_t* y_bf16, uint8_t* xq,
                                 float* xs, uint32_t flags, w8a8_stream_t stream) {
  if (m < 0 || n < 0 || k < 0 || m >= kMaxDim) return W8A8_ERR_SHAPE;
  if ((flags & ~(uint32_t)(W8A8_GEMM_STATIC_WEIGHTS | W8A8_LINEAR_SINGLE_KERNEL)) != 0)
    return W8A8_ERR_UNSUPPORTED;
  if (k % 16 != 0 || n % 8 != 0 || n >= kMaxDim || k >= kMaxDim) return W8A8_ERR_SHAPE;
  if (m == 0 || n == 0) return W8A8_OK;
  if ((xq == nullptr) != (xs == nullptr)) return W8A8_ERR_NULL;
  if (!y_bf16 || (k > 0 && (!x_bf16 || !wq || !ws))) return W8A8_ERR_NULL;
  if (!aligned(y_bf16, 16) || (k > 0 && (!aligned(x_bf16, 16) || !aligned(wq, 16) ||
                                         !aligned(ws, 4))))
    return W8A8_ERR_ALIGN;
  if (xq && (!aligned(xq, 16) || !aligned(xs, 4))) return W8A8_ERR_ALIGN;
  const bool stat = (flags & W8A8_GEMM_STATIC_WEIGHTS) != 0;
  const bool single = (flags & W8A8_LINEAR_SINGLE_KERNEL) != 0;
  if (k > 0 && (single ? w8a8::linear_fused_possible(m, n, k) : w8a8::linear_fused_serves(m, n, k)))
    return from_cuda(w8a8::launch_linear_fused(x_bf16, wq, ws, y_bf16, xq, xs, m, n, k, stat,
                                               cs(stream)));
  // two kernels: the activation quantizer writes xq and xs, then the GEMM
  if (k > 0 && !xq) return W8A8_ERR_NULL;
  if (k == 0) return from_cuda(cudaMemsetAsync(y_bf16, 0, (size_t)(m * n * 2), cs(stream)));
  w8a8_status st = from_cuda(w8a8::launch_act_quant(x_bf16, m, k, xq, xs, cs(stream)));
  if (st != W8A8_OK) return st;
  return fp8_block_gemm_ex(xq, xs, wq, ws, y_bf16, m, n, k, flags & W8A8_GEMM_STATIC_WEIGHTS,
                           stream);
}

W8A8_API w8a8_status fp8_grouped_gemm(const uint8_t* xq, const float* xs, int64_t rows_x,
                                      const int32_t* row_idx, const int32_t* group_offsets,
                                      int32_t g, int64_t total_rows, const uint8_t* wq,
                                      const float* ws, uint16_t* y_bf16, int64_t n, int64_t k,
                                      w8a8_stream_t stream) {
  if (g < 0 || total_rows < 0 || rows_x < 0 || n < 0 || k < 0) return W8A8_ERR_SHAPE;
  if (total_rows >= kMaxDim || rows_x >= kMaxDim) return W8A8_ERR_SHAPE;
  if (g > w8a8::grouped_gemm_max_groups()) return W8A8_ERR_UNSUPPORTED;
  if (total_rows == 0 || n == 0 || g == 0)
    return (k % 16 == 0 && n % 8 == 0) ? W8A8_OK : W8A8_ERR_SHAPE;
  if (!group_offsets) return W8A8_ERR_NULL;
  if (!aligned(group_offsets, 4) || (row_idx && !aligned(row_idx, 4))) return W8A8_ERR_ALIGN;
  if (!row_idx && total_rows > rows_x) return W8A8_ERR_SHAPE;  // identity gather reads row r
  if ((int64_t)g * n >= kMaxDim) return W8A8_ERR_SHAPE;
  w8a8_status st = check_gemm_common(xq, xs, wq, ws, y_bf16, n, k);
  if (st != W8A8_OK) return st;
  if (k > 0 && rows_x == 0) return W8A8_ERR_SHAPE;
  return from_cuda(w8a8::launch_grouped_gemm(xq, xs, rows_x, row_idx, group_offsets, g,
                                             total_rows, wq, ws, y_bf16, n, k, cs(stream)));
}

// --------------------------------------------------------------- KV cache

W8A8_API w8a8_status kv_amax_quantize(const uint16_t* x_bf16, int64_t numel, uint8_t* q,
                                      float* scale, float* amax, int mode, w8a8_stream_t stream) {
  if (numel < 0) return W8A8_ERR_SHAPE;
  if (mode != W8A8_KV_AMAX_AND_QUANT && mode != W8A8_KV_AMAX_ONLY && mode != W8A8_KV_QUANT_ONLY)
    return W8A8_ERR_UNSUPPORTED;
  if (!scale) return W8A8_ERR_NULL;
  if (mode != W8A8_KV_QUANT_ONLY && !amax) return W8A8_ERR_NULL;
  if (numel > 0 && !x_bf16) return W8A8_ERR_NULL;
  if (numel > 0 && mode != W8A8_KV_AMAX_ONLY && !q) return W8A8_ERR_NULL;
  if (!aligned(scale, 4) || (amax && !aligned(amax, 4))) return W8A8_ERR_ALIGN;
  if (numel > 0 && !aligned(x_bf16, 16)) return W8A8_ERR_ALIGN;
  if (numel > 0 && mode != W8A8_KV_AMAX_ONLY && !aligned(q, 16)) return W8A8_ERR_ALIGN;
  return from_cuda(w8a8::launch_kv_amax_quantize(x_bf16, numel, q, scale, amax, mode, cs(stream)));
}

// ------------------------------------------------------------ diagnostics

W8A8_API w8a8_status w8a8_consume_device_error(int* code) {
  if (!code) return W8A8_ERR_NULL;
  int g = 0, sg = 0, pg = 0, q = 0, a = 0, bt = 0;
  w8a8_status st = from_cuda(w8a8::consume_device_error(&g));
  if (st != W8A8_OK) return st;
  st = from_cuda(w8a8::consume_small_gemm_error(&sg));
  if (st != W8A8_OK) return st;
  st = from_cuda(w8a8::consume_pow2_gemm_error(&pg));
  if (st != W8A8_OK) return st;
  if (g == 0) g = sg != 0 ? sg : pg;
  st = from_cuda(w8a8::consume_batch_error(&bt));
  if (st != W8A8_OK) return st;
  st = from_cuda(w8a8::consume_quant_error(&q));
  if (st != W8A8_OK) return st;
  st = from_cuda(w8a8::consume_attention_error(&a));
  *code = g != 0 ? g : (q != 0 ? q : (a != 0 ? a : bt));
  return st;
}

W8A8_API w8a8_status w8a8_debug_force_wait_timeout(int on) {
  const int v = on ? 1 : 0;
  w8a8_status st = from_cuda(w8a8::set_gemm_force_timeout(v));
  if (st != W8A8_OK) return st;
  st = from_cuda(w8a8::set_small_gemm_force_timeout(v));
  if (st != W8A8_OK) return st;
  st = from_cuda(w8a8::set_pow2_gemm_force_timeout(v));
  if (st != W8A8_OK) return st;
  st = from_cuda(w8a8::set_attn_force_timeout(v));
  if (st != W8A8_OK) return st;
  return from_cuda(w8a8::set_quant_force_timeout(v));
}
