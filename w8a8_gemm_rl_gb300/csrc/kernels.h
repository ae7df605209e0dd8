// kernels.h -- internal launchers behind the C ABI.  Each returns the CUDA
// error of its launch(es); argument checking is done by the callers in
// api.cu before any of these run.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace w8a8 {

// Number of SMs of the current device (cached per device).
int sm_count();

cudaError_t launch_e4m3_encode(const float* x, int64_t n, uint8_t* q, cudaStream_t st);
cudaError_t launch_e4m3_decode(const uint8_t* q, int64_t n, float* x, cudaStream_t st);

// pow2: power-of-two scales (the smallest 2^e with 448 * 2^e >= amax).
cudaError_t launch_act_quant(const uint16_t* x, int64_t m, int64_t k, uint8_t* q, float* s,
                             cudaStream_t st, bool pow2 = false);

// Output row r quantizes x row row_idx[r] (zeros when outside [0, rows_x)).
cudaError_t launch_act_quant_gather(const uint16_t* x, int64_t rows_x, int64_t k,
                                    const int32_t* row_idx, int64_t total_rows, uint8_t* q,
                                    float* s, cudaStream_t st);

struct WeightJob {
  const uint16_t* w;
  uint8_t* wq;
  float* ws;
  int64_t n, k;
};
cudaError_t launch_weight_quant(const WeightJob* jobs, int count, cudaStream_t st,
                                bool pow2 = false);

// Per-tensor KV quantization; mode as in the public header.
cudaError_t launch_kv_amax_quantize(const uint16_t* x, int64_t n, uint8_t* q, float* scale,
                                    float* amax, int mode, cudaStream_t st);

// dequant.cu: y = BF16(dec(q) * S) over br x bc scale blocks, and the
// per-report-block error statistics [max |x - x_hat|, sum e^2, sum x^2].
cudaError_t launch_dequant(const uint8_t* q, const float* s, int64_t rows, int64_t cols,
                           int64_t br, int64_t bc, uint16_t* y, cudaStream_t st);
// batch.cu: the same two over many matrices at once, 128 x 128 scale blocks
// (and, for the report, 128 x 128 report blocks).
struct BlockJob {
  const uint16_t* x;  // report: BF16 inputs [n, k]
  const uint8_t* q;   // codes [n, k]
  const float* s;     // scales [ceil(n/128), ceil(k/128)]
  uint16_t* y;        // dequantize: BF16 output [n, k]
  double* stats;      // report: [ceil(n/128), ceil(k/128), 3]
  int64_t n, k;
};
cudaError_t launch_dequant_batch(const BlockJob* jobs, int count, cudaStream_t st);
cudaError_t launch_quant_error_batch(const BlockJob* jobs, int count, cudaStream_t st);

cudaError_t launch_quant_error(const uint16_t* x, const uint8_t* q, const float* s, int64_t rows,
                               int64_t cols, int64_t sbr, int64_t sbc, int64_t rbr, int64_t rbc,
                               double* stats, cudaStream_t st);

// attention.cu: causal prefill attention over FP8 Q, K, V (head dim 128).
cudaError_t launch_prefill_attention(const uint8_t* q, const float* sq, const uint8_t* k,
                                     const float* sk, const uint8_t* v, const float* sv,
                                     int64_t batch, int64_t seq, int hq, int hkv,
                                     float softmax_scale, uint16_t* out, cudaStream_t st);

// attention.cu: decode attention over the FP8 KV cache (head dim 128).
cudaError_t launch_decode_attention(const uint8_t* q, const float* sq, const uint8_t* k,
                                    const float* sk, const uint8_t* v, const float* sv,
                                    const int32_t* lens, int64_t batch, int64_t smax, int hq,
                                    int hkv, float softmax_scale, uint16_t* out,
                                    cudaStream_t st);

cudaError_t launch_block_gemm(const uint8_t* xq, const float* xs, const uint8_t* wq,
                              const float* ws, uint16_t* y, int64_t m, int64_t n, int64_t k,
                              cudaStream_t st);

// The same GEMM for power-of-two scales on the block-scaled MMA
// (gemm_pow2.cu): the scales become UE8M0 factors of the tensor cores'
// products and the accumulator spans all of K.
cudaError_t launch_block_gemm_pow2(const uint8_t* xq, const float* xs, const uint8_t* wq,
                                   const float* ws, uint16_t* y, int64_t m, int64_t n, int64_t k,
                                   cudaStream_t st);

// The same GEMM for m <= 256 rows (gemm_small_m.cu): weights streamed once
// by every SM, K split over a thread-block cluster.  static_weights: wq and
// ws may be read while the previous kernel on the stream is still running.
cudaError_t launch_block_gemm_small_m(const uint8_t* xq, const float* xs, const uint8_t* wq,
                                      const float* ws, uint16_t* y, int64_t m, int64_t n,
                                      int64_t k, bool static_weights, cudaStream_t st);
// The same kernel fed with BF16 activations x [m, k]: the 1 x 128 activation
// quantization happens inside it (bit-exact with launch_act_quant); its codes
// and scales are also written to xq_out / xs_out when those are not NULL.
cudaError_t launch_linear_fused(const uint16_t* x, const uint8_t* wq, const float* ws,
                                uint16_t* y, uint8_t* xq_out, float* xs_out, int64_t m,
                                int64_t n, int64_t k, bool static_weights, cudaStream_t st);
// Whether that kernel is the faster choice (narrow outputs), and whether it
// can run at all (m <= 128, k <= 32768).
bool linear_fused_serves(int64_t m, int64_t n, int64_t k);
bool linear_fused_possible(int64_t m, int64_t n, int64_t k);

// Whether the kernel above is the one for an m x n x k product (m <= 256,
// k <= 32768, and past m = 128 only where the general kernel has few tiles).
bool block_gemm_small_m_serves(int64_t m, int64_t n, int64_t k);

cudaError_t launch_grouped_gemm(const uint8_t* xq, const float* xs, int64_t rows_x,
                                const int32_t* row_idx, const int32_t* group_offsets, int32_t g,
                                int64_t total_rows, const uint8_t* wq, const float* ws,
                                uint16_t* y, int64_t n, int64_t k, cudaStream_t st);

}  // namespace w8a8
