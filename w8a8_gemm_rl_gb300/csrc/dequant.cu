// dequant.cu -- the inverse of the quantizers and the error report the pages
// build on it ("Unified FP8" notes, the fake-quant versus real-quant
// experiments behind the quantization-error analysis):
//
//   x_hat[r, c] = dec(q[r, c]) * S[r / br, c / bc]    one binary32 multiply
//   y[r, c]     = BF16_RN(x_hat[r, c])                 (dequantize_blockwise)
//
// and, per report block of the matrix, max |x - x_hat|, sum (x - x_hat)^2
// and sum x^2 (quant_error_report).  Both stream their inputs once: HBM-bound.
#include "common.cuh"
#include "kernels.h"

namespace w8a8 {

namespace {

inline unsigned grid_for(int64_t work, int64_t per_cta) {
  const int64_t need = (work + per_cta - 1) / per_cta;
  const int64_t cap = (int64_t)sm_count() * 8;
  return (unsigned)(need < 1 ? 1 : (need < cap ? need : cap));
}

}  // namespace

__device__ __forceinline__ void dequant_store16(uint4 w, float S, uint16_t* dst) {
  uint4 o0, o1;
  o0.x = dequant_pair(w.x & 0xFFFFu, S);
  o0.y = dequant_pair(w.x >> 16, S);
  o0.z = dequant_pair(w.y & 0xFFFFu, S);
  o0.w = dequant_pair(w.y >> 16, S);
  o1.x = dequant_pair(w.z & 0xFFFFu, S);
  o1.y = dequant_pair(w.z >> 16, S);
  o1.z = dequant_pair(w.w & 0xFFFFu, S);
  o1.w = dequant_pair(w.w >> 16, S);
  st_stream_v4(dst, o0);
  st_stream_v4(dst + 8, o1);
}

// 16 consecutive codes that share one scale (cols and bc multiples of 16);
// each thread has U such vectors in flight.
constexpr int DQ_U = 4;
__global__ void __launch_bounds__(256) dequant_v16_kernel(const uint8_t* __restrict__ q,
                                                          const float* __restrict__ s,
                                                          int64_t cols, int64_t br, int64_t bc,
                                                          int64_t nbc, int64_t nvec,
                                                          uint16_t* __restrict__ y) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t v0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v0 < nvec;
       v0 += stride * DQ_U) {
    uint4 w[DQ_U];
    float S[DQ_U];
#pragma unroll
    for (int u = 0; u < DQ_U; ++u) {
      const int64_t v = v0 + u * stride;
      if (v < nvec) {
        const int64_t e = v * 16;
        const int64_t r = e / cols, c = e - r * cols;
        S[u] = s[(r / br) * nbc + c / bc];
        w[u] = ld_stream_v4(q + e);
      }
    }
#pragma unroll
    for (int u = 0; u < DQ_U; ++u) {
      const int64_t v = v0 + u * stride;
      if (v < nvec) dequant_store16(w[u], S[u], y + v * 16);
    }
  }
}


// Any shape: one element per thread step.
__global__ void __launch_bounds__(256) dequant_scalar_kernel(const uint8_t* __restrict__ q,
                                                             const float* __restrict__ s,
                                                             int64_t rows, int64_t cols,
                                                             int64_t br, int64_t bc, int64_t nbc,
                                                             uint16_t* __restrict__ y) {
  const int64_t n = rows * cols;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = e / cols, c = e - r * cols;
    const float S = s[(r / br) * nbc + c / bc];
    y[e] = (uint16_t)(dequant_pair(q[e], S) & 0xFFFFu);
  }
}

cudaError_t launch_dequant(const uint8_t* q, const float* s, int64_t rows, int64_t cols,
                           int64_t br, int64_t bc, uint16_t* y, cudaStream_t st) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  const int64_t nbc = (cols + bc - 1) / bc;
  if (cols % 16 == 0 && bc % 16 == 0) {
    const int64_t nvec = rows * cols / 16;
    dequant_v16_kernel<<<grid_for(nvec, 256 * DQ_U), 256, 0, st>>>(q, s, cols, br, bc, nbc, nvec,
                                                                   y);
  } else {
    dequant_scalar_kernel<<<grid_for(rows * cols, 256 * 8), 256, 0, st>>>(q, s, rows, cols, br,
                                                                          bc, nbc, y);
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Quantization-error report: one warp (small blocks) or one CTA (blocks of
// 4096 elements and more) per report block.  e = x - x_hat is
// formed in binary32, which is exact whenever x_hat lies within a factor 2
// of x (Sterbenz) -- every pair the quantizers produce -- so the block
// maximum is exact.  The lanes walk the block's 8-element row chunks in
// row-major order, ERR_U chunks in flight each; squares are summed over
// those 32 elements in binary32 and then accumulated in binary64 (binary64
// arithmetic is scarce on this part, so it runs once per 32 elements).
// ---------------------------------------------------------------------------
constexpr int ERR_U = 4;
struct ErrLayout {
  int64_t rows, cols;
  int64_t sbr, sbc, nsbc;  // quantization blocks
  int64_t rbr, rbc, nrbc;  // report blocks
  int64_t nblocks;
};

__device__ __forceinline__ void err_accumulate8(uint4 xv, uint2 qv, float S, float& mx, float& e2,
                                                float& x2) {
  const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
  const uint32_t qw[2] = {qv.x, qv.y};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 d = e4m3x2_to_float2((uint16_t)((qw[i >> 1] >> ((i & 1) * 16)) & 0xFFFFu));
    const float x0 = bf16_lo(xw[i]), x1 = bf16_hi(xw[i]);
    const float e0 = __fsub_rn(x0, __fmul_rn(d.x, S));
    const float e1 = __fsub_rn(x1, __fmul_rn(d.y, S));
    mx = fmaxf(mx, fmaxf(fabsf(e0), fabsf(e1)));
    e2 = __fmaf_rn(e0, e0, e2);
    e2 = __fmaf_rn(e1, e1, e2);
    x2 = __fmaf_rn(x0, x0, x2);
    x2 = __fmaf_rn(x1, x1, x2);
  }
}

// kCta: one CTA (8 warps) walks each report block -- for large blocks, so
// that a few blocks still keep enough loads in flight; otherwise one warp.
template <bool kVec, bool kCta>
__global__ void __launch_bounds__(256) quant_error_kernel(const uint16_t* __restrict__ x,
                                                          const uint8_t* __restrict__ q,
                                                          const float* __restrict__ s,
                                                          ErrLayout L, double* __restrict__ stats) {
  __shared__ double red[8][3];
  const int lane = threadIdx.x & 31;
  const uint32_t nthr = kCta ? 256u : 32u;
  const uint32_t tid = kCta ? threadIdx.x : (uint32_t)lane;
  const int64_t unit = kCta ? (int64_t)blockIdx.x
                            : (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t nunits = kCta ? (int64_t)gridDim.x : (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t b = unit; b < L.nblocks; b += nunits) {
    const int64_t br = b / L.nrbc, bc = b - br * L.nrbc;
    const int64_t r0 = br * L.rbr, c0 = bc * L.rbc;
    const int64_t r1 = min(L.rows, r0 + L.rbr), c1 = min(L.cols, c0 + L.rbc);
    float mx = 0.0f;
    double se = 0.0, sx = 0.0;
    if (kVec) {
      // a report block holds at most 2^20 elements: chunk indices are 32-bit
      const uint32_t cpr = (uint32_t)((c1 - c0) / 8);  // 8-element chunks per block row
      // the usual case: the whole report block lies in one scale block
      const bool one_scale = r0 / L.sbr == (r1 - 1) / L.sbr && c0 / L.sbc == (c1 - 1) / L.sbc;
      const float S1 = one_scale ? s[(r0 / L.sbr) * L.nsbc + c0 / L.sbc] : 0.0f;
      // chunk i = dr * cpr + dc walked as (dr, dc) with carries, no division
      const uint32_t nr = (uint32_t)(r1 - r0);
      const uint32_t sq = nthr / cpr, sm = nthr % cpr;
      uint32_t dr0 = tid / cpr, dc0 = tid % cpr;
      while (dr0 < nr) {
        uint4 xv[ERR_U];
        uint2 qv[ERR_U];
        float S[ERR_U];
        bool ok[ERR_U];
        uint32_t dr = dr0, dc = dc0;
#pragma unroll
        for (int u = 0; u < ERR_U; ++u) {
          ok[u] = dr < nr;
          if (ok[u]) {
            const int64_t rr = r0 + dr, cc = c0 + (int64_t)dc * 8;
            xv[u] = ld_stream_v4(x + rr * L.cols + cc);
            qv[u] = *reinterpret_cast<const uint2*>(q + rr * L.cols + cc);
            S[u] = one_scale ? S1 : s[(rr / L.sbr) * L.nsbc + cc / L.sbc];
          }
          dr += sq;
          dc += sm;
          if (dc >= cpr) { dc -= cpr; ++dr; }
        }
        dr0 = dr;
        dc0 = dc;
        float e2 = 0.0f, x2 = 0.0f;
#pragma unroll
        for (int u = 0; u < ERR_U; ++u)
          if (ok[u]) err_accumulate8(xv[u], qv[u], S[u], mx, e2, x2);
        se += (double)e2;
        sx += (double)x2;
      }
    } else {
      const int64_t w = c1 - c0;
      const int64_t n = (r1 - r0) * w;
      for (int64_t i = tid; i < n; i += nthr) {
        const int64_t r = r0 + i / w, c = c0 + i % w;
        const float S = s[(r / L.sbr) * L.nsbc + c / L.sbc];
        const float d = e4m3x2_to_float2(q[r * L.cols + c]).x;
        const float xv = bf16_lo(x[r * L.cols + c]);
        const float e = __fsub_rn(xv, __fmul_rn(d, S));
        mx = fmaxf(mx, fabsf(e));
        se += (double)e * (double)e;
        sx += (double)xv * (double)xv;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
      se += __shfl_xor_sync(0xFFFFFFFFu, se, o);
      sx += __shfl_xor_sync(0xFFFFFFFFu, sx, o);
    }
    if (kCta) {
      // warps' partials combined in a fixed order: the result does not
      // depend on scheduling
      if (lane == 0) {
        red[threadIdx.x >> 5][0] = (double)mx;
        red[threadIdx.x >> 5][1] = se;
        red[threadIdx.x >> 5][2] = sx;
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        double m = 0.0, a = 0.0, c = 0.0;
        for (int wi = 0; wi < 8; ++wi) {
          m = fmax(m, red[wi][0]);
          a += red[wi][1];
          c += red[wi][2];
        }
        stats[3 * b + 0] = m;
        stats[3 * b + 1] = a;
        stats[3 * b + 2] = c;
      }
      __syncthreads();
    } else if (lane == 0) {
      stats[3 * b + 0] = (double)mx;
      stats[3 * b + 1] = se;
      stats[3 * b + 2] = sx;
    }
  }
}

cudaError_t launch_quant_error(const uint16_t* x, const uint8_t* q, const float* s, int64_t rows,
                               int64_t cols, int64_t sbr, int64_t sbc, int64_t rbr, int64_t rbc,
                               double* stats, cudaStream_t st) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  ErrLayout L;
  L.rows = rows;
  L.cols = cols;
  L.sbr = sbr;
  L.sbc = sbc;
  L.nsbc = (cols + sbc - 1) / sbc;
  L.rbr = rbr;
  L.rbc = rbc;
  L.nrbc = (cols + rbc - 1) / rbc;
  L.nblocks = ((rows + rbr - 1) / rbr) * L.nrbc;
  // 8-element vectors stay inside one row, one report block and one scale
  const bool vec = cols % 8 == 0 && rbc % 8 == 0 && sbc % 8 == 0;
  // a CTA per block while blocks are few (so that enough loads are in
  // flight); a warp per block once there are plenty (less reduction work)
  if (rbr * rbc >= 4096 && L.nblocks < 16 * (int64_t)sm_count()) {
    const unsigned grid = grid_for(L.nblocks, 1);
    if (vec)
      quant_error_kernel<true, true><<<grid, 256, 0, st>>>(x, q, s, L, stats);
    else
      quant_error_kernel<false, true><<<grid, 256, 0, st>>>(x, q, s, L, stats);
  } else {  // a warp per block, 8 per CTA
    const unsigned grid = grid_for(L.nblocks, 8);
    if (vec)
      quant_error_kernel<true, false><<<grid, 256, 0, st>>>(x, q, s, L, stats);
    else
      quant_error_kernel<false, false><<<grid, 256, 0, st>>>(x, q, s, L, stats);
  }
  return cudaGetLastError();
}

}  // namespace w8a8
