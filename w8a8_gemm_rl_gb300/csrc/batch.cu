// batch.cu -- the dequantizer and the quantization-error report over a whole
// batch of weight matrices in one launch each ("Unified FP8" notes: the
// fake-quant versus real-quant experiments and the quantization-error
// analysis, applied to every weight matrix a weight sync produces), for
// 128 x 128 scale blocks:
//
//   dequantize:  y[r, c] = BF16_RN( RN32( dec(q[r, c]) * S[r/128, c/128] ) )
//   report:      per 128 x 128 block, max |x - x_hat|, sum (x - x_hat)^2 and
//                sum x^2 with x_hat = RN32(dec(q) * S)
//
// the same arithmetic as dequantize_blockwise and quant_error_report.
//
// Like the batched weight quantizer: persistent CTAs (several per SM), one
// producer warp and 8 consumer warps each, over a shared-memory ring of whole
// blocks.  The producer brings each block by 2-D TMA (codes: 128 rows x 128
// bytes; for the report also the BF16 block, 128 rows x 256 bytes; rows and
// columns past the edge arrive as zeros); the consumers read it with 16-byte
// shared loads.  A CTA walks the blocks of the whole batch in increasing
// order and finds each block's matrix by advancing the previous one.  Every
// wait is bounded; a wait that gives up records an error (codes 41..43) and
// the CTA stops after draining its copies.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tmap.h"

namespace w8a8 {

__device__ int g_w8a8_batch_error = 0;

namespace batch {

constexpr uint64_t WAIT_NS = 2000000000ull;
constexpr int CONSUMER_WARPS = 8;
constexpr int THREADS = 32 * (CONSUMER_WARPS + 1);
constexpr int Q_BYTES = 128 * 128;      // a block of codes
constexpr int X_BYTES = 128 * 128 * 2;  // a block of BF16 inputs

template <bool kReport>
struct Cfg {
  static constexpr int STAGES = kReport ? 2 : 4;
  static constexpr int STAGE_BYTES = Q_BYTES + (kReport ? X_BYTES : 0);
  static constexpr int SMEM = STAGES * STAGE_BYTES + 2 * STAGES * 8 + 2 * 8 * 3 * 8 + 64;
};

template <int kMax, bool kReport>
struct Batch {
  CUtensorMap tq[kMax];                     // codes [n, k] u8, box 128 x 128
  CUtensorMap tx[kReport ? kMax : 1];       // report: inputs [n, k] BF16, box 128 x 128
  const float* s[kMax];
  uint16_t* y[kMax];                        // dequantize: output
  double* stats[kMax];                      // report: [ceil(n/128), ceil(k/128), 3]
  int64_t n[kMax];
  int64_t k[kMax];
  int64_t first[kMax + 1];                  // first block of each matrix; first[count] = total
  int count;
};

__device__ __forceinline__ void record_error(int code) { atomicCAS(&g_w8a8_batch_error, 0, code); }

template <int kMax, bool kReport>
__global__ void __launch_bounds__(THREADS, 2) block_pass_kernel(const __grid_constant__ Batch<kMax, kReport> b) {
  using C = Cfg<kReport>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = ptx::smem_addr(smem);
  const uint32_t bar0 = sbase + C::STAGES * C::STAGE_BYTES;
  double* red = reinterpret_cast<double*>(smem + C::STAGES * C::STAGE_BYTES + 2 * C::STAGES * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(
      smem + C::STAGES * C::STAGE_BYTES + 2 * C::STAGES * 8 + 2 * 8 * 3 * 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), CONSUMER_WARPS);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  const int64_t total = b.first[b.count];

  if (warp == CONSUMER_WARPS) {
    // ------------------------------------------------------------ producer
    int64_t issued = 0;
    int mat = 0;
    for (int64_t blk = blockIdx.x; blk < total; blk += gridDim.x, ++issued) {
      const int s = (int)(issued % C::STAGES);
      const uint32_t par = (uint32_t)((issued / C::STAGES) & 1);
      uint32_t ok = 1;
      if (lane == 0) {
        ok = ptx::mbar_wait(empty_bar(s), par ^ 1u, WAIT_NS) ? 1u : 0u;
        if (!ok) { record_error(41); *abort_flag = 1; }
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok || *abort_flag) break;
      while (kMax > 1 && b.first[mat + 1] <= blk) ++mat;
      const uint32_t nbk = (uint32_t)((b.k[mat] + 127) >> 7);
      const uint32_t local = (uint32_t)(blk - b.first[mat]);
      const int bi = (int)(local / nbk), bj = (int)(local - (uint32_t)bi * nbk);
      if (lane == 0) {
        const uint32_t st = sbase + s * C::STAGE_BYTES;
        ptx::mbar_arrive_expect_tx(full_bar(s), C::STAGE_BYTES);
        ptx::tma_load_2d(st, &b.tq[mat], full_bar(s), bj * 128, bi * 128);
        if (kReport) ptx::tma_load_2d(st + Q_BYTES, &b.tx[mat], full_bar(s), bj * 128, bi * 128);
      }
    }
    // drain: no copy may still be landing when the CTA exits
    if (lane == 0) {
      const int64_t first = issued > C::STAGES ? issued - C::STAGES : 0;
      for (int64_t i = first; i < issued; ++i)
        if (!ptx::mbar_wait(full_bar((int)(i % C::STAGES)), (uint32_t)((i / C::STAGES) & 1),
                            WAIT_NS))
          record_error(42);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int t = threadIdx.x;  // 0..255
  int64_t it = 0;
  int mat = 0;
  for (int64_t blk = blockIdx.x; blk < total; blk += gridDim.x, ++it) {
    while (kMax > 1 && b.first[mat + 1] <= blk) ++mat;
    const int64_t n = b.n[mat], k = b.k[mat];
    const uint32_t nbk = (uint32_t)((k + 127) >> 7);
    const uint32_t local = (uint32_t)(blk - b.first[mat]);
    const int64_t bi = local / nbk, bj = local - (uint32_t)bi * nbk;
    const int rows = (int)min((int64_t)128, n - bi * 128);
    const int cols = (int)min((int64_t)128, k - bj * 128);
    const float S = b.s[mat][bi * nbk + bj];  // independent of the data: before the wait
    const int s = (int)(it % C::STAGES);
    const uint32_t par = (uint32_t)((it / C::STAGES) & 1);
    uint32_t ok = 1;
    if (lane == 0) ok = ptx::mbar_wait(full_bar(s), par, WAIT_NS) ? 1u : 0u;
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    if (!ok && lane == 0) record_error(43);
    const uint32_t stq = sbase + s * C::STAGE_BYTES;
    if (!kReport) {
      // 16 codes per chunk, 8 chunks per row: thread t takes chunk t % 8 of
      // rows t / 8 + 32 j; a warp writes four whole 256-byte output rows
      uint4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = ptx::lds128(stq + ((t >> 3) + 32 * j) * 128 + (t & 7) * 16);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(empty_bar(s));
      // the warps' wait outcomes meet at one named barrier, so that all
      // consumers stop together and none waits on a barrier alone
      int* okw = reinterpret_cast<int*>(red) + (it & 1) * 8;
      if (lane == 0) okw[warp] = (int)ok;
      ptx::named_bar_sync(1, 32 * CONSUMER_WARPS);
      bool stop = false;
      for (int wi = 0; wi < CONSUMER_WARPS; ++wi) stop |= okw[wi] == 0;
      if (stop) break;
      const int c = (t & 7) * 16;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = (t >> 3) + 32 * j;
        if (r < rows && c < cols) {
          uint16_t* dst = b.y[mat] + (bi * 128 + r) * k + bj * 128 + c;
          uint4 o0, o1;
          o0.x = dequant_pair(v[j].x & 0xFFFFu, S);
          o0.y = dequant_pair(v[j].x >> 16, S);
          o0.z = dequant_pair(v[j].y & 0xFFFFu, S);
          o0.w = dequant_pair(v[j].y >> 16, S);
          o1.x = dequant_pair(v[j].z & 0xFFFFu, S);
          o1.y = dequant_pair(v[j].z >> 16, S);
          o1.z = dequant_pair(v[j].w & 0xFFFFu, S);
          o1.w = dequant_pair(v[j].w >> 16, S);
          st_stream_v4(dst, o0);
          st_stream_v4(dst + 8, o1);
        }
      }
    } else {
      // 8 elements per chunk, 16 chunks per row: thread t takes chunk t % 16
      // of rows t / 16 + 16 j.  Elements outside the matrix read as zeros on
      // both sides (x = 0, code 0), so they add nothing.
      const uint32_t stx = stq + Q_BYTES;
      const int ch = t & 15;
      float mx = 0.0f, e2 = 0.0f, x2 = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int r = (t >> 4) + 16 * j;
        const uint4 xv = ptx::lds128(stx + r * 256 + ch * 16);
        uint2 qv;
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(qv.x), "=r"(qv.y)
                     : "r"(stq + r * 128 + ch * 8));
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
        const uint32_t qw[2] = {qv.x, qv.y};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 d = e4m3x2_to_float2((uint16_t)((qw[i >> 1] >> ((i & 1) * 16)) & 0xFFFFu));
          const float x0 = bf16_lo(xw[i]), x1 = bf16_hi(xw[i]);
          const float ea = __fsub_rn(x0, __fmul_rn(d.x, S));
          const float eb = __fsub_rn(x1, __fmul_rn(d.y, S));
          mx = fmaxf(mx, fmaxf(fabsf(ea), fabsf(eb)));
          e2 = __fmaf_rn(ea, ea, e2);
          e2 = __fmaf_rn(eb, eb, e2);
          x2 = __fmaf_rn(x0, x0, x2);
          x2 = __fmaf_rn(x1, x1, x2);
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(empty_bar(s));
      // 64 squares per thread summed in binary32, then a binary32 tree over
      // the warp (butterfly) and the 8 warps' partials summed in binary64 in
      // index order by one thread: the result does not depend on scheduling.
      // The terms are non-negative, so the 64 running-sum steps and the 5
      // tree levels add at most 69 roundings of relative 2^-24: below
      // 4.2e-6, inside the report's 1e-5.  Binary64 arithmetic is scarce on
      // this part: it runs once per block.
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        e2 += __shfl_xor_sync(0xFFFFFFFFu, e2, o);
        x2 += __shfl_xor_sync(0xFFFFFFFFu, x2, o);
      }
      float* rb = reinterpret_cast<float*>(red) + (it & 1) * 24;
      if (lane == 0) {
        rb[3 * warp + 0] = ok ? mx : -1.0f;
        rb[3 * warp + 1] = e2;
        rb[3 * warp + 2] = x2;
      }
      ptx::named_bar_sync(1, 32 * CONSUMER_WARPS);
      bool stop = false;
      for (int wi = 0; wi < CONSUMER_WARPS; ++wi) stop |= rb[3 * wi] < 0.0f;
      if (stop) break;  // every consumer takes the same decision
      if (t == 0) {
        double m = 0.0, a = 0.0, c = 0.0;
        for (int wi = 0; wi < CONSUMER_WARPS; ++wi) {
          m = fmax(m, (double)rb[3 * wi]);
          a += (double)rb[3 * wi + 1];
          c += (double)rb[3 * wi + 2];
        }
        double* out = b.stats[mat] + 3 * (bi * nbk + bj);
        out[0] = m;
        out[1] = a;
        out[2] = c;
      }
    }
  }
}

template <int kMax, bool kReport>
static cudaError_t launch_chunk(const BlockJob* jobs, int count, cudaStream_t st) {
  using C = Cfg<kReport>;
  Batch<kMax, kReport> b;
  int64_t total = 0;
  b.count = count;
  for (int i = 0; i < count; ++i) {
    const BlockJob& j = jobs[i];
    if (!make_tmap_2d(&b.tq[i], j.q, 1, (uint64_t)j.n, (uint64_t)j.k, 128, 128,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
    if (kReport && !make_tmap_2d(&b.tx[i], j.x, 2, (uint64_t)j.n, (uint64_t)j.k, 128, 128,
                                 CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
    b.s[i] = j.s;
    b.y[i] = j.y;
    b.stats[i] = j.stats;
    b.n[i] = j.n;
    b.k[i] = j.k;
    b.first[i] = total;
    total += ((j.n + 127) / 128) * ((j.k + 127) / 128);
  }
  for (int i = count; i <= kMax; ++i) b.first[i] = total;
  for (int i = count; i < kMax; ++i) {
    b.s[i] = nullptr; b.y[i] = nullptr; b.stats[i] = nullptr; b.n[i] = 0; b.k[i] = 0;
  }
  if (total == 0) return cudaSuccess;
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(block_pass_kernel<kMax, kReport>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = 1;
  }
  const unsigned grid = (unsigned)std::min<int64_t>(total, 2 * (int64_t)sm_count());
  block_pass_kernel<kMax, kReport><<<grid, THREADS, C::SMEM, st>>>(b);
  return cudaGetLastError();
}

// Kernel parameters hold up to ~32 KB: 160 matrices for the dequantizer
// (one tensor map each), 96 for the report (two).
template <bool kReport>
static cudaError_t launch_all(const BlockJob* jobs, int count, cudaStream_t st) {
  constexpr int kBatch = kReport ? 96 : 160;
  for (int i0 = 0; i0 < count; i0 += kBatch) {
    const int c = std::min(kBatch, count - i0);
    cudaError_t e = c == 1 ? launch_chunk<1, kReport>(jobs + i0, 1, st)
                           : launch_chunk<kBatch, kReport>(jobs + i0, c, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace batch

cudaError_t launch_dequant_batch(const BlockJob* jobs, int count, cudaStream_t st) {
  return batch::launch_all<false>(jobs, count, st);
}

cudaError_t launch_quant_error_batch(const BlockJob* jobs, int count, cudaStream_t st) {
  return batch::launch_all<true>(jobs, count, st);
}

cudaError_t consume_batch_error(int* code) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_w8a8_batch_error, sizeof(int));
  if (e != cudaSuccess) return e;
  if (v != 0) {
    int z = 0;
    e = cudaMemcpyToSymbol(g_w8a8_batch_error, &z, sizeof(int));
  }
  *code = v;
  return e;
}

}  // namespace w8a8
