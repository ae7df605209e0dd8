// quant.cu -- the HBM-bound kernels of the path: E4M3 codec, 1x128
// per-token activation quantizer, 128x128 blockwise weight quantizer and the
// per-tensor KV-cache quantizer.
//
// Every quantizer computes, per group G ("Unified FP8" notes, scale and
// quantization equations; NeMo RL FP8 Table 1 and Table 3 granularities):
//   amax = max_{x in G} |x|,  S = RN32(amax / 448) (1 if amax = 0),
//   q = E4M3(RN32(x / S))     round to nearest even, saturating at 448,
// bit-exactly (see common.cuh for the coding of x / S).
//
// Design for GB300: 16-byte coalesced BF16 loads with the non-coherent,
// no-L1-allocate hint; a group of 128 BF16 values is 256 contiguous bytes
// handled by 16 lanes, its amax reduced with 4 butterfly shuffles; several
// groups in flight per thread so each SM keeps tens of KB of loads
// outstanding; codes leave as 8-byte stores.  Grids are multiples of the SM
// count.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tmap.h"

namespace w8a8 {

// Set (first error wins) when a bounded wait in a quantization kernel gives up.
__device__ int g_w8a8_quant_error = 0;
// Test hook (w8a8_debug_force_wait_timeout): when set, the weight
// quantizer's consumers give up on their first block at once, as if the
// wait's time limit had passed, so that the abort path runs on demand.
__device__ int g_w8a8_quant_force_timeout = 0;

cudaError_t set_quant_force_timeout(int on) {
  return cudaMemcpyToSymbol(g_w8a8_quant_force_timeout, &on, sizeof(int));
}

cudaError_t consume_quant_error(int* code) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_w8a8_quant_error, sizeof(int));
  if (e == cudaSuccess && v != 0) {
    const int z = 0;
    e = cudaMemcpyToSymbol(g_w8a8_quant_error, &z, sizeof(int));
  }
  *code = v;
  return e;
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

__host__ __device__ inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Grid for a grid-stride kernel: enough CTAs to cover `work` items of
// `per_cta` each, capped at `waves` CTAs per SM.
static inline unsigned grid_for(int64_t work, int64_t per_cta, int waves) {
  int64_t want = cdiv(std::max<int64_t>(work, 1), per_cta);
  int64_t cap = (int64_t)sm_count() * waves;
  return (unsigned)std::max<int64_t>(1, std::min(want, cap));
}

// =====================================================================
// E4M3 codec
// =====================================================================

__global__ void __launch_bounds__(256) e4m3_encode_kernel(const float* __restrict__ x, int64_t n,
                                                          uint8_t* __restrict__ q) {
  const int64_t nv = n / 8;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (int64_t i = tid; i < nv; i += stride) {
    const uint4 a = ld_stream_v4(x + i * 8);
    const uint4 b = ld_stream_v4(x + i * 8 + 4);
    uint2 c;
    c.x = cvt_e4m3x2(__uint_as_float(a.x), __uint_as_float(a.y)) |
          (cvt_e4m3x2(__uint_as_float(a.z), __uint_as_float(a.w)) << 16);
    c.y = cvt_e4m3x2(__uint_as_float(b.x), __uint_as_float(b.y)) |
          (cvt_e4m3x2(__uint_as_float(b.z), __uint_as_float(b.w)) << 16);
    st_stream_v2(q + i * 8, c);
  }
  for (int64_t i = nv * 8 + tid; i < n; i += stride)
    q[i] = (uint8_t)(cvt_e4m3x2(x[i], 0.0f) & 0xFFu);
}

__global__ void __launch_bounds__(256) e4m3_decode_kernel(const uint8_t* __restrict__ q, int64_t n,
                                                          float* __restrict__ x) {
  const int64_t nv = n / 16;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (int64_t i = tid; i < nv; i += stride) {
    const uint4 c = ld_stream_v4(q + i * 16);
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 lo = e4m3x2_to_float2((uint16_t)(w[j] & 0xFFFFu));
      const float2 hi = e4m3x2_to_float2((uint16_t)(w[j] >> 16));
      uint4 o = make_uint4(__float_as_uint(lo.x), __float_as_uint(lo.y), __float_as_uint(hi.x),
                           __float_as_uint(hi.y));
      st_stream_v4(x + i * 16 + j * 4, o);
    }
  }
  for (int64_t i = nv * 16 + tid; i < n; i += stride) x[i] = e4m3x2_to_float2(q[i]).x;
}

cudaError_t launch_e4m3_encode(const float* x, int64_t n, uint8_t* q, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  e4m3_encode_kernel<<<grid_for(n, 256 * 8, 8), 256, 0, st>>>(x, n, q);
  return cudaGetLastError();
}

cudaError_t launch_e4m3_decode(const uint8_t* q, int64_t n, float* x, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  e4m3_decode_kernel<<<grid_for(n, 256 * 16, 8), 256, 0, st>>>(q, n, x);
  return cudaGetLastError();
}

// =====================================================================
// Generic block quantizer (any block shape, any row length): one CTA per
// block, scalar loads, two passes.  Serves rows whose length is not a
// multiple of 8 BF16 values, where 16-byte row segments do not exist.
// =====================================================================

template <bool kPow2>
__global__ void __launch_bounds__(256) block_quant_generic_kernel(const uint16_t* __restrict__ x,
                                                                  int64_t rows, int64_t cols,
                                                                  int64_t br, int64_t bc,
                                                                  uint8_t* __restrict__ q,
                                                                  float* __restrict__ s) {
  __shared__ float red[8];
  const int64_t nbc = cdiv(cols, bc);
  const int64_t blk = blockIdx.x;
  const int64_t bi = blk / nbc, bj = blk - bi * nbc;
  const int64_t r0 = bi * br, r1 = min(r0 + br, rows);
  const int64_t c0 = bj * bc, c1 = min(c0 + bc, cols);
  const int64_t w = c1 - c0, cnt = (r1 - r0) * w;
  float a = 0.0f;
  for (int64_t t = threadIdx.x; t < cnt; t += blockDim.x) {
    const int64_t r = r0 + t / w, c = c0 + t % w;
    a = fmaxf(a, fabsf(bf16_lo(x[r * cols + c])));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
  __syncthreads();
  a = red[0];
  for (int i = 1; i < (int)(blockDim.x >> 5); ++i) a = fmaxf(a, red[i]);
  const float S = group_scale<kPow2>(a);
  const QuantScale qs = make_quant_scale(S);
  for (int64_t t = threadIdx.x; t < cnt; t += blockDim.x) {
    const int64_t r = r0 + t / w, c = c0 + t % w;
    q[r * cols + c] = (uint8_t)quant_one(bf16_lo(x[r * cols + c]), qs);
  }
  if (threadIdx.x == 0) s[blk] = S;
}

static cudaError_t launch_generic(const uint16_t* x, int64_t rows, int64_t cols, int64_t br,
                                  int64_t bc, uint8_t* q, float* s, cudaStream_t st,
                                  bool pow2 = false) {
  const int64_t nb = cdiv(rows, br) * cdiv(cols, bc);
  if (nb == 0) return cudaSuccess;
  if (nb > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  if (pow2)
    block_quant_generic_kernel<true><<<(unsigned)nb, 256, 0, st>>>(x, rows, cols, br, bc, q, s);
  else
    block_quant_generic_kernel<false><<<(unsigned)nb, 256, 0, st>>>(x, rows, cols, br, bc, q, s);
  return cudaGetLastError();
}

// =====================================================================
// 1x128 per-token activation quantizer (row length a multiple of 8)
// =====================================================================
// A warp quantizes 2 groups per unit (lanes 0-15 and 16-31, 8 BF16 values
// per lane) and U units per iteration, loads first, so 4 KB per warp are in
// flight.  Consecutive warps take consecutive groups: the access stream is
// contiguous.

// With row_idx, output row r quantizes x row row_idx[r] (a zero row when the
// index is outside [0, rows_x)); without it, row r quantizes row r.
template <typename IdxT, bool kPow2>
__global__ void __launch_bounds__(256) act_quant_kernel(const uint16_t* __restrict__ x, IdxT m,
                                                        IdxT k, uint8_t* __restrict__ q,
                                                        float* __restrict__ s,
                                                        const int32_t* __restrict__ row_idx,
                                                        IdxT rows_x) {
  constexpr int U = 4;
  const IdxT gpr = (k + 127) / 128;
  const IdxT G = m * gpr;
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4, l16 = lane & 15;
  const IdxT warp = (IdxT)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const IdxT nwarps = (IdxT)gridDim.x * (blockDim.x >> 5);
  for (IdxT base = warp * (2 * U); base < G; base += nwarps * (2 * U)) {
    uint4 v[U];
    IdxT off[U];
    bool ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const IdxT g = base + 2 * u + half;
      const IdxT row = g / gpr;
      const IdxT col = (g - row * gpr) * 128 + l16 * 8;
      ok[u] = (g < G) && (col < k);
      off[u] = row * k + col;
      bool rd = ok[u];
      IdxT src = row;
      if (row_idx != nullptr && rd) {
        const int64_t r = row_idx[row];
        rd = r >= 0 && r < (int64_t)rows_x;
        src = rd ? (IdxT)r : 0;
      }
      v[u] = rd ? ld_stream_v4(x + src * k + col) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float a = absmax_bf16x2(v[u].x, 0.0f);
      a = absmax_bf16x2(v[u].y, a);
      a = absmax_bf16x2(v[u].z, a);
      a = absmax_bf16x2(v[u].w, a);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
      const float S = group_scale<kPow2>(a);
      const QuantScale qs = make_quant_scale(S);
      if (ok[u]) {
        uint2 c;
        c.x = quant_bf16x4(v[u].x, v[u].y, qs);
        c.y = quant_bf16x4(v[u].z, v[u].w, qs);
        st_stream_v2(q + off[u], c);
      }
      const IdxT g = base + 2 * u + half;
      if (l16 == 0 && g < G) s[g] = S;
    }
  }
}

// Rows that are whole multiples of 128: group g is the 256 bytes at g * 128
// elements and its scale is s[g], so no row/column arithmetic is needed.
// Four lanes share a group (32 values each, four 16-byte loads), which
// spreads the per-group work -- two butterfly steps, S and the reciprocal --
// over 32 values per lane; a warp covers 8 consecutive groups (2 KB) per
// unit and U units are loaded before any is used.
//
// Launched as a programmatic dependent, and letting the next kernel on the
// stream launch at once: in a chain quantizer -> GEMM the GEMM's prologue
// (and, with static weights, its first weight reads) overlaps this kernel,
// and this kernel's launch overlaps the end of the one before it.  Nothing
// is read or written before that previous kernel has completed.
template <int U, bool kPow2>
__global__ void __launch_bounds__(256) act_quant_k128_kernel(const uint16_t* __restrict__ x,
                                                             int64_t G, uint8_t* __restrict__ q,
                                                             float* __restrict__ s) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int sub = lane & 3, gi = lane >> 2;
  const int64_t warp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t base = warp * (8 * U); base < G; base += nwarps * (8 * U)) {
    uint4 v[U][4];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t g = base + 8 * u + gi;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        v[u][j] = g < G ? ld_stream_v4(x + g * 128 + (sub + 4 * j) * 8) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t g = base + 8 * u + gi;
      float a = absmax_bf16x8_tree<4>(v[u]);
      a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
      a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
      const float S = group_scale<kPow2>(a);
      const QuantScale qs = make_quant_scale(S);
      if (g < G) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint2 c;
          c.x = quant_bf16x4(v[u][j].x, v[u][j].y, qs);
          c.y = quant_bf16x4(v[u][j].z, v[u][j].w, qs);
          st_stream_v2(q + g * 128 + (sub + 4 * j) * 8, c);
        }
        if (sub == 0) s[g] = S;
      }
    }
  }
}

// The same over routed rows, rows a multiple of 128: output group g (row
// g / gpr, group g % gpr) reads the group of x row row_idx[g / gpr], or zeros
// when that index is outside [0, rows_x).  Group counts fit in 32 bits.
template <int U>
__global__ void __launch_bounds__(256) act_quant_gather_k128_kernel(
    const uint16_t* __restrict__ x, int64_t rows_x, const int32_t* __restrict__ row_idx,
    uint32_t gpr, uint32_t G, uint8_t* __restrict__ q, float* __restrict__ s) {
  const int lane = threadIdx.x & 31;
  const int sub = lane & 3, gi = lane >> 2;
  const uint32_t warp = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const uint32_t nwarps = gridDim.x * (blockDim.x >> 5);
  for (uint32_t base = warp * (8 * U); base < G; base += nwarps * (8 * U)) {
    const uint16_t* src[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t g = base + 8 * u + gi;
      src[u] = nullptr;
      if (g < G) {
        const uint32_t r = g / gpr;
        const int64_t sr = row_idx[r];
        if (sr >= 0 && sr < rows_x) src[u] = x + ((uint64_t)sr * gpr + (g - r * gpr)) * 128;
      }
    }
    uint4 v[U][4];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int j = 0; j < 4; ++j)
        v[u][j] = src[u] ? ld_stream_v4(src[u] + (sub + 4 * j) * 8) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t g = base + 8 * u + gi;
      float a = absmax_bf16x8_tree<4>(v[u]);
      a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
      a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
      const float S = scale_from_amax(a);
      const QuantScale qs = make_quant_scale(S);
      if (g < G) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint2 c;
          c.x = quant_bf16x4(v[u][j].x, v[u][j].y, qs);
          c.y = quant_bf16x4(v[u][j].z, v[u][j].w, qs);
          st_stream_v2(q + (uint64_t)g * 128 + (sub + 4 * j) * 8, c);
        }
        if (sub == 0) s[g] = S;
      }
    }
  }
}

template <bool kPow2>
static cudaError_t launch_act_quant_t(const uint16_t* x, int64_t m, int64_t k, uint8_t* q,
                                      float* s, cudaStream_t st) {
  if (m == 0 || k == 0) return cudaSuccess;
  if (k % 8 != 0) return launch_generic(x, m, k, 1, 128, q, s, st, kPow2);
  const int64_t G = m * cdiv(k, 128);
  if (k % 128 == 0) {
    constexpr int U = 2;
    const unsigned grid = grid_for(G, 8 * 8 * U, 8);  // 8 warps x 8 groups x U per CTA pass
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, act_quant_k128_kernel<U, kPow2>, x, G, q, s);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  const unsigned grid = grid_for(G, 8 * 8, 16);  // 8 warps x 8 groups per CTA iteration
  if (m * k < (int64_t)0x7FFFFFFF)
    act_quant_kernel<uint32_t, kPow2><<<grid, 256, 0, st>>>(x, (uint32_t)m, (uint32_t)k, q, s,
                                                            nullptr, (uint32_t)m);
  else
    act_quant_kernel<int64_t, kPow2><<<grid, 256, 0, st>>>(x, m, k, q, s, nullptr, m);
  return cudaGetLastError();
}

cudaError_t launch_act_quant(const uint16_t* x, int64_t m, int64_t k, uint8_t* q, float* s,
                             cudaStream_t st, bool pow2) {
  return pow2 ? launch_act_quant_t<true>(x, m, k, q, s, st)
              : launch_act_quant_t<false>(x, m, k, q, s, st);
}

cudaError_t launch_act_quant_gather(const uint16_t* x, int64_t rows_x, int64_t k,
                                    const int32_t* row_idx, int64_t total_rows, uint8_t* q,
                                    float* s, cudaStream_t st) {
  if (total_rows == 0 || k == 0) return cudaSuccess;
  if (k % 8 != 0) return cudaErrorNotSupported;
  const int64_t G = total_rows * cdiv(k, 128);
  if (k % 128 == 0 && G < (int64_t)0x7FFFFFFF) {
    constexpr int U = 2;
    const unsigned grid = grid_for(G, 8 * 8 * U, 8);
    act_quant_gather_k128_kernel<U><<<grid, 256, 0, st>>>(x, rows_x, row_idx, (uint32_t)(k / 128),
                                                          (uint32_t)G, q, s);
    return cudaGetLastError();
  }
  const unsigned grid = grid_for(G, 8 * 8, 16);
  act_quant_kernel<int64_t, false><<<grid, 256, 0, st>>>(x, total_rows, k, q, s, row_idx, rows_x);
  return cudaGetLastError();
}

// =====================================================================
// 128x128 blockwise weight quantizer (row length a multiple of 8)
// =====================================================================
// Persistent CTAs (2 per SM), each a producer warp plus 8 consumer warps,
// over a 3-stage shared-memory ring of 32 KB blocks:
//   producer  one 2-D TMA tensor load per block (128 rows x 256 bytes; rows
//             and columns past the matrix edge arrive as zeros), completing
//             on the stage's mbarrier, up to 3 blocks ahead;
//   consumers 16-byte conflict-free shared loads (lanes 0-15 one row, 16-31
//             the next), release the stage, block amax (butterfly + 8
//             partials through shared memory + a named barrier), S, then
//             the codes straight to global memory as 8-byte stores.
// A batch of matrices is one launch; a CTA finds the matrix of a block from
// the block prefix sums held in the kernel parameters.
// All waits are bounded; a wait that gives up records an error and the CTA
// stops after draining its copies.

template <int kMax>
struct WeightBatch {
  CUtensorMap tmap[kMax];  // [n, k] BF16, box 128 x 128, zero fill outside
  const uint16_t* w[kMax];
  uint8_t* wq[kMax];
  float* ws[kMax];
  int64_t n[kMax];
  int64_t k[kMax];
  int64_t first[kMax + 1];  // first block index of each matrix; first[count] = total
  int count;
};

constexpr int WQ_STAGES = 3;
constexpr int WQ_CONSUMER_WARPS = 8;
constexpr int WQ_THREADS = 32 * (WQ_CONSUMER_WARPS + 1);
constexpr int WQ_STAGE_BYTES = 128 * 256;
constexpr int WQ_SMEM = WQ_STAGES * WQ_STAGE_BYTES + 2 * WQ_STAGES * 8 + 2 * 8 * 4 + 16;
constexpr uint64_t WQ_WAIT_NS = 2000000000ull;

struct BlockRef {
  int mat;
  int64_t bi, bj, nbk;
  int rows;  // valid rows in the block
  int cols;  // valid columns (multiple of 8)
};

// The matrix holding block blk.  A CTA visits its blocks in increasing
// order, so the previous answer (hint) is advanced instead of searched for:
// usually no step at all (matrices hold >= 1024 blocks, a CTA strides ~300).
template <int kMax>
__device__ __forceinline__ int find_matrix(const WeightBatch<kMax>& b, int64_t blk, int hint) {
  int lo = hint;
  if (kMax > 1)
    while (b.first[lo + 1] <= blk) ++lo;
  return lo;
}

template <int kMax>
__device__ __forceinline__ BlockRef locate_block(const WeightBatch<kMax>& b, int64_t blk, int lo) {
  BlockRef r;
  r.mat = lo;
  const int64_t n = b.n[lo], k = b.k[lo];
  // block counts of one matrix fit in 32 bits (rows and columns are < 2^31)
  const uint32_t nbk = (uint32_t)((k + 127) >> 7);
  const uint32_t local = (uint32_t)(blk - b.first[lo]);
  const uint32_t bi = local / nbk;
  r.nbk = nbk;
  r.bi = bi;
  r.bj = local - bi * nbk;
  r.rows = (int)min((int64_t)128, n - r.bi * 128);
  r.cols = (int)min((int64_t)128, k - r.bj * 128);
  return r;
}

template <int kMax, bool kPow2>
__global__ void __launch_bounds__(WQ_THREADS, 2)
    weight_quant_kernel(const __grid_constant__ WeightBatch<kMax> b) {
  extern __shared__ __align__(1024) uint8_t wq_smem[];
  const uint32_t sbase = ptx::smem_addr(wq_smem);
  const uint32_t bar0 = sbase + WQ_STAGES * WQ_STAGE_BYTES;
  float* red = reinterpret_cast<float*>(wq_smem + WQ_STAGES * WQ_STAGE_BYTES + 2 * WQ_STAGES * 8);
  volatile int* abort_flag =
      reinterpret_cast<volatile int*>(wq_smem + WQ_STAGES * WQ_STAGE_BYTES + 2 * WQ_STAGES * 8 + 64);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (WQ_STAGES + s); };
  if (threadIdx.x == 0) {
    for (int s = 0; s < WQ_STAGES; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), WQ_CONSUMER_WARPS);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  const int64_t total = b.first[b.count];

  if (warp == WQ_CONSUMER_WARPS) {
    // ------------------------------------------------------------ producer
    int64_t issued = 0;
    int mat = 0;
    for (int64_t blk = blockIdx.x; blk < total; blk += gridDim.x, ++issued) {
      const int s = (int)(issued % WQ_STAGES);
      const uint32_t par = (uint32_t)((issued / WQ_STAGES) & 1);
      uint32_t ok = 1;
      if (lane == 0) {
        ok = ptx::mbar_wait(empty_bar(s), par ^ 1u, WQ_WAIT_NS) ? 1u : 0u;
        if (!ok) { atomicCAS(&g_w8a8_quant_error, 0, 11); *abort_flag = 1; }
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok || *abort_flag) break;
      mat = find_matrix(b, blk, mat);
      const BlockRef r = locate_block(b, blk, mat);
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(full_bar(s), WQ_STAGE_BYTES);
        ptx::tma_load_2d(sbase + s * WQ_STAGE_BYTES, &b.tmap[r.mat], full_bar(s), (int)(r.bj * 128),
                         (int)(r.bi * 128));
      }
    }
    // drain: no copy may still be landing when the CTA exits
    if (lane == 0) {
      const int64_t first = issued > WQ_STAGES ? issued - WQ_STAGES : 0;
      for (int64_t i = first; i < issued; ++i)
        if (!ptx::mbar_wait(full_bar((int)(i % WQ_STAGES)), (uint32_t)((i / WQ_STAGES) & 1), WQ_WAIT_NS))
          atomicCAS(&g_w8a8_quant_error, 0, 12);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int t = threadIdx.x;  // 0..255
  const int ch = t & 15;      // 16-byte chunk within a 256-byte row
  int64_t it = 0;
  int mat = 0;
  for (int64_t blk = blockIdx.x; blk < total; blk += gridDim.x, ++it) {
    // the block's place does not depend on its data: find it before waiting
    mat = find_matrix(b, blk, mat);
    const BlockRef r = locate_block(b, blk, mat);
    const int s = (int)(it % WQ_STAGES);
    const uint32_t par = (uint32_t)((it / WQ_STAGES) & 1);
    uint32_t ok = 1;
    if (lane == 0)
      ok = (it == 0 && g_w8a8_quant_force_timeout) ? 0u
                                                    : (ptx::mbar_wait(full_bar(s), par, WQ_WAIT_NS) ? 1u : 0u);
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    if (!ok && lane == 0) atomicCAS(&g_w8a8_quant_error, 0, 13);
    const uint32_t stage = sbase + s * WQ_STAGE_BYTES;
    const bool col_ok = ch * 8 < r.cols;
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = ptx::lds128(stage + ((t >> 4) + 16 * j) * 256 + ch * 16);
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(empty_bar(s));
    float a = absmax_bf16x8_tree<8>(v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
    // Partials (and each warp's wait outcome) meet at one named barrier; the
    // decision to stop is taken from the same shared values by every
    // consumer, so all leave together and none waits on a barrier alone.
    float* rb = red + (it & 1) * 8;
    if (lane == 0) rb[warp] = ok ? a : -1.0f;
    ptx::named_bar_sync(1, 32 * WQ_CONSUMER_WARPS);
    if (fminf(fminf(fminf(rb[0], rb[1]), fminf(rb[2], rb[3])),
              fminf(fminf(rb[4], rb[5]), fminf(rb[6], rb[7]))) < 0.0f)
      break;
    a = fmaxf(fmaxf(fmaxf(rb[0], rb[1]), fmaxf(rb[2], rb[3])),
              fmaxf(fmaxf(rb[4], rb[5]), fmaxf(rb[6], rb[7])));
    const float S = group_scale<kPow2>(a);
    const QuantScale qs = make_quant_scale(S);
    const int64_t k = b.k[r.mat];
    uint8_t* dstq = b.wq[r.mat] + (r.bi * 128) * k + r.bj * 128 + ch * 8;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int row = (t >> 4) + 16 * j;
      if (col_ok && row < r.rows) {
        uint2 c;
        c.x = quant_bf16x4(v[j].x, v[j].y, qs);
        c.y = quant_bf16x4(v[j].z, v[j].w, qs);
        st_stream_v2(dstq + row * k, c);
      }
    }
    if (t == 0) b.ws[r.mat][r.bi * r.nbk + r.bj] = S;
  }
}

template <int kMax, bool kPow2>
static cudaError_t launch_weight_batch(const WeightJob* jobs, int count, cudaStream_t st) {
  WeightBatch<kMax> b;
  int64_t total = 0;
  b.count = count;
  for (int i = 0; i < count; ++i) {
    if (!make_tmap_2d(&b.tmap[i], jobs[i].w, 2, (uint64_t)jobs[i].n, (uint64_t)jobs[i].k, 128, 128,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
    b.w[i] = jobs[i].w;
    b.wq[i] = jobs[i].wq;
    b.ws[i] = jobs[i].ws;
    b.n[i] = jobs[i].n;
    b.k[i] = jobs[i].k;
    b.first[i] = total;
    total += cdiv(jobs[i].n, 128) * cdiv(jobs[i].k, 128);
  }
  for (int i = count; i <= kMax; ++i) b.first[i] = total;
  for (int i = count; i < kMax; ++i) {
    b.w[i] = nullptr; b.wq[i] = nullptr; b.ws[i] = nullptr; b.n[i] = 0; b.k[i] = 0;
  }
  if (total == 0) return cudaSuccess;
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(weight_quant_kernel<kMax, kPow2>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             WQ_SMEM);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = 1;
  }
  const unsigned grid = (unsigned)std::min<int64_t>(total, 2 * (int64_t)sm_count());
  weight_quant_kernel<kMax, kPow2><<<grid, WQ_THREADS, WQ_SMEM, st>>>(b);
  return cudaGetLastError();
}

template <bool kPow2>
static cudaError_t launch_weight_quant_t(const WeightJob* jobs, int count, cudaStream_t st) {
  constexpr int kBatch = 160;  // ~28 KB of kernel parameters (tensor maps included)
  WeightJob fast[kBatch];
  int nf = 0;
  for (int i = 0; i < count; ++i) {
    const WeightJob& j = jobs[i];
    if (j.n == 0 || j.k == 0) continue;
    if (j.k % 8 != 0) {
      cudaError_t e = launch_generic(j.w, j.n, j.k, 128, 128, j.wq, j.ws, st, kPow2);
      if (e != cudaSuccess) return e;
      continue;
    }
    fast[nf++] = j;
    if (nf == kBatch) {
      cudaError_t e = launch_weight_batch<kBatch, kPow2>(fast, nf, st);
      if (e != cudaSuccess) return e;
      nf = 0;
    }
  }
  if (nf == 1) return launch_weight_batch<1, kPow2>(fast, 1, st);
  if (nf > 1) return launch_weight_batch<kBatch, kPow2>(fast, nf, st);
  return cudaSuccess;
}

cudaError_t launch_weight_quant(const WeightJob* jobs, int count, cudaStream_t st, bool pow2) {
  return pow2 ? launch_weight_quant_t<true>(jobs, count, st)
              : launch_weight_quant_t<false>(jobs, count, st);
}

// =====================================================================
// Per-tensor KV-cache quantizer: pass 1 amax, pass 2 code
// =====================================================================
// Pass 1 folds |x| into one float per CTA and combines CTAs with atomicMax
// on the float's bit pattern (non-negative floats order like their bits), so
// the result does not depend on the order.  Pass 2 reads the amax, forms S
// and codes every element; it walks the tensor backwards so that the last
// tens of MB pass 1 read are still in L2 when pass 2 starts.  The stream
// orders the passes: no grid-wide wait inside a kernel.

__global__ void __launch_bounds__(256) kv_amax_kernel(const uint16_t* __restrict__ x, int64_t n,
                                                      unsigned int* __restrict__ amax_bits) {
  __shared__ float red[8];
  constexpr int U = 4;
  const int64_t nv = n / 8;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  float a = 0.0f;
  int64_t i = tid;
  for (; i + (U - 1) * stride < nv; i += U * stride) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) v[u] = ld_stream_v4(x + (i + u * stride) * 8);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      a = absmax_bf16x2(v[u].x, a);
      a = absmax_bf16x2(v[u].y, a);
      a = absmax_bf16x2(v[u].z, a);
      a = absmax_bf16x2(v[u].w, a);
    }
  }
  for (; i < nv; i += stride) {
    const uint4 v = ld_stream_v4(x + i * 8);
    a = absmax_bf16x2(v.x, a);
    a = absmax_bf16x2(v.y, a);
    a = absmax_bf16x2(v.z, a);
    a = absmax_bf16x2(v.w, a);
  }
  for (int64_t j = nv * 8 + tid; j < n; j += stride) a = fmaxf(a, fabsf(bf16_lo(x[j])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) a = fmaxf(a, red[w]);
    atomicMax(amax_bits, __float_as_uint(a));
  }
}

__global__ void __launch_bounds__(256) kv_quant_kernel(const uint16_t* __restrict__ x, int64_t n,
                                                       uint8_t* __restrict__ q,
                                                       float* __restrict__ scale,
                                                       const float* __restrict__ amax,
                                                       int mode) {
  float S;
  if (mode == 2) {
    S = *scale;
  } else {
    S = scale_from_amax(*amax);
    if (blockIdx.x == 0 && threadIdx.x == 0) *scale = S;
    if (mode == 1) return;
  }
  // a scale handed in by the caller may make x / S overflow: code by division
  const QuantScale qs = mode == 2 ? make_quant_scale_division(S) : make_quant_scale(S);
  constexpr int U = 4;
  const int64_t nv = n / 8;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  // tail first (it is at the end, which pass 1 read last)
  for (int64_t j = nv * 8 + tid; j < n; j += stride)
    q[j] = (uint8_t)quant_one(bf16_lo(x[j]), qs);
  int64_t i = tid;
  for (; i + (U - 1) * stride < nv; i += U * stride) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) v[u] = ld_stream_v4(x + (nv - 1 - (i + u * stride)) * 8);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      uint2 c;
      c.x = quant_bf16x4(v[u].x, v[u].y, qs);
      c.y = quant_bf16x4(v[u].z, v[u].w, qs);
      st_stream_v2(q + (nv - 1 - (i + u * stride)) * 8, c);
    }
  }
  for (; i < nv; i += stride) {
    const uint4 v = ld_stream_v4(x + (nv - 1 - i) * 8);
    uint2 c;
    c.x = quant_bf16x4(v.x, v.y, qs);
    c.y = quant_bf16x4(v.z, v.w, qs);
    st_stream_v2(q + (nv - 1 - i) * 8, c);
  }
}

cudaError_t launch_kv_amax_quantize(const uint16_t* x, int64_t n, uint8_t* q, float* scale,
                                    float* amax, int mode, cudaStream_t st) {
  if (mode != 2) {
    cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), st);
    if (e != cudaSuccess) return e;
    if (n > 0) {
      kv_amax_kernel<<<grid_for(n, 256 * 8 * 4, 8), 256, 0, st>>>(
          x, n, reinterpret_cast<unsigned int*>(amax));
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  const unsigned grid = (mode == 1) ? 1u : grid_for(n, 256 * 8 * 4, 8);
  if (mode == 2 && n == 0) return cudaSuccess;
  kv_quant_kernel<<<grid, 256, 0, st>>>(x, n, q, scale, amax, mode);
  return cudaGetLastError();
}

}  // namespace w8a8
