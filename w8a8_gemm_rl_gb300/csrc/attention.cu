// attention.cu -- decode attention over the FP8 KV cache (NeMo RL FP8 blog,
// Table 3 and the FP8 KV-cache section: Q, K and V carry one FP32 scale each;
// FP8-RL section 4: attention reads the FP8 KV cache):
//
//   score_t = softmax_scale * sq * sk * sum_d dec(q[b,h,d]) * dec(k[b,t,kh,d])
//   out_d   = sv * sum_{t < len_b} softmax(score)_t * dec(v[b,t,kh,d])
//
// one query token per sequence, grouped-query heads (query head h reads KV
// head h / (hq / hkv)), head dim 128.  Each CTA reads one (sequence, KV
// head) slice of K and V exactly once for up to 4 query heads, so the
// kernel streams the cache: it is HBM-bound, and runs on the CUDA cores.
//
// Layout inside a CTA (4 warps): warp w takes a contiguous quarter of the
// tokens and streams it through its own ring of shared-memory stages, each
// filled by two TMA tile loads (16 tokens of K, 16 of V: the 128-byte rows
// of one KV head sit hkv * 128 bytes apart in the cache, a 2-D box of
// 16 rows x 128 bytes).  Lane 0 keeps AT_STAGES - 1 chunks in flight while
// the warp computes on the oldest.  In a warp, lane group g (lanes
// 8g..8g+7) takes every 4th token of a chunk and lane l8 = lane % 8 holds
// dims 16 l8 .. 16 l8 + 15.  Scores are in log2 units (log2 e and every
// scale folded into the query), kept by an online softmax per lane group;
// the groups, then the warps, are merged at the end.  Binary32 arithmetic
// throughout; dot products and the value update use packed two-lane FMAs
// (even and odd dims in the two halves).
#include <math.h>

#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tmap.h"

namespace w8a8 {

// Set (first code wins) when a bounded wait of the decode attention kernel
// gives up: 21 = a chunk's TMA loads did not land in time, 22 = the drain
// of the loads still in flight after that also timed out.
__device__ int g_w8a8_attn_error = 0;

cudaError_t consume_attention_error(int* code) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_w8a8_attn_error, sizeof(int));
  if (e == cudaSuccess && v != 0) {
    const int z = 0;
    e = cudaMemcpyToSymbol(g_w8a8_attn_error, &z, sizeof(int));
  }
  *code = v;
  return e;
}

namespace {

constexpr int AT_D = 128;
constexpr int AT_WARPS = 4;
constexpr int AT_THREADS = 32 * AT_WARPS;
constexpr int AT_U = 4;                            // tokens per lane group per chunk
constexpr int AT_CHUNK = 4 * AT_U;                 // tokens per chunk (4 lane groups)
constexpr int AT_STAGES = 4;                       // ring depth per warp
constexpr int AT_TILE = AT_CHUNK * AT_D;           // bytes of K (or of V) per chunk
constexpr int AT_STAGE = 2 * AT_TILE;              // K tile, then V tile
constexpr int AT_RING = AT_STAGES * AT_STAGE;      // per warp
constexpr int AT_BAR_OFF = AT_WARPS * AT_RING;     // mbarriers after the rings
constexpr int AT_SPLIT = 4;                        // CTAs (one cluster) per slice
constexpr int AT_DYN_SMEM = AT_BAR_OFF + AT_WARPS * AT_STAGES * 8;
constexpr uint64_t AT_WAIT_LIMIT_NS = 2000000000ull;
static_assert(AT_TILE % 128 == 0 && AT_STAGE % 128 == 0, "TMA destinations stay 128-byte aligned");

// 16 codes (one 16-byte vector) -> 8 pairs (even dim, odd dim), exactly.
__device__ __forceinline__ void decode16(const uint4& c, float2 (&f)[8]) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i + 0] = e4m3x2_to_float2((uint16_t)(w[i] & 0xFFFFu));
    f[2 * i + 1] = e4m3x2_to_float2((uint16_t)(w[i] >> 16));
  }
}

__device__ __forceinline__ uint16_t bf16_rn(float x) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
  return r;
}

// Thread-block cluster helpers: a full cluster barrier (release / acquire,
// so shared-memory writes before it are visible to every CTA after it) and
// a load from the shared memory of another CTA of the cluster.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ float ld_cluster_f32(const float* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(ptx::smem_addr(p)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(r) : "memory");
  return v;
}

// Factors that bring two online-softmax states (running maxima m, m2 in
// log2 units; -inf for an empty state) to their common maximum.
__device__ __forceinline__ float2 merge_factors(float m, float m2, float& mt) {
  mt = fmaxf(m, m2);
  return make_float2(m == -INFINITY ? 0.0f : exp2f(m - mt), m2 == -INFINITY ? 0.0f : exp2f(m2 - mt));
}

}  // namespace

template <int GH>
__global__ void __cluster_dims__(AT_SPLIT, 1, 1) __launch_bounds__(AT_THREADS, 2)
    decode_attention_kernel(const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v,
                            const uint8_t* __restrict__ q, const float* __restrict__ sq_p,
                            const float* __restrict__ sk_p, const float* __restrict__ sv_p,
                            const int32_t* __restrict__ lens, int64_t smax, int hq, int hkv,
                            int hgroups, float softmax_scale, uint16_t* __restrict__ out) {
  extern __shared__ __align__(1024) uint8_t at_smem[];
  __shared__ float s_acc[AT_WARPS][GH][AT_D];
  __shared__ float s_ml[AT_WARPS][GH][2];
  __shared__ float s_ca[GH][AT_D];  // this CTA's merged state, read by the cluster
  __shared__ float s_cm[GH][2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane >> 3, l8 = lane & 7;
  const int rank = blockIdx.x % AT_SPLIT;  // rank in the cluster (clusters run along x)
  const int unit = blockIdx.x / AT_SPLIT;
  const int hg = unit % hgroups;
  const int64_t bk = unit / hgroups;
  const int kh = (int)(bk % hkv);
  const int64_t b = bk / hkv;
  const int h0 = kh * (hq / hkv) + hg * GH;  // first query head of this CTA
  // lengths are device data the host cannot check: clamp to [0, smax]
  const int len = (int)min((int64_t)max(lens[b], 0), smax);

  // the cluster's CTAs split the tokens into AT_SPLIT contiguous parts,
  // and each CTA's warps split its part into AT_WARPS
  const int pc = (len + AT_SPLIT - 1) / AT_SPLIT;
  const int c_lo = min(len, rank * pc), c_hi = min(len, c_lo + pc);
  const int per = (c_hi - c_lo + AT_WARPS - 1) / AT_WARPS;
  const int t0 = min(c_hi, c_lo + warp * per), t1 = min(c_hi, t0 + per);
  const int nch = (t1 - t0 + AT_CHUNK - 1) / AT_CHUNK;
  const uint32_t ring = ptx::smem_addr(at_smem) + warp * AT_RING;
  const uint32_t bar0 = ptx::smem_addr(at_smem) + AT_BAR_OFF + warp * AT_STAGES * 8;
  // cache row of token t of this sequence is b * smax + t (fits: checked on the host)
  const int row0 = (int)(b * smax) + t0;
  const int x0 = kh * AT_D;  // byte column of this KV head: a multiple of 128

  auto issue = [&](int c) {
    const uint32_t st = ring + (c % AT_STAGES) * AT_STAGE;
    const uint32_t bar = bar0 + (c % AT_STAGES) * 8;
    ptx::mbar_arrive_expect_tx(bar, AT_STAGE);
    ptx::tma_load_2d(st, &tm_k, bar, x0, row0 + c * AT_CHUNK);
    ptx::tma_load_2d(st + AT_TILE, &tm_v, bar, x0, row0 + c * AT_CHUNK);
  };
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < AT_STAGES; ++s) ptx::mbar_init(bar0 + s * 8, 1);
    ptx::fence_mbar_init();
    for (int c = 0; c < AT_STAGES && c < nch; ++c) issue(c);
  }

  // query slice, all factors folded in: scores come out in log2 units
  const float qk = softmax_scale * sq_p[0] * sk_p[0] * 1.4426950408889634f;
  float2 qf[GH][8];
#pragma unroll
  for (int h = 0; h < GH; ++h) {
    const uint4 c = *reinterpret_cast<const uint4*>(q + ((b * hq) + h0 + h) * AT_D + 16 * l8);
    decode16(c, qf[h]);
#pragma unroll
    for (int i = 0; i < 8; ++i) qf[h][i] = __fmul2_rn(qf[h][i], make_float2(qk, qk));
  }
  float m[GH], l[GH];
  float2 acc[GH][8];
#pragma unroll
  for (int h = 0; h < GH; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[h][i] = make_float2(0.0f, 0.0f);
  }
  __syncwarp();  // the barriers are initialised before any lane polls them

  // Every lane runs the same chunks (the warp-wide shuffles below need all
  // 32 lanes); a lane group whose token is past the end skips the update.
  int c = 0;
  bool ok = true;
  for (; c < nch; ++c) {
    const int s = c % AT_STAGES;
    const bool landed = ptx::mbar_wait(bar0 + s * 8, (uint32_t)(c / AT_STAGES) & 1u, AT_WAIT_LIMIT_NS);
    if (!__all_sync(0xFFFFFFFFu, landed)) {
      ok = false;
      break;
    }
    const uint32_t st = ring + s * AT_STAGE;
    const int tc = t0 + c * AT_CHUNK;
    // the scores of the lane group's AT_U tokens for every head: independent
    // chains, reduced over the 8 lanes of the group together
    float sc[AT_U][GH];
#pragma unroll
    for (int u = 0; u < AT_U; ++u) {
      float2 kf[8];
      decode16(ptx::lds128(st + (grp + 4 * u) * AT_D + 16 * l8), kf);
#pragma unroll
      for (int h = 0; h < GH; ++h) {
        float2 a = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int i = 0; i < 8; ++i) a = __ffma2_rn(qf[h][i], kf[i], a);
        sc[u][h] = a.x + a.y;
      }
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1)
#pragma unroll
      for (int u = 0; u < AT_U; ++u)
#pragma unroll
        for (int h = 0; h < GH; ++h) sc[u][h] += __shfl_xor_sync(0xFFFFFFFFu, sc[u][h], o);
    // one online-softmax step per head over the chunk's tokens: the running
    // maximum moves to the chunk's maximum (a factor of exactly 1 when it
    // does not move), then each valid token adds its weight
    float pw[AT_U][GH];
#pragma unroll
    for (int h = 0; h < GH; ++h) {
      float mx = m[h];
#pragma unroll
      for (int u = 0; u < AT_U; ++u)
        if (tc + grp + 4 * u < t1) mx = fmaxf(mx, sc[u][h]);
      const float ms = mx == -INFINITY ? 0.0f : mx;  // no token yet: nothing to weigh
      const float cr = exp2f(m[h] - ms);
      float ps = 0.0f;
#pragma unroll
      for (int u = 0; u < AT_U; ++u) {
        pw[u][h] = tc + grp + 4 * u < t1 ? exp2f(sc[u][h] - ms) : 0.0f;
        ps += pw[u][h];
      }
      l[h] = __fmaf_rn(l[h], cr, ps);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[h][i] = __fmul2_rn(acc[h][i], make_float2(cr, cr));
      m[h] = mx;
    }
#pragma unroll
    for (int u = 0; u < AT_U; ++u) {
      float2 vf[8];
      decode16(ptx::lds128(st + AT_TILE + (grp + 4 * u) * AT_D + 16 * l8), vf);
#pragma unroll
      for (int h = 0; h < GH; ++h)
#pragma unroll
        for (int i = 0; i < 8; ++i)
          acc[h][i] = __ffma2_rn(make_float2(pw[u][h], pw[u][h]), vf[i], acc[h][i]);
    }
    // every lane has used this stage: lane 0 refills it with chunk c + AT_STAGES
    __syncwarp();
    if (lane == 0 && c + AT_STAGES < nch) {
      ptx::fence_proxy_async_smem();
      issue(c + AT_STAGES);
    }
  }
  if (!ok && lane == 0) {
    // chunks c .. c + AT_STAGES - 1 may still be in flight: let them land
    // (bounded) before the shared memory is given up
    atomicCAS(&g_w8a8_attn_error, 0, 21);
    for (int j = c; j < nch && j < c + AT_STAGES; ++j)
      if (!ptx::mbar_wait(bar0 + (j % AT_STAGES) * 8, (uint32_t)(j / AT_STAGES) & 1u,
                          AT_WAIT_LIMIT_NS))
        atomicCAS(&g_w8a8_attn_error, 0, 22);
  }

  // merge the 4 lane groups of the warp (lanes with equal l8 hold equal dims)
#pragma unroll
  for (int o = 8; o < 32; o <<= 1) {
#pragma unroll
    for (int h = 0; h < GH; ++h) {
      const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m[h], o);
      const float l2 = __shfl_xor_sync(0xFFFFFFFFu, l[h], o);
      float mt;
      const float2 f = merge_factors(m[h], m2, mt);
      l[h] = l[h] * f.x + l2 * f.y;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float ax = __shfl_xor_sync(0xFFFFFFFFu, acc[h][i].x, o);
        const float ay = __shfl_xor_sync(0xFFFFFFFFu, acc[h][i].y, o);
        acc[h][i].x = acc[h][i].x * f.x + ax * f.y;
        acc[h][i].y = acc[h][i].y * f.x + ay * f.y;
      }
      m[h] = mt;
    }
  }
  if (grp == 0) {
#pragma unroll
    for (int h = 0; h < GH; ++h) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        s_acc[warp][h][16 * l8 + 2 * i] = acc[h][i].x;
        s_acc[warp][h][16 * l8 + 2 * i + 1] = acc[h][i].y;
      }
      if (l8 == 0) {
        s_ml[warp][h][0] = m[h];
        s_ml[warp][h][1] = l[h];
      }
    }
  }
  __syncthreads();
  // merge the warps in a fixed order: thread d holds dim d of every head
  const int d = threadIdx.x;
#pragma unroll
  for (int h = 0; h < GH; ++h) {
    float mm = -INFINITY, ll = 0.0f, aa = 0.0f;
#pragma unroll
    for (int w = 0; w < AT_WARPS; ++w) {
      float mt;
      const float2 f = merge_factors(mm, s_ml[w][h][0], mt);
      ll = ll * f.x + s_ml[w][h][1] * f.y;
      aa = aa * f.x + s_acc[w][h][d] * f.y;
      mm = mt;
    }
    s_ca[h][d] = aa;
    if (d == 0) {
      s_cm[h][0] = mm;
      s_cm[h][1] = ll;
    }
  }
  // then the cluster's CTAs in rank order: CTA r finishes heads r, r + AT_SPLIT, ...
  cluster_sync_all();
  const float sv = sv_p[0];
  for (int h = rank; h < GH; h += AT_SPLIT) {
    float mm = -INFINITY, ll = 0.0f, aa = 0.0f;
#pragma unroll
    for (int r = 0; r < AT_SPLIT; ++r) {
      float mt;
      const float2 f = merge_factors(mm, ld_cluster_f32(&s_cm[h][0], r), mt);
      ll = ll * f.x + ld_cluster_f32(&s_cm[h][1], r) * f.y;
      aa = aa * f.x + ld_cluster_f32(&s_ca[h][d], r) * f.y;
      mm = mt;
    }
    const float y = ll > 0.0f ? aa / ll * sv : 0.0f;
    out[((b * hq) + h0 + h) * AT_D + d] = bf16_rn(y);
  }
  cluster_sync_all();  // no CTA leaves while another may still read its shared memory
}

template <int GH>
static cudaError_t launch_attn(const CUtensorMap& tm_k, const CUtensorMap& tm_v, const uint8_t* q,
                               const float* sq, const float* sk, const float* sv,
                               const int32_t* lens, int64_t smax, int hq, int hkv, int hgroups,
                               float softmax_scale, uint16_t* out, unsigned grid,
                               cudaStream_t st) {
  static bool configured[64] = {};  // the attribute belongs to each device's context
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(decode_attention_kernel<GH>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, AT_DYN_SMEM);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  decode_attention_kernel<GH><<<grid, AT_THREADS, AT_DYN_SMEM, st>>>(
      tm_k, tm_v, q, sq, sk, sv, lens, smax, hq, hkv, hgroups, softmax_scale, out);
  return cudaGetLastError();
}

cudaError_t launch_decode_attention(const uint8_t* q, const float* sq, const uint8_t* k,
                                    const float* sk, const uint8_t* v, const float* sv,
                                    const int32_t* lens, int64_t batch, int64_t smax, int hq,
                                    int hkv, float softmax_scale, uint16_t* out,
                                    cudaStream_t st) {
  if (batch == 0) return cudaSuccess;
  const int g = hq / hkv;
  const int gh = g >= 4 ? 4 : g;
  const int hgroups = g / gh;
  const int64_t grid = batch * hkv * hgroups * AT_SPLIT;
  // TMA row coordinates are 32-bit: the last chunk may start AT_CHUNK rows
  // before batch * smax and run past it (those rows read as zero)
  if (grid > 0x7FFFFFFFLL || batch * smax > 0x7FFFFFFFLL - AT_CHUNK) return cudaErrorInvalidValue;
  // K and V as 2-D row-major [batch * smax, hkv * 128] byte matrices; a box
  // is 16 token rows of one KV head
  CUtensorMap tm_k, tm_v;
  const uint64_t rows = (uint64_t)(batch * smax), cols = (uint64_t)hkv * AT_D;
  if (rows == 0) {
    // no tokens at all: the kernel issues no load, but a map needs a row
    if (!make_tmap_2d(&tm_k, k, 1, 1, cols, AT_CHUNK, AT_D, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_tmap_2d(&tm_v, v, 1, 1, cols, AT_CHUNK, AT_D, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  } else if (!make_tmap_2d(&tm_k, k, 1, rows, cols, AT_CHUNK, AT_D, CU_TENSOR_MAP_SWIZZLE_NONE) ||
             !make_tmap_2d(&tm_v, v, 1, rows, cols, AT_CHUNK, AT_D, CU_TENSOR_MAP_SWIZZLE_NONE)) {
    return cudaErrorInvalidValue;
  }
  switch (gh) {
    case 1:
      return launch_attn<1>(tm_k, tm_v, q, sq, sk, sv, lens, smax, hq, hkv, hgroups, softmax_scale,
                            out, (unsigned)grid, st);
    case 2:
      return launch_attn<2>(tm_k, tm_v, q, sq, sk, sv, lens, smax, hq, hkv, hgroups, softmax_scale,
                            out, (unsigned)grid, st);
    default:
      return launch_attn<4>(tm_k, tm_v, q, sq, sk, sv, lens, smax, hq, hkv, hgroups, softmax_scale,
                            out, (unsigned)grid, st);
  }
}

}  // namespace w8a8
