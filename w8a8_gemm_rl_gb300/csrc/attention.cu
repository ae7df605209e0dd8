// attention.cu -- decode attention over the FP8 KV cache (NeMo RL FP8 blog,
// Table 3 and the FP8 KV-cache section: Q, K and V carry one FP32 scale each;
// FP8-RL section 4: attention reads the FP8 KV cache):
//
//   score_t = softmax_scale * sq * sk * sum_d dec(q[b,h,d]) * dec(k[b,t,kh,d])
//   out_d   = sv * sum_{t < len_b} softmax(score)_t * dec(v[b,t,kh,d])
//
// one query token per sequence, grouped-query heads (query head h reads KV
// head h / (hq / hkv)), head dim 128.  A cluster of 1 to 8 CTAs (chosen at
// launch from the number of slices) reads one (sequence, KV head) slice of
// K and V exactly once for up to 8 query heads, so the kernel streams the
// cache and is HBM-bound.
//
// Each CTA takes a contiguous part of the slice's tokens and each of its 4
// warps a contiguous quarter of that, streamed through the warp's own ring
// of shared-memory stages: two TMA tile loads per chunk of 32 tokens (the
// 128-byte rows of one KV head sit hkv * 128 bytes apart in the cache, a
// 2-D box of 32 rows x 128 bytes, stored with the 128-byte swizzle so that
// the 8-row matrix loads below hit distinct banks).  Lane 0 keeps
// AT_STAGES - 1 chunks in flight while the warp computes on the oldest.
//
// Both contractions of a chunk run on the tensor cores (mma.sync), with the
// query heads as the MMA rows:
//   S[h, t] = sum_d q[h, d] k[t, d]: m16n8k32 on the raw E4M3 codes (the
//     products are exact, f32 accumulation); K fragments come from the
//     stage by ldmatrix, rows 8-15 of A are zero;
//   O[h, d] += P[h, t] v[t, d]: m16n8k16 in f16 with f32 accumulation.  The
//     accumulator of S is already laid out as the A operand P; V fragments
//     come from ldmatrix.trans on the raw tile, a byte permute and one
//     exact widening to f16.  P = 2^15 p is split into two f16 parts (hi +
//     lo carries 22 bits of it, so the weights lose nothing that binary32
//     would keep): the high parts fill A rows 0-7 and the low parts rows
//     8-15, so one MMA carries both.
// The softmax is online, in log2 units, one step per chunk per head.  The
// warps' states, then the cluster's CTAs' states (through distributed
// shared memory), are merged at the end.
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
constexpr int AT_CHUNK = 32;                       // tokens per chunk (a multiple of 16)
constexpr int AT_NT = AT_CHUNK / 8;                // 8-token n tiles of S per chunk
constexpr int AT_STAGES = 3;                       // ring depth per warp
constexpr int AT_TILE = AT_CHUNK * AT_D;           // bytes of K (or of V) per chunk
constexpr int AT_STAGE = 2 * AT_TILE;              // K tile, then V tile
constexpr int AT_RING = AT_STAGES * AT_STAGE;      // per warp
constexpr int AT_BAR_OFF = AT_WARPS * AT_RING;     // mbarriers after the rings
constexpr int AT_MAX_SPLIT = 8;                    // CTAs (one cluster) per slice, at most
// + 1024: the rings start at the first 1024-byte boundary of the dynamic
// shared memory (which follows the kernel's static shared arrays)
constexpr int AT_DYN_SMEM = AT_BAR_OFF + AT_WARPS * AT_STAGES * 8 + 1024;
constexpr uint64_t AT_WAIT_LIMIT_NS = 2000000000ull;
constexpr float AT_P_LOG2 = 15.0f;                 // weights are formed as 2^15 p <= 2^15
static_assert(AT_TILE % 1024 == 0 && AT_STAGE % 1024 == 0 && AT_RING % 1024 == 0,
              "128-byte-swizzled tiles start on 1024-byte boundaries");

// four E4M3 codes (bytes 0..3) -> f16x2 of bytes 0, 1 and f16x2 of bytes 2, 3,
// exactly (every E4M3 value is an f16 value)
__device__ __forceinline__ void e4m3x4_f16x2x2(uint32_t c, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(c));
}
// 2^x by the hardware approximation (an error of a few ulp, far inside the
// tolerance the parity tests hold; 0 for x = -inf and for results below the
// normal range)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// (lo, hi) -> f16x2 with lo in the low half, round to nearest even
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float2 unpack_f16x2(uint32_t h2) {
  float lo, hi;
  asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(h2));
  return make_float2(lo, hi);
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
// d += A B on one full m16n8k16 tile (f16 in, f32 accumulate): a0 / a2 the
// fragments of row g, a1 / a3 those of row g + 8; d0, d1 row g, d2, d3 row g + 8.
__device__ __forceinline__ void mma_rows16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                           uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// (d0, d1) += A B on one m16n8k32 tile of E4M3 codes (f32 accumulate)
// whose A rows 8..15 are zero (their results are dropped): a0 / a2 hold
// bytes 4 tig .. 4 tig + 3 of the two 16-byte halves of row g's k range,
// b0 / b1 the same of column g.
__device__ __forceinline__ void mma_e4m3_rows8(float& d0, float& d1, uint32_t a0, uint32_t a2,
                                               uint32_t b0, uint32_t b1) {
  asm("{\n\t.reg .f32 z2, z3;\n\t"
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, z2, z3}, {%2, %3, %4, %3}, "
      "{%5, %6}, {%0, %1, %7, %7};\n\t}"
      : "+f"(d0), "+f"(d1)
      : "r"(a0), "r"(0u), "r"(a2), "r"(b0), "r"(b1), "f"(0.0f));
}

// d += A B on one full m16n8k32 tile of E4M3 codes (f32 accumulate): a[0] /
// a[2] bytes 4 tig .. 4 tig + 3 of the two 16-byte halves of row g's k
// range, a[1] / a[3] the same of row g + 8; d[0], d[1] row g, d[2], d[3] row
// g + 8.
__device__ __forceinline__ void mma_e4m3_rows16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                                uint32_t b1) {
  asm("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
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
__global__ void __launch_bounds__(AT_THREADS, 2)
    decode_attention_kernel(const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v,
                            const uint8_t* __restrict__ q, const float* __restrict__ sq_p,
                            const float* __restrict__ sk_p, const float* __restrict__ sv_p,
                            const int32_t* __restrict__ lens, int64_t smax, int hq, int hkv,
                            int hgroups, int nsplit, float softmax_scale,
                            uint16_t* __restrict__ out) {
  extern __shared__ __align__(16) uint8_t at_smem[];
  __shared__ float s_acc[AT_WARPS][GH][AT_D];
  __shared__ float s_ml[AT_WARPS][GH][2];
  __shared__ float s_ca[GH][AT_D];  // this CTA's merged state, read by the cluster
  __shared__ float s_cm[GH][2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;  // fragment row (query head) and column pair
  const int rank = blockIdx.x % nsplit;  // rank in the cluster of nsplit CTAs (along x)
  const int unit = blockIdx.x / nsplit;
  const int hg = unit % hgroups;
  const int64_t bk = unit / hgroups;
  const int kh = (int)(bk % hkv);
  const int64_t b = bk / hkv;
  const int h0 = kh * (hq / hkv) + hg * GH;  // first query head of this CTA
  // lengths are device data the host cannot check: clamp to [0, smax]
  const int len = (int)min((int64_t)max(lens[b], 0), smax);

  // the cluster's CTAs split the tokens into nsplit contiguous parts, and
  // each CTA's warps split its part into AT_WARPS
  const int pc = (len + nsplit - 1) / nsplit;
  const int c_lo = min(len, rank * pc), c_hi = min(len, c_lo + pc);
  const int per = (c_hi - c_lo + AT_WARPS - 1) / AT_WARPS;
  const int t0 = min(c_hi, c_lo + warp * per), t1 = min(c_hi, t0 + per);
  const int nch = (t1 - t0 + AT_CHUNK - 1) / AT_CHUNK;
  const uint32_t base = (ptx::smem_addr(at_smem) + 1023u) & ~1023u;  // swizzle atoms: 1024-aligned
  const uint32_t ring = base + warp * AT_RING;
  const uint32_t bar0 = base + AT_BAR_OFF + warp * AT_STAGES * 8;
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

  // Q as the A operand of S = Q K^T (raw E4M3 codes), row g = query head
  // h0 + g (zero past GH); k step ks covers dims 32 ks .. 32 ks + 31
  uint32_t qa[4][2];
#pragma unroll
  for (int ks = 0; ks < 4; ++ks)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
      qa[ks][hh] = g < GH ? *reinterpret_cast<const uint32_t*>(q + ((b * hq) + h0 + g) * AT_D +
                                                              32 * ks + 16 * hh + 4 * tig)
                          : 0u;
  const float qk = softmax_scale * sq_p[0] * sk_p[0] * 1.4426950408889634f;
  // online-softmax state of head g (the 4 lanes of a row agree on m; each
  // sums its own tokens into l), and O[g, d] for d = 16 s + 4 tig + e + 2 i
  // in two parts: acc[s][e][i] from the high halves of the weights (MMA row
  // g), acc[s][e][2 + i] from the low halves (row g + 8)
  float m = -INFINITY, l = 0.0f;
  float acc[8][2][4];
#pragma unroll
  for (int s = 0; s < 8; ++s)
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[s][e][i] = 0.0f;
  __syncwarp();  // the barriers are initialised before any lane polls them

  // ldmatrix row address of this lane inside a tile: matrix lane / 8 holds
  // tokens 8 ((lane / 8) & 1) + 0..7 of segment pair base + lane / 16; the
  // 128-byte swizzle stores 16-byte chunk c of row r at chunk c ^ (r & 7)
  const int mrow = (lane & 7) + ((lane >> 3) & 1) * 8;
  const int mseg = lane >> 4;

  int c = 0;
  bool ok = true;
  for (; c < nch; ++c) {
    const int s = c % AT_STAGES;
    const bool landed = ptx::mbar_wait(bar0 + s * 8, (uint32_t)(c / AT_STAGES) & 1u, AT_WAIT_LIMIT_NS);
    if (!__all_sync(0xFFFFFFFFu, landed)) {
      ok = false;
      break;
    }
    const uint32_t tk = ring + s * AT_STAGE, tv = tk + AT_TILE;
    const int tc = t0 + c * AT_CHUNK;

    // S for the chunk: n tile j holds tokens 8 j + 0..7; this lane gets
    // head g, tokens 8 j + 2 tig + {0, 1}.  Two partial sums per tile (even
    // and odd k steps) keep more MMA chains in flight.
    float sp2[2][AT_NT][2] = {};
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
#pragma unroll
      for (int tb = 0; tb < AT_CHUNK / 16; ++tb) {
        // tokens 16 tb + 0-7 / 8-15 of segment 2 ks, then of segment 2 ks + 1
        uint32_t r[4];
        const int row = 16 * tb + mrow;
        ldsm_x4(tk + row * AT_D + (((2 * ks + mseg) ^ (row & 7)) << 4), r);
#pragma unroll
        for (int jj = 0; jj < 2; ++jj)
          mma_e4m3_rows8(sp2[ks & 1][2 * tb + jj][0], sp2[ks & 1][2 * tb + jj][1], qa[ks][0],
                         qa[ks][1], r[jj], r[jj + 2]);
      }
    float sc[AT_NT][2];
#pragma unroll
    for (int j = 0; j < AT_NT; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) sc[j][e] = sp2[0][j][e] + sp2[1][j][e];
    // one online-softmax step over the chunk: scores in log2 units, tokens
    // past the end weigh nothing; the maximum covers the chunk's first
    // token, so it is finite
    float mx = m;
    if (tc + AT_CHUNK <= t1) {  // a full chunk (all but a warp's last)
#pragma unroll
      for (int j = 0; j < AT_NT; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          sc[j][e] *= qk;
          mx = fmaxf(mx, sc[j][e]);
        }
    } else {
#pragma unroll
      for (int j = 0; j < AT_NT; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float x = tc + 8 * j + 2 * tig + e < t1 ? sc[j][e] * qk : -INFINITY;
          sc[j][e] = x;
          mx = fmaxf(mx, x);
        }
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
    // 0 for the first step, exactly 1 while the maximum holds
    const float cr = m == mx ? 1.0f : ex2_approx(m - mx);
    float pp[AT_NT][2], ps = 0.0f;
#pragma unroll
    for (int j = 0; j < AT_NT; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        pp[j][e] = ex2_approx(sc[j][e] - mx + AT_P_LOG2);
        ps += pp[j][e];
      }
    l = __fmaf_rn(l, cr, ps);
    m = mx;
    if (__any_sync(0xFFFFFFFFu, cr != 1.0f)) {
#pragma unroll
      for (int s2 = 0; s2 < 8; ++s2)
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[s2][e][i] *= cr;
    }
    // P in the A layout of O += P V, one k16 step per 16 tokens (k slots =
    // the tokens, where the S tiles left them), as hi + lo f16 parts: the
    // high parts in rows 0-7 and the low parts in rows 8-15 of one tile, so
    // one MMA carries both
#pragma unroll
    for (int kk = 0; kk < AT_CHUNK / 16; ++kk) {
      const uint32_t ph0 = pack_f16x2(pp[2 * kk][0], pp[2 * kk][1]);
      const uint32_t ph1 = pack_f16x2(pp[2 * kk + 1][0], pp[2 * kk + 1][1]);
      const float2 f0 = unpack_f16x2(ph0), f1 = unpack_f16x2(ph1);
      const uint32_t pl0 = pack_f16x2(pp[2 * kk][0] - f0.x, pp[2 * kk][1] - f0.y);
      const uint32_t pl1 = pack_f16x2(pp[2 * kk + 1][0] - f1.x, pp[2 * kk + 1][1] - f1.y);
#pragma unroll
      for (int sp = 0; sp < 8; sp += 2) {
        // transposed: tokens 16 kk + 2 tig + {0, 1} (+ 8) of dims 2 g, 2 g + 1 of a segment
        uint32_t r[4];
        const int row = 16 * kk + mrow;
        ldsm_x4_trans(tv + row * AT_D + (((sp + mseg) ^ (row & 7)) << 4), r);
#pragma unroll
        for (int hs = 0; hs < 2; ++hs) {
          const int seg = sp + hs;
          // bytes (t, 2g) (t, 2g+1) (t+1, 2g) (t+1, 2g+1) -> (t, 2g) (t+1, 2g) | (t, 2g+1) (t+1, 2g+1)
          const uint32_t x0v = __byte_perm(r[2 * hs], 0u, 0x3120u);
          const uint32_t x1v = __byte_perm(r[2 * hs + 1], 0u, 0x3120u);
          uint32_t b0[2], b1[2];  // [e]: n tile of dims 16 seg + 2 n + e
          e4m3x4_f16x2x2(x0v, b0[0], b0[1]);
          e4m3x4_f16x2x2(x1v, b1[0], b1[1]);
#pragma unroll
          for (int e = 0; e < 2; ++e) mma_rows16(acc[seg][e], ph0, pl0, ph1, pl1, b0[e], b1[e]);
        }
      }
    }
    // every lane has used this stage (each ldmatrix result has fed an MMA
    // issued above, so the reads are complete): lane 0 refills it with
    // chunk c + AT_STAGES
    __syncwarp();
    if (lane == 0 && c + AT_STAGES < nch) issue(c + AT_STAGES);
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

  // the warp's state: l summed over the 4 lanes of each row
  l += __shfl_xor_sync(0xFFFFFFFFu, l, 1);
  l += __shfl_xor_sync(0xFFFFFFFFu, l, 2);
  if (g < GH) {
#pragma unroll
    for (int s2 = 0; s2 < 8; ++s2)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        s_acc[warp][g][16 * s2 + 4 * tig + e] = acc[s2][e][0] + acc[s2][e][2];
        s_acc[warp][g][16 * s2 + 4 * tig + e + 2] = acc[s2][e][1] + acc[s2][e][3];
      }
    if (tig == 0) {
      s_ml[warp][g][0] = m;
      s_ml[warp][g][1] = l;
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
  // then the cluster's CTAs in rank order: CTA r finishes heads r, r + nsplit, ...
  cluster_sync_all();
  const float sv = sv_p[0];
  for (int h = rank; h < GH; h += nsplit) {
    float mm = -INFINITY, ll = 0.0f, aa = 0.0f;
    for (int r = 0; r < nsplit; ++r) {
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
                               int nsplit, float softmax_scale, uint16_t* out, unsigned grid,
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(AT_THREADS);
  cfg.dynamicSmemBytes = AT_DYN_SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)nsplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_attention_kernel<GH>, tm_k, tm_v, q, sq, sk, sv, lens,
                            smax, hq, hkv, hgroups, nsplit, softmax_scale, out);
}

cudaError_t launch_decode_attention(const uint8_t* q, const float* sq, const uint8_t* k,
                                    const float* sk, const uint8_t* v, const float* sv,
                                    const int32_t* lens, int64_t batch, int64_t smax, int hq,
                                    int hkv, float softmax_scale, uint16_t* out,
                                    cudaStream_t st) {
  if (batch == 0) return cudaSuccess;
  const int g = hq / hkv;
  // query heads per CTA: the 8 used rows of the MMA tiles when they divide
  // the group, else 4, else the whole group (1 or 2)
  const int gh = g % 8 == 0 ? 8 : (g % 4 == 0 ? 4 : g);
  const int hgroups = g / gh;
  // CTAs per slice (measured on the 32 x 8192 x 8 x 128 cache and its
  // neighbours): each extra CTA costs a pipeline fill and a merge, so split
  // finely only while SMs would otherwise idle; around one or two slices
  // per SM take them whole (long ones in 4 parts, which pays for the
  // fills), beyond that in 2 parts for a finer balance over the SMs
  const int64_t units = batch * hkv * hgroups;
  const int64_t sms = sm_count();
  int nsplit;
  if (units * 4 <= sms)
    nsplit = AT_MAX_SPLIT;
  else if (units * 2 <= sms)
    nsplit = 4;
  else if (units <= sms)
    nsplit = 2;
  else if (units <= 2 * sms)
    nsplit = smax >= 16384 ? 4 : 1;
  else
    nsplit = 2;
  const int64_t grid = units * nsplit;
  // TMA row coordinates are 32-bit: the last chunk may start AT_CHUNK rows
  // before batch * smax and run past it (those rows read as zero)
  if (grid > 0x7FFFFFFFLL || batch * smax > 0x7FFFFFFFLL - AT_CHUNK) return cudaErrorInvalidValue;
  // K and V as 2-D row-major [batch * smax, hkv * 128] byte matrices; a box
  // is 16 token rows of one KV head, stored with the 128-byte swizzle
  CUtensorMap tm_k, tm_v;
  const uint64_t rows = (uint64_t)(batch * smax), cols = (uint64_t)hkv * AT_D;
  if (rows == 0) {
    // no tokens at all: the kernel issues no load, but a map needs a row
    if (!make_tmap_2d(&tm_k, k, 1, 1, cols, AT_CHUNK, AT_D, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_2d(&tm_v, v, 1, 1, cols, AT_CHUNK, AT_D, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  } else if (!make_tmap_2d(&tm_k, k, 1, rows, cols, AT_CHUNK, AT_D, CU_TENSOR_MAP_SWIZZLE_128B) ||
             !make_tmap_2d(&tm_v, v, 1, rows, cols, AT_CHUNK, AT_D, CU_TENSOR_MAP_SWIZZLE_128B)) {
    return cudaErrorInvalidValue;
  }
  switch (gh) {
    case 1:
      return launch_attn<1>(tm_k, tm_v, q, sq, sk, sv, lens, smax, hq, hkv, hgroups, nsplit,
                            softmax_scale, out, (unsigned)grid, st);
    case 2:
      return launch_attn<2>(tm_k, tm_v, q, sq, sk, sv, lens, smax, hq, hkv, hgroups, nsplit,
                            softmax_scale, out, (unsigned)grid, st);
    case 4:
      return launch_attn<4>(tm_k, tm_v, q, sq, sk, sv, lens, smax, hq, hkv, hgroups, nsplit,
                            softmax_scale, out, (unsigned)grid, st);
    default:
      return launch_attn<8>(tm_k, tm_v, q, sq, sk, sv, lens, smax, hq, hkv, hgroups, nsplit,
                            softmax_scale, out, (unsigned)grid, st);
  }
}


// ================================================================ prefill
// Causal prefill attention (NeMo RL FP8 blog, Table 3: per-tensor Q, K and V
// scales): the prompt's tokens attend to their sequence's tokens up to
// themselves,
//   score_j = softmax_scale * sq * sk * sum_d dec(q[b,i,h,d]) * dec(k[b,j,kh,d])
//   out_d   = sv * sum_{j <= i} softmax(score)_j * dec(v[b,j,kh,d]),
// q [batch, seq, hq, 128], k and v [batch, seq, hkv, 128] (the KV cache's
// layout), out [batch, seq, hq, 128] BF16.
//
// A CTA takes 64 query tokens of one (sequence, query head); each of its 4
// warps 16 of them, as the rows of m16 MMA tiles.  The keys come in chunks
// of 64 tokens (K and V tiles by TMA, 128-byte swizzle, a 3-stage ring
// shared by the warps): S = Q K^T on the raw E4M3 codes (m16n8k32, f32
// accumulation), one online-softmax step per chunk in log2 units, then
// O += P V in f16 with the weights P = 2^15 p split into high and low f16
// parts (two MMAs; together they carry 22 bits of each weight), V widened
// exactly from E4M3.  The diagonal chunk masks the keys after each query.
// Query blocks are launched longest (most keys) first.
namespace {
constexpr int PF_ROWS = 64;                    // query tokens per CTA
constexpr int PF_KEYS = 64;                    // keys per chunk (= PF_ROWS: chunk qb is the diagonal)
constexpr int PF_STAGES = 3;
constexpr int PF_TILE = PF_KEYS * AT_D;        // bytes of K (or of V) per chunk
constexpr int PF_STAGE = 2 * PF_TILE;
constexpr int PF_BAR_OFF = PF_STAGES * PF_STAGE;
constexpr int PF_DYN_SMEM = PF_BAR_OFF + PF_STAGES * 8 + 1024;
static_assert(PF_TILE % 1024 == 0, "128-byte-swizzled tiles start on 1024-byte boundaries");
static_assert(PF_ROWS == 16 * AT_WARPS && PF_KEYS == PF_ROWS, "one diagonal chunk per query block");
}  // namespace

// 3 CTAs per SM (168 registers): 6-7% faster than 2 (180 registers)
__global__ void __launch_bounds__(AT_THREADS, 3)
    prefill_attention_kernel(const __grid_constant__ CUtensorMap tm_k,
                             const __grid_constant__ CUtensorMap tm_v,
                             const uint8_t* __restrict__ q, const float* __restrict__ sq_p,
                             const float* __restrict__ sk_p, const float* __restrict__ sv_p,
                             int seq, int hq, int hkv, int nqb, float softmax_scale,
                             uint16_t* __restrict__ out) {
  extern __shared__ __align__(16) uint8_t at_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;
  const int qb = nqb - 1 - (int)blockIdx.x;  // the longest blocks first
  const int h = (int)blockIdx.y;
  const int64_t b = blockIdx.z;
  const int kh = h / (hq / hkv);
  const int r0 = qb * PF_ROWS + 16 * warp;  // this warp's first query token
  const int nch = qb + 1;                   // key chunks 0 .. qb
  const uint32_t base = (ptx::smem_addr(at_smem) + 1023u) & ~1023u;
  const uint32_t bar0 = base + PF_BAR_OFF;
  // cache row of token t of this sequence is b * seq + t (fits: checked on the host)
  const int krow0 = (int)(b * seq);
  const int x0 = kh * AT_D;
  auto issue = [&](int c) {
    const uint32_t st = base + (c % PF_STAGES) * PF_STAGE;
    const uint32_t bar = bar0 + (c % PF_STAGES) * 8;
    ptx::mbar_arrive_expect_tx(bar, PF_STAGE);
    ptx::tma_load_2d(st, &tm_k, bar, x0, krow0 + c * PF_KEYS);
    ptx::tma_load_2d(st + PF_TILE, &tm_v, bar, x0, krow0 + c * PF_KEYS);
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < PF_STAGES; ++s) ptx::mbar_init(bar0 + s * 8, 1);
    ptx::fence_mbar_init();
    for (int c = 0; c < PF_STAGES && c < nch; ++c) issue(c);
  }
  __syncthreads();  // the barriers are initialised before any thread polls them

  // Q as the A operand of S = Q K^T (raw E4M3 codes): rows g and g + 8 are
  // query tokens r0 + g and r0 + g + 8 (zero past the sequence); k step ks
  // covers dims 32 ks .. 32 ks + 31
  uint32_t qa[4][4];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int tok = r0 + g + 8 * hh;
    const uint8_t* qp = q + (((b * seq + tok) * hq) + h) * (int64_t)AT_D + 4 * tig;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      qa[ks][hh] = tok < seq ? *reinterpret_cast<const uint32_t*>(qp + 32 * ks) : 0u;
      qa[ks][2 + hh] = tok < seq ? *reinterpret_cast<const uint32_t*>(qp + 32 * ks + 16) : 0u;
    }
  }
  const float qk = softmax_scale * sq_p[0] * sk_p[0] * 1.4426950408889634f;
  // online-softmax state of rows g (index 0) and g + 8 (index 1): the 4
  // lanes of a row agree on m, each sums its own keys into l; O[row, d] for
  // d = 16 s + 4 tig + e + 2 i: acc[s][e][i] (row g), acc[s][e][2 + i] (row g + 8)
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.0f, 0.0f};
  float acc[8][2][4];
#pragma unroll
  for (int s = 0; s < 8; ++s)
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[s][e][i] = 0.0f;
  // ldmatrix row address of this lane inside a tile (as in the decode kernel)
  const int mrow = (lane & 7) + ((lane >> 3) & 1) * 8;
  const int mseg = lane >> 4;

  int c = 0;
  bool ok = true;
  for (; c < nch; ++c) {
    const int s = c % PF_STAGES;
    const bool landed = ptx::mbar_wait(bar0 + s * 8, (uint32_t)(c / PF_STAGES) & 1u, AT_WAIT_LIMIT_NS);
    if (!__syncthreads_and(landed ? 1 : 0)) {
      ok = false;
      break;
    }
    const uint32_t tk = base + s * PF_STAGE, tv = tk + PF_TILE;
    const bool diag = c == qb;
    // S for the chunk: n tile j holds keys 64 c + 8 j + 0..7; this lane gets
    // keys 64 c + 8 j + 2 tig + {0, 1} of rows g and g + 8
    float sp[PF_KEYS / 8][4];
#pragma unroll
    for (int j = 0; j < PF_KEYS / 8; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) sp[j][i] = 0.0f;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
#pragma unroll
      for (int tb = 0; tb < PF_KEYS / 16; ++tb) {
        uint32_t r[4];
        const int row = 16 * tb + mrow;
        ldsm_x4(tk + row * AT_D + (((2 * ks + mseg) ^ (row & 7)) << 4), r);
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) mma_e4m3_rows16(sp[2 * tb + jj], qa[ks], r[jj], r[jj + 2]);
      }
    // one online-softmax step per row: scores in log2 units, keys after the
    // query weigh nothing (the diagonal chunk only); every row has key 0 in
    // chunk 0, so its maximum is finite from the first step on
    float mx[2] = {m[0], m[1]};
#pragma unroll
    for (int j = 0; j < PF_KEYS / 8; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int key = c * PF_KEYS + 8 * j + 2 * tig + (i & 1);
        const int row = r0 + g + 8 * (i >> 1);
        const float x = diag && key > row ? -INFINITY : sp[j][i] * qk;
        sp[j][i] = x;
        mx[i >> 1] = fmaxf(mx[i >> 1], x);
      }
    float cr[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xFFFFFFFFu, mx[hh], 1));
      mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xFFFFFFFFu, mx[hh], 2));
      // 0 for the first step, exactly 1 while the maximum holds
      cr[hh] = m[hh] == mx[hh] ? 1.0f : ex2_approx(m[hh] - mx[hh]);
    }
    float ps[2] = {0.0f, 0.0f};
#pragma unroll
    for (int j = 0; j < PF_KEYS / 8; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        sp[j][i] = ex2_approx(sp[j][i] - mx[i >> 1] + AT_P_LOG2);
        ps[i >> 1] += sp[j][i];
      }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      l[hh] = __fmaf_rn(l[hh], cr[hh], ps[hh]);
      m[hh] = mx[hh];
    }
    if (__any_sync(0xFFFFFFFFu, cr[0] != 1.0f || cr[1] != 1.0f)) {
#pragma unroll
      for (int s2 = 0; s2 < 8; ++s2)
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[s2][e][i] *= cr[i >> 1];
    }
    // O += P V, one k16 step per 16 keys: P in the A layout (rows g, g + 8;
    // k slots = the keys, where the S tiles left them), as high and low f16
    // parts, each one MMA against the same V fragments
#pragma unroll
    for (int kk = 0; kk < PF_KEYS / 16; ++kk) {
      uint32_t ah[4], al[4];  // a0: row g keys 0-7 of the step, a1: row g + 8, a2 / a3: keys 8-15
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const float p0 = sp[2 * kk + t][2 * hh], p1 = sp[2 * kk + t][2 * hh + 1];
          const uint32_t hi = pack_f16x2(p0, p1);
          const float2 f = unpack_f16x2(hi);
          ah[2 * t + hh] = hi;
          al[2 * t + hh] = pack_f16x2(p0 - f.x, p1 - f.y);
        }
#pragma unroll
      for (int spg = 0; spg < 8; spg += 2) {
        // transposed: keys 16 kk + 2 tig + {0, 1} (+ 8) of dims 2 g, 2 g + 1 of a segment
        uint32_t r[4];
        const int row = 16 * kk + mrow;
        ldsm_x4_trans(tv + row * AT_D + (((spg + mseg) ^ (row & 7)) << 4), r);
#pragma unroll
        for (int hs = 0; hs < 2; ++hs) {
          const int seg = spg + hs;
          const uint32_t x0v = __byte_perm(r[2 * hs], 0u, 0x3120u);
          const uint32_t x1v = __byte_perm(r[2 * hs + 1], 0u, 0x3120u);
          uint32_t b0[2], b1[2];  // [e]: n tile of dims 16 seg + 2 n + e
          e4m3x4_f16x2x2(x0v, b0[0], b0[1]);
          e4m3x4_f16x2x2(x1v, b1[0], b1[1]);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            mma_rows16(acc[seg][e], ah[0], ah[1], ah[2], ah[3], b0[e], b1[e]);
            mma_rows16(acc[seg][e], al[0], al[1], al[2], al[3], b0[e], b1[e]);
          }
        }
      }
    }
    // every warp has used this stage (each ldmatrix result has fed an MMA
    // above): refill it with chunk c + PF_STAGES
    __syncthreads();
    if (threadIdx.x == 0 && c + PF_STAGES < nch) issue(c + PF_STAGES);
  }
  if (!ok && threadIdx.x == 0) {
    // chunks c .. c + PF_STAGES - 1 may still be in flight: let them land
    // (bounded) before the shared memory is given up
    atomicCAS(&g_w8a8_attn_error, 0, 23);
    for (int j = c; j < nch && j < c + PF_STAGES; ++j)
      if (!ptx::mbar_wait(bar0 + (j % PF_STAGES) * 8, (uint32_t)(j / PF_STAGES) & 1u,
                          AT_WAIT_LIMIT_NS))
        atomicCAS(&g_w8a8_attn_error, 0, 24);
  }
  if (!ok) return;
  const float sv = sv_p[0];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    float lt = l[hh];
    lt += __shfl_xor_sync(0xFFFFFFFFu, lt, 1);
    lt += __shfl_xor_sync(0xFFFFFFFFu, lt, 2);
    const int tok = r0 + g + 8 * hh;
    if (tok >= seq) continue;
    const float f = sv / lt;
    uint16_t* o = out + (((b * seq + tok) * hq) + h) * (int64_t)AT_D;
#pragma unroll
    for (int s2 = 0; s2 < 8; ++s2)
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        // dims 16 s2 + 4 tig + 2 i + {0, 1}
        const uint32_t v2 = (uint32_t)bf16_rn(acc[s2][0][2 * hh + i] * f) |
                            ((uint32_t)bf16_rn(acc[s2][1][2 * hh + i] * f) << 16);
        *reinterpret_cast<uint32_t*>(o + 16 * s2 + 4 * tig + 2 * i) = v2;
      }
  }
}

cudaError_t launch_prefill_attention(const uint8_t* q, const float* sq, const uint8_t* k,
                                     const float* sk, const uint8_t* v, const float* sv,
                                     int64_t batch, int64_t seq, int hq, int hkv,
                                     float softmax_scale, uint16_t* out, cudaStream_t st) {
  if (batch == 0 || seq == 0) return cudaSuccess;
  const int64_t nqb = (seq + PF_ROWS - 1) / PF_ROWS;
  // grid y / z limits; TMA row coordinates are 32-bit: the last chunk may
  // run PF_KEYS rows past batch * seq (those rows read as zero)
  if (hq > 65535 || batch > 65535 || nqb > 0x7FFFFFFFLL ||
      batch * seq > 0x7FFFFFFFLL - PF_KEYS)
    return cudaErrorInvalidValue;
  CUtensorMap tm_k, tm_v;
  const uint64_t rows = (uint64_t)(batch * seq), cols = (uint64_t)hkv * AT_D;
  if (!make_tmap_2d(&tm_k, k, 1, rows, cols, PF_KEYS, AT_D, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tm_v, v, 1, rows, cols, PF_KEYS, AT_D, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(prefill_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             PF_DYN_SMEM);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  const dim3 grid((unsigned)nqb, (unsigned)hq, (unsigned)batch);
  prefill_attention_kernel<<<grid, AT_THREADS, PF_DYN_SMEM, st>>>(
      tm_k, tm_v, q, sq, sk, sv, (int)seq, hq, hkv, (int)nqb, softmax_scale, out);
  return cudaGetLastError();
}

}  // namespace w8a8
