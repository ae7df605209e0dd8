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

#include <type_traits>

#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tmap.h"

namespace w8a8 {

// Set (first code wins) when a bounded wait of an attention kernel gives
// up: 21 = a decode chunk's TMA loads did not land in time, 22 = the drain
// of the loads still in flight after that also timed out, 23 = a wait of
// the prefill kernel.
__device__ int g_w8a8_attn_error = 0;

// Test hook (w8a8_debug_force_wait_timeout): when set, each decode warp's
// wait for its first chunk, and the prefill MMA issuer before its first
// MMA, behave as if they had run out of time.
__device__ int g_w8a8_attn_force_timeout = 0;

cudaError_t set_attn_force_timeout(int on) {
  return cudaMemcpyToSymbol(g_w8a8_attn_force_timeout, &on, sizeof(int));
}

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
  // the test hook, read while the first loads are in flight
  const bool force_timeout = *reinterpret_cast<volatile int*>(&g_w8a8_attn_force_timeout) != 0;
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
    bool landed = ptx::mbar_wait(bar0 + s * 8, (uint32_t)(c / AT_STAGES) & 1u, AT_WAIT_LIMIT_NS);
    if (c == 0 && force_timeout) landed = false;
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
// Both contractions run on the 5th-generation tensor cores with the
// accumulators in tensor memory.  A query block is 128 query tokens of one
// (sequence, query head); keys come in chunks of 128 tokens, so chunk qb of
// block qb is the diagonal one.  The kernel is persistent: one CTA per SM
// takes its share of the blocks in turn, longest (most keys) first.
//   warp 0     TMA: each block's Q tile (once the previous block's S MMAs
//              are done with the buffer), then its K and V tiles (E4M3,
//              128-byte swizzle) into a 3-stage ring;
//   warp 1     allocates 512 TMEM columns: two S buffers, two PV buffers.
//              Lane 0 issues S(j) = Q K_j^T on the raw E4M3 codes
//              (kind::f8f6f4, M = 128 queries, N = 128 keys, f32
//              accumulation) into S buffer j % 2, and PV(j) = P_j V_j
//              (kind::f16, M = 128 queries, N = 128 dims, K = 128 keys, A
//              read from tensor memory, the weights' high then low f16
//              parts) into PV buffer j % 2;
//   warps 2-3  widen each V tile to f16, transposed (V^T [dim][key], the
//              K-major B operand), exactly;
//   warps 4-11 two threads per query row (one in each of two warps on the
//              same TMEM lanes), each with half of the keys and half of the
//              output dims: the row's maximum over S(j) (the pair's partial
//              maxima exchanged), then the weights P = 2^15 p (online
//              softmax in log2 units, later keys masked in the diagonal
//              chunk) as high and low f16 parts (together 22 bits of each
//              weight), written over the row of S(j) in tensor memory, where
//              PV(j) reads them; then, one chunk behind,
//              O = O * correction + PV(j - 1) in FP32 registers, so that
//              PV(j) runs while the next chunk's weights are formed.
// The softmax passes keep their 32-column loops rolled: fully unrolled, the
// loop body outgrew the instruction cache and the kernel ran ~30% slower.
// Every mbarrier wait is bounded; a wait that gives up records error 23 and
// stops the CTA's roles.
namespace {
constexpr int PT_ROWS = 128;                        // query tokens per block
constexpr int PT_KEYS = 128;                        // keys per chunk
constexpr int PT_TILE = PT_KEYS * AT_D;             // 16 KB: a Q, K or V tile (E4M3)
constexpr int PT_HALF = 128 * 128;                  // 16 KB: 128 rows x 64 f16 (128 bytes)
constexpr int PT_STAGES = 3;                        // K/V ring
constexpr int PT_OFF_Q = 0;
constexpr int PT_OFF_KV = PT_OFF_Q + PT_TILE;                   // stages of (K, V)
constexpr int PT_OFF_VT = PT_OFF_KV + 2 * PT_STAGES * PT_TILE;  // 2 buffers of V^T f16 (2 halves each)
constexpr int PT_OFF_BAR = PT_OFF_VT + 4 * PT_HALF;
constexpr int PT_NBAR = 2 * PT_STAGES + 23;
constexpr int PT_OFF_MISC = PT_OFF_BAR + PT_NBAR * 8;
constexpr int PT_OFF_X = PT_OFF_MISC + 16;  // row maxima and sums exchanged by warp pairs
constexpr int PT_DYN_SMEM = PT_OFF_X + 2 * 2 * PT_ROWS * 4 + 1024;
constexpr int PT_THREADS = 384;
constexpr uint32_t PT_IDESC = ptx::idesc_e4m3_f32(128, 128);  // also kind::f16 with F16 A, B
static_assert(PT_OFF_KV % 1024 == 0 && PT_OFF_VT % 1024 == 0,
              "swizzled tiles start on 1024-byte boundaries");
static_assert(PT_DYN_SMEM <= 232448, "shared memory");

// D (TMEM) (+)= A (TMEM, 128 lanes = rows, two f16 per 32-bit column along
// K) x B (shared memory descriptor), kind::f16
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 lanes x 4 consecutive 32-bit columns from registers
__device__ __forceinline__ void tmem_st_x4(uint32_t taddr, uint32_t v0, uint32_t v1, uint32_t v2,
                                           uint32_t v3) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
               "r"(v0), "r"(v1), "r"(v2), "r"(v3)
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// bounded mbarrier wait that also gives up once another role has
__device__ __forceinline__ bool pt_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer() - t0 > AT_WAIT_LIMIT_NS) {
      atomicCAS(&g_w8a8_attn_error, 0, 23);
      *abort_flag = 1;
      return false;
    }
  }
}

// the same wait taken by lane 0 and broadcast to the warp
__device__ __forceinline__ bool pt_wait_warp(uint32_t bar, uint32_t parity,
                                             volatile int* abort_flag, int lane) {
  uint32_t okw = lane == 0 ? (pt_wait(bar, parity, abort_flag) ? 1u : 0u) : 0u;
  return __shfl_sync(0xFFFFFFFFu, okw, 0) != 0u;
}
}  // namespace

// The k-th query block of CTA x (of G): blocks are numbered longest first
// (then sequence, then query head, so the query heads of one KV head are
// neighbours), dealt in rounds of G, every other round in reverse order so
// that the CTAs' totals even out.
struct PtBlock {
  int qb, h, b;
};
__device__ __forceinline__ bool pt_block(int k, int x, int G, int64_t total, int nqb, int hq,
                                         int batch, PtBlock& blk) {
  const int64_t u = (int64_t)k * G + ((k & 1) ? G - 1 - x : x);
  if (u >= total) return false;
  const int64_t per = (int64_t)hq * batch;
  blk.qb = nqb - 1 - (int)(u / per);
  const int64_t rem = u % per;
  blk.h = (int)(rem % hq);
  blk.b = (int)(rem / hq);
  return true;
}

__global__ void __launch_bounds__(PT_THREADS, 1)
    prefill_attention_kernel(const __grid_constant__ CUtensorMap tm_q,
                             const __grid_constant__ CUtensorMap tm_k,
                             const __grid_constant__ CUtensorMap tm_v,
                             const float* __restrict__ sq_p, const float* __restrict__ sk_p,
                             const float* __restrict__ sv_p, int seq, int hq, int hkv, int nqb,
                             int batch, float softmax_scale, uint16_t* __restrict__ out) {
  extern __shared__ __align__(16) uint8_t at_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = (int)gridDim.x, x = (int)blockIdx.x;
  const int64_t total = (int64_t)nqb * hq * batch;
  const int group = hq / hkv;
  const uint32_t base = (ptx::smem_addr(at_smem) + 1023u) & ~1023u;
  uint8_t* gbase = at_smem + (base - ptx::smem_addr(at_smem));
  const uint32_t bar0 = base + PT_OFF_BAR;
  const uint32_t q_full = bar0;
  auto kv_full = [&](int t) { return bar0 + 8u * (1 + t); };
  auto kv_empty = [&](int t) { return bar0 + 8u * (1 + PT_STAGES + t); };  // S commit + 2 converter warps
  const uint32_t bar2 = bar0 + 8u * (1 + 2 * PT_STAGES);  // then pairs, indexed by chunk % 2
  auto s_full = [&](int s) { return bar2 + 8u * (0 + s); };    // S MMA commit
  auto p_full = [&](int s) { return bar2 + 8u * (2 + s); };    // 8 softmax warps
  auto vt_full = [&](int s) { return bar2 + 8u * (4 + s); };   // 2 converter warps
  auto vt_empty = [&](int s) { return bar2 + 8u * (6 + s); };  // PV MMA commit
  auto pv_full = [&](int s) { return bar2 + 8u * (8 + s); };   // PV MMA commit
  auto pv_empty = [&](int s) { return bar2 + 8u * (10 + s); }; // 8 softmax warps
  const uint32_t mma_done = bar2 + 8u * 12;                     // the last MMAs completed
  const uint32_t q_empty = bar2 + 8u * 13;                      // a block's last S MMA completed
  // exchange e of the softmax warp pair of TMEM lane quarter q: buffer e % 2
  auto xbar = [&](int e, int q) { return bar2 + 8u * (14 + 4 * (e & 1) + q); };  // 64 threads
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + PT_OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + PT_OFF_MISC + 4);
  auto next_block = [&](int k, PtBlock& blk) {
    return pt_block(k, x, G, total, nqb, hq, batch, blk);
  };

  if (threadIdx.x == 0) {
    ptx::mbar_init(q_full, 1);
    ptx::mbar_init(q_empty, 1);
    for (int t = 0; t < PT_STAGES; ++t) {
      ptx::mbar_init(kv_full(t), 1);
      ptx::mbar_init(kv_empty(t), 3);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(s_full(s), 1);
      ptx::mbar_init(p_full(s), 8);
      ptx::mbar_init(vt_full(s), 2);
      ptx::mbar_init(vt_empty(s), 1);
      ptx::mbar_init(pv_full(s), 1);
      ptx::mbar_init(pv_empty(s), 8);
    }
    for (int q = 0; q < 8; ++q) ptx::mbar_init(xbar(q >> 2, q & 3), 64);
    ptx::mbar_init(mma_done, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  auto tS = [&](int s) { return tmem_base + 128u * (uint32_t)s; };         // S(j), then P(j)
  auto tPV = [&](int s) { return tmem_base + 256u + 128u * (uint32_t)s; };  // PV(j)

  // Chunks are counted over all of the CTA's blocks (g): the rings, the
  // TMEM buffers and their barriers' phases follow g, so one block's first
  // loads and MMAs overlap the previous block's last steps.
  if (warp == 0) {
    // ------------------------------------------------------------------ TMA
    if (lane == 0) {
      int g = 0, nblk = 0;
      bool ok = true;
      PtBlock blk;
      for (int k = 0; ok && next_block(k, blk); ++k) {
        const int krow0 = blk.b * seq;  // cache row of the sequence's token 0 (checked on the host)
        const int kh = blk.h / group;
        for (int c = 0; c <= blk.qb; ++c) {
          const int t = g % PT_STAGES;
          if (!pt_wait(kv_empty(t), (uint32_t)(((g / PT_STAGES) & 1) ^ 1), abort_flag)) { ok = false; break; }
          const uint32_t st = base + PT_OFF_KV + t * 2 * PT_TILE;
          ptx::mbar_arrive_expect_tx(kv_full(t), 2 * PT_TILE);
          ptx::tma_load_2d(st, &tm_k, kv_full(t), kh * AT_D, krow0 + c * PT_KEYS);
          ptx::tma_load_2d(st + PT_TILE, &tm_v, kv_full(t), kh * AT_D, krow0 + c * PT_KEYS);
          ++g;
          if (c == 0) {
            // Q of this block, once the previous block's S MMAs are done with the tile
            if (!pt_wait(q_empty, (uint32_t)((k & 1) ^ 1), abort_flag)) { ok = false; break; }
            ptx::mbar_arrive_expect_tx(q_full, PT_TILE);
            ptx::tma_load_2d(base + PT_OFF_Q, &tm_q, q_full, blk.h * AT_D, krow0 + blk.qb * PT_ROWS);
            ++nblk;
          }
        }
      }
      // no copy may still be landing when the CTA retires
      if (nblk > 0) {
        const uint64_t t0 = ptx::globaltimer();
        while (!ptx::mbar_try_wait(q_full, (uint32_t)((nblk - 1) & 1)))
          if (ptx::globaltimer() - t0 > AT_WAIT_LIMIT_NS) { atomicCAS(&g_w8a8_attn_error, 0, 23); break; }
      }
      for (int j = g > PT_STAGES ? g - PT_STAGES : 0; j < g; ++j) {
        const uint64_t t1 = ptx::globaltimer();
        while (!ptx::mbar_try_wait(kv_full(j % PT_STAGES), (uint32_t)((j / PT_STAGES) & 1)))
          if (ptx::globaltimer() - t1 > AT_WAIT_LIMIT_NS) { atomicCAS(&g_w8a8_attn_error, 0, 23); break; }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA
    if (lane == 0) {
      bool ok = true;
      if (*reinterpret_cast<volatile int*>(&g_w8a8_attn_force_timeout) != 0) {
        atomicCAS(&g_w8a8_attn_error, 0, 23);
        *abort_flag = 1;
        ok = false;
      }
      const uint64_t qdesc = ptx::smem_desc_kmajor_sw128(base + PT_OFF_Q);
      // S cursor: block ks, its chunk cs, overall chunk gs
      int ks = 0, cs = 0, gs = 0;
      PtBlock bs;
      bool s_more = next_block(0, bs);
      auto issue_s = [&]() {
        if (cs == 0 && !pt_wait(q_full, (uint32_t)(ks & 1), abort_flag)) return false;
        const int t = gs % PT_STAGES;
        if (!pt_wait(kv_full(t), (uint32_t)((gs / PT_STAGES) & 1), abort_flag)) return false;
        ptx::tc_fence_after();
        const uint64_t kdesc = ptx::smem_desc_kmajor_sw128(base + PT_OFF_KV + t * 2 * PT_TILE);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // 32 dims (bytes) per MMA
          ptx::mma_f8f6f4(tS(gs & 1), qdesc + 2u * kk, kdesc + 2u * kk, PT_IDESC, kk > 0 ? 1u : 0u);
        ptx::mma_commit(s_full(gs & 1));
        ptx::mma_commit(kv_empty(t));
        ++gs;
        if (++cs > bs.qb) {  // the block's last S: its Q tile may be replaced once it completes
          ptx::mma_commit(q_empty);
          cs = 0;
          s_more = next_block(++ks, bs);
        }
        return true;
      };
      // PV cursor: block kp, its chunk cp, overall chunk gp (two behind S)
      int kp = 0, cp = 0, gp = 0;
      PtBlock bp;
      bool p_more = next_block(0, bp);
      if (ok && s_more) ok = issue_s();
      if (ok && s_more) ok = issue_s();
      while (ok && p_more) {
        // PV(gp): the weights of chunk gp in S buffer s, V^T widened, PV
        // buffer s read out (chunk gp - 2)
        const int s = gp & 1;
        const uint32_t ph = (uint32_t)((gp >> 1) & 1);
        if (!pt_wait(p_full(s), ph, abort_flag) || !pt_wait(vt_full(s), ph, abort_flag) ||
            !pt_wait(pv_empty(s), ph ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t vt = base + PT_OFF_VT + s * 2 * PT_HALF;
#pragma unroll
        for (int part = 0; part < 2; ++part) {  // the weights' high, then low f16 parts
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {  // 16 keys per MMA: 8 columns of P
            const uint32_t a = tS(s) + 32u * (uint32_t)(kk >> 1) + 16u * (uint32_t)part +
                               8u * (uint32_t)(kk & 1);
            const uint64_t bdesc = ptx::smem_desc_kmajor_sw128(vt + (uint32_t)(kk >> 2) * PT_HALF) +
                                   2u * (kk & 3);
            mma_f16_tmem_a(tPV(s), a, bdesc, PT_IDESC, (part | kk) ? 1u : 0u);
          }
        }
        ptx::mma_commit(pv_full(s));
        ptx::mma_commit(vt_empty(s));
        if (s_more) {
          // S(gp + 2) goes where P(gp) is: after PV(gp) has completed
          if (!pt_wait(pv_full(s), ph, abort_flag)) { ok = false; break; }
          ptx::tc_fence_after();
          ok = issue_s();
        }
        ++gp;
        if (++cp > bp.qb) {
          cp = 0;
          p_more = next_block(++kp, bp);
        }
      }
      // every MMA issued has completed before the CTA frees TMEM
      ptx::mma_commit(mma_done);
      const uint64_t t0 = ptx::globaltimer();
      while (!ptx::mbar_try_wait(mma_done, 0))
        if (ptx::globaltimer() - t0 > AT_WAIT_LIMIT_NS) { atomicCAS(&g_w8a8_attn_error, 0, 23); break; }
    }
    __syncwarp();
  } else if (warp < 4) {
    // ------------------------------------------------------ V -> V^T (f16)
    // a block is 16 dims x 8 keys: 8 LDS.128 from key rows (128-byte swizzle
    // of the TMA tile), transposed with byte permutes, widened exactly to
    // f16, 16 STS.128 into V^T rows (128-byte swizzle of the K-major operand:
    // 16-byte chunk c of row d at c ^ (d & 7)). Lane l of converter warp wv
    // takes key octet (l & 7) + 8 wv and dim groups l >> 3, (l >> 3) + 4:
    // the stores of a warp fill whole 128-byte lines, the loads two-way.
    const int wv = warp - 2;
    const int ko = (lane & 7) + 8 * wv;
    int g = 0;
    bool okc = true;
    PtBlock blk;
    for (int k = 0; okc && next_block(k, blk); ++k) {
      for (int c = 0; c <= blk.qb; ++c, ++g) {
        const int t = g % PT_STAGES, s = g & 1;
        bool okl = pt_wait(kv_full(t), (uint32_t)((g / PT_STAGES) & 1), abort_flag) &&
                   pt_wait(vt_empty(s), (uint32_t)(((g >> 1) & 1) ^ 1), abort_flag);
        if (!__all_sync(0xFFFFFFFFu, okl)) { okc = false; break; }
        const uint32_t vsrc = base + PT_OFF_KV + t * 2 * PT_TILE + PT_TILE;
        const uint32_t vt = base + PT_OFF_VT + s * 2 * PT_HALF + (uint32_t)wv * PT_HALF;
#pragma unroll 1
        for (int i = 0; i < 2; ++i) {
          const int gq = (lane >> 3) + 4 * i;  // dims 16 gq .. 16 gq + 15
          uint4 w[8];
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            w[kk] = ptx::lds128(vsrc + (8 * ko + kk) * 128 + ((gq ^ kk) << 4));
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t xw[8];
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              xw[kk] = j == 0 ? w[kk].x : j == 1 ? w[kk].y : j == 2 ? w[kk].z : w[kk].w;
#pragma unroll
            for (int dd = 0; dd < 4; ++dd) {
              // dim 16 gq + 4 j + dd of keys 8 ko .. 8 ko + 7: byte dd of each
              // word (low two bytes: byte dd of the first word, then of the second)
              const uint32_t sel = (uint32_t)dd | ((uint32_t)(dd + 4) << 4);
              const uint32_t k01 = __byte_perm(xw[0], xw[1], sel);
              const uint32_t k23 = __byte_perm(xw[2], xw[3], sel);
              const uint32_t k45 = __byte_perm(xw[4], xw[5], sel);
              const uint32_t k67 = __byte_perm(xw[6], xw[7], sel);
              const uint32_t k0123 = __byte_perm(k01, k23, 0x5410u);
              const uint32_t k4567 = __byte_perm(k45, k67, 0x5410u);
              uint32_t f[4];
              e4m3x4_f16x2x2(k0123, f[0], f[1]);
              e4m3x4_f16x2x2(k4567, f[2], f[3]);
              const int d = 16 * gq + 4 * j + dd;
              ptx::sts128(vt + d * 128 + ((((ko & 7) ^ (d & 7))) << 4), f[0], f[1], f[2], f[3]);
            }
          }
        }
        ptx::fence_proxy_async_smem();  // generic writes -> the MMA's reads
        __syncwarp();
        if (lane == 0) {
          ptx::mbar_arrive(vt_full(s));
          ptx::mbar_arrive(kv_empty(t));
        }
      }
    }
  } else {
    // ------------------------------------------------------------- softmax
    // Two warps per TMEM lane quarter: thread rrow of half hf takes keys
    // 64 hf .. 64 hf + 63 of each chunk of query row rrow and dims
    // 64 hf .. 64 hf + 63 of its output.  The pair exchanges its partial
    // row maxima once per chunk and its sums once per block, through shared
    // memory and an mbarrier per exchange (bounded waits).
    const int quarter = warp & 3, hf = (warp - 4) >> 2;
    const int rrow = quarter * 32 + lane;  // query row in the block (TMEM lane)
    const uint32_t lanes = (uint32_t)(quarter * 32) << 16;
    const float qk = softmax_scale * sq_p[0] * sk_p[0] * 1.4426950408889634f;
    const float fv = sv_p[0];
    float* xv = reinterpret_cast<float*>(gbase + PT_OFF_X);  // [buffer][half][row]
    float o[64];
    float m, l;
    int qb = 0, tok = 0, ex = 0;
    // the partner's value of exchange ex (this thread's own is v)
    auto exchange = [&](float v, float& other) {
      const int bx = ex & 1;
      xv[(bx * 2 + hf) * PT_ROWS + rrow] = v;
      ptx::mbar_arrive(xbar(ex, quarter));  // releases the store above
      const bool okx = pt_wait(xbar(ex, quarter), (uint32_t)((ex >> 1) & 1), abort_flag);
      if (!__all_sync(0xFFFFFFFFu, okx)) return false;
      other = xv[(bx * 2 + (hf ^ 1)) * PT_ROWS + rrow];
      ++ex;
      return true;
    };
    // pass 1 of chunk c (overall gc): the row's new maximum and the
    // correction of what came before; four running maxima (independent
    // chains) of this half's raw scores, the diagonal chunk's keys after the
    // query left out, scaled once (rounding is monotone and qk >= 0, so this
    // is the maximum of the scaled scores; an empty half gives NaN, which
    // fmaxf passes over), then the pair's two maxima
    auto pass1 = [&](int c, int gc, float& mx, float& cr) {
      if (!pt_wait_warp(s_full(gc & 1), (uint32_t)((gc >> 1) & 1), abort_flag, lane)) return false;
      ptx::tc_fence_after();
      const uint32_t ts = tS(gc & 1) + lanes;
      const int lim = c == qb ? tok - c * PT_KEYS : PT_KEYS;
      float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
      for (int cc = 2 * hf; cc < 2 * hf + 2; ++cc) {
        uint32_t r[32];
        ptx::tmem_ld_32x32b_x32(ts + 32 * cc, r);
        ptx::tmem_wait_ld_dep32(r);
        if (!__any_sync(0xFFFFFFFFu, lim < 32 * cc + 31)) {
#pragma unroll
          for (int i = 0; i < 32; ++i) mq[i & 3] = fmaxf(mq[i & 3], __uint_as_float(r[i]));
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * cc + i <= lim) mq[i & 3] = fmaxf(mq[i & 3], __uint_as_float(r[i]));
        }
      }
      const float mh = fmaxf(m, fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * qk);
      float mo;
      if (!exchange(mh, mo)) return false;
      mx = fmaxf(mh, mo);
      cr = m == mx ? 1.0f : ex2_approx(m - mx);
      m = mx;
      return true;
    };
    // O = O * cr + PV(gc) over this half's dims, then PV buffer gc % 2 is
    // free again (once both halves have read it)
    auto o_update = [&](int gc, float cr) {
      if (!pt_wait_warp(pv_full(gc & 1), (uint32_t)((gc >> 1) & 1), abort_flag, lane)) return false;
      ptx::tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t r[32];
        ptx::tmem_ld_32x32b_x32(tPV(gc & 1) + lanes + 64 * hf + 32 * cc, r);
        ptx::tmem_wait_ld_dep32(r);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[32 * cc + i] = __fmaf_rn(o[32 * cc + i], cr, __uint_as_float(r[i]));
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(pv_empty(gc & 1));
      return true;
    };
    // the weights of 32 keys (one 32-column block of S) as high and low f16
    // parts over the block: columns 0 .. 15 the high parts (two keys per
    // column), 16 .. 31 the low parts; keys past lim weigh 0.  bias is
    // log2(2^15) minus the row's maximum.
    auto weights = [&](uint32_t taddr, const uint32_t (&r)[32], float bias, int lim,
                       float (&psq)[4], auto masked) {
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {  // 8 keys: 4 columns of each part
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float pv[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int i = 8 * q8 + 2 * e + u;
            pv[u] = ex2_approx(__fmaf_rn(__uint_as_float(r[i]), qk, bias));
            if (decltype(masked)::value && i > lim) pv[u] = 0.0f;
            psq[e] += pv[u];
          }
          hi[e] = pack_f16x2(pv[0], pv[1]);
          const float2 fh = unpack_f16x2(hi[e]);
          lo[e] = pack_f16x2(pv[0] - fh.x, pv[1] - fh.y);
        }
        tmem_st_x4(taddr + 4 * q8, hi[0], hi[1], hi[2], hi[3]);
        tmem_st_x4(taddr + 16 + 4 * q8, lo[0], lo[1], lo[2], lo[3]);
      }
    };
    int g = 0;
    bool ok = true;
    PtBlock blk;
    for (int k = 0; ok && next_block(k, blk); ++k) {
      qb = blk.qb;
      tok = qb * PT_ROWS + rrow;
      const int nch = qb + 1;  // key chunks 0 .. qb; chunk qb is the diagonal
#pragma unroll
      for (int i = 0; i < 64; ++i) o[i] = 0.0f;
      m = -INFINITY;
      l = 0.0f;
      float mx_c = 0.0f, cr_c = 0.0f, cr_lag = 0.0f;
      ok = pass1(0, g, mx_c, cr_c);
      for (int c = 0; c < nch && ok; ++c) {
        const int gc = g + c;
        const uint32_t ts = tS(gc & 1) + lanes;
        const int lim = c == qb ? tok - c * PT_KEYS : PT_KEYS;
        // pass 2: the weights over this half of the row of S(c), four
        // partial sums
        float psq[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        const float bias = AT_P_LOG2 - mx_c;
#pragma unroll 1
        for (int cc = 2 * hf; cc < 2 * hf + 2; ++cc) {
          uint32_t r[32];
          ptx::tmem_ld_32x32b_x32(ts + 32 * cc, r);
          ptx::tmem_wait_ld_dep32(r);
          // tcgen05.st is warp-collective: the choice of path is the warp's
          if (!__any_sync(0xFFFFFFFFu, lim < 32 * cc + 31))
            weights(ts + 32 * cc, r, bias, 0, psq, std::false_type{});
          else
            weights(ts + 32 * cc, r, bias, lim - 32 * cc, psq, std::true_type{});
        }
        const float ps = (psq[0] + psq[1]) + (psq[2] + psq[3]);
        l = __fmaf_rn(l, cr_c, ps);
        tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(p_full(gc & 1));
        // one chunk behind: O += PV(c - 1) while the tensor cores compute PV(c)
        if (c > 0 && !o_update(gc - 1, cr_lag)) { ok = false; break; }
        cr_lag = cr_c;
        if (c + 1 < nch && !pass1(c + 1, gc + 1, mx_c, cr_c)) { ok = false; break; }
      }
      if (ok) ok = o_update(g + nch - 1, cr_lag);
      g += nch;
      float lo_sum = 0.0f;
      if (ok) ok = exchange(l, lo_sum);
      if (ok && tok < seq) {
        const float f = fv / (l + lo_sum);
        uint4* dst = reinterpret_cast<uint4*>(
            out + ((((int64_t)blk.b * seq + tok) * hq) + blk.h) * (int64_t)AT_D + 64 * hf);
#pragma unroll
        for (int v8 = 0; v8 < 8; ++v8) {
          uint4 w;
          w.x = (uint32_t)bf16_rn(o[8 * v8 + 0] * f) | ((uint32_t)bf16_rn(o[8 * v8 + 1] * f) << 16);
          w.y = (uint32_t)bf16_rn(o[8 * v8 + 2] * f) | ((uint32_t)bf16_rn(o[8 * v8 + 3] * f) << 16);
          w.z = (uint32_t)bf16_rn(o[8 * v8 + 4] * f) | ((uint32_t)bf16_rn(o[8 * v8 + 5] * f) << 16);
          w.w = (uint32_t)bf16_rn(o[8 * v8 + 6] * f) | ((uint32_t)bf16_rn(o[8 * v8 + 7] * f) << 16);
          dst[v8] = w;
        }
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, 512);
  }
}

cudaError_t launch_prefill_attention(const uint8_t* q, const float* sq, const uint8_t* k,
                                     const float* sk, const uint8_t* v, const float* sv,
                                     int64_t batch, int64_t seq, int hq, int hkv,
                                     float softmax_scale, uint16_t* out, cudaStream_t st) {
  if (batch == 0 || seq == 0) return cudaSuccess;
  const int64_t nqb = (seq + PT_ROWS - 1) / PT_ROWS;
  if (hq > 65535 || batch > 65535 || nqb > 0x7FFFFFFFLL ||
      batch * seq > 0x7FFFFFFFLL - PT_KEYS)
    return cudaErrorInvalidValue;
  CUtensorMap tm_q, tm_k, tm_v;
  const uint64_t rows = (uint64_t)(batch * seq);
  if (!make_tmap_2d(&tm_q, q, 1, rows, (uint64_t)hq * AT_D, PT_ROWS, AT_D, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tm_k, k, 1, rows, (uint64_t)hkv * AT_D, PT_KEYS, AT_D, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tm_v, v, 1, rows, (uint64_t)hkv * AT_D, PT_KEYS, AT_D, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(prefill_attention_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, PT_DYN_SMEM);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  // persistent: one CTA per SM walks its share of the query blocks
  const int64_t blocks = nqb * hq * batch;
  const unsigned grid = (unsigned)std::min<int64_t>(blocks, sm_count());
  prefill_attention_kernel<<<grid, PT_THREADS, PT_DYN_SMEM, st>>>(
      tm_q, tm_k, tm_v, sq, sk, sv, (int)seq, hq, hkv, (int)nqb, (int)batch, softmax_scale, out);
  return cudaGetLastError();
}

}  // namespace w8a8
