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
// tokens; in a warp, lane group g (lanes 8g..8g+7) takes every 4th token and
// lane l8 = lane % 8 holds dims 16 l8 .. 16 l8 + 15 (16 bytes of K and of V
// per token).  Scores are in log2 units (log2 e and every scale folded into
// the query), kept by an online softmax per lane group; the groups, then
// the warps, are merged at the end.  Binary32 arithmetic throughout.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace w8a8 {

namespace {

constexpr int AT_D = 128;
constexpr int AT_WARPS = 4;
constexpr int AT_THREADS = 32 * AT_WARPS;
constexpr int AT_U = 4;  // tokens per lane group in flight

// 16 codes (one 16-byte vector) -> 16 binary32 values, exactly.
__device__ __forceinline__ void decode16(const uint4& c, float (&f)[16]) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 a = e4m3x2_to_float2((uint16_t)(w[i] & 0xFFFFu));
    const float2 b = e4m3x2_to_float2((uint16_t)(w[i] >> 16));
    f[4 * i + 0] = a.x;
    f[4 * i + 1] = a.y;
    f[4 * i + 2] = b.x;
    f[4 * i + 3] = b.y;
  }
}

__device__ __forceinline__ uint16_t bf16_rn(float x) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
  return r;
}

// Merge another (m, l, acc) state into this one (m in log2 units; -inf for
// an empty state).
template <int N>
__device__ __forceinline__ void merge_state(float& m, float& l, float (&acc)[N], float m2, float l2,
                                            const float (&acc2)[N]) {
  const float mt = fmaxf(m, m2);
  const float c1 = m == -INFINITY ? 0.0f : exp2f(m - mt);
  const float c2 = m2 == -INFINITY ? 0.0f : exp2f(m2 - mt);
  l = l * c1 + l2 * c2;
#pragma unroll
  for (int i = 0; i < N; ++i) acc[i] = acc[i] * c1 + acc2[i] * c2;
  m = mt;
}

}  // namespace

template <int GH>
__global__ void __launch_bounds__(AT_THREADS, 2)
    decode_attention_kernel(const uint8_t* __restrict__ q, const float* __restrict__ sq_p,
                            const uint8_t* __restrict__ k, const float* __restrict__ sk_p,
                            const uint8_t* __restrict__ v, const float* __restrict__ sv_p,
                            const int32_t* __restrict__ lens, int64_t smax, int hq, int hkv,
                            int hgroups, float softmax_scale, uint16_t* __restrict__ out) {
  __shared__ float s_acc[AT_WARPS][GH][AT_D];
  __shared__ float s_ml[AT_WARPS][GH][2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane >> 3, l8 = lane & 7;
  const int hg = blockIdx.x % hgroups;
  const int64_t bk = blockIdx.x / hgroups;
  const int kh = (int)(bk % hkv);
  const int64_t b = bk / hkv;
  const int h0 = kh * (hq / hkv) + hg * GH;  // first query head of this CTA
  // lengths are device data the host cannot check: clamp to [0, smax]
  const int len = (int)min((int64_t)max(lens[b], 0), smax);

  // query slice, all factors folded in: scores come out in log2 units
  const float qk = softmax_scale * sq_p[0] * sk_p[0] * 1.4426950408889634f;
  float qf[GH][16];
#pragma unroll
  for (int h = 0; h < GH; ++h) {
    const uint4 c = *reinterpret_cast<const uint4*>(q + ((b * hq) + h0 + h) * AT_D + 16 * l8);
    decode16(c, qf[h]);
#pragma unroll
    for (int i = 0; i < 16; ++i) qf[h][i] *= qk;
  }
  float m[GH], l[GH], acc[GH][16];
#pragma unroll
  for (int h = 0; h < GH; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[h][i] = 0.0f;
  }

  const int per = (len + AT_WARPS - 1) / AT_WARPS;
  const int t0 = min(len, warp * per), t1 = min(len, t0 + per);
  const int64_t tstride = (int64_t)hkv * AT_D;
  const uint8_t* kbase = k + ((b * smax) * hkv + kh) * AT_D + 16 * l8;
  const uint8_t* vbase = v + ((b * smax) * hkv + kh) * AT_D + 16 * l8;
  // Every lane runs the same number of iterations (the warp-wide shuffles
  // below need all 32 lanes); a lane group whose token is past the end
  // loads nothing and skips the update.  AT_U tokens per lane group are
  // loaded before any is used, so that enough bytes are in flight.
  for (int tb = t0; tb < t1; tb += 4 * AT_U) {
    uint4 kc[AT_U], vc[AT_U];
#pragma unroll
    for (int u = 0; u < AT_U; ++u) {
      const int t = tb + grp + 4 * u;
      const bool tok = t < t1;
      kc[u] = tok ? ld_stream_v4(kbase + t * tstride) : make_uint4(0u, 0u, 0u, 0u);
      vc[u] = tok ? ld_stream_v4(vbase + t * tstride) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < AT_U; ++u) {
      const bool tok = tb + grp + 4 * u < t1;
      float kf[16], vf[16];
      decode16(kc[u], kf);
      float s[GH];
#pragma unroll
      for (int h = 0; h < GH; ++h) {
        float a = 0.0f, c = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          a = __fmaf_rn(qf[h][i], kf[i], a);
          c = __fmaf_rn(qf[h][i + 1], kf[i + 1], c);
        }
        s[h] = a + c;
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1)
#pragma unroll
        for (int h = 0; h < GH; ++h) s[h] += __shfl_xor_sync(0xFFFFFFFFu, s[h], o);
      decode16(vc[u], vf);
#pragma unroll
      for (int h = 0; h < GH; ++h) {
        if (!tok) continue;
        if (s[h] > m[h]) {  // a new running maximum: rescale what was summed so far
          const float cr = exp2f(m[h] - s[h]);
          l[h] *= cr;
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[h][i] *= cr;
          m[h] = s[h];
        }
        const float p = exp2f(s[h] - m[h]);
        l[h] += p;
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[h][i] = __fmaf_rn(p, vf[i], acc[h][i]);
      }
    }
  }

  // merge the 4 lane groups of the warp (lanes with equal l8 hold equal dims)
#pragma unroll
  for (int o = 8; o < 32; o <<= 1) {
#pragma unroll
    for (int h = 0; h < GH; ++h) {
      const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m[h], o);
      const float l2 = __shfl_xor_sync(0xFFFFFFFFu, l[h], o);
      float a2[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) a2[i] = __shfl_xor_sync(0xFFFFFFFFu, acc[h][i], o);
      merge_state(m[h], l[h], acc[h], m2, l2, a2);
    }
  }
  if (grp == 0) {
#pragma unroll
    for (int h = 0; h < GH; ++h) {
#pragma unroll
      for (int i = 0; i < 16; ++i) s_acc[warp][h][16 * l8 + i] = acc[h][i];
      if (l8 == 0) {
        s_ml[warp][h][0] = m[h];
        s_ml[warp][h][1] = l[h];
      }
    }
  }
  __syncthreads();
  // merge the warps in a fixed order; thread d writes dim d of every head
  const float sv = sv_p[0];
  const int d = threadIdx.x;
#pragma unroll
  for (int h = 0; h < GH; ++h) {
    float mm = -INFINITY, ll = 0.0f, aa[1] = {0.0f};
#pragma unroll
    for (int w = 0; w < AT_WARPS; ++w) {
      const float a2[1] = {s_acc[w][h][d]};
      merge_state(mm, ll, aa, s_ml[w][h][0], s_ml[w][h][1], a2);
    }
    const float y = ll > 0.0f ? aa[0] / ll * sv : 0.0f;
    out[((b * hq) + h0 + h) * AT_D + d] = bf16_rn(y);
  }
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
  const int64_t grid = batch * hkv * hgroups;
  if (grid > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  switch (gh) {
    case 1:
      decode_attention_kernel<1><<<(unsigned)grid, AT_THREADS, 0, st>>>(
          q, sq, k, sk, v, sv, lens, smax, hq, hkv, hgroups, softmax_scale, out);
      break;
    case 2:
      decode_attention_kernel<2><<<(unsigned)grid, AT_THREADS, 0, st>>>(
          q, sq, k, sk, v, sv, lens, smax, hq, hkv, hgroups, softmax_scale, out);
      break;
    default:
      decode_attention_kernel<4><<<(unsigned)grid, AT_THREADS, 0, st>>>(
          q, sq, k, sk, v, sv, lens, smax, hq, hkv, hgroups, softmax_scale, out);
      break;
  }
  return cudaGetLastError();
}

}  // namespace w8a8
