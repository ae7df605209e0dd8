// gemm_small_m.cu -- the blockwise-scaled FP8 GEMM for few token rows
// (m <= 256: decode-sized batches), shaped to stream the weights at HBM rate.
//
// What is computed is fp8_block_gemm's definition (NeMo RL FP8 blog, Table 1;
// "Unified FP8" notes, scale choice: FP32 scales):
//   Y[i,j] = BF16( sum_kb xs[i,kb] * ws[j/128,kb] * P[i,j,kb] ),
//   P[i,j,kb] = sum_{k in 128-wide slab kb} dec(xq[i,k]) * dec(wq[j,k]),
// FP32 accumulation, one FP32 promotion per slab.
//
// With m <= 256 the weights are almost all of the bytes, so the kernel is
// laid out around reading them once, from every SM at once:
//   * Operands swapped: a CTA owns 128 weight rows (one 128-row scale
//     block), which are the MMA's M = 128 rows; the tokens, padded to NT in
//     {32, 64, 128, 256}, are the MMA's N.  The accumulator is 128 lanes x
//     NT columns of TMEM, and a slab's weight scale is one number per CTA.
//   * Split K over a thread-block cluster of C CTAs (C = 1..8, chosen from
//     the tile and slab counts and the number of clusters that fit at once):
//     CTA r of the cluster takes a contiguous range of K slabs of the same
//     128 rows.  After the main loop every CTA sends the partial sums of
//     the token rows that CTA q owns to q's shared memory (one bulk copy
//     through distributed shared memory per peer); each CTA then adds the C
//     partials of its token rows in cluster-rank order (deterministic),
//     rounds and stores them.  No global scratch memory is used.
//   * Weight slabs come by TMA (the tensor-copy engine), token slabs by
//     16-byte cp.async from dedicated warps: an SM's TMA engine moves about
//     one 128-byte row per 5 cycles, so the NT token rows of a slab would
//     otherwise cost as much as its 128 weight rows.
//
// Roles:
//   warp 0      producer: per slab one TMA box of 128 weight rows x 128 B
//               into a STAGES-deep ring;
//   warp 1      allocates 2 x NT TMEM columns; lane 0 issues 4 x
//               tcgen05.mma.kind::f8f6f4 (128 x NT x 32) per slab into one of
//               two TMEM buffers and commits;
//   warps 2..   token loaders (1 or 2 warps): each slab's NT x 128 B of
//               codes by cp.async into the 128-byte-swizzled operand layout
//               (rows past m and bytes past k are zero-filled);
//   the rest    promotion (4 or 8 warps): tcgen05.ld of the slab's partial,
//               acc += P * (xs[token] * ws) in FP32 registers (thread =
//               weight row, registers = token columns).
//
// Every mbarrier wait is bounded (2 s of wall time); a wait that gives up
// records an error code (31..37) in this kernel's device error word, stops
// the other roles of its CTA and still takes part in the cluster barriers,
// so no CTA of the cluster is left waiting.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tmap.h"

namespace w8a8 {

// Device error word of this kernel (each translation unit has its own).
__device__ int g_w8a8_small_gemm_error = 0;
// Test hook (w8a8_debug_force_wait_timeout): when set, the MMA issuer's
// first wait gives up at once, so that the abort path runs on demand.
__device__ int g_w8a8_small_gemm_force_timeout = 0;

namespace sgemm {

constexpr int BW = 128;  // weight rows per CTA (the MMA's M)
constexpr int BK = 128;  // K bytes per slab: one 128-byte swizzle row
constexpr int W_BYTES = BW * BK;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr int MAX_SPLIT = 8;  // portable cluster size

// kFused: the token rows come as BF16 and are quantized (1 x 128 groups) by
// the loader warps on their way into shared memory.
template <int NT, bool kFused = false>
struct Cfg {
  static constexpr int X_BYTES = NT * BK;
  // fused: each stage also holds the slab's BF16 token rows (NT x 256 B)
  static constexpr int XB_BYTES = kFused ? NT * BK * 2 : 0;
  static constexpr int STAGE_BYTES = W_BYTES + X_BYTES + XB_BYTES;
  static constexpr int STAGES = kFused && NT >= 128 ? 3 : 4;
  // The CTA's scales are loaded once, at the start: xs of every token for
  // each of the CTA's slabs, transposed to [slab][token], and the tile's ws
  // per slab.  A CTA takes at most MAX_SLABS slabs (the split is chosen so,
  // and longer K goes to the general kernel).
  static constexpr int MAX_SLABS = 32;
  static constexpr int XS_BYTES = MAX_SLABS * NT * 4;
  static constexpr int WS_BYTES = MAX_SLABS * 4;
  static constexpr int XW = kFused ? (NT >= 128 ? 4 : 2) : (NT >= 128 ? 2 : 1);  // token loaders
  // Fused: the loaders' group scales pass to the promotion warps through a
  // ring of scale slots (each slab's NT scales), deep enough that the
  // loaders never wait on it in steady state: they run at most STAGES slabs
  // ahead of the MMA, and the MMA at most 2 ahead of the promotion.
  static constexpr int SLOTS = STAGES + 2;
  static constexpr int EPI_WARPS = NT >= 256 ? 8 : 4;
  static constexpr int EPI_WARP0 = 2 + XW;
  static constexpr int COLS = NT >= 256 ? 128 : NT;  // token columns per promotion thread
  static constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
  static constexpr int TMEM_COLS = 2 * NT;  // a power of two >= 64
  static constexpr int RING = STAGES * STAGE_BYTES;
  // The reduction reuses the ring: a send area of up to NTR = min(NT, 128)
  // token rows of 128 FP32, then a receive area of split - 1 slots of the
  // ceil(rows / split) token rows a CTA owns, at most NTR + split rows.
  // With 256 tokens all rows go in one round where the send area and the
  // slots fit below the barriers (the ring and the scale tables).
  static constexpr int NTR = NT < 128 ? NT : 128;
  static constexpr int RECV_OFF = NTR * BW * 4;
  static constexpr int RED_BYTES = RECV_OFF + (NTR + MAX_SPLIT) * BW * 4;
  static constexpr int OFF_XS = RING > RED_BYTES ? RING : RED_BYTES;
  static constexpr int OFF_WS = OFF_XS + XS_BYTES;
  static constexpr int OFF_BARS = OFF_WS + WS_BYTES;
  // full, empty, sfull, sempty, tfull[2], tempty[2], done, recv
  static constexpr int NUM_BARS = 2 * STAGES + 2 * SLOTS + 4 + 3;  // + done, recv, scales
  static constexpr int OFF_MISC = OFF_BARS + NUM_BARS * 8;
  static constexpr int SMEM = 1024 + OFF_MISC + 16;
  static constexpr uint32_t IDESC = ptx::idesc_e4m3_f32(BW, NT);
  static_assert(STAGE_BYTES % 1024 == 0, "swizzle atoms are 1024-byte aligned");
  static_assert(SMEM <= 232448, "shared memory");
  static_assert(COLS % 16 == 0 && COLS >= 32, "TMEM loads: 16 columns each, at least two");
  static_assert(NT % (4 * XW) == 0, "token rows split evenly over the loader warps");
  static_assert(!kFused || (NT <= 128 && NT % (8 * XW) == 0 && SLOTS <= MAX_SLABS),
                "fused: up to 128 tokens, 8 rows per loader warp step");
  // Registers: with 256 tokens the 8 promotion warps hold 128 FP32 sums
  // each; during the main loop the first warpgroup (producer, MMA, loaders)
  // gives them its share: 128 * 64 + 256 * 216 <= 384 * 168 (the launch's
  // register budget), and every warp returns to 168 for the reduction.
  static constexpr bool SPLIT_REGS = NT >= 256;
  // Who fetches the CTA's scale tables (asynchronously, after the
  // dependency wait): with 256 tokens the token loaders, which signal the
  // promotion warps through an mbarrier (the promotion warps' register share
  // has no room for the fetch); otherwise the promotion warps themselves.
  static constexpr bool LOADER_SCALES = NT >= 256 && !kFused;
  static constexpr int REGS_CTRL = 64, REGS_EPI = 216;
  // TMEM columns per promotion load step: 32 for 128 token columns (fewer,
  // longer load round trips; measured 3-5% faster with 256 tokens), else 16
  // (the fused kernel's registers hold no two 32-column buffers next to 128
  // sums)
  static constexpr int PROM_STEP = COLS >= 128 && !kFused ? 32 : 16;
  static_assert(!SPLIT_REGS || (EPI_WARP0 == 4 && 128 * REGS_CTRL + 256 * REGS_EPI <= THREADS * 168),
                "register split");
};

// tcgen05.ld of N (16 or 32) consecutive columns, and the wait for it
template <int N>
__device__ __forceinline__ void tmem_load(uint32_t taddr, uint32_t (&r)[N]) {
  if constexpr (N == 32) ptx::tmem_ld_32x32b_x32(taddr, r);
  else ptx::tmem_ld_32x32b_x16(taddr, r);
}
template <int N>
__device__ __forceinline__ void tmem_wait(uint32_t (&r)[N]) {
  if constexpr (N == 32) ptx::tmem_wait_ld_dep32(r);
  else ptx::tmem_wait_ld_dep(r);
}

struct Params {
  const uint8_t* xq;
  const float* xs;
  const uint16_t* xb;  // fused: BF16 tokens [m, k]
  uint8_t* xq_out;     // fused: codes and scales written here when not NULL
  float* xs_out;
  const float* ws;
  uint16_t* y;
  int32_t m, n, k, nkb, split;
  int32_t static_weights;  // wq, ws may be read before the previous kernel completes
};

__device__ __forceinline__ void record_error(int code) {
  atomicCAS(&g_w8a8_small_gemm_error, 0, code);
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         int code) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer() - t0 > WAIT_LIMIT_NS) {
      record_error(code);
      *abort_flag = 1;
      return false;
    }
  }
}

// First token row owned (rounded and stored) by K-split rank r; rank r owns
// [owned_lo(r), owned_lo(r + 1)), at most ceil(m / split) rows (r <= 8 and
// m <= 256: the product fits 32 bits).
__device__ __forceinline__ int owned_lo(int r, int m, int split) {
  return (int)((uint32_t)(r * m) / (uint32_t)split);
}

// Token rows the cluster reduction takes per round: all m at once where the
// send area (m rows of 128 FP32) and the receive slots of the split - 1 peers
// fit in the shared memory the main loop has finished with (the ring and the
// scale tables), else rounds of 128.
template <int NT, bool kFused>
__device__ __forceinline__ int reduce_rows_per_round(int m, int split) {
  if (NT <= 128) return m;
  const int own = (m + split - 1) / split;
  return (m + (split - 1) * own) * BW * 4 <= Cfg<NT, kFused>::OFF_BARS ? m : 128;
}

// The cluster reduction and the store of the output rows, run by every warp
// of the CTA after its role in the main loop: the promotion warps pass their
// sums (kAcc), the others take part in the barriers and the final sums.
// Each role calls it from its own branch, so that it runs with the registers
// that role holds.
template <int NT, bool kFused, bool kAcc>
__device__ __forceinline__ void reduce_store(const Params& p, uint8_t* smem, uint32_t sbase,
                                             uint32_t recv_bar, int rank, int split, int n0,
                                             int warp, int lane, int c0,
                                             const float2 (&acc)[Cfg<NT, kFused>::COLS / 2]) {
  using C = Cfg<NT, kFused>;
  // -------------------------------------------------- cluster reduction
  // Per round of token rows (one round unless the shared memory is short):
  //  1. arrive on the cluster barrier: this thread is past the main loop (or
  //     the previous round's sums) -- every copy and MMA touching the ring
  //     has been seen complete on an mbarrier, so the arrive is relaxed;
  //  2. the promotion threads store their partial sums as FP32 rows
  //     [token][weight row] in the send area at the start of the ring
  //     (consecutive lanes: consecutive words) -- the ring is this CTA's own
  //     and every slab in it has been consumed;
  //  3. wait on the cluster barrier: every peer is past its main loop, so
  //     its receive area (after its send area) is free;
  //  4. lane q of warp 0 sends peer q the rows that peer owns with one bulk
  //     copy into the peer's receive slot for this sender, completing on
  //     the peer's receive mbarrier; lane 0 waits for this CTA's own rows;
  //  5. arrive (relaxed) on the cluster barrier again: every copy into this
  //     CTA has landed, as its receive mbarrier showed, so the senders'
  //     areas are free;
  //  6. the CTA adds its rows' partials in rank order (its own read in
  //     place), rounds to BF16 and stores them;
  //  7. wait on the cluster barrier: every copy out of this CTA has landed,
  //     so it may reuse its send area or exit.
  const int m = p.m;
  const int rr = reduce_rows_per_round<NT, kFused>(m, split);
  const int rounds = (m + rr - 1) / rr;
  const int recv_off = rr * BW * 4;
  for (int h = 0; h < rounds; ++h) {
    const int t0 = rr * h;
    const int mh = min(rr, m - t0);
    const int own_rows = (mh + split - 1) / split;
    const int mlo = owned_lo(rank, mh, split), mhi = owned_lo(rank + 1, mh, split);
    if (split > 1) ptx::cluster_arrive_relaxed();
    if (kAcc && c0 < t0 + mh && c0 + C::COLS > t0) {
      const int row = (warp & 3) * 32 + lane;
      float* send = reinterpret_cast<float*>(smem);
#pragma unroll
      for (int i = 0; i < C::COLS; ++i) {
        const int u = c0 + i - t0;
        if (u >= 0 && u < mh) send[u * BW + row] = (i & 1) ? acc[i >> 1].y : acc[i >> 1].x;
      }
      ptx::fence_proxy_async_smem();  // generic writes -> the bulk copies' reads
    }
    __syncthreads();
    if (split > 1) ptx::cluster_wait();
    if (split > 1 && warp == 0) {
      const int q = lane;
      if (q < split && q != rank) {
        const int qlo = owned_lo(q, mh, split), qhi = owned_lo(q + 1, mh, split);
        if (qhi > qlo) {
          // a receiver's slots skip its own rank
          const int slot = rank < q ? rank : rank - 1;
          const uint32_t dst = sbase + (uint32_t)(recv_off + slot * own_rows * BW * 4);
          ptx::bulk_copy_to_peer(ptx::mapa_shared(dst, (uint32_t)q),
                                 sbase + (uint32_t)(qlo * BW * 4),
                                 (uint32_t)((qhi - qlo) * BW * 4),
                                 ptx::mapa_shared(recv_bar, (uint32_t)q));
        }
      }
    }
    if (split > 1 && threadIdx.x == 0) {
      const uint64_t tw = ptx::globaltimer();
      while (!ptx::mbar_try_wait(recv_bar, (uint32_t)(h & 1))) {
        if (ptx::globaltimer() - tw > WAIT_LIMIT_NS) { record_error(37); break; }
      }
      if (h + 1 < rounds) {
        const int mn = min(rr, m - t0 - rr);
        const int cnt = owned_lo(rank + 1, mn, split) - owned_lo(rank, mn, split);
        ptx::mbar_arrive_expect_tx(recv_bar, (uint32_t)((split - 1) * cnt * BW * 4));
      }
    }
    __syncthreads();
    if (split > 1) ptx::cluster_arrive_relaxed();
    // warp = token row, lane = 4 consecutive weight rows: 16-byte shared
    // loads, and a warp stores one 256-byte output row segment
    const int col4 = lane * 4;
    for (int u = mlo + warp; u < mhi; u += C::THREADS / 32) {
      float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int q = 0; q < split; ++q) {
        const int off = q == rank ? (u * BW + col4) * 4
                                  : recv_off + (((q < rank ? q : q - 1) * own_rows + (u - mlo)) * BW + col4) * 4;
        const float4 v = *reinterpret_cast<const float4*>(smem + off);
        s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
      }
      if (n0 + col4 < p.n) {
        uint2 o;
        o.x = ptx::pack_bf16x2(s.x, s.y);
        o.y = ptx::pack_bf16x2(s.z, s.w);
        *reinterpret_cast<uint2*>(p.y + (int64_t)(t0 + u) * p.n + n0 + col4) = o;
      }
    }
    if (split > 1) ptx::cluster_wait();
  }
}

template <int NT, bool kFused>
__global__ void __launch_bounds__(Cfg<NT, kFused>::THREADS, NT <= 64 ? 2 : 1)
    fp8_gemm_small_m_kernel(const __grid_constant__ CUtensorMap tmap_w,
                            const __grid_constant__ Params p) {
  using C = Cfg<NT, kFused>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_addr(smem);
  const uint32_t bar0 = sbase + C::OFF_BARS;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
  auto sfull_bar = [&](int s) { return bar0 + 8u * (2 * C::STAGES + s); };
  auto sempty_bar = [&](int s) { return bar0 + 8u * (2 * C::STAGES + C::SLOTS + s); };
  constexpr int TB0 = 2 * C::STAGES + 2 * C::SLOTS;
  auto tfull_bar = [&](int b) { return bar0 + 8u * (TB0 + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (TB0 + 2 + b); };
  const uint32_t done_bar = bar0 + 8u * (TB0 + 4);
  const uint32_t recv_bar = bar0 + 8u * (TB0 + 5);
  const uint32_t scales_bar = bar0 + 8u * (TB0 + 6);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  // unfused: xs of every slab [slab][token]; fused: the scale-slot ring
  float* xs_tab = reinterpret_cast<float*>(smem + C::OFF_XS);
  float* ws_tab = reinterpret_cast<float*>(smem + C::OFF_WS);   // [slab]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // clusters are runs of `split` consecutive CTAs along x: the K-split rank
  // is the rank in the cluster
  const int split = p.split;
  const int rank = (int)(blockIdx.x % (unsigned)split);
  const int tile = (int)(blockIdx.x / (unsigned)split);
  const int n0 = tile * BW;
  const int kb0 = (int)((int64_t)rank * p.nkb / split);
  const int nsl = (int)((int64_t)(rank + 1) * p.nkb / split) - kb0;  // >= 1

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(full_bar(s), 1 + 32 * C::XW);  // W expect_tx + token loaders' lanes
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int s = 0; s < C::SLOTS; ++s) {
      ptx::mbar_init(sfull_bar(s), 32 * C::XW);  // the token loaders' lanes
      ptx::mbar_init(sempty_bar(s), C::EPI_WARPS);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(tfull_bar(b), 1);
      ptx::mbar_init(tempty_bar(b), C::EPI_WARPS);
    }
    ptx::mbar_init(done_bar, 1);
    // the reduction's first round: (split - 1) peers each send the rows this
    // CTA owns (armed before any peer can send: they send only after a
    // cluster barrier that follows this)
    ptx::mbar_init(recv_bar, 1);
    ptx::mbar_init(scales_bar, 32 * C::XW);  // the token loaders' lanes
    {
      const int mh = reduce_rows_per_round<NT, kFused>(p.m, split);
      const int cnt = owned_lo(rank + 1, mh, split) - owned_lo(rank, mh, split);
      ptx::mbar_arrive_expect_tx(recv_bar, (uint32_t)((split - 1) * cnt * BW * 4));
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) ptx::prefetch_tmap(&tmap_w);
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  // The next kernel on the stream may start its own prologue now (it waits
  // for this one to complete before it reads anything this one writes).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // With static weights the first ring stages of weight slabs, and the
  // weight scales, are fetched before the wait below, so that they stream
  // in while the previous kernel on the stream finishes.
  const int pre = p.static_weights ? min(C::STAGES, nsl) : 0;
  if (threadIdx.x == 0) {
    for (int j = 0; j < pre; ++j) {
      ptx::mbar_arrive_expect_tx(full_bar(j), W_BYTES);
      ptx::tma_load_2d(sbase + j * C::STAGE_BYTES, &tmap_w, full_bar(j), (kb0 + j) * BK, n0);
    }
  }
  // Launched as a programmatic dependent: everything above may overlap the
  // end of the previous kernel on the stream; nothing below runs before that
  // kernel has completed and its memory is visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // The register re-split is issued at the top of each side's branch: code
  // after a join of the two would compile at the smaller share.
  if (warp < C::EPI_WARP0) {
    if (C::SPLIT_REGS) ptx::reg_dealloc<C::REGS_CTRL>();
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      // slabs [0, pre) were issued before the wait (pre <= STAGES)
      uint32_t stage = (uint32_t)(pre % C::STAGES), phase = pre == C::STAGES ? 1u : 0u;
      int issued = pre;
      for (int j = pre; j < nsl; ++j) {
        const int kb = kb0 + j;
        uint32_t okw = 1;
        if (lane == 0) okw = wait_bar(empty_bar(stage), phase ^ 1u, abort_flag, 31) ? 1u : 0u;
        okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
        if (!okw) break;
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx(full_bar(stage), W_BYTES);
          ptx::tma_load_2d(sbase + stage * C::STAGE_BYTES, &tmap_w, full_bar(stage), kb * BK, n0);
        }
        ++issued;
        if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
      }
      // no TMA copy may still be landing when the ring is reused or the CTA
      // retires: wait (bounded) for the last phase of each stage filled
      if (lane == 0 && issued > 0) {
        const int first = issued > C::STAGES ? issued - C::STAGES : 0;
        for (int i = first; i < issued; ++i) {
          const uint32_t s = (uint32_t)(i % C::STAGES);
          const uint32_t par = (uint32_t)((i / C::STAGES) & 1);
          const uint64_t t0 = ptx::globaltimer();
          while (!ptx::mbar_try_wait(full_bar(s), par)) {
            if (ptx::globaltimer() - t0 > WAIT_LIMIT_NS) { record_error(33); break; }
          }
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      // ------------------------------------------------------------- MMA issue
      if (lane == 0) {
        uint32_t stage = 0, phase = 0, tb = 0, tphase = 0;
        for (int j = 0; j < nsl; ++j) {
          if (!wait_bar(tempty_bar(tb), tphase ^ 1u, abort_flag, 34)) break;
          if (g_w8a8_small_gemm_force_timeout) { record_error(35); *abort_flag = 1; break; }
          if (!wait_bar(full_bar(stage), phase, abort_flag, 35)) break;
          // the token rows were written by cp.async (generic proxy); the MMA
          // reads them through the async proxy
          ptx::fence_proxy_async_smem();
          ptx::tc_fence_after();
          const uint32_t sa = sbase + stage * C::STAGE_BYTES;
          const uint64_t adesc = ptx::smem_desc_kmajor_sw128(sa);
          const uint64_t bdesc = ptx::smem_desc_kmajor_sw128(sa + W_BYTES);
          const uint32_t dcol = tmem_base + tb * NT;
  #pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk)  // K = 32 bytes per MMA: +2 in the >>4 field
            ptx::mma_f8f6f4(dcol, adesc + 2u * kk, bdesc + 2u * kk, C::IDESC, kk > 0 ? 1u : 0u);
          ptx::mma_commit(empty_bar(stage));
          ptx::mma_commit(tfull_bar(tb));
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
          if (++tb == 2) { tb = 0; tphase ^= 1u; }
        }
        ptx::mma_commit(done_bar);
        const uint64_t t0 = ptx::globaltimer();
        while (!ptx::mbar_try_wait(done_bar, 0)) {
          if (ptx::globaltimer() - t0 > WAIT_LIMIT_NS) { record_error(36); break; }
        }
      }
      __syncwarp();
    } else if (kFused) {
      // ------------------------------------------- token loaders + quantizer
      // Loader warp w owns token rows 8 (i XW + w) + [0, 8), i = 0, 1, ...
      // It copies them, BF16, into the stage's staging area by 16-byte
      // cp.async, STAGES slabs ahead (one copy group per slab), and codes
      // them from there once they have landed:
      //  * four lanes take one 1 x 128 group (row r, slab kb); lane `sub`
      //    holds elements [32 sub, 32 sub + 32);
      //  * the group's amax is reduced over the four lanes, S = RN32(amax /
      //    448) (S = 1 for an all-zero group), and each element is coded as
      //    E4M3(RN32(x / S)) -- the activation quantizer's arithmetic, bit
      //    for bit;
      //  * lane `sub`'s 32 codes (code chunks 2 sub, 2 sub + 1) go to chunk
      //    c ^ (r % 8) of the row (the 128-byte swizzle), S to the slab's
      //    scale slot.
      // Rows past m and elements past k read as zero (codes 0, S = 1).  In
      // the staging area chunk c of row r sits at (c & 8) | ((c ^ r) & 7), so
      // the 8 rows a warp reads at once fall in distinct banks.  The CTAs of
      // the first weight tile also write the codes and scales out.
      const int w = warp - 2;
      const int sub = lane & 3, gi = lane >> 2;
      constexpr int ITERS = NT / (8 * C::XW);
      const bool write_out = tile == 0 && p.xq_out != nullptr;
      auto staging = [&](int st) { return sbase + st * C::STAGE_BYTES + W_BYTES + C::X_BYTES; };
      // copies of slab j (this warp's rows) into stage j % STAGES
      auto copy_slab = [&](int j) {
        const uint32_t xb = staging(j % C::STAGES);
        const int c = lane & 15;
        const int col = (kb0 + j) * BK + 8 * c;
  #pragma unroll
        for (int it = 0; it < ITERS; ++it) {
  #pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int r = 8 * (it * C::XW + w) + 2 * t + (lane >> 4);
            const bool in = r < p.m && col < p.k;
            ptx::cp_async_16(xb + (uint32_t)(r * 256 + (((c & 8) | ((c ^ r) & 7)) << 4)),
                             in ? p.xb + (int64_t)r * p.k + col : p.xb, in ? 16u : 0u);
          }
        }
        ptx::cp_async_commit();
      };
      for (int j = 0; j < min(C::STAGES, nsl); ++j) copy_slab(j);
      uint32_t stage = 0, phase = 0;
      for (int j = 0; j < nsl; ++j) {
        const int sl = j % C::SLOTS;
        // this lane's copies of slab j have landed, then every lane's
        if (nsl - 1 - j >= C::STAGES - 1) ptx::cp_async_wait_group<C::STAGES - 1>();
        else ptx::cp_async_wait_group<0>();
        __syncwarp();
        uint32_t okw = 1;
        if (lane == 0)
          okw = (wait_bar(empty_bar(stage), phase ^ 1u, abort_flag, 31) &&
                 wait_bar(sempty_bar(sl), (uint32_t)(((j / C::SLOTS) & 1) ^ 1), abort_flag, 31))
                    ? 1u : 0u;
        okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
        if (!okw) break;
        const int kb = kb0 + j;
        const uint32_t sx = sbase + stage * C::STAGE_BYTES + W_BYTES;
        const uint32_t xb = staging(stage);
        float* slot = xs_tab + sl * NT;
  #pragma unroll
        for (int it = 0; it < ITERS; ++it) {
          const int r = 8 * (it * C::XW + w) + gi;
          const bool rin = r < p.m;
          const int col = kb * BK + 32 * sub;
          uint4 v[4];
  #pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int c = 4 * sub + i;
            v[i] = ptx::lds128(xb + (uint32_t)(r * 256 + (((c & 8) | ((c ^ r) & 7)) << 4)));
          }
          float a = absmax_bf16x8_tree<4>(v);
          a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
          a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
          const float S = scale_from_amax(a);
          const QuantScale qs = make_quant_scale(S);
          uint32_t cw[8];
  #pragma unroll
          for (int i = 0; i < 4; ++i) {
            cw[2 * i] = quant_bf16x4(v[i].x, v[i].y, qs);
            cw[2 * i + 1] = quant_bf16x4(v[i].z, v[i].w, qs);
          }
          const uint32_t rb = sx + (uint32_t)(r * 128);
          ptx::sts128(rb + ((uint32_t)((2 * sub) ^ (r & 7)) << 4), cw[0], cw[1], cw[2], cw[3]);
          ptx::sts128(rb + ((uint32_t)((2 * sub + 1) ^ (r & 7)) << 4), cw[4], cw[5], cw[6], cw[7]);
          if (sub == 0) slot[r] = S;
          if (write_out && rin) {
            uint8_t* dst = p.xq_out + (int64_t)r * p.k + col;
            if (col < p.k) *reinterpret_cast<uint4*>(dst) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
            if (col + 16 < p.k)
              *reinterpret_cast<uint4*>(dst + 16) = make_uint4(cw[4], cw[5], cw[6], cw[7]);
            if (sub == 0) p.xs_out[(int64_t)r * p.nkb + kb] = S;
          }
        }
        // the codes were written by the generic proxy; the MMA reads them
        // through the async proxy
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(full_bar(stage));
        ptx::mbar_arrive(sfull_bar(sl));
        // the staging rows of this stage are free again: next slab for it
        __syncwarp();
        if (j + C::STAGES < nsl) copy_slab(j + C::STAGES);
        if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
      }
      ptx::cp_async_wait_all();
      __syncwarp();
    } else {
      // -------------------------------------------------------- token loaders
      // Lane l of loader warp w copies 16-byte chunk l % 8 of token rows
      // 4 (i XW + w) + l / 8, i = 0, 1, ...: each warp-wide copy moves four
      // whole 128-byte rows.  Chunk c of row r sits at chunk c ^ (r % 8) of
      // the row (the 128-byte swizzle the MMA descriptor names).
      const int w = warp - 2;
      const int q = lane >> 3, c = lane & 7;
      constexpr int ITERS = NT / (4 * C::XW);
      if (C::LOADER_SCALES) {
        // the CTA's scale tables first: xs[token][kb0 .. kb0 + nsl) transposed
        // to [slab][token] (tokens past m read as 0; loader thread lt takes
        // token lt % 32 + 32 i, every slab) and ws[tile][kb0 .. kb0 + nsl);
        // their arrival is signalled on scales_bar
        const int lt = threadIdx.x - 64;
        constexpr int LT = 32 * C::XW;
        for (int t = lt; t < NT; t += LT) {
          const bool in = t < p.m;
          const float* src = p.xs + (in ? (int64_t)t * p.nkb + kb0 : 0);
          for (int j = 0; j < nsl; ++j)
            ptx::cp_async_4(ptx::smem_addr(xs_tab + j * NT + t), in ? src + j : p.xs, in ? 4u : 0u);
        }
        for (int j = lt; j < nsl; j += LT)
          ptx::cp_async_4(ptx::smem_addr(ws_tab + j), p.ws + (int64_t)tile * p.nkb + kb0 + j, 4u);
        ptx::cp_async_arrive_noinc(scales_bar);
      }
      uint32_t stage = 0, phase = 0;
      for (int j = 0; j < nsl; ++j) {
        uint32_t okw = 1;
        if (lane == 0) okw = wait_bar(empty_bar(stage), phase ^ 1u, abort_flag, 31) ? 1u : 0u;
        okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
        if (!okw) break;
        const uint32_t sx = sbase + stage * C::STAGE_BYTES + W_BYTES;
        const int kc = (kb0 + j) * BK + c * 16;
        const bool kin = kc < p.k;
  #pragma unroll
        for (int i = 0; i < ITERS; ++i) {
          const int r = 4 * (i * C::XW + w) + q;
          const bool in = kin && r < p.m;
          ptx::cp_async_16(sx + (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)),
                           in ? p.xq + (int64_t)r * p.k + kc : p.xq, in ? 16u : 0u);
        }
        ptx::cp_async_arrive_noinc(full_bar(stage));
        if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
      }
      ptx::cp_async_wait_all();
      __syncwarp();
    }
    const float2 none[C::COLS / 2] = {};
    reduce_store<NT, kFused, false>(p, smem, sbase, recv_bar, rank, split, n0, warp, lane, 0, none);
  } else {
    if (C::SPLIT_REGS) ptx::reg_alloc<C::REGS_EPI>();
    // ------------------------------------------------------------ promotion
    const int ew = warp - C::EPI_WARP0;
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int c0 = (ew >> 2) * C::COLS;  // first token column of this warp
    // The CTA's scales, fetched by these warps alone while the first slabs
    // stream in: xs[token][kb0 .. kb0 + nsl) transposed to [slab][token]
    // (tokens past m read as 0; thread et takes token et % NT, every
    // (ET / NT)-th slab) and ws[tile][kb0 .. kb0 + nsl).
    const int et = threadIdx.x - 32 * C::EPI_WARP0;
    constexpr int ET = 32 * C::EPI_WARPS;
    if (C::LOADER_SCALES) {
      // the token loaders' fetch of the scale tables has landed: every lane
      // waits on the barrier itself, since every lane reads the tables next
      // (on a timeout the abort flag stops the loop below)
      wait_bar(scales_bar, 0, abort_flag, 32);
    } else {
      static_assert(ET % NT == 0 || kFused, "whole tokens per thread group");
      if (!kFused) {
        const int t = et % NT;
        const bool in = t < p.m;
        const float* src = p.xs + (in ? (int64_t)t * p.nkb + kb0 : 0);
        for (int j = et / NT; j < nsl; j += ET / NT)
          ptx::cp_async_4(ptx::smem_addr(xs_tab + j * NT + t), in ? src + j : p.xs, in ? 4u : 0u);
      }
      for (int j = et; j < nsl; j += ET)
        ptx::cp_async_4(ptx::smem_addr(ws_tab + j), p.ws + (int64_t)tile * p.nkb + kb0 + j, 4u);
      ptx::cp_async_wait_all();
      ptx::named_bar_sync(1, ET);
    }
    if (!kFused) {
      // Each slab's token scales times the tile's weight scale, once per
      // CTA: s[j][t] = xs[t][kb0 + j] * ws[tile][kb0 + j], the factor every
      // partial of slab j, token t is multiplied by.
      for (int i = et; i < nsl * NT; i += ET) xs_tab[i] *= ws_tab[i / NT];
      ptx::named_bar_sync(1, ET);
    }
    float2 acc[C::COLS / 2];
#pragma unroll
    for (int i = 0; i < C::COLS / 2; ++i) acc[i] = make_float2(0.0f, 0.0f);
    uint32_t tb = 0, tphase = 0;
    for (int j = 0; j < nsl; ++j) {
      const int sl = j % C::SLOTS;
      uint32_t okw = 1;
      if (lane == 0)
        okw = (wait_bar(tfull_bar(tb), tphase, abort_flag, 32) &&
               (!kFused ||
                wait_bar(sfull_bar(sl), (uint32_t)((j / C::SLOTS) & 1), abort_flag, 32)))
                  ? 1u : 0u;
      okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
      if (!okw) break;
      ptx::tc_fence_after();
      const float* slot = xs_tab + (kFused ? sl : j) * NT;
      const float2 w2 = make_float2(ws_tab[j], ws_tab[j]);
      const uint32_t tcol = tmem_base + ((uint32_t)(quarter * 32) << 16) + tb * NT + c0;
      // The slab's partial comes out of TMEM STEP columns at a time, the
      // next step's load in flight while the current one is multiplied in.
      constexpr int STEP = C::PROM_STEP, NSTEP = C::COLS / STEP;
      auto hand_back = [&]() {
        // the buffer's last load has landed: hand it back to the MMA
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(tempty_bar(tb));
      };
      uint32_t ra[STEP], rb[STEP];
      tmem_load<STEP>(tcol, ra);
      tmem_wait<STEP>(ra);
      if (NSTEP == 1) hand_back();
#pragma unroll
      for (int cc = 0; cc < NSTEP; ++cc) {
        uint32_t(&cur)[STEP] = (cc & 1) ? rb : ra;
        uint32_t(&nxt)[STEP] = (cc & 1) ? ra : rb;
        if (cc + 1 < NSTEP) tmem_load<STEP>(tcol + (cc + 1) * STEP, nxt);
#pragma unroll
        for (int e = 0; e < STEP / 4; ++e) {
          const float4 x4 = *reinterpret_cast<const float4*>(slot + c0 + cc * STEP + 4 * e);
          float2 s01 = make_float2(x4.x, x4.y), s23 = make_float2(x4.z, x4.w);
          if (kFused) {  // unfused: the table holds the products already
            s01 = __fmul2_rn(s01, w2);
            s23 = __fmul2_rn(s23, w2);
          }
          const int a = cc * (STEP / 2) + 2 * e;
          acc[a] = __ffma2_rn(
              make_float2(__uint_as_float(cur[4 * e]), __uint_as_float(cur[4 * e + 1])), s01,
              acc[a]);
          acc[a + 1] = __ffma2_rn(
              make_float2(__uint_as_float(cur[4 * e + 2]), __uint_as_float(cur[4 * e + 3])), s23,
              acc[a + 1]);
        }
        if (cc + 1 < NSTEP) tmem_wait<STEP>(nxt);
        if (cc + 2 == NSTEP) hand_back();
      }
      if (kFused) {
        // the slab's scales have been read: hand the slot back to the loaders
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(sempty_bar(sl));
      }
      if (++tb == 2) { tb = 0; tphase ^= 1u; }
    }
    reduce_store<NT, kFused, true>(p, smem, sbase, recv_bar, rank, split, n0, warp, lane, c0, acc);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// Most clusters of `split` CTAs that fit on the device at once (cached per
// device).
template <int NT, bool kFused>
static int max_active_clusters(int split) {
  static int cache[64][MAX_SPLIT + 1] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cache[dev][split] > 0) return cache[dev][split];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)split, 1, 1);
  cfg.blockDim = dim3(Cfg<NT, kFused>::THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg<NT, kFused>::SMEM;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fp8_gemm_small_m_kernel<NT, kFused>, &cfg) !=
          cudaSuccess ||
      n <= 0) {
    cudaGetLastError();  // the query failed: assume one cluster per `split` SMs
    n = std::max(1, sm_count() / split);
  }
  cache[dev][split] = n;
  return n;
}

// Split of K over a cluster, chosen by a cost model fitted to timings of
// the Qwen3-8B decode linears on GB300: a wave of clusters costs a fixed
// part (launch, prologue, pipeline fill, reduction) worth FILL slabs plus
// the slabs of each CTA, and the model makes waves x (FILL + slabs per CTA)
// smallest.  The occupancy query counts one CTA per SM; up to 64 tokens two
// CTAs share an SM, which doubles the clusters resident at once.
template <int NT, bool kFused>
static int choose_split(int tiles, int nkb) {
  constexpr double FILL = NT <= 64 ? 23.0 : (NT <= 128 ? 20.0 : 13.0);
  constexpr int PER_SM = (NT <= 64 && !kFused) ? 2 : 1;
  int best = MAX_SPLIT;
  double best_cost = 1e30;
  for (int s = 1; s <= std::min(MAX_SPLIT, nkb); ++s) {
    if ((nkb + s - 1) / s > Cfg<NT, kFused>::MAX_SLABS) continue;  // the scale table's size
    const int fit = PER_SM * max_active_clusters<NT, kFused>(s);
    const double waves = (double)((tiles + fit - 1) / fit);
    const double cost = waves * (FILL + (double)((nkb + s - 1) / s));
    if (cost < best_cost - 1e-9) { best_cost = cost; best = s; }
  }
  return best;
}

// p: every field but split set by the caller.
template <int NT, bool kFused>
static cudaError_t launch_nt(Params p, const uint8_t* wq, cudaStream_t st) {
  using C = Cfg<NT, kFused>;
  CUtensorMap tw;
  if (!make_tmap_2d(&tw, wq, 1, (uint64_t)p.n, (uint64_t)p.k, BW, BK,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(fp8_gemm_small_m_kernel<NT, kFused>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = 1;
  }
  const int tiles = (p.n + BW - 1) / BW;
  p.split = choose_split<NT, kFused>(tiles, p.nkb);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.split * tiles), 1, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch: the prologue (barriers, TMEM, tensor-map
  // prefetch) overlaps the previous kernel's tail
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, fp8_gemm_small_m_kernel<NT, kFused>, tw, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

static Params make_params(const float* ws, uint16_t* y, int64_t m, int64_t n, int64_t k,
                          bool static_weights) {
  Params p{};
  p.ws = ws; p.y = y;
  p.m = (int32_t)m; p.n = (int32_t)n; p.k = (int32_t)k;
  p.nkb = (int32_t)((k + BK - 1) / BK);
  p.static_weights = static_weights ? 1 : 0;
  return p;
}

}  // namespace sgemm

constexpr int BW_TILE = sgemm::BW;
constexpr int FUSED_MAX_TILES = 8;

bool block_gemm_small_m_serves(int64_t m, int64_t n, int64_t k) {
  // a split of at most MAX_SPLIT CTAs must leave each at most MAX_SLABS slabs
  if (m < 1 || m > 256 || k < 1 ||
      (k + sgemm::BK * sgemm::MAX_SPLIT - 1) / (sgemm::BK * sgemm::MAX_SPLIT) >
          sgemm::Cfg<256>::MAX_SLABS)
    return false;
  // Past 128 rows the token operand outweighs a 128-row weight tile, and
  // the 128 x 256-tile kernel is faster wherever its tiles alone fill a
  // quarter of the SMs (measured on the Qwen3-8B linears at m = 256: qkv
  // 22.6 against 41.9 us, gate_up 41.2 against 87.1 us; o and down, with 32
  // tiles each, 21.6 and 39.5 us here against 22.6 and 54.2 us there).
  if (m > 128) return ((m + 127) / 128) * ((n + 255) / 256) * 4 < (int64_t)sm_count();
  return true;
}

cudaError_t set_small_gemm_force_timeout(int on) {
  return cudaMemcpyToSymbol(g_w8a8_small_gemm_force_timeout, &on, sizeof(int));
}

cudaError_t consume_small_gemm_error(int* code) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_w8a8_small_gemm_error, sizeof(int));
  if (e != cudaSuccess) return e;
  if (v != 0) {
    int z = 0;
    e = cudaMemcpyToSymbol(g_w8a8_small_gemm_error, &z, sizeof(int));
  }
  *code = v;
  return e;
}

cudaError_t launch_block_gemm_small_m(const uint8_t* xq, const float* xs, const uint8_t* wq,
                                      const float* ws, uint16_t* y, int64_t m, int64_t n,
                                      int64_t k, bool static_weights, cudaStream_t st) {
  using namespace sgemm;
  if (!block_gemm_small_m_serves(m, n, k) || n <= 0) return cudaErrorInvalidValue;
  Params p = make_params(ws, y, m, n, k, static_weights);
  p.xq = xq; p.xs = xs;
  if (m <= 32) return launch_nt<32, false>(p, wq, st);
  if (m <= 64) return launch_nt<64, false>(p, wq, st);
  if (m <= 128) return launch_nt<128, false>(p, wq, st);
  return launch_nt<256, false>(p, wq, st);
}

bool linear_fused_possible(int64_t m, int64_t n, int64_t k);

bool linear_fused_serves(int64_t m, int64_t n, int64_t k) {
  // Every weight-tile CTA quantizes the token rows of its slabs, so the
  // quantization is repeated once per 128 output columns: measured on the
  // Qwen3-8B linears at m = 64 (48 to 192 tiles) the single kernel took 55
  // to 73 us a linear against 19 us for quantizer + GEMM.  It is kept for
  // narrow outputs, where that repetition is small.
  return linear_fused_possible(m, n, k) && (n + BW_TILE - 1) / BW_TILE <= FUSED_MAX_TILES;
}

bool linear_fused_possible(int64_t m, int64_t n, int64_t k) {
  return m <= 128 && block_gemm_small_m_serves(m, n, k);
}

cudaError_t launch_linear_fused(const uint16_t* x, const uint8_t* wq, const float* ws,
                                uint16_t* y, uint8_t* xq_out, float* xs_out, int64_t m,
                                int64_t n, int64_t k, bool static_weights, cudaStream_t st) {
  using namespace sgemm;
  if (!linear_fused_possible(m, n, k) || n <= 0) return cudaErrorInvalidValue;
  Params p = make_params(ws, y, m, n, k, static_weights);
  p.xb = x; p.xq_out = xq_out; p.xs_out = xs_out;
  if (m <= 32) return launch_nt<32, true>(p, wq, st);
  if (m <= 64) return launch_nt<64, true>(p, wq, st);
  return launch_nt<128, true>(p, wq, st);
}

}  // namespace w8a8
