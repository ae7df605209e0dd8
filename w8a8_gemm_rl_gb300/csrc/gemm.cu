// gemm.cu -- blockwise-scaled FP8 (E4M3) GEMM and its grouped (MoE) variant
// on the 5th-generation tensor cores of sm_103a.
//
// What is computed (NeMo RL FP8 blog, Table 1; "Unified FP8" notes, scale
// choice: FP32 scales):
//   Y[i,j] = BF16( sum_kb xs[i,kb] * ws[j/128,kb] * P[i,j,kb] ),
//   P[i,j,kb] = sum_{k in 128-wide slab kb} dec(xq[i,k]) * dec(wq[j,k]),
// FP32 accumulation.  The scales are FP32 and differ per (row, slab) and per
// (128-column block, slab), so they cannot ride on the hardware's UE8M0
// block-scaled MMA; instead every slab's partial P is produced on its own in
// tensor memory and promoted into FP32 registers with its scale.
//
// Kernel structure (persistent, one CTA per SM, warp-specialized):
//   warp 0      producer: TMA of the A and B K-slabs into a 3-stage
//               shared-memory ring (for routed MoE rows, B by TMA and A rows
//               0-63 by a cp.async gather);
//   warp 1      allocates 512 TMEM columns; lane 0 issues 4 x
//               tcgen05.mma.kind::f8f6f4 (128 x 256 x 32) per slab into one
//               of two 256-column TMEM buffers, then commits to mbarriers;
//   warp 2      waits for each slab's MMAs and releases the promotion warps
//               through a named barrier per TMEM buffer;
//   warp 3      stages each slab's scales (xs of the tile's rows, ws of its
//               two column blocks) into a shared-memory ring, two slabs ahead;
//               for routed MoE rows it gathers A rows 64-127 instead, and
//               warp 2 stages the scales;
//   warps 4..11 promotion: tcgen05.ld of the slab partial, acc += P * s in
//               FP32 registers (128 per thread), release the TMEM buffer,
//               and after the last slab round to BF16 and store.
// With two TMEM buffers the MMA of slab kb+1 overlaps the promotion of slab
// kb.  Tiles are 128 x 256; tiles are visited in groups of 8 M-tiles so the
// CTAs running at once share A and B tiles through L2.
//
// Every mbarrier wait is bounded (2 s of wall time).  A wait that gives up
// records an error code in g_w8a8_gemm_error, tells the other roles to stop,
// waits for its own copies / MMAs in flight, frees TMEM and returns.
#include <algorithm>

#include "kernels.h"
#include "ptx.cuh"
#include "tmap.h"

namespace w8a8 {

__device__ int g_w8a8_gemm_error = 0;
// Test hook (w8a8_debug_force_wait_timeout): when set, the MMA issuer's
// first wait gives up at once, as if its time limit had passed, so that the
// abort path (stop, drain copies and MMAs, free TMEM) runs on demand.
__device__ int g_w8a8_gemm_force_timeout = 0;

namespace gemm {

constexpr int BM = 128;
// Tile width: 256 columns, or 128 for the dense GEMM when 256-wide tiles
// would leave SMs idle (few rows); each of the 8 promotion warps takes half.
constexpr int BN = 256;
constexpr int BN_NARROW = 128;
constexpr int BK = 128;  // FP8 elements = bytes = one 128-byte swizzle row
constexpr int STAGES = 3;
constexpr int A_BYTES = BM * BK;
__host__ __device__ constexpr int b_bytes(int bn) { return bn * BK; }
__host__ __device__ constexpr int ring_stage_bytes(int bn) { return A_BYTES + b_bytes(bn); }
constexpr int NUM_EPI_WARPS = 8;
constexpr int EPI_WARP0 = 4;  // warpgroup 0: producer, MMA, hand-off, gather
constexpr int THREADS = 32 * EPI_WARP0 + 32 * NUM_EPI_WARPS;
// Registers: launched at 168 per thread (384 threads = 64512); warpgroup 0
// drops to 72 and the two promotion warpgroups rise to 216:
// 128 * 72 + 256 * 216 = 64512.
constexpr int REGS_LAUNCH = 168, REGS_CTRL = 72, REGS_EPI = 216;
static_assert(128 * REGS_CTRL + 256 * REGS_EPI <= THREADS * REGS_LAUNCH, "register split");
constexpr int RASTER_M = 8;
constexpr int MAX_GROUPS = 1024;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr uint64_t ABORT_DRAIN_LIMIT_NS = 10000000000ull;
// named barriers 1 and 2 (0 is __syncthreads): warp 2 hands the slab in
// TMEM buffer b to the promotion warps on barrier BAR_SLAB + b
constexpr uint32_t BAR_SLAB = 1;
constexpr uint32_t BAR_SLAB_THREADS = 32 * (1 + NUM_EPI_WARPS);

// shared-memory map (offsets from a 1024-byte aligned base)
__host__ __device__ constexpr int off_bars(int bn) { return STAGES * ring_stage_bytes(bn); }
// full, empty, tfull[2], tempty[2], done, then the scale slots' sfull, sempty
constexpr int NUM_BARS = 2 * STAGES + 4 + 1 + 2 * 4;
__host__ __device__ constexpr int off_misc(int bn) { return off_bars(bn) + NUM_BARS * 8; }
enum Mode { DENSE = 0, GROUPED = 1, GATHER = 2 };
// Output staging: each promotion warp writes its 32 rows x bn / 2 columns, in
// bn / 2 / store_cols passes, into private boxes of 32 rows x store_cols BF16
// columns laid out as the TMA's 128-byte swizzle, and one lane stores each
// box to global memory by TMA (64-column boxes: 2% faster than 32-column
// ones, which were 3-6% faster for the grouped GEMM than 16-column ones).
// Each warp has two boxes.  Where a warp's share of a tile takes two passes
// (tiles 256 wide) each pass has its own box, so a tile's stores never wait
// for one another (the one wait, before the first pass, is for the previous
// tile's stores).  With one pass per tile (128 wide) the boxes alternate per
// TMA store issued (not per pass: a partial last N tile issues fewer stores
// than passes, and the box written next must never be the source of the
// newest store, which cp.async.bulk.wait_group.read 1 does not retire).
__host__ __device__ constexpr int store_cols(int) { return 64; }
__host__ __device__ constexpr int stage_boxes(int, int) { return 2; }
// swizzle atoms: 1024-byte aligned
__host__ __device__ constexpr int off_stage(int bn) { return (off_misc(bn) + 16 + 1023) / 1024 * 1024; }
__host__ __device__ constexpr int stage_bytes(int mode, int bn) {
  return NUM_EPI_WARPS * stage_boxes(mode, bn) * 32 * store_cols(mode) * 2;
}
// The promotion's per-slab scales, staged by the hand-off warp: SCALE_SLOTS
// slots, each the 128 row scales xs[row, kb] of the tile and its two
// column-block scales ws[nb, kb] (padded to 16 bytes), filled
// SCALE_LOOKAHEAD slabs ahead of the slab being released.
constexpr int SCALE_SLOTS = 4;
static_assert(NUM_BARS == 2 * STAGES + 5 + 2 * SCALE_SLOTS, "barrier count");
constexpr int SCALE_LOOKAHEAD = 2;
constexpr int SCALE_SLOT_FLOATS = 132;
static_assert(SCALE_SLOTS >= SCALE_LOOKAHEAD + 2, "slots staged ahead plus the two in use");
__host__ __device__ constexpr int off_scales(int mode, int bn) { return off_stage(bn) + stage_bytes(mode, bn); }
__host__ __device__ constexpr int off_groups(int mode, int bn) {
  return off_scales(mode, bn) + SCALE_SLOTS * SCALE_SLOT_FLOATS * 4;
}
__host__ __device__ constexpr int smem_bytes(int mode, int g, int bn) {
  return 1024 + off_groups(mode, bn) + 2 * 4 * (g + 1);
}
static_assert(smem_bytes(DENSE, 1, BN) <= 232448, "shared memory");
static_assert(smem_bytes(DENSE, 1, BN_NARROW) <= 232448, "shared memory");
static_assert(smem_bytes(GATHER, MAX_GROUPS, BN) <= 232448, "shared memory");

struct Params {
  const uint8_t* xq;
  const float* xs;
  const float* ws;
  uint16_t* y;
  const int32_t* row_idx;
  const int32_t* group_offsets;
  int64_t m;       // dense: rows of X and Y; grouped: total routed rows
  int64_t rows_x;  // rows of xq / xs
  int32_t n, k, nkb, nnb;
  int32_t g;
  int32_t num_m_tiles;  // dense
  int32_t num_n_tiles;
};

struct Tile {
  int32_t e;
  int32_t rows;  // valid rows (<= BM)
  int64_t row0;  // first output row (routed order for grouped)
  int32_t n0;
};

__device__ __forceinline__ void record_error(int code) { atomicCAS(&g_w8a8_gemm_error, 0, code); }
__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

// Wait that also gives up early when another role has aborted.
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

template <int kMode, int kBN>
__device__ __forceinline__ Tile decode_tile(const Params& p, int64_t t, const int32_t* s_prefix,
                                            const int32_t* s_start) {
  Tile T;
  // tile indices fit in 32 bits (the launchers check), and 32-bit division
  // is several times cheaper than 64-bit on the tile-boundary critical path
  const uint32_t tt = (uint32_t)t;
  if (kMode == DENSE) {
    const uint32_t per_group = (uint32_t)RASTER_M * (uint32_t)p.num_n_tiles;
    const uint32_t grp = tt / per_group;
    const int32_t first_m = (int32_t)(grp * RASTER_M);
    const uint32_t gm = (uint32_t)min(RASTER_M, p.num_m_tiles - first_m);
    const uint32_t r = tt - grp * per_group;
    const int32_t mt = first_m + (int32_t)(r % gm);
    const int32_t nt = (int32_t)(r / gm);
    T.e = 0;
    T.row0 = (int64_t)mt * BM;
    T.rows = (int32_t)min64(BM, p.m - T.row0);
    T.n0 = nt * kBN;
  } else {
    const int32_t mt_all = (int32_t)(tt / (uint32_t)p.num_n_tiles);
    const int32_t nt = (int32_t)(tt - (uint32_t)mt_all * (uint32_t)p.num_n_tiles);
    int lo = 0, hi = p.g;  // s_prefix[lo] <= mt_all < s_prefix[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_prefix[mid] <= mt_all) lo = mid; else hi = mid;
    }
    const int32_t mt = mt_all - s_prefix[lo];
    const int64_t gstart = s_start[lo];
    const int64_t gend = s_start[lo + 1] > gstart ? s_start[lo + 1] : gstart;
    T.e = lo;
    T.row0 = gstart + (int64_t)mt * BM;
    T.rows = (int32_t)min64(BM, gend - T.row0);
    T.n0 = nt * kBN;
  }
  return T;
}

// A lane's share of one tile's scale sources: rows lane + 32 i (i < 4) of
// xs (row index, or invalid: past the tile, past rows_x, or a routed index
// out of range) and the tile's two column blocks of ws (first element of the
// block's row of slabs, or invalid: past n).
struct ScaleSrc {
  int32_t row[4];
  uint32_t row_ok;  // bit i: row[i] valid
  int64_t blk[2];
  uint32_t blk_ok;  // bit h: blk[h] valid
};

template <int kMode>
__device__ __forceinline__ ScaleSrc scale_sources(const Params& p, const Tile& T, int lane) {
  ScaleSrc S;
  S.row_ok = 0;
  S.blk_ok = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = lane + 32 * i;
    int64_t sr = -1;
    if (r < T.rows) sr = kMode == GATHER ? (int64_t)p.row_idx[T.row0 + r] : T.row0 + r;
    const bool v = sr >= 0 && sr < p.rows_x;
    S.row[i] = v ? (int32_t)sr : 0;
    S.row_ok |= (v ? 1u : 0u) << i;
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int nb = (T.n0 >> 7) + h;
    const bool v = nb < p.nnb;
    S.blk[h] = ((int64_t)T.e * p.nnb + (v ? nb : 0)) * p.nkb;
    S.blk_ok |= (v ? 1u : 0u) << h;
  }
  return S;
}

// Slab kb's scales into a slot: 128 row scales, then the two block scales
// (4-byte cp.async; invalid sources write 0).
__device__ __forceinline__ void stage_scales(const Params& p, const ScaleSrc& S, int kb,
                                             uint32_t slot, int lane) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool v = (S.row_ok >> i) & 1u;
    ptx::cp_async_4(slot + 4u * (uint32_t)(lane + 32 * i),
                    v ? p.xs + (int64_t)S.row[i] * p.nkb + kb : p.xs, v ? 4u : 0u);
  }
  if (lane < 2) {
    const bool v = (S.blk_ok >> lane) & 1u;
    const int64_t b = lane == 0 ? S.blk[0] : S.blk[1];
    ptx::cp_async_4(slot + 4u * (uint32_t)(128 + lane), v ? p.ws + b + kb : p.ws, v ? 4u : 0u);
  }
}

template <int kMode, int kBN>
__global__ void __launch_bounds__(THREADS, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                    const __grid_constant__ CUtensorMap tmap_b,
                    const __grid_constant__ CUtensorMap tmap_y, const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_addr(smem);
  constexpr int STAGE_BYTES = ring_stage_bytes(kBN);
  constexpr int TMEM_COLS = 2 * kBN;
  constexpr uint32_t IDESC = ptx::idesc_e4m3_f32(BM, kBN);
  constexpr int OFF_MISC = off_misc(kBN);
  const uint32_t bar0 = sbase + off_bars(kBN);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t done_bar = bar0 + 8u * (2 * STAGES + 4);
  auto sfull_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + 5 + s); };
  auto sempty_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + 5 + SCALE_SLOTS + s); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  int32_t* s_prefix = reinterpret_cast<int32_t*>(smem + off_groups(kMode, kBN));
  int32_t* s_start = s_prefix + (p.g + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(full_bar(s), kMode == GATHER ? 1 + 64 : 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(tfull_bar(b), 1);
      ptx::mbar_init(tempty_bar(b), NUM_EPI_WARPS);
    }
    ptx::mbar_init(done_bar, 1);
    for (int s = 0; s < SCALE_SLOTS; ++s) {
      ptx::mbar_init(sfull_bar(s), 32);  // the scale stager's lanes (cp.async arrivals)
      ptx::mbar_init(sempty_bar(s), 1);  // the hand-off warp, once the slot is read
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmap_b);
    if (kMode != GATHER) ptx::prefetch_tmap(&tmap_a);
    ptx::prefetch_tmap(&tmap_y);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), TMEM_COLS);
    ptx::tmem_relinquish();
  }
  int64_t num_tiles;
  if (kMode == DENSE) {
    num_tiles = (int64_t)p.num_m_tiles * p.num_n_tiles;
  } else {
    // per-group start row (clamped to [0, m]) and prefix sums of M-tiles
    if (warp == 2) {
      const int G = p.g;
      const int per = (G + 31) / 32;
      const int e0 = min(lane * per, G), e1 = min(e0 + per, G);
      int32_t local = 0;
      for (int e = e0; e < e1; ++e) {
        int64_t a = p.group_offsets[e], b = p.group_offsets[e + 1];
        a = min64(max64(a, 0), p.m);
        b = min64(max64(b, a), p.m);
        s_start[e] = (int32_t)a;
        local += (int32_t)((b - a + BM - 1) / BM);
      }
      int32_t incl = local;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
      }
      int32_t run = incl - local;
      for (int e = e0; e < e1; ++e) {
        s_prefix[e] = run;
        int64_t a = s_start[e], b = p.group_offsets[e + 1];
        b = min64(max64(b, a), p.m);
        run += (int32_t)((b - a + BM - 1) / BM);
      }
      if (lane == 31) {
        s_prefix[G] = incl;
        int64_t last = p.group_offsets[G];
        s_start[G] = (int32_t)min64(max64(last, 0), p.m);
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (kMode != DENSE) num_tiles = (int64_t)s_prefix[p.g] * p.num_n_tiles;

  const int nkb = p.nkb;

  if (warp < EPI_WARP0) {
  // warpgroup 0 hands registers to the promotion warpgroups (one setmaxnreg
  // for the whole warpgroup)
  ptx::reg_dealloc<REGS_CTRL>();
  if (warp == 0 || (kMode == GATHER && warp == 3)) {
    // ------------------------------------------------------------ producer
    uint32_t stage = 0, phase = 0;
    int64_t issued = 0;  // stages whose B slab (and A slab) lane 0 of warp 0 loaded by TMA
    bool ok = true;
    if (kMode != GATHER) {
      if (lane == 0) {
        for (int64_t t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
          const Tile T = decode_tile<kMode, kBN>(p, t, s_prefix, s_start);
          const int brow = T.e * p.n + T.n0;
          for (int kb = 0; kb < nkb; ++kb) {
            if (!wait_bar(empty_bar(stage), phase ^ 1u, abort_flag, 1)) { ok = false; break; }
            const uint32_t sa = sbase + stage * STAGE_BYTES;
            ptx::mbar_arrive_expect_tx(full_bar(stage), STAGE_BYTES);
            ptx::tma_load_2d(sa, &tmap_a, full_bar(stage), kb * BK, (int)T.row0);
            ptx::tma_load_2d(sa + A_BYTES, &tmap_b, full_bar(stage), kb * BK, brow);
            ++issued;
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
        }
      }
    } else {
      // Routed rows: warps 0 and 3 copy tile rows 0-63 and 64-127 of each A
      // slab with 16-byte cp.async into the 128-byte-swizzled layout the MMA
      // expects; lane 0 of warp 0 also brings the B slab by TMA.  Lane l
      // takes chunk l % 8 of rows 64w + 4j + l / 8 (j = 0..15), so every
      // warp-wide copy moves four whole 128-byte rows.  A row past the
      // group's end, or whose index lies outside [0, rows_x), is zero-filled.
      // Each lane's copies of a stage arrive on the stage's full barrier once
      // they have landed (cp.async.mbarrier.arrive), so the warps never wait
      // for their own copies and keep up to STAGES slabs in flight.
      const int w = warp == 0 ? 0 : 1;
      const int q = lane >> 3, c = lane & 7;
      // swizzled offset of (row 64w + 4j + q, chunk c): (row & 7) = 4 (j & 1) + q
      const uint32_t dofs_even = (uint32_t)((64 * w + q) * 128 + ((c ^ q) << 4));
      const uint32_t dofs_odd = (uint32_t)((64 * w + q) * 128 + ((c ^ (q | 4)) << 4));
      for (int64_t t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        const Tile T = decode_tile<kMode, kBN>(p, t, s_prefix, s_start);
        const int brow = T.e * p.n + T.n0;
        int32_t src_row[16];
        uint32_t valid = 0;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int r = 64 * w + 4 * j + q;
          int64_t sr = -1;
          if (r < T.rows) sr = p.row_idx[T.row0 + r];
          const bool v = sr >= 0 && sr < p.rows_x;
          src_row[j] = v ? (int32_t)sr : 0;
          valid |= (v ? 1u : 0u) << j;
        }
        for (int kb = 0; kb < nkb; ++kb) {
          uint32_t okw = 1;
          if (lane == 0) okw = wait_bar(empty_bar(stage), phase ^ 1u, abort_flag, 2) ? 1u : 0u;
          okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
          if (!okw) { ok = false; break; }
          const uint32_t sa = sbase + stage * STAGE_BYTES;
          if (warp == 0 && lane == 0) {
            ptx::mbar_arrive_expect_tx(full_bar(stage), b_bytes(kBN));
            ptx::tma_load_2d(sa + A_BYTES, &tmap_b, full_bar(stage), kb * BK, brow);
            ++issued;
          }
          const int kc = kb * BK + c * 16;
          const uint32_t vk = kc < p.k ? valid : 0u;
          const uint8_t* xk = p.xq + kc;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const bool in = (vk >> j) & 1u;
            ptx::cp_async_16(sa + 512u * j + ((j & 1) ? dofs_odd : dofs_even),
                             in ? xk + (int64_t)src_row[j] * p.k : p.xq, in ? 16u : 0u);
          }
          ptx::cp_async_arrive_noinc(full_bar(stage));
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      ptx::cp_async_wait_all();
    }
    // Before leaving, make sure no TMA copy is still landing in shared
    // memory: wait (bounded) for the last phase of each stage filled.
    if (warp == 0 && lane == 0 && issued > 0) {
      const int64_t first = issued > STAGES ? issued - STAGES : 0;
      for (int64_t i = first; i < issued; ++i) {
        const uint32_t s = (uint32_t)(i % STAGES);
        const uint32_t par = (uint32_t)((i / STAGES) & 1);
        const uint64_t t0 = ptx::globaltimer();
        while (!ptx::mbar_try_wait(full_bar(s), par)) {
          if (ptx::globaltimer() - t0 > WAIT_LIMIT_NS) { record_error(3); break; }
        }
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------ slab hand-off
    // Lane 0 waits for each slab's MMAs to finish; then the warp releases the
    // eight promotion warps through the named barrier of the slab's TMEM
    // buffer.  A hardware barrier wakes all eight at once; waiting on the
    // MMA's mbarrier (or polling a shared-memory word) themselves, they woke
    // hundreds of cycles apart, and the slowest one gates the next MMA into
    // that buffer.
    //
    // Why the promotion warps can never be left waiting: this warp arrives
    // exactly once per slab of the CTA's tile sequence, and the promotion
    // warps wait exactly once per slab, on barrier 1 + buffer.  An arrival
    // for slab j on buffer b's barrier must not come before all eight warps
    // have passed that barrier for slab j-2, or the two generations would
    // mix.  Normally this holds because slab j's MMA was issued only after
    // the eight warps released buffer b (tempty) after slab j-2.  After an
    // abort (no more MMAs to wait for) the warp waits for that release
    // itself, which the promotion warps always make: they wait on nothing
    // but these barriers.
    //
    // Each slab's scales reach the promotion warps through shared memory, so
    // that those warps keep no global load in flight across their barriers
    // and fences (each of which would wait for it): slot j % SCALE_SLOTS (j
    // counts the CTA's slabs) holds the tile's 128 row scales xs[source row,
    // kb] and its two column-block scales ws[e, nb, kb]; rows past the tile or
    // the operand, routed rows whose index lies outside [0, rows_x), and
    // blocks past n read as 0 (their partial sums are 0).  The slots are
    // filled SCALE_LOOKAHEAD slabs ahead by warp 3, which takes part in no
    // barrier of the slab loop, and handed over through the sfull / sempty
    // mbarriers: this warp releases slab j only once slab j's slot is full
    // (every lane waits, so that the release follows the copies in each
    // lane), and frees slab j - 2's slot once slab j's MMAs have finished
    // (the promotion warps are then done with slab j - 2).  With routed rows
    // warp 3 gathers operand rows instead, and this warp stages the scales
    // itself with cp.async groups: slab j's copies are waited for before its
    // release, and slab j + SCALE_LOOKAHEAD is staged right after it (issued
    // before, they held the release up).
    const uint32_t scale_ring = sbase + (uint32_t)off_scales(kMode, kBN);
    auto slot_addr = [&](int64_t j) {
      return scale_ring + (uint32_t)((j % SCALE_SLOTS) * SCALE_SLOT_FLOATS * 4);
    };
    // routed rows: load cursor (tile, slab, CTA slab count) for the staging
    int64_t lt = blockIdx.x;
    int lkb = 0;
    int64_t lj = 0;
    ScaleSrc src{};
    auto stage_next = [&]() {  // one commit group per call (empty past the end)
      if (lt < num_tiles) {
        stage_scales(p, src, lkb, slot_addr(lj), lane);
        ++lj;
        if (++lkb == nkb) {
          lkb = 0;
          lt += gridDim.x;
          if (lt < num_tiles) src = scale_sources<kMode>(p, decode_tile<kMode, kBN>(p, lt, s_prefix, s_start), lane);
        }
      }
      ptx::cp_async_commit();
    };
    if (kMode == GATHER) {
      if (lt < num_tiles) src = scale_sources<kMode>(p, decode_tile<kMode, kBN>(p, lt, s_prefix, s_start), lane);
#pragma unroll 1
      for (int i = 0; i < SCALE_LOOKAHEAD; ++i) stage_next();
    }
    uint32_t tb = 0, tphase = 0;
    bool ok = true;
    int64_t j = 0;
    for (int64_t t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      for (int kb = 0; kb < nkb; ++kb, ++j) {
        // slab j's scales first: they are normally staged long before its
        // MMAs finish, and the check then stays off the release's path
        if (kMode == GATHER) {
          ptx::cp_async_wait_group<SCALE_LOOKAHEAD - 1>();
        } else if (!*abort_flag) {
          wait_bar(sfull_bar((int)(j % SCALE_SLOTS)), (uint32_t)((j / SCALE_SLOTS) & 1), abort_flag,
                   10);
        }
        if (lane == 0) {
          if (ok) ok = wait_bar(tfull_bar(tb), tphase, abort_flag, 7);
          if (!ok && !ptx::mbar_wait(tempty_bar(tb), tphase ^ 1u, ABORT_DRAIN_LIMIT_NS))
            record_error(8);
        }
        __syncwarp();
        ptx::named_bar_arrive(BAR_SLAB + tb, BAR_SLAB_THREADS);
        if (kMode == GATHER) stage_next();
        else if (lane == 0 && j >= 2) ptx::mbar_arrive(sempty_bar((int)((j - 2) % SCALE_SLOTS)));
        if (++tb == 2) { tb = 0; tphase ^= 1u; }
      }
    }
    if (kMode == GATHER) ptx::cp_async_wait_all();
  } else if (kMode != GATHER && warp == 3) {
    // ------------------------------------------------------ scale staging
    // Fills slab j's slot (above) once slab j - SCALE_SLOTS's slot is free,
    // by 4-byte cp.async whose completion arrives on the slot's sfull.
    // Every lane waits for the slot itself, before its copies overwrite it.
    const uint32_t scale_ring = sbase + (uint32_t)off_scales(kMode, kBN);
    int64_t j = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
      const ScaleSrc src = scale_sources<kMode>(p, decode_tile<kMode, kBN>(p, t, s_prefix, s_start), lane);
      for (int kb = 0; kb < nkb; ++kb, ++j) {
        const int sl = (int)(j % SCALE_SLOTS);
        const bool okl = wait_bar(sempty_bar(sl), (uint32_t)(((j / SCALE_SLOTS) & 1) ^ 1),
                                  abort_flag, 9);
        if (!__all_sync(0xFFFFFFFFu, okl)) { ok = false; break; }
        stage_scales(p, src, kb, scale_ring + (uint32_t)(sl * SCALE_SLOT_FLOATS * 4), lane);
        ptx::cp_async_arrive_noinc(sfull_bar(sl));
      }
    }
    ptx::cp_async_wait_all();
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issue
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, tb = 0, tphase = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_bar(tempty_bar(tb), tphase ^ 1u, abort_flag, 4)) { ok = false; break; }
          if (g_w8a8_gemm_force_timeout) { record_error(5); *abort_flag = 1; ok = false; break; }
          if (!wait_bar(full_bar(stage), phase, abort_flag, 5)) { ok = false; break; }
          // gathered A rows were written by cp.async (generic proxy); the
          // MMA reads them through the async proxy
          if (kMode == GATHER) ptx::fence_proxy_async_smem();
          ptx::tc_fence_after();
          const uint32_t sa = sbase + stage * STAGE_BYTES;
          const uint64_t adesc = ptx::smem_desc_kmajor_sw128(sa);
          const uint64_t bdesc = ptx::smem_desc_kmajor_sw128(sa + A_BYTES);
          const uint32_t dcol = tmem_base + tb * kBN;
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk)  // K = 32 bytes per MMA: +2 in the >>4 field
            ptx::mma_f8f6f4(dcol, adesc + 2u * kk, bdesc + 2u * kk, IDESC, kk > 0 ? 1u : 0u);
          ptx::mma_commit(empty_bar(stage));
          ptx::mma_commit(tfull_bar(tb));
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          if (++tb == 2) { tb = 0; tphase ^= 1u; }
        }
      }
      // all MMAs issued by this thread have finished once done_bar fires
      ptx::mma_commit(done_bar);
      const uint64_t t0 = ptx::globaltimer();
      while (!ptx::mbar_try_wait(done_bar, 0)) {
        if (ptx::globaltimer() - t0 > WAIT_LIMIT_NS) { record_error(6); break; }
      }
    }
  }
  } else {
    // ------------------------------------------------------------ promotion
    ptx::reg_alloc<REGS_EPI>();
    // Thread (quarter, lane) owns tile row quarter*32+lane; warps 4-7 take
    // columns 0-127 of the tile, warps 8-11 columns 128-255 (one weight-scale
    // block each).  Per slab: s = xs[row,kb] * ws[nb,kb] (loads issued two
    // slabs ahead), then the partial comes out of TMEM 16 columns at a time
    // -- the next load in flight while the current one is folded in with
    // packed FMAs -- and the TMEM buffer is handed back as soon as the last
    // load has landed.
    const int ew = warp - EPI_WARP0;
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int half = ew >> 2;      // which half of the tile's columns
    constexpr int COLS = kBN / 2;  // columns per promotion warp
    const int lrow = quarter * 32 + lane;
    uint32_t tb = 0;

    // per-tile state, filled for the next tile before the current one is stored
    Tile T;
    auto setup_tile = [&](int64_t t) { T = decode_tile<kMode, kBN>(p, t, s_prefix, s_start); };
    if ((int64_t)blockIdx.x < num_tiles) setup_tile(blockIdx.x);
    // this thread's row scale and column-block scale in each staged slot
    const float* scales = reinterpret_cast<const float*>(smem + off_scales(kMode, kBN));
    uint32_t js = 0;  // slabs of this CTA so far (slot = js % SCALE_SLOTS)
    constexpr int SC = store_cols(kMode);
    constexpr int CPR = SC / 8;  // 16-byte chunks per staged row
    constexpr int RPI = 32 / CPR;  // rows per warp-wide copy (partial-tile path)
    constexpr int SWZ_SHIFT = CPR == 8 ? 0 : (CPR == 4 ? 1 : 2);  // 128/64/32-byte swizzle
    constexpr uint32_t BUF_BYTES = 32 * SC * 2;
    constexpr int PASSES = COLS / SC;
    constexpr int NBOX = stage_boxes(kMode, kBN);
    constexpr bool WHOLE_TILE = NBOX == PASSES;
    const uint32_t stg0 = sbase + off_stage(kBN) + (uint32_t)ew * NBOX * BUF_BYTES;
    uint32_t nstores = 0;  // TMA stores this warp has issued (over all its tiles)
    for (int64_t t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      const int64_t cur_row0 = T.row0;
      const int cur_rows = T.rows;
      const int c0 = T.n0 + half * COLS;
      float2 acc[COLS / 2];
#pragma unroll
      for (int j = 0; j < COLS / 2; ++j) acc[j] = make_float2(0.0f, 0.0f);
      for (int kb = 0; kb < nkb; ++kb) {
        ptx::named_bar_sync(BAR_SLAB + tb, BAR_SLAB_THREADS);  // slab kb is in TMEM buffer tb
        const float* slot = scales + (js % SCALE_SLOTS) * SCALE_SLOT_FLOATS;
        const float s = slot[lrow] * slot[128 + half * COLS / 128];
        ++js;
        ptx::tc_fence_after();
        const uint32_t tcol = tmem_base + ((uint32_t)(quarter * 32) << 16) + tb * kBN + half * COLS;
        const float2 s2 = make_float2(s, s);
        uint32_t ra[16], rb[16];
        ptx::tmem_ld_32x32b_x16(tcol, ra);
        ptx::tmem_wait_ld_dep(ra);
#pragma unroll
        for (int c = 0; c < COLS / 16; ++c) {
          uint32_t(&cur)[16] = (c & 1) ? rb : ra;
          uint32_t(&nxt)[16] = (c & 1) ? ra : rb;
          if (c + 1 < COLS / 16) ptx::tmem_ld_32x32b_x16(tcol + (c + 1) * 16, nxt);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            acc[c * 8 + j] = __ffma2_rn(
                make_float2(__uint_as_float(cur[2 * j]), __uint_as_float(cur[2 * j + 1])), s2,
                acc[c * 8 + j]);
          if (c + 1 < COLS / 16) ptx::tmem_wait_ld_dep(nxt);
          if (c + 2 == COLS / 16) {
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(tempty_bar(tb));
          }
        }
        tb ^= 1u;
      }
      // BF16 out.  Lane = row writes its chunks of 8 columns into the staging
      // area (chunk ch at position ch ^ swizzle(row): conflict-free, and the
      // layout the TMA store expects).  A warp whose 32 rows all lie in the
      // tile stores the box by TMA; the rows of a partial tile (the last one
      // of a group, or past M) go out by plain row-segment copies instead,
      // so that no row beyond the tile is written.
      const bool full_rows = quarter * 32 + 32 <= cur_rows;
      // the next tile's decode and first scale loads overlap the stores
      // (started inside the last slab instead, they slowed it down)
      if (t + gridDim.x < num_tiles) setup_tile(t + gridDim.x);
      if (WHOLE_TILE) {
        // the previous tile's TMA stores have read this warp's boxes
        if (lane == 0) ptx::bulk_wait_read_0();
        __syncwarp();
      }
#pragma unroll
      for (int pass = 0; pass < PASSES; ++pass) {
        const int col0 = c0 + pass * SC;
        if (col0 >= p.n) break;  // columns past n (warp-uniform)
        const uint32_t stg =
            stg0 + (WHOLE_TILE ? (uint32_t)pass : (nstores & 1u)) * BUF_BYTES;
        if (!WHOLE_TILE) {
          // every store but the newest (from the other box) has read its box
          if (lane == 0) ptx::bulk_wait_read_1();
          __syncwarp();
        }
#pragma unroll
        for (int ch = 0; ch < CPR; ++ch) {
          const int v = pass * CPR + ch;
          const uint32_t pos = (uint32_t)(ch ^ ((lane >> SWZ_SHIFT) & (CPR - 1)));
          ptx::sts128(stg + (uint32_t)(lane * SC * 2) + pos * 16u,
                      ptx::pack_bf16x2(acc[v * 4 + 0].x, acc[v * 4 + 0].y),
                      ptx::pack_bf16x2(acc[v * 4 + 1].x, acc[v * 4 + 1].y),
                      ptx::pack_bf16x2(acc[v * 4 + 2].x, acc[v * 4 + 2].y),
                      ptx::pack_bf16x2(acc[v * 4 + 3].x, acc[v * 4 + 3].y));
        }
        if (full_rows) {
          ptx::fence_proxy_async_smem();  // staging writes -> TMA (async proxy)
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_2d(&tmap_y, stg, col0, (int)(cur_row0 + quarter * 32));
            ptx::bulk_commit();
          }
          ++nstores;
        } else {
          __syncwarp();
#pragma unroll
          for (int it = 0; it < 32 / RPI; ++it) {
            const int r = it * RPI + lane / CPR;
            const int ch = lane % CPR;
            const uint32_t pos = (uint32_t)(ch ^ ((r >> SWZ_SHIFT) & (CPR - 1)));
            const uint4 o = ptx::lds128(stg + (uint32_t)(r * SC * 2) + pos * 16u);
            const int trow = quarter * 32 + r;
            const int col = col0 + ch * 8;
            if (trow < cur_rows && col < p.n)
              *reinterpret_cast<uint4*>(p.y + (cur_row0 + trow) * (int64_t)p.n + col) = o;
          }
          __syncwarp();
        }
      }
    }
    // every TMA store of this warp has completed before the CTA retires
    if (lane == 0) ptx::bulk_wait_all();
  }


  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace gemm

// ---------------------------------------------------------------- host side

// Row-major [rows, cols] bytes, box [box_rows, 128 bytes], 128-byte swizzle.
static bool make_tmap_u8(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                         uint32_t box_rows) {
  return make_tmap_2d(map, base, 1, rows, cols, box_rows, 128, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int kMode, int kBN>
static cudaError_t prepare_kernel(int smem) {
  // Raise the dynamic shared-memory limit once per device and size class.
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || smem > configured[dev]) {
    e = cudaFuncSetAttribute(gemm::fp8_gemm_kernel<kMode, kBN>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = smem;
  }
  return cudaSuccess;
}

// p: every field but num_n_tiles set by the caller.
template <int kBN>
static cudaError_t launch_dense(const CUtensorMap& ta, const CUtensorMap& ty, const uint8_t* wq,
                                gemm::Params p, cudaStream_t st) {
  using namespace gemm;
  CUtensorMap tb;
  if (!make_tmap_u8(&tb, wq, (uint64_t)p.n, (uint64_t)p.k, kBN)) return cudaErrorInvalidValue;
  p.num_n_tiles = (int32_t)((p.n + kBN - 1) / kBN);
  const int64_t tiles = (int64_t)p.num_m_tiles * p.num_n_tiles;
  if (tiles > INT32_MAX) return cudaErrorNotSupported;  // 2^31 tiles of output cannot exist
  const int smem = smem_bytes(DENSE, 1, kBN);
  cudaError_t e = prepare_kernel<DENSE, kBN>(smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)std::min<int64_t>(tiles, sm_count());
  fp8_gemm_kernel<DENSE, kBN><<<grid, THREADS, smem, st>>>(ta, tb, ty, p);
  return cudaGetLastError();
}

cudaError_t launch_block_gemm(const uint8_t* xq, const float* xs, const uint8_t* wq,
                              const float* ws, uint16_t* y, int64_t m, int64_t n, int64_t k,
                              cudaStream_t st) {
  using namespace gemm;
  if (m == 0 || n == 0) return cudaSuccess;
  if (k == 0) return cudaMemsetAsync(y, 0, (size_t)(m * n * 2), st);
  CUtensorMap ta;
  if (!make_tmap_u8(&ta, xq, (uint64_t)m, (uint64_t)k, BM)) return cudaErrorInvalidValue;
  CUtensorMap ty;
  if (!make_tmap_2d(&ty, y, 2, (uint64_t)m, (uint64_t)n, 32, store_cols(DENSE),
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  Params p{};
  p.xq = xq; p.xs = xs; p.ws = ws; p.y = y;
  p.row_idx = nullptr; p.group_offsets = nullptr;
  p.m = m; p.rows_x = m;
  p.n = (int32_t)n; p.k = (int32_t)k;
  p.nkb = (int32_t)((k + 127) / 128);
  p.nnb = (int32_t)((n + 127) / 128);
  p.g = 1;
  p.num_m_tiles = (int32_t)((m + BM - 1) / BM);
  // 128-wide tiles where 256-wide ones would not give every SM a tile: twice
  // the CTAs, and each promotion warp's chain per slab half as long
  const int64_t wide_tiles = (int64_t)p.num_m_tiles * ((n + BN - 1) / BN);
  if (wide_tiles < (int64_t)sm_count()) return launch_dense<BN_NARROW>(ta, ty, wq, p, st);
  return launch_dense<BN>(ta, ty, wq, p, st);
}

cudaError_t launch_grouped_gemm(const uint8_t* xq, const float* xs, int64_t rows_x,
                                const int32_t* row_idx, const int32_t* group_offsets, int32_t g,
                                int64_t total_rows, const uint8_t* wq, const float* ws,
                                uint16_t* y, int64_t n, int64_t k, cudaStream_t st) {
  using namespace gemm;
  if (total_rows == 0 || n == 0 || g == 0) return cudaSuccess;
  if (k == 0) return cudaMemsetAsync(y, 0, (size_t)(total_rows * n * 2), st);
  CUtensorMap ta, tb;
  const bool gather = row_idx != nullptr;
  // The A map is only used for the identity gather (rows of a group are
  // contiguous); with a gather it is still encoded (over xq) but never read.
  if (!make_tmap_u8(&ta, xq, (uint64_t)std::max<int64_t>(rows_x, 1), (uint64_t)k, BM))
    return cudaErrorInvalidValue;
  if (!make_tmap_u8(&tb, wq, (uint64_t)g * (uint64_t)n, (uint64_t)k, BN))
    return cudaErrorInvalidValue;
  CUtensorMap ty;
  if (!make_tmap_2d(&ty, y, 2, (uint64_t)total_rows, (uint64_t)n, 32, store_cols(GROUPED),
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  Params p{};
  p.xq = xq; p.xs = xs; p.ws = ws; p.y = y;
  p.row_idx = row_idx; p.group_offsets = group_offsets;
  p.m = total_rows; p.rows_x = rows_x;
  p.n = (int32_t)n; p.k = (int32_t)k;
  p.nkb = (int32_t)((k + 127) / 128);
  p.nnb = (int32_t)((n + 127) / 128);
  p.g = g;
  p.num_m_tiles = 0;
  p.num_n_tiles = (int32_t)((n + BN - 1) / BN);
  const int64_t max_tiles = ((total_rows + BM - 1) / BM + g) * (int64_t)p.num_n_tiles;
  if (max_tiles > INT32_MAX) return cudaErrorNotSupported;
  const int smem = smem_bytes(gather ? GATHER : GROUPED, g, BN);
  const unsigned grid = (unsigned)std::min<int64_t>(max_tiles, sm_count());
  cudaError_t e;
  if (gather) {
    e = prepare_kernel<GATHER, BN>(smem);
    if (e != cudaSuccess) return e;
    fp8_gemm_kernel<GATHER, BN><<<grid, THREADS, smem, st>>>(ta, tb, ty, p);
  } else {
    e = prepare_kernel<GROUPED, BN>(smem);
    if (e != cudaSuccess) return e;
    fp8_gemm_kernel<GROUPED, BN><<<grid, THREADS, smem, st>>>(ta, tb, ty, p);
  }
  return cudaGetLastError();
}

int grouped_gemm_max_groups() { return gemm::MAX_GROUPS; }

cudaError_t set_gemm_force_timeout(int on) {
  return cudaMemcpyToSymbol(g_w8a8_gemm_force_timeout, &on, sizeof(int));
}

cudaError_t consume_device_error(int* code) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_w8a8_gemm_error, sizeof(int));
  if (e != cudaSuccess) return e;
  if (v != 0) {
    int z = 0;
    e = cudaMemcpyToSymbol(g_w8a8_gemm_error, &z, sizeof(int));
  }
  *code = v;
  return e;
}

}  // namespace w8a8
