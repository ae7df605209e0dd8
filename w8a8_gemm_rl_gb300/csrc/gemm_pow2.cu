// gemm_pow2.cu -- the blockwise FP8 GEMM for power-of-two scales, on the
// tensor cores' block-scaled MMA, issued for CTA pairs.
//
// The NeMo RL FP8 blog lists power-of-two scaling factors as a recipe
// option; with them every scale is 2^e, which the MMA's UE8M0 block scale
// factors carry exactly ("Unified FP8" notes, FP8 scale choice: E8M0 versus
// FP32).  What is computed is fp8_block_gemm's definition,
//   Y[i,j] = BF16( sum_kb xs[i,kb] * ws[j/128,kb] * P[i,j,kb] ),
// but the scaling happens inside tcgen05.mma.kind::mxf8f6f4.block_scale:
// row i of A and column j of B carry the UE8M0 factors of xs[i,kb] and
// ws[j/128,kb] for each 32-wide K block (the same factor for the four blocks
// of a 128-wide slab), and the tensor cores accumulate the scaled products
// of the whole K extent in FP32 in tensor memory.  Nothing is promoted
// through registers per slab; the accumulator is read once per tile.
//
// CTA pairs: a cluster of two CTAs computes a 256 x 256 tile with
// tcgen05.mma.cta_group::2 issued by the even CTA.  CTA r stages A rows
// 128r..128r+127 of the tile and B rows (output columns) 128r..128r+127, so
// each SM's shared memory takes 32 KB of TMA writes and serves 32 KB of MMA
// reads per 128-wide K slab instead of 48 KB each for a 128 x 256 tile on one
// SM: shared-memory bandwidth, not the tensor cores, bounded the one-SM
// form.  CTA r's tensor memory holds the accumulator of its own 128 rows.
// The odd CTA's copies complete on the even CTA's stage barriers; the MMA
// completions are multicast to both CTAs' barriers.
//
// Scale factors in tensor memory (each CTA its own), each word's byte
// replicated 4 times (one per 32-wide K block): the factor of the CTA's A row
// i is read from column base_a + i / 32, lane i % 32 of lane quarter i / 32
// (so quarter q needs only column q); the factor of the tile's B column j
// from column base_b + j / 32, lane j % 32, which every lane quarter holds.
// A slab's factors take 16 columns (A at 0..3, B at 8..15); the ring holds
// 4 slots of 4 slabs, so the scale warps hand over 4 slabs at a time.
//
// Roles in each CTA (persistent, one CTA per SM, one pair tile at a time):
//   warps 0-3   scale factors: warp q writes the factors of 4 slabs at a
//               time into lane quarter q of a ring of TMEM slots;
//   warps 4-11  epilogue: wait for a tile's accumulator, read the CTA's 128
//               rows (32 rows x 128 columns per warp), hand the accumulator
//               back, round to BF16 and store through swizzled staging by TMA;
//   warp 12     allocates 512 TMEM columns for the pair (accumulator 0..255,
//               scale slots 256..319); in the even CTA lane 0 issues 4
//               block-scaled MMAs per slab and commits;
//   warp 13     producer: TMA of the CTA's A and B halves of each slab into a
//               ring of stages.
// Every mbarrier wait is bounded (2 s); a wait that gives up records an
// error code (51..58) in this kernel's device error word, stops the roles of
// both CTAs of the pair, drains copies and MMAs in flight and frees TMEM.  A
// scale that is not a power of two in [2^-127, 2^127] records code 59 (its
// rows of Y are then wrong; nothing else is affected).
#include <algorithm>

#include "kernels.h"
#include "ptx.cuh"
#include "tmap.h"

namespace w8a8 {

__device__ int g_w8a8_pow2_gemm_error = 0;
// Test hook: while nonzero, the MMA issuer gives up before its first slab as
// if its wait had run out of time (code 55).
__device__ int g_w8a8_pow2_gemm_force_timeout = 0;

namespace p2 {

constexpr int BM = 128;       // A rows per CTA
constexpr int PAIR_M = 256;   // A rows per pair tile
constexpr int BN = 256;       // output columns per tile (B rows, 128 per CTA)
constexpr int BK = 128;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK, B_BYTES = (BN / 2) * BK;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;   // one CTA's half of a slab
// Scale factors live in a ring of SF_SLOTS slots of SF_GROUP slabs each; a
// slab's factors take 16 columns: A's at 0..3, B's at 8..15.
constexpr int SF_GROUP = 4;
constexpr int SF_SLOTS = 4;
constexpr int SF_COL0 = 256;       // first scale-slot column
constexpr int SF_SLAB_COLS = 16;
constexpr int SF_SLOT_COLS = SF_GROUP * SF_SLAB_COLS;
constexpr int SF_B_COL = 8;
static_assert(SF_COL0 + SF_SLOTS * SF_SLOT_COLS <= 512, "tensor memory");
constexpr int TMEM_COLS = 512;
constexpr int SF_WARPS = 4;
constexpr int EPI_WARP0 = 4, NUM_EPI_WARPS = 8;
constexpr int MMA_WARP = EPI_WARP0 + NUM_EPI_WARPS;
constexpr int TMA_WARP = MMA_WARP + 1;
constexpr int THREADS = 32 * (TMA_WARP + 1);
constexpr int RASTER_M = 4;  // pair tiles (256 rows each) per raster group
constexpr uint16_t PAIR_MASK = 0x3;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr int STORE_COLS = 32;  // BF16 columns per TMA store box
constexpr int OFF_BARS = STAGES * STAGE_BYTES;
// full, empty, sf_full, sf_empty, acc_full, acc_empty, done
constexpr int NUM_BARS = 2 * STAGES + 2 * SF_SLOTS + 3;
constexpr int OFF_MISC = OFF_BARS + NUM_BARS * 8;
constexpr int OFF_STAGE = (OFF_MISC + 16 + 1023) / 1024 * 1024;
constexpr int STAGE_BUF_BYTES = 32 * STORE_COLS * 2;  // 32 rows x 32 BF16 columns
constexpr int SMEM = 1024 + OFF_STAGE + NUM_EPI_WARPS * 2 * STAGE_BUF_BYTES;
static_assert(SMEM <= 232448, "shared memory");

// Instruction descriptor of kind::mxf8f6f4 with block scaling: E4M3 A and B
// (format 0), both K-major, N >> 3 in bits 17-22, UE8M0 scale factors (bit
// 23), M >> 4 in bits 24-28, and the byte of each scale word this MMA uses
// (bits 29-30 for A, 4-5 for B); K = 32 per MMA.
__host__ __device__ constexpr uint32_t idesc_block_scaled(int M, int N, int sf_byte) {
  return ((uint32_t)sf_byte << 4) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
         ((uint32_t)(M >> 4) << 24) | ((uint32_t)sf_byte << 29);
}

struct Params {
  const float* xs;
  const float* ws;
  uint16_t* y;
  int64_t m;
  int32_t n, k, nkb, nnb, num_m_tiles, num_n_tiles;  // tiles: 256 x 256 pair tiles
};

__device__ __forceinline__ void record_error(int code) {
  atomicCAS(&g_w8a8_pow2_gemm_error, 0, code);
}

// Stop both CTAs of the pair: this CTA's flag and the peer's.
__device__ __forceinline__ void abort_pair(volatile int* abort_flag, uint32_t peer_flag) {
  *abort_flag = 1;
  ptx::st_cluster_u32(peer_flag, 1u);
}

// Bounded wait on a barrier of this CTA.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         uint32_t peer_flag, int code) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer() - t0 > WAIT_LIMIT_NS) {
      record_error(code);
      abort_pair(abort_flag, peer_flag);
      return false;
    }
  }
}

// UE8M0 byte of a power-of-two scale 2^e, -127 <= e <= 127: the binary32
// exponent field, which is 0 for 2^-127 (a binary32 subnormal); the byte is
// replicated into the four K blocks of a slab.
__device__ __forceinline__ uint32_t ue8m0_x4(float s) {
  return ((__float_as_uint(s) >> 23) & 0xFFu) * 0x01010101u;
}
// A scale the UE8M0 format holds exactly: +2^e with -127 <= e <= 127.
__device__ __forceinline__ bool ue8m0_exact(float s) {
  const uint32_t b = __float_as_uint(s);
  const uint32_t e = b >> 23;  // sign and exponent
  return ((b & 0x007FFFFFu) == 0 && e >= 1 && e <= 254) || b == 0x00400000u;
}

// Pair tile t as seen by CTA `rank`: its 128 A rows start at row0 (rows of
// them inside the matrix, possibly none); the tile's columns start at n0.
// Pair tiles are visited in groups of RASTER_M along M, so the pairs running
// at once share A and B slabs through L2.
struct Tile {
  int64_t row0;
  int32_t rows, n0;
};

__device__ __forceinline__ Tile decode_tile(const Params& p, uint32_t t, uint32_t rank) {
  const uint32_t per_group = (uint32_t)RASTER_M * (uint32_t)p.num_n_tiles;
  const uint32_t grp = t / per_group;
  const int32_t first_m = (int32_t)(grp * RASTER_M);
  const uint32_t gm = (uint32_t)min(RASTER_M, p.num_m_tiles - first_m);
  const uint32_t r = t - grp * per_group;
  Tile T;
  T.row0 = (int64_t)(first_m + (int32_t)(r % gm)) * PAIR_M + (int64_t)rank * BM;
  T.rows = (int32_t)max((int64_t)0, min((int64_t)BM, p.m - T.row0));
  T.n0 = (int32_t)(r / gm) * BN;
  return T;
}

__global__ void __launch_bounds__(THREADS, 1)
    fp8_gemm_pow2_kernel(const __grid_constant__ CUtensorMap tmap_a,
                         const __grid_constant__ CUtensorMap tmap_b,
                         const __grid_constant__ CUtensorMap tmap_y, const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_addr(smem);
  const uint32_t bar0 = sbase + OFF_BARS;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto sf_full_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + s); };
  auto sf_empty_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + SF_SLOTS + s); };
  const uint32_t acc_full = bar0 + 8u * (2 * STAGES + 2 * SF_SLOTS);
  const uint32_t acc_empty = acc_full + 8u;
  const uint32_t done_bar = acc_full + 16u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  // the even CTA's barriers, as cluster addresses (its own for the leader)
  const uint32_t lead_bar0 = ptx::mapa_shared(bar0, 0);
  const uint32_t peer_flag = ptx::mapa_shared(ptx::smem_addr(smem + OFF_MISC + 4), rank ^ 1u);
  const uint32_t pair = blockIdx.x >> 1, num_pairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int s = 0; s < SF_SLOTS; ++s) {
      ptx::mbar_init(sf_full_bar(s), 2 * SF_WARPS);
      ptx::mbar_init(sf_empty_bar(s), 1);
    }
    ptx::mbar_init(acc_full, 1);
    ptx::mbar_init(acc_empty, 2 * NUM_EPI_WARPS);
    ptx::mbar_init(done_bar, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == TMA_WARP && lane == 0) {
    ptx::prefetch_tmap(&tmap_a);
    ptx::prefetch_tmap(&tmap_b);
    ptx::prefetch_tmap(&tmap_y);
  }
  if (warp == MMA_WARP) {
    ptx::tmem_alloc_pair(ptx::smem_addr(tmem_slot), TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  // both CTAs' barriers are initialized before either touches the other's
  ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t num_tiles = (uint32_t)p.num_m_tiles * (uint32_t)p.num_n_tiles;
  const int nkb = p.nkb;

  if (warp < SF_WARPS) {
    // --------------------------------------------------------- scale factors
    // Warp q writes its lane quarter: A column q (the CTA's rows 32q + lane)
    // and all 8 B columns.  The scales of a group of SF_GROUP slabs are
    // loaded into a register ring indexed statically (the inner loops are
    // unrolled), right after the previous group's handover: issued before
    // it, they held up that arrive, which waits for the warp's loads in
    // flight.
    const uint32_t lane_q = (uint32_t)(warp * 32) << 16;  // this warp's lane quarter
    const uint32_t lead_sf_full0 = lead_bar0 + 8u * (2 * STAGES);
    uint32_t slot = 0, sphase = 0;
    bool ok = true;
    for (uint32_t t = pair; t < num_tiles && ok; t += num_pairs) {
      const Tile T = decode_tile(p, t, rank);
      const int nb0 = T.n0 / BN * 2;  // first 128-column weight-scale block
      // a row past m reads row 0's scale (its codes are zero, so any factor
      // gives zero)
      const int64_t row = T.row0 + 32 * warp + lane;
      const float* xsr = p.xs + (row < p.m ? row : 0) * (int64_t)nkb;
      const float* wsr0 = p.ws + (int64_t)min(nb0, p.nnb - 1) * nkb;
      const float* wsr1 = p.ws + (int64_t)min(nb0 + 1, p.nnb - 1) * nkb;
      float ra[SF_GROUP], rw0[SF_GROUP], rw1[SF_GROUP];
#pragma unroll
      for (int u = 0; u < SF_GROUP; ++u) {
        if (u < nkb) {
          ra[u] = xsr[u];
          rw0[u] = wsr0[u];
          rw1[u] = wsr1[u];
        }
      }
      for (int kb0 = 0; kb0 < nkb; kb0 += SF_GROUP) {
        uint32_t okw = 1;
        if (lane == 0)
          okw = wait_bar(sf_empty_bar(slot), sphase ^ 1u, abort_flag, peer_flag, 52) ? 1u : 0u;
        okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
        if (!okw) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t col = tmem_base + lane_q + SF_COL0 + slot * SF_SLOT_COLS;
#pragma unroll
        for (int u = 0; u < SF_GROUP; ++u) {
          const int kb = kb0 + u;
          if (kb < nkb) {
            if (!(ue8m0_exact(ra[u]) && ue8m0_exact(rw0[u]) && ue8m0_exact(rw1[u])))
              record_error(59);
            // B columns 0..127 of the tile take weight block nb0, 128..255
            // block nb0 + 1
            const uint32_t b0 = ue8m0_x4(rw0[u]), b1 = ue8m0_x4(rw1[u]);
            const uint32_t cu = col + (uint32_t)(u * SF_SLAB_COLS);
            asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(cu + (uint32_t)warp),
                         "r"(ue8m0_x4(ra[u]))
                         : "memory");
            asm volatile(
                "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
                    cu + SF_B_COL),
                "r"(b0), "r"(b0), "r"(b0), "r"(b0), "r"(b1), "r"(b1), "r"(b1), "r"(b1)
                : "memory");
          }
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_cluster(lead_sf_full0 + 8u * slot);
        if (++slot == SF_SLOTS) { slot = 0; sphase ^= 1u; }
        // the next group's scales
#pragma unroll
        for (int u = 0; u < SF_GROUP; ++u) {
          const int kb = kb0 + SF_GROUP + u;
          if (kb < nkb) {
            ra[u] = xsr[kb];
            rw0[u] = wsr0[kb];
            rw1[u] = wsr1[kb];
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == TMA_WARP) {
    // -------------------------------------------------------------- producer
    // this CTA's halves of each slab; the bytes complete on the even CTA's
    // stage barrier, which expects both halves
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (uint32_t t = pair; t < num_tiles && ok; t += num_pairs) {
        const Tile T = decode_tile(p, t, rank);
        const int brow = T.n0 + (int)rank * (BN / 2);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_bar(empty_bar(stage), phase ^ 1u, abort_flag, peer_flag, 51)) { ok = false; break; }
          const uint32_t sa = sbase + stage * STAGE_BYTES;
          const uint32_t lead_full = lead_bar0 + 8u * stage;
          if (leader) ptx::mbar_arrive_expect_tx(full_bar(stage), 2 * STAGE_BYTES);
          ptx::tma_load_2d_pair(sa, &tmap_a, lead_full, kb * BK, (int)T.row0);
          ptx::tma_load_2d_pair(sa + A_BYTES, &tmap_b, lead_full, kb * BK, brow);
          ++issued;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      // no TMA copy may still be landing when the CTA retires: the even CTA
      // waits for its last stages' barriers (which count both CTAs' bytes);
      // the odd CTA is held by the final cluster barrier until then
      if (leader) {
        const int64_t first = issued > STAGES ? issued - STAGES : 0;
        for (int64_t i = first; i < issued; ++i) {
          const uint64_t t0 = ptx::globaltimer();
          while (!ptx::mbar_try_wait(full_bar((int)(i % STAGES)), (uint32_t)((i / STAGES) & 1))) {
            if (ptx::globaltimer() - t0 > WAIT_LIMIT_NS) { record_error(53); break; }
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------- MMA issue
    if (leader && lane == 0) {
      uint32_t stage = 0, phase = 0, slot = 0, sphase = 0, tphase = 0;
      bool ok = true;
      if (*reinterpret_cast<volatile int*>(&g_w8a8_pow2_gemm_force_timeout) != 0) {
        record_error(55);
        abort_pair(abort_flag, peer_flag);
        ok = false;
      }
      for (uint32_t t = pair; t < num_tiles && ok; t += num_pairs) {
        // both CTAs' epilogues have read the previous tile's accumulator
        if (!wait_bar(acc_empty, tphase ^ 1u, abort_flag, peer_flag, 54)) break;
        for (int kb = 0; kb < nkb; ++kb) {
          const int u = kb % SF_GROUP;  // slab within its scale group
          if (!wait_bar(full_bar(stage), phase, abort_flag, peer_flag, 55)) { ok = false; break; }
          if (u == 0 && !wait_bar(sf_full_bar(slot), sphase, abort_flag, peer_flag, 56)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = sbase + stage * STAGE_BYTES;
          const uint64_t adesc = ptx::smem_desc_kmajor_sw128(sa);
          const uint64_t bdesc = ptx::smem_desc_kmajor_sw128(sa + A_BYTES);
          const uint32_t sfa = tmem_base + SF_COL0 + slot * SF_SLOT_COLS + u * SF_SLAB_COLS;
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk) {
            const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
                "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X "
                "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(tmem_base),
                "l"(adesc + 2u * kk), "l"(bdesc + 2u * kk),
                "r"(idesc_block_scaled(PAIR_M, BN, kk)), "r"(sfa), "r"(sfa + (uint32_t)SF_B_COL),
                "r"(acc)
                : "memory");
          }
          ptx::mma_commit_pair(empty_bar(stage), PAIR_MASK);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          // the group's last slab (or the tile's) frees its scale slot
          if (u == SF_GROUP - 1 || kb == nkb - 1) {
            ptx::mma_commit_pair(sf_empty_bar(slot), PAIR_MASK);
            if (++slot == SF_SLOTS) { slot = 0; sphase ^= 1u; }
          }
        }
        if (!ok) break;
        ptx::mma_commit_pair(acc_full, PAIR_MASK);
        tphase ^= 1u;
      }
      ptx::mma_commit_pair(done_bar, 0x1);
      const uint64_t t0 = ptx::globaltimer();
      while (!ptx::mbar_try_wait(done_bar, 0)) {
        if (ptx::globaltimer() - t0 > WAIT_LIMIT_NS) { record_error(57); break; }
      }
    }
    __syncwarp();
  } else if (warp >= EPI_WARP0) {
    // -------------------------------------------------------------- epilogue
    const int ew = warp - EPI_WARP0;
    const int quarter = warp & 3;
    const int half = ew >> 2;
    const uint32_t stg0 = sbase + OFF_STAGE + (uint32_t)ew * 2 * STAGE_BUF_BYTES;
    const uint32_t lead_acc_empty = lead_bar0 + 8u * (2 * STAGES + 2 * SF_SLOTS + 1);
    uint32_t tphase = 0;
    uint32_t nstores = 0;  // TMA stores this warp has issued (over all its tiles)
    for (uint32_t t = pair; t < num_tiles; t += num_pairs) {
      const Tile T = decode_tile(p, t, rank);
      uint32_t okw = 1;
      if (lane == 0) okw = wait_bar(acc_full, tphase, abort_flag, peer_flag, 58) ? 1u : 0u;
      okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
      if (!okw) break;
      ptx::tc_fence_after();
      // the warp's 32 rows x 128 columns of the accumulator, in two halves of
      // 64 columns, each rounded to packed BF16 pairs at once (64 registers
      // hold the warp's 32 x 128 outputs)
      uint32_t pk[64];
      const uint32_t tcol = tmem_base + ((uint32_t)(quarter * 32) << 16) + half * 128;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t r[64];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t(&rc)[16] = *reinterpret_cast<uint32_t(*)[16]>(&r[16 * c]);
          ptx::tmem_ld_32x32b_x16(tcol + 64 * h + 16 * c, rc);
        }
        // the waits tie the loaded registers, so no use moves above them
        ptx::tmem_wait_ld_dep32(*reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        ptx::tmem_wait_ld_dep32(*reinterpret_cast<uint32_t(*)[32]>(&r[32]));
#pragma unroll
        for (int i = 0; i < 32; ++i)
          pk[32 * h + i] = ptx::pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
      }
      // hand the accumulator back: the pair's next tile may start
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(lead_acc_empty);
      tphase ^= 1u;
      // BF16 out: lane = row, chunks of 8 columns into a 64-byte-swizzled
      // staging buffer (conflict-free, the TMA store's layout); a warp whose
      // 32 rows lie in the matrix stores by TMA, else by row segments
      const bool full_rows = quarter * 32 + 32 <= T.rows;
      const bool any_rows = quarter * 32 < T.rows;
      const int c0 = T.n0 + half * 128;
#pragma unroll
      for (int pass = 0; pass < 128 / STORE_COLS; ++pass) {
        const int col0 = c0 + pass * STORE_COLS;
        if (col0 >= p.n || !any_rows) break;  // nothing of the matrix (warp-uniform)
        // the two buffers alternate per TMA store issued, not per pass: the
        // one written now is never the source of the newest store, and every
        // older store has read its source once all but the newest have
        const uint32_t stg = stg0 + (nstores & 1u) * STAGE_BUF_BYTES;
        if (lane == 0) ptx::bulk_wait_read_1();
        __syncwarp();
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const int v = pass * 4 + ch;
          const uint32_t pos = (uint32_t)(ch ^ ((lane >> 1) & 3));
          ptx::sts128(stg + (uint32_t)(lane * STORE_COLS * 2) + pos * 16u, pk[4 * v + 0],
                      pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
        if (full_rows) {
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_2d(&tmap_y, stg, col0, (int)(T.row0 + quarter * 32));
            ptx::bulk_commit();
          }
          ++nstores;
        } else {
          __syncwarp();
#pragma unroll
          for (int it = 0; it < 8; ++it) {
            const int r = it * 4 + (lane >> 2);
            const int ch = lane & 3;
            const uint32_t pos = (uint32_t)(ch ^ ((r >> 1) & 3));
            const uint4 o = ptx::lds128(stg + (uint32_t)(r * STORE_COLS * 2) + pos * 16u);
            const int trow = quarter * 32 + r;
            const int col = col0 + ch * 8;
            if (trow < T.rows && col < p.n)
              *reinterpret_cast<uint4*>(p.y + (T.row0 + trow) * (int64_t)p.n + col) = o;
          }
          __syncwarp();
        }
      }
    }
    if (lane == 0) ptx::bulk_wait_all();
  }

  // the pair's MMAs have completed (the even CTA's issuer waited for them)
  // and both CTAs' accumulator reads are done before the pair frees TMEM;
  // the barrier also keeps each CTA's shared memory alive while the other
  // may still use it
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();
  if (warp == MMA_WARP) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

}  // namespace p2

cudaError_t launch_block_gemm_pow2(const uint8_t* xq, const float* xs, const uint8_t* wq,
                                   const float* ws, uint16_t* y, int64_t m, int64_t n, int64_t k,
                                   cudaStream_t st) {
  using namespace p2;
  if (m == 0 || n == 0) return cudaSuccess;
  if (k == 0) return cudaMemsetAsync(y, 0, (size_t)(m * n * 2), st);
  CUtensorMap ta, tb, ty;
  if (!make_tmap_2d(&ta, xq, 1, (uint64_t)m, (uint64_t)k, BM, BK, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (!make_tmap_2d(&tb, wq, 1, (uint64_t)n, (uint64_t)k, BN / 2, BK, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (!make_tmap_2d(&ty, y, 2, (uint64_t)m, (uint64_t)n, 32, STORE_COLS, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  Params p{};
  p.xs = xs; p.ws = ws; p.y = y; p.m = m;
  p.n = (int32_t)n; p.k = (int32_t)k;
  p.nkb = (int32_t)((k + BK - 1) / BK);
  p.nnb = (int32_t)((n + 127) / 128);
  p.num_m_tiles = (int32_t)((m + PAIR_M - 1) / PAIR_M);
  p.num_n_tiles = (int32_t)((n + BN - 1) / BN);
  const int64_t tiles = (int64_t)p.num_m_tiles * p.num_n_tiles;
  if (tiles > INT32_MAX) return cudaErrorNotSupported;
  // per device: the shared-memory attribute, and how many pairs fit at once
  static int max_pairs[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int pairs_fit = (dev >= 0 && dev < 64) ? max_pairs[dev] : 0;
  if (pairs_fit == 0) {
    e = cudaFuncSetAttribute(fp8_gemm_pow2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(2 * (unsigned)(sm_count() / 2));
    e = cudaOccupancyMaxActiveClusters(&pairs_fit, fp8_gemm_pow2_kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (pairs_fit <= 0) return cudaErrorNotSupported;
    if (dev >= 0 && dev < 64) max_pairs[dev] = pairs_fit;
  }
  const unsigned pairs = (unsigned)std::min<int64_t>(tiles, pairs_fit);
  cfg.gridDim = dim3(2 * pairs);
  e = cudaLaunchKernelEx(&cfg, fp8_gemm_pow2_kernel, ta, tb, ty, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t set_pow2_gemm_force_timeout(int on) {
  return cudaMemcpyToSymbol(g_w8a8_pow2_gemm_force_timeout, &on, sizeof(int));
}

cudaError_t consume_pow2_gemm_error(int* code) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_w8a8_pow2_gemm_error, sizeof(int));
  if (e != cudaSuccess) return e;
  if (v != 0) {
    int z = 0;
    e = cudaMemcpyToSymbol(g_w8a8_pow2_gemm_error, &z, sizeof(int));
  }
  *code = v;
  return e;
}

}  // namespace w8a8
