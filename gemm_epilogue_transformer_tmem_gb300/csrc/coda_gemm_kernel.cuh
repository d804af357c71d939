// The fused GEMM + on-chip epilogue kernel for sm_103a.
//
// CODA article (d9bl.com, §3.1 and Fig. 1): the GEMM produces the output tile
// and the epilogue f is applied to it before the single global write of D.
// agentlenshq.com ("仕組み"): the GEMM mainloop is fixed, the epilogue is built
// from composable primitives.  zeli.app (augment_me): the RMSNorm row scale is
// gathered as per-row partial sums over the K tiles and applied after the
// projection.
//
// GB300 design: one persistent CTA per SM, or a cluster of two CTAs sharing a
// tcgen05 cta_group::2 MMA on a 256-row tile (each CTA stages half of B);
// warp-specialised:
//   warp 0      TMA producer: A [128 x 64] and B [256 x 64] bf16 tiles into a
//               ring of 128-byte-swizzled shared-memory stages
//   warp 1      MMA issuer: tcgen05.mma (M=128, N=256, K=16) into one of two
//               fp32 accumulators in tensor memory (2 x 256 columns)
//   warp 2      allocates / frees the 512 tensor-memory columns
//   warp 3      (dynamic tile order only) asks cluster launch control for the
//               tile of a cluster that has not started yet
//   warps 4-7   epilogue: tcgen05.ld drains the accumulator one 32-column chunk
//               at a time (thread = row), runs the op list, packs bf16 (RNE)
//               into swizzled staging and TMA-stores it; aux tiles (residual,
//               Z, Xhat) arrive by TMA one chunk ahead.  While they work on
//               tile i, the MMA warp already fills the other accumulator.
//   warps 8-11  (commuted RMSNorm, single CTA) read every A stage from shared
//               memory and accumulate sum_k x^2 for their row, then
//               r = rsqrt(s/K+eps).  A CTA pair takes r from a pre-pass kernel
//               that overlaps the pair's mainloop (programmatic dependent launch).
// On each CTA's last tile warps 0-3 (one per tensor-memory lane quarter) join
// the epilogue once the last accumulator is complete and take its odd chunks.
// Every mbarrier wait is bounded: on expiry the kernel records a timeout in the
// device error word, lets in-flight copies land, frees tensor memory and exits.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "coda_internal.h"
#include "coda_ops.cuh"
#include "coda_ptx.cuh"

namespace coda {

__device__ __forceinline__ void record_error(uint32_t* err, uint32_t role, uint32_t tile) {
  if (atomicCAS(err, 0u, static_cast<uint32_t>(CODA_ERR_TIMEOUT)) == 0u) {
    err[1] = blockIdx.x;
    err[2] = role;
    err[3] = tile;
  }
}

// Longest sleep of one barrier poll: bounds how late a waiter sees the abort
// flag or its time limit.
constexpr uint32_t kWaitSleepNs = 20000;

static __device__ __noinline__ bool wait_slow(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag,
                                       uint64_t timeout_ns, uint32_t* err, uint32_t role, uint32_t tile) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    // sleep on the barrier between checks of the abort flag and the clock
    if (mbar_try_wait_sleep(bar, parity, kWaitSleepNs)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > timeout_ns) {
      record_error(err, role, tile);
      *abort_flag = 1u;
      return false;
    }
  }
}

// bounded wait used only on the abort path; ignores the abort flag
static __device__ __noinline__ bool wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

struct Waiter {
  Ctl* ctl;
  uint64_t timeout;
  uint32_t* err;
  uint32_t role;
  __device__ __forceinline__ bool operator()(uint64_t* bar, uint32_t parity, uint32_t tile) const {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, &ctl->abort_flag, timeout, err, role, tile);
  }
};

// Tile order: groups of `group_m` row blocks; within a group the row block
// varies fastest, then the column block.  The CTAs working at any moment share
// a few row blocks of A and a few column blocks of B, so A is read from DRAM
// once and B once per group, instead of A once per column block.  With
// raster_cols the roles swap: groups of column blocks, the column block
// fastest, so B is read once and A once per group (for a B smaller than A).
__device__ __forceinline__ void tile_coords(int tile, const GemmParams& p, int& m_tile, int& n_tile) {
  const int outer = p.raster_cols ? p.num_n_tiles : p.num_m_tiles;
  const int inner = p.raster_cols ? p.num_m_tiles : p.num_n_tiles;
  const int group_tiles = p.group_m * inner;
  const int g = tile / group_tiles;
  const int first = g * p.group_m;
  const int gsz = min(p.group_m, outer - first);
  const int local = tile - g * group_tiles;
  const int a = first + local % gsz;
  const int b = local / gsz;
  m_tile = p.raster_cols ? b : a;
  n_tile = p.raster_cols ? a : b;
}

// Row scale of the commuted norm for one row, from the pre-pass kernel's r or
// from the caller's row sums of squares of A
__device__ __forceinline__ float row_rms_scale(const GemmParams& p, int row) {
  const float v = p.rms_vec[row];
  return p.rms_from_sumsq ? rsqrtf(fmaf(v, p.inv_K, p.rms_eps)) : v;
}

// Work of one CTA (of one cluster, for CTA pairs).  Normally whole tiles,
// tile0, tile0 + step, ... (tile0: the cluster's index, step: the number of
// clusters).  With the split over K (stream-K), the first p.sk_tiles tiles are
// shared out as (tile, k-block) units: their U = sk_tiles x num_kb units are
// cut into `step` equal runs, and cluster c starts with units
// [c U / step, (c+1) U / step) -- the tail of one tile, maybe whole tiles, and
// the head of another.  The tiles after them follow in whole-tile waves
// (sk_tiles = num_tiles: the whole problem is split, for problems with fewer
// tiles than SMs; otherwise sk_tiles is what the last, partly filled wave and
// the one before it held, so that no cluster idles at the end).  The split
// tiles come first so that a tile's last contributor applies the epilogue --
// adding the other contributor's published partial -- while its MMAs already
// run the next tile.  Every role walks the same sequence.
struct Item {
  int tile, kb0, kb1;
};

struct WorkIter {
  int t, t_end;           // whole tiles: t, t + step, ... below t_end
  int64_t u, u_end;       // stream-K units of this cluster (unit u: tile u / num_kb)
  int step;
  bool split;
  // Dynamic order (cluster launch control, p.clc): the grid has one cluster per
  // tile; a cluster starts with its own tile and takes each later one from the
  // scheduler thread's responses, which every tile-walking role reads in turn
  // from a ring of kSchedSlots and releases on the leader CTA's barrier.
  bool dyn;
  bool started;
  int slot;
  uint32_t ph;
  __device__ __forceinline__ WorkIter(const GemmParams& p, bool split_, int tile0, int tile_step)
      : t(tile0), t_end(p.num_tiles), u(0), u_end(0), step(tile_step), split(split_),
        dyn(!split_ && p.clc != 0), started(false), slot(0), ph(0) {
    if (split) {
      t = p.sk_tiles + tile0;
      const int64_t U = static_cast<int64_t>(p.sk_tiles) * p.num_kb;
      u = U * tile0 / tile_step;
      u_end = U * (tile0 + 1) / tile_step;
    }
  }
  // One thread (or, with warp_call, a whole warp whose lane 0 waits) takes the
  // next item.  `sched_ok` turns false when the wait for a response gave up.
  __device__ __forceinline__ bool next(const GemmParams& p, Item& w, Ctl* ctl, const Waiter& W, uint32_t rank,
                                       int csize, bool warp_call, int lane, bool& sched_ok) {
    if (dyn) {
      int tile = t;
      if (started) {
        if (!warp_call || lane == 0) {
          if (W(&ctl->sched_full[slot], ph, static_cast<uint32_t>(t))) {
            tile = clc_response_ctaid_x(smem_u32(&ctl->sched_resp[slot][0]));
            if (tile >= 0) tile /= csize;
            if (rank == 0)
              mbar_arrive(&ctl->sched_empty[slot]);
            else
              mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->sched_empty[slot]), 0u));
          } else {
            tile = -2;
          }
        }
        if (warp_call) tile = __shfl_sync(0xFFFFFFFFu, tile, 0);
        if (++slot == kSchedSlots) {
          slot = 0;
          ph ^= 1u;
        }
      }
      started = true;
      if (tile == -2) sched_ok = false;
      if (tile < 0) return false;
      t = tile;
      w.tile = tile;
      w.kb0 = 0;
      w.kb1 = p.num_kb;
      return true;
    }
    if (u < u_end) {
      w.tile = static_cast<int>(u / p.num_kb);
      w.kb0 = static_cast<int>(u - static_cast<int64_t>(w.tile) * p.num_kb);
      const int64_t end = static_cast<int64_t>(w.kb0) + (u_end - u);
      w.kb1 = end < p.num_kb ? static_cast<int>(end) : p.num_kb;
      u += w.kb1 - w.kb0;
      return true;
    }
    if (t >= t_end) return false;
    w.tile = t;
    w.kb0 = 0;
    w.kb1 = p.num_kb;
    t += step;
    return true;
  }
};

// Tensor-memory accumulator of a CTA's local-th tile and the parity of its
// barrier phases: two accumulators used in turn, or (MX kernels, whose scales
// take the other half of tensor memory) one accumulator used by every tile.
template <bool kMX>
__device__ __forceinline__ int acc_index(int local) {
  return kMX ? 0 : (local & 1);
}
template <bool kMX>
__device__ __forceinline__ uint32_t acc_parity(int local) {
  return kMX ? static_cast<uint32_t>(local & 1) : static_cast<uint32_t>((local >> 1) & 1);
}

// The CTA whose run holds unit u: the largest c with floor(c U / G) <= u.
__device__ __forceinline__ int unit_owner(int64_t u, int64_t U, int64_t G) {
  return static_cast<int>(((u + 1) * G + U - 1) / U) - 1;
}

// Warp-wide wait of the roles that wait once per tile or chunk (epilogue,
// helpers, row statistics): lane 0 polls the barrier, then the outcome is
// broadcast and __syncwarp orders the other lanes' subsequent reads after
// lane 0's acquire.  (Polls by every lane measured the same there; the
// producer and MMA warps, which wait once per stage, use warp_wait_poll.)
__device__ __forceinline__ bool warp_wait(const Waiter& W, uint64_t* bar, uint32_t parity, uint32_t tile, int lane) {
  int ok = 1;
  if (lane == 0) ok = W(bar, parity, tile) ? 1 : 0;
  ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
  __syncwarp();
  return ok != 0;
}

// Warp-wide wait of the producer and MMA warps, whose loops run on every lane:
// every lane polls the barrier (the try_wait may suspend the warp until the
// phase completes) and a vote keeps the warp converged; past a bounded number
// of polls, lane 0 takes the bounded slow path and broadcasts the outcome.
// (Polling by lane 0 alone, with the other lanes parked at a shuffle, cost the
// CTA-pair workloads 4-9%: the warp reconverges late after each wait.)
__device__ __forceinline__ bool warp_wait_poll(const Waiter& W, uint64_t* bar, uint32_t parity, uint32_t tile,
                                               int lane) {
  for (int i = 0; i < 64; ++i)
    if (__all_sync(0xFFFFFFFFu, mbar_try_wait(bar, parity) ? 1 : 0)) return true;
  return warp_wait(W, bar, parity, tile, lane);
}

// Aux values of one 32-row x 32-column box staged with the 64-byte swizzle:
// 16-byte chunk c of row r sits at r*64 + ((c ^ ((r >> 1) & 3)) * 16).
struct SmemAux {
  const uint8_t* base;   // staging buffer of aux tensor 0 for the current chunk
  int r;                 // row inside the box (the lane)
  __device__ __forceinline__ void load(int k, float (&out)[32]) const {
    const uint8_t* rowp = base + k * (2 * kBoxBytes) + r * 64;
    const int sw = (r >> 1) & 3;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 q = *reinterpret_cast<const uint4*>(rowp + ((c ^ sw) << 4));
      unpack8(q, out + 8 * c);
    }
  }
};

// kAMN: A is given as [K, M] (MN-major operand: the weight gradient X^T dY
// reads the stored activations X [tokens, features] directly).
// kFP8: A and B are FP8 E4M3, both K-major; a stage then holds 128 elements of
// K (the same 128-byte rows), four MMAs of K = 32 (kind::f8f6f4).
// kMX (with kFP8): MX block-scaled E4M3 (kind::mxf8f6f4, one E8M0 scale per 32
// elements of K).  Each stage also brings the scale tiles of its rows (512 bytes
// per 128 rows, tmSA / tmSB); the MMA warp copies them into tensor memory
// (tcgen05.cp) ahead of the stage's four MMAs.  The scales need tensor-memory
// columns, so the MX kernel keeps one accumulator (256 columns) instead of two.
template <bool kGLU, bool kBMN, bool kRowStats, bool kPair, class Epi, bool kAMN, bool kFP8, bool kMX = false>
__global__ void __launch_bounds__((kRowStats || kMX) ? 384 : 256, 1)
    coda_gemm_epilogue_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                              const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmX0,
                              const __grid_constant__ CUtensorMap tmX1, const __grid_constant__ CUtensorMap tmX2,
                              const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                              const __grid_constant__ GemmParams p) {
  static_assert(!kMX || kFP8, "MX operands are 8-bit");
  static_assert(!(kMX && kRowStats), "MX kernels have no row-statistics warps");
  // epilogue warp groups: MX kernels, whose one accumulator holds the next
  // tile's MMAs back until it is drained, run two groups of four warps (warps
  // 4-7 take the even chunks, 8-11 the odd ones); the others one group
  constexpr int kEpiGroups = kMX ? 2 : 1;
  constexpr int kEpiW = kEpiWarps * kEpiGroups;
  // Per-CTA tile geometry.  A CTA pair shares one 256-row tile: rank r of the
  // pair owns rows r*128 .. r*128+127 of it and stages half of B.
  constexpr int kTileM = kPair ? 2 * BM : BM;
  constexpr int kCsize = kPair ? 2 : 1;   // CTAs per cluster
  constexpr int kStageB = kPair ? kPairStageBBytes : kStageBBytes;
  // MX scale tiles per stage and CTA: A's 128 rows, and both 128-row halves of B
  constexpr int kStageSF = kMX ? kMxStageSFBytes : 0;
  // bytes the leader's full barrier expects per stage (both CTAs' loads for a pair)
  constexpr uint32_t kExpectTx = kPair ? 2u * (kPairStageBytes + kStageSF) : static_cast<uint32_t>(kStageBytes + kStageSF);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + p.smem_ctl_off);
  uint8_t* sA = smem;
  uint8_t* sB = smem + p.stages * kStageABytes;
  uint8_t* sSF = sB + p.stages * kStageB;   // MX scale tiles (kMX only)
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const bool leader = rank == 0u;
  // split-K grids run without row-statistics warps (and never with MX operands)
  const bool split = !kRowStats && !kMX && p.split != 0;
  const int tile0 = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int tile_step = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&ctl->full[s], 1);
      // a stage is free once the MMA commit and the four row-statistics warps arrived
      mbar_init(&ctl->empty[s], 1 + (kRowStats ? 4 : 0));
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&ctl->tfull[a], 1);
      mbar_init(&ctl->tempty[a], (kPair ? 256 : 128) * kEpiGroups);
      mbar_init(&ctl->rsfull[a], 128);
      mbar_init(&ctl->rsempty[a], 128);
    }
    for (int q = 0; q < kEpiW; ++q)
      for (int b = 0; b < 2; ++b) mbar_init(&ctl->auxfull[q][b], 1);
    for (int b = 0; b < 2; ++b)
      for (int q = 0; q < kEpiWarps; ++q) mbar_init(&ctl->gfull[b][q], 1);
    mbar_init(&ctl->drain, 1);
    mbar_init(&ctl->esync, kEpiWarps);
    for (int q = 0; q < kEpiWarps; ++q) {
      mbar_init(&ctl->helpdone[q], 1);
      mbar_init(&ctl->haux[q][0], 1);
      mbar_init(&ctl->haux[q][1], 1);
    }
    for (int s = 0; s < kSchedSlots; ++s) {
      mbar_init(&ctl->sched_full[s], 1);
      // tile-walking roles: the producers, the MMA issuer and the epilogue warps
      // of the cluster (the row-statistics variant runs in static order)
      mbar_init(&ctl->sched_empty[s], kPair ? 2 + 1 + 2 * kEpiW : 1 + 1 + kEpiW);
    }
    ctl->abort_flag = 0u;
    fence_mbar_init();
    if (p.num_kb > 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      if (kMX) {
        tma_prefetch_desc(&tmSA);
        tma_prefetch_desc(&tmSB);
      }
    }
    tma_prefetch_desc(&tmD);
  }
  if (warp == 2) {
    if constexpr (kPair) {
      tmem_alloc_pair(&ctl->tmem_base, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&ctl->tmem_base, kTmemCols);
      tmem_relinquish();
    }
  }
  __syncwarp();   // warp 0 diverged around the initialisation above
  tc_fence_before_sync();
  __syncthreads();
  if constexpr (kPair) cluster_sync();   // the peer's barriers are initialised before any remote use
  tc_fence_after_sync();
  const uint32_t tmem_base = ctl->tmem_base;
  // The row-statistics finish launched behind this grid may be scheduled now:
  // it waits (griddepcontrol.wait) for this grid to complete before reading.
  if (threadIdx.x == 0) griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp walks the tiles and stages (warp-uniform coordinates);
    // one elected lane arms the stage's barrier and issues its copies.
    if (p.num_kb > 0) {
      const Waiter W{ctl, p.timeout_ns, p.err, ROLE_PRODUCER};
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_phase = 0;
      bool ok = true;
      WorkIter wi(p, split, tile0, tile_step);
      Item w;
      while (ok && wi.next(p, w, ctl, W, rank, kCsize, true, lane, ok)) {
        const int tile = w.tile;
        int m_tile, n_tile;
        tile_coords(tile, p, m_tile, n_tile);
        const int m0 = m_tile * kTileM + static_cast<int>(rank) * BM;
        // B columns (N index) of this tile held by this CTA: for SwiGLU the G
        // half and the U half of the same output columns
        int nb0, nb1;
        if constexpr (kPair) {
          nb0 = kGLU ? (rank == 0u ? n_tile * (BN / 2) : p.half + n_tile * (BN / 2))
                     : n_tile * BN + static_cast<int>(rank) * (BN / 2);
          nb1 = nb0;
        } else {
          nb0 = kGLU ? n_tile * (BN / 2) : n_tile * BN;
          nb1 = kGLU ? p.half + n_tile * (BN / 2) : nb0 + BN / 2;
        }
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!warp_wait_poll(W, &ctl->empty[stage], phase ^ 1u, tile, lane)) {
            ok = false;
            break;
          }
          uint64_t* fb = &ctl->full[stage];
          if (leader) {
            armed |= 1u << stage;
            armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
          }
          const bool issuer = elect_one();
          if (issuer && leader) mbar_arrive_expect_tx(fb, kExpectTx);
          const int k0 = kb * (kFP8 ? 2 * BK : BK);   // elements of K
          uint8_t* a_dst = sA + stage * kStageABytes;
          uint8_t* b_dst = sB + stage * kStageB;
          if (issuer) {
          if constexpr (kMX) {
            // scale tiles of this k-block: A's 128 rows (this CTA's), B's two
            // 128-row halves of the tile (both in each CTA of a pair)
            uint8_t* sf_dst = sSF + stage * kStageSF;
            const int ca = (m0 / BM) * p.num_kb + kb;
            int b0, b1;
            if constexpr (kPair) {
              b0 = kGLU ? n_tile * (BN / 2) : n_tile * BN;
              b1 = kGLU ? p.half + n_tile * (BN / 2) : b0 + BN / 2;
            } else {
              b0 = nb0;
              b1 = nb1;
            }
            const int cb0 = (b0 / BM) * p.num_kb + kb;
            const int cb1 = (b1 / BM) * p.num_kb + kb;
            if constexpr (kPair) {
              const uint32_t fbc = mapa_shared(smem_u32(fb), 0u);
              tma_load_2d_pair(sf_dst, &tmSA, fbc, 0, ca);
              tma_load_2d_pair(sf_dst + 512, &tmSB, fbc, 0, cb0);
              tma_load_2d_pair(sf_dst + 1024, &tmSB, fbc, 0, cb1);
            } else {
              tma_load_2d(sf_dst, &tmSA, fb, 0, ca);
              tma_load_2d(sf_dst + 512, &tmSB, fb, 0, cb0);
              tma_load_2d(sf_dst + 1024, &tmSB, fb, 0, cb1);
            }
          }
          if constexpr (kPair) {
            const uint32_t fbc = mapa_shared(smem_u32(fb), 0u);   // the leader's barrier
            if (kAMN) {
              tma_load_2d_pair(a_dst, &tmA, fbc, m0, k0);
              tma_load_2d_pair(a_dst + 8192, &tmA, fbc, m0 + 64, k0);
            } else {
              tma_load_2d_pair(a_dst, &tmA, fbc, k0, m0);
            }
            if (kBMN) {
              tma_load_2d_pair(b_dst, &tmB, fbc, nb0, k0);
              tma_load_2d_pair(b_dst + 8192, &tmB, fbc, nb0 + 64, k0);
            } else {
              tma_load_2d_pair(b_dst, &tmB, fbc, k0, nb0);
            }
          } else {
            if (kAMN) {
              tma_load_2d(a_dst, &tmA, fb, m0, k0);
              tma_load_2d(a_dst + 8192, &tmA, fb, m0 + 64, k0);
            } else {
              tma_load_2d(a_dst, &tmA, fb, k0, m0);
            }
            if (kBMN) {
              tma_load_2d(b_dst, &tmB, fb, nb0, k0);
              tma_load_2d(b_dst + 8192, &tmB, fb, nb0 + 64, k0);
              tma_load_2d(b_dst + 16384, &tmB, fb, nb1, k0);
              tma_load_2d(b_dst + 24576, &tmB, fb, nb1 + 64, k0);
            } else {
              tma_load_2d(b_dst, &tmB, fb, k0, nb0);
              tma_load_2d(b_dst + 16384, &tmB, fb, k0, nb1);
            }
          }
          }
          __syncwarp();
          if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && lane == 0) {
        // give copies already issued a bounded time to land before the CTA exits
        for (int s = 0; s < p.stages; ++s)
          if (armed & (1u << s)) wait_drain(&ctl->full[s], (armed_phase >> s) & 1u, 2000000ull);
        if (kPair) {
          const uint64_t t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < 200000ull) {
          }
        }
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // The whole warp walks the tiles and stages, so that stage addresses and
    // operand descriptors are warp-uniform values; one elected lane issues the
    // tensor-memory copies, the MMAs and the commits.
    if (leader) {
      const Waiter W{ctl, p.timeout_ns, p.err, ROLE_MMA};
      constexpr uint32_t idesc = kMX ? make_idesc_mx_e4m3(kTileM, BN)
                                     : (kFP8 ? make_idesc_e4m3(kTileM, BN) : make_idesc_bf16(kTileM, BN, kBMN, kAMN));
      // per UMMA_K step the operand start address advances 32 bytes along a
      // K-major row, or 16 k-rows of 128 bytes (2 KB) in an MN-major tile; in
      // 16-byte units, the descriptor's start-address field
      constexpr uint64_t kStepA = kAMN ? (2048 >> 4) : (32 >> 4);
      constexpr uint64_t kStepB = kBMN ? (2048 >> 4) : (32 >> 4);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      WorkIter wi(p, split, tile0, tile_step);
      Item w;
      for (; ok && wi.next(p, w, ctl, W, rank, kCsize, true, lane, ok); ++local) {
        const int tile = w.tile;
        const int acc = acc_index<kMX>(local);
        const uint32_t acc_phase = acc_parity<kMX>(local);
        if (!warp_wait_poll(W, &ctl->tempty[acc], acc_phase ^ 1u, tile, lane)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * kAccCols;
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!warp_wait_poll(W, &ctl->full[stage], phase, tile, lane)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a_addr = smem_u32(sA + stage * kStageABytes);
          const uint32_t b_addr = smem_u32(sB + stage * kStageB);
          // MN-major operands: 64-element groups 8 KB apart
          const uint64_t ad0 = make_smem_desc(a_addr, kAMN ? 8192 : 16, 1024);
          const uint64_t bd0 = make_smem_desc(b_addr, kBMN ? 8192 : 16, 1024);
          const bool first = kb == w.kb0;
          if constexpr (kMX) {
            // the stage's scale tiles into tensor memory: A's at columns sf+0..3,
            // B's halves at sf+4..7 and sf+8..11 (one 32-bit word per row and
            // 32-row group, its four bytes the stage's four 32-element blocks);
            // the MMAs below are issued after these copies by the same lane.
            // (Issuing the next stage's copies ahead of this stage's MMAs, once
            // its tiles had landed, measured 13% slower: the copies hold up the
            // MMAs queued behind them instead of overlapping them.)
            const uint32_t sf = tmem_base + kMxSFCol0 + stage * kMxSFColsPerStage;
            const uint32_t ss = smem_u32(sSF + stage * kStageSF);
            const uint64_t sd0 = make_smem_desc_rows16(ss);
            const uint64_t sd1 = make_smem_desc_rows16(ss + 512);
            const uint64_t sd2 = make_smem_desc_rows16(ss + 1024);
            if (elect_one()) {
              tmem_cp_32x128b_x4<kPair>(sf, sd0);
              tmem_cp_32x128b_x4<kPair>(sf + 4, sd1);
              tmem_cp_32x128b_x4<kPair>(sf + 8, sd2);
#pragma unroll
              for (int k = 0; k < BK / UMMA_K; ++k) {
                const uint64_t ad = ad0 + k * kStepA;
                const uint64_t bd = bd0 + k * kStepB;
                const uint32_t acc_in = (first && k == 0) ? 0u : 1u;
                const uint32_t id = idesc_sf_ids(idesc, static_cast<uint32_t>(k), static_cast<uint32_t>(k));
                if constexpr (kPair)
                  mma_mxf8_ss_pair(d_tmem, ad, bd, id, sf, sf + 4, acc_in);
                else
                  mma_mxf8_ss(d_tmem, ad, bd, id, sf, sf + 4, acc_in);
              }
              if constexpr (kPair)
                mma_commit_pair_mc(&ctl->empty[stage], 0x3);
              else
                mma_commit(&ctl->empty[stage]);
            }
          } else {
            if (elect_one()) {
#pragma unroll
              for (int k = 0; k < BK / UMMA_K; ++k) {
                const uint64_t ad = ad0 + k * kStepA;
                const uint64_t bd = bd0 + k * kStepB;
                const uint32_t acc_in = (first && k == 0) ? 0u : 1u;
                if constexpr (kFP8) {
                  if constexpr (kPair)
                    mma_f8_ss_pair(d_tmem, ad, bd, idesc, acc_in);
                  else
                    mma_f8_ss(d_tmem, ad, bd, idesc, acc_in);
                } else {
                  if constexpr (kPair)
                    mma_bf16_ss_pair(d_tmem, ad, bd, idesc, acc_in);
                  else
                    mma_bf16_ss(d_tmem, ad, bd, idesc, acc_in);
                }
              }
              if constexpr (kPair)
                mma_commit_pair_mc(&ctl->empty[stage], 0x3);
              else
                mma_commit(&ctl->empty[stage]);
            }
          }
          __syncwarp();
          if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (elect_one()) {
          if constexpr (kPair)
            mma_commit_pair_mc(&ctl->tfull[acc], 0x3);
          else
            mma_commit(&ctl->tfull[acc]);
        }
        __syncwarp();
      }
      // no MMA may still write tensor memory when it is freed (in a pair both
      // CTAs learn it: their helper warps wait for it too)
      if (lane == 0) {
        if constexpr (kPair)
          mma_commit_pair_mc(&ctl->drain, 0x3);
        else
          mma_commit(&ctl->drain);
        wait_drain(&ctl->drain, 0u, 2000000ull);
      }
      __syncwarp();
    }
  } else if (warp == 3) {
    // ------------------------------------------------- tile scheduler (dynamic order)
    // The leader asks for the tile of a cluster that has not started, at most
    // kSchedSlots responses ahead of the slowest role; each CTA arms its own
    // barrier for the response, which lands in every CTA of the cluster.  After
    // the first response that took nothing, no further request is made.
    if (lane == 0 && p.clc != 0 && !split) {
      const Waiter W{ctl, p.timeout_ns, p.err, ROLE_SCHEDULER};
      int slot = 0;
      uint32_t ph = 0;
      for (int i = 0;; ++i) {
        if (leader && i >= kSchedSlots && !W(&ctl->sched_empty[slot], ph ^ 1u, 0u)) break;
        mbar_arrive_expect_tx(&ctl->sched_full[slot], 16u);
        if (leader) {
          fence_proxy_async_smem();   // the roles' reads of the previous response come first
          clc_try_cancel<kPair>(smem_u32(&ctl->sched_resp[slot][0]), smem_u32(&ctl->sched_full[slot]));
        }
        if (!W(&ctl->sched_full[slot], ph, 0u)) {
          // a request may still be in flight: give it a bounded time to land
          // (in a pair the other CTA's copy too, as after the producer's abort)
          wait_drain(&ctl->sched_full[slot], ph, 2000000ull);
          if (kPair) {
            const uint64_t t0 = globaltimer_ns();
            while (globaltimer_ns() - t0 < 200000ull) {
            }
          }
          break;
        }
        if (clc_response_ctaid_x(smem_u32(&ctl->sched_resp[slot][0])) < 0) break;
        if (++slot == kSchedSlots) {
          slot = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp >= 4 && warp < 4 + kEpiW) {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 4;             // epilogue warp index (staging, aux barriers)
    const int q = ew & (kEpiWarps - 1);  // tensor-memory lane quarter
    const int grp = ew / kEpiWarps;      // chunk group: chunks c with c % kEpiGroups == grp
    const Waiter W{ctl, p.timeout_ns, p.err, ROLE_EPILOGUE};
    constexpr int kOutCols = kGLU ? BN / 2 : BN;
    uint8_t* wbase = smem + p.smem_epi_off + ew * p.epi_warp_bytes;
    uint8_t* out_stage = wbase;
    uint8_t* aux_stage = wbase + 2 * kBoxBytes;
    // the tile's slices of the op list's column vectors (cv_smem), fp32 [n_colpf][kOutCols]
    float* cv_stage = reinterpret_cast<float*>(wbase + 2 * kBoxBytes + p.n_aux * 2 * kBoxBytes);
    const int n_aux = p.n_aux;
    const int r_in_tile = q * 32 + lane;
    uint32_t aux_phase = 0;   // bit b: parity of the next completion of buffer b
    uint32_t aux_armed = 0;   // bit b: buffer b has a load that was not waited for
    int abuf = 0;
    int sbuf = 0;
    int local = 0;
    bool ok = true;

    // aux tiles and D are touched once: mark them first to leave L2, so the
    // A and B tiles that other CTAs reuse stay resident
    const uint64_t stream_policy = policy_evict_first();
    auto issue_aux = [&](int b, int col, int row0) {
      __syncwarp();
      if (lane == 0) {
        uint64_t* bar = &ctl->auxfull[ew][b];
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n_aux * kBoxBytes));
        tma_load_2d_hint(aux_stage + (0 * 2 + b) * kBoxBytes, &tmX0, bar, col, row0, stream_policy);
        if (n_aux > 1) tma_load_2d_hint(aux_stage + (1 * 2 + b) * kBoxBytes, &tmX1, bar, col, row0, stream_policy);
        if (n_aux > 2) tma_load_2d_hint(aux_stage + (2 * 2 + b) * kBoxBytes, &tmX2, bar, col, row0, stream_policy);
      }
      aux_armed |= 1u << b;
    };

    bool gd_waited = false;
    uint32_t es_par = 0;      // parity of the next esync phase
    // Meet the other epilogue warps: every warp arrives once per phase and
    // waits (bounded) for the phase, so no warp runs more than a phase ahead
    // and a warp that gave up (timeout, abort) cannot leave the others blocked.
    // Warp 0 of the epilogue may publish a flag to eflag[phase parity] first.
    auto esync = [&](int tile) -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->esync);
      const bool r = warp_wait(W, &ctl->esync, es_par, tile, lane);
      es_par ^= 1u;
      return r;
    };
    WorkIter wi(p, split, tile0, tile_step);
    Item w;
    for (; ok && wi.next(p, w, ctl, W, rank, kCsize, true, lane, ok); ++local) {
      const int tile = w.tile;
      int m_tile, n_tile;
      tile_coords(tile, p, m_tile, n_tile);
      const int m0 = m_tile * kTileM + static_cast<int>(rank) * BM;
      const int row = m0 + r_in_tile;
      const bool row_ok = row < p.M;
      const int col_base = n_tile * kOutCols;
      int nch = (p.N_out - col_base + kChunk - 1) / kChunk;
      if (nch > kOutCols / kChunk) nch = kOutCols / kChunk;
      const int acc = acc_index<kMX>(local);
      const uint32_t acc_phase = acc_parity<kMX>(local);
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kAccCols;
      const bool partial = split && !(w.kb0 == 0 && w.kb1 == p.num_kb);
      if (n_aux > 0 && !partial && grp < nch) issue_aux(abuf, col_base + grp * kChunk, m0 + q * 32);
      // Each chunk reads its 32 entries of every column vector of the op list
      // with warp-uniform loads, which from L2 would each stall the chunk.
      // While the tile's accumulator is computed, copy the tile's slices to
      // this warp's shared memory (fp32, 0 past N_out; lane l takes columns
      // l, l + 32, ...), or, where there is no room, prefetch them into L1
      // (lane l the l-th 128-byte line of a slice; every line it touches holds
      // at least one entry of the slice).
      if (p.cv_smem) {
        __syncwarp();   // every lane is done with the previous tile's slices
        for (int e = 0; e < p.n_colpf; ++e) {
          float x[kOutCols / 32];
          if (p.colpf_shift[e] == 1) {
            const uint16_t* src = static_cast<const uint16_t*>(p.colpf[e]);
#pragma unroll
            for (int i = 0; i < kOutCols / 32; ++i) {
              const int col = col_base + i * 32 + lane;
              x[i] = col < p.N_out ? __uint_as_float(static_cast<uint32_t>(__ldg(src + col)) << 16) : 0.0f;
            }
          } else {
            const float* src = static_cast<const float*>(p.colpf[e]);
#pragma unroll
            for (int i = 0; i < kOutCols / 32; ++i) {
              const int col = col_base + i * 32 + lane;
              x[i] = col < p.N_out ? __ldg(src + col) : 0.0f;
            }
          }
#pragma unroll
          for (int i = 0; i < kOutCols / 32; ++i) cv_stage[e * kOutCols + i * 32 + lane] = x[i];
        }
        __syncwarp();
      } else if (p.n_colpf > 0) {
        const int col_end = min(col_base + kOutCols, p.N_out);
        for (int e = 0; e < p.n_colpf && col_end > col_base; ++e) {
          const int sh = p.colpf_shift[e];
          const uint64_t v = reinterpret_cast<uint64_t>(p.colpf[e]);
          const uint64_t first = v + (static_cast<uint64_t>(col_base) << sh);
          const uint64_t last = v + (static_cast<uint64_t>(col_end) << sh) - 1;
          const uint64_t line = (first & ~uint64_t(127)) + static_cast<uint64_t>(lane) * 128;
          if (line <= last) prefetch_l1(line);
        }
      }

      bool okw = warp_wait(W, &ctl->tfull[acc], acc_phase, tile, lane);
      if (!okw) {
        ok = false;
        break;
      }
      tc_fence_after_sync();

      // Split tiles: the CTA that completes a tile's k-range last applies the
      // epilogue to the sum of every segment's partial accumulator.  No CTA
      // ever waits for another: each publishes its partial (fence, then a
      // counter increment) and only the one that sees the count complete goes
      // on (the fence-and-count reduction of the CUDA programming guide).
      bool src_tmem = true;    // accumulator values come from tensor memory
      int n_seg = 0;           // partial segments to add from the workspace
      int skip_seg = -1;       // ... except this one (the CTA's own, still in tensor memory)
      const float* seg_base = nullptr;
      if (partial) {
        const int64_t U = static_cast<int64_t>(p.sk_tiles) * p.num_kb;
        const int64_t tile_u = static_cast<int64_t>(tile) * p.num_kb;
        const int first = unit_owner(tile_u, U, tile_step);
        const int nseg = unit_owner(tile_u + p.num_kb - 1, U, tile_step) - first + 1;
        const int seg = tile0 - first;
        // Partial slots (one per segment) and the arrival counter of a split
        // tile: per tile where the whole problem is split (few tiles); in the
        // split waves of a large problem per CTA of the tile's first
        // contributor, which is the first contributor of no other split tile
        // (only the last tile that starts inside its run can end beyond it).
        const int owner = p.sk_tiles == p.num_tiles ? tile : first * kCsize + static_cast<int>(rank);
        float* slots = p.ws_part + static_cast<size_t>(owner) * kSplitSegs * kPartFloats;
        uint32_t* cnt = p.ws_cnt + owner;
        const bool leader_thread = q == 0 && lane == 0;
        // every other segment already published: finish from tensor memory
        if (leader_thread) ctl->eflag[es_par] = ld_acquire_gpu(cnt) == static_cast<uint32_t>(nseg - 1) ? 1u : 0u;
        if (!esync(tile)) {
          ok = false;
          break;
        }
        const bool last_now = ctl->eflag[es_par ^ 1u] != 0u;
        if (last_now) {
          __threadfence();
          skip_seg = seg;
        } else {
          // partial layout: float4 (row r, columns 4q..4q+3) at index q * BM + r,
          // so one store instruction of a warp covers 512 contiguous bytes
          float4* mine = reinterpret_cast<float4*>(slots + static_cast<size_t>(seg) * kPartFloats) + r_in_tile;
#pragma unroll 1
          for (int c = 0; c < BN / kChunk; ++c) {
            float v[32];
            tmem_ld32(t_row + c * kChunk, v);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              __stcg(mine + (c * 8 + j) * BM, make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
          }
          tc_fence_before_sync();
          if constexpr (kPair)
            mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->tempty[acc]), 0u));
          else
            mbar_arrive(&ctl->tempty[acc]);
          __threadfence();
          if (!esync(tile)) {     // every partial store is fenced before the count
            ok = false;
            break;
          }
          if (leader_thread) {
            __threadfence();
            ctl->eflag[es_par] = atomicAdd(cnt, 1u) == static_cast<uint32_t>(nseg - 1) ? 1u : 0u;
            __threadfence();
          }
          if (!esync(tile)) {
            ok = false;
            break;
          }
          if (ctl->eflag[es_par ^ 1u] == 0u) continue;
          __threadfence();
          src_tmem = false;
        }
        n_seg = nseg;
        seg_base = slots + static_cast<size_t>(r_in_tile) * 4;
        if (n_aux > 0) issue_aux(abuf, col_base, m0 + q * 32);
      }

      float r_rms = 1.0f, mu = 0.0f;
      if (kRowStats) {
        okw = warp_wait(W, &ctl->rsfull[acc], acc_phase, tile, lane);
        if (!okw) {
          ok = false;
          break;
        }
        r_rms = ctl->rs[acc][r_in_tile];
        mu = ctl->rmu[acc][r_in_tile];
        mbar_arrive(&ctl->rsempty[acc]);
      } else if (p.rms_vec != nullptr) {
        // row statistics from the pre-pass kernel, which may still have been
        // running when this grid started: wait for it before the first read
        if (!gd_waited) {
          griddep_wait();
          gd_waited = true;
        }
        r_rms = row_ok ? row_rms_scale(p, row) : 1.0f;
        if (p.mu_vec != nullptr) mu = row_ok ? p.mu_vec[row] : 0.0f;
      }

      // The CTA's last tile (static order): the helper warp of this lane quarter
      // takes its odd chunks.  Row reductions keep even and odd chunks apart in
      // every tile, so that the sum does not depend on who took which chunk.
      const bool helped = !kRowStats && !kMX && p.helpers != 0 && !split && tile + tile_step >= p.num_tiles;
      float red0[CODA_MAX_REDUCTIONS] = {0.0f, 0.0f, 0.0f, 0.0f};
      float red1[CODA_MAX_REDUCTIONS] = {0.0f, 0.0f, 0.0f, 0.0f};
      uint32_t keep = 0;
      // Aux tiles of chunk c: prefetch the group's next chunk, wait for this one.
      auto aux_step = [&](int c) -> bool {
        if (n_aux == 0) return true;
        const int col = col_base + c * kChunk;
        const int next = helped ? 2 : kEpiGroups;   // the helpers take the odd chunks
        if (c + next < nch) issue_aux(abuf ^ 1, col + next * kChunk, m0 + q * 32);
        if (!warp_wait(W, &ctl->auxfull[ew][abuf], (aux_phase >> abuf) & 1u, tile, lane)) return false;
        aux_phase ^= 1u << abuf;
        aux_armed &= ~(1u << abuf);
        return true;
      };
      // The op list on chunk c's accumulator values, the row reductions kept by
      // chunk parity, and the bf16 store of the chunk.
      auto epi_chunk = [&](int c, float(&v)[32], float(&u)[32]) {
        const int col = col_base + c * kChunk;
        int nvalid = p.N_out - col;
        if (nvalid > kChunk) nvalid = kChunk;
        const RowCtx rc{row, row_ok, col, nvalid, p.half, p.N_out, p.M, r_rms, mu,
                        p.cv_smem ? cv_stage + c * kChunk : nullptr, kOutCols};
        const SmemAux ax{aux_stage + abuf * kBoxBytes, lane};
        if constexpr (kRowStats) {   // never helped: one running sum
          Epi::template run<32, kGLU>(p.prog, v, u, rc, ax, red0, keep);
        } else {
          float cred[CODA_MAX_REDUCTIONS] = {0.0f, 0.0f, 0.0f, 0.0f};
          Epi::template run<32, kGLU>(p.prog, v, u, rc, ax, cred, keep);
          if (c & 1) {
#pragma unroll
            for (int r = 0; r < CODA_MAX_REDUCTIONS; ++r) red1[r] += cred[r];
          } else {
#pragma unroll
            for (int r = 0; r < CODA_MAX_REDUCTIONS; ++r) red0[r] += cred[r];
          }
        }

        // stage bf16 row chunk (64-byte swizzle) and TMA-store the 32x32 box
        uint8_t* ob = out_stage + sbuf * kBoxBytes;
        if (lane == 0) bulk_wait_group_read<1>();
        __syncwarp();
        {
          uint8_t* rowp = ob + lane * 64;
          const int sw = (lane >> 1) & 3;
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)
            *reinterpret_cast<uint4*>(rowp + ((cc ^ sw) << 4)) = pack8(v + 8 * cc);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d_hint(&tmD, ob, col, m0 + q * 32, stream_policy);
          bulk_commit_group();
        }
        sbuf ^= 1;
        if (n_aux > 0) abuf ^= 1;
      };

      if constexpr (kMX) {
        // One accumulator: the next tile's MMAs wait for its release.  Load all
        // of this group's chunks (two of SwiGLU's G/U pairs, or four plain
        // chunks; columns past the matrix edge hold zero products and are not
        // stored) in one round trip, release, then work from registers.
        float pv[4][32];
        if constexpr (kGLU)
          tmem_ld32x4(t_row + grp * kChunk, t_row + BN / 2 + grp * kChunk, t_row + (grp + 2) * kChunk,
                      t_row + BN / 2 + (grp + 2) * kChunk, pv);
        else
          tmem_ld32x4(t_row + grp * kChunk, t_row + (grp + 2) * kChunk, t_row + (grp + 4) * kChunk,
                      t_row + (grp + 6) * kChunk, pv);
        tc_fence_before_sync();
        if constexpr (kPair)
          mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->tempty[acc]), 0u));
        else
          mbar_arrive(&ctl->tempty[acc]);
        constexpr int kPer = kGLU ? 2 : 4;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int c = grp + i * kEpiGroups;
          if (c >= nch) break;
          if (!aux_step(c)) {
            ok = false;
            break;
          }
          if constexpr (kGLU)
            epi_chunk(c, pv[2 * i], pv[2 * i + 1]);
          else
            epi_chunk(c, pv[i], pv[i]);
        }
      } else {
      for (int c = grp; c < nch; c += kEpiGroups) {
        if (helped && (c & 1)) continue;
        if (!aux_step(c)) {
          ok = false;
          break;
        }
        float v[32], u[32];
        if (p.num_kb > 0 && src_tmem) {
          if constexpr (kGLU)
            tmem_ld32x2(t_row + c * kChunk, v, t_row + BN / 2 + c * kChunk, u);
          else
            tmem_ld32(t_row + c * kChunk, v);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            v[j] = 0.0f;
            u[j] = 0.0f;
          }
        }
#pragma unroll 1
        for (int sg = 0; sg < n_seg; ++sg) {
          if (sg == skip_seg) continue;
          const float4* sp = reinterpret_cast<const float4*>(seg_base + static_cast<size_t>(sg) * kPartFloats);
          float4 a[8], b[8];   // all loads of this segment in flight before the adds
#pragma unroll
          for (int j = 0; j < 8; ++j) a[j] = __ldcg(sp + (c * 8 + j) * BM);
          if (kGLU) {
#pragma unroll
            for (int j = 0; j < 8; ++j) b[j] = __ldcg(sp + ((BN / 2) / 4 + c * 8 + j) * BM);
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            v[4 * j] += a[j].x;
            v[4 * j + 1] += a[j].y;
            v[4 * j + 2] += a[j].z;
            v[4 * j + 3] += a[j].w;
            if (kGLU) {
              u[4 * j] += b[j].x;
              u[4 * j + 1] += b[j].y;
              u[4 * j + 2] += b[j].z;
              u[4 * j + 3] += b[j].w;
            }
          }
        }
        if (c + kEpiGroups >= nch && src_tmem) {
          // this group's last chunk of the accumulator is in registers: release
          // it to the MMA warp (the leader's barrier)
          tc_fence_before_sync();
          if constexpr (kPair)
            mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->tempty[acc]), 0u));
          else
            mbar_arrive(&ctl->tempty[acc]);
        }
        epi_chunk(c, v, u);
      }
      }
      if (!ok) break;
      if (kEpiGroups > 1 && !kMX && grp >= nch && src_tmem) {
        // a group with no chunk in this tile releases the accumulator all the same
        tc_fence_before_sync();
        if constexpr (kPair)
          mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->tempty[acc]), 0u));
        else
          mbar_arrive(&ctl->tempty[acc]);
      }
      if (kEpiGroups > 1 && (p.prog.n_red > 0 || p.ws_keep != nullptr)) {
        // the odd-chunk group hands its row partials and keep counts to the
        // even-chunk group of its lane quarter, in the slot of the tile's
        // parity: the group can be at most one tile ahead (the accumulator
        // of the tile after next needs the even group's release, which comes
        // after the even group read this slot)
        const int slot = local & 1;
        if (grp == 1) {
#pragma unroll
          for (int r = 0; r < CODA_MAX_REDUCTIONS; ++r) ctl->g.gred[slot][q][r][lane] = red1[r];
          ctl->g.gkeep[slot][q][lane] = keep;
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl->gfull[slot][q]);
          continue;
        }
        if (!warp_wait(W, &ctl->gfull[slot][q], static_cast<uint32_t>((local >> 1) & 1), tile, lane)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int r = 0; r < CODA_MAX_REDUCTIONS; ++r)
          if (r < p.prog.n_red) red1[r] = ctl->g.gred[slot][q][r][lane];
        keep += ctl->g.gkeep[slot][q][lane];
      } else if (kEpiGroups > 1 && grp == 1) {
        continue;
      }
      if (helped && (p.prog.n_red > 0 || p.ws_keep != nullptr)) {
        if (!warp_wait(W, &ctl->helpdone[q], 0u, tile, lane)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int r = 0; r < CODA_MAX_REDUCTIONS; ++r)
          if (r < p.prog.n_red) red1[r] = ctl->h.hred[q][r][lane];
        keep += ctl->h.hkeep[q][lane];
      }
      if (row_ok) {
        const size_t Ms = static_cast<size_t>(p.M);
#pragma unroll
        for (int r = 0; r < CODA_MAX_REDUCTIONS; ++r)
          if (r < p.prog.n_red)
            p.ws_red[(static_cast<size_t>(r) * p.num_n_tiles + n_tile) * Ms + row] = red0[r] + red1[r];
        if (p.ws_keep != nullptr) p.ws_keep[static_cast<size_t>(n_tile) * Ms + row] = keep;
        if (kRowStats && p.rms_slot >= 0 && n_tile == 0) {
          p.row_stats[static_cast<size_t>(p.rms_slot) * Ms + row] = r_rms;
          if (p.norm_ln) p.row_stats[static_cast<size_t>(p.rms_slot + 1) * Ms + row] = mu;
        }
      }
    }
    // the stores' shared-memory reads must be done before the CTA exits; the
    // grid's completion makes their global writes visible to later work
    if (lane == 0) {
      bulk_wait_group_read<0>();
      if (!ok) {
        for (int b = 0; b < 2; ++b)
          if (aux_armed & (1u << b)) wait_drain(&ctl->auxfull[ew][b], (aux_phase >> b) & 1u, 2000000ull);
      }
    }
    __syncwarp();
  } else if (kRowStats && warp >= 8) {
    // ------------------- row statistics (commuted RMSNorm / LayerNorm)
    // Each A stage is read alongside the MMA as soon as it is in shared memory;
    // one arrival per warp frees the stage.  (CTA pairs get their row scales
    // from a pre-pass kernel instead: there the A halves signal the leader's
    // barrier, not their own CTA's.  So do split-K grids, where a CTA sees only
    // part of a row's K range.)
    const int q = warp - 8;
    const int r = q * 32 + lane;
    const Waiter W{ctl, p.timeout_ns, p.err, ROLE_ROWSTATS};
    int stage = 0;
    uint32_t phase = 0;
    int local = 0;
    bool ok = true;
    for (int tile = tile0; ok && tile < p.num_tiles; tile += tile_step, ++local) {
      // LayerNorm sums are taken about the row's first element (shifted data),
      // so the variance cancels only as far as the row's spread; RMSNorm
      // needs the raw sum of squares (shift 0)
      float s = 0.0f, s1 = 0.0f, shift = 0.0f;
      for (int kb = 0; kb < p.num_kb; ++kb) {
        const bool okw = warp_wait(W, &ctl->full[stage], phase, tile, lane);
        if (!okw) {
          ok = false;
          break;
        }
        // row r of the 128B-swizzled A stage: its eight 16-byte chunks in an
        // order that spreads the warp over all banks (the sum ignores order)
        const uint8_t* arow = sA + stage * kStageABytes + r * 128;
        if (kb == 0 && p.norm_ln)   // logical chunk 0 sits at physical chunk (r & 7)
          shift = __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(arow + ((r & 7) << 4))) << 16);
        // the last k-block may run past K: TMA fills those columns with zeros,
        // which must not enter the shifted sums (x - shift would be -shift)
        const int kvalid = p.K - kb * BK;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 w = *reinterpret_cast<const uint4*>(arow + ((j ^ (r & 7)) << 4));
          float x[8];
          unpack8(w, x);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float d = (8 * j + e < kvalid) ? x[e] - shift : 0.0f;
            s = fmaf(d, d, s);
            s1 += d;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->empty[stage]);
        if (++stage == p.stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      const bool okw = warp_wait(W, &ctl->rsempty[acc], acc_phase ^ 1u, tile, lane);
      if (!okw) break;
      if (p.norm_ln) {
        // LayerNorm: mean = shift + mean(d), variance = mean(d^2) - mean(d)^2
        const float m = s1 * p.inv_K;
        const float var = fmaxf(fmaf(s, p.inv_K, -m * m), 0.0f);
        ctl->rmu[acc][r] = shift + m;
        ctl->rs[acc][r] = rsqrtf(var + p.rms_eps);
      } else {
        ctl->rmu[acc][r] = 0.0f;
        ctl->rs[acc][r] = rsqrtf(fmaf(s, p.inv_K, p.rms_eps));
      }
      mbar_arrive(&ctl->rsfull[acc]);
    }
  }

  if constexpr (!kRowStats) {
    // ------------------------------------------ helpers on the CTA's last tile
    // Once the last accumulator is complete nothing is left to load or issue:
    // the producer, MMA, allocator and scheduler warps (lane quarters 0-3) take
    // the odd chunks of the CTA's last tile, halving the epilogue that nothing
    // overlaps; their aux tiles come by TMA into the idle ring, one chunk ahead.
    // Only in the static order, without a split.
    if (!kMX && p.helpers != 0 && !split && warp < kEpiWarps) {
      __syncwarp();
      const int q = warp;
      const Waiter W{ctl, p.timeout_ns, p.err, ROLE_EPILOGUE};
      const int n_local = tile0 < p.num_tiles ? (p.num_tiles - 1 - tile0) / tile_step + 1 : 0;
      if (n_local > 0 && p.num_kb > 0) {
        constexpr int kOutCols = kGLU ? BN / 2 : BN;
        const int local = n_local - 1;
        const int tile = tile0 + local * tile_step;
        int m_tile, n_tile;
        tile_coords(tile, p, m_tile, n_tile);
        const int m0 = m_tile * kTileM + static_cast<int>(rank) * BM;
        const int row = m0 + q * 32 + lane;
        const bool row_ok = row < p.M;
        const int col_base = n_tile * kOutCols;
        int nch = (p.N_out - col_base + kChunk - 1) / kChunk;
        if (nch > kOutCols / kChunk) nch = kOutCols / kChunk;
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc_index<kMX>(local) * kAccCols;
        // every MMA of the CTA has completed (used once: no phase ambiguity)
        if (warp_wait(W, &ctl->drain, 0u, static_cast<uint32_t>(tile), lane)) {
          tc_fence_after_sync();
          float r_rms = 1.0f, mu = 0.0f;
          if (p.rms_vec != nullptr) {
            griddep_wait();
            r_rms = row_ok ? row_rms_scale(p, row) : 1.0f;
            if (p.mu_vec != nullptr) mu = row_ok ? p.mu_vec[row] : 0.0f;
          }
          const uint64_t stream_policy = policy_evict_first();
          // staging in the ring, whose copies have all landed and been consumed:
          // two output boxes, then two aux buffers of n_aux boxes (aux k of
          // buffer b at (2k + b) boxes, as in the epilogue warps' staging)
          const int n_aux = p.n_aux;
          uint8_t* hstage = smem + q * (2 + 2 * n_aux) * kBoxBytes;
          uint8_t* haux = hstage + 2 * kBoxBytes;
          uint32_t haux_phase = 0, haux_armed = 0;
          int hb = 0;
          auto h_issue = [&](int b, int col) {
            __syncwarp();
            if (lane == 0) {
              uint64_t* bar = &ctl->haux[q][b];
              mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n_aux * kBoxBytes));
              tma_load_2d_hint(haux + (0 * 2 + b) * kBoxBytes, &tmX0, bar, col, m0 + q * 32, stream_policy);
              if (n_aux > 1) tma_load_2d_hint(haux + (1 * 2 + b) * kBoxBytes, &tmX1, bar, col, m0 + q * 32, stream_policy);
              if (n_aux > 2) tma_load_2d_hint(haux + (2 * 2 + b) * kBoxBytes, &tmX2, bar, col, m0 + q * 32, stream_policy);
            }
            haux_armed |= 1u << b;
          };
          bool hok = true;
          if (n_aux > 0 && 1 < nch) h_issue(0, col_base + kChunk);
          float hred[CODA_MAX_REDUCTIONS] = {0.0f, 0.0f, 0.0f, 0.0f};
          uint32_t keep = 0;
          int sbuf = 0;
          for (int c = 1; c < nch; c += 2) {
            const int col = col_base + c * kChunk;
            if (n_aux > 0) {
              if (c + 2 < nch) h_issue(hb ^ 1, col + 2 * kChunk);
              if (!warp_wait(W, &ctl->haux[q][hb], (haux_phase >> hb) & 1u, static_cast<uint32_t>(tile), lane)) {
                hok = false;
                break;
              }
              haux_phase ^= 1u << hb;
              haux_armed &= ~(1u << hb);
            }
            const SmemAux ax{haux + hb * kBoxBytes, lane};
            float v[32], u[32];
            if constexpr (kGLU)
              tmem_ld32x2(t_row + c * kChunk, v, t_row + BN / 2 + c * kChunk, u);
            else
              tmem_ld32(t_row + c * kChunk, v);
            int nvalid = p.N_out - col;
            if (nvalid > kChunk) nvalid = kChunk;
            const RowCtx rc{row, row_ok, col, nvalid, p.half, p.N_out, p.M, r_rms, mu};
            float cred[CODA_MAX_REDUCTIONS] = {0.0f, 0.0f, 0.0f, 0.0f};
            Epi::template run<32, kGLU>(p.prog, v, u, rc, ax, cred, keep);
#pragma unroll
            for (int r = 0; r < CODA_MAX_REDUCTIONS; ++r) hred[r] += cred[r];
            uint8_t* ob = hstage + sbuf * kBoxBytes;
            if (lane == 0) bulk_wait_group_read<1>();
            __syncwarp();
            {
              uint8_t* rowp = ob + lane * 64;
              const int sw = (lane >> 1) & 3;
#pragma unroll
              for (int cc = 0; cc < 4; ++cc)
                *reinterpret_cast<uint4*>(rowp + ((cc ^ sw) << 4)) = pack8(v + 8 * cc);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d_hint(&tmD, ob, col, m0 + q * 32, stream_policy);
              bulk_commit_group();
            }
            sbuf ^= 1;
            if (n_aux > 0) hb ^= 1;
          }
          if (!hok && lane == 0) {
            // aux copies still in flight land before the CTA exits
            for (int b = 0; b < 2; ++b)
              if (haux_armed & (1u << b)) wait_drain(&ctl->haux[q][b], (haux_phase >> b) & 1u, 2000000ull);
          }
          if (hok && (p.prog.n_red > 0 || p.ws_keep != nullptr)) {
#pragma unroll
            for (int r = 0; r < CODA_MAX_REDUCTIONS; ++r) ctl->h.hred[q][r][lane] = hred[r];
            ctl->h.hkeep[q][lane] = keep;
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->helpdone[q]);
          }
          if (lane == 0) bulk_wait_group_read<0>();
          __syncwarp();
        }
      }
    }
  }

  // Lanes 1-31 of the scheduler warp got here while lane 0 was still in its
  // loop: reconverge every warp first, so that the CTA barrier (an aligned
  // barrier, which counts whole warps) waits for every role to finish
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if constexpr (kPair) cluster_sync();   // neither CTA leaves while its peer may still signal it
  if (warp == 2) {
    tc_fence_after_sync();
    if constexpr (kPair)
      tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <bool kGLU, bool kBMN, bool kRowStats, bool kPair, class Epi, bool kAMN = false, bool kFP8 = false,
          bool kMX = false>
cudaError_t launch_gemm_t(const CUtensorMap* maps, const GemmParams& p, int grid, size_t smem, cudaStream_t st) {
  auto kern = &coda_gemm_epilogue_kernel<kGLU, kBMN, kRowStats, kPair, Epi, kAMN, kFP8, kMX>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // Programmatic launch only behind the row-scale pre-pass, whose one output
  // (r) the epilogue reads after griddepcontrol.wait.  Row sums of squares
  // supplied by the caller come with an A that the previous kernel on the stream
  // may have written itself, and the mainloop reads A without such a wait.
  const bool after_prepass = p.rms_vec != nullptr && !p.rms_from_sumsq;
  if constexpr (!kPair) {
    if (!after_prepass) {
      kern<<<grid, (kRowStats || kMX) ? 384 : 256, smem, st>>>(maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6],
                                                       maps[7], p);
      return cudaGetLastError();
    }
    // after the row-scale pre-pass (split-K grids): start the mainloop early,
    // the epilogue waits
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3((kRowStats || kMX) ? 384 : 256, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], maps[7],
                              p);
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3((kRowStats || kMX) ? 384 : 256, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // after a row-scale pre-pass: start the mainloop early, the epilogue waits
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_prepass ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], maps[7],
                              p);
  }
}

// Largest number of CTA pairs of this kernel that can be resident at once.
template <bool kGLU, bool kBMN, bool kRowStats>
cudaError_t max_active_pairs_t(size_t smem, int* pairs) {
  auto kern = &coda_gemm_epilogue_kernel<kGLU, kBMN, kRowStats, true, EpiInterp, false, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kRowStats ? 384 : 256, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(pairs, kern, &cfg);
}

}  // namespace coda

namespace coda {

// Launch the kernel variant for (A layout, B layout, row-statistics warps, CTA
// pair) with epilogue policy Epi.  kRowStatsOK: the policy can be launched with
// row-statistics warps (its op sequence has a commuted norm); kAMNOK: it is
// built for A given as [K, M] too (never with row statistics).
template <class Epi, bool kGLU, bool kRowStatsOK, bool kAMNOK = false>
cudaError_t launch_variant(bool a_mn_major, bool b_mn_major, bool row_stats, bool pair, const CUtensorMap* maps,
                           const GemmParams& p, int grid, size_t smem, cudaStream_t st) {
  if (a_mn_major) {
    if constexpr (kAMNOK) {
      if (row_stats) return cudaErrorNotSupported;
      if (pair)
        return b_mn_major ? launch_gemm_t<kGLU, true, false, true, Epi, true>(maps, p, grid, smem, st)
                          : launch_gemm_t<kGLU, false, false, true, Epi, true>(maps, p, grid, smem, st);
      return b_mn_major ? launch_gemm_t<kGLU, true, false, false, Epi, true>(maps, p, grid, smem, st)
                        : launch_gemm_t<kGLU, false, false, false, Epi, true>(maps, p, grid, smem, st);
    } else {
      return cudaErrorNotSupported;
    }
  }
  if (pair) {
    if (row_stats) return cudaErrorNotSupported;   // pairs take row scales from the pre-pass
    return b_mn_major ? launch_gemm_t<kGLU, true, false, true, Epi>(maps, p, grid, smem, st)
                      : launch_gemm_t<kGLU, false, false, true, Epi>(maps, p, grid, smem, st);
  }
  if (row_stats) {
    if constexpr (kRowStatsOK) {
      return b_mn_major ? launch_gemm_t<kGLU, true, true, false, Epi>(maps, p, grid, smem, st)
                        : launch_gemm_t<kGLU, false, true, false, Epi>(maps, p, grid, smem, st);
    } else {
      return cudaErrorNotSupported;
    }
  }
  return b_mn_major ? launch_gemm_t<kGLU, true, false, false, Epi>(maps, p, grid, smem, st)
                    : launch_gemm_t<kGLU, false, false, false, Epi>(maps, p, grid, smem, st);
}

// FP8 E4M3 operands (A [M, K], B [N, K], both K-major; no row statistics)
template <class Epi, bool kGLU>
cudaError_t launch_variant_fp8(bool pair, const CUtensorMap* maps, const GemmParams& p, int grid, size_t smem,
                               cudaStream_t st) {
  return pair ? launch_gemm_t<kGLU, false, false, true, Epi, false, true>(maps, p, grid, smem, st)
              : launch_gemm_t<kGLU, false, false, false, Epi, false, true>(maps, p, grid, smem, st);
}

// MX block-scaled E4M3 operands (scales in maps[6], maps[7])
template <class Epi, bool kGLU>
cudaError_t launch_variant_mx(bool pair, const CUtensorMap* maps, const GemmParams& p, int grid, size_t smem,
                              cudaStream_t st) {
  return pair ? launch_gemm_t<kGLU, false, false, true, Epi, false, true, true>(maps, p, grid, smem, st)
              : launch_gemm_t<kGLU, false, false, false, Epi, false, true, true>(maps, p, grid, smem, st);
}

}  // namespace coda
