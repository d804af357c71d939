// Internal definitions shared by the host API and the kernels of the CODA
// GEMM+epilogue library (not part of the public C ABI).
#pragma once

#include <cstddef>
#include <cstdint>

#include "../../include/coda.h"

namespace coda {

// Tile shape of the fused kernel: one 128-row x 256-column fp32 accumulator per
// tcgen05 MMA chain (M=128, N=256, K=16 instructions), K staged 64 bf16 at a time
// (one 128-byte swizzle atom per row).
constexpr int BM = 128;
constexpr int BN = 256;            // MMA N: columns of B per tile (G|U halves for SwiGLU)
constexpr int BK = 64;
constexpr int UMMA_K = 16;
constexpr int kAccCols = 256;      // TMEM columns per accumulator buffer
constexpr int kTmemCols = 512;     // two accumulator buffers
constexpr int kEpiWarps = 4;        // epilogue warps per group (one per tensor-memory lane quarter)
constexpr int kMaxEpiGroups = 2;    // MX kernels: two groups, even and odd chunks
constexpr int kChunk = 32;         // epilogue columns per TMEM load / TMA store box
constexpr int kStageABytes = BM * BK * 2;          // 16 KB
constexpr int kStageBBytes = BN * BK * 2;          // 32 KB
constexpr int kStageBytes = kStageABytes + kStageBBytes;
// CTA pair (cta_group::2): a 256 x 256 tile; each CTA stages its 128 rows of A
// and half (128 columns) of B
constexpr int kPairStageBBytes = (BN / 2) * BK * 2;  // 16 KB
constexpr int kPairStageBytes = kStageABytes + kPairStageBBytes;
constexpr int kBoxBytes = 32 * kChunk * 2;         // 32 rows x 32 bf16 = 2 KB
constexpr int kMaxStages = 8;
// MX operands: per stage and CTA, the scale tiles of A's 128 rows and of B's two
// 128-row halves (512 bytes each); in tensor memory, after the one 256-column
// accumulator, 16 columns per stage (A's tile at +0..3, B's at +4..7, +8..11)
constexpr int kMxStageSFBytes = 3 * 512;
constexpr int kMxSFCol0 = kAccCols;
constexpr int kMxSFColsPerStage = 16;
static_assert(kMxSFCol0 + kMaxStages * kMxSFColsPerStage <= kTmemCols, "MX scales must fit in tensor memory");
// Split over K (stream-K): a tile's k-blocks may be shared by up to kSplitSegs
// clusters, each CTA publishing a BM x BN fp32 partial accumulator as float4
// vectors, vector (row r, columns 4q..4q+3) at index q * BM + r (a warp's 32
// rows of one vector column are 512 contiguous bytes).  Slots and arrival
// counters are indexed by tile where the whole problem is split, and by the
// CTAs of a split tile's first contributor where only the last waves are: the
// workspace then holds them for kMaxSplitCtas CTAs (a larger grid does not
// split).
constexpr int kSplitSegs = 3;
constexpr int kPartFloats = BN * BM;
constexpr int kMaxSplitCtas = 160;
// column vectors whose slices the epilogue stages (or prefetches) per tile
constexpr int kMaxColPrefetch = 8;
constexpr int kMaxAux = 3;                         // residual, z, xhat
// Dynamic tile order (cluster launch control): responses in flight at once
constexpr int kSchedSlots = 2;

// aux tensor kinds (index into the aux tensor-map array)
enum AuxKind : int { AUX_RESIDUAL = 0, AUX_Z = 1, AUX_XHAT = 2 };

// One compiled epilogue op.  `red` is the reduction register (0..3) for the
// reduction ops; `u` carries the dropout threshold; f1 the dropout scale.
struct DevOp {
  uint32_t code;
  uint32_t slot;
  float f0;
  float f1;
  uint64_t u;
  int32_t red;
  int32_t aux;      // staging index of the aux tensor this op reads, or -1
  int32_t cv;       // its first column-vector slice staged in shared memory, or -1
                    // (GemmParams::cv_smem; an op's slices are consecutive)
};

struct RedInfo {
  int32_t slot[CODA_MAX_REDUCTIONS];
  int32_t is_mean[CODA_MAX_REDUCTIONS];
};

struct EpiProgram {
  int32_t n_ops;
  int32_t glu_pos;         // index of the SWIGLU op, -1 if none
  int32_t n_red;
  int32_t has_dropout;
  uint64_t seed;
  DevOp ops[CODA_MAX_OPS];
  RedInfo red;
  const uint16_t* col_vec[CODA_MAX_COL_VECS];
  const float* row_vec[CODA_MAX_ROW_VECS];
  uint16_t* preact;
  int32_t preact_width;
  int32_t pad;
  const float* ln_colsum;  // LN_ROWSCALE: c (fp32 [width])
  const float* ln_bias;    // LN_ROWSCALE: b (fp32 [width]) or null
  int32_t n_colred;        // column reductions
  int32_t num_rb;          // 32-row blocks, ceil(M / 32)
  int32_t colred_slot[CODA_MAX_COL_REDUCTIONS];
  float* ws_col;           // [n_colred][num_rb][N_out] per-32-row-block column partials
  const float* col_scale_f32;  // COL_SCALE_F32: fp32 [width]
};

struct GemmParams {
  int32_t M, N, K;
  int32_t N_out;           // output width (N/2 with SWIGLU)
  int32_t half;            // N/2 with SWIGLU, else 0
  int32_t num_m_tiles, num_n_tiles, num_tiles, num_kb, stages;
  int32_t group_m;         // row (or, with raster_cols, column) blocks per rasterization group
  int32_t raster_cols;     // 1: groups of column blocks, column block fastest (see tile_coords)
  int32_t n_aux;           // aux tensors staged by TMA
  int32_t rms_slot;        // row-stat slot for r_i, -1 if none
  float rms_eps;
  float inv_K;
  uint64_t timeout_ns;
  float* row_stats;
  float* ws_red;           // [n_red][num_n_tiles][M]
  uint32_t* ws_keep;       // [num_n_tiles][M]
  uint32_t smem_epi_off;   // offset of the epilogue staging region
  uint32_t smem_ctl_off;   // offset of the control block
  uint32_t epi_warp_bytes; // staging bytes per epilogue warp
  uint32_t* err;           // device error word (4 x u32)
  const float* rms_vec;    // commuted-norm row scales r from the pre-pass kernel (or, with
                           // rms_from_sumsq, the caller's row sums of squares of A), or null
  int32_t rms_from_sumsq;  // 1: rms_vec holds sum_k A[i,k]^2; r = rsqrt(s / K + eps)
  const float* mu_vec;     // commuted LayerNorm row means from the pre-pass kernel, or null
  int32_t norm_ln;         // the row statistics are LayerNorm's (mean and centred variance)
  int32_t split;           // 1: clusters take equal runs of (tile, k-block) units (stream-K) ...
  int32_t sk_tiles;        // ... of the first sk_tiles tiles (the rest follow in whole-tile waves)
  float* ws_part;          // split: [slots][kSplitSegs][kPartFloats] partial accumulators (slots:
                           // num_tiles with sk_tiles == num_tiles, else kMaxSplitCtas)
  uint32_t* ws_cnt;        // split: [slots] arrival counters, zero at launch
  int32_t clc;             // 1: one cluster launched per tile; running clusters take
                           // the tiles of clusters not yet started (cluster launch control)
  int32_t helpers;         // 1: warps 0-3 take the odd chunks of each CTA's last tile
  int32_t n_colpf;         // column vectors the op list reads (bias, column scales, LayerNorm's
                           // c and b; the SwiGLU up half of one as an entry of its own) ...
  int32_t colpf_shift[kMaxColPrefetch];     // ... log2 of their element bytes (1: bf16, 2: fp32)
  const void* colpf[kMaxColPrefetch];       // ... and their first elements
  int32_t cv_smem;         // 1: each epilogue warp copies the tile's slices of them to its shared
                           // memory (fp32 [n_colpf][output columns of a tile]) before the tile's
                           // accumulator is ready; 0: they are prefetched into L1 instead
  EpiProgram prog;
};

// Shared-memory control block of the fused kernel (mbarriers, tensor-memory
// base address, abort flag, commuted-RMSNorm row scales for both accumulators).
struct Ctl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t rsfull[2];
  uint64_t rsempty[2];
  uint64_t auxfull[kMaxEpiGroups * kEpiWarps][2];
  uint64_t drain;
  uint64_t esync;          // the four epilogue warps meet here on split tiles (one arrival each)
  uint32_t eflag[2];       // flag broadcast through esync, by phase parity
  uint64_t sched_full[kSchedSlots];    // a cluster-launch-control response landed (16 bytes)
  uint64_t sched_empty[kSchedSlots];   // every tile-walking role read it (leader CTA's barrier)
  alignas(16) uint32_t sched_resp[kSchedSlots][4];
  uint64_t helpdone[kEpiWarps];                           // a helper warp's row partials are in place
  uint64_t haux[kEpiWarps][2];                            // a helper warp's aux tiles landed (two buffers)
  // two epilogue groups (MX kernels): the odd-chunk group's row partials and
  // keep counts of a tile, handed to the even-chunk group, by tile parity
  uint64_t gfull[2][kEpiWarps];
  // tail helpers run in the other kernels only: their partials share the space
  union {
    struct {
      float hred[kEpiWarps][CODA_MAX_REDUCTIONS][32];     // helper row-reduction partials (last tile)
      uint32_t hkeep[kEpiWarps][32];                      // helper dropout keep counts (last tile)
    } h;
    struct {
      float gred[2][kEpiWarps][CODA_MAX_REDUCTIONS][32];
      uint32_t gkeep[2][kEpiWarps][32];
    } g;
  };
  uint32_t tmem_base;
  uint32_t abort_flag;
  float rs[2][BM];
  float rmu[2][BM];        // commuted LayerNorm: row means for both accumulators
};

// device error word layout: [0] code, [1] block, [2] role, [3] tile
enum ErrRole : uint32_t { ROLE_PRODUCER = 1, ROLE_MMA = 2, ROLE_EPILOGUE = 3, ROLE_ROWSTATS = 4, ROLE_SCHEDULER = 5 };

}  // namespace coda
