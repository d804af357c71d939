// Host side of the C ABI declared in include/coda.h: argument and op-list
// validation, compilation of the op list into the kernels' program, TMA tensor
// map encoding, launch on the caller's stream, and the device error word.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "coda_internal.h"
#include "coda_launch.h"
#include "coda_sequences.h"

namespace coda {

// first device-side failure: code, block, role, tile (see coda_check_device_error)
__device__ uint32_t g_coda_err[4];

namespace {

std::atomic<uint64_t> g_launches{0};
std::atomic<uint64_t> g_timeout_ns{1000000000ull};
std::atomic<int> g_max_ctas{0};
std::atomic<int> g_pair_mode{0};   // 0 auto, 1 single CTAs only, 2 CTA pairs whenever K > 0
std::atomic<int> g_split_mode{0};  // 0 auto, 1 never split over K, 2 split whenever eligible
std::atomic<int> g_dynamic_tiles{0};  // 1: cluster-launch-control tile order where it applies
std::atomic<int> g_tail_helpers{1};   // 1: warps 0-3 help with each CTA's last tile where it applies
std::atomic<int> g_fixed_seqs{1};  // 1: use the fixed op sequences, 0: always the interpreter
std::atomic<int> g_raster_mode{0};   // 0 auto, 1 row groups, 2 column groups
std::atomic<int> g_raster_group{0};  // blocks per group (<= 0: the 48 MB group)
thread_local coda_plan g_last_plan{};

constexpr int kMaxDevices = 64;
struct DevInfo {
  bool init;
  int sms;
  int max_smem;
  uint32_t* err;
};
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

coda_status device_info(DevInfo& out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CODA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return CODA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (!d.init) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return CODA_ERR_CUDA;
    // the kernels are compiled for sm_103a only
    if (major != 10 || minor != 3) return CODA_ERR_UNSUPPORTED;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_coda_err) != cudaSuccess) return CODA_ERR_CUDA;
    d.err = static_cast<uint32_t*>(p);
    d.init = true;
  }
  out = d;
  return CODA_OK;
}

coda_status encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode ? CODA_OK : CODA_ERR_CUDA;
}

// No L2 sector promotion: the boxes' rows are 64 or 128 bytes and their neighbours are
// fetched by their own copies soon after; promoting each row to 256 bytes measured
// 2.5% slower on the workload with two aux tensors (dgrad) and no faster elsewhere.
// 2-D row-major tensor [outer, inner] of bf16 (or, u8 = true, of bytes) with box [box_outer, box_inner]
coda_status make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                     uint32_t box_outer, CUtensorMapSwizzle sw, bool u8 = false) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * (u8 ? 1 : 2)};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(m, u8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                              const_cast<void*>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CODA_OK : CODA_ERR_CUDA;
}

// The tiled MX scales of an operand as `chunks` 512-byte tiles (128 words each),
// one tile per box
coda_status make_map_sf(CUtensorMap* m, const void* base, uint64_t chunks) {
  cuuint64_t dims[2] = {128, chunks};
  cuuint64_t strides[1] = {512};
  cuuint32_t box[2] = {128, 1};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CODA_OK : CODA_ERR_CUDA;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// The op list after validation, in the form the kernels read.
struct Compiled {
  EpiProgram prog;
  bool glu = false;
  int n_aux = 0;
  const void* aux_ptr[kMaxAux] = {nullptr, nullptr, nullptr};
  bool has_rms = false;   // RMS_ROWSCALE or LN_ROWSCALE (row statistics of A)
  const float* rms_sumsq = nullptr;   // RMS_SUMSQ_ROWSCALE: the caller's row sums of squares of A
  bool is_ln = false;     // ... and it is LN_ROWSCALE
  int rms_slot = -1;
  float rms_eps = 0.0f;
  bool needs_row_stats = false;
  int max_stat_slot = -1;
  float* col_stats = nullptr;   // column-reduction output (aux.col_stats)
};

coda_status compile_epilogue(const coda_epilogue* epi, const coda_aux* aux, int64_t N, int64_t K, bool fused,
                             Compiled& c) {
  std::memset(&c.prog, 0, sizeof(c.prog));
  c.prog.glu_pos = -1;
  const uint32_t n_ops = epi ? epi->n_ops : 0u;
  if (n_ops > CODA_MAX_OPS) return CODA_ERR_INVALID_ARG;
  if (epi && epi->reserved != 0) return CODA_ERR_INVALID_ARG;
  c.prog.n_ops = static_cast<int32_t>(n_ops);
  c.prog.seed = epi ? epi->seed : 0ull;
  static const coda_aux kNoAux = {};
  const coda_aux& ax = aux ? *aux : kNoAux;

  // pass 1: the SWIGLU position
  for (uint32_t o = 0; o < n_ops; ++o)
    if (epi->ops[o].opcode == CODA_OP_SWIGLU) {
      if (c.prog.glu_pos >= 0) return CODA_ERR_INVALID_ARG;
      c.prog.glu_pos = static_cast<int32_t>(o);
    }
  c.glu = c.prog.glu_pos >= 0;
  if (c.glu && (N % 16) != 0) return CODA_ERR_INVALID_ARG;
  const int64_t n_out = c.glu ? N / 2 : N;

  int aux_index[kMaxAux] = {-1, -1, -1};
  auto use_aux = [&](int kind, const void* ptr) -> int {
    if (aux_index[kind] < 0) {
      aux_index[kind] = c.n_aux;
      c.aux_ptr[c.n_aux] = ptr;
      ++c.n_aux;
    }
    return aux_index[kind];
  };
  bool seen_preact = false;
  for (uint32_t o = 0; o < n_ops; ++o) {
    const coda_op& op = epi->ops[o];
    DevOp& d = c.prog.ops[o];
    d.code = op.opcode;
    d.slot = op.slot;
    d.f0 = op.f0;
    d.f1 = 0.0f;
    d.u = 0;
    d.red = -1;
    d.aux = -1;
    d.cv = -1;
    if (op.f1 != 0.0f || !std::isfinite(op.f0)) return CODA_ERR_INVALID_ARG;
    const bool after_glu = !c.glu || static_cast<int32_t>(o) > c.prog.glu_pos;
    switch (op.opcode) {
      case CODA_OP_SCALE:
      case CODA_OP_GELU_TANH:
      case CODA_OP_GELU_ERF:
      case CODA_OP_SILU:
      case CODA_OP_SWIGLU:
        break;
      case CODA_OP_COL_SCALE:
      case CODA_OP_BIAS:
        if (op.slot >= CODA_MAX_COL_VECS || ax.col_vec[op.slot] == nullptr) return CODA_ERR_INVALID_ARG;
        if (!aligned16(ax.col_vec[op.slot])) return CODA_ERR_ALIGNMENT;
        c.prog.col_vec[op.slot] = static_cast<const uint16_t*>(ax.col_vec[op.slot]);
        break;
      case CODA_OP_COL_SCALE_F32:
        if (ax.col_scale_f32 == nullptr) return CODA_ERR_INVALID_ARG;
        if (!aligned16(ax.col_scale_f32)) return CODA_ERR_ALIGNMENT;
        c.prog.col_scale_f32 = ax.col_scale_f32;
        break;
      case CODA_OP_ROW_SCALE:
        if (op.slot >= CODA_MAX_ROW_VECS || ax.row_vec[op.slot] == nullptr) return CODA_ERR_INVALID_ARG;
        if (!aligned4(ax.row_vec[op.slot])) return CODA_ERR_ALIGNMENT;
        c.prog.row_vec[op.slot] = ax.row_vec[op.slot];
        break;
      case CODA_OP_RMS_ROWSCALE:
        if (!fused) return CODA_ERR_UNSUPPORTED;
        if (c.has_rms || c.rms_sumsq || K <= 0 || op.f0 < 0.0f) return CODA_ERR_INVALID_ARG;
        if (op.slot != CODA_NO_SLOT) {
          if (op.slot >= CODA_MAX_STAT_SLOTS) return CODA_ERR_INVALID_ARG;
          c.rms_slot = static_cast<int>(op.slot);
          c.needs_row_stats = true;
          if (c.rms_slot > c.max_stat_slot) c.max_stat_slot = c.rms_slot;
        }
        c.has_rms = true;
        c.rms_eps = op.f0;
        break;
      case CODA_OP_RMS_SUMSQ_ROWSCALE:
        // r_i from the caller's sums of squares: the kernels then apply the row
        // factor exactly as for RMS_ROWSCALE, without a pass over A
        if (!fused) return CODA_ERR_UNSUPPORTED;
        if (c.has_rms || c.rms_sumsq || K <= 0 || op.f0 < 0.0f) return CODA_ERR_INVALID_ARG;
        if (op.slot >= CODA_MAX_ROW_VECS || ax.row_vec[op.slot] == nullptr) return CODA_ERR_INVALID_ARG;
        if (!aligned4(ax.row_vec[op.slot])) return CODA_ERR_ALIGNMENT;
        c.rms_sumsq = ax.row_vec[op.slot];
        c.rms_eps = op.f0;
        d.code = CODA_OP_RMS_ROWSCALE;
        break;
      case CODA_OP_LN_ROWSCALE:
        if (!fused) return CODA_ERR_UNSUPPORTED;
        if (c.has_rms || c.rms_sumsq || K <= 0 || op.f0 < 0.0f) return CODA_ERR_INVALID_ARG;
        if (ax.ln_colsum == nullptr) return CODA_ERR_INVALID_ARG;
        if (!aligned16(ax.ln_colsum) || (ax.ln_bias != nullptr && !aligned16(ax.ln_bias))) return CODA_ERR_ALIGNMENT;
        if (op.slot != CODA_NO_SLOT) {
          // r_i to row_stats[slot], mu_i to row_stats[slot + 1]
          if (op.slot + 1 >= CODA_MAX_STAT_SLOTS) return CODA_ERR_INVALID_ARG;
          c.rms_slot = static_cast<int>(op.slot);
          c.needs_row_stats = true;
          if (c.rms_slot + 1 > c.max_stat_slot) c.max_stat_slot = c.rms_slot + 1;
        }
        c.has_rms = true;
        c.is_ln = true;
        c.rms_eps = op.f0;
        c.prog.ln_colsum = ax.ln_colsum;
        c.prog.ln_bias = ax.ln_bias;
        break;
      case CODA_OP_GELU_TANH_GRAD:
      case CODA_OP_GELU_ERF_GRAD:
        if (!after_glu || ax.z == nullptr) return CODA_ERR_INVALID_ARG;
        if (!aligned16(ax.z)) return CODA_ERR_ALIGNMENT;
        d.aux = use_aux(AUX_Z, ax.z);
        break;
      case CODA_OP_DROPOUT: {
        if (!after_glu || c.prog.has_dropout) return CODA_ERR_INVALID_ARG;
        if (!(op.f0 >= 0.0f && op.f0 < 1.0f)) return CODA_ERR_INVALID_ARG;
        c.prog.has_dropout = 1;
        const double keep = 1.0 - static_cast<double>(op.f0);
        // T = floor((1-p) * 2^64) in fp64.  Keep-all (p == 0, or T not below
        // 2^64 for a tiny p) is flagged to the kernel by f0 == 0.
        const double t = std::ldexp(keep, 64);
        if (op.f0 == 0.0f || t >= 18446744073709551616.0) {
          d.f0 = 0.0f;
          d.u = ~0ull;
        } else {
          d.u = static_cast<uint64_t>(t);
        }
        d.f1 = static_cast<float>(1.0 / keep);
        break;
      }
      case CODA_OP_RESIDUAL:
        if (!after_glu || ax.residual == nullptr) return CODA_ERR_INVALID_ARG;
        if (!aligned16(ax.residual)) return CODA_ERR_ALIGNMENT;
        d.aux = use_aux(AUX_RESIDUAL, ax.residual);
        break;
      case CODA_OP_STORE_PREACT:
        if (seen_preact || ax.preact_out == nullptr) return CODA_ERR_INVALID_ARG;
        if (!aligned16(ax.preact_out)) return CODA_ERR_ALIGNMENT;
        seen_preact = true;
        c.prog.preact = static_cast<uint16_t*>(ax.preact_out);
        c.prog.preact_width = static_cast<int32_t>(after_glu ? n_out : N);
        break;
      case CODA_OP_ROW_SUM:
      case CODA_OP_ROW_MEAN:
      case CODA_OP_ROW_SUMSQ:
      case CODA_OP_ROW_DOT_AUX:
        if (!after_glu || op.slot >= CODA_MAX_STAT_SLOTS) return CODA_ERR_INVALID_ARG;
        if (c.prog.n_red >= CODA_MAX_REDUCTIONS) return CODA_ERR_INVALID_ARG;
        if (op.opcode == CODA_OP_ROW_DOT_AUX) {
          if (ax.xhat == nullptr) return CODA_ERR_INVALID_ARG;
          if (!aligned16(ax.xhat)) return CODA_ERR_ALIGNMENT;
          d.aux = use_aux(AUX_XHAT, ax.xhat);
        }
        d.red = c.prog.n_red;
        c.prog.red.slot[c.prog.n_red] = static_cast<int32_t>(op.slot);
        c.prog.red.is_mean[c.prog.n_red] = op.opcode == CODA_OP_ROW_MEAN ? 1 : 0;
        ++c.prog.n_red;
        c.needs_row_stats = true;
        if (static_cast<int>(op.slot) > c.max_stat_slot) c.max_stat_slot = static_cast<int>(op.slot);
        break;
      case CODA_OP_COL_SUM:
      case CODA_OP_COL_SUMSQ:
      case CODA_OP_COL_DOT_AUX:
      case CODA_OP_COL_DOT_NORM:
        if (!fused) return CODA_ERR_UNSUPPORTED;
        if (op.opcode == CODA_OP_COL_DOT_NORM) {
          if (ax.row_vec[0] == nullptr) return CODA_ERR_INVALID_ARG;
          if (!aligned4(ax.row_vec[0]) || (ax.row_vec[1] && !aligned4(ax.row_vec[1]))) return CODA_ERR_ALIGNMENT;
          c.prog.row_vec[0] = ax.row_vec[0];
          c.prog.row_vec[1] = ax.row_vec[1];
        }
        if (!after_glu || op.slot >= CODA_MAX_STAT_SLOTS) return CODA_ERR_INVALID_ARG;
        if (c.prog.n_colred >= CODA_MAX_COL_REDUCTIONS || ax.col_stats == nullptr) return CODA_ERR_INVALID_ARG;
        if (!aligned4(ax.col_stats)) return CODA_ERR_ALIGNMENT;
        if (op.opcode == CODA_OP_COL_DOT_AUX || op.opcode == CODA_OP_COL_DOT_NORM) {
          if (ax.xhat == nullptr) return CODA_ERR_INVALID_ARG;
          if (!aligned16(ax.xhat)) return CODA_ERR_ALIGNMENT;
          d.aux = use_aux(AUX_XHAT, ax.xhat);
        }
        d.red = c.prog.n_colred;
        c.prog.colred_slot[c.prog.n_colred] = static_cast<int32_t>(op.slot);
        ++c.prog.n_colred;
        c.col_stats = ax.col_stats;
        break;
      default:
        return CODA_ERR_INVALID_ARG;
    }
  }
  return CODA_OK;
}

struct Geometry {
  int64_t n_out;
  int out_cols;
  int num_m_tiles, num_n_tiles, num_kb;
  int64_t num_tiles;
};

// tile_m: rows per tile (128 for one CTA, 256 for a CTA pair); fp8: 128 elements of K per k-block
Geometry geometry(int64_t M, int64_t N, int64_t K, bool glu, int tile_m = BM, bool fp8 = false) {
  Geometry g{};
  g.n_out = glu ? N / 2 : N;
  g.out_cols = glu ? BN / 2 : BN;
  g.num_m_tiles = static_cast<int>((M + tile_m - 1) / tile_m);
  g.num_n_tiles = static_cast<int>((g.n_out + g.out_cols - 1) / g.out_cols);
  const int bk = fp8 ? 2 * BK : BK;
  g.num_kb = static_cast<int>((K + bk - 1) / bk);
  g.num_tiles = static_cast<int64_t>(g.num_m_tiles) * g.num_n_tiles;
  return g;
}

// Workspace layout: row-reduction partials [n_red][column tiles][M] fp32, then
// keep-count partials [column tiles][M] u32, then the commuted-norm row scales
// [M] fp32 (and means [M] for LayerNorm, written by the pre-pass kernel), then
// column-reduction partials [n_colred][ceil(M/32)][N_out] fp32.
size_t col_partials_offset(int64_t M, const Geometry& g, const Compiled& c) {
  size_t b = static_cast<size_t>(c.prog.n_red) * g.num_n_tiles * static_cast<size_t>(M) * sizeof(float);
  if (c.prog.has_dropout) b += static_cast<size_t>(g.num_n_tiles) * static_cast<size_t>(M) * sizeof(uint32_t);
  if (c.has_rms) b += static_cast<size_t>(M) * sizeof(float) * (c.is_ln ? 2 : 1);   // r [M] (+ mu [M])
  return b;
}

size_t workspace_bytes_for(int64_t M, const Geometry& g, const Compiled& c) {
  size_t b = col_partials_offset(M, g, c);
  b += static_cast<size_t>(c.prog.n_colred) * static_cast<size_t>((M + 31) / 32) * static_cast<size_t>(g.n_out) *
       sizeof(float);
  return b;
}

// CTA pairs once there are two row blocks (mode 0), always (2) or never (1)
bool use_pair(int64_t M, int64_t K) {
  const int mode = g_pair_mode.load();
  return K > 0 && (mode == 2 || (mode == 0 && M > BM));
}

// Whether a problem may split K ranges over CTAs (stream-K), and for how many
// partial slots the workspace holds room.  Two uses: problems with few tiles
// (single CTAs; at most 76 tiles of 128 rows, half of GB300's 152 SMs, and at
// least 16 k-blocks, K >= 1024), whose idle SMs take part of every tile's K
// range (slots per tile); and problems of many tiles (at least
// kSplitWaveTiles), whose last, partly filled wave of tiles is shared out
// evenly instead (slots per CTA, kMaxSplitCtas).  The decision to split also
// checks the device's SM count and the grid; the slots alone size the
// workspace, so it is independent of the device and so is
// coda_workspace_size.  Forced: any problem with two k-blocks or more.
constexpr int64_t kSplitWaveTiles = 128;
int64_t split_slots(const Geometry& g, bool pair) {
  const int mode = g_split_mode.load();
  if (mode == 1 || g.num_kb < 2) return 0;
  const bool few = !pair && (mode == 2 || (g.num_kb >= 16 && g.num_tiles <= 76));
  const bool waves = mode == 2 || g.num_tiles >= kSplitWaveTiles;
  int64_t n = few ? g.num_tiles : 0;
  if (waves && n < kMaxSplitCtas) n = kMaxSplitCtas;
  return n;
}
bool split_eligible(const Geometry& g, bool pair) { return split_slots(g, pair) > 0; }

// Split-K part of the workspace, after the rest rounded up to 256 bytes:
// partial accumulators [tiles][kSplitSegs][BN x BM] fp32, then a u32 arrival
// counter per tile.
// The column vectors the op list reads, for the epilogue's per-tile staging
// (or L1 prefetch): each op's slices consecutive from its `cv` index, in the
// order the ops read them (a vector, then its SwiGLU up half where the op runs
// before SWIGLU; LayerNorm's c before b).  An op list that needs more than
// kMaxColPrefetch slices stages none (its ops read global memory) and
// prefetches the first kMaxColPrefetch.  Returns whether the slices can be staged.
bool plan_colvecs(EpiProgram& prog, int32_t half, GemmParams& p) {
  p.n_colpf = 0;
  bool fits = true;
  auto add = [&](const void* v, int shift) {
    if (p.n_colpf == kMaxColPrefetch) {
      fits = false;
      return;
    }
    p.colpf[p.n_colpf] = v;
    p.colpf_shift[p.n_colpf] = shift;
    ++p.n_colpf;
  };
  for (int o = 0; o < prog.n_ops; ++o) {
    DevOp& op = prog.ops[o];
    op.cv = -1;
    const bool pre = half > 0 && o < prog.glu_pos;
    auto both = [&](const void* v, int shift) {
      add(v, shift);
      if (pre) add(static_cast<const char*>(v) + (static_cast<size_t>(half) << shift), shift);
    };
    switch (op.code) {
      case CODA_OP_BIAS:
      case CODA_OP_COL_SCALE:
        if (op.slot < CODA_MAX_COL_VECS && prog.col_vec[op.slot] != nullptr) {
          op.cv = p.n_colpf;
          both(prog.col_vec[op.slot], 1);
        }
        break;
      case CODA_OP_COL_SCALE_F32:
        if (prog.col_scale_f32 != nullptr) {
          op.cv = p.n_colpf;
          both(prog.col_scale_f32, 2);
        }
        break;
      case CODA_OP_LN_ROWSCALE:
        if (prog.ln_colsum != nullptr) {
          op.cv = p.n_colpf;
          both(prog.ln_colsum, 2);
          if (prog.ln_bias != nullptr) both(prog.ln_bias, 2);
        }
        break;
      default:
        break;
    }
  }
  if (!fits)
    for (int o = 0; o < prog.n_ops; ++o) prog.ops[o].cv = -1;
  return fits && p.n_colpf > 0;
}

// The fixed op sequence whose opcodes are exactly this list's, or SEQ_INTERP.
// RMS_SUMSQ_ROWSCALE runs as RMS_ROWSCALE (only the source of r differs).
int match_sequence(const coda_epilogue* epi, bool glu) {
  if (!g_fixed_seqs.load()) return SEQ_INTERP;
  const uint32_t n = epi ? epi->n_ops : 0u;
  for (const SeqDef& d : kSeqDefs) {
    if (d.glu != glu || static_cast<uint32_t>(d.n) != n) continue;
    bool same = true;
    for (uint32_t o = 0; o < n && same; ++o) {
      uint32_t code = epi->ops[o].opcode;
      if (code == CODA_OP_RMS_SUMSQ_ROWSCALE) code = CODA_OP_RMS_ROWSCALE;
      same = code == d.codes[o];
    }
    if (same) return d.id;
  }
  return SEQ_INTERP;
}

cudaError_t launch_gemm_seq(int seq, bool glu, bool a_mn_major, bool b_mn_major, bool row_stats, bool pair,
                            const CUtensorMap* maps, const GemmParams& p, int grid, size_t smem, cudaStream_t st) {
  switch (seq) {
    case SEQ_RMS:
    case SEQ_LN:
      return launch_gemm_norm(seq, a_mn_major, b_mn_major, row_stats, pair, maps, p, grid, smem, st);
    case SEQ_RMS_SWIGLU:
      return launch_gemm_norm_glu(seq, a_mn_major, b_mn_major, row_stats, pair, maps, p, grid, smem, st);
    case SEQ_NONE:
    case SEQ_RESIDUAL:
    case SEQ_BIAS_GELU_RESIDUAL:
    case SEQ_RESIDUAL_SUMSQ:
      return launch_gemm_fwd(seq, a_mn_major, b_mn_major, row_stats, pair, maps, p, grid, smem, st);
    case SEQ_SWIGLU:
    case SEQ_SWIGLU_DROPOUT:
      return launch_gemm_fwd_glu(seq, a_mn_major, b_mn_major, row_stats, pair, maps, p, grid, smem, st);
    case SEQ_DGRAD:
    case SEQ_WGRAD:
      return launch_gemm_bwd(seq, a_mn_major, b_mn_major, row_stats, pair, maps, p, grid, smem, st);
    case SEQ_BIAS:
    case SEQ_BIAS_GELU:
    case SEQ_BIAS_GELU_ERF:
    case SEQ_BIAS_RESIDUAL:
    case SEQ_GELU:
      return launch_gemm_gpt(seq, a_mn_major, b_mn_major, row_stats, pair, maps, p, grid, smem, st);
    case SEQ_DEQUANT:
    case SEQ_DEQUANT_SWIGLU:
      return cudaErrorNotSupported;   // built for FP8 operands only
    default:
      return launch_gemm_interp(glu, a_mn_major, b_mn_major, row_stats, pair, maps, p, grid, smem, st);
  }
}

// Tile order: groups of row blocks (A's group resident in L2, B streamed once
// per group) or of column blocks (B's group resident, A streamed once per
// group), each group holding about 48 MB of its resident operand.  Automatic:
// the order with fewer modelled DRAM reads (A + B x row groups, or B + A x
// column groups); row groups on a tie.
void raster_plan(const Geometry& g, int tile_m, int64_t K, int elem_bytes, int32_t& group, int32_t& cols) {
  const int64_t kk = K > 0 ? K : 1;
  const int64_t budget = int64_t{48} << 20;
  const int64_t a_blk = static_cast<int64_t>(tile_m) * kk * elem_bytes;
  const int64_t b_blk = static_cast<int64_t>(BN) * kk * elem_bytes;
  auto clamp = [](int64_t v, int64_t hi) { return v < 1 ? int64_t{1} : (v > hi ? hi : v); };
  const int64_t gr = clamp(budget / a_blk, g.num_m_tiles);
  const int64_t gc = clamp(budget / b_blk, g.num_n_tiles);
  const double a_tot = static_cast<double>(g.num_m_tiles) * static_cast<double>(a_blk);
  const double b_tot = static_cast<double>(g.num_n_tiles) * static_cast<double>(b_blk);
  const double tr = a_tot + b_tot * static_cast<double>((g.num_m_tiles + gr - 1) / gr);
  const double tc = b_tot + a_tot * static_cast<double>((g.num_n_tiles + gc - 1) / gc);
  const int mode = g_raster_mode.load();
  const int want = g_raster_group.load();
  bool use_cols = mode == 2 || (mode == 0 && tc < tr);
  int64_t n = use_cols ? gc : gr;
  if (mode != 0 && want > 0) n = clamp(want, use_cols ? g.num_n_tiles : g.num_m_tiles);
  group = static_cast<int32_t>(n);
  cols = use_cols ? 1 : 0;
}

size_t split_base(size_t b) { return (b + 255) & ~size_t(255); }
size_t split_bytes(const Geometry& g, bool pair) {
  const size_t n = static_cast<size_t>(split_slots(g, pair));
  return n * kSplitSegs * kPartFloats * sizeof(float) + n * sizeof(uint32_t);
}

coda_status check_dims(int64_t M, int64_t N, int64_t K) {
  const int64_t lim = (int64_t{1} << 31) - 1;
  if (M < 0 || N < 0 || K < 0 || M > lim || N > lim || K > lim) return CODA_ERR_INVALID_ARG;
  if ((N % 8) != 0 || (K % 8) != 0) return CODA_ERR_INVALID_ARG;
  return CODA_OK;
}

coda_status from_cuda(cudaError_t e) { return e == cudaSuccess ? CODA_OK : CODA_ERR_CUDA; }

}  // namespace
}  // namespace coda

namespace coda {
coda_status workspace_need(int64_t M, int64_t N, int64_t K, const coda_epilogue* epi, bool with_split,
                           size_t* bytes) {
  if (bytes == nullptr) return CODA_ERR_INVALID_ARG;
  *bytes = 0;
  coda_status s = check_dims(M, N, K);
  if (s != CODA_OK) return s;
  // sizes only: validate the op list without its aux tensors being present
  Compiled c;
  coda_aux dummy{};
  static const uint16_t kAligned[8] __attribute__((aligned(16))) = {};
  for (int i = 0; i < CODA_MAX_COL_VECS; ++i) dummy.col_vec[i] = kAligned;
  for (int i = 0; i < CODA_MAX_ROW_VECS; ++i) dummy.row_vec[i] = reinterpret_cast<const float*>(kAligned);
  dummy.residual = dummy.z = dummy.xhat = kAligned;
  dummy.preact_out = const_cast<uint16_t*>(kAligned);
  dummy.ln_colsum = dummy.ln_bias = reinterpret_cast<const float*>(kAligned);
  dummy.col_stats = const_cast<float*>(reinterpret_cast<const float*>(kAligned));
  dummy.col_scale_f32 = reinterpret_cast<const float*>(kAligned);
  s = compile_epilogue(epi, &dummy, N, K, true, c);
  if (s != CODA_OK) return s;
  const bool pair = use_pair(M, K);
  const Geometry g = geometry(M, N, K, c.glu, pair ? 2 * BM : BM);
  const size_t base = workspace_bytes_for(M, g, c);
  *bytes = (with_split && split_eligible(g, pair)) ? split_base(base) + split_bytes(g, pair) : base;
  return CODA_OK;
}
}  // namespace coda

using namespace coda;

extern "C" {


coda_status coda_workspace_size(int64_t M, int64_t N, int64_t K, const coda_epilogue* epi, size_t* bytes) {
  return workspace_need(M, N, K, epi, true, bytes);
}

}  // extern "C"

namespace coda {
namespace {

// The fused call.  sfa / sfb: the tiled MX scales of A and B (MX operands, with
// CODA_AB_E4M3 | CODA_B_NK), or null.
coda_status gemm_impl(const void* A, const void* B, int64_t M, int64_t N, int64_t K, int32_t b_layout,
                      const coda_epilogue* epi, const coda_aux* aux, void* D, float* row_stats,
                      uint32_t* row_keep_count, void* workspace, size_t workspace_bytes, void* stream,
                      const void* sfa, const void* sfb) {
  coda_status s = check_dims(M, N, K);
  if (s != CODA_OK) return s;
  if ((b_layout & ~(CODA_B_NK | CODA_A_KM | CODA_AB_E4M3)) != 0) return CODA_ERR_INVALID_ARG;
  const bool a_mn = (b_layout & CODA_A_KM) != 0;   // A given as [K, M]
  const bool fp8 = (b_layout & CODA_AB_E4M3) != 0;  // A and B are E4M3 bytes
  const bool mx = sfa != nullptr;                   // ... with MX block scales
  b_layout &= CODA_B_NK;
  if (a_mn && (M % 8) != 0) return CODA_ERR_INVALID_ARG;   // 16-byte rows of A [K, M]
  if (fp8 && (a_mn || b_layout != CODA_B_NK || (K % 16) != 0)) return CODA_ERR_INVALID_ARG;
  if (mx && (!fp8 || (K % 32) != 0)) return CODA_ERR_INVALID_ARG;
  Compiled c;
  s = compile_epilogue(epi, aux, N, K, true, c);
  if (s != CODA_OK) return s;
  if ((a_mn || fp8) && c.has_rms) return CODA_ERR_UNSUPPORTED;   // row statistics read bf16 A by rows
  if (mx && c.rms_sumsq) return CODA_ERR_UNSUPPORTED;
  // the U half of an MX SwiGLU weight must start on a 128-row scale tile
  if (mx && c.glu && ((N / 2) % BM) != 0) return CODA_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return CODA_OK;
  if (D == nullptr || (K > 0 && (A == nullptr || B == nullptr))) return CODA_ERR_INVALID_ARG;
  if (!aligned16(D) || (K > 0 && (!aligned16(A) || !aligned16(B)))) return CODA_ERR_ALIGNMENT;
  if (mx && K > 0 && (sfb == nullptr || !aligned16(sfa) || !aligned16(sfb))) return sfb ? CODA_ERR_ALIGNMENT
                                                                                      : CODA_ERR_INVALID_ARG;
  if (c.needs_row_stats && row_stats == nullptr) return CODA_ERR_INVALID_ARG;
  if (row_stats && !aligned4(row_stats)) return CODA_ERR_ALIGNMENT;
  if (row_keep_count && !aligned4(row_keep_count)) return CODA_ERR_ALIGNMENT;
  // CTA pairs (cta_group::2, 256-row tiles) once there are at least two row blocks
  const bool pair = use_pair(M, K);
  const Geometry g = geometry(M, N, K, c.glu, pair ? 2 * BM : BM, fp8);
  if (g.num_tiles > (int64_t{1} << 31) - 1) return CODA_ERR_UNSUPPORTED;
  const size_t ws_need = workspace_bytes_for(M, g, c);
  if (ws_need > 0 && (workspace == nullptr || workspace_bytes < ws_need)) return CODA_ERR_WORKSPACE;
  const bool split_room = !mx && split_eligible(g, pair) && workspace != nullptr &&
                          workspace_bytes >= split_base(ws_need) + split_bytes(g, pair);
  if (workspace && !aligned16(workspace)) return CODA_ERR_ALIGNMENT;

  DevInfo dev;
  s = device_info(dev);
  if (s != CODA_OK) return s;
  s = encoder();
  if (s != CODA_OK) return s;

  CUtensorMap maps[8];   // A, B, D, aux 0-2, MX scales of A and B
  std::memset(maps, 0, sizeof(maps));
  s = make_map(&maps[2], D, static_cast<uint64_t>(g.n_out), static_cast<uint64_t>(M), kChunk, 32,
               CU_TENSOR_MAP_SWIZZLE_64B);
  if (s != CODA_OK) return s;
  if (K > 0) {
    if (fp8)   // E4M3 bytes: 128-byte rows of 128 elements of K
      s = make_map(&maps[0], A, static_cast<uint64_t>(K), static_cast<uint64_t>(M), 2 * BK, BM,
                   CU_TENSOR_MAP_SWIZZLE_128B, true);
    else if (a_mn)   // [K, M]: two 64-wide boxes of M per 128-row tile, 64 rows of K
      s = make_map(&maps[0], A, static_cast<uint64_t>(M), static_cast<uint64_t>(K), 64, BK,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    else
      s = make_map(&maps[0], A, static_cast<uint64_t>(K), static_cast<uint64_t>(M), BK, BM,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    if (s != CODA_OK) return s;
    if (fp8)
      s = make_map(&maps[1], B, static_cast<uint64_t>(K), static_cast<uint64_t>(N), 2 * BK, BN / 2,
                   CU_TENSOR_MAP_SWIZZLE_128B, true);
    else if (b_layout == CODA_B_KN)
      s = make_map(&maps[1], B, static_cast<uint64_t>(N), static_cast<uint64_t>(K), 64, BK,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    else
      s = make_map(&maps[1], B, static_cast<uint64_t>(K), static_cast<uint64_t>(N), BK, BN / 2,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    if (s != CODA_OK) return s;
  } else {
    maps[0] = maps[2];
    maps[1] = maps[2];
  }
  for (int k = 0; k < 3; ++k) {
    if (k < c.n_aux) {
      s = make_map(&maps[3 + k], c.aux_ptr[k], static_cast<uint64_t>(g.n_out), static_cast<uint64_t>(M), kChunk,
                   32, CU_TENSOR_MAP_SWIZZLE_64B);
      if (s != CODA_OK) return s;
    } else {
      maps[3 + k] = maps[2];
    }
  }
  if (mx && K > 0) {
    const uint64_t kbt = static_cast<uint64_t>((K + 127) / 128);
    s = make_map_sf(&maps[6], sfa, static_cast<uint64_t>((M + BM - 1) / BM) * kbt);
    if (s != CODA_OK) return s;
    s = make_map_sf(&maps[7], sfb, static_cast<uint64_t>((N + BM - 1) / BM) * kbt);
    if (s != CODA_OK) return s;
  } else {
    maps[6] = maps[2];
    maps[7] = maps[2];
  }

  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  p.M = static_cast<int32_t>(M);
  p.N = static_cast<int32_t>(N);
  p.K = static_cast<int32_t>(K);
  p.N_out = static_cast<int32_t>(g.n_out);
  p.half = c.glu ? static_cast<int32_t>(N / 2) : 0;
  p.num_m_tiles = g.num_m_tiles;
  raster_plan(g, pair ? 2 * BM : BM, K, fp8 ? 1 : 2, p.group_m, p.raster_cols);
  p.num_n_tiles = g.num_n_tiles;
  p.num_tiles = static_cast<int32_t>(g.num_tiles);
  p.num_kb = g.num_kb;
  p.n_aux = c.n_aux;
  p.rms_slot = c.rms_slot;
  p.norm_ln = c.is_ln ? 1 : 0;
  p.rms_eps = c.rms_eps;
  p.inv_K = K > 0 ? static_cast<float>(1.0 / static_cast<double>(K)) : 0.0f;
  p.timeout_ns = g_timeout_ns.load();
  p.row_stats = row_stats;
  float* rms_ws = nullptr;
  if (ws_need > 0) {
    p.ws_red = static_cast<float*>(workspace);
    uint32_t* keep_ws = reinterpret_cast<uint32_t*>(static_cast<float*>(workspace) +
                                                    static_cast<size_t>(c.prog.n_red) * g.num_n_tiles * M);
    if (c.prog.has_dropout && row_keep_count != nullptr) p.ws_keep = keep_ws;
    rms_ws = reinterpret_cast<float*>(keep_ws + (c.prog.has_dropout ? static_cast<size_t>(g.num_n_tiles) * M : 0));
    if (c.prog.n_colred > 0)
      c.prog.ws_col = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + col_partials_offset(M, g, c));
  }
  c.prog.num_rb = static_cast<int32_t>((M + 31) / 32);
  p.epi_warp_bytes = static_cast<uint32_t>(2 * kBoxBytes + c.n_aux * 2 * kBoxBytes);
  // MX kernels run two epilogue warp groups (even and odd chunks), each warp with its own staging
  const size_t n_epi_warps = static_cast<size_t>(kEpiWarps) * (mx ? kMaxEpiGroups : 1);
  const size_t ctl_bytes = (sizeof(Ctl) + 127) & ~size_t(127);
  const size_t stage_bytes = (pair ? kPairStageBytes : kStageBytes) + (mx ? kMxStageSFBytes : 0);
  auto stages_for = [&](size_t warp_bytes) -> int {
    const size_t fixed_b = 1024 + n_epi_warps * warp_bytes + ctl_bytes;
    if (static_cast<size_t>(dev.max_smem) < fixed_b + 2 * stage_bytes) return 0;
    const int s = static_cast<int>((static_cast<size_t>(dev.max_smem) - fixed_b) / stage_bytes);
    return s > kMaxStages ? kMaxStages : s;
  };
  // Column vectors: staged per tile in each epilogue warp's shared memory
  // where that costs no pipeline stage (a stage is worth more), else
  // prefetched into L1.
  const bool cv_fit = plan_colvecs(c.prog, p.half, p);
  const size_t cv_bytes = static_cast<size_t>(p.n_colpf) * (c.glu ? BN / 2 : BN) * sizeof(float);
  if (cv_fit && stages_for(p.epi_warp_bytes + cv_bytes) == stages_for(p.epi_warp_bytes)) {
    p.cv_smem = 1;
    p.epi_warp_bytes += static_cast<uint32_t>(cv_bytes);
  } else {
    for (int o = 0; o < c.prog.n_ops; ++o) c.prog.ops[o].cv = -1;
  }
  const size_t epi_bytes = n_epi_warps * p.epi_warp_bytes;
  const size_t fixed = 1024 + epi_bytes + ctl_bytes;
  if (static_cast<size_t>(dev.max_smem) < fixed + 2 * stage_bytes) return CODA_ERR_UNSUPPORTED;
  int stages = static_cast<int>((static_cast<size_t>(dev.max_smem) - fixed) / stage_bytes);
  if (stages > kMaxStages) stages = kMaxStages;
  p.stages = stages;
  p.smem_epi_off = static_cast<uint32_t>(stages * stage_bytes);
  p.smem_ctl_off = static_cast<uint32_t>(stages * stage_bytes + epi_bytes);
  p.err = dev.err;
  p.prog = c.prog;
  const size_t smem = fixed + static_cast<size_t>(stages) * stage_bytes;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool mn = b_layout == CODA_B_KN;
  const int cap = g_max_ctas.load();
  int grid = dev.sms;
  if (cap > 0 && cap < grid) grid = cap;
  cudaError_t e;
  // Split over K (stream-K): clusters take equal runs of (tile, k-block) units
  // and CTAs that share a tile publish fp32 partials to the workspace.
  bool split = false;
  auto arm_split = [&](int64_t sk_tiles) -> cudaError_t {
    const size_t slots = sk_tiles == g.num_tiles ? static_cast<size_t>(g.num_tiles) : static_cast<size_t>(kMaxSplitCtas);
    split = true;
    p.split = 1;
    p.sk_tiles = static_cast<int32_t>(sk_tiles);
    p.ws_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + split_base(ws_need));
    p.ws_cnt = reinterpret_cast<uint32_t*>(p.ws_part + slots * kSplitSegs * kPartFloats);
    return cudaMemsetAsync(p.ws_cnt, 0, slots * sizeof(uint32_t), st);
  };
  // slots the workspace holds (per tile, or per CTA for the last waves)
  const int64_t slots_room = split_room ? split_slots(g, pair) : 0;
  // Few tiles (single CTAs): the whole problem, in runs at least half a tile
  // long so that a tile has at most kSplitSegs contributors.
  if (!pair && slots_room >= g.num_tiles) {
    const int64_t units = g.num_tiles * g.num_kb;
    int64_t G = units / ((g.num_kb + 1) / 2);
    if (G > grid) G = grid;
    if (G > kMaxSplitCtas) G = kMaxSplitCtas;
    // automatic: only when at most half the SMs would have a tile.  Above that
    // the tiles' own weight streams already come close to HBM bandwidth
    // (86 CTAs pull ~6 TB/s), and publishing and re-reading the fp32 partials
    // costs more than the shorter mainloop saves.
    const bool idle = g_split_mode.load() == 2 || g.num_tiles * 2 <= static_cast<int64_t>(grid);
    if (idle && G > g.num_tiles) {
      grid = static_cast<int>(G);
      e = arm_split(g.num_tiles);
      if (e != cudaSuccess) return CODA_ERR_CUDA;
    }
  }
  // CTA pairs and split-K grids take the commuted-norm row scales from a
  // pre-pass kernel (a pair's A halves signal the leader's barrier; a split
  // CTA sees only part of each row), so they run no row-statistics warps.  So
  // does a single-CTA grid with fewer tiles than SMs: such a problem is bound
  // by the weight stream and the per-SM shared-memory traffic, and the
  // side path's reads of every A stage add to the latter.
  const bool rowstat_warps = c.has_rms && !pair && !split && g.num_tiles >= grid;
  if (c.rms_sumsq != nullptr) {   // the caller's row sums of squares: no pre-pass
    p.rms_vec = c.rms_sumsq;
    p.rms_from_sumsq = 1;
  }
  if (c.has_rms && !rowstat_warps) {
    float* mu_ws = c.is_ln ? rms_ws + M : nullptr;
    e = launch_rms_rowscale(A, M, K, p.inv_K, c.rms_eps, c.is_ln, rms_ws,
                            c.rms_slot >= 0 ? row_stats + static_cast<size_t>(c.rms_slot) * M : nullptr, mu_ws,
                            (c.is_ln && c.rms_slot >= 0) ? row_stats + static_cast<size_t>(c.rms_slot + 1) * M : nullptr,
                            st);
    p.mu_vec = mu_ws;
    if (e != cudaSuccess) return CODA_ERR_CUDA;
    g_launches.fetch_add(1);
    p.rms_vec = rms_ws;
  }
  if (pair) {
    int pairs = 0;
    e = max_pairs(c.glu, mn, smem, &pairs);
    if (e != cudaSuccess) return CODA_ERR_CUDA;
    if (pairs < 1) return CODA_ERR_UNSUPPORTED;
    if (pairs > grid / 2) pairs = grid / 2 > 0 ? grid / 2 : 1;
    if (g.num_tiles < pairs) pairs = static_cast<int>(g.num_tiles);
    grid = 2 * pairs;
  } else if (!split && g.num_tiles < grid) {
    grid = static_cast<int>(g.num_tiles);
  }
  const int csize = pair ? 2 : 1;
  // Many tiles: the whole-tile waves take ceil(T / C) tile times on C
  // clusters, the last wave partly idle.  Where that idle share is above 5% of
  // the run's cluster time, the tiles of the last, partly filled wave and of
  // the one before it (C to 2C - 1 tiles) are shared out as stream-K units
  // instead, ahead of the whole tiles (each run at least a tile long, so a
  // split tile has two contributors): every cluster then runs T / C tile
  // times, the partials' publish and re-read overlapping later tiles'
  // mainloops.  Measured, the idle share costs far less than its size: under
  // the power cap a partly filled last wave runs at higher clocks, so the
  // split gains little and its partials (publish ~10 us, re-read ~10 us per
  // cluster) can cost more; wgrad (9.5% idle) gains 1-5%, the LLaMA out- and
  // down-projections (3.8%) and rmsproj (3.7%) lose 1-15% when split.
  if (!split && slots_room >= kMaxSplitCtas && !rowstat_warps && grid <= kMaxSplitCtas) {
    const int64_t C = grid / csize;
    const int64_t T = g.num_tiles;
    if (C > 0 && T >= 2 * C) {
      const int64_t waves = (T + C - 1) / C;
      const int64_t idle = waves * C - T;   // cluster-tile slots left idle in the last wave
      if (g_split_mode.load() == 2 || idle * 20 > waves * C) {
        e = arm_split(T - (T / C - 1) * C);
        if (e != cudaSuccess) return CODA_ERR_CUDA;
      }
    }
  }
  // Dynamic tile order: one cluster per tile, where the tiles outnumber the
  // clusters that are resident at once (otherwise every cluster has one tile)
  p.clc = 0;
  if (g_dynamic_tiles.load() != 0 && !split && !rowstat_warps && cap == 0 && g.num_kb > 0 &&
      g.num_tiles > static_cast<int64_t>(grid / csize) && g.num_tiles * csize <= 0x7FFFFFFF) {
    p.clc = 1;
    grid = static_cast<int>(g.num_tiles * csize);
  }
  // Helpers on each CTA's last tile: measured +1.5% (rmsproj, 7 tiles per
  // cluster) to +3% (skinny, 1 tile; lnproj) and -0.4% on grids of ~36 tiles per
  // cluster (swiglu), where the last tile's epilogue is a small share of the run;
  // an epilogue with aux tiles is long enough to gain up to 64 (dgrad, 27: +0.6%)
  const int64_t tiles_per_cluster = (g.num_tiles + grid / csize - 1) / (grid / csize);
  // (their aux tiles are staged in the ring: four warps' output and aux buffers must fit in it)
  const bool ring_room = static_cast<size_t>(kEpiWarps) * (2 + 2 * c.n_aux) * kBoxBytes <=
                         static_cast<size_t>(stages) * stage_bytes;
  p.helpers = (g_tail_helpers.load() != 0 && !mx && !split && p.clc == 0 && ring_room && !rowstat_warps &&
               g.num_kb > 0 && (tiles_per_cluster <= 16 || (c.n_aux > 0 && tiles_per_cluster <= 64))) ? 1 : 0;
  int seq = match_sequence(epi, c.glu);
  auto launch = [&](int sq) {
    return mx ? launch_gemm_mx(sq, c.glu, pair, maps, p, grid, smem, st)
              : (fp8 ? launch_gemm_fp8(sq, c.glu, pair, maps, p, grid, smem, st)
                     : launch_gemm_seq(sq, c.glu, a_mn, mn, rowstat_warps, pair, maps, p, grid, smem, st));
  };
  e = launch(seq);
  if (e == cudaErrorNotSupported && seq != SEQ_INTERP) {
    (void)cudaGetLastError();   // the sequence has no kernel for this variant: interpret
    seq = SEQ_INTERP;
    e = launch(seq);
  }
  if (e != cudaSuccess) return CODA_ERR_CUDA;
  g_launches.fetch_add(1);
  g_last_plan = coda_plan{pair ? 1 : 0, split ? 1 : 0, grid, stages, g.num_tiles,
                          (p.rms_vec != nullptr && !p.rms_from_sumsq) ? 1 : 0, seq, p.clc,
                          p.cv_smem ? p.n_colpf : -p.n_colpf};
  if (c.prog.n_colred > 0) {
    e = launch_finalize_cols(c.prog.ws_col, c.prog.n_colred, c.prog.num_rb, g.n_out, c.prog.colred_slot,
                             c.col_stats, st);
    if (e != cudaSuccess) return CODA_ERR_CUDA;
    g_launches.fetch_add(1);
  }
  const bool need_keep = c.prog.has_dropout && row_keep_count != nullptr;
  if (c.prog.n_red > 0 || need_keep) {
    e = launch_finalize(p.ws_red, p.ws_keep, p.M, g.num_n_tiles, c.prog.n_red, c.prog.red,
                        static_cast<float>(1.0 / static_cast<double>(g.n_out)), row_stats,
                        need_keep ? row_keep_count : nullptr, st);
    if (e != cudaSuccess) return CODA_ERR_CUDA;
    g_launches.fetch_add(1);
  }
  return CODA_OK;
}

}  // namespace
}  // namespace coda

extern "C" {

coda_status coda_gemm_epilogue(const void* A, const void* B, int64_t M, int64_t N, int64_t K, int32_t b_layout,
                               const coda_epilogue* epi, const coda_aux* aux, void* D, float* row_stats,
                               uint32_t* row_keep_count, void* workspace, size_t workspace_bytes, void* stream) {
  return gemm_impl(A, B, M, N, K, b_layout, epi, aux, D, row_stats, row_keep_count, workspace, workspace_bytes,
                   stream, nullptr, nullptr);
}

coda_status coda_gemm_epilogue_mx(const void* A, const void* scale_A, const void* B, const void* scale_B, int64_t M,
                                  int64_t N, int64_t K, const coda_epilogue* epi, const coda_aux* aux, void* D,
                                  float* row_stats, uint32_t* row_keep_count, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  if (K > 0 && M > 0 && N > 0 && (scale_A == nullptr || scale_B == nullptr)) return CODA_ERR_INVALID_ARG;
  // K == 0 has no scales to read; the kernel path still needs a non-null marker
  static const uint8_t kNone[16] __attribute__((aligned(16))) = {};
  return gemm_impl(A, B, M, N, K, CODA_B_NK | CODA_AB_E4M3, epi, aux, D, row_stats, row_keep_count, workspace,
                   workspace_bytes, stream, scale_A ? scale_A : kNone, scale_B ? scale_B : kNone);
}

coda_status coda_fold_gamma(const void* W, const void* gamma, void* W_out, int64_t K, int64_t N, int32_t b_layout,
                            void* stream) {
  coda_status s = check_dims(0, N, K);
  if (s != CODA_OK) return s;
  if (b_layout != CODA_B_KN && b_layout != CODA_B_NK) return CODA_ERR_INVALID_ARG;
  if (K == 0 || N == 0) return CODA_OK;
  if (!W || !gamma || !W_out) return CODA_ERR_INVALID_ARG;
  if (!aligned16(W) || !aligned16(gamma) || !aligned16(W_out)) return CODA_ERR_ALIGNMENT;
  DevInfo dev;
  s = device_info(dev);
  if (s != CODA_OK) return s;
  const cudaError_t e =
      launch_fold_gamma(W, gamma, W_out, K, N, b_layout == CODA_B_KN, dev.sms, static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) g_launches.fetch_add(1);
  return from_cuda(e);
}

coda_status coda_fold_layernorm(const void* W, const void* gamma, const void* beta, void* W_out, float* colsum_out,
                                float* bias_out, int64_t K, int64_t N, int32_t b_layout, void* stream) {
  coda_status s = check_dims(0, N, K);
  if (s != CODA_OK) return s;
  if (b_layout != CODA_B_KN && b_layout != CODA_B_NK) return CODA_ERR_INVALID_ARG;
  if (K == 0 || N == 0) return CODA_OK;
  if (!W || !gamma || !W_out || !colsum_out || !bias_out || W_out == W) return CODA_ERR_INVALID_ARG;
  if (!aligned16(W) || !aligned16(gamma) || !aligned16(W_out) || (beta && !aligned16(beta)) ||
      !aligned4(colsum_out) || !aligned4(bias_out))
    return CODA_ERR_ALIGNMENT;
  DevInfo dev;
  s = device_info(dev);
  if (s != CODA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool kn = b_layout == CODA_B_KN;
  cudaError_t e = launch_fold_gamma(W, gamma, W_out, K, N, kn, dev.sms, st);
  if (e != cudaSuccess) return CODA_ERR_CUDA;
  g_launches.fetch_add(1);
  e = launch_ln_colsum(W_out, W, beta, K, N, kn, colsum_out, bias_out, st);
  if (e != cudaSuccess) return CODA_ERR_CUDA;
  g_launches.fetch_add(1);
  return CODA_OK;
}

coda_status coda_layernorm(const void* X, const void* gamma, const void* beta, int64_t M, int64_t K, float eps,
                           void* Xn_out, void* stream) {
  coda_status s = check_dims(M, 8, K);
  if (s != CODA_OK) return s;
  if (!std::isfinite(eps) || eps < 0.0f || K == 0) return CODA_ERR_INVALID_ARG;
  if (M == 0) return CODA_OK;
  if (!X || !gamma || !Xn_out) return CODA_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(gamma) || !aligned16(Xn_out) || (beta && !aligned16(beta))) return CODA_ERR_ALIGNMENT;
  DevInfo dev;
  s = device_info(dev);
  if (s != CODA_OK) return s;
  const cudaError_t e = launch_layernorm(X, gamma, beta, M, K, eps, Xn_out, static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) g_launches.fetch_add(1);
  return from_cuda(e);
}

coda_status coda_norm_backward(const void* g, const void* X, const float* r, const float* mu, const float* sum_g,
                               const float* sum_gx, int64_t M, int64_t K, void* dX, void* stream) {
  coda_status s = check_dims(M, 8, K);
  if (s != CODA_OK) return s;
  if (K == 0 || M == 0) return CODA_OK;
  if (!g || !X || !r || !sum_gx || !dX) return CODA_ERR_INVALID_ARG;
  if ((mu == nullptr) != (sum_g == nullptr)) return CODA_ERR_INVALID_ARG;   // LayerNorm needs both
  if (!aligned16(g) || !aligned16(X) || !aligned16(dX)) return CODA_ERR_ALIGNMENT;
  if (!aligned4(r) || !aligned4(sum_gx) || (mu && !aligned4(mu)) || (sum_g && !aligned4(sum_g)))
    return CODA_ERR_ALIGNMENT;
  DevInfo dev;
  s = device_info(dev);
  if (s != CODA_OK) return s;
  const cudaError_t e = launch_norm_backward(g, X, r, mu, sum_g, sum_gx, M, K, dX, dev.sms,
                                             static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) g_launches.fetch_add(1);
  return from_cuda(e);
}

coda_status coda_quantize_e4m3_rows(const void* X, int64_t M, int64_t K, void* Q, float* scale, void* stream) {
  coda_status s = check_dims(M, 16, K);
  if (s != CODA_OK) return s;
  if ((K % 16) != 0) return CODA_ERR_INVALID_ARG;
  if (M == 0 || K == 0) return CODA_OK;
  if (!X || !Q || !scale) return CODA_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(Q) || !aligned4(scale)) return CODA_ERR_ALIGNMENT;
  DevInfo dev;
  s = device_info(dev);
  if (s != CODA_OK) return s;
  const cudaError_t e = launch_quantize_e4m3_rows(X, M, K, Q, scale, static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) g_launches.fetch_add(1);
  return from_cuda(e);
}

size_t coda_mx_scale_bytes(int64_t R, int64_t K) {
  if (R <= 0 || K <= 0) return 0;
  return static_cast<size_t>((R + 127) / 128) * static_cast<size_t>((K + 127) / 128) * 512u;
}

coda_status coda_quantize_mx_e4m3(const void* X, int64_t R, int64_t K, void* Q, void* scales, void* stream) {
  coda_status s = check_dims(R, 32, K);
  if (s != CODA_OK) return s;
  if ((K % 32) != 0) return CODA_ERR_INVALID_ARG;
  if (R == 0 || K == 0) return CODA_OK;
  if (!X || !Q || !scales) return CODA_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(Q) || !aligned16(scales)) return CODA_ERR_ALIGNMENT;
  DevInfo dev;
  s = device_info(dev);
  if (s != CODA_OK) return s;
  const cudaError_t e = launch_quantize_mx_e4m3(X, R, K, Q, scales, coda_mx_scale_bytes(R, K), dev.sms,
                                                static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) g_launches.fetch_add(1);
  return from_cuda(e);
}

coda_status coda_rmsnorm(const void* X, const void* gamma, int64_t M, int64_t K, float eps, void* Xn_out,
                         float* rstd_out, void* stream) {
  coda_status s = check_dims(M, 8, K);
  if (s != CODA_OK) return s;
  if (!std::isfinite(eps) || eps < 0.0f || K == 0) return CODA_ERR_INVALID_ARG;
  if (M == 0) return CODA_OK;
  if (!X || !gamma || !Xn_out) return CODA_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(gamma) || !aligned16(Xn_out) || (rstd_out && !aligned4(rstd_out)))
    return CODA_ERR_ALIGNMENT;
  DevInfo dev;
  s = device_info(dev);
  if (s != CODA_OK) return s;
  const cudaError_t e = launch_rmsnorm(X, gamma, M, K, eps, Xn_out, rstd_out, static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) g_launches.fetch_add(1);
  return from_cuda(e);
}

coda_status coda_epilogue_apply(const void* C, int64_t M, int64_t N, const coda_epilogue* epi, const coda_aux* aux,
                                void* D, float* row_stats, uint32_t* row_keep_count, void* stream) {
  coda_status s = check_dims(M, N, 8);
  if (s != CODA_OK) return s;
  Compiled c;
  s = compile_epilogue(epi, aux, N, 8, false, c);
  if (s != CODA_OK) return s;
  if (M == 0 || N == 0) return CODA_OK;
  if (!C || !D) return CODA_ERR_INVALID_ARG;
  if (!aligned16(C) || !aligned16(D)) return CODA_ERR_ALIGNMENT;
  if (c.needs_row_stats && row_stats == nullptr) return CODA_ERR_INVALID_ARG;
  if ((row_stats && !aligned4(row_stats)) || (row_keep_count && !aligned4(row_keep_count)))
    return CODA_ERR_ALIGNMENT;
  DevInfo dev;
  s = device_info(dev);
  if (s != CODA_OK) return s;
  const int64_t n_out = c.glu ? N / 2 : N;
  const cudaError_t e = launch_epilogue_apply(C, D, M, static_cast<int>(N), static_cast<int>(n_out),
                                              c.glu ? static_cast<int>(N / 2) : 0, c.aux_ptr, row_stats,
                                              c.prog.has_dropout ? row_keep_count : nullptr, c.prog,
                                              static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) g_launches.fetch_add(1);
  return from_cuda(e);
}

coda_status coda_check_device_error(void* stream, uint32_t* info) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return CODA_ERR_CUDA;
  DevInfo dev;
  coda_status s = device_info(dev);
  if (s != CODA_OK) return s;
  uint32_t h[4] = {0, 0, 0, 0};
  if (cudaMemcpy(h, dev.err, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return CODA_ERR_CUDA;
  if (info) std::memcpy(info, h, sizeof(h));
  if (h[0] == 0) return CODA_OK;
  const uint32_t z[4] = {0, 0, 0, 0};
  if (cudaMemcpy(dev.err, z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess) return CODA_ERR_CUDA;
  return static_cast<coda_status>(h[0]);
}

const char* coda_status_string(coda_status status) {
  switch (status) {
    case CODA_OK: return "CODA_OK";
    case CODA_ERR_INVALID_ARG: return "CODA_ERR_INVALID_ARG";
    case CODA_ERR_UNSUPPORTED: return "CODA_ERR_UNSUPPORTED";
    case CODA_ERR_ALIGNMENT: return "CODA_ERR_ALIGNMENT";
    case CODA_ERR_CUDA: return "CODA_ERR_CUDA";
    case CODA_ERR_TIMEOUT: return "CODA_ERR_TIMEOUT";
    case CODA_ERR_WORKSPACE: return "CODA_ERR_WORKSPACE";
    default: return "CODA_ERR_UNKNOWN";
  }
}

uint64_t coda_launch_count(void) { return g_launches.load(); }

void coda_set_pipeline_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns == 0 ? 1000000000ull : ns); }

void coda_set_max_ctas(int32_t n) { g_max_ctas.store(n < 0 ? 0 : n); }

void coda_set_cta_pair(int32_t mode) { g_pair_mode.store(mode < 0 || mode > 2 ? 0 : mode); }

void coda_set_fixed_sequences(int32_t enable) { g_fixed_seqs.store(enable != 0 ? 1 : 0); }

void coda_set_split_k(int32_t mode) { g_split_mode.store(mode < 0 || mode > 2 ? 0 : mode); }

void coda_set_tile_scheduler(int32_t dynamic) { g_dynamic_tiles.store(dynamic != 0 ? 1 : 0); }

void coda_set_tail_helpers(int32_t enable) { g_tail_helpers.store(enable != 0 ? 1 : 0); }

void coda_set_raster(int32_t mode, int32_t group) {
  g_raster_mode.store(mode < 0 || mode > 2 ? 0 : mode);
  g_raster_group.store(group);
}

void coda_last_plan(coda_plan* out) {
  if (out != nullptr) *out = g_last_plan;
}

}  // extern "C"
