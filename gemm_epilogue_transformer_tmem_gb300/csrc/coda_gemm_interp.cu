// Instantiations of the fused kernel with the op-list interpreter (any op list)
// for plain (unpaired) outputs, and the CTA-pair occupancy queries; the
// SwiGLU-paired instantiations are compiled in coda_gemm_interp_glu.cu.
#include <mutex>

#include "coda_gemm_kernel.cuh"
#include "coda_launch.h"

namespace coda {

cudaError_t launch_gemm_interp(bool glu, bool a_mn_major, bool b_mn_major, bool row_stats, bool pair,
                               const CUtensorMap* maps, const GemmParams& p, int grid, size_t smem, cudaStream_t st) {
  if (glu) return launch_gemm_interp_glu(a_mn_major, b_mn_major, row_stats, pair, maps, p, grid, smem, st);
  return launch_variant<EpiInterp, false, true, true>(a_mn_major, b_mn_major, row_stats, pair, maps, p, grid, smem, st);
}

// The occupancy query costs a driver round trip; its answer depends only on
// the device, the variant and the shared memory, so it is kept (a handful of
// entries per process).
cudaError_t max_pairs(bool glu, bool b_mn_major, size_t smem, int* pairs) {
  struct Entry {
    int dev, glu, mn;
    size_t smem;
    int pairs;
  };
  static std::mutex mu;
  static Entry cache[32];
  static int n_cached = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < n_cached; ++i)
      if (cache[i].dev == dev && cache[i].glu == glu && cache[i].mn == b_mn_major && cache[i].smem == smem) {
        *pairs = cache[i].pairs;
        return cudaSuccess;
      }
  }
  if (glu)
    e = max_pairs_glu(b_mn_major, smem, pairs);
  else
    e = b_mn_major ? max_active_pairs_t<false, true, false>(smem, pairs)
                   : max_active_pairs_t<false, false, false>(smem, pairs);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  if (n_cached < 32) cache[n_cached++] = Entry{dev, glu ? 1 : 0, b_mn_major ? 1 : 0, smem, *pairs};
  return cudaSuccess;
}

}  // namespace coda
