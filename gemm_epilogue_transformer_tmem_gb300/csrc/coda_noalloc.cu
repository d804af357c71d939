// coda_gemm_epilogue_noalloc: the fused GEMM + epilogue for callers that cannot
// allocate device memory when they call it.
//
// Some callers cannot call cudaMalloc at call time: a serving loop that fixes
// its device-memory footprint at start-up and forbids allocation afterwards
// (cudaMalloc can synchronise the device and has no latency bound), or a host
// runtime whose device memory is owned entirely by another allocator.  This
// entry point needs no workspace from them: the cross-tile row-reduction and
// keep-count partials live in one fixed buffer compiled into the library.
//
// The buffer is a file-scope __device__ array of CODA_NOALLOC_SCRATCH_BYTES.
// Every GPU that loads the library holds it until the process exits.  Host code
// cannot use the array's name as a device address (on the host it names a
// stand-in object), so the device address is looked up with
// cudaGetSymbolAddress once per device, with that device current, on the first
// call made on that device, and then passed to the kernels as their workspace.
//
// All calls share the one buffer, and it keeps whatever the last call wrote.
// Nothing in it has to start at zero: the fused kernel writes every partial
// (one per reduction, column tile and row) before the finishing kernel reads
// it.  Calls whose kernels can overlap on the GPU (different streams, or
// different host threads on the same device) race on the buffer.
#include <cuda_runtime.h>

#include <mutex>

#include "coda_internal.h"
#include "coda_launch.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[CODA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// device address of g_noalloc_scratch on the current device
coda_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CODA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return CODA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return CODA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return CODA_OK;
}

}  // namespace

extern "C" CODA_API coda_status coda_gemm_epilogue_noalloc(const void* A, const void* B, int64_t M, int64_t N,
                                                           int64_t K, int32_t b_layout, const coda_epilogue* epi,
                                                           const coda_aux* aux, void* D, float* row_stats,
                                                           uint32_t* row_keep_count, void* stream) {
  // the minimum the problem needs; the whole buffer is offered, so the split
  // over K runs when its partials fit as well
  size_t need = 0;
  coda_status s = coda::workspace_need(M, N, K, epi, false, &need);
  if (s != CODA_OK) return s;
  if (need > static_cast<size_t>(CODA_NOALLOC_SCRATCH_BYTES)) return CODA_ERR_WORKSPACE;
  void* scratch = nullptr;
  s = scratch_address(&scratch);
  if (s != CODA_OK) return s;
  return coda_gemm_epilogue(A, B, M, N, K, b_layout, epi, aux, D, row_stats, row_keep_count, scratch,
                            CODA_NOALLOC_SCRATCH_BYTES, stream);
}
