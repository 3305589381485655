// Small C-ABI utilities: status strings, version, the device's SM count the grids
// are sized from, and the library exponential exposed for cross-checking.
#include <atomic>

#include "api_util.h"
#include "gs_common.cuh"

namespace gs {

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];  // 0 until queried
}  // namespace

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();  // leave no sticky error behind for launch_status
    return 1;
  }
  int c = g_sm_count[dev].load(std::memory_order_relaxed);
  if (c > 0) return c;
  if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0) {
    cudaGetLastError();
    return 1;
  }
  g_sm_count[dev].store(c, std::memory_order_relaxed);
  return c;
}

__global__ void k_expf(const float* __restrict__ x, float* __restrict__ y, int64_t n) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) y[i] = gs_expf(x[i]);
}

}  // namespace gs

extern "C" gs_status gs_util_expf(const float* x, float* y, int64_t n, cudaStream_t stream) {
  using namespace gs;
  if (n < 0 || (n > 0 && (!x || !y))) return GS_ERR_INVALID_ARG;
  if (n == 0) return GS_OK;
  k_expf<<<grid_for(n, 256, sm_count() * 16), 256, 0, stream>>>(x, y, n);
  return launch_status();
}

extern "C" int32_t gs_sm_count(void) { return gs::sm_count(); }

extern "C" const char* gs_status_str(uint32_t status) {
  if (status == 0) return "ok";
  if (status & GS_ERR_INVALID_ARG) return "invalid argument";
  if (status & GS_ERR_CUDA) return "CUDA launch failed";
  if (status & GS_ERR_CAPACITY) return "tile intersections exceed capacity";
  if (status & GS_ERR_TIMEOUT) return "bounded device wait gave up";
  if (status & GS_ERR_NONFINITE) return "non-finite Gaussian parameters";
  if (status & GS_ERR_SCRATCH_LIMIT) return "sizes exceed the fixed scratch of gs_bin_sort_noalloc";
  return "unknown status";
}

extern "C" const char* gs_version(void) { return "gs-gb300 0.1 sm_103a"; }
