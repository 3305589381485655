// gs_bin_sort_noalloc (see below): gs_bin_sort with its scratch in a fixed array.
#include <mutex>

#include "api_util.h"
#include "binsort_layout.h"

// ---------------------------------------------------------------------------
// gs_bin_sort_noalloc: the same binning for callers that may not allocate device
// memory, e.g. a real-time loop whose memory is all reserved at start-up, or an
// application that embeds the library while its own allocator owns the GPU.  The
// sort's scratch lives in the file-scope array below, which every GPU that loads
// this module holds until the process exits.  It is the only object of this
// translation unit.  Under lazy module loading (the CUDA default) the module that
// carries it is loaded by the first call on a device, and that load is itself a
// device allocation; with CUDA_MODULE_LOADING=EAGER every process that loads the
// library holds the array on each GPU it uses.  Either way a caller makes one call
// during start-up, before it stops allocating and before any stream capture.  The
// array's device address is looked up once per device and kept: that assumes the
// device's primary context, with no cudaDeviceReset after the first call (a reset
// would leave the kept address stale).  Its size is the workspace of
// n = GS_NOALLOC_MAX_N Gaussians, capacity_K = GS_NOALLOC_MAX_K intersections and
// GS_NOALLOC_MAX_TILES tiles, which covers every smaller problem.
namespace gs {

constexpr size_t kNoAllocBytes = sort_layout(GS_NOALLOC_MAX_N, GS_NOALLOC_MAX_K, GS_NOALLOC_MAX_TILES).total;
static_assert(kNoAllocBytes == 71860736, "fixed scratch size changed");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

}  // namespace gs

extern "C" gs_status gs_bin_sort_noalloc(gs_dims dims, const gs_proj* proj, const gs_camera* cam,
                                         uint32_t capacity_K, gs_bins bins, uint32_t* dev_status,
                                         cudaStream_t stream) {
  using namespace gs;
  if (!dims_ok(dims) || !camera_ok(cam)) return GS_ERR_INVALID_ARG;
  const int64_t tiles = n_tiles(cam);
  if (dims.n > GS_NOALLOC_MAX_N || capacity_K > GS_NOALLOC_MAX_K || tiles > GS_NOALLOC_MAX_TILES)
    return GS_ERR_SCRATCH_LIMIT;
  const size_t need = sort_layout(dims.n, capacity_K, tiles).total;
  if (need > kNoAllocBytes) return GS_ERR_SCRATCH_LIMIT;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return GS_ERR_CUDA;
  void* scratch = nullptr;
  {
    // once per device, with that device current: the device address of the array
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return GS_ERR_CUDA;
      g_noalloc_ptr[dev] = p;
    }
    scratch = g_noalloc_ptr[dev];
  }
  return gs_bin_sort(dims, proj, cam, capacity_K, bins, scratch, kNoAllocBytes, dev_status, stream);
}
