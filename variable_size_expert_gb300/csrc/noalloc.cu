// mgg_route_noalloc: the device router with its scratch in a fixed,
// library-owned device array instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory at the moment they need
// routing: code running inside an allocator-free region (a custom memory
// manager that hands out only the tensors it planned, an inference engine
// whose arena is sealed after start-up), or a host path where calling
// cudaMalloc would synchronise the device.  For them this entry point uses
// a 1 MiB array that every GPU loading the library reserves once (and keeps
// until the process exits); nothing is allocated or freed per call.
#include <mutex>

#include "../../include/mgg.h"
#include "internal.h"

namespace mgg {
namespace {

constexpr size_t kScratchBytes = MGG_NOALLOC_SCRATCH_BYTES;

// Per-chunk expert histogram of the router (see router.cu).  One instance
// per device; shared by every call on that device.
static __device__ __align__(256) int32_t g_route_scratch[kScratchBytes / sizeof(int32_t)];

std::mutex g_mu;
void* g_scratch_ptr[64] = {};

// Device address of this device's scratch array, looked up once per device
// with that device current (the host-side symbol is only a stand-in).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace mgg

extern "C" mgg_status mgg_route_noalloc(const int32_t* expert_ids, const float* topk_weights,
                                        int T, int k, int E, int N, mgg_dtype dtype,
                                        const mgg_routing* routing, int32_t* dev_status,
                                        void* stream) {
  const mgg::NvtxRange nvtx("mgg_route_noalloc");
  using namespace mgg;
  if (!expert_ids || !topk_weights || !dev_status || !routing || !routing->counts ||
      !routing->end_offs || !routing->start || !routing->tile_start || !routing->row_assign ||
      !routing->row_token || !routing->row_weight || !routing->assign_row)
    return MGG_ERR_INVALID_ARG;
  if (T < 1 || k < 1 || E < 1 || N < 1 || E > kMaxExperts) return MGG_ERR_INVALID_ARG;
  if (static_cast<long long>(T) * k > (1LL << 30)) return MGG_ERR_INVALID_ARG;
  if (dtype != MGG_BF16 && dtype != MGG_F32 && dtype != MGG_FP8_E4M3) return MGG_ERR_DTYPE;
  // the fixed array must hold the per-chunk histogram
  if (route_ws_bytes(T, k, E) > kScratchBytes) return MGG_ERR_WORKSPACE;
  // only sm_103 images are built: check before touching the device symbol
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MGG_ERR_CUDA;
  if (major != 10 || minor != 3) return MGG_ERR_UNSUPPORTED_ARCH;
  // mgg_route then validates the rest and launches the router kernels on
  // the fixed array
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MGG_ERR_CUDA;
  return mgg_route(expert_ids, topk_weights, T, k, E, N, dtype, routing, dev_status, scratch,
                   kScratchBytes, stream);
}
