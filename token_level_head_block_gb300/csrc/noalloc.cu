// mhla_forward_noalloc: the MHLA forward for callers that are not allowed to
// allocate device memory.
//
// Some callers cannot call cudaMalloc (or cudaMallocAsync) at the point where
// they run the forward pass: an inference engine's plugin that executes inside
// the engine's enqueue step, where the engine owns every byte of device memory
// and forbids allocation on the serving path; a latency-critical loop that plans
// all memory once at start-up because cudaFree synchronises the whole device and
// an allocation can fail under fragmentation at the worst moment.  Those callers
// still own and pass their inputs and outputs, but the forward's scratch
// (summaries, mixed summaries, the bf16 copy of W) comes from a fixed-size array
// that lives in this library's device image, so the call itself allocates
// nothing.
#include <cuda_runtime.h>

#include <mutex>

#include "mhla_internal.h"

namespace mhla {
namespace {

constexpr size_t kScratchBytes = MHLA_NOALLOC_SCRATCH_BYTES;

// One copy per GPU that loads this library, held until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The name
// g_noalloc_scratch in host code is only a host-side stand-in for the symbol,
// so the address is looked up once per device, with that device current.
void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return nullptr;
    g_scratch_addr[dev] = ptr;
  }
  return g_scratch_addr[dev];
}

}  // namespace
}  // namespace mhla

extern "C" mhla_status_t mhla_forward_noalloc(const mhla_tensor_t* q, const mhla_tensor_t* k,
                                              const mhla_tensor_t* v, const float* W,
                                              const mhla_shape3_t* grid, const mhla_shape3_t* block,
                                              const mhla_phi_t* phi, const mhla_tensor_t* out, void* stream,
                                              int32_t path) {
  // Reject a problem whose scratch would not fit before touching the device.
  size_t need = 0;
  const mhla_status_t sz = mhla_workspace_size(q, grid, block, path, &need);
  if (sz != MHLA_OK) return sz;
  if (need > mhla::kScratchBytes) return MHLA_ERR_WORKSPACE;
  void* scratch = mhla::scratch_on_current_device();
  if (!scratch) return MHLA_ERR_CUDA;
  // mhla_forward re-checks the need for the path it actually takes against the
  // array's capacity and returns MHLA_ERR_WORKSPACE when it does not fit.
  return mhla_forward(q, k, v, W, grid, block, phi, out, scratch, mhla::kScratchBytes, stream, path);
}
