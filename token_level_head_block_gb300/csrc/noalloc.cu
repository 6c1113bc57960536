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
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "mhla_internal.h"

namespace mhla {
namespace {

constexpr size_t kScratchBytes = MHLA_NOALLOC_SCRATCH_BYTES;

// One copy per GPU that loads this library, held until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// cuCtxGetCurrent through the runtime's driver entry point (no link-time
// dependency on libcuda).
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Device address of the array in each context it was looked up in.  The key is
// the CUDA context, not the device index: a context created after a reset of
// the device holds its own copy of the array at its own address.
constexpr int kMaxContexts = 64;
std::mutex g_mu;
CUcontext g_ctx[kMaxContexts] = {};
void* g_addr[kMaxContexts] = {};
int g_used = 0;

// The name g_noalloc_scratch in host code is only a host-side stand-in for the
// symbol, so its device address is looked up once per context, with the
// caller's device current.  The first lookup in a context loads this file's
// device code there, and the driver allocates the array's memory at that
// moment: the reason callers make their first call at start-up.
void* scratch_in_current_context() {
  CtxGetCurrentFn get = ctx_get_current();
  CUcontext ctx = nullptr;
  if (!get || get(&ctx) != CUDA_SUCCESS) return nullptr;
  if (!ctx) {
    // No context is current on this thread yet: make the current device's
    // primary context current (cudaSetDevice initialises it; no memory is
    // allocated for this library).
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || cudaSetDevice(dev) != cudaSuccess) return nullptr;
    if (get(&ctx) != CUDA_SUCCESS || !ctx) return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  for (int e = 0; e < g_used; ++e)
    if (g_ctx[e] == ctx) return g_addr[e];
  if (g_used == kMaxContexts) return nullptr;
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return nullptr;
  g_ctx[g_used] = ctx;
  g_addr[g_used] = ptr;
  ++g_used;
  return ptr;
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
  void* scratch = mhla::scratch_in_current_context();
  if (!scratch) return MHLA_ERR_CUDA;
  // mhla_forward re-checks the need for the path it actually takes against the
  // array's capacity and returns MHLA_ERR_WORKSPACE when it does not fit.
  return mhla_forward(q, k, v, W, grid, block, phi, out, scratch, mhla::kScratchBytes, stream, path);
}
