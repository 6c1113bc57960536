// Per-kernel CUDA-event timing behind mhla_profile_begin / mhla_profile_end,
// and an NVTX range named after the kernel around every launch (a no-op unless
// a profiler such as Nsight Systems or Nsight Compute is attached; ncu can then
// select launches with --nvtx-include).
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "mhla_internal.h"

namespace mhla {
namespace {

struct Record {
  const char* name;
  cudaEvent_t start, stop;
};

std::mutex g_mu;
std::atomic<bool> g_active{false};
std::vector<Record> g_records;

}  // namespace

KernelTimer::KernelTimer(const char* name, void* stream) : name_(name), stream_(stream), start_(nullptr) {
  nvtxRangePushA(name);
  if (!g_active.load(std::memory_order_acquire)) return;
  cudaEvent_t e;
  if (cudaEventCreate(&e) != cudaSuccess) return;
  if (cudaEventRecord(e, static_cast<cudaStream_t>(stream_)) != cudaSuccess) {
    cudaEventDestroy(e);
    return;
  }
  start_ = e;
}

KernelTimer::~KernelTimer() {
  nvtxRangePop();
  if (!start_) return;
  cudaEvent_t stop;
  if (cudaEventCreate(&stop) != cudaSuccess || cudaEventRecord(stop, static_cast<cudaStream_t>(stream_)) != cudaSuccess) {
    cudaEventDestroy(static_cast<cudaEvent_t>(start_));
    return;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  g_records.push_back(Record{name_, static_cast<cudaEvent_t>(start_), stop});
}

}  // namespace mhla

using namespace mhla;

extern "C" mhla_status_t mhla_profile_begin(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (Record& r : g_records) {
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  g_records.clear();
  g_active.store(true, std::memory_order_release);
  return MHLA_OK;
}

extern "C" mhla_status_t mhla_profile_end(mhla_kernel_time_t* out, int32_t capacity, int32_t* count) {
  if (!count || (capacity > 0 && !out)) return MHLA_ERR_INVALID_ARG;
  g_active.store(false, std::memory_order_release);
  std::lock_guard<std::mutex> lk(g_mu);
  struct Sum { std::string name; int32_t launches; double ms; };
  std::vector<Sum> sums;
  mhla_status_t st = MHLA_OK;
  for (Record& r : g_records) {
    float ms = 0.0f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess)
      st = MHLA_ERR_CUDA;
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
    Sum* slot = nullptr;
    for (Sum& s : sums)
      if (s.name == r.name) slot = &s;
    if (!slot) {
      sums.push_back(Sum{r.name, 0, 0.0});
      slot = &sums.back();
    }
    slot->launches += 1;
    slot->ms += ms;
  }
  g_records.clear();
  *count = static_cast<int32_t>(sums.size());
  for (int32_t i = 0; i < capacity && i < static_cast<int32_t>(sums.size()); ++i) {
    std::memset(out[i].name, 0, sizeof(out[i].name));
    std::strncpy(out[i].name, sums[i].name.c_str(), sizeof(out[i].name) - 1);
    out[i].launches = sums[i].launches;
    out[i].total_ms = static_cast<float>(sums[i].ms);
  }
  return st;
}
