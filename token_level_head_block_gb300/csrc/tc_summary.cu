// tc_summary: the first step of the tensor-core path of the MHLA forward on
// sm_103a, [S_j | z_j] = phi(K_j)^T [V_j | 1] per (b, head group, block j)
// ([P2] "MHLA: Restoring Expressivity of Linear Attention via Token-Level
// Multi-Head", section 4 "Architecture": local key-value summaries; [P1]
// 171host.com/767426.html, section 7, MHLA.forward: kv = k^T v, k_sum).

// The pipeline itself lives in tc_fwd_bodies.cuh (shared with the fused
// launch).  Every mbarrier wait is bounded (time and poll count); a wait that
// gives up raises a per-CTA abort flag so the other roles stop waiting too, sets
// bit 0 of this file's device error word, and the CTA drains its copies,
// releases tensor memory and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "mhla_internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"
#include "tc_fwd_bodies.cuh"
#include "tma_host.h"

namespace mhla {

__device__ unsigned int g_sum_error = 0;

namespace {

using namespace ptx;
using namespace tc;

// ============================================================================
// tc_summary: the summary pipeline (tc_fwd_bodies.cuh) in a launch of its own.
// Its prologue also rounds W to bf16 for the mixing GEMM that follows.
// ============================================================================
constexpr int kTcThreads = 320;  // producer, MMA, 4 phi warps, 4 epilogue warps
constexpr int kSumCtrl = 1024;

template <int D>
constexpr size_t sum_smem() {
  return SumCfg<D>::DATA + kSumCtrl + 1024;
}

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
tc_summary(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v, TcGeom g,
           int32_t G, int64_t n_items, int phi_kind, float eps,
           __nv_bfloat16* __restrict__ Sbuf, const float* __restrict__ W, __nv_bfloat16* __restrict__ Wb,
           __nv_bfloat16* __restrict__ WbT, int64_t Mp, int32_t Mw, int32_t upb) {
  using Cfg = SumCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  uint8_t* stages = smem;
  uint8_t* ctrl = smem + Cfg::DATA;
  const SumBars bars = sum_bars<D>(ctrl);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 512);
  volatile uint32_t* abortf = tmem_slot + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    sum_init<D>(bars);
    *abortf = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  sum_fill_ones<D>(stages, threadIdx.x, kTcThreads);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Launched as a dependent grid: the set-up above overlaps the previous kernel's
  // tail; W, k and v (which that kernel may have written) are read only after it.
  grid_dep_wait();
  // W rounded to bf16 for the mixing GEMM, [M][Mp] with zero padding (and, when
  // WbT is given, W^T likewise); every CTA converts a slice (the GEMM runs after
  // this kernel on the same stream).  Wb null: summaries only.  upb > 0: the
  // summaries are of causal units (upb per block of the Mw x Mw matrix W), and
  // Wb is the unit-level W': W[b(i)][b(j)] for a past block, W[b(i)][b(i)] for
  // an earlier unit of the same block, 0 otherwise.
  if (Wb) {
    const int64_t n = static_cast<int64_t>(g.M) * Mp;
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * kTcThreads + threadIdx.x; e < n;
         e += static_cast<int64_t>(gridDim.x) * kTcThreads) {
      const int64_t i = e / Mp, j = e % Mp;
      float x = 0.0f;
      if (j < g.M) {
        if (upb > 0) {
          const int64_t bi = i / upb, bj = j / upb;
          if (bj < bi || (bj == bi && j < i)) x = W[bi * Mw + bj];
        } else {
          x = W[i * g.M + j];
        }
      }
      Wb[e] = __float2bfloat16_rn(x);
      if (WbT) WbT[e] = __float2bfloat16_rn(j < g.M ? W[j * g.M + i] : 0.0f);   // W^T for the backward
    }
  }
  summary_roles<D>(&tm_k, &tm_v, g, G, blockIdx.x, gridDim.x, n_items, phi_kind, eps, Sbuf, stages, bars, tmem,
                   abortf, &g_sum_error, nullptr);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::TMEM_COLS);
  }
}

template <int D>
int run_summary(const Problem& p, const float* W, __nv_bfloat16* Wb, __nv_bfloat16* WbT, int64_t Mp,
                __nv_bfloat16* Sbuf, int32_t Mw, int32_t upb, cudaStream_t stream) {
  using Cfg = SumCfg<D>;
  constexpr size_t SMEM = sum_smem<D>();
  const int sms = device_sm_count();
  if (sms <= 0) return MHLA_ERR_CUDA;
  ChunkPlan c64;
  if (!chunk_plan(p, 64, &c64)) return MHLA_ERR_UNSUPPORTED;
  CUtensorMap tk, tv;
  if (!operand_map(p, p.k, c64.box_y, c64.box_t, &tk) || !operand_map(p, p.v, c64.box_y, c64.box_t, &tv))
    return MHLA_ERR_CUDA;
  const int32_t G = static_cast<int32_t>((p.H + Cfg::HP - 1) / Cfg::HP);
  const int64_t n_items = p.B * G * p.M;
  if (cudaFuncSetAttribute(tc_summary<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(SMEM)) != cudaSuccess)
    return MHLA_ERR_CUDA;
  const int per_sm = std::max(1, occupancy(tc_summary<D>, kTcThreads, SMEM));
  const int grid = static_cast<int>(std::min<int64_t>(n_items, static_cast<int64_t>(sms) * per_sm));
  KernelTimer timer("tc_summary", stream);
  const cudaError_t e = launch_dependent(tc_summary<D>, dim3(grid), dim3(kTcThreads), SMEM, stream, tk, tv,
                                         make_geom(p, c64), G, n_items, p.phi_kind, p.eps, Sbuf, W, Wb, WbT, Mp, Mw,
                                         upb);
  return e == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
}

}  // namespace

int tc_run_summary(const Problem& p, const float* W, void* Wb, void* WbT, int64_t Mp, void* Sbuf, void* stream,
                   int32_t Mw, int32_t upb) {
  auto* wb = static_cast<__nv_bfloat16*>(Wb);
  auto* wbt = static_cast<__nv_bfloat16*>(WbT);
  auto* sb = static_cast<__nv_bfloat16*>(Sbuf);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return p.d == 64 ? run_summary<64>(p, W, wb, wbt, Mp, sb, Mw, upb, s)
                   : run_summary<32>(p, W, wb, wbt, Mp, sb, Mw, upb, s);
}

int read_and_clear_summary_error(void* stream, uint32_t* flags) { return read_and_clear_word(g_sum_error, stream, flags); }

MHLA_DEFINE_STALL_SETTER(set_stall_summary)

}  // namespace mhla
