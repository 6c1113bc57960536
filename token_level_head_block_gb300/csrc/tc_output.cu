// tc_output: the readout step of the tensor-core path, per (b, h, block i),
// 128 tokens at a time: o_t = phi(q_t) S~_i / (phi(q_t) . z~_i + eps)
// ([P2] "MHLA: Restoring Expressivity of Linear Attention via Token-Level
// Multi-Head", section 4 "Token-Level Adaptivity"; [P1] 171host.com/767426.html,
// section 5(4) and section 7, MHLA.forward).

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

__device__ unsigned int g_out_error = 0;

namespace {

using namespace ptx;
using namespace tc;

// ============================================================================
// tc_output: the readout pipeline (tc_fwd_bodies.cuh) in a launch of its own,
// items taken in a fixed order (blockIdx.x, + gridDim.x, ...).
// ============================================================================
constexpr int kOutThreadsTC = 512;   // 16 warps: see the roles in tc_fwd_bodies.cuh

template <int D>
constexpr size_t out_smem() {
  return OutCfg<D>::DATA + 2048 + 1024;
}

template <int D, bool PAIR>
__global__ void __launch_bounds__(kOutThreadsTC, 1)
tc_output(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_o,
          const __grid_constant__ CUtensorMap tm_st, TcGeom g, int64_t n_items, int phi_kind, float eps,
          const float* __restrict__ zt, const __nv_bfloat16* St) {
  using Cfg = OutCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  uint8_t* ctrl = smem + Cfg::DATA;
  const OutBars bars = out_bars<D>(ctrl);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 1536);
  volatile uint32_t* abortf = tmem_slot + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    out_init<D>(bars);
    *abortf = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_o);
    prefetch_tmap(&tm_st);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  if (PAIR) {
    out_zero_offdiag<D, PAIR>(smem + Cfg::NQ * Cfg::QT, threadIdx.x, kOutThreadsTC);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const OutSched sc{blockIdx.x, gridDim.x, n_items, nullptr, nullptr, 1};
  output_roles<D, PAIR>(&tm_q, &tm_o, &tm_st, g, sc, phi_kind, eps, zt, St, smem, bars, tmem, abortf,
                        &g_out_error);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::TMEM_COLS);
  }
}

// ----------------------------------------------------------------- host side

template <int D, bool PAIR>
int run_output(const Problem& p, const __nv_bfloat16* St, const float* zt, cudaStream_t stream) {
  using Cfg = OutCfg<D>;
  constexpr size_t SMEM = out_smem<D>();
  const int sms = device_sm_count();
  if (sms <= 0) return MHLA_ERR_CUDA;
  // PAIR: the problem seen with heads of 64 channels, two real heads each
  Problem v = p;
  if (PAIR) {
    v.d = 64;
    v.H = p.H / 2;
    v.q.sh = 2 * p.q.sh;
    v.o.sh = 2 * p.o.sh;
  }
  ChunkPlan c128;
  if (!chunk_plan(v, 128, &c128)) return MHLA_ERR_UNSUPPORTED;
  CUtensorMap tq, to;
  if (!operand_map(v, v.q, c128.box_y, c128.box_t, &tq) || !operand_map(v, v.o, c128.box_y, c128.box_t, &to))
    return MHLA_ERR_CUDA;
  // S~ tiles (row-major [BH*M][d][d]) seen as (c % 8, r, c / 8, tile): a
  // (8, d, d/8, 1) box lands as 16-byte rows of 8 columns, d rows per column
  // group: the unswizzled MN-major operand layout (PAIR: one column group per box).
  CUtensorMap tst;
  {
    const cuuint64_t dims[4] = {8u, static_cast<cuuint64_t>(p.d), static_cast<cuuint64_t>(p.d / 8),
                                static_cast<cuuint64_t>(p.BH() * p.M)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(p.d * 2), 16u, static_cast<cuuint64_t>(p.d * p.d * 2)};
    const cuuint32_t box[4] = {8u, static_cast<cuuint32_t>(p.d), PAIR ? 1u : static_cast<cuuint32_t>(p.d / 8), 1u};
    if (!encode_tensor_map(&tst, 4, const_cast<__nv_bfloat16*>(St), dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE))
      return MHLA_ERR_CUDA;
  }
  const int64_t n_items = v.BH() * v.M;
  if (cudaFuncSetAttribute(tc_output<D, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(SMEM)) != cudaSuccess)
    return MHLA_ERR_CUDA;
  const int per_sm =
      std::max(1, std::min(occupancy(tc_output<D, PAIR>, kOutThreadsTC, SMEM), 512 / Cfg::TMEM_COLS));
  const int grid = static_cast<int>(std::min<int64_t>(n_items, static_cast<int64_t>(sms) * per_sm));
  KernelTimer timer("tc_output", stream);
  const cudaError_t e = launch_dependent(tc_output<D, PAIR>, dim3(grid), dim3(kOutThreadsTC), SMEM, stream, tq,
                                         to, tst, make_geom(v, c128), n_items, p.phi_kind, p.eps, zt, St);
  if (e != cudaSuccess) return MHLA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
}

}  // namespace

// d = 32 with an even number of adjacent heads reads out head pairs as 64-channel rows.
bool output_pairs_heads(const Problem& p) {
  return p.d == 32 && p.H % 2 == 0 && p.q.sh == 32 && p.o.sh == 32 && operand_tma_ok(p, p.q) &&
         operand_tma_ok(p, p.o);
}

int tc_run_output(const Problem& p, const void* St, const float* zt, void* stream) {
  auto* st = static_cast<const __nv_bfloat16*>(St);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.d == 64) return run_output<64, false>(p, st, zt, s);
  return output_pairs_heads(p) ? run_output<64, true>(p, st, zt, s) : run_output<32, false>(p, st, zt, s);
}

int read_and_clear_output_error(void* stream, uint32_t* flags) { return read_and_clear_word(g_out_error, stream, flags); }

MHLA_DEFINE_STALL_SETTER(set_stall_output)

}  // namespace mhla
