// tc_summary: the first step of the tensor-core path of the MHLA forward on
// sm_103a, [S_j | z_j] = phi(K_j)^T [V_j | 1] per (b, head group, block j)
// ([P2] "MHLA: Restoring Expressivity of Linear Attention via Token-Level
// Multi-Head", section 4 "Architecture": local key-value summaries; [P1]
// 171host.com/767426.html, section 7, MHLA.forward: kv = k^T v, k_sum).

// Every mbarrier wait is bounded (time and poll count); a wait that gives up
// raises a per-CTA abort flag so the other roles stop waiting too, sets bit 0 of
// this file's device error word, and the CTA drains its copies, releases tensor
// memory and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "mhla_internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"
#include "tma_host.h"

namespace mhla {

__device__ unsigned int g_sum_error = 0;

namespace {

using namespace ptx;
using namespace tc;

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag) {
  return wait_bounded_on(bar, parity, abort_flag, &g_sum_error);
}
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag) {
  return warp_wait_on(bar, parity, abort_flag, &g_sum_error);
}
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) { drain_wait_on(bar, parity, &g_sum_error); }

// ============================================================================
// tc_summary
// Work item = (b, j, head group) with the head group fastest, so the CTAs that
// fetch the other heads of the same tokens run side by side.
// ============================================================================
template <int D>
struct SumCfg {
  static constexpr int HP = 128 / D;                 // heads per work item
  static constexpr int C = 64;                       // tokens per stage
  static constexpr int ROWB = D * 2;                 // bytes per token row
  static constexpr int TILE = C * ROWB;              // one head's K or V chunk
  static constexpr int STAGE = (2 * HP + 1) * TILE;  // K tiles, V tiles, ones tile
  static constexpr int LOADB = 2 * HP * TILE;        // bytes TMA delivers per stage
  static constexpr int NS = D == 64 ? 5 : 6;
  static constexpr uint32_t SBO = 8 * ROWB;
  static constexpr uint32_t LAYOUT = D == 64 ? 2u : 4u;
  static constexpr int NMMA = 128 + 16;              // 128 value columns + z column block
  static constexpr int ACC_STRIDE = 256;             // TMEM columns between accumulators
  static constexpr int TMEM_COLS = 512;
  static constexpr int CTRL = 1024;
  static constexpr size_t SMEM = static_cast<size_t>(NS) * STAGE + CTRL + 1024;
};
constexpr int kTcThreads = 320;  // producer, MMA, 4 phi warps, 4 epilogue warps

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
  uint8_t* ctrl = smem + Cfg::NS * Cfg::STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* phid = full + Cfg::NS;
  uint64_t* empty = phid + Cfg::NS;
  uint64_t* tfull = empty + Cfg::NS;
  uint64_t* tempty = tfull + 2;
  uint64_t* fin = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 512);
  volatile uint32_t* abortf = tmem_slot + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::NS; ++s) {
      mbar_init(full + s, 1);
      mbar_init(phid + s, 128);
      mbar_init(empty + s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull + a, 1);
      mbar_init(tempty + a, 128);
    }
    mbar_init(fin, 1);
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
  // Constant ones operand of every stage: row t holds (1, 0, ..., 0), so the
  // MMA column that reads it sums phi(k) over the tokens: z_j.
  for (int idx = threadIdx.x; idx < Cfg::NS * Cfg::C * (D / 8); idx += kTcThreads) {
    const int s = idx / (Cfg::C * (D / 8));
    const int rem = idx % (Cfg::C * (D / 8));
    const int row = rem / (D / 8), phys = rem % (D / 8);
    const int logical = phys ^ swz<D>(row);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (logical == 0) v.x = 0x3F80u;   // bf16 1.0 in the low half
    *reinterpret_cast<uint4*>(stages + s * Cfg::STAGE + 2 * Cfg::HP * Cfg::TILE + row * Cfg::ROWB + phys * 16) = v;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int s = 0;
      uint32_t ph = 0;
      uint64_t fills = 0;
      bool ok = true;
      for (int64_t item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        const int32_t grp = static_cast<int32_t>(item % G);
        const int64_t rest = item / G;
        const int32_t j = static_cast<int32_t>(rest % g.M), b = static_cast<int32_t>(rest / g.M);
        for (int c = 0; c < g.chunks; ++c) {
          if (!wait_bounded(empty + s, ph ^ 1u, abortf)) { ok = false; break; }
          mbar_arrive_expect_tx(full + s, Cfg::LOADB);
          int32_t x, y, z;
          chunk_coords(g, j, c, b, x, y, z);
          uint8_t* st = stages + s * Cfg::STAGE;
#pragma unroll
          for (int hh = 0; hh < Cfg::HP; ++hh) {
            const int32_t h = grp * Cfg::HP + hh;   // h >= H reads zeros (out of bounds)
            tma_load_5d(st + hh * Cfg::TILE, &tm_k, full + s, 0, h, x, y, z, pol);
            tma_load_5d(st + (Cfg::HP + hh) * Cfg::TILE, &tm_v, full + s, 0, h, x, y, z, pol);
          }
          ++fills;
          if (++s == Cfg::NS) { s = 0; ph ^= 1u; }
        }
      }
      // Every fill must have landed before the CTA's shared memory goes away.
      for (int st = 0; st < Cfg::NS; ++st) {
        const uint64_t n = fills / Cfg::NS + (static_cast<uint64_t>(st) < fills % Cfg::NS ? 1 : 0);
        if (n > 0) drain_wait(full + st, static_cast<uint32_t>((n - 1) & 1));
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, Cfg::NMMA, true, true);
      int s = 0;
      uint32_t ph = 0, local = 0;
      bool ok = true;
      for (int64_t item = blockIdx.x; ok && item < n_items; item += gridDim.x, ++local) {
        const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
        if (!wait_bounded(tempty + acc, aph ^ 1u, abortf)) break;
        tc_fence_after();
        const uint32_t dt = tmem + acc * Cfg::ACC_STRIDE;
        for (int c = 0; c < g.chunks; ++c) {
          if (!wait_bounded(phid + s, ph, abortf)) { ok = false; break; }
          tc_fence_after();
          const uint32_t base = smem_u32(stages + s * Cfg::STAGE);
#pragma unroll
          for (int ks = 0; ks < Cfg::C / 16; ++ks) {
            const uint64_t a = smem_desc(base + ks * 2 * Cfg::SBO, Cfg::TILE, Cfg::SBO, Cfg::LAYOUT);
            const uint64_t bd =
                smem_desc(base + Cfg::HP * Cfg::TILE + ks * 2 * Cfg::SBO, Cfg::TILE, Cfg::SBO, Cfg::LAYOUT);
            mma_bf16(dt, a, bd, idesc, (c | ks) != 0 ? 1u : 0u);
          }
          mma_commit(empty + s);
          if (++s == Cfg::NS) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        mma_commit(tfull + acc);
      }
      mma_commit(fin);
      drain_wait(fin, 0);
    }
  } else if (warp < 6) {
    // ---------------------------------------------------------- phi on K
    const int rt = threadIdx.x - 64;
    const int hh = rt / D, u = rt % D;
    const int rg = u / (D / 8), p = u % (D / 8);
    uint8_t* head_tile = stages + hh * Cfg::TILE + rg * Cfg::ROWB + p * 16;
    const bool add_eps = phi_kind == MHLA_PHI_RELU_EPS;
    const __nv_bfloat162 eps2 = __float2bfloat162_rn(eps);
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int64_t item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      for (int c = 0; c < g.chunks; ++c) {
        if (!warp_wait(full + s, ph, abortf)) { ok = false; break; }
        uint8_t* base = head_tile + s * Cfg::STAGE;
#pragma unroll
        for (int m = 0; m < Cfg::C / 8; ++m) {
          uint4* ptr = reinterpret_cast<uint4*>(base + m * 8 * Cfg::ROWB);
          *ptr = phi8_packed(*ptr, add_eps, eps2);
        }
        fence_proxy_async_smem();
        mbar_arrive(phid + s);
        if (++s == Cfg::NS) { s = 0; ph ^= 1u; }
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int q4 = warp & 3;
    const int row = 32 * q4 + lane;          // TMEM lane = channel row of head hh
    const int hh = row / D, r = row % D;
    uint32_t local = 0;
    for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x, ++local) {
      const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
      if (!warp_wait(tfull + acc, aph, abortf)) break;
      tc_fence_after();
      const uint32_t tb = tmem + acc * Cfg::ACC_STRIDE + (static_cast<uint32_t>(32 * q4) << 16);
      uint32_t v0[32], v1[32], vz[16];
      tmem_ld_x32(tb + hh * D, v0);
      if (D == 64) tmem_ld_x32(tb + hh * D + 32, v1);
      tmem_ld_x16(tb + 128, vz);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(tempty + acc);
      const int32_t grp = static_cast<int32_t>(item % G);
      const int64_t rest = item / G;
      const int32_t j = static_cast<int32_t>(rest % g.M), b = static_cast<int32_t>(rest / g.M);
      const int32_t h = grp * Cfg::HP + hh;
      if (h < g.H) {
        // Sbuf is blocked by groups of 128 columns: column col of source block j
        // lives at ((col / 128) * M + j) * 128 + col % 128.  A row of D columns
        // starting at a multiple of D stays inside one group.
        const int64_t col = (static_cast<int64_t>(b) * g.H + h) * (D + 1) * D + r * D;
        const int64_t grow = (col >> 7) * g.M + j;
        uint4* drow = reinterpret_cast<uint4*>(Sbuf + grow * 128 + (col & 127));
        const uint64_t keep = policy_evict_last();
#pragma unroll
        for (int q = 0; q < 4; ++q)
          st_global_v4_hint(drow + q, make_uint4(pack_bf16(__uint_as_float(v0[8 * q]), __uint_as_float(v0[8 * q + 1])),
                               pack_bf16(__uint_as_float(v0[8 * q + 2]), __uint_as_float(v0[8 * q + 3])),
                               pack_bf16(__uint_as_float(v0[8 * q + 4]), __uint_as_float(v0[8 * q + 5])),
                               pack_bf16(__uint_as_float(v0[8 * q + 6]), __uint_as_float(v0[8 * q + 7]))), keep);
        if (D == 64) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            st_global_v4_hint(drow + 4 + q, make_uint4(pack_bf16(__uint_as_float(v1[8 * q]), __uint_as_float(v1[8 * q + 1])),
                                     pack_bf16(__uint_as_float(v1[8 * q + 2]), __uint_as_float(v1[8 * q + 3])),
                                     pack_bf16(__uint_as_float(v1[8 * q + 4]), __uint_as_float(v1[8 * q + 5])),
                                     pack_bf16(__uint_as_float(v1[8 * q + 6]), __uint_as_float(v1[8 * q + 7]))), keep);
        }
        const int64_t zcol = (static_cast<int64_t>(b) * g.H + h) * (D + 1) * D + D * D + r;
        Sbuf[((zcol >> 7) * g.M + j) * 128 + (zcol & 127)] = __float2bfloat16_rn(__uint_as_float(vz[0]));
      }
    }
  }
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
                           static_cast<int>(Cfg::SMEM)) != cudaSuccess)
    return MHLA_ERR_CUDA;
  const int per_sm = std::max(1, occupancy(tc_summary<D>, kTcThreads, Cfg::SMEM));
  const int grid = static_cast<int>(std::min<int64_t>(n_items, static_cast<int64_t>(sms) * per_sm));
  KernelTimer timer("tc_summary", stream);
  tc_summary<D><<<grid, kTcThreads, Cfg::SMEM, stream>>>(tk, tv, make_geom(p, c64), G, n_items, p.phi_kind, p.eps,
                                                         Sbuf, W, Wb, WbT, Mp, Mw, upb);
  return cudaGetLastError() == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
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

}  // namespace mhla
