// Tensor-core path of the MHLA forward on sm_103a: TMA-fed, tcgen05 MMAs with
// float32 accumulators in tensor memory, persistent warp-specialised CTAs.
//
// The three steps of the method ([P2] "MHLA: Restoring Expressivity of Linear
// Attention via Token-Level Multi-Head", section 4 "Architecture", "Multi-Head
// Mixing", "Token-Level Adaptivity"; [P1] 171host.com/767426.html, section 7,
// MHLA.forward):
//
//   tc_summary  per (b, head group, block j): [S_j | z_j] = phi(K_j)^T [V_j | 1]
//               (its prologue also rounds W to bf16 for the mixing GEMM)
//               K and V chunks of 64 tokens arrive by 5-D TMA (d, H, X, Y, B*T);
//               phi is applied in shared memory; 128/d heads share one
//               128 x (128+16) MMA whose diagonal d x d blocks are the S_j and
//               whose column 128 (a constant "ones" operand) is z_j.
//   tc_mix      S~ = W . S as one GEMM over the source blocks j:
//               D[i, col] = sum_j W[i][j] Sbuf[j][col], col = (b, h, row, c).
//   tc_output   per (b, h, block i), 128 tokens at a time:
//               o_t = phi(q_t) S~_i / (phi(q_t) . z~_i + eps); numerator and
//               denominator from one MMA (z~_i rides as two extra B columns),
//               the result scaled, rounded and stored by TMA in the input layout.
//
// Every mbarrier wait is bounded (time and poll count); a wait that gives up
// raises a per-CTA abort flag so the other roles stop waiting too, sets bit 0 of
// the device error word, and the CTA drains its copies, releases tensor memory
// and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "mhla_internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"
#include "tma_host.h"

namespace mhla {

__device__ unsigned int g_tc_error = 0;

namespace {

using namespace ptx;

using namespace tc;

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag) {
  return wait_bounded_on(bar, parity, abort_flag, &g_tc_error);
}
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag) {
  return warp_wait_on(bar, parity, abort_flag, &g_tc_error);
}
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) { drain_wait_on(bar, parity, &g_tc_error); }

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
           __nv_bfloat16* __restrict__ WbT, int64_t Mp) {
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
  // this kernel on the same stream).
  {
    const int64_t n = static_cast<int64_t>(g.M) * Mp;
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * kTcThreads + threadIdx.x; e < n;
         e += static_cast<int64_t>(gridDim.x) * kTcThreads) {
      const int64_t i = e / Mp, j = e % Mp;
      Wb[e] = __float2bfloat16_rn(j < g.M ? W[i * g.M + j] : 0.0f);
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
#pragma unroll
        for (int q = 0; q < 4; ++q)
          drow[q] = make_uint4(pack_bf16(__uint_as_float(v0[8 * q]), __uint_as_float(v0[8 * q + 1])),
                               pack_bf16(__uint_as_float(v0[8 * q + 2]), __uint_as_float(v0[8 * q + 3])),
                               pack_bf16(__uint_as_float(v0[8 * q + 4]), __uint_as_float(v0[8 * q + 5])),
                               pack_bf16(__uint_as_float(v0[8 * q + 6]), __uint_as_float(v0[8 * q + 7])));
        if (D == 64) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            drow[4 + q] = make_uint4(pack_bf16(__uint_as_float(v1[8 * q]), __uint_as_float(v1[8 * q + 1])),
                                     pack_bf16(__uint_as_float(v1[8 * q + 2]), __uint_as_float(v1[8 * q + 3])),
                                     pack_bf16(__uint_as_float(v1[8 * q + 4]), __uint_as_float(v1[8 * q + 5])),
                                     pack_bf16(__uint_as_float(v1[8 * q + 6]), __uint_as_float(v1[8 * q + 7])));
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

// ============================================================================
// tc_mix:  D[i, col] = sum_j W[i][j] * Sbuf[j][col]
// One tile = 128 query blocks i x 256 columns col = (b, h, row, c) of Sbuf; the
// tensor-memory row of query block i then holds S~_i (and z~_i) contiguously.
// ============================================================================
struct MixCfg {
  static constexpr int ROWS = 128;               // query blocks per tile (MMA M)
  static constexpr int COLS = 256;               // Sbuf columns per tile (MMA N)
  static constexpr int KC = 64;                  // source blocks j per stage
  static constexpr int A_BYTES = ROWS * KC * 2;  // W chunk, K-major
  static constexpr int B_BYTES = KC * COLS * 2;  // Sbuf chunk, four 64-column MN-major chunks
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int NS = 4;
  static constexpr int ACC_STRIDE = 256;
  static constexpr int TMEM_COLS = 512;
  static constexpr int CTRL = 1024;
  static constexpr size_t SMEM = static_cast<size_t>(NS) * STAGE + CTRL + 1024;
};
constexpr int kMixThreadsTC = 320;   // producer, MMA, two epilogue warpgroups taking alternate tiles

template <int D>
__global__ void __launch_bounds__(kMixThreadsTC, 1)
tc_mix(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_s, int32_t M,
       int64_t ncols, int32_t n_col_tiles, int32_t n_i_tiles, __nv_bfloat16* __restrict__ St,
       float* __restrict__ zt) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  uint8_t* stages = smem;
  uint8_t* ctrl = smem + MixCfg::NS * MixCfg::STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + MixCfg::NS;
  uint64_t* tfull = empty + MixCfg::NS;
  uint64_t* tempty = tfull + 2;
  uint64_t* fin = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 512);
  volatile uint32_t* abortf = tmem_slot + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n_tiles = static_cast<int64_t>(n_col_tiles) * n_i_tiles;
  const int nk = (M + MixCfg::KC - 1) / MixCfg::KC;
  if (threadIdx.x == 0) {
    for (int s = 0; s < MixCfg::NS; ++s) {
      mbar_init(full + s, 1);
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
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_s);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, MixCfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Tiles run query-tile fastest, so the query tiles that read the same Sbuf
  // columns run side by side and share them in L2.
  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_last();
      const uint64_t pol_s = policy_evict_first();
      int s = 0;
      uint32_t ph = 0;
      uint64_t fills = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
        const int32_t i0 = static_cast<int32_t>(t % n_i_tiles) * MixCfg::ROWS;
        const int32_t col0 = static_cast<int32_t>(t / n_i_tiles) * MixCfg::COLS;
        for (int kc = 0; kc < nk; ++kc) {
          if (!wait_bounded(empty + s, ph ^ 1u, abortf)) { ok = false; break; }
          mbar_arrive_expect_tx(full + s, MixCfg::STAGE);
          uint8_t* st = stages + s * MixCfg::STAGE;
          tma_load_2d(st, &tm_w, full + s, kc * MixCfg::KC, i0, pol_w);
#pragma unroll
          for (int a = 0; a < MixCfg::COLS / 64; ++a) {
            const int32_t col = col0 + 64 * a;                    // 64 columns inside one 128-column group
            tma_load_3d(st + MixCfg::A_BYTES + a * (MixCfg::KC * 128), &tm_s, full + s, col & 127,
                        kc * MixCfg::KC, col >> 7, pol_s);
          }
          ++fills;
          if (++s == MixCfg::NS) { s = 0; ph ^= 1u; }
        }
      }
      for (int st = 0; st < MixCfg::NS; ++st) {
        const uint64_t n = fills / MixCfg::NS + (static_cast<uint64_t>(st) < fills % MixCfg::NS ? 1 : 0);
        if (n > 0) drain_wait(full + st, static_cast<uint32_t>((n - 1) & 1));
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(MixCfg::ROWS, MixCfg::COLS, /*a K-major*/ false,
                                                /*b MN-major*/ true);
      int s = 0;
      uint32_t ph = 0, local = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; ok && t < n_tiles; t += gridDim.x, ++local) {
        const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
        if (!wait_bounded(tempty + acc, aph ^ 1u, abortf)) break;
        tc_fence_after();
        const uint32_t dt = tmem + acc * MixCfg::ACC_STRIDE;
        for (int kc = 0; kc < nk; ++kc) {
          if (!wait_bounded(full + s, ph, abortf)) { ok = false; break; }
          tc_fence_after();
          const uint32_t base = smem_u32(stages + s * MixCfg::STAGE);
#pragma unroll
          for (int ks = 0; ks < MixCfg::KC / 16; ++ks) {
            const uint64_t a = smem_desc(base + ks * 32, 16, 1024, 2);
            const uint64_t b = smem_desc(base + MixCfg::A_BYTES + ks * 2048, MixCfg::KC * 128, 1024, 2);
            mma_bf16(dt, a, b, idesc, (kc | ks) != 0 ? 1u : 0u);
          }
          mma_commit(empty + s);
          if (++s == MixCfg::NS) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        mma_commit(tfull + acc);
      }
      mma_commit(fin);
      drain_wait(fin, 0);
    }
  } else {
    // warpgroup wg (warps 2-5 or 6-9) drains accumulator wg: the tiles with local % 2 == wg
    constexpr int32_t PER_BH = (D + 1) * D;            // Sbuf columns of one (b, h): d rows of S, then z
    const int wg = (warp - 2) >> 2;
    const int q4 = warp & 3;
    const int row = 32 * q4 + lane;                    // query block within the tile
    uint32_t local = 0;
    for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x, ++local) {
      if (static_cast<int>(local & 1u) != wg) continue;
      const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
      if (!warp_wait(tfull + acc, aph, abortf)) break;
      tc_fence_after();
      const int32_t i = static_cast<int32_t>(t % n_i_tiles) * MixCfg::ROWS + row;
      const int32_t col0 = static_cast<int32_t>(t / n_i_tiles) * MixCfg::COLS;
      // column col0 + cc is (bh, rem) with rem = rr * D + c: one division per tile
      int32_t bh = col0 / PER_BH, rem = col0 - bh * PER_BH;
      const uint32_t tb = tmem + acc * MixCfg::ACC_STRIDE + (static_cast<uint32_t>(32 * q4) << 16);
#pragma unroll 1
      for (int cc = 0; cc < MixCfg::COLS; cc += 32) {
        uint32_t v[32];
        tmem_ld_x32(tb + cc, v);
        tmem_ld_wait();
        if (i < M && col0 + cc < ncols) {
          const int32_t rr = rem / D, c0 = rem % D;    // 32 columns of one row rr of one (b, h)
          const int64_t tile_id = static_cast<int64_t>(bh) * M + i;
          if (rr < D) {
            __nv_bfloat16* tile = St + tile_id * D * D + rr * D + c0;     // S~_i row-major
#pragma unroll
            for (int q = 0; q < 4; ++q)
              *reinterpret_cast<uint4*>(tile + q * 8) =
                  make_uint4(pack_bf16(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
                             pack_bf16(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                             pack_bf16(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                             pack_bf16(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
          } else {
            uint4* dst = reinterpret_cast<uint4*>(zt + tile_id * D + c0);
#pragma unroll
            for (int q = 0; q < 8; ++q) dst[q] = make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          }
        }
        rem += 32;
        if (rem >= PER_BH) { rem -= PER_BH; ++bh; }
      }
      tc_fence_before();
      mbar_arrive(tempty + acc);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, MixCfg::TMEM_COLS);
  }
}

// ============================================================================
// tc_mix_resident: the same GEMM for M <= 256 with all of W (bf16, <= 128 KB)
// resident in shared memory, computed transposed: D[col][i] = sum_j
// Sbuf[j][col] W[i][j].  One tile = 128 Sbuf columns (MMA M, the TMEM lanes) x
// all query blocks (MMA N <= 256): per 16 source blocks a single 128 x N x 16
// MMA, A = the Sbuf chunk as it landed (MN-major), B = W (K-major).  With the
// columns on TMEM lanes, the 32 lanes of an epilogue warp hold 32 consecutive
// columns of one query block, so each store writes 64 contiguous bytes of S~
// (or 128 of z~).  Two accumulator sets alternate between tiles; both
// epilogue warpgroups drain every tile, each half of the query blocks.
// ============================================================================
struct MixResCfg {
  static constexpr int COLS = 128;                // Sbuf columns per tile (MMA M)
  static constexpr int NMAX = 256;                // query blocks (MMA N, at most)
  static constexpr int KC = 64;                   // source blocks per stage
  static constexpr int W_CHUNK = NMAX * KC * 2;   // W rows i for 64 source blocks, K-major
  static constexpr int W_BYTES = 4 * W_CHUNK;     // up to 256 x 256
  static constexpr int STAGE = KC * COLS * 2;     // Sbuf chunk: two 64-column MN-major halves
  static constexpr int NS = 6;
  static constexpr int SET = NMAX;                // TMEM columns of one accumulator set
  static constexpr int TMEM_COLS = 512;
  static constexpr int CTRL = 1024;
  static constexpr size_t SMEM = static_cast<size_t>(W_BYTES) + static_cast<size_t>(NS) * STAGE + CTRL + 1024;
};

template <int D>
__global__ void __launch_bounds__(kMixThreadsTC, 1)
tc_mix_resident(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_s, int32_t M,
                int32_t NP, int64_t ncols, int32_t n_tiles, __nv_bfloat16* __restrict__ St, float* __restrict__ zt) {
  using Cfg = MixResCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  uint8_t* wres = smem;                                  // [k chunk] W rows i, K-major
  uint8_t* stages = smem + Cfg::W_BYTES;
  uint8_t* ctrl = stages + Cfg::NS * Cfg::STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + Cfg::NS;
  uint64_t* tfull = empty + Cfg::NS;
  uint64_t* tempty = tfull + 2;
  uint64_t* wfull = tempty + 2;
  uint64_t* fin = wfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 512);
  volatile uint32_t* abortf = tmem_slot + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = (M + Cfg::KC - 1) / Cfg::KC;           // 1..4 source chunks
  const uint32_t wchunk = static_cast<uint32_t>(NP) * Cfg::KC * 2;
  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::NS; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull + a, 1);
      mbar_init(tempty + a, 256);
    }
    mbar_init(wfull, 1);
    mbar_init(fin, 1);
    *abortf = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_s);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_last();
      const uint64_t pol_s = policy_evict_first();
      // all of W once: chunk kc holds rows i < NP (rows >= M read as zeros) of source blocks kc*64 ..
      mbar_arrive_expect_tx(wfull, static_cast<uint32_t>(nk) * wchunk);
      for (int kc = 0; kc < nk; ++kc) tma_load_2d(wres + kc * wchunk, &tm_w, wfull, kc * Cfg::KC, 0, pol_w);
      int s = 0;
      uint32_t ph = 0;
      uint64_t fills = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
        for (int kc = 0; kc < nk; ++kc) {
          if (!wait_bounded(empty + s, ph ^ 1u, abortf)) { ok = false; break; }
          mbar_arrive_expect_tx(full + s, Cfg::STAGE);
          uint8_t* st = stages + s * Cfg::STAGE;
          // one 128-column group of Sbuf, rows j contiguous; rows j >= M read as zeros
          tma_load_3d(st, &tm_s, full + s, 0, kc * Cfg::KC, static_cast<int32_t>(t), pol_s);
          tma_load_3d(st + Cfg::STAGE / 2, &tm_s, full + s, 64, kc * Cfg::KC, static_cast<int32_t>(t), pol_s);
          ++fills;
          if (++s == Cfg::NS) { s = 0; ph ^= 1u; }
        }
      }
      drain_wait(wfull, 0);
      for (int st = 0; st < Cfg::NS; ++st) {
        const uint64_t n = fills / Cfg::NS + (static_cast<uint64_t>(st) < fills % Cfg::NS ? 1 : 0);
        if (n > 0) drain_wait(full + st, static_cast<uint32_t>((n - 1) & 1));
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(Cfg::COLS, NP, /*a MN-major*/ true, /*b K-major*/ false);
      int s = 0;
      uint32_t ph = 0, local = 0;
      bool ok = wait_bounded(wfull, 0, abortf);
      tc_fence_after();
      const uint32_t wbase = smem_u32(wres);
      for (int64_t t = blockIdx.x; ok && t < n_tiles; t += gridDim.x, ++local) {
        const uint32_t set = local & 1u, sph = (local >> 1) & 1u;
        if (!wait_bounded(tempty + set, sph ^ 1u, abortf)) break;
        tc_fence_after();
        for (int kc = 0; kc < nk; ++kc) {
          if (!wait_bounded(full + s, ph, abortf)) { ok = false; break; }
          tc_fence_after();
          const uint32_t base = smem_u32(stages + s * Cfg::STAGE);
#pragma unroll
          for (int ks = 0; ks < Cfg::KC / 16; ++ks) {
            const uint64_t a = smem_desc(base + ks * 2048, Cfg::STAGE / 2, 1024, 2);
            const uint64_t b = smem_desc(wbase + kc * wchunk + ks * 32, 16, 1024, 2);
            mma_bf16(tmem + set * Cfg::SET, a, b, idesc, (kc | ks) != 0 ? 1u : 0u);
          }
          mma_commit(empty + s);
          if (++s == Cfg::NS) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        mma_commit(tfull + set);
      }
      mma_commit(fin);
      drain_wait(fin, 0);
    }
  } else {
    // warpgroup wg (warps 2-5 or 6-9) drains query blocks [128 wg, 128 wg + 128) of every tile
    constexpr int32_t PER_BH = (D + 1) * D;            // Sbuf columns of one (b, h): d rows of S, then z
    const int wg = (warp - 2) >> 2;
    const int q4 = warp & 3;
    const int i_lo = wg * 128, i_hi = min(M, i_lo + 128);
    uint32_t local = 0;
    for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x, ++local) {
      const uint32_t set = local & 1u, sph = (local >> 1) & 1u;
      if (!warp_wait(tfull + set, sph, abortf)) break;
      tc_fence_after();
      // this lane's column; 32-column runs never cross a row of S (d is a multiple of 32)
      const int64_t col = t * Cfg::COLS + 32 * q4 + lane;
      const bool live = col < ncols;
      const int64_t bh = col / PER_BH;
      const int32_t rem = static_cast<int32_t>(col - bh * PER_BH);
      const int32_t rr = rem / D, c = rem % D;
      const uint32_t tb = tmem + set * Cfg::SET + (static_cast<uint32_t>(32 * q4) << 16);
#pragma unroll 1
      for (int i0 = i_lo; i0 < i_hi; i0 += 32) {
        uint32_t v[32];
        tmem_ld_x32(tb + i0, v);
        tmem_ld_wait();
        if (live) {
          if (rr < D) {
            __nv_bfloat16* dst = St + (bh * M + i0) * (D * D) + rr * D + c;   // S~_i row-major
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (i0 + e < i_hi) dst[static_cast<int64_t>(e) * D * D] = __float2bfloat16_rn(__uint_as_float(v[e]));
          } else {
            float* dst = zt + (bh * M + i0) * D + c;
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (i0 + e < i_hi) dst[static_cast<int64_t>(e) * D] = __uint_as_float(v[e]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(tempty + set);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::TMEM_COLS);
  }
}

// ============================================================================
// tc_output
// Work item = (b, i, h) with the head fastest, so neighbouring CTAs read the
// neighbouring 128-byte head rows of the same tokens at about the same time.
// One MMA per 16 channels gives numerator and denominator together:
//   D[t][0..d)  = phi(q_t) S~_i                   (B columns 0..d-1: S~_i)
//   D[t][d]     = phi(q_t) . hi(z~_i)             (B column d:   z~_i rounded to bf16)
//   D[t][d+1]   = phi(q_t) . (z~_i - hi(z~_i))    (B column d+1: the rounding remainder)
// so the float32 denominator keeps about 16 bits more than a bf16 z~ would.
//
// The kernel streams q at the rate HBM allows only if enough loads are in
// flight: under full load a q chunk takes several microseconds to arrive, so
// shared memory goes almost entirely to q stages.  The output of a chunk is
// written back into its own q stage (the MMA has consumed it by then) and
// stored from there; the S~_i tiles, one per work item, have their own small
// ring fed by a second producer warp.
// ============================================================================
template <int D>
struct OutCfg {
  static constexpr int C = 128;                 // tokens per chunk = MMA M
  static constexpr int N = D + 16;              // S~ columns + the two z~ columns (+ 14 unused)
  static constexpr int ROWB = D * 2;
  static constexpr int QT = C * ROWB;           // q tile, then the output tile of the chunk
  static constexpr int KG = D / 8;              // core matrices along K (= rows of S~)
  static constexpr int B_SBO = KG * 128;        // bytes between column groups of 8
  static constexpr int ST_BYTES = D * D * 2;    // S~_i tile as written by tc_mix
  static constexpr int BOPS = (N / 8) * B_SBO;  // B operand: S~ columns and the z~ column groups
  static constexpr int ZRAW = D * 4;              // z~_i in float32, copied in after the operand
  static constexpr int BT = (BOPS + ZRAW + 1023) / 1024 * 1024;
  static constexpr int NQ = D == 64 ? 9 : 16;   // q stages
  static constexpr int NB = D == 64 ? 6 : 10;   // B slots (one per work item)
  static constexpr uint32_t A_SBO = 8 * ROWB;
  static constexpr uint32_t A_LAYOUT = D == 64 ? 2u : 4u;
  static constexpr int ACC_STRIDE = D == 64 ? 128 : 64;
  static constexpr int TMEM_COLS = 2 * ACC_STRIDE;
  static constexpr int CTRL = 1024;
  static constexpr size_t SMEM = static_cast<size_t>(NQ) * QT + static_cast<size_t>(NB) * BT + CTRL + 1024;
};
// q producer, MMA, 4 phi warps, two epilogue warpgroups taking alternate
// chunks, B producer, store issuer
constexpr int kOutThreadsTC = 512;
constexpr int kOutStoresInFlight = 3;   // TMA stores allowed to be reading shared memory at once

template <int D>
__global__ void __launch_bounds__(kOutThreadsTC, 1)
tc_output(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_o,
          const __grid_constant__ CUtensorMap tm_st, TcGeom g, int64_t n_items, int phi_kind, float eps,
          const float* __restrict__ zt) {
  using Cfg = OutCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  uint8_t* qst = smem;                                   // [NQ] q / output tiles
  uint8_t* bslot = smem + Cfg::NQ * Cfg::QT;             // [NB] S~ tiles + z~ columns
  uint8_t* ctrl = bslot + Cfg::NB * Cfg::BT;
  uint64_t* qfull = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* phid = qfull + Cfg::NQ;
  uint64_t* ostore = phid + Cfg::NQ;
  uint64_t* qempty = ostore + Cfg::NQ;
  uint64_t* bfull = qempty + Cfg::NQ;
  uint64_t* bempty = bfull + Cfg::NB;
  uint64_t* tfull = bempty + Cfg::NB;
  uint64_t* tempty = tfull + 2;
  uint64_t* fin = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 768);
  volatile uint32_t* abortf = tmem_slot + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::NQ; ++s) {
      mbar_init(qfull + s, 1);
      mbar_init(phid + s, 128);
      mbar_init(ostore + s, 128);
      mbar_init(qempty + s, 1);
    }
    for (int k = 0; k < Cfg::NB; ++k) {
      mbar_init(bfull + k, 1);
      mbar_init(bempty + k, 1);
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
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_o);
    prefetch_tmap(&tm_st);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------- q producer
    if (lane == 0) {
      const uint64_t pol_q = policy_evict_first();
      int s = 0;
      uint32_t ph = 0;
      uint64_t fills = 0;
      bool ok = true;
      for (int64_t item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        const int32_t h = static_cast<int32_t>(item % g.H);
        const int64_t rest = item / g.H;
        const int32_t i = static_cast<int32_t>(rest % g.M), b = static_cast<int32_t>(rest / g.M);
        for (int c = 0; c < g.chunks; ++c) {
          if (!wait_bounded(qempty + s, ph ^ 1u, abortf)) { ok = false; break; }
          mbar_arrive_expect_tx(qfull + s, Cfg::QT);
          int32_t x, y, z;
          chunk_coords(g, i, c, b, x, y, z);
          tma_load_5d(qst + s * Cfg::QT, &tm_q, qfull + s, 0, h, x, y, z, pol_q);
          ++fills;
          if (++s == Cfg::NQ) { s = 0; ph ^= 1u; }
        }
      }
      for (int st = 0; st < Cfg::NQ; ++st) {
        const uint64_t n = fills / Cfg::NQ + (static_cast<uint64_t>(st) < fills % Cfg::NQ ? 1 : 0);
        if (n > 0) drain_wait(qfull + st, static_cast<uint32_t>((n - 1) & 1));
      }
    }
  } else if (warp == 14) {
    // ------------------------------------------- B producer: one slot per item
    // Per item: S~_i (row-major in global memory) through a 4-D tensor view
    // (c % 8, r, c / 8, tile) whose box lands exactly in the unswizzled
    // MN-major core-matrix layout the MMA reads, and z~_i (float32) by a plain
    // bulk copy behind it.  Nothing here waits on a load, so the producer runs
    // up to NB items ahead.
    if (lane == 0) {
      const uint64_t pol_s = policy_evict_last();
      int kb = 0;
      uint32_t bph = 0;
      uint64_t fills = 0;
      for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int64_t h = item % g.H, rest = item / g.H;
        const int64_t i = rest % g.M, b = rest / g.M;
        const int64_t tile = (b * g.H + h) * g.M + i;
        if (!wait_bounded(bempty + kb, bph ^ 1u, abortf)) break;
        uint8_t* slot = bslot + kb * Cfg::BT;
        mbar_arrive_expect_tx(bfull + kb, Cfg::ST_BYTES + Cfg::ZRAW);
        tma_load_4d(slot, &tm_st, bfull + kb, 0, 0, 0, static_cast<int32_t>(tile), pol_s);
        bulk_load(slot + Cfg::BOPS, zt + tile * D, Cfg::ZRAW, bfull + kb, pol_s);
        ++fills;
        if (++kb == Cfg::NB) { kb = 0; bph ^= 1u; }
      }
      for (int st = 0; st < Cfg::NB; ++st) {
        const uint64_t n = fills / Cfg::NB + (static_cast<uint64_t>(st) < fills % Cfg::NB ? 1 : 0);
        if (n > 0) drain_wait(bfull + st, static_cast<uint32_t>((n - 1) & 1));
      }
    }
  } else if (warp == 15) {
    // ------------------------------------------- store issuer
    // Chunks in order: once the epilogue has written a chunk's output tile,
    // store it by TMA; a stage goes back to the q producer as soon as its
    // store has read it (up to kOutStoresInFlight stores read at once).
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      int pend[kOutStoresInFlight + 1];
      int npend = 0;
      bool ok = true;
      for (int64_t item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        const int32_t h = static_cast<int32_t>(item % g.H);
        const int64_t rest = item / g.H;
        const int32_t i = static_cast<int32_t>(rest % g.M), b = static_cast<int32_t>(rest / g.M);
        for (int c = 0; c < g.chunks; ++c) {
          if (!wait_bounded(ostore + s, ph, abortf)) { ok = false; break; }
          int32_t x, y, z;
          chunk_coords(g, i, c, b, x, y, z);
          tma_store_5d(&tm_o, qst + s * Cfg::QT, 0, h, x, y, z);
          bulk_commit_group();
          pend[npend++] = s;
          if (npend > kOutStoresInFlight) {
            bulk_wait_group_read<kOutStoresInFlight>();   // the oldest store has read its tile
            mbar_arrive(qempty + pend[0]);
#pragma unroll
            for (int e = 0; e < kOutStoresInFlight; ++e) pend[e] = pend[e + 1];
            --npend;
          }
          if (++s == Cfg::NQ) { s = 0; ph ^= 1u; }
        }
      }
      bulk_wait_group0();
    }
  } else if (warp == 1) {
    // ------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, Cfg::N, /*a K-major*/ false, /*b MN-major*/ true);
      int s = 0, kb = 0;
      uint32_t ph = 0, cnt = 0, bph = 0;
      bool ok = true;
      for (int64_t item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        // the slot of this item: S~ copy landed and z~ columns written
        if (!wait_bounded(bfull + kb, bph, abortf)) break;
        const uint32_t bbase = smem_u32(bslot + kb * Cfg::BT);
        for (int c = 0; c < g.chunks; ++c, ++cnt) {
          const uint32_t acc = cnt & 1u, aph = (cnt >> 1) & 1u;
          if (!wait_bounded(tempty + acc, aph ^ 1u, abortf)) { ok = false; break; }
          if (!wait_bounded(phid + s, ph, abortf)) { ok = false; break; }
          tc_fence_after();
          const uint32_t base = smem_u32(qst + s * Cfg::QT);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint64_t a = smem_desc(base + ks * 32, 16, Cfg::A_SBO, Cfg::A_LAYOUT);
            const uint64_t b = smem_desc(bbase + ks * 256, 128, Cfg::B_SBO, 0);
            mma_bf16(tmem + acc * Cfg::ACC_STRIDE, a, b, idesc, ks != 0 ? 1u : 0u);
          }
          mma_commit(tfull + acc);
          if (++s == Cfg::NQ) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        mma_commit(bempty + kb);              // slot reusable once this item's MMAs are done
        if (++kb == Cfg::NB) { kb = 0; bph ^= 1u; }
      }
      mma_commit(fin);
      drain_wait(fin, 0);
    }
  } else if (warp < 6) {
    // ------------------------------------------- phi on q; the z~ columns of B
    constexpr int CPR = D / 8;            // 16-byte chunks per row
    constexpr int RP = 128 / CPR;         // rows covered per pass
    const int rt = threadIdx.x - 64;
    const int rg = rt / CPR, p = rt % CPR;
    const bool add_eps = phi_kind == MHLA_PHI_RELU_EPS;
    const __nv_bfloat162 eps2 = __float2bfloat162_rn(eps);
    // thread rt < D owns row rt of z~_i: column D of B holds hi, column D+1 lo
    const int zoff = (D / 8) * Cfg::B_SBO + (rt >> 3) * 128 + (rt & 7) * 16;
    int s = 0, kb = 0;
    uint32_t ph = 0, bph = 0;
    bool ok = true;
    for (int64_t item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      // the item's slot: S~_i and the float32 z~_i have landed (the producer runs ahead)
      if (!warp_wait(bfull + kb, bph, abortf)) break;
      if (rt < D) {
        uint8_t* slot = bslot + kb * Cfg::BT;
        const float zv = *reinterpret_cast<const float*>(slot + Cfg::BOPS + rt * 4);
        const __nv_bfloat16 hi = __float2bfloat16_rn(zv);
        const __nv_bfloat16 lo = __float2bfloat16_rn(zv - __bfloat162float(hi));
        *reinterpret_cast<uint32_t*>(slot + zoff) =
            static_cast<uint32_t>(__bfloat16_as_ushort(hi)) | (static_cast<uint32_t>(__bfloat16_as_ushort(lo)) << 16);
      }
      if (++kb == Cfg::NB) { kb = 0; bph ^= 1u; }
      for (int c = 0; c < g.chunks; ++c) {
        if (!warp_wait(qfull + s, ph, abortf)) { ok = false; break; }
        uint8_t* tile = qst + s * Cfg::QT;
#pragma unroll
        for (int m = 0; m < Cfg::C / RP; ++m) {
          uint4* ptr = reinterpret_cast<uint4*>(tile + (rg + RP * m) * Cfg::ROWB + p * 16);
          *ptr = phi8_packed(*ptr, add_eps, eps2);
        }
        // also publishes this item's z~ columns to the MMA (first chunk)
        fence_proxy_async_smem();
        mbar_arrive(phid + s);
        if (++s == Cfg::NQ) { s = 0; ph ^= 1u; }
      }
    }
  } else {
    // ------------------------------------------- epilogue: scale and write back
    // Warpgroup wg (warps 6-9 or 10-13) takes the chunks with cnt % 2 == wg, which
    // are exactly the chunks accumulated in TMEM accumulator wg.
    const int wg = (warp - 6) >> 2;
    const int q4 = warp & 3;
    const int row = 32 * q4 + lane;      // token row of the chunk
    int s = 0;
    uint32_t ph = 0, cnt = 0;
    bool ok = true;
    for (int64_t item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      for (int c = 0; c < g.chunks; ++c, ++cnt) {
        const int cs = s;
        if (++s == Cfg::NQ) { s = 0; ph ^= 1u; }
        if (static_cast<int>(cnt & 1u) != wg) continue;
        const uint32_t acc = wg, aph = (cnt >> 1) & 1u;
        if (!warp_wait(tfull + acc, aph, abortf)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tb = tmem + acc * Cfg::ACC_STRIDE + (static_cast<uint32_t>(32 * q4) << 16);
        uint32_t v0[32], v1[32], vz[16];
        tmem_ld_x32(tb, v0);
        if (D == 64) tmem_ld_x32(tb + 32, v1);
        tmem_ld_x16(tb + D, vz);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(tempty + acc);
        const float inv = 1.0f / (__uint_as_float(vz[0]) + __uint_as_float(vz[1]) + eps);
        // the MMA has finished reading the q tile: the output row goes in its place
        uint8_t* orow = qst + cs * Cfg::QT + row * Cfg::ROWB;
#pragma unroll
        for (int q = 0; q < D / 8; ++q) {
          const uint32_t* src = (q < 4) ? (v0 + 8 * q) : (v1 + 8 * (q - 4));
          const uint4 packed = make_uint4(
              pack_bf16(__uint_as_float(src[0]) * inv, __uint_as_float(src[1]) * inv),
              pack_bf16(__uint_as_float(src[2]) * inv, __uint_as_float(src[3]) * inv),
              pack_bf16(__uint_as_float(src[4]) * inv, __uint_as_float(src[5]) * inv),
              pack_bf16(__uint_as_float(src[6]) * inv, __uint_as_float(src[7]) * inv));
          *reinterpret_cast<uint4*>(orow + ((q ^ swz<D>(row)) * 16)) = packed;
        }
        fence_proxy_async_smem();
        mbar_arrive(ostore + cs);
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

// ----------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool encode(CUtensorMap* m, int rank, void* base, const cuuint64_t* dims, const cuuint64_t* strides_bytes,
            const cuuint32_t* box, CUtensorMapSwizzle swz, CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return fn(m, dt, static_cast<cuuint32_t>(rank), base, dims, strides_bytes, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct TcLayout {
  size_t wb_off, sbuf_off, st_off, zt_off, total;
  int64_t Mp, ncols, ngroups;
};

TcLayout tc_layout(const Problem& p) {
  TcLayout L;
  L.Mp = (p.M + 7) / 8 * 8;
  L.ncols = p.BH() * (p.d + 1) * p.d;
  L.ngroups = (L.ncols + 127) / 128;                    // Sbuf column groups of 128
  size_t off = 0;
  L.wb_off = off;
  off += align_up(static_cast<size_t>(p.M) * L.Mp * 2);
  L.sbuf_off = off;
  off += align_up(static_cast<size_t>(p.M) * L.ngroups * 128 * 2);
  L.st_off = off;
  off += align_up(static_cast<size_t>(p.BH()) * p.M * p.d * p.d * 2);
  L.zt_off = off;
  off += align_up(static_cast<size_t>(p.BH()) * p.M * p.d * 4);
  L.total = off;
  return L;
}

int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

template <typename K>
int occupancy(K kernel, int threads, size_t smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess) return 0;
  return n;
}

template <int D>
int run_summary(const Problem& p, const float* W, __nv_bfloat16* Wb, __nv_bfloat16* WbT, int64_t Mp,
                __nv_bfloat16* Sbuf, cudaStream_t stream) {
  using Cfg = SumCfg<D>;
  const int sms = device_sms();
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
                                                         Sbuf, W, Wb, WbT, Mp);
  return cudaGetLastError() == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
}

// D[i, col] = sum_j Wm[i][j] Sbuf[j][col] for the ncols = BH (d + 1) d columns:
// S~ (row-major [BH][M][d][d]) and z~ (float32 [BH][M][d]).
template <int D>
int run_mix(const Problem& p, const __nv_bfloat16* Wm, int64_t Mp, const __nv_bfloat16* Sbuf, __nv_bfloat16* St,
            float* zt, cudaStream_t stream) {
  const int sms = device_sms();
  if (sms <= 0) return MHLA_ERR_CUDA;
  const int64_t ncols = p.BH() * (p.d + 1) * p.d;
  const int64_t ngroups = (ncols + 127) / 128;
  // Sbuf as (128 columns, M source blocks, G groups)
  const cuuint64_t sdims[3] = {128u, static_cast<cuuint64_t>(p.M), static_cast<cuuint64_t>(ngroups)};
  const cuuint64_t sstrides[2] = {256u, static_cast<cuuint64_t>(p.M * 256)};
  const cuuint64_t wdims[2] = {static_cast<cuuint64_t>(p.M), static_cast<cuuint64_t>(p.M)};
  const cuuint64_t wstrides[1] = {static_cast<cuuint64_t>(Mp * 2)};
  void* wptr = const_cast<__nv_bfloat16*>(Wm);
  void* sptr = const_cast<__nv_bfloat16*>(Sbuf);
  if (p.M <= 256) {   // all of W in shared memory
    CUtensorMap tw, ts;
    const int32_t NP = static_cast<int32_t>((p.M + 15) / 16 * 16);   // MMA N: query blocks rounded up to 16
    const cuuint32_t wbox[2] = {static_cast<cuuint32_t>(MixResCfg::KC), static_cast<cuuint32_t>(NP)};
    const cuuint32_t sbox[3] = {64u, static_cast<cuuint32_t>(MixResCfg::KC), 1u};
    if (!encode(&tw, 2, wptr, wdims, wstrides, wbox, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode(&ts, 3, sptr, sdims, sstrides, sbox, CU_TENSOR_MAP_SWIZZLE_128B))
      return MHLA_ERR_CUDA;
    const int32_t n_tiles = static_cast<int32_t>((ncols + MixResCfg::COLS - 1) / MixResCfg::COLS);
    if (cudaFuncSetAttribute(tc_mix_resident<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(MixResCfg::SMEM)) != cudaSuccess)
      return MHLA_ERR_CUDA;
    const int grid = static_cast<int>(std::min<int64_t>(n_tiles, sms));
    KernelTimer timer("tc_mix", stream);
    tc_mix_resident<D><<<grid, kMixThreadsTC, MixResCfg::SMEM, stream>>>(tw, ts, static_cast<int32_t>(p.M), NP,
                                                                          ncols, n_tiles, St, zt);
    return cudaGetLastError() == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
  }
  CUtensorMap tw, ts;
  const cuuint32_t wbox[2] = {static_cast<cuuint32_t>(MixCfg::KC), static_cast<cuuint32_t>(MixCfg::ROWS)};
  const cuuint32_t sbox[3] = {64u, static_cast<cuuint32_t>(MixCfg::KC), 1u};
  if (!encode(&tw, 2, wptr, wdims, wstrides, wbox, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode(&ts, 3, sptr, sdims, sstrides, sbox, CU_TENSOR_MAP_SWIZZLE_128B))
    return MHLA_ERR_CUDA;
  const int32_t n_col_tiles = static_cast<int32_t>((ncols + MixCfg::COLS - 1) / MixCfg::COLS);
  const int32_t n_i_tiles = static_cast<int32_t>((p.M + MixCfg::ROWS - 1) / MixCfg::ROWS);
  if (cudaFuncSetAttribute(tc_mix<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(MixCfg::SMEM)) !=
      cudaSuccess)
    return MHLA_ERR_CUDA;
  const int64_t n_tiles = static_cast<int64_t>(n_col_tiles) * n_i_tiles;
  const int grid = static_cast<int>(std::min<int64_t>(n_tiles, sms));
  KernelTimer timer("tc_mix", stream);
  tc_mix<D><<<grid, kMixThreadsTC, MixCfg::SMEM, stream>>>(tw, ts, static_cast<int32_t>(p.M), ncols, n_col_tiles,
                                                            n_i_tiles, St, zt);
  return cudaGetLastError() == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
}

template <int D>
int run_output(const Problem& p, const __nv_bfloat16* St, const float* zt, cudaStream_t stream) {
  using Cfg = OutCfg<D>;
  const int sms = device_sms();
  if (sms <= 0) return MHLA_ERR_CUDA;
  ChunkPlan c128;
  if (!chunk_plan(p, 128, &c128)) return MHLA_ERR_UNSUPPORTED;
  CUtensorMap tq, to;
  if (!operand_map(p, p.q, c128.box_y, c128.box_t, &tq) || !operand_map(p, p.o, c128.box_y, c128.box_t, &to))
    return MHLA_ERR_CUDA;
  // S~ tiles (row-major [BH*M][d][d]) seen as (c % 8, r, c / 8, tile): a
  // (8, d, d/8, 1) box lands as 16-byte rows of 8 columns, d rows per column
  // group: the unswizzled MN-major operand layout.
  CUtensorMap tst;
  {
    const cuuint64_t dims[4] = {8u, static_cast<cuuint64_t>(p.d), static_cast<cuuint64_t>(p.d / 8),
                                static_cast<cuuint64_t>(p.BH() * p.M)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(p.d * 2), 16u, static_cast<cuuint64_t>(p.d * p.d * 2)};
    const cuuint32_t box[4] = {8u, static_cast<cuuint32_t>(p.d), static_cast<cuuint32_t>(p.d / 8), 1u};
    if (!encode(&tst, 4, const_cast<__nv_bfloat16*>(St), dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE))
      return MHLA_ERR_CUDA;
  }
  const int64_t n_items = p.BH() * p.M;
  if (cudaFuncSetAttribute(tc_output<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(Cfg::SMEM)) !=
      cudaSuccess)
    return MHLA_ERR_CUDA;
  const int per_sm = std::max(1, std::min(occupancy(tc_output<D>, kOutThreadsTC, Cfg::SMEM), 512 / Cfg::TMEM_COLS));
  const int grid = static_cast<int>(std::min<int64_t>(n_items, static_cast<int64_t>(sms) * per_sm));
  KernelTimer timer("tc_output", stream);
  tc_output<D><<<grid, kOutThreadsTC, Cfg::SMEM, stream>>>(tq, to, tst, make_geom(p, c128), n_items, p.phi_kind, p.eps,
                                                            zt);
  return cudaGetLastError() == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
}

template <int D>
int launch_tc_d(const Problem& p, const float* W, void* workspace, cudaStream_t stream) {
  const TcLayout L = tc_layout(p);
  char* ws = static_cast<char*>(workspace);
  __nv_bfloat16* Wb = reinterpret_cast<__nv_bfloat16*>(ws + L.wb_off);
  __nv_bfloat16* Sbuf = reinterpret_cast<__nv_bfloat16*>(ws + L.sbuf_off);
  __nv_bfloat16* St = reinterpret_cast<__nv_bfloat16*>(ws + L.st_off);
  float* zt = reinterpret_cast<float*>(ws + L.zt_off);
  int rc = run_summary<D>(p, W, Wb, nullptr, L.Mp, Sbuf, stream);
  if (rc == MHLA_OK) rc = run_mix<D>(p, Wb, L.Mp, Sbuf, St, zt, stream);
  if (rc == MHLA_OK) rc = run_output<D>(p, St, zt, stream);
  return rc;
}

}  // namespace

bool encode_tensor_map(CUtensorMap* m, int rank, void* base, const cuuint64_t* dims,
                       const cuuint64_t* strides_bytes, const cuuint32_t* box, CUtensorMapSwizzle swz) {
  return encode(m, rank, base, dims, strides_bytes, box, swz);
}

int device_sm_count() { return device_sms(); }

int tc_run_summary(const Problem& p, const float* W, void* Wb, void* WbT, int64_t Mp, void* Sbuf, void* stream) {
  auto* wb = static_cast<__nv_bfloat16*>(Wb);
  auto* wbt = static_cast<__nv_bfloat16*>(WbT);
  auto* sb = static_cast<__nv_bfloat16*>(Sbuf);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return p.d == 64 ? run_summary<64>(p, W, wb, wbt, Mp, sb, s) : run_summary<32>(p, W, wb, wbt, Mp, sb, s);
}

int tc_run_mix(const Problem& p, const void* Wm, int64_t Mp, const void* Sbuf, void* St, float* zt, void* stream) {
  auto* wm = static_cast<const __nv_bfloat16*>(Wm);
  auto* sb = static_cast<const __nv_bfloat16*>(Sbuf);
  auto* st = static_cast<__nv_bfloat16*>(St);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return p.d == 64 ? run_mix<64>(p, wm, Mp, sb, st, zt, s) : run_mix<32>(p, wm, Mp, sb, st, zt, s);
}

bool tc_eligible(const Problem& p) {
  if (p.dtype != MHLA_BF16) return false;
  if (p.d != 32 && p.d != 64) return false;
  if (p.B < 1 || p.H < 1) return false;
  ChunkPlan cp;
  if (!chunk_plan(p, 64, &cp) || !chunk_plan(p, 128, &cp)) return false;
  for (const Operand* o : {&p.q, &p.k, &p.v, &p.o})
    if (!operand_tma_ok(p, *o)) return false;
  const int64_t lim32 = int64_t{1} << 31;
  const int64_t ncols = p.BH() * (p.d + 1) * p.d;
  if (p.BH() * p.M * p.d >= lim32 || ncols >= lim32 || p.M >= (int64_t{1} << 16)) return false;
  if (p.X >= lim32 || p.Y >= lim32 || p.B * p.T >= lim32 || p.H >= lim32) return false;
  if (p.B * ((p.H + 1) / 2) * p.M >= lim32) return false;
  return true;
}

size_t tc_workspace_bytes(const Problem& p) { return tc_layout(p).total; }

int launch_tc(const Problem& p, const float* W, void* workspace, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.d == 64) return launch_tc_d<64>(p, W, workspace, s);
  return launch_tc_d<32>(p, W, workspace, s);
}

int read_and_clear_device_error(void* stream, uint32_t* flags) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int host = 0;
  if (cudaMemcpyFromSymbolAsync(&host, g_tc_error, sizeof(host), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MHLA_ERR_CUDA;
  const unsigned int zero = 0;
  if (cudaMemcpyToSymbolAsync(g_tc_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return MHLA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MHLA_ERR_CUDA;
  *flags = host;
  return host ? MHLA_ERR_TIMEOUT : MHLA_OK;
}

}  // namespace mhla
