// Tensor-core path of the MHLA forward on sm_103a: TMA-fed, tcgen05 MMAs with
// float32 accumulators in tensor memory, persistent warp-specialised CTAs.
//
// The three steps of the method ([P2] "MHLA: Restoring Expressivity of Linear
// Attention via Token-Level Multi-Head", section 4 "Architecture", "Multi-Head
// Mixing", "Token-Level Adaptivity"; [P1] 171host.com/767426.html, section 7,
// MHLA.forward):
//
//   tc_summary  per (b, head group, block j): [S_j | z_j] = phi(K_j)^T [V_j | 1]
//               K and V chunks of 64 tokens arrive by 5-D TMA (d, H, X, Y, B*T);
//               phi is applied in shared memory; 128/d heads share one
//               128 x (128+16) MMA whose diagonal d x d blocks are the S_j and
//               whose column 128 (a constant "ones" operand) is z_j.
//   tc_mix      S~ = W . S as one GEMM over the source blocks j:
//               D[col, i] = sum_j Sbuf[j][col] W[i][j], col = (b, h, row, c).
//   tc_output   per (b, h, block i), 128 tokens at a time:
//               o_t = phi(q_t) S~_i / (phi(q_t) . z~_i + eps); the numerator on
//               the tensor core, the denominator in float32 on CUDA cores while
//               phi is applied, the result stored by TMA in the input layout.
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

namespace mhla {

__device__ unsigned int g_tc_error = 0;

namespace {

using namespace ptx;

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr uint32_t kWaitLimitPolls = 1u << 28;
constexpr uint64_t kDrainLimitNs = 50000000ull;   // 50 ms for copies already in flight

__device__ __noinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1; it < kWaitLimitPolls; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > kWaitLimitNs) break;
    }
  }
  *abort_flag = 1u;
  atomicOr(&g_tc_error, 1u);
  return false;
}

// Every lane waits, then the warp agrees: warp-collective instructions that
// follow (shuffles, tcgen05.ld) run either on all lanes or on none.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag) {
  const bool ok = wait_bounded(bar, parity, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// Wait for a phase that must already be under way (copies or MMAs in flight),
// without consulting the abort flag.
__device__ __noinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 0; it < kWaitLimitPolls; ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 63u) == 63u && globaltimer() - t0 > kDrainLimitNs) {
      atomicOr(&g_tc_error, 2u);
      return;
    }
  }
}

// Token-grid geometry of one launch (all int32: checked on the host).
struct TcGeom {
  int32_t M, nbx, nby;     // block grid, x fastest
  int32_t bx, by, bt, T;   // block extents; frames per batch image (1 for 2-D)
  int32_t box_y, box_t;    // TMA box of one chunk along y and t (x: whole block rows)
  int32_t nyc;             // chunks stacked along y inside one frame of a block
  int32_t chunks;          // chunks per block
  int32_t H, B;
};

// Coordinates (x, y, z = b*T + t) of chunk c of block j of batch b.
__device__ __forceinline__ void chunk_coords(const TcGeom& g, int32_t j, int32_t c, int32_t b, int32_t& x,
                                             int32_t& y, int32_t& z) {
  const int32_t jx = j % g.nbx, jr = j / g.nbx;
  const int32_t jy = jr % g.nby, jt = jr / g.nby;
  x = jx * g.bx;
  y = jy * g.by + (c % g.nyc) * g.box_y;
  z = b * g.T + jt * g.bt + (c / g.nyc) * g.box_t;
}

// phi on eight bf16 values in place; returns the float32 values for callers
// that need them (ReLU is exact in bf16; the + eps variant rounds once).
__device__ __forceinline__ uint4 phi8(uint4 raw, int phi_kind, float eps, float (&f)[8]) {
  const float add = phi_kind == MHLA_PHI_RELU_EPS ? eps : 0.0f;
  __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&raw);
  uint4 out;
  __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&out);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 v = __bfloat1622float2(h2[e]);
    const float a = fmaxf(v.x, 0.0f) + add, b = fmaxf(v.y, 0.0f) + add;
    f[2 * e] = a;
    f[2 * e + 1] = b;
    o2[e] = __floats2bfloat162_rn(a, b);
  }
  return out;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// 16-byte chunk position inside a swizzled row: 128-byte swizzle for d = 64
// (row r XORs chunk bits with r mod 8), 64-byte swizzle for d = 32.
template <int D>
__device__ __forceinline__ int swz(int row) {
  return D == 64 ? (row & 7) : ((row >> 1) & 3);
}

// ============================================================================
// tc_summary
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
           int32_t G, int64_t n_items, int64_t ncols, int phi_kind, float eps,
           __nv_bfloat16* __restrict__ Sbuf) {
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
        const int32_t j = static_cast<int32_t>(item % g.M);
        const int64_t rest = item / g.M;
        const int32_t grp = static_cast<int32_t>(rest % G), b = static_cast<int32_t>(rest / G);
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
          float f[8];
          *ptr = phi8(*ptr, phi_kind, eps, f);
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
      const int32_t j = static_cast<int32_t>(item % g.M);
      const int64_t rest = item / g.M;
      const int32_t grp = static_cast<int32_t>(rest % G), b = static_cast<int32_t>(rest / G);
      const int32_t h = grp * Cfg::HP + hh;
      if (h < g.H) {
        __nv_bfloat16* dst = Sbuf + static_cast<int64_t>(j) * ncols +
                             (static_cast<int64_t>(b) * g.H + h) * (D + 1) * D;
        uint4* drow = reinterpret_cast<uint4*>(dst + r * D);
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
        dst[D * D + r] = __float2bfloat16_rn(__uint_as_float(vz[0]));
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
// tc_mix:  D[col, i] = sum_j Sbuf[j][col] * W[i][j]
// ============================================================================
struct MixCfg {
  static constexpr int COLS = 128;     // GEMM M: Sbuf columns per tile
  static constexpr int KC = 64;        // source blocks j per stage
  static constexpr int A_BYTES = COLS * KC * 2;   // two 64-column MN-major chunks
  static constexpr int NS = 4;
  static constexpr int CTRL = 1024;
};
constexpr int kMixThreadsTC = 192;   // producer, MMA, 4 epilogue warps

__global__ void __launch_bounds__(kMixThreadsTC, 1)
tc_mix(const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_w, int32_t M, int32_t N,
       int32_t stage_bytes, int32_t tmem_cols, int32_t acc_stride, int64_t ncols, int32_t n_col_tiles,
       int32_t n_i_tiles, int32_t d, __nv_bfloat16* __restrict__ St, float* __restrict__ zt) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  uint8_t* stages = smem;
  uint8_t* ctrl = smem + MixCfg::NS * stage_bytes;
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
    prefetch_tmap(&tm_s);
    prefetch_tmap(&tm_w);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, static_cast<uint32_t>(tmem_cols));
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_s = policy_evict_first();
      const uint64_t pol_w = policy_evict_last();
      int s = 0;
      uint32_t ph = 0;
      uint64_t fills = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
        const int32_t col0 = static_cast<int32_t>(t % n_col_tiles) * MixCfg::COLS;
        const int32_t i0 = static_cast<int32_t>(t / n_col_tiles) * 256;
        for (int kc = 0; kc < nk; ++kc) {
          if (!wait_bounded(empty + s, ph ^ 1u, abortf)) { ok = false; break; }
          mbar_arrive_expect_tx(full + s, static_cast<uint32_t>(MixCfg::A_BYTES + N * 128));
          uint8_t* st = stages + s * stage_bytes;
          tma_load_2d(st, &tm_s, full + s, col0, kc * MixCfg::KC, pol_s);
          tma_load_2d(st + MixCfg::A_BYTES / 2, &tm_s, full + s, col0 + 64, kc * MixCfg::KC, pol_s);
          tma_load_2d(st + MixCfg::A_BYTES, &tm_w, full + s, kc * MixCfg::KC, i0, pol_w);
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
      const uint32_t idesc = idesc_bf16_f32(128, N, /*a MN-major*/ true, /*b K-major*/ false);
      int s = 0;
      uint32_t ph = 0, local = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; ok && t < n_tiles; t += gridDim.x, ++local) {
        const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
        if (!wait_bounded(tempty + acc, aph ^ 1u, abortf)) break;
        tc_fence_after();
        const uint32_t dt = tmem + acc * static_cast<uint32_t>(acc_stride);
        for (int kc = 0; kc < nk; ++kc) {
          if (!wait_bounded(full + s, ph, abortf)) { ok = false; break; }
          tc_fence_after();
          const uint32_t base = smem_u32(stages + s * stage_bytes);
#pragma unroll
          for (int ks = 0; ks < MixCfg::KC / 16; ++ks) {
            const uint64_t a = smem_desc(base + ks * 2048, MixCfg::A_BYTES / 2, 1024, 2);
            const uint64_t b = smem_desc(base + MixCfg::A_BYTES + ks * 32, 16, 1024, 2);
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
    const int q4 = warp & 3;
    const int row = 32 * q4 + lane;
    const int64_t per_bh = static_cast<int64_t>(d + 1) * d;
    uint32_t local = 0;
    for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x, ++local) {
      const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
      if (!warp_wait(tfull + acc, aph, abortf)) break;
      tc_fence_after();
      const int64_t col = static_cast<int64_t>(t % n_col_tiles) * MixCfg::COLS + row;
      const int32_t i0 = static_cast<int32_t>(t / n_col_tiles) * 256;
      const bool live = col < ncols;
      const int64_t bh = col / per_bh, rem = col % per_bh;
      const int rr = static_cast<int>(rem / d), c = static_cast<int>(rem % d);
      const uint32_t tb = tmem + acc * static_cast<uint32_t>(acc_stride) + (static_cast<uint32_t>(32 * q4) << 16);
      for (int cc = 0; cc < N; cc += 32) {
        uint32_t v[32];
        if (N - cc >= 32) {
          tmem_ld_x32(tb + cc, v);
        } else {
          uint32_t h16[16];
          tmem_ld_x16(tb + cc, h16);
#pragma unroll
          for (int u = 0; u < 16; ++u) v[u] = h16[u];
#pragma unroll
          for (int u = 16; u < 32; ++u) v[u] = 0u;
        }
        tmem_ld_wait();
        if (live) {
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            const int32_t i = i0 + cc + u;
            if (cc + u < N && i < M) {
              const float val = __uint_as_float(v[u]);
              if (rr < d)
                St[((bh * M + i) * d + rr) * d + c] = __float2bfloat16_rn(val);
              else
                zt[(bh * M + i) * d + c] = val;
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(tempty + acc);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, static_cast<uint32_t>(tmem_cols));
  }
}

// ============================================================================
// tc_output
// ============================================================================
template <int D>
struct OutCfg {
  static constexpr int C = 128;                 // tokens per chunk = MMA M
  static constexpr int ROWB = D * 2;
  static constexpr int QT = C * ROWB;           // q (then o) tile
  static constexpr int BT = D * ROWB;           // S~_i tile
  static constexpr int STAGE = ((QT + BT + 1023) / 1024) * 1024;
  static constexpr int NS = 6;
  static constexpr uint32_t SBO = 8 * ROWB;
  static constexpr uint32_t LAYOUT = D == 64 ? 2u : 4u;
  static constexpr int TMEM_COLS = 2 * D < 32 ? 32 : 2 * D;
  static constexpr int CTRL = 1024 + NS * C * 4;  // barriers + denominators
  static constexpr size_t SMEM = static_cast<size_t>(NS) * STAGE + CTRL + 1024;
};

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
tc_output(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_o,
          const __grid_constant__ CUtensorMap tm_st, TcGeom g, int64_t n_items, int phi_kind, float eps,
          const float* __restrict__ zt) {
  using Cfg = OutCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  uint8_t* stages = smem;
  uint8_t* ctrl = smem + Cfg::NS * Cfg::STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* phid = full + Cfg::NS;
  uint64_t* empty = phid + Cfg::NS;
  uint64_t* ostore = empty + Cfg::NS;
  uint64_t* tfull = ostore + Cfg::NS;
  uint64_t* tempty = tfull + 2;
  uint64_t* fin = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 512);
  volatile uint32_t* abortf = tmem_slot + 1;
  float* den_s = reinterpret_cast<float*>(ctrl + 1024);   // [NS][C]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::NS; ++s) {
      mbar_init(full + s, 1);
      mbar_init(phid + s, 128);
      mbar_init(empty + s, 1);
      mbar_init(ostore + s, 128);
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
    if (lane == 0) {
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_s = policy_evict_last();
      int s = 0;
      uint32_t ph = 0;
      uint64_t fills = 0;
      bool ok = true;
      for (int64_t item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        const int32_t i = static_cast<int32_t>(item % g.M);
        const int64_t bh = item / g.M;
        const int32_t b = static_cast<int32_t>(bh / g.H), h = static_cast<int32_t>(bh % g.H);
        for (int c = 0; c < g.chunks; ++c) {
          if (!wait_bounded(empty + s, ph ^ 1u, abortf)) { ok = false; break; }
          mbar_arrive_expect_tx(full + s, Cfg::QT + Cfg::BT);
          int32_t x, y, z;
          chunk_coords(g, i, c, b, x, y, z);
          uint8_t* st = stages + s * Cfg::STAGE;
          tma_load_5d(st, &tm_q, full + s, 0, h, x, y, z, pol_q);
          tma_load_2d(st + Cfg::QT, &tm_st, full + s, 0, static_cast<int32_t>(item * D), pol_s);
          ++fills;
          if (++s == Cfg::NS) { s = 0; ph ^= 1u; }
        }
      }
      for (int st = 0; st < Cfg::NS; ++st) {
        const uint64_t n = fills / Cfg::NS + (static_cast<uint64_t>(st) < fills % Cfg::NS ? 1 : 0);
        if (n > 0) drain_wait(full + st, static_cast<uint32_t>((n - 1) & 1));
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, D, /*a K-major*/ false, /*b MN-major*/ true);
      int s = 0;
      uint32_t ph = 0, cnt = 0;
      bool ok = true;
      for (int64_t item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        for (int c = 0; c < g.chunks; ++c, ++cnt) {
          const uint32_t acc = cnt & 1u, aph = (cnt >> 1) & 1u;
          if (!wait_bounded(tempty + acc, aph ^ 1u, abortf)) { ok = false; break; }
          if (!wait_bounded(phid + s, ph, abortf)) { ok = false; break; }
          tc_fence_after();
          const uint32_t base = smem_u32(stages + s * Cfg::STAGE);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint64_t a = smem_desc(base + ks * 32, 16, Cfg::SBO, Cfg::LAYOUT);
            const uint64_t b = smem_desc(base + Cfg::QT + ks * 2 * Cfg::SBO, 16, Cfg::SBO, Cfg::LAYOUT);
            mma_bf16(tmem + acc * D, a, b, idesc, ks != 0 ? 1u : 0u);
          }
          mma_commit(tfull + acc);
          if (++s == Cfg::NS) { s = 0; ph ^= 1u; }
        }
      }
      mma_commit(fin);
      drain_wait(fin, 0);
    }
  } else if (warp < 6) {
    // ------------------------------------------- phi on q, denominators
    constexpr int CPR = D / 8;            // 16-byte chunks per row
    constexpr int RP = 128 / CPR;         // rows covered per pass
    const int rt = threadIdx.x - 64;
    const int rg = rt / CPR, p = rt % CPR;
    const int lc = p ^ swz<D>(rg);        // logical chunk: channels lc*8 .. lc*8+7
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int64_t item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      const float4* zp = reinterpret_cast<const float4*>(zt + item * D + lc * 8);
      const float4 za = __ldg(zp), zb = __ldg(zp + 1);
      const float zr[8] = {za.x, za.y, za.z, za.w, zb.x, zb.y, zb.z, zb.w};
      for (int c = 0; c < g.chunks; ++c) {
        if (!warp_wait(full + s, ph, abortf)) { ok = false; break; }
        uint8_t* tile = stages + s * Cfg::STAGE;
#pragma unroll
        for (int m = 0; m < Cfg::C / RP; ++m) {
          const int r = rg + RP * m;
          uint4* ptr = reinterpret_cast<uint4*>(tile + r * Cfg::ROWB + p * 16);
          float f[8];
          *ptr = phi8(*ptr, phi_kind, eps, f);
          float part = 0.0f;
#pragma unroll
          for (int e = 0; e < 8; ++e) part = fmaf(f[e], zr[e], part);
#pragma unroll
          for (int off = 1; off < CPR; off <<= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
          if (p == 0) den_s[s * Cfg::C + r] = part;
        }
        fence_proxy_async_smem();
        mbar_arrive(phid + s);
        if (++s == Cfg::NS) { s = 0; ph ^= 1u; }
      }
    }
  } else {
    // ------------------------------------------- epilogue: divide, store by TMA
    const int q4 = warp & 3;
    const int row = 32 * q4 + lane;      // token row of the chunk
    const bool store_thread = (warp == 6 && lane == 0);
    int s = 0;
    uint32_t ph = 0, cnt = 0;
    bool ok = true;
    for (int64_t item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      const int32_t i = static_cast<int32_t>(item % g.M);
      const int64_t bh = item / g.M;
      const int32_t b = static_cast<int32_t>(bh / g.H), h = static_cast<int32_t>(bh % g.H);
      for (int c = 0; c < g.chunks; ++c, ++cnt) {
        const uint32_t acc = cnt & 1u, aph = (cnt >> 1) & 1u;
        if (!warp_wait(tfull + acc, aph, abortf)) { ok = false; break; }
        // den_s was written by the phi warps before they released this stage.
        if (!warp_wait(phid + s, ph, abortf)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tb = tmem + acc * D + (static_cast<uint32_t>(32 * q4) << 16);
        uint32_t v0[32], v1[32];
        tmem_ld_x32(tb, v0);
        if (D == 64) tmem_ld_x32(tb + 32, v1);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(tempty + acc);
        const float den = den_s[s * Cfg::C + row] + eps;
        uint8_t* orow = stages + s * Cfg::STAGE + row * Cfg::ROWB;
#pragma unroll
        for (int q = 0; q < D / 8; ++q) {
          const uint32_t* src = (q < 4) ? (v0 + 8 * q) : (v1 + 8 * (q - 4));
          const uint4 packed = make_uint4(
              pack_bf16(__uint_as_float(src[0]) / den, __uint_as_float(src[1]) / den),
              pack_bf16(__uint_as_float(src[2]) / den, __uint_as_float(src[3]) / den),
              pack_bf16(__uint_as_float(src[4]) / den, __uint_as_float(src[5]) / den),
              pack_bf16(__uint_as_float(src[6]) / den, __uint_as_float(src[7]) / den));
          *reinterpret_cast<uint4*>(orow + ((q ^ swz<D>(row)) * 16)) = packed;
        }
        fence_proxy_async_smem();
        mbar_arrive(ostore + s);
        if (store_thread) {
          if (wait_bounded(ostore + s, ph, abortf)) {
            int32_t x, y, z;
            chunk_coords(g, i, c, b, x, y, z);
            tma_store_5d(&tm_o, stages + s * Cfg::STAGE, 0, h, x, y, z);
            bulk_commit_group();
            bulk_wait_group_read0();
          } else {
            ok = false;
          }
          mbar_arrive(empty + s);
        }
        ok = __all_sync(0xffffffffu, ok);
        if (++s == Cfg::NS) { s = 0; ph ^= 1u; }
      }
    }
    if (store_thread) bulk_wait_group0();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::TMEM_COLS);
  }
}

// W (float32, M x M) -> bf16 [M][Mp], zero padded columns.
__global__ void convert_w(const float* __restrict__ W, __nv_bfloat16* __restrict__ Wb, int64_t M, int64_t Mp) {
  const int64_t n = M * Mp;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < n;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t i = e / Mp, j = e % Mp;
    Wb[e] = __float2bfloat16_rn(j < M ? W[i * M + j] : 0.0f);
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

struct ChunkPlan {
  int64_t box_y, box_t, nyc, chunks;
};

// Split every block into chunks of C tokens made of whole block rows (and,
// where a frame holds fewer than C tokens, whole frames).
bool chunk_plan(const Problem& p, int64_t C, ChunkPlan* cp) {
  if (p.w % C != 0 || C % p.bx != 0 || p.bx > 256) return false;
  const int64_t rows = C / p.bx;
  if (rows <= p.by) {
    if (p.by % rows != 0) return false;
    cp->box_y = rows;
    cp->box_t = 1;
    cp->nyc = p.by / rows;
  } else {
    if (rows % p.by != 0) return false;
    const int64_t frames = rows / p.by;
    if (p.bt % frames != 0) return false;
    cp->box_y = p.by;
    cp->box_t = frames;
    cp->nyc = 1;
  }
  if (cp->box_y > 256 || cp->box_t > 256) return false;
  cp->chunks = p.w / C;
  return true;
}

bool operand_tma_ok(const Problem& p, const Operand& o) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(o.data);
  if (a % 16 != 0) return false;
  if (o.sh % 8 != 0 || o.sn % 8 != 0 || o.sb % 8 != 0) return false;
  if ((p.H > 1 && o.sh <= 0) || o.sn <= 0) return false;
  if (p.T > 1 && o.sb != p.T * p.Y * p.X * o.sn) return false;   // (b, t) fold into one dimension
  const int64_t zstride = p.T > 1 ? p.Y * p.X * o.sn : o.sb;
  if (p.B > 1 && zstride <= 0) return false;
  const int64_t lim = int64_t{1} << 39;   // strides in bytes below 2^40
  return o.sh < lim && o.sn * p.X < lim && zstride < lim;
}

bool operand_map(const Problem& p, const Operand& o, int64_t box_y, int64_t box_t, CUtensorMap* m) {
  const int64_t zstride = p.T > 1 ? p.Y * p.X * o.sn : (p.B > 1 ? o.sb : p.Y * p.X * o.sn);
  const int64_t sh = p.H > 1 ? o.sh : p.d;
  const cuuint64_t dims[5] = {static_cast<cuuint64_t>(p.d), static_cast<cuuint64_t>(p.H),
                              static_cast<cuuint64_t>(p.X), static_cast<cuuint64_t>(p.Y),
                              static_cast<cuuint64_t>(p.B * p.T)};
  const cuuint64_t strides[4] = {static_cast<cuuint64_t>(sh * 2), static_cast<cuuint64_t>(o.sn * 2),
                                 static_cast<cuuint64_t>(p.X * o.sn * 2), static_cast<cuuint64_t>(zstride * 2)};
  const cuuint32_t box[5] = {static_cast<cuuint32_t>(p.d), 1u, static_cast<cuuint32_t>(p.bx),
                             static_cast<cuuint32_t>(box_y), static_cast<cuuint32_t>(box_t)};
  return encode(m, 5, o.data, dims, strides, box,
                p.d == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}

struct TcLayout {
  size_t wb_off, sbuf_off, st_off, zt_off, total;
  int64_t Mp, ncols;
};

TcLayout tc_layout(const Problem& p) {
  TcLayout L;
  L.Mp = (p.M + 7) / 8 * 8;
  L.ncols = p.BH() * (p.d + 1) * p.d;
  size_t off = 0;
  L.wb_off = off;
  off += align_up(static_cast<size_t>(p.M) * L.Mp * 2);
  L.sbuf_off = off;
  off += align_up(static_cast<size_t>(p.M) * L.ncols * 2);
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

TcGeom make_geom(const Problem& p, const ChunkPlan& cp) {
  TcGeom g;
  g.M = static_cast<int32_t>(p.M);
  g.nbx = static_cast<int32_t>(p.nbx);
  g.nby = static_cast<int32_t>(p.nby);
  g.bx = static_cast<int32_t>(p.bx);
  g.by = static_cast<int32_t>(p.by);
  g.bt = static_cast<int32_t>(p.bt);
  g.T = static_cast<int32_t>(p.T);
  g.box_y = static_cast<int32_t>(cp.box_y);
  g.box_t = static_cast<int32_t>(cp.box_t);
  g.nyc = static_cast<int32_t>(cp.nyc);
  g.chunks = static_cast<int32_t>(cp.chunks);
  g.H = static_cast<int32_t>(p.H);
  g.B = static_cast<int32_t>(p.B);
  return g;
}

template <int D>
int launch_tc_d(const Problem& p, const float* W, void* workspace, cudaStream_t stream) {
  const TcLayout L = tc_layout(p);
  char* ws = static_cast<char*>(workspace);
  __nv_bfloat16* Wb = reinterpret_cast<__nv_bfloat16*>(ws + L.wb_off);
  __nv_bfloat16* Sbuf = reinterpret_cast<__nv_bfloat16*>(ws + L.sbuf_off);
  __nv_bfloat16* St = reinterpret_cast<__nv_bfloat16*>(ws + L.st_off);
  float* zt = reinterpret_cast<float*>(ws + L.zt_off);
  const int sms = device_sms();
  if (sms <= 0) return MHLA_ERR_CUDA;

  ChunkPlan c64, c128;
  if (!chunk_plan(p, 64, &c64) || !chunk_plan(p, 128, &c128)) return MHLA_ERR_UNSUPPORTED;

  // ---- step 0: W -> bf16
  {
    const int64_t n = p.M * L.Mp;
    const int blocks = static_cast<int>(std::min<int64_t>((n + 255) / 256, 4096));
    KernelTimer timer("convert_w", stream);
    convert_w<<<blocks, 256, 0, stream>>>(W, Wb, p.M, L.Mp);
    if (cudaGetLastError() != cudaSuccess) return MHLA_ERR_CUDA;
  }

  // ---- step 1: summaries
  {
    using Cfg = SumCfg<D>;
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
    tc_summary<D><<<grid, kTcThreads, Cfg::SMEM, stream>>>(tk, tv, make_geom(p, c64), G, n_items, L.ncols,
                                                           p.phi_kind, p.eps, Sbuf);
    if (cudaGetLastError() != cudaSuccess) return MHLA_ERR_CUDA;
  }

  // ---- step 2: mixing GEMM
  {
    const int32_t N = static_cast<int32_t>(std::min<int64_t>(256, (p.M + 15) / 16 * 16));
    int32_t tcols = 32;
    while (tcols < N) tcols *= 2;
    const int32_t acc_stride = tcols;
    const int32_t tmem_cols = 2 * tcols;
    const int32_t stage_bytes = MixCfg::A_BYTES + ((N * 128 + 1023) / 1024) * 1024;
    const size_t smem = static_cast<size_t>(MixCfg::NS) * stage_bytes + MixCfg::CTRL + 1024;
    CUtensorMap ts, tw;
    {
      const cuuint64_t dims[2] = {static_cast<cuuint64_t>(L.ncols), static_cast<cuuint64_t>(p.M)};
      const cuuint64_t strides[1] = {static_cast<cuuint64_t>(L.ncols * 2)};
      const cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(MixCfg::KC)};
      if (!encode(&ts, 2, Sbuf, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return MHLA_ERR_CUDA;
    }
    {
      const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.M), static_cast<cuuint64_t>(p.M)};
      const cuuint64_t strides[1] = {static_cast<cuuint64_t>(L.Mp * 2)};
      const cuuint32_t box[2] = {static_cast<cuuint32_t>(MixCfg::KC), static_cast<cuuint32_t>(N)};
      if (!encode(&tw, 2, Wb, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return MHLA_ERR_CUDA;
    }
    const int32_t n_col_tiles = static_cast<int32_t>((L.ncols + MixCfg::COLS - 1) / MixCfg::COLS);
    const int32_t n_i_tiles = static_cast<int32_t>((p.M + 255) / 256);
    if (cudaFuncSetAttribute(tc_mix, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess)
      return MHLA_ERR_CUDA;
    const int per_sm = std::max(1, std::min(occupancy(tc_mix, kMixThreadsTC, smem), 512 / tmem_cols));
    const int64_t n_tiles = static_cast<int64_t>(n_col_tiles) * n_i_tiles;
    const int grid = static_cast<int>(std::min<int64_t>(n_tiles, static_cast<int64_t>(sms) * per_sm));
    KernelTimer timer("tc_mix", stream);
    tc_mix<<<grid, kMixThreadsTC, smem, stream>>>(ts, tw, static_cast<int32_t>(p.M), N, stage_bytes, tmem_cols,
                                                   acc_stride, L.ncols, n_col_tiles, n_i_tiles,
                                                   static_cast<int32_t>(p.d), St, zt);
    if (cudaGetLastError() != cudaSuccess) return MHLA_ERR_CUDA;
  }

  // ---- step 3: outputs
  {
    using Cfg = OutCfg<D>;
    CUtensorMap tq, to, tst;
    if (!operand_map(p, p.q, c128.box_y, c128.box_t, &tq) || !operand_map(p, p.o, c128.box_y, c128.box_t, &to))
      return MHLA_ERR_CUDA;
    {
      const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.d), static_cast<cuuint64_t>(p.BH() * p.M * p.d)};
      const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.d * 2)};
      const cuuint32_t box[2] = {static_cast<cuuint32_t>(p.d), static_cast<cuuint32_t>(p.d)};
      if (!encode(&tst, 2, St, dims, strides, box,
                  p.d == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
        return MHLA_ERR_CUDA;
    }
    const int64_t n_items = p.BH() * p.M;
    if (cudaFuncSetAttribute(tc_output<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(Cfg::SMEM)) != cudaSuccess)
      return MHLA_ERR_CUDA;
    const int per_sm = std::max(1, std::min(occupancy(tc_output<D>, kTcThreads, Cfg::SMEM), 512 / Cfg::TMEM_COLS));
    const int grid = static_cast<int>(std::min<int64_t>(n_items, static_cast<int64_t>(sms) * per_sm));
    KernelTimer timer("tc_output", stream);
    tc_output<D><<<grid, kTcThreads, Cfg::SMEM, stream>>>(tq, to, tst, make_geom(p, c128), n_items, p.phi_kind,
                                                          p.eps, zt);
    if (cudaGetLastError() != cudaSuccess) return MHLA_ERR_CUDA;
  }
  return MHLA_OK;
}

}  // namespace

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
