// Tensor-core causal (chunkwise) MHLA on sm_103a: bf16, d in {32, 64},
// contiguous blocks of w = 64 tokens or a multiple of 128, N a multiple of 128.
//
// [P2] "MHLA: Restoring Expressivity of Linear Attention via Token-Level
// Multi-Head", App. B "Causal MHLA": block-specific mixed summaries, each
// block's mixture reused, causal at the cost of chunkwise linear attention.
// Read as the causal restriction of the two-stage form: token t of block i sees
// every past block j < i through W[i][j] and the tokens s <= t of its own block
// through W[i][i].
//
// The sequence is cut into units of U = min(w, 128) tokens.  With S_u the
// summary of unit u, the state a unit starts from is
//   S'_u = sum_{u'} W'[u][u'] S_u',  W'[u][u'] = W[b(u)][b(u')] if b(u') < b(u),
//                                               W[b(u)][b(u)]  if b(u') = b(u), u' < u,
//                                               0 otherwise,
// (z'_u likewise): one GEMM with the forward's mixing kernel on the expanded
// unit-level W'.  Then per 128-token tile (1 or 2 units), with phi(Q)_u the
// tile's rows of unit u and P[t][s] = W[b(t)][b(t)] phi(q_t) . phi(k_s) for
// s <= t in the same block (0 otherwise):
//   [num | den]_t = P_t [V | 1] + phi(q_t) [S'_u(t) | z'_u(t)]
// numerator and denominator from the same MMAs.
//
// With two units per tile the state term of each unit gets its own
// accumulator (A = the whole phi(Q) tile, each row reads its own unit's), so
// the state MMAs run while the workers form P.
//
// tc_causal_tile: persistent CTAs; warp 9 issues the TMA loads, warp 8 the
// MMAs, warps 0-7 (two warpgroups) apply phi, form P and write the output, one
// tile ahead (phi and the scores of the next tile run under this tile's MMAs and
// output).  q, k, v tiles and the state tiles are double-buffered.  Every wait is bounded; a wait that gives up sets
// bit 0 of this file's device error word and an abort flag, the CTA drains
// what it issued and releases tensor memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "mhla_internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"
#include "tma_host.h"

namespace mhla {

__device__ unsigned int g_causal_error = 0;

namespace {

using namespace tc;

__device__ __forceinline__ bool cwait(uint64_t* bar, uint32_t parity, volatile uint32_t* abortf) {
  return wait_bounded_on(bar, parity, abortf, &g_causal_error);
}
__device__ __forceinline__ bool cwarp_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abortf) {
  return warp_wait_on(bar, parity, abortf, &g_causal_error);
}
__device__ __forceinline__ void cdrain(uint64_t* bar, uint32_t parity) { drain_wait_on(bar, parity, &g_causal_error); }

constexpr int kCtWorkers = 256;
constexpr int kCtThreads = kCtWorkers + 64;   // workers, MMA issuer, load producer
constexpr int kTile = 128;

template <int D, int NU>
struct CtCfg {
  static constexpr int ROWB = D * 2;
  static constexpr int TILE = kTile * ROWB;           // one [128][D] token tile
  static constexpr uint32_t SBO = 8 * ROWB;
  static constexpr uint32_t LAYOUT = D == 64 ? 2u : 4u;
  static constexpr int ST = D * D * 2;                // one state tile (row-major, swizzled like a token tile)
  static constexpr int P_CHUNK = kTile * 128;         // 64 keys of P, K-major, 128-byte swizzle
  static constexpr int QT_OFF = 0;                    // [2] phi(q) tiles
  static constexpr int KT_OFF = QT_OFF + 2 * TILE;    // [2] phi(k) tiles
  static constexpr int VT_OFF = KT_OFF + 2 * TILE;    // [2] v tiles, then the ones atom
  static constexpr int ONES_OFF = VT_OFF + 2 * TILE;
  static constexpr int P_OFF = ONES_OFF + TILE;
  static constexpr int SLOT = NU * 2 * ST;            // per unit: state tile, z' atom
  static constexpr int SZ_OFF = P_OFF + 2 * P_CHUNK;  // [2] slots
  static constexpr int ZRAW_OFF = SZ_OFF + 2 * SLOT;  // [2][NU][D] float32
  static constexpr int CTRL_OFF = ZRAW_OFF + 2 * NU * D * 4;
  static constexpr size_t SMEM = CTRL_OFF + 128 + 1024;
  static constexpr int NO = D + 16;                   // MMA 2 columns: d values, the denominator block
  // scores [0, 128); P [V | 1] (and, with one unit, its state term) at 128;
  // with two units, their state terms at 256 and 384
  static constexpr int TMEM_COLS = NU > 1 ? 512 : 256;
  static __host__ __device__ constexpr int state_col(int k) { return NU > 1 ? 256 + 128 * k : 128; }
};

struct CtGeom {
  int32_t N, H, M, w, U, Mu, nt;   // tokens, heads, blocks, block and unit length, units, tiles per (b, h)
};

// INTRA = false (the non-causal forward on 64-token contiguous blocks): units
// are the blocks, the states are the ordinary mixed summaries S~, z~, and only
// the state MMAs run (no k, v tiles, no scores).
template <int D, int NU, bool INTRA>
__global__ void __launch_bounds__(kCtThreads, 1)
tc_causal_tile(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_st, CtGeom g,
               int64_t n_units, int phi_kind, float eps, const float* __restrict__ W,
               const float* __restrict__ zt, __nv_bfloat16* __restrict__ out, int64_t osb, int64_t osn,
               int64_t osh) {
  using Cfg = CtCfg<D, NU>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  uint8_t* qt = smem + Cfg::QT_OFF;
  uint8_t* kt = smem + Cfg::KT_OFF;
  uint8_t* vt = smem + Cfg::VT_OFF;
  uint8_t* ones = smem + Cfg::ONES_OFF;
  uint8_t* sp = smem + Cfg::P_OFF;
  uint8_t* sz = smem + Cfg::SZ_OFF;
  float* zraw = reinterpret_cast<float*>(smem + Cfg::ZRAW_OFF);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::CTRL_OFF);   // [2] q (k, v) of a stage landed
  uint64_t* full_st = full + 2;       // [2] state tiles and z' of a slot landed
  uint64_t* phid = full + 4;          // workers: phi applied
  uint64_t* done1 = full + 5;         // MMA 1 (scores) complete
  uint64_t* zready = full + 6;        // workers: the z' atoms of the slot written
  uint64_t* ready = full + 7;         // workers: P written
  uint64_t* done2 = full + 8;         // every MMA of the tile complete
  uint64_t* odone = full + 9;         // workers: the accumulators read
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(full + 10);
  volatile uint32_t* abortf = tmem_slot + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == kCtWorkers) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(full + i, 1);
      mbar_init(full_st + i, 1);
    }
    mbar_init(phid, kCtWorkers / 32);
    mbar_init(done1, 1);
    mbar_init(zready, kCtWorkers / 32);
    mbar_init(ready, kCtWorkers / 32);
    mbar_init(done2, 1);
    mbar_init(odone, kCtWorkers / 32);
    *abortf = 0u;
    fence_mbar_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_st);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  if (tid < kCtWorkers) {
    // ones atom of [V | 1]: row s holds (1, 0, ..., 0); the z' atoms start at zero
    for (int idx = tid; idx < kTile * (D / 8); idx += kCtWorkers) {
      const int row = idx / (D / 8), phys = idx % (D / 8);
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if ((phys ^ swz<D>(row)) == 0) v.x = 0x3F80u;
      *reinterpret_cast<uint4*>(ones + row * Cfg::ROWB + phys * 16) = v;
    }
    for (int e = tid; e < 2 * Cfg::SLOT / 16; e += kCtWorkers)
      reinterpret_cast<uint4*>(sz)[e] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // unit -> (b, h, tile), in 32-bit arithmetic (n_units < 2^31, checked on the host)
  auto coords = [&](int64_t u, int32_t& b, int32_t& h, int32_t& tile) {
    const uint32_t uu = static_cast<uint32_t>(u);
    tile = static_cast<int32_t>(uu % static_cast<uint32_t>(g.nt));
    const uint32_t bh = uu / static_cast<uint32_t>(g.nt);
    h = static_cast<int32_t>(bh % static_cast<uint32_t>(g.H));
    b = static_cast<int32_t>(bh / static_cast<uint32_t>(g.H));
  };

  // stage st: q (k, v) tiles and the state slot of unit u
  auto issue = [&](int st, int64_t u, uint64_t pol, uint64_t pol_st) {
    int32_t b, h, tile;
    coords(u, b, h, tile);
    mbar_arrive_expect_tx(full + st, (INTRA ? 3 : 1) * Cfg::TILE);
    tma_load_4d(qt + st * Cfg::TILE, &tm_q, full + st, 0, h, tile * kTile, b, pol);
    if (INTRA) {
      tma_load_4d(kt + st * Cfg::TILE, &tm_k, full + st, 0, h, tile * kTile, b, pol);
      tma_load_4d(vt + st * Cfg::TILE, &tm_v, full + st, 0, h, tile * kTile, b, pol);
    }
    mbar_arrive_expect_tx(full_st + st, NU * (Cfg::ST + D * 4));
    for (int k = 0; k < NU; ++k) {
      const int64_t su = (static_cast<int64_t>(b) * g.H + h) * g.Mu + static_cast<int64_t>(tile) * NU + k;
      tma_load_2d(sz + st * Cfg::SLOT + k * 2 * Cfg::ST, &tm_st, full_st + st, 0, static_cast<int32_t>(su * D),
                  pol_st);
      bulk_load(zraw + (st * NU + k) * D, zt + su * D, D * 4, full_st + st, pol_st);
    }
  };

  if (warp == kCtWorkers / 32 + 1) {
    // ------------------------------------------------------------ load producer
    // Tiles n and n + 1 up front; tile n + 2 into stage n % 2 as soon as every MMA
    // of tile n is complete.
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const uint64_t pol_st = policy_evict_last();
      uint32_t n_stage[2] = {0, 0};
      const int64_t u0 = blockIdx.x, stride = gridDim.x;
      for (int st = 0; st < 2; ++st)
        if (u0 + st * stride < n_units) {
          issue(st, u0 + st * stride, pol, pol_st);
          n_stage[st] = 1;
        }
      uint32_t it = 0;
      for (int64_t u = u0; u + 2 * stride < n_units; u += stride, ++it) {
        if (!cwait(done2, it & 1u, abortf)) break;
        const int st = static_cast<int>(it & 1u);
        issue(st, u + 2 * stride, pol, pol_st);
        ++n_stage[st];
      }
      for (int st = 0; st < 2; ++st)
        if (n_stage[st]) {
          cdrain(full + st, (n_stage[st] - 1) & 1u);
          cdrain(full_st + st, (n_stage[st] - 1) & 1u);
        }
    }
  } else if (warp == kCtWorkers / 32) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t n_m1 = 0, n_m2 = 0;
      const int64_t u0 = blockIdx.x, stride = gridDim.x;
      // MMA 1 of a tile: scores = phi(Q) phi(K)^T, 128 x 128 (TMEM columns 0..127)
      auto mma1 = [&](int st) {
        constexpr uint32_t idesc = idesc_bf16_f32(128, kTile, /*a K-major*/ false, /*b K-major*/ false);
        const uint32_t qa = smem_u32(qt + st * Cfg::TILE), ka = smem_u32(kt + st * Cfg::TILE);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_bf16(tmem, smem_desc(qa + ks * 32, 16, Cfg::SBO, Cfg::LAYOUT),
                   smem_desc(ka + ks * 32, 16, Cfg::SBO, Cfg::LAYOUT), idesc, ks > 0 ? 1u : 0u);
        mma_commit(done1);
        ++n_m1;
      };
      bool ok = u0 < n_units && cwait(full, 0, abortf) && cwait(phid, 0, abortf);
      if (ok) {
        tc_fence_after();
        if (INTRA) mma1(0);
      }
      uint32_t it = 0;
      for (int64_t u = u0; ok && u < n_units; u += stride, ++it) {
        const uint32_t par = it & 1u, par2 = (it >> 1) & 1u;
        const int st = static_cast<int>(it & 1u);
        const bool has_next = u + stride < n_units;
        const uint32_t qa = smem_u32(qt + st * Cfg::TILE);
        // the previous tile's output has read the accumulators
        if (it > 0 && !cwait(odone, par ^ 1u, abortf)) break;
        constexpr uint32_t idesc2 = idesc_bf16_f32(128, Cfg::NO, /*a K-major*/ false, /*b MN-major*/ true);
        if (INTRA) {   // P [V | 1] into column 128
          if (!cwait(ready, par, abortf)) break;
          tc_fence_after();
          const uint32_t pa = smem_u32(sp), va = smem_u32(vt + st * Cfg::TILE);
          const uint32_t lbo_v = static_cast<uint32_t>(Cfg::ONES_OFF - (Cfg::VT_OFF + st * Cfg::TILE));
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks)
            mma_bf16(tmem + 128, smem_desc(pa + (ks >> 2) * Cfg::P_CHUNK + (ks & 3) * 32, 16, 1024, 2),
                     smem_desc(va + ks * 2 * Cfg::SBO, lbo_v, Cfg::SBO, Cfg::LAYOUT), idesc2, ks > 0 ? 1u : 0u);
        }
        // state MMAs: phi(Q) [S'_u | z'_u hi lo], one accumulator per unit; with one
        // unit (NU == 1) it is the accumulator of P [V | 1] (column 128) and adds to it
        if (!cwait(full_st + st, par2, abortf) || !cwait(zready, par, abortf)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < NU; ++k) {
          const uint32_t sb = smem_u32(sz + st * Cfg::SLOT + k * 2 * Cfg::ST);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            mma_bf16(tmem + Cfg::state_col(k), smem_desc(qa + ks * 32, 16, Cfg::SBO, Cfg::LAYOUT),
                     smem_desc(sb + ks * 2 * Cfg::SBO, Cfg::ST, Cfg::SBO, Cfg::LAYOUT), idesc2,
                     (ks > 0 || (INTRA && NU == 1)) ? 1u : 0u);
        }
        // the next tile's phi is done before this tile's MMAs are reported (so its
        // phid arrival cannot run a phase ahead of this wait); then its scores
        // (columns 0..127, read out into P before this tile's P [V | 1] was issued)
        if (has_next) {
          const int sn = st ^ 1;
          if (!cwait(full + sn, ((it + 1) >> 1) & 1u, abortf) || !cwait(phid, par ^ 1u, abortf)) break;
          tc_fence_after();
        }
        mma_commit(done2);
        ++n_m2;
        if (INTRA && has_next) mma1(st ^ 1);
      }
      if (n_m1) cdrain(done1, (n_m1 - 1) & 1u);
      if (n_m2) cdrain(done2, (n_m2 - 1) & 1u);
    }
  } else {
    // ------------------------------------------------------------ workers
    // One tile ahead: phi of tile n + 1 runs under this tile's MMAs, and the
    // scores of tile n + 1 under this tile's output.
    const int row = tid & 127;                    // query row = TMEM lane
    const int half = tid >> 7;                    // key chunks and output columns of this warpgroup
    const int q4 = warp & 3;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    const int my_unit = NU > 1 ? q4 >> 1 : 0;     // rows 0-63 unit 0, 64-127 unit 1: uniform per warp
    const bool add_eps = phi_kind == MHLA_PHI_RELU_EPS;
    const __nv_bfloat162 eps2 = __float2bfloat162_rn(eps);
    const int swr = row & 7;
    // phi on the q (and k) tiles of a stage
    auto apply_phi = [&](int st) {
      for (int e = tid; e < (INTRA ? 2 : 1) * Cfg::TILE / 16; e += kCtWorkers) {
        uint4* p = reinterpret_cast<uint4*>(e < Cfg::TILE / 16 ? qt + st * Cfg::TILE : kt + st * Cfg::TILE) +
                   (e % (Cfg::TILE / 16));
        *p = phi8_packed(*p, add_eps, eps2);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(phid);
    };
    // z' atoms of a slot (row r: columns 0, 1 = hi, lo)
    auto write_z = [&](int st) {
      if (tid < NU * D) {
        const int k = tid / D, r = tid % D;
        const float zv = zraw[(st * NU + k) * D + r];
        const __nv_bfloat16 hi = __float2bfloat16_rn(zv);
        const __nv_bfloat16 lo = __float2bfloat16_rn(zv - __bfloat162float(hi));
        *reinterpret_cast<uint32_t*>(sz + st * Cfg::SLOT + k * 2 * Cfg::ST + Cfg::ST + r * Cfg::ROWB + swz<D>(r) * 16) =
            static_cast<uint32_t>(__bfloat16_as_ushort(hi)) | (static_cast<uint32_t>(__bfloat16_as_ushort(lo)) << 16);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(zready);
    };
    // W_ii of this row's block in tile u (read ahead of the scores)
    auto row_weight = [&](int64_t u) {
      const int32_t tile = static_cast<int32_t>(static_cast<uint32_t>(u) % static_cast<uint32_t>(g.nt));
      const int32_t blk = (tile * kTile + row) / g.w;
      return INTRA ? __ldg(W + static_cast<int64_t>(blk) * g.M + blk) : 0.0f;
    };
    // P = W_ii * score for keys s <= t of the same block, from the scores of tile u
    auto form_p = [&](int64_t u, float wii) {
      int32_t b, h, tile;
      coords(u, b, h, tile);
      const int32_t n0 = tile * kTile;
      const int32_t blk = (n0 + row) / g.w;
      const int32_t first = blk * g.w - n0;      // first key of this row's block inside the tile (may be < 0)
      for (int m = half; m < kTile / 32; m += 2) {   // 32 keys per step
        uint32_t r[32];
        tmem_ld_x32(lane_base + m * 32, r);
        tmem_ld_wait();
        uint32_t packed[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int s0 = m * 32 + e;
          const bool k0 = s0 <= row && s0 >= first;
          const bool k1 = s0 + 1 <= row && s0 + 1 >= first;
          packed[e >> 1] =
              pack_bf16(k0 ? __uint_as_float(r[e]) * wii : 0.0f, k1 ? __uint_as_float(r[e + 1]) * wii : 0.0f);
        }
        uint8_t* prow = sp + (m >> 1) * Cfg::P_CHUNK + row * 128;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4*>(prow + ((((m & 1) * 4 + q) ^ swr) * 16)) =
              make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ready);
    };

    bool ok = static_cast<int64_t>(blockIdx.x) < n_units;
    if (ok) {
      ok = cwarp_wait(full, 0, abortf);
      if (ok) apply_phi(0);
      if (ok && INTRA) {
        const float wii0 = row_weight(blockIdx.x);
        ok = cwarp_wait(done1, 0, abortf);
        if (ok) {
          tc_fence_after();
          form_p(blockIdx.x, wii0);
        }
      }
      ok = ok && cwarp_wait(full_st, 0, abortf);
      if (ok) write_z(0);
    }
    uint32_t it = 0;
    for (int64_t u = blockIdx.x; ok && u < n_units; u += gridDim.x, ++it) {
      const uint32_t par = it & 1u;
      const int st = static_cast<int>(it & 1u), sn = st ^ 1;
      const uint32_t parn2 = ((it + 1) >> 1) & 1u;
      const bool has_next = u + gridDim.x < n_units;
      int32_t b, h, tile;
      coords(u, b, h, tile);
      const float wii_next = has_next ? row_weight(u + gridDim.x) : 0.0f;
      // ---- phi of the next tile
      if (has_next) {
        if (!cwarp_wait(full + sn, parn2, abortf)) break;
        apply_phi(sn);
      }
      // ---- output: o_t = num_t / (den_t + eps), this warpgroup's half of the columns
      if (!cwarp_wait(done2, par, abortf)) break;
      tc_fence_after();
      const int32_t n0 = tile * kTile;
      constexpr int HC = D / 2;
      uint32_t o[HC], dn[2];
      const uint32_t sc = lane_base + Cfg::state_col(my_unit);
      if constexpr (HC == 32) {
        tmem_ld_x32(sc + half * HC, o);
      } else {
        tmem_ld_x16(sc + half * HC, o);
      }
      tmem_ld_x1(sc + D, dn[0]);
      tmem_ld_x1(sc + D + 1, dn[1]);
      tmem_ld_wait();
      float den = __uint_as_float(dn[0]) + __uint_as_float(dn[1]);
      if (INTRA && NU > 1) {   // add P [V | 1] from column 128
        uint32_t o2[HC], d2;
        if constexpr (HC == 32) {
          tmem_ld_x32(lane_base + 128 + half * HC, o2);
        } else {
          tmem_ld_x16(lane_base + 128 + half * HC, o2);
        }
        tmem_ld_x1(lane_base + 128 + D, d2);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < HC; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) + __uint_as_float(o2[e]));
        den += __uint_as_float(d2);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(odone);
      const float inv = 1.0f / (den + eps);
      uint4* dstp = reinterpret_cast<uint4*>(out + b * osb + static_cast<int64_t>(n0 + row) * osn + h * osh +
                                             half * HC);
#pragma unroll
      for (int q = 0; q < HC / 8; ++q)
        dstp[q] = make_uint4(pack_bf16(__uint_as_float(o[8 * q]) * inv, __uint_as_float(o[8 * q + 1]) * inv),
                             pack_bf16(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv),
                             pack_bf16(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv),
                             pack_bf16(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv));
      // ---- the next tile's P (after this tile's P [V | 1] has read P), then its z'
      // atoms (after this tile's state MMAs, so zready stays one phase ahead at most)
      if (has_next) {
        if (INTRA) {
          if (!cwarp_wait(done1, par ^ 1u, abortf)) break;
          tc_fence_after();
          form_p(u + gridDim.x, wii_next);
        }
        if (!cwarp_wait(full_st + sn, parn2, abortf)) break;
        write_z(sn);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::TMEM_COLS);
  }
}

// ----------------------------------------------------------------- host side

struct CtLayout {
  size_t wu_off, sbuf_off, st_off, zt_off, total;
  int64_t Mp, Mu;
  int32_t U;
};

CtLayout ct_layout(const Problem& p) {
  CtLayout L;
  L.U = p.w == 64 ? 64 : 128;
  L.Mu = p.N / L.U;
  L.Mp = (L.Mu + 7) / 8 * 8;
  const int64_t ncols = p.BH() * (p.d + 1) * p.d;
  const int64_t ngroups = (ncols + 127) / 128;
  size_t off = 0;
  L.wu_off = off;
  off += align_up(static_cast<size_t>(L.Mu) * L.Mp * 2);
  L.sbuf_off = off;
  off += align_up(static_cast<size_t>(L.Mu) * ngroups * 128 * 2);
  L.st_off = off;
  off += align_up(static_cast<size_t>(p.BH()) * L.Mu * p.d * p.d * 2);
  L.zt_off = off;
  off += align_up(static_cast<size_t>(p.BH()) * L.Mu * p.d * 4);
  L.total = off;
  return L;
}

// The problem seen as 64-token rows cut into units of U tokens (same tensors).
Problem unit_problem(const Problem& p, int32_t U) {
  Problem u = p;
  u.ndim = 2;
  u.T = 1;
  u.Y = p.N / 64;
  u.X = 64;
  u.bt = 1;
  u.by = U / 64;
  u.bx = 64;
  u.nbt = 1;
  u.nby = p.N / U;
  u.nbx = 1;
  u.M = p.N / U;
  u.w = U;
  return u;
}

bool ct_map(const Problem& p, const Operand& o, CUtensorMap* m) {
  const int64_t sh = p.H > 1 ? o.sh : p.d;
  const int64_t sn = o.sn;
  const int64_t sb = p.B > 1 ? o.sb : p.N * p.H * p.d;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(p.d), static_cast<cuuint64_t>(p.H),
                              static_cast<cuuint64_t>(p.N), static_cast<cuuint64_t>(p.B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(sh * 2), static_cast<cuuint64_t>(sn * 2),
                                 static_cast<cuuint64_t>(sb * 2)};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(p.d), 1u, static_cast<cuuint32_t>(kTile), 1u};
  return encode_tensor_map(m, 4, o.data, dims, strides, box,
                           p.d == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}

template <int D, int NU, bool INTRA>
int launch_ct_tile(const Problem& p, const float* W, int64_t Mu, const __nv_bfloat16* St, const float* zt,
                   cudaStream_t stream) {
  using Cfg = CtCfg<D, NU>;
  CUtensorMap tq, tk, tv, tst;
  if (!ct_map(p, p.q, &tq) || !ct_map(p, p.k, &tk) || !ct_map(p, p.v, &tv)) return MHLA_ERR_CUDA;
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(p.BH() * Mu * D)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D * 2)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(D), static_cast<cuuint32_t>(D)};
    if (!encode_tensor_map(&tst, 2, const_cast<__nv_bfloat16*>(St), dims, strides, box,
                           D == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
      return MHLA_ERR_CUDA;
  }
  CtGeom g;
  g.N = static_cast<int32_t>(p.N);
  g.H = static_cast<int32_t>(p.H);
  g.M = static_cast<int32_t>(p.M);
  g.w = static_cast<int32_t>(p.w);
  g.U = static_cast<int32_t>(p.N / Mu);
  g.Mu = static_cast<int32_t>(Mu);
  g.nt = static_cast<int32_t>(p.N / kTile);
  const int64_t n_units = p.BH() * g.nt;
  if (n_units >= (int64_t{1} << 31)) return MHLA_ERR_UNSUPPORTED;   // the kernel decodes units in 32 bits
  const int sms = device_sm_count();
  if (sms <= 0) return MHLA_ERR_CUDA;
  if (cudaFuncSetAttribute(tc_causal_tile<D, NU, INTRA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(Cfg::SMEM)) != cudaSuccess)
    return MHLA_ERR_CUDA;
  const int grid = static_cast<int>(std::min<int64_t>(n_units, sms));
  KernelTimer timer(INTRA ? "tc_causal_tile" : "tc_tile_output", stream);
  tc_causal_tile<D, NU, INTRA><<<grid, kCtThreads, Cfg::SMEM, stream>>>(
      tq, tk, tv, tst, g, n_units, p.phi_kind, p.eps, W, zt, static_cast<__nv_bfloat16*>(p.o.data), p.o.sb, p.o.sn,
      p.o.sh);
  return cudaGetLastError() == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
}

}  // namespace

bool tc_causal_eligible(const Problem& p) {
  if (!blocks_contiguous(p)) return false;
  if (p.dtype != MHLA_BF16 || (p.d != 32 && p.d != 64)) return false;
  if (p.B < 1 || p.H < 1 || p.N % kTile != 0) return false;
  if (p.w != 64 && p.w % 128 != 0) return false;
  for (const Operand* o : {&p.q, &p.k, &p.v, &p.o}) {
    if (reinterpret_cast<uintptr_t>(o->data) % 16 != 0) return false;
    if (o->sb % 8 != 0 || o->sn % 8 != 0 || o->sh % 8 != 0 || o->sn <= 0) return false;
    if ((p.H > 1 && o->sh <= 0) || (p.B > 1 && o->sb <= 0)) return false;
    const int64_t lim = int64_t{1} << 39;
    if (o->sb >= lim || o->sn * 64 >= lim || o->sh >= lim) return false;
  }
  const Problem u = unit_problem(p, p.w == 64 ? 64 : 128);
  for (const Operand* o : {&u.k, &u.v})
    if (!operand_tma_ok(u, *o)) return false;
  const int64_t lim32 = int64_t{1} << 31;
  return p.BH() * u.M * p.d < lim32 && p.BH() * (p.N / kTile) < lim32 && p.BH() * (p.d + 1) * p.d < lim32;
}

size_t tc_causal_workspace_bytes(const Problem& p) { return ct_layout(p).total; }

int launch_tc_causal(const Problem& p, const float* W, void* workspace, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const CtLayout L = ct_layout(p);
  char* ws = static_cast<char*>(workspace);
  auto* Wu = reinterpret_cast<__nv_bfloat16*>(ws + L.wu_off);
  auto* St = reinterpret_cast<__nv_bfloat16*>(ws + L.st_off);
  auto* zt = reinterpret_cast<float*>(ws + L.zt_off);
  const Problem pu = unit_problem(p, L.U);
  // unit summaries, and the unit-level causal W' in the summary kernel's prologue
  int rc = tc_run_summary(pu, W, Wu, nullptr, L.Mp, ws + L.sbuf_off, stream, static_cast<int32_t>(p.M),
                          static_cast<int32_t>(p.w / L.U < 1 ? 1 : p.w / L.U));
  if (rc == MHLA_OK) rc = tc_run_mix(pu, Wu, L.Mp, ws + L.sbuf_off, St, zt, stream, /*discard_input=*/true);
  if (rc != MHLA_OK) return rc;
  const int NU = L.U == 64 ? 2 : 1;
  if (p.d == 64)
    return NU == 2 ? launch_ct_tile<64, 2, true>(p, W, L.Mu, St, zt, s) : launch_ct_tile<64, 1, true>(p, W, L.Mu, St, zt, s);
  return NU == 2 ? launch_ct_tile<32, 2, true>(p, W, L.Mu, St, zt, s) : launch_ct_tile<32, 1, true>(p, W, L.Mu, St, zt, s);
}

bool tc_tile_eligible(const Problem& p) {
  return p.w == 64 && blocks_contiguous(p) && tc_causal_eligible(p);
}

int launch_tc_tile_forward(const Problem& p, const float* W, void* Wb, int64_t Mp, void* Sbuf, void* St, float* zt,
                           void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Problem pu = unit_problem(p, 64);   // units are the blocks
  int rc = tc_run_summary(pu, W, Wb, nullptr, Mp, Sbuf, stream);
  if (rc == MHLA_OK) rc = tc_run_mix(pu, Wb, Mp, Sbuf, St, zt, stream, /*discard_input=*/true);
  if (rc != MHLA_OK) return rc;
  const auto* st = static_cast<const __nv_bfloat16*>(St);
  return p.d == 64 ? launch_ct_tile<64, 2, false>(p, W, p.M, st, zt, s) : launch_ct_tile<32, 2, false>(p, W, p.M, st, zt, s);
}

bool tc_causal_states_eligible(const Problem& p) { return (p.w == 64 || p.w == 128) && tc_causal_eligible(p); }

size_t tc_causal_states_bytes(const Problem& p) { return ct_layout(p).total; }

int launch_tc_causal_states(const Problem& p, const float* W, void* region, void* stream, CausalStates* out) {
  const CtLayout L = ct_layout(p);   // U = w: the units are the blocks, W' is W's strict lower triangle
  char* ws = static_cast<char*>(region);
  auto* Wu = reinterpret_cast<__nv_bfloat16*>(ws + L.wu_off);
  auto* St = reinterpret_cast<__nv_bfloat16*>(ws + L.st_off);
  auto* zt = reinterpret_cast<float*>(ws + L.zt_off);
  const Problem pu = unit_problem(p, L.U);
  int rc = tc_run_summary(pu, W, Wu, nullptr, L.Mp, ws + L.sbuf_off, stream, static_cast<int32_t>(p.M), 1);
  if (rc == MHLA_OK) rc = tc_run_mix(pu, Wu, L.Mp, ws + L.sbuf_off, St, zt, stream, /*discard_input=*/false);
  out->Sbuf = ws + L.sbuf_off;
  out->St = St;
  out->zt = zt;
  out->Wu = Wu;
  out->Mp = L.Mp;
  return rc;
}

int launch_tc_causal_mix(const Problem& p, const void* Wm, int64_t Mp, const void* Sbuf, void* St, float* zt,
                         void* stream) {
  const CtLayout L = ct_layout(p);
  return tc_run_mix(unit_problem(p, L.U), Wm, Mp, Sbuf, St, zt, stream, /*discard_input=*/true);
}

int read_and_clear_causal_error(void* stream, uint32_t* flags) {
  return read_and_clear_word(g_causal_error, stream, flags);
}

MHLA_DEFINE_STALL_SETTER(set_stall_causal)

}  // namespace mhla
