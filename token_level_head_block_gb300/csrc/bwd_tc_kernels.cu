// Tensor-core backward pass of MHLA on sm_103a (bf16, d in {32, 64}, tokens
// per block a multiple of 128 in whole block rows).
//
// The pages print no backward pass; W is learnable ([P2] "MHLA: Restoring
// Expressivity of Linear Attention via Token-Level Multi-Head", section 4
// "Multi-Head Mixing"; [P1] 171host.com/767426.html, section 7: a 1x1
// convolution's weight), so these kernels form the chain-rule derivatives of
// the forward's three steps in reverse, for L = sum(dout * o):
//
//   (forward summaries and mixing, recomputed by the forward's kernels)
//   tc_bwd_query  per (b, query block i, head group), 128 tokens at a time:
//                 MMA A   [num | den] = phi(Q) [S~ | z~hi z~lo]
//                 epilogue dnum = g / den, dden = -(g . o) / den (CUDA cores)
//                 MMA B   dphi(Q) = [dnum | dden] [S~^T ; z~hi z~lo]
//                 MMA C   [dS~ | dz~] += phi(Q)^T [dnum | dden], over the block
//                 dq = dphi(Q) * [q > 0]; dS~, dz~ go to a buffer laid out like
//                 the forward's summaries, so the forward's mixing GEMM with W^T
//                 turns them into dS, dz
//   tc_dw         dW[i][j] = sum over summary columns of dS~[i][col] S[j][col]:
//                 one GEMM over the 128-column groups, split over CTAs, then a
//                 fixed-order sum of the partial products (deterministic)
//   tc_bwd_key    per (b, source block j, head group), 128 tokens at a time:
//                 MMA D   dv = phi(K) dS
//                 MMA E   dphi(K) = [v | 1 1] [dS^T ; dz hi lo]
//                 dk = dphi(K) * [k > 0]
// phi'(x) is 1 for x > 0 and 0 otherwise; masks come from the raw inputs.
//
// Every wait is bounded; a wait that gives up sets bit 0 of this file's device
// error word and an abort flag, the CTA drains what it issued (bit 1 if that
// drain gives up), releases tensor memory and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "mhla_internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"
#include "tma_host.h"

namespace mhla {

__device__ unsigned int g_bwd_error = 0;

namespace {

using namespace tc;

__device__ __forceinline__ bool bwait(uint64_t* bar, uint32_t parity, volatile uint32_t* abortf) {
  return wait_bounded_on(bar, parity, abortf, &g_bwd_error);
}
__device__ __forceinline__ void bdrain(uint64_t* bar, uint32_t parity) { drain_wait_on(bar, parity, &g_bwd_error); }

// 16-byte unit of a row in a 128-byte-swizzled tile (rows of 128 bytes).
__device__ __forceinline__ int swz128(int row) { return row & 7; }

// ============================================================================
// tc_bwd_query
// ============================================================================
template <int D>
struct BqCfg {
  static constexpr int HP = 128 / D;             // heads per work item
  static constexpr int C = 128;                  // tokens per chunk (MMA M)
  static constexpr int ROWB = D * 2;
  static constexpr int TILE = C * ROWB;          // one head's [128][D] token tile
  static constexpr int HT = HP * TILE;           // all heads of a chunk
  static constexpr uint32_t SBO = 8 * ROWB;
  static constexpr uint32_t LAYOUT = D == 64 ? 2u : 4u;
  static constexpr int ST = D * D * 2;           // one S~ tile (row-major, swizzled like a token tile)
  static constexpr int EXT = C * 128;            // [128][64] 128-byte-swizzled K-extension tile
  static constexpr int ZB = D * 128;             // [D][64] K-extension of S~^T for MMA B
  // shared memory
  static constexpr int QT_OFF = 0;                       // phi(q), HP tiles
  static constexpr int GT_OFF = QT_OFF + HT;             // dout, HP tiles
  static constexpr int DN_OFF = GT_OFF + HT;             // dnum, HP tiles, then DDC; later dq
  static constexpr int DDC_OFF = DN_OFF + HT;            // dden as N columns (MN-major, layout of D)
  static constexpr int DDA_OFF = DDC_OFF + TILE;         // dden as K columns (K-major, 128-byte swizzle)
  static constexpr int SZ_OFF = DDA_OFF + EXT;           // per head: S~ tile, then the z~ N atom
  static constexpr int ZB_OFF = SZ_OFF + HP * 2 * ST;    // per head: z~ K-extension
  static constexpr int ZRAW_OFF = ZB_OFF + HP * ZB;      // z~ float32, HP x D
  static constexpr int MASK_OFF = ZRAW_OFF + HP * D * 4; // [HP][128][D/8] bits of q > 0
  static constexpr int CTRL_OFF = MASK_OFF + HP * C * (D / 8);
  static constexpr size_t SMEM = CTRL_OFF + 128 + 1024;
  static constexpr int ASTR = D == 64 ? 128 : 64;        // TMEM columns per head of MMA A
  static constexpr int CCOL = 256;                       // MMA C accumulator (128 + 16 columns)
  static constexpr int TMEM_COLS = 512;
};
constexpr int kBqThreads = 256;

template <int D>
__global__ void __launch_bounds__(kBqThreads, 1)
tc_bwd_query(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_g,
             const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_st, TcGeom g,
             int32_t G, int64_t n_items, int phi_kind, float eps, const float* __restrict__ zt,
             __nv_bfloat16* __restrict__ dSbuf) {
  using Cfg = BqCfg<D>;
  constexpr int HP = Cfg::HP;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  uint8_t* qt = smem + Cfg::QT_OFF;
  uint8_t* gt = smem + Cfg::GT_OFF;
  uint8_t* dn = smem + Cfg::DN_OFF;
  uint8_t* ddc = smem + Cfg::DDC_OFF;
  uint8_t* dda = smem + Cfg::DDA_OFF;
  uint8_t* sz = smem + Cfg::SZ_OFF;
  uint8_t* zb = smem + Cfg::ZB_OFF;
  float* zraw = reinterpret_cast<float*>(smem + Cfg::ZRAW_OFF);
  uint8_t* mask = smem + Cfg::MASK_OFF;
  uint64_t* bq = reinterpret_cast<uint64_t*>(smem + Cfg::CTRL_OFF);   // q tiles landed
  uint64_t* bg = bq + 1;                                               // dout tiles landed
  uint64_t* bs = bq + 2;                                               // S~, z~ of an item landed
  uint64_t* bm1 = bq + 3;                                              // MMA A complete
  uint64_t* bm2 = bq + 4;                                              // MMA B and C complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bq + 5);
  volatile uint32_t* abortf = tmem_slot + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(bq, 1);
    mbar_init(bg, 1);
    mbar_init(bs, 1);
    mbar_init(bm1, 1);
    mbar_init(bm2, 1);
    *abortf = 0u;
    fence_mbar_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_g);
    prefetch_tmap(&tm_dq);
    prefetch_tmap(&tm_st);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  // The dden and z~ extension tiles: only their first columns are ever written.
  for (int e = tid; e < (Cfg::TILE + Cfg::EXT) / 16; e += kBqThreads)
    reinterpret_cast<uint4*>(ddc)[e] = make_uint4(0u, 0u, 0u, 0u);
  for (int e = tid; e < HP * 2 * Cfg::ST / 16; e += kBqThreads)
    reinterpret_cast<uint4*>(sz)[e] = make_uint4(0u, 0u, 0u, 0u);
  for (int e = tid; e < HP * Cfg::ZB / 16; e += kBqThreads)
    reinterpret_cast<uint4*>(zb)[e] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const uint64_t pol_stream = policy_evict_first();
  const uint64_t pol_keep = policy_evict_last();
  // item -> (grp, i, b), head group fastest
  auto item_coords = [&](int64_t item, int32_t& grp, int32_t& i, int32_t& b) {
    grp = static_cast<int32_t>(item % G);
    const int64_t rest = item / G;
    i = static_cast<int32_t>(rest % g.M);
    b = static_cast<int32_t>(rest / g.M);
  };
  auto issue_tiles = [&](const CUtensorMap* map, uint8_t* dst, uint64_t* bar, int64_t item, int c) {
    int32_t grp, i, b;
    item_coords(item, grp, i, b);
    int32_t x, y, z;
    chunk_coords(g, i, c, b, x, y, z);
    mbar_arrive_expect_tx(bar, Cfg::HT);
#pragma unroll
    for (int hh = 0; hh < HP; ++hh)   // heads >= H read zeros
      tma_load_5d(dst + hh * Cfg::TILE, map, bar, 0, grp * HP + hh, x, y, z, pol_stream);
  };
  auto issue_sz = [&](int64_t item) {
    int32_t grp, i, b;
    item_coords(item, grp, i, b);
    uint32_t bytes = 0;
    for (int hh = 0; hh < HP; ++hh)
      if (grp * HP + hh < g.H) bytes += Cfg::ST + D * 4;
    mbar_arrive_expect_tx(bs, bytes);
    for (int hh = 0; hh < HP; ++hh) {
      const int32_t h = grp * HP + hh;
      if (h >= g.H) continue;
      const int64_t tile = (static_cast<int64_t>(b) * g.H + h) * g.M + i;
      tma_load_2d(sz + hh * 2 * Cfg::ST, &tm_st, bs, 0, static_cast<int32_t>(tile * D), pol_keep);
      bulk_load(zraw + hh * D, zt + tile * D, D * 4, bs, pol_keep);
    }
  };

  // Issued (thread 0) and consumed (every thread) phase counts.
  uint32_t n_q = 0, n_g = 0, n_s = 0, n_m1 = 0, n_m2 = 0;
  uint32_t c_q = 0, c_g = 0, c_s = 0, c_m1 = 0, c_m2 = 0;
  if (tid == 0 && static_cast<int64_t>(blockIdx.x) < n_items) {
    issue_sz(blockIdx.x);
    issue_tiles(&tm_q, qt, bq, blockIdx.x, 0);
    issue_tiles(&tm_g, gt, bg, blockIdx.x, 0);
    n_s = n_q = n_g = 1;
  }
  const bool add_eps = phi_kind == MHLA_PHI_RELU_EPS;
  const __nv_bfloat162 eps2 = __float2bfloat162_rn(eps);
  const int row = 32 * (warp & 3) + lane;      // token row of the chunk = TMEM lane
  const int wg = warp >> 2;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
  bool ok = true;

  for (int64_t item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
    int32_t grp, i, b;
    item_coords(item, grp, i, b);
    // ---- the item's S~ and z~: build the z~ operand pieces
    if (!__syncthreads_and(bwait(bs, c_s & 1u, abortf))) break;
    ++c_s;
    if (tid < HP * D) {
      const int hh = tid / D, r = tid % D;
      const float zv = grp * HP + hh < g.H ? zraw[hh * D + r] : 0.0f;
      const __nv_bfloat16 hi = __float2bfloat16_rn(zv);
      const __nv_bfloat16 lo = __float2bfloat16_rn(zv - __bfloat162float(hi));
      const uint32_t hilo = static_cast<uint32_t>(__bfloat16_as_ushort(hi)) |
                            (static_cast<uint32_t>(__bfloat16_as_ushort(lo)) << 16);
      // MMA A, N atom after S~: row r (K), columns 0, 1 = hi, lo (unit 0 of the row)
      *reinterpret_cast<uint32_t*>(sz + hh * 2 * Cfg::ST + Cfg::ST + r * Cfg::ROWB + swz<D>(r) * 16) = hilo;
      // MMA B, K extension: row r (N), K columns hh = hi, HP + hh = lo
      uint8_t* zrow = zb + hh * Cfg::ZB + r * 128 + swz128(r) * 16;
      *reinterpret_cast<__nv_bfloat16*>(zrow + hh * 2) = hi;
      *reinterpret_cast<__nv_bfloat16*>(zrow + (HP + hh) * 2) = lo;
    }
    fence_proxy_async_smem();
    __syncthreads();

    for (int c = 0; c < g.chunks; ++c) {
      const bool last = c + 1 == g.chunks;
      const int64_t nitem = last ? item + gridDim.x : item;
      const int nc = last ? 0 : c + 1;
      const bool has_next = nitem < n_items;
      // ---- phi in place on the q tiles, and the q > 0 bits
      if (!__syncthreads_and(bwait(bq, c_q & 1u, abortf))) { ok = false; break; }
      ++c_q;
      for (int e = tid; e < Cfg::HT / 16; e += kBqThreads) {
        const int hh = e / (Cfg::TILE / 16), rem = e % (Cfg::TILE / 16);
        const int t = rem / (D / 8), p = rem % (D / 8);
        uint4* ptr = reinterpret_cast<uint4*>(qt) + e;
        const uint4 raw = *ptr;
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
        uint32_t bits = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const __nv_bfloat162 v2 = *reinterpret_cast<const __nv_bfloat162*>(&w[k]);
          bits |= (__low2float(v2) > 0.0f ? 1u : 0u) << (2 * k);
          bits |= (__high2float(v2) > 0.0f ? 1u : 0u) << (2 * k + 1);
        }
        mask[(hh * Cfg::C + t) * (D / 8) + (p ^ swz<D>(t))] = static_cast<uint8_t>(bits);
        *ptr = phi8_packed(raw, add_eps, eps2);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();

      // ---- MMA A: [num | den] = phi(q) [S~ | z~]
      if (tid == 0) {
        bulk_wait_group_read<0>();   // the previous chunk's dq stores have read the dn tiles
        tc_fence_after();
        constexpr uint32_t idesc = idesc_bf16_f32(128, D + 16, /*a K-major*/ false, /*b MN-major*/ true);
#pragma unroll
        for (int hh = 0; hh < HP; ++hh) {
          const uint32_t qa = smem_u32(qt + hh * Cfg::TILE), sb = smem_u32(sz + hh * 2 * Cfg::ST);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            mma_bf16(tmem + hh * Cfg::ASTR, smem_desc(qa + ks * 32, 16, Cfg::SBO, Cfg::LAYOUT),
                     smem_desc(sb + ks * 2 * Cfg::SBO, Cfg::ST, Cfg::SBO, Cfg::LAYOUT), idesc, ks > 0 ? 1u : 0u);
        }
        mma_commit(bm1);
        ++n_m1;
      }
      if (!__syncthreads_and(bwait(bm1, c_m1 & 1u, abortf))) { ok = false; break; }
      ++c_m1;
      if (!__syncthreads_and(bwait(bg, c_g & 1u, abortf))) { ok = false; break; }
      ++c_g;
      tc_fence_after();

      // ---- epilogue 1: dnum = g / den, dden = -(g . o) / den
      for (int hh = wg; hh < HP; hh += 2) {
        const uint32_t tb = lane_base + hh * Cfg::ASTR;
        uint32_t nv[D];
        uint32_t dv2[2];
        if constexpr (D == 64) {
          tmem_ld_x32(tb, *reinterpret_cast<uint32_t(*)[32]>(nv));
          tmem_ld_x32(tb + 32, *reinterpret_cast<uint32_t(*)[32]>(nv + 32));
        } else {
          tmem_ld_x32(tb, *reinterpret_cast<uint32_t(*)[32]>(nv));
        }
        tmem_ld_x1(tb + D, dv2[0]);
        tmem_ld_x1(tb + D + 1, dv2[1]);
        tmem_ld_wait();
        const float den = __uint_as_float(dv2[0]) + __uint_as_float(dv2[1]) + eps;
        // heads past H (zero inputs) contribute exact zeros, whatever eps is
        const float inv = grp * HP + hh < g.H ? 1.0f / den : 0.0f;
        const uint8_t* grow = gt + hh * Cfg::TILE + row * Cfg::ROWB;
        float go = 0.0f;
#pragma unroll
        for (int u = 0; u < D / 8; ++u) {
          const uint4 gr = *reinterpret_cast<const uint4*>(grow + ((u ^ swz<D>(row)) * 16));
          const uint32_t gw[4] = {gr.x, gr.y, gr.z, gr.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const __nv_bfloat162 g2 = *reinterpret_cast<const __nv_bfloat162*>(&gw[k]);
            go = fmaf(__low2float(g2), __uint_as_float(nv[8 * u + 2 * k]), go);
            go = fmaf(__high2float(g2), __uint_as_float(nv[8 * u + 2 * k + 1]), go);
          }
        }
        const float dden = -go * inv * inv;   // -(g . num / den) / den
        uint8_t* drow = dn + hh * Cfg::TILE + row * Cfg::ROWB;
#pragma unroll
        for (int u = 0; u < D / 8; ++u) {
          const uint4 gr = *reinterpret_cast<const uint4*>(grow + ((u ^ swz<D>(row)) * 16));
          const uint32_t gw[4] = {gr.x, gr.y, gr.z, gr.w};
          uint32_t ow[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const __nv_bfloat162 g2 = *reinterpret_cast<const __nv_bfloat162*>(&gw[k]);
            ow[k] = pack_bf16(__low2float(g2) * inv, __high2float(g2) * inv);
          }
          *reinterpret_cast<uint4*>(drow + ((u ^ swz<D>(row)) * 16)) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
        }
        const __nv_bfloat16 ddb = __float2bfloat16_rn(dden);
        // MMA C's B: N column hh of the dden atom (row = token, unit 0 of the row)
        *reinterpret_cast<__nv_bfloat16*>(ddc + row * Cfg::ROWB + swz<D>(row) * 16 + hh * 2) = ddb;
        // MMA B's A: K columns hh and HP + hh (they meet z~ hi and lo)
        uint8_t* arow = dda + row * 128 + swz128(row) * 16;
        *reinterpret_cast<__nv_bfloat16*>(arow + hh * 2) = ddb;
        *reinterpret_cast<__nv_bfloat16*>(arow + (HP + hh) * 2) = ddb;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();

      // ---- MMA B (dphi(q)) and MMA C (dS~, dz~); the dout tiles are free
      if (tid == 0) {
        if (has_next) {
          issue_tiles(&tm_g, gt, bg, nitem, nc);
          ++n_g;
        }
        tc_fence_after();
        constexpr uint32_t idb = idesc_bf16_f32(128, D, /*a K-major*/ false, /*b K-major*/ false);
#pragma unroll
        for (int hh = 0; hh < HP; ++hh) {
          const uint32_t da = smem_u32(dn + hh * Cfg::TILE), sb = smem_u32(sz + hh * 2 * Cfg::ST);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            mma_bf16(tmem + hh * D, smem_desc(da + ks * 32, 16, Cfg::SBO, Cfg::LAYOUT),
                     smem_desc(sb + ks * 32, 16, Cfg::SBO, Cfg::LAYOUT), idb, ks > 0 ? 1u : 0u);
          mma_bf16(tmem + hh * D, smem_desc(smem_u32(dda), 16, 1024, 2),
                   smem_desc(smem_u32(zb + hh * Cfg::ZB), 16, 1024, 2), idb, 1u);
        }
        constexpr uint32_t idc = idesc_bf16_f32(128, 128 + 16, /*a MN-major*/ true, /*b MN-major*/ true);
        const uint32_t qa = smem_u32(qt), da = smem_u32(dn);
#pragma unroll
        for (int ks = 0; ks < Cfg::C / 16; ++ks)
          mma_bf16(tmem + Cfg::CCOL, smem_desc(qa + ks * 2 * Cfg::SBO, Cfg::TILE, Cfg::SBO, Cfg::LAYOUT),
                   smem_desc(da + ks * 2 * Cfg::SBO, Cfg::TILE, Cfg::SBO, Cfg::LAYOUT), idc,
                   (c > 0 || ks > 0) ? 1u : 0u);
        mma_commit(bm2);
        ++n_m2;
      }
      if (!__syncthreads_and(bwait(bm2, c_m2 & 1u, abortf))) { ok = false; break; }
      ++c_m2;
      tc_fence_after();
      if (tid == 0 && has_next) {   // phi(q), S~ and z~ are consumed
        if (last) {
          issue_sz(nitem);
          ++n_s;
        }
        issue_tiles(&tm_q, qt, bq, nitem, nc);
        ++n_q;
      }

      // ---- epilogue 2: dq = dphi(q) * [q > 0] into the dn tiles, then stored
      for (int hh = wg; hh < HP; hh += 2) {
        uint32_t v[D];
        if constexpr (D == 64) {
          tmem_ld_x32(lane_base + hh * D, *reinterpret_cast<uint32_t(*)[32]>(v));
          tmem_ld_x32(lane_base + hh * D + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
        } else {
          tmem_ld_x32(lane_base + hh * D, *reinterpret_cast<uint32_t(*)[32]>(v));
        }
        tmem_ld_wait();
        const uint8_t* mrow = mask + (hh * Cfg::C + row) * (D / 8);
        uint8_t* orow = dn + hh * Cfg::TILE + row * Cfg::ROWB;
#pragma unroll
        for (int u = 0; u < D / 8; ++u) {
          const uint32_t bits = mrow[u];
          uint32_t ow[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float a0 = (bits >> (2 * k)) & 1u ? __uint_as_float(v[8 * u + 2 * k]) : 0.0f;
            const float a1 = (bits >> (2 * k + 1)) & 1u ? __uint_as_float(v[8 * u + 2 * k + 1]) : 0.0f;
            ow[k] = pack_bf16(a0, a1);
          }
          *reinterpret_cast<uint4*>(orow + ((u ^ swz<D>(row)) * 16)) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      if (tid == 0) {
        int32_t x, y, z;
        chunk_coords(g, i, c, b, x, y, z);
        for (int hh = 0; hh < HP; ++hh)
          if (grp * HP + hh < g.H) tma_store_5d(&tm_dq, dn + hh * Cfg::TILE, 0, grp * HP + hh, x, y, z);
        bulk_commit_group();
      }

      // ---- epilogue 3 (after the block's last chunk): dS~ and dz~ to dSbuf
      if (last) {
        // thread: TMEM lane row = (hh, r); warpgroup wg takes half of the d columns
        const int hh = row / D, r = row % D;
        const uint32_t tb = lane_base + Cfg::CCOL + hh * D + wg * (D / 2);
        uint32_t v[D / 2];
        if constexpr (D == 64) {
          tmem_ld_x32(tb, *reinterpret_cast<uint32_t(*)[32]>(v));
        } else {
          tmem_ld_x16(tb, *reinterpret_cast<uint32_t(*)[16]>(v));
        }
        uint32_t vz = 0;
        tmem_ld_x1(lane_base + Cfg::CCOL + 128 + hh, vz);
        tmem_ld_wait();
        const int32_t h = grp * HP + hh;
        if (h < g.H) {
          constexpr int32_t PER_BH = (D + 1) * D;
          const int64_t col = (static_cast<int64_t>(b) * g.H + h) * PER_BH + r * D + wg * (D / 2);
          uint4* drow = reinterpret_cast<uint4*>(dSbuf + ((col >> 7) * g.M + i) * 128 + (col & 127));
#pragma unroll
          for (int q = 0; q < D / 16; ++q)
            drow[q] = make_uint4(pack_bf16(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
                                 pack_bf16(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                                 pack_bf16(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                                 pack_bf16(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
          if (wg == 0) {
            const int64_t zcol = (static_cast<int64_t>(b) * g.H + h) * PER_BH + D * D + r;
            dSbuf[((zcol >> 7) * g.M + i) * 128 + (zcol & 127)] = __float2bfloat16_rn(__uint_as_float(vz));
          }
        }
        tc_fence_before();
        __syncthreads();
      }
    }
  }

  if (tid == 0) {
    bulk_wait_group0();
    if (n_q > c_q) bdrain(bq, (n_q - 1) & 1u);
    if (n_g > c_g) bdrain(bg, (n_g - 1) & 1u);
    if (n_s > c_s) bdrain(bs, (n_s - 1) & 1u);
    if (n_m1 > c_m1) bdrain(bm1, (n_m1 - 1) & 1u);
    if (n_m2 > c_m2) bdrain(bm2, (n_m2 - 1) & 1u);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::TMEM_COLS);
  }
}

// ============================================================================
// tc_bwd_key
// ============================================================================
template <int D>
struct BkCfg {
  static constexpr int HP = 128 / D;
  static constexpr int C = 128;
  static constexpr int ROWB = D * 2;
  static constexpr int TILE = C * ROWB;
  static constexpr int HT = HP * TILE;
  static constexpr uint32_t SBO = 8 * ROWB;
  static constexpr uint32_t LAYOUT = D == 64 ? 2u : 4u;
  static constexpr int ST = D * D * 2;           // one dS tile (row-major, swizzled)
  static constexpr int EXT = C * 128;            // ones K-extension of v: [128][64], 128-byte swizzle
  static constexpr int ZB = D * 128;             // dz K-extension of dS^T: [D][64]
  static constexpr int STAGE = 2 * HT;           // k tiles then v tiles (then dk, dv in place)
  static constexpr int NS = 2;
  static constexpr int ST_OFF = NS * STAGE;
  static constexpr int ONES_OFF = ST_OFF + HP * ST;
  static constexpr int ZB_OFF = ONES_OFF + EXT;
  static constexpr int ZRAW_OFF = ZB_OFF + HP * ZB;
  static constexpr int MASK_OFF = ZRAW_OFF + HP * D * 4;
  static constexpr int MASK_BYTES = HP * C * (D / 8);
  static constexpr int CTRL_OFF = MASK_OFF + NS * MASK_BYTES;
  static constexpr size_t SMEM = CTRL_OFF + 128 + 1024;
  static constexpr int TMEM_COLS = 256;           // per head: dv (D columns), dphi(k) (D columns)
};
constexpr int kBkThreads = 256;

template <int D>
__global__ void __launch_bounds__(kBkThreads, 1)
tc_bwd_key(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
           const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
           const __grid_constant__ CUtensorMap tm_ds, TcGeom g, int32_t G, int64_t n_items, int phi_kind,
           float eps, const float* __restrict__ dz) {
  using Cfg = BkCfg<D>;
  constexpr int HP = Cfg::HP;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  uint8_t* stages = smem;
  uint8_t* dst = smem + Cfg::ST_OFF;
  uint8_t* ones = smem + Cfg::ONES_OFF;
  uint8_t* zb = smem + Cfg::ZB_OFF;
  float* zraw = reinterpret_cast<float*>(smem + Cfg::ZRAW_OFF);
  uint8_t* masks = smem + Cfg::MASK_OFF;
  uint64_t* bl = reinterpret_cast<uint64_t*>(smem + Cfg::CTRL_OFF);   // [2] k, v tiles landed
  uint64_t* bs = bl + 2;                                               // dS, dz of an item landed
  uint64_t* bm = bl + 3;                                               // MMAs complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bl + 4);
  volatile uint32_t* abortf = tmem_slot + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(bl, 1);
    mbar_init(bl + 1, 1);
    mbar_init(bs, 1);
    mbar_init(bm, 1);
    *abortf = 0u;
    fence_mbar_init();
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_dk);
    prefetch_tmap(&tm_dv);
    prefetch_tmap(&tm_ds);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  // ones extension of v (K columns 0, 1 = 1 for every token) and the dz tiles
  for (int e = tid; e < Cfg::EXT / 16; e += kBkThreads) {
    const int r = e / 8, p = e % 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if ((p ^ swz128(r)) == 0) v.x = 0x3F803F80u;   // bf16 1.0, 1.0
    reinterpret_cast<uint4*>(ones)[e] = v;
  }
  for (int e = tid; e < HP * Cfg::ZB / 16; e += kBkThreads)
    reinterpret_cast<uint4*>(zb)[e] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const uint64_t pol_stream = policy_evict_first();
  const uint64_t pol_keep = policy_evict_last();
  auto item_coords = [&](int64_t item, int32_t& grp, int32_t& j, int32_t& b) {
    grp = static_cast<int32_t>(item % G);
    const int64_t rest = item / G;
    j = static_cast<int32_t>(rest % g.M);
    b = static_cast<int32_t>(rest / g.M);
  };
  auto issue_kv = [&](int st, int64_t item, int c) {
    int32_t grp, j, b;
    item_coords(item, grp, j, b);
    int32_t x, y, z;
    chunk_coords(g, j, c, b, x, y, z);
    uint8_t* base = stages + st * Cfg::STAGE;
    mbar_arrive_expect_tx(bl + st, Cfg::STAGE);
#pragma unroll
    for (int hh = 0; hh < HP; ++hh) {
      tma_load_5d(base + hh * Cfg::TILE, &tm_k, bl + st, 0, grp * HP + hh, x, y, z, pol_stream);
      tma_load_5d(base + Cfg::HT + hh * Cfg::TILE, &tm_v, bl + st, 0, grp * HP + hh, x, y, z, pol_stream);
    }
  };
  auto issue_ds = [&](int64_t item) {
    int32_t grp, j, b;
    item_coords(item, grp, j, b);
    uint32_t bytes = 0;
    for (int hh = 0; hh < HP; ++hh)
      if (grp * HP + hh < g.H) bytes += Cfg::ST + D * 4;
    mbar_arrive_expect_tx(bs, bytes);
    for (int hh = 0; hh < HP; ++hh) {
      const int32_t h = grp * HP + hh;
      if (h >= g.H) continue;
      const int64_t tile = (static_cast<int64_t>(b) * g.H + h) * g.M + j;
      tma_load_2d(dst + hh * Cfg::ST, &tm_ds, bs, 0, static_cast<int32_t>(tile * D), pol_keep);
      bulk_load(zraw + hh * D, dz + tile * D, D * 4, bs, pol_keep);
    }
  };

  uint32_t n_l[2] = {0, 0}, n_s = 0, n_m = 0;
  uint32_t c_l[2] = {0, 0}, c_s = 0, c_m = 0;
  uint32_t chunk_no = 0;   // chunks processed by this CTA (stage = chunk_no & 1)
  if (tid == 0 && static_cast<int64_t>(blockIdx.x) < n_items) {
    issue_ds(blockIdx.x);
    issue_kv(0, blockIdx.x, 0);
    n_s = n_l[0] = 1;
  }
  const bool add_eps = phi_kind == MHLA_PHI_RELU_EPS;
  const __nv_bfloat162 eps2 = __float2bfloat162_rn(eps);
  const int row = 32 * (warp & 3) + lane;
  const int wg = warp >> 2;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
  bool ok = true;

  for (int64_t item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
    int32_t grp, j, b;
    item_coords(item, grp, j, b);
    if (!__syncthreads_and(bwait(bs, c_s & 1u, abortf))) break;
    ++c_s;
    if (tid < HP * D) {   // dz hi, lo into K columns 0, 1 of row r of the extension
      const int hh = tid / D, r = tid % D;
      const float zv = grp * HP + hh < g.H ? zraw[hh * D + r] : 0.0f;
      const __nv_bfloat16 hi = __float2bfloat16_rn(zv);
      const __nv_bfloat16 lo = __float2bfloat16_rn(zv - __bfloat162float(hi));
      *reinterpret_cast<uint32_t*>(zb + hh * Cfg::ZB + r * 128 + swz128(r) * 16) =
          static_cast<uint32_t>(__bfloat16_as_ushort(hi)) | (static_cast<uint32_t>(__bfloat16_as_ushort(lo)) << 16);
    }
    fence_proxy_async_smem();
    __syncthreads();

    for (int c = 0; c < g.chunks; ++c, ++chunk_no) {
      const int st = chunk_no & 1;
      uint8_t* kt = stages + st * Cfg::STAGE;
      uint8_t* vt = kt + Cfg::HT;
      uint8_t* mask = masks + st * Cfg::MASK_BYTES;
      const bool last = c + 1 == g.chunks;
      const int64_t nitem = last ? item + gridDim.x : item;
      const int nc = last ? 0 : c + 1;
      const bool has_next = nitem < n_items;
      if (!__syncthreads_and(bwait(bl + st, c_l[st] & 1u, abortf))) { ok = false; break; }
      ++c_l[st];
      // ---- phi in place on the k tiles, and the k > 0 bits
      for (int e = tid; e < Cfg::HT / 16; e += kBkThreads) {
        const int hh = e / (Cfg::TILE / 16), rem = e % (Cfg::TILE / 16);
        const int t = rem / (D / 8), p = rem % (D / 8);
        uint4* ptr = reinterpret_cast<uint4*>(kt) + e;
        const uint4 raw = *ptr;
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
        uint32_t bits = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const __nv_bfloat162 v2 = *reinterpret_cast<const __nv_bfloat162*>(&w[k]);
          bits |= (__low2float(v2) > 0.0f ? 1u : 0u) << (2 * k);
          bits |= (__high2float(v2) > 0.0f ? 1u : 0u) << (2 * k + 1);
        }
        mask[(hh * Cfg::C + t) * (D / 8) + (p ^ swz<D>(t))] = static_cast<uint8_t>(bits);
        *ptr = phi8_packed(raw, add_eps, eps2);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();

      if (tid == 0) {
        tc_fence_after();
        // MMA D: dv = phi(k) dS;  MMA E: dphi(k) = [v | 1 1] [dS^T ; dz hi lo]
        constexpr uint32_t idd = idesc_bf16_f32(128, D, /*a K-major*/ false, /*b MN-major*/ true);
        constexpr uint32_t ide = idesc_bf16_f32(128, D, /*a K-major*/ false, /*b K-major*/ false);
#pragma unroll
        for (int hh = 0; hh < HP; ++hh) {
          const uint32_t ka = smem_u32(kt + hh * Cfg::TILE), va = smem_u32(vt + hh * Cfg::TILE);
          const uint32_t sb = smem_u32(dst + hh * Cfg::ST);
          const uint32_t dvc = tmem + hh * 2 * D, dkc = dvc + D;
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            mma_bf16(dvc, smem_desc(ka + ks * 32, 16, Cfg::SBO, Cfg::LAYOUT),
                     smem_desc(sb + ks * 2 * Cfg::SBO, Cfg::ST, Cfg::SBO, Cfg::LAYOUT), idd, ks > 0 ? 1u : 0u);
            mma_bf16(dkc, smem_desc(va + ks * 32, 16, Cfg::SBO, Cfg::LAYOUT),
                     smem_desc(sb + ks * 32, 16, Cfg::SBO, Cfg::LAYOUT), ide, ks > 0 ? 1u : 0u);
          }
          mma_bf16(dkc, smem_desc(smem_u32(ones), 16, 1024, 2), smem_desc(smem_u32(zb + hh * Cfg::ZB), 16, 1024, 2),
                   ide, 1u);
        }
        mma_commit(bm);
        ++n_m;
        // the other stage: its dk, dv stores must have read it, then the next chunk loads into it
        if (has_next) {
          bulk_wait_group_read<0>();
          issue_kv(st ^ 1, nitem, nc);
          ++n_l[st ^ 1];
        }
      }
      if (!__syncthreads_and(bwait(bm, c_m & 1u, abortf))) { ok = false; break; }
      ++c_m;
      tc_fence_after();
      if (tid == 0 && has_next && last) {   // dS, dz consumed by this item's last MMAs
        issue_ds(nitem);
        ++n_s;
      }

      // ---- epilogue: dv into the v tiles, dk = dphi(k) * [k > 0] into the k tiles
      for (int hh = wg; hh < HP; hh += 2) {
        uint32_t a[D];
        if constexpr (D == 64) {
          tmem_ld_x32(lane_base + hh * 2 * D, *reinterpret_cast<uint32_t(*)[32]>(a));
          tmem_ld_x32(lane_base + hh * 2 * D + 32, *reinterpret_cast<uint32_t(*)[32]>(a + 32));
        } else {
          tmem_ld_x32(lane_base + hh * 2 * D, *reinterpret_cast<uint32_t(*)[32]>(a));
        }
        tmem_ld_wait();
        uint8_t* vrow = vt + hh * Cfg::TILE + row * Cfg::ROWB;
#pragma unroll
        for (int u = 0; u < D / 8; ++u)
          *reinterpret_cast<uint4*>(vrow + ((u ^ swz<D>(row)) * 16)) =
              make_uint4(pack_bf16(__uint_as_float(a[8 * u]), __uint_as_float(a[8 * u + 1])),
                         pack_bf16(__uint_as_float(a[8 * u + 2]), __uint_as_float(a[8 * u + 3])),
                         pack_bf16(__uint_as_float(a[8 * u + 4]), __uint_as_float(a[8 * u + 5])),
                         pack_bf16(__uint_as_float(a[8 * u + 6]), __uint_as_float(a[8 * u + 7])));
        if constexpr (D == 64) {
          tmem_ld_x32(lane_base + hh * 2 * D + D, *reinterpret_cast<uint32_t(*)[32]>(a));
          tmem_ld_x32(lane_base + hh * 2 * D + D + 32, *reinterpret_cast<uint32_t(*)[32]>(a + 32));
        } else {
          tmem_ld_x32(lane_base + hh * 2 * D + D, *reinterpret_cast<uint32_t(*)[32]>(a));
        }
        tmem_ld_wait();
        const uint8_t* mrow = mask + (hh * Cfg::C + row) * (D / 8);
        uint8_t* krow = kt + hh * Cfg::TILE + row * Cfg::ROWB;
#pragma unroll
        for (int u = 0; u < D / 8; ++u) {
          const uint32_t bits = mrow[u];
          uint32_t ow[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float a0 = (bits >> (2 * k)) & 1u ? __uint_as_float(a[8 * u + 2 * k]) : 0.0f;
            const float a1 = (bits >> (2 * k + 1)) & 1u ? __uint_as_float(a[8 * u + 2 * k + 1]) : 0.0f;
            ow[k] = pack_bf16(a0, a1);
          }
          *reinterpret_cast<uint4*>(krow + ((u ^ swz<D>(row)) * 16)) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      if (tid == 0) {
        int32_t x, y, z;
        chunk_coords(g, j, c, b, x, y, z);
        for (int hh = 0; hh < HP; ++hh) {
          if (grp * HP + hh >= g.H) continue;
          tma_store_5d(&tm_dk, kt + hh * Cfg::TILE, 0, grp * HP + hh, x, y, z);
          tma_store_5d(&tm_dv, vt + hh * Cfg::TILE, 0, grp * HP + hh, x, y, z);
        }
        bulk_commit_group();
      }
    }
  }

  if (tid == 0) {
    bulk_wait_group0();
    for (int st = 0; st < 2; ++st)
      if (n_l[st] > c_l[st]) bdrain(bl + st, (n_l[st] - 1) & 1u);
    if (n_s > c_s) bdrain(bs, (n_s - 1) & 1u);
    if (n_m > c_m) bdrain(bm, (n_m - 1) & 1u);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::TMEM_COLS);
  }
}

// ============================================================================
// tc_dw: part[s][i][j] = sum over the column groups of split s of
//        dSbuf[i][col] Sbuf[j][col]   (both [G][M][128] bf16, K-major tiles)
// One CTA per (i tile of 128, j tile of up to 256, split).  Warp 0 loads
// 64-column halves of a group into a 4-stage ring, warp 1 issues the MMAs,
// warps 4-7 write the float32 tile.
// ============================================================================
struct DwCfg {
  static constexpr int IT = 128;                  // rows i per tile (MMA M)
  static constexpr int JT = 256;                  // rows j per tile (MMA N, at most)
  static constexpr int A_BYTES = IT * 128;        // [128][64] K-major, 128-byte swizzle
  static constexpr int B_BYTES = JT * 128;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int NS = 4;
  static constexpr size_t SMEM = static_cast<size_t>(NS) * STAGE + 256 + 1024;
  static constexpr int TMEM_COLS = 256;
};
constexpr int kDwThreads = 256;

__global__ void __launch_bounds__(kDwThreads, 1)
tc_dw(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b, int32_t M, int32_t n_jt,
      int32_t JN, int64_t ngroups, int32_t nsplit, float* __restrict__ part) {
  using Cfg = DwCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::NS * Cfg::STAGE);
  uint64_t* empty = full + Cfg::NS;
  uint64_t* done = empty + Cfg::NS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile uint32_t* abortf = tmem_slot + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int32_t split = static_cast<int32_t>(blockIdx.x % nsplit);
  const int32_t tile = static_cast<int32_t>(blockIdx.x / nsplit);
  const int32_t i0 = (tile / n_jt) * Cfg::IT, j0 = (tile % n_jt) * Cfg::JT;
  const int64_t g0 = ngroups * split / nsplit, g1 = ngroups * (split + 1) / nsplit;
  const int32_t nsteps = static_cast<int32_t>(2 * (g1 - g0));   // 64-column halves
  if (tid == 0) {
    for (int s = 0; s < Cfg::NS; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    mbar_init(done, 1);
    *abortf = 0u;
    fence_mbar_init();
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_b);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t bbytes = static_cast<uint32_t>(JN * 128);

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int s = 0;
      uint32_t ph = 0;
      uint64_t fills = 0;
      for (int32_t st = 0; st < nsteps; ++st) {
        if (!bwait(empty + s, ph ^ 1u, abortf)) break;
        const int32_t grp = static_cast<int32_t>(g0 + st / 2), half = st & 1;
        mbar_arrive_expect_tx(full + s, Cfg::A_BYTES + bbytes);
        uint8_t* base = stages + s * Cfg::STAGE;
        tma_load_3d(base, &tm_a, full + s, half * 64, i0, grp, pol);            // rows i >= M read zeros
        tma_load_3d(base + Cfg::A_BYTES, &tm_b, full + s, half * 64, j0, grp, pol);
        ++fills;
        if (++s == Cfg::NS) { s = 0; ph ^= 1u; }
      }
      for (int st = 0; st < Cfg::NS; ++st) {
        const uint64_t n = fills / Cfg::NS + (static_cast<uint64_t>(st) < fills % Cfg::NS ? 1 : 0);
        if (n > 0) bdrain(full + st, static_cast<uint32_t>((n - 1) & 1));
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, JN, /*a K-major*/ false, /*b K-major*/ false);
      int s = 0;
      uint32_t ph = 0;
      for (int32_t st = 0; st < nsteps; ++st) {
        if (!bwait(full + s, ph, abortf)) break;
        tc_fence_after();
        const uint32_t base = smem_u32(stages + s * Cfg::STAGE);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tmem, smem_desc(base + ks * 32, 16, 1024, 2), smem_desc(base + Cfg::A_BYTES + ks * 32, 16, 1024, 2),
                   idesc, (st > 0 || ks > 0) ? 1u : 0u);
        mma_commit(empty + s);
        if (++s == Cfg::NS) { s = 0; ph ^= 1u; }
      }
      mma_commit(done);
      bdrain(done, 0);
    }
  } else if (warp >= 4) {
    const int q4 = warp & 3;
    const int32_t i = i0 + 32 * q4 + lane;
    const bool ok = __all_sync(0xffffffffu, bwait(done, 0, abortf));
    if (ok) {
      tc_fence_after();
      const uint32_t tb = tmem + (static_cast<uint32_t>(32 * q4) << 16);
      float* prow = part + (static_cast<int64_t>(split) * M + i) * M;
      for (int cc = 0; cc < JN; cc += 32) {
        uint32_t v[32];
        tmem_ld_x32(tb + cc, v);
        tmem_ld_wait();
        if (i < M) {
          if (nsteps == 0) {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = 0u;
          }
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (j0 + cc + e < M) prow[j0 + cc + e] = __uint_as_float(v[e]);
        }
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

// dW = the partial products summed over the splits in a fixed order.
__global__ void tc_dw_reduce(const float* __restrict__ part, float* __restrict__ dW, int64_t MM, int32_t nsplit) {
  const int64_t x = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (x >= MM) return;
  float s = 0.0f;
  for (int32_t k = 0; k < nsplit; ++k) s += part[k * MM + x];
  dW[x] = s;
}

// ----------------------------------------------------------------- host side

struct BwdLayout {
  size_t wb_off, wbt_off, sbuf_off, dsbuf_off, st_off, zt_off, part_off, total;
  int64_t Mp, ngroups;
  int32_t n_it, n_jt, JN, nsplit;
};

// CTAs the dW product is split over (about one per SM of a GB300); a constant,
// so that the workspace size does not depend on the device.
constexpr int64_t kDwTargetCtas = 152;

BwdLayout bwd_layout(const Problem& p) {
  BwdLayout L;
  L.Mp = (p.M + 7) / 8 * 8;
  const int64_t ncols = p.BH() * (p.d + 1) * p.d;
  L.ngroups = (ncols + 127) / 128;
  L.n_it = static_cast<int32_t>((p.M + DwCfg::IT - 1) / DwCfg::IT);
  L.n_jt = static_cast<int32_t>((p.M + DwCfg::JT - 1) / DwCfg::JT);
  L.JN = static_cast<int32_t>(std::min<int64_t>(DwCfg::JT, (p.M + 15) / 16 * 16));
  const int64_t tiles = static_cast<int64_t>(L.n_it) * L.n_jt;
  L.nsplit = static_cast<int32_t>(
      std::max<int64_t>(1, std::min<int64_t>(L.ngroups, (kDwTargetCtas + tiles - 1) / tiles)));
  size_t off = 0;
  L.wb_off = off;
  off += align_up(static_cast<size_t>(p.M) * L.Mp * 2);
  L.wbt_off = off;
  off += align_up(static_cast<size_t>(p.M) * L.Mp * 2);
  L.sbuf_off = off;
  off += align_up(static_cast<size_t>(p.M) * L.ngroups * 128 * 2);
  L.dsbuf_off = off;
  off += align_up(static_cast<size_t>(p.M) * L.ngroups * 128 * 2);
  L.st_off = off;
  off += align_up(static_cast<size_t>(p.BH()) * p.M * p.d * p.d * 2);
  L.zt_off = off;
  off += align_up(static_cast<size_t>(p.BH()) * p.M * p.d * 4);
  L.part_off = off;
  off += align_up(static_cast<size_t>(L.nsplit) * p.M * p.M * 4);
  L.total = off;
  return L;
}

// Row-major [rows][D] bf16 tiles stacked in one tensor: a (D, D) box lands as
// the tile with the swizzle of D (rows of 2 D bytes).
bool tile_rows_map(void* base, int64_t rows, int d, CUtensorMap* m) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d * 2)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(d), static_cast<cuuint32_t>(d)};
  return encode_tensor_map(m, 2, base, dims, strides, box,
                           d == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}

template <int D>
int launch_tc_bwd_d(const Problem& p, const float* W, const BwdOperands& bo, void* workspace, cudaStream_t stream) {
  const int sms = device_sm_count();
  if (sms <= 0) return MHLA_ERR_CUDA;
  const BwdLayout L = bwd_layout(p);
  char* ws = static_cast<char*>(workspace);
  void* Wb = ws + L.wb_off;
  void* WbT = ws + L.wbt_off;
  void* Sbuf = ws + L.sbuf_off;
  auto* dSbuf = reinterpret_cast<__nv_bfloat16*>(ws + L.dsbuf_off);
  auto* St = reinterpret_cast<__nv_bfloat16*>(ws + L.st_off);
  auto* zt = reinterpret_cast<float*>(ws + L.zt_off);
  auto* part = reinterpret_cast<float*>(ws + L.part_off);
  ChunkPlan c128;
  if (!chunk_plan(p, 128, &c128)) return MHLA_ERR_UNSUPPORTED;
  const TcGeom geo = make_geom(p, c128);
  const int32_t G = static_cast<int32_t>((p.H + 128 / D - 1) / (128 / D));
  const int64_t n_items = p.B * G * p.M;

  // b1: summaries (with W, W^T in bf16) and the mixing, as in the forward
  int rc = tc_run_summary(p, W, Wb, WbT, L.Mp, Sbuf, stream);
  if (rc == MHLA_OK) rc = tc_run_mix(p, Wb, L.Mp, Sbuf, St, zt, stream);
  if (rc != MHLA_OK) return rc;

  // b2: query blocks
  {
    using Cfg = BqCfg<D>;
    CUtensorMap tq, tg, tdq, tst;
    if (!operand_map(p, p.q, c128.box_y, c128.box_t, &tq) || !operand_map(p, bo.dout, c128.box_y, c128.box_t, &tg) ||
        !operand_map(p, bo.dq, c128.box_y, c128.box_t, &tdq) || !tile_rows_map(St, p.BH() * p.M * D, D, &tst))
      return MHLA_ERR_CUDA;
    if (cudaFuncSetAttribute(tc_bwd_query<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(Cfg::SMEM)) != cudaSuccess)
      return MHLA_ERR_CUDA;
    const int grid = static_cast<int>(std::min<int64_t>(n_items, sms));
    KernelTimer timer("tc_bwd_query", stream);
    tc_bwd_query<D><<<grid, kBqThreads, Cfg::SMEM, stream>>>(tq, tg, tdq, tst, geo, G, n_items, p.phi_kind, p.eps,
                                                             zt, dSbuf);
    if (cudaGetLastError() != cudaSuccess) return MHLA_ERR_CUDA;
  }
  // b3: dW from dS~ and S, then dS = W^T dS~ (into the S~ buffers)
  {
    CUtensorMap ta, tb;
    const cuuint64_t dims[3] = {128u, static_cast<cuuint64_t>(p.M), static_cast<cuuint64_t>(L.ngroups)};
    const cuuint64_t strides[2] = {256u, static_cast<cuuint64_t>(p.M * 256)};
    const cuuint32_t abox[3] = {64u, static_cast<cuuint32_t>(DwCfg::IT), 1u};
    const cuuint32_t bbox[3] = {64u, static_cast<cuuint32_t>(L.JN), 1u};
    if (!encode_tensor_map(&ta, 3, dSbuf, dims, strides, abox, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map(&tb, 3, Sbuf, dims, strides, bbox, CU_TENSOR_MAP_SWIZZLE_128B))
      return MHLA_ERR_CUDA;
    if (cudaFuncSetAttribute(tc_dw, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(DwCfg::SMEM)) !=
        cudaSuccess)
      return MHLA_ERR_CUDA;
    const int64_t ctas = static_cast<int64_t>(L.n_it) * L.n_jt * L.nsplit;
    {
      KernelTimer timer("tc_dw", stream);
      tc_dw<<<static_cast<unsigned>(ctas), kDwThreads, DwCfg::SMEM, stream>>>(
          ta, tb, static_cast<int32_t>(p.M), L.n_jt, L.JN, L.ngroups, L.nsplit, part);
      if (cudaGetLastError() != cudaSuccess) return MHLA_ERR_CUDA;
      const int64_t MM = p.M * p.M;
      tc_dw_reduce<<<static_cast<unsigned>((MM + 255) / 256), 256, 0, stream>>>(part, bo.dW, MM, L.nsplit);
      if (cudaGetLastError() != cudaSuccess) return MHLA_ERR_CUDA;
    }
    rc = tc_run_mix(p, WbT, L.Mp, dSbuf, St, zt, stream);
    if (rc != MHLA_OK) return rc;
  }
  // b4: source blocks
  {
    using Cfg = BkCfg<D>;
    CUtensorMap tk, tv, tdk, tdv, tds;
    if (!operand_map(p, p.k, c128.box_y, c128.box_t, &tk) || !operand_map(p, p.v, c128.box_y, c128.box_t, &tv) ||
        !operand_map(p, bo.dk, c128.box_y, c128.box_t, &tdk) || !operand_map(p, bo.dv, c128.box_y, c128.box_t, &tdv) ||
        !tile_rows_map(St, p.BH() * p.M * D, D, &tds))
      return MHLA_ERR_CUDA;
    if (cudaFuncSetAttribute(tc_bwd_key<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(Cfg::SMEM)) != cudaSuccess)
      return MHLA_ERR_CUDA;
    const int grid = static_cast<int>(std::min<int64_t>(n_items, sms));
    KernelTimer timer("tc_bwd_key", stream);
    tc_bwd_key<D><<<grid, kBkThreads, Cfg::SMEM, stream>>>(tk, tv, tdk, tdv, tds, geo, G, n_items, p.phi_kind, p.eps,
                                                           zt);
    if (cudaGetLastError() != cudaSuccess) return MHLA_ERR_CUDA;
  }
  return MHLA_OK;
}

}  // namespace

bool tc_bwd_eligible(const Problem& p, const BwdOperands& bo) {
  if (!tc_eligible(p)) return false;
  for (const Operand* o : {&bo.dout, &bo.dq, &bo.dk, &bo.dv})
    if (!operand_tma_ok(p, *o)) return false;
  return p.BH() * p.M * p.d < (int64_t{1} << 31);
}

size_t tc_bwd_workspace_bytes(const Problem& p) { return bwd_layout(p).total; }

int launch_tc_bwd(const Problem& p, const float* W, const BwdOperands& bo, void* workspace, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.d == 64) return launch_tc_bwd_d<64>(p, W, bo, workspace, s);
  return launch_tc_bwd_d<32>(p, W, bo, workspace, s);
}

int read_and_clear_bwd_error(void* stream, uint32_t* flags) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int host = 0;
  if (cudaMemcpyFromSymbolAsync(&host, g_bwd_error, sizeof(host), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MHLA_ERR_CUDA;
  const unsigned int zero = 0;
  if (cudaMemcpyToSymbolAsync(g_bwd_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return MHLA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MHLA_ERR_CUDA;
  *flags = host;
  return host ? MHLA_ERR_TIMEOUT : MHLA_OK;
}

}  // namespace mhla
