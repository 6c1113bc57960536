// The three warp-specialised pipelines of the tensor-core MHLA forward as device
// functions, shared by the separate launches (tc_summary.cu, tc_mix.cu,
// tc_output.cu) and the single persistent launch of tc_fused.cu:
//
//   summary  [S_j | z_j] = phi(K_j)^T [V_j | 1] per (b, head group, block j)
//            ([P2] "MHLA: Restoring Expressivity of Linear Attention via
//            Token-Level Multi-Head", section 4 "Architecture": local key-value
//            summaries; [P1] 171host.com/767426.html, section 7, MHLA.forward:
//            kv = k^T v, k_sum);
//   mixing   S~ = W . S over the source blocks for every (b, h) at once ([P2]
//            section 4 "Multi-Head Mixing"; [P1] section 7: piece_attn, a 1x1
//            convolution over the block axis);
//   readout  o_t = phi(q_t) S~_i / (phi(q_t) . z~_i + eps) per (b, h, block i)
//            ([P2] section 4 "Token-Level Adaptivity"; [P1] section 5(4) and
//            section 7, MHLA.forward).
//
// Each pipeline has three parts: *_bars carves its mbarriers out of a control
// region, *_init initialises them (one thread), *_roles runs the warp roles.
// A caller initialises, fences, synchronises the CTA and then calls *_roles
// from every thread; warps a pipeline does not use return at once.
//
// Hooks of the fused launch (null or false in the separate launches):
//   - the summary epilogue raises a per-batch counter after each item's stores;
//   - the mixing producer waits for the summaries of a tile's batches before
//     loading them, takes W from shared memory the caller filled, and its
//     epilogue raises a per-batch counter after each tile's stores;
//   - the readout takes its items from a global queue (a ring in shared memory
//     hands them to every role in the same order) and its S~ producer waits for
//     the mixing of an item's batch.
// Counters are raised with release semantics after a proxy fence and read with
// acquire semantics followed by a proxy fence, so the TMA and bulk copies of
// the reading CTA see the generic stores of the writing CTA.  Every wait is
// bounded (time and poll count): one that gives up raises the CTA's abort flag
// (the other roles stop waiting too) and sets bit 0 of the caller's error word;
// the producers then drain their copies in flight.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mhla_internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace mhla {
namespace tc {

// Publishes a warp's global stores to other CTAs through a counter (every lane
// fences; lane 0 adds): the writer's half of the fused launch's dependencies.
static __device__ __forceinline__ void warp_publish(uint32_t* counter, uint32_t lane) {
  fence_proxy_async_global();
  __threadfence();
  __syncwarp();
  if (lane == 0) red_release_gpu_add(counter, 1u);
}

// ============================================================================
// summary
// Work item = (b, j, head group) with the head group fastest, so the CTAs that
// fetch the other heads of the same tokens run side by side.  Roles: warp 0
// TMA producer, warp 1 MMA issuer, warps 2-5 phi on K, warps 6-9 epilogue.
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
  static constexpr int NV = 128;                     // value columns of the MMA
  static constexpr int NZ = 16;                      // then the ones tile's columns (column 0: z)
  static constexpr int ACC_STRIDE = 256;             // TMEM columns between accumulators
  static constexpr int TMEM_COLS = 512;
  // A shared ones tile with six stages (the z columns as a second MMA) was
  // measured 3.5 us slower on DiT-S/2 than a ones tile in each of five stages.
  static constexpr size_t DATA = static_cast<size_t>(NS) * STAGE;
  static constexpr int WARPS = 10;
};

struct SumBars {
  uint64_t *full, *phid, *empty, *tfull, *tempty, *fin;
};

template <int D>
__device__ __forceinline__ SumBars sum_bars(uint8_t* ctrl) {
  constexpr int NS = SumCfg<D>::NS;
  SumBars b;
  b.full = reinterpret_cast<uint64_t*>(ctrl);
  b.phid = b.full + NS;
  b.empty = b.phid + NS;
  b.tfull = b.empty + NS;
  b.tempty = b.tfull + 2;
  b.fin = b.tempty + 2;
  return b;
}

template <int D>
__device__ __forceinline__ void sum_init(const SumBars& b) {
  for (int s = 0; s < SumCfg<D>::NS; ++s) {
    mbar_init(b.full + s, 1);
    mbar_init(b.phid + s, 128);
    mbar_init(b.empty + s, 1);
  }
  for (int a = 0; a < 2; ++a) {
    mbar_init(b.tfull + a, 1);
    mbar_init(b.tempty + a, 128);
  }
  mbar_init(b.fin, 1);
}

// Constant ones operand of every stage: row t holds (1, 0, ..., 0), so the MMA
// column that reads it sums phi(k) over the tokens: z_j.  Every thread of the
// CTA takes a share; the caller fences the async proxy afterwards.
template <int D>
__device__ __forceinline__ void sum_fill_ones(uint8_t* stages, int tid, int nthreads) {
  using Cfg = SumCfg<D>;
  for (int idx = tid; idx < Cfg::NS * Cfg::C * (D / 8); idx += nthreads) {
    const int s = idx / (Cfg::C * (D / 8));
    const int rem = idx % (Cfg::C * (D / 8));
    const int row = rem / (D / 8), phys = rem % (D / 8);
    const int logical = phys ^ swz<D>(row);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (logical == 0) v.x = 0x3F80u;   // bf16 1.0 in the low half
    *reinterpret_cast<uint4*>(stages + s * Cfg::STAGE + 2 * Cfg::HP * Cfg::TILE + row * Cfg::ROWB + phys * 16) = v;
  }
}

// Items first, first + stride, ... below n_items.  done (fused launch): per
// batch counter raised once per epilogue warp and item after its stores.
template <int D>
__device__ __forceinline__ void summary_roles(const CUtensorMap* tm_k, const CUtensorMap* tm_v, const TcGeom& g,
                                              int32_t G, int64_t first, int64_t stride, int64_t n_items,
                                              int phi_kind, float eps, __nv_bfloat16* __restrict__ Sbuf,
                                              uint8_t* stages, const SumBars& bars, uint32_t tmem,
                                              volatile uint32_t* abortf, unsigned int* err, uint32_t* done) {
  using Cfg = SumCfg<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int s = 0;
      uint32_t ph = 0;
      uint64_t fills = 0;
      bool ok = true;
      for (int64_t item = first; ok && item < n_items; item += stride) {
        const uint32_t it32 = static_cast<uint32_t>(item), rest = it32 / static_cast<uint32_t>(G);
        const int32_t grp = static_cast<int32_t>(it32 - rest * static_cast<uint32_t>(G));
        const int32_t j = static_cast<int32_t>(rest % static_cast<uint32_t>(g.M));
        const int32_t b = static_cast<int32_t>(rest / static_cast<uint32_t>(g.M));
        for (int c = 0; c < g.chunks; ++c) {
          if (!wait_bounded_on(bars.empty + s, ph ^ 1u, abortf, err)) { ok = false; break; }
          mbar_arrive_expect_tx(bars.full + s, Cfg::LOADB);
          int32_t x, y, z;
          chunk_coords(g, j, c, b, x, y, z);
          uint8_t* st = stages + s * Cfg::STAGE;
#pragma unroll
          for (int hh = 0; hh < Cfg::HP; ++hh) {
            const int32_t h = grp * Cfg::HP + hh;   // h >= H reads zeros (out of bounds)
            tma_load_5d(st + hh * Cfg::TILE, tm_k, bars.full + s, 0, h, x, y, z, pol);
            tma_load_5d(st + (Cfg::HP + hh) * Cfg::TILE, tm_v, bars.full + s, 0, h, x, y, z, pol);
          }
          ++fills;
          if (++s == Cfg::NS) { s = 0; ph ^= 1u; }
        }
      }
      // Every fill must have landed before the CTA's shared memory is reused.
      for (int st = 0; st < Cfg::NS; ++st) {
        const uint64_t n = fills / Cfg::NS + (static_cast<uint64_t>(st) < fills % Cfg::NS ? 1 : 0);
        if (n > 0) drain_wait_on(bars.full + st, static_cast<uint32_t>((n - 1) & 1), err);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_v = idesc_bf16_f32(128, Cfg::NV + Cfg::NZ, true, true);
      int s = 0;
      uint32_t ph = 0, local = 0;
      bool ok = true;
      for (int64_t item = first; ok && item < n_items; item += stride, ++local) {
        const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
        if (!wait_bounded_on(bars.tempty + acc, aph ^ 1u, abortf, err)) break;
        tc_fence_after();
        const uint32_t dt = tmem + acc * Cfg::ACC_STRIDE;
        for (int c = 0; c < g.chunks; ++c) {
          if (!wait_bounded_on(bars.phid + s, ph, abortf, err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t base = smem_u32(stages + s * Cfg::STAGE);
#pragma unroll
          for (int ks = 0; ks < Cfg::C / 16; ++ks) {
            // columns 0..127: phi(K)^T V of every head pair; 128..143: phi(K)^T ones
            const uint64_t a = smem_desc(base + ks * 2 * Cfg::SBO, Cfg::TILE, Cfg::SBO, Cfg::LAYOUT);
            const uint64_t bv =
                smem_desc(base + Cfg::HP * Cfg::TILE + ks * 2 * Cfg::SBO, Cfg::TILE, Cfg::SBO, Cfg::LAYOUT);
            mma_bf16(dt, a, bv, idesc_v, (c | ks) != 0 ? 1u : 0u);
          }
          mma_commit(bars.empty + s);
          if (++s == Cfg::NS) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        mma_commit(bars.tfull + acc);
      }
      mma_commit(bars.fin);
      drain_wait_on(bars.fin, 0, err);
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
    for (int64_t item = first; ok && item < n_items; item += stride) {
      for (int c = 0; c < g.chunks; ++c) {
        if (!warp_wait_on(bars.full + s, ph, abortf, err)) { ok = false; break; }
        uint8_t* base = head_tile + s * Cfg::STAGE;
#pragma unroll
        for (int m = 0; m < Cfg::C / 8; ++m) {
          uint4* ptr = reinterpret_cast<uint4*>(base + m * 8 * Cfg::ROWB);
          *ptr = phi8_packed(*ptr, add_eps, eps2);
        }
        fence_proxy_async_smem();
        mbar_arrive(bars.phid + s);
        if (++s == Cfg::NS) { s = 0; ph ^= 1u; }
      }
    }
  } else if (warp < Cfg::WARPS) {
    // ---------------------------------------------------------- epilogue
    const int q4 = warp & 3;
    const int row = 32 * q4 + lane;          // TMEM lane = channel row of head hh
    const int hh = row / D, r = row % D;
    uint32_t local = 0;
    for (int64_t item = first; item < n_items; item += stride, ++local) {
      const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
      if (!warp_wait_on(bars.tfull + acc, aph, abortf, err)) break;
      tc_fence_after();
      const uint32_t tb = tmem + acc * Cfg::ACC_STRIDE + (static_cast<uint32_t>(32 * q4) << 16);
      uint32_t v0[32], v1[32], vz[16];
      tmem_ld_x32(tb + hh * D, v0);
      if (D == 64) tmem_ld_x32(tb + hh * D + 32, v1);
      tmem_ld_x16(tb + 128, vz);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(bars.tempty + acc);
      const uint32_t it32 = static_cast<uint32_t>(item), rest = it32 / static_cast<uint32_t>(G);
      const int32_t grp = static_cast<int32_t>(it32 - rest * static_cast<uint32_t>(G));
      const int32_t j = static_cast<int32_t>(rest % static_cast<uint32_t>(g.M));
      const int32_t b = static_cast<int32_t>(rest / static_cast<uint32_t>(g.M));
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
      if (done) warp_publish(done + b, lane);
    }
  }
}

// ============================================================================
// mixing, M <= 256: all of W (bf16) resident in shared memory, computed
// transposed: D[col][i] = sum_j Sbuf[j][col] W[i][j].  One tile = 128 Sbuf
// columns (MMA M, the TMEM lanes) x all query blocks (MMA N <= 256): per 16
// source blocks a single 128 x N x 16 MMA, A = the Sbuf chunk as it landed
// (MN-major), B = W (K-major).  With the columns on TMEM lanes, the 32 lanes of
// an epilogue warp hold 32 consecutive columns of one query block, so each
// store writes 64 contiguous bytes of S~ (or 128 of z~).  Two accumulator sets
// alternate between tiles; both epilogue warpgroups drain every tile, each half
// of the query blocks.  Roles: warp 0 TMA producer, warp 1 MMA issuer, warps
// 2-9 epilogue.
// ============================================================================
template <int NS_>
struct MixResCfg {
  static constexpr int COLS = 128;                // Sbuf columns per tile (MMA M)
  static constexpr int NMAX = 256;                // query blocks (MMA N, at most)
  static constexpr int KC = 64;                   // source blocks per stage
  static constexpr int W_CHUNK = NMAX * KC * 2;   // W rows i for 64 source blocks, K-major
  static constexpr int W_BYTES = 4 * W_CHUNK;     // up to 256 x 256
  static constexpr int STAGE = KC * COLS * 2;     // Sbuf chunk: two 64-column MN-major halves
  static constexpr int NS = NS_;
  static constexpr int SET = NMAX;                // TMEM columns of one accumulator set
  static constexpr int TMEM_COLS = 512;
  static constexpr size_t DATA = static_cast<size_t>(W_BYTES) + static_cast<size_t>(NS) * STAGE;
  static constexpr int WARPS = 10;
};

struct MixBars {
  uint64_t *full, *empty, *tfull, *tempty, *wfull, *fin;
};

template <int NS>
__device__ __forceinline__ MixBars mix_bars(uint8_t* ctrl) {
  MixBars b;
  b.full = reinterpret_cast<uint64_t*>(ctrl);
  b.empty = b.full + NS;
  b.tfull = b.empty + NS;
  b.tempty = b.tfull + 2;
  b.wfull = b.tempty + 2;
  b.fin = b.wfull + 1;
  return b;
}

template <int NS>
__device__ __forceinline__ void mix_init(const MixBars& b) {
  for (int s = 0; s < NS; ++s) {
    mbar_init(b.full + s, 1);
    mbar_init(b.empty + s, 1);
  }
  for (int a = 0; a < 2; ++a) {
    mbar_init(b.tfull + a, 1);
    mbar_init(b.tempty + a, 256);
  }
  mbar_init(b.wfull, 1);
  mbar_init(b.fin, 1);
}

// W (float32 [M][M], row i = query block) rounded to bf16 into the resident
// operand as TMA would have placed it: per chunk of 64 source blocks, row i is
// 128 bytes of W[i][64 kc .. 64 kc + 63], 16-byte units XOR-swizzled by i mod 8;
// rows i >= M and source blocks j >= M hold zeros.  Every thread of the CTA
// takes a share; the caller fences the async proxy afterwards.
template <int NS>
__device__ __forceinline__ void mix_fill_w(uint8_t* wres, const float* __restrict__ W, int32_t M, int32_t NP,
                                           int tid, int nthreads) {
  const int nk = (M + 63) / 64;
  const int units = nk * NP * 8;                    // 16-byte units of the operand
  for (int u = tid; u < units; u += nthreads) {
    const int kc = u / (NP * 8), rem = u % (NP * 8);
    const int i = rem / 8, c = rem % 8;              // logical unit c: source blocks 64 kc + 8 c ..
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j0 = 64 * kc + 8 * c + 2 * e;
      const float a = (i < M && j0 < M) ? W[static_cast<int64_t>(i) * M + j0] : 0.0f;
      const float b = (i < M && j0 + 1 < M) ? W[static_cast<int64_t>(i) * M + j0 + 1] : 0.0f;
      w[e] = pack_bf16(a, b);
    }
    *reinterpret_cast<uint4*>(wres + static_cast<size_t>(kc) * NP * 128 + i * 128 + ((c ^ (i & 7)) * 16)) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Dependencies of the fused launch: tile t covers columns [128 t, 128 t + 128)
// of Sbuf, i.e. the batches per_b_cols-wide column ranges it touches.
struct MixDeps {
  const uint32_t* sum_done;   // per batch; null: none (a separate launch)
  uint32_t sum_target;        // per batch
  uint32_t* mix_done;         // per batch, raised once per epilogue warp and tile
  int64_t per_b_cols;         // Sbuf columns of one batch: H (d + 1) d
};

template <int NS, int D>
__device__ __forceinline__ void mix_roles(const CUtensorMap* tm_w, const CUtensorMap* tm_s, int32_t M, int32_t NP,
                                          int64_t ncols, int64_t first, int64_t stride, int64_t n_tiles,
                                          __nv_bfloat16* __restrict__ St, float* __restrict__ zt,
                                          const __nv_bfloat16* discard_s, uint8_t* smem, const MixBars& bars,
                                          uint32_t tmem, volatile uint32_t* abortf, unsigned int* err,
                                          const MixDeps& dep) {
  using Cfg = MixResCfg<NS>;
  uint8_t* wres = smem;                                  // [k chunk] W rows i, K-major
  uint8_t* stages = smem + Cfg::W_BYTES;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = (M + Cfg::KC - 1) / Cfg::KC;           // 1..4 source chunks
  const uint32_t wchunk = static_cast<uint32_t>(NP) * Cfg::KC * 2;
  const bool w_resident = tm_w == nullptr;               // W already in shared memory
  const int64_t last_col = ncols - 1;
  if (warp == 0) {
    if (lane == 0) {
      if (!dep.sum_done) grid_dep_wait();   // separate launch: W in bf16 and Sbuf come from the summary launch
      const uint64_t pol_w = policy_evict_last();
      const uint64_t pol_s = policy_evict_first();
      if (!w_resident) {
        // all of W once: chunk kc holds rows i < NP (rows >= M read as zeros) of source blocks kc*64 ..
        mbar_arrive_expect_tx(bars.wfull, static_cast<uint32_t>(nk) * wchunk);
        for (int kc = 0; kc < nk; ++kc) tma_load_2d(wres + kc * wchunk, tm_w, bars.wfull, kc * Cfg::KC, 0, pol_w);
      }
      int s = 0;
      uint32_t ph = 0;
      uint64_t fills = 0;
      bool ok = true;
      int64_t ready_to = -1;                             // summaries of batches <= ready_to are complete
      for (int64_t t = first; ok && t < n_tiles; t += stride) {
        if (dep.sum_done) {
          const int64_t b_hi = min(t * Cfg::COLS + Cfg::COLS - 1, last_col) / dep.per_b_cols;
          for (int64_t b = max(ready_to + 1, t * Cfg::COLS / dep.per_b_cols); ok && b <= b_hi; ++b)
            ok = wait_counter_on(dep.sum_done + b, dep.sum_target, abortf, err);
          if (!ok) break;
          ready_to = max(ready_to, b_hi);
        }
        for (int kc = 0; kc < nk; ++kc) {
          if (!wait_bounded_on(bars.empty + s, ph ^ 1u, abortf, err)) { ok = false; break; }
          mbar_arrive_expect_tx(bars.full + s, Cfg::STAGE);
          uint8_t* st = stages + s * Cfg::STAGE;
          // one 128-column group of Sbuf, rows j contiguous; rows j >= M read as zeros
          tma_load_3d(st, tm_s, bars.full + s, 0, kc * Cfg::KC, static_cast<int32_t>(t), pol_s);
          tma_load_3d(st + Cfg::STAGE / 2, tm_s, bars.full + s, 64, kc * Cfg::KC, static_cast<int32_t>(t), pol_s);
          ++fills;
          if (++s == Cfg::NS) { s = 0; ph ^= 1u; }
        }
      }
      if (!w_resident) drain_wait_on(bars.wfull, 0, err);
      for (int st = 0; st < Cfg::NS; ++st) {
        const uint64_t n = fills / Cfg::NS + (static_cast<uint64_t>(st) < fills % Cfg::NS ? 1 : 0);
        if (n > 0) drain_wait_on(bars.full + st, static_cast<uint32_t>((n - 1) & 1), err);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(Cfg::COLS, NP, /*a MN-major*/ true, /*b K-major*/ false);
      int s = 0;
      uint32_t ph = 0, local = 0;
      bool ok = w_resident || wait_bounded_on(bars.wfull, 0, abortf, err);
      tc_fence_after();
      const uint32_t wbase = smem_u32(wres);
      for (int64_t t = first; ok && t < n_tiles; t += stride, ++local) {
        const uint32_t set = local & 1u, sph = (local >> 1) & 1u;
        if (!wait_bounded_on(bars.tempty + set, sph ^ 1u, abortf, err)) break;
        tc_fence_after();
        for (int kc = 0; kc < nk; ++kc) {
          if (!wait_bounded_on(bars.full + s, ph, abortf, err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t base = smem_u32(stages + s * Cfg::STAGE);
#pragma unroll
          for (int ks = 0; ks < Cfg::KC / 16; ++ks) {
            const uint64_t a = smem_desc(base + ks * 2048, Cfg::STAGE / 2, 1024, 2);
            const uint64_t b = smem_desc(wbase + kc * wchunk + ks * 32, 16, 1024, 2);
            mma_bf16(tmem + set * Cfg::SET, a, b, idesc, (kc | ks) != 0 ? 1u : 0u);
          }
          mma_commit(bars.empty + s);
          if (++s == Cfg::NS) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        mma_commit(bars.tfull + set);
      }
      mma_commit(bars.fin);
      drain_wait_on(bars.fin, 0, err);
    }
  } else if (warp < Cfg::WARPS) {
    // warpgroup wg (warps 2-5 or 6-9) drains query blocks [128 wg, 128 wg + 128) of every tile
    constexpr int32_t PER_BH = (D + 1) * D;            // Sbuf columns of one (b, h): d rows of S, then z
    const int wg = (warp - 2) >> 2;
    const int q4 = warp & 3;
    const int i_lo = wg * 128, i_hi = min(M, i_lo + 128);
    uint32_t local = 0;
    for (int64_t t = first; t < n_tiles; t += stride, ++local) {
      const uint32_t set = local & 1u, sph = (local >> 1) & 1u;
      if (!warp_wait_on(bars.tfull + set, sph, abortf, err)) break;
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
      mbar_arrive(bars.tempty + set);
      if (dep.mix_done) {
        const int64_t b_lo = t * Cfg::COLS / dep.per_b_cols;
        const int64_t b_hi = min(t * Cfg::COLS + Cfg::COLS - 1, last_col) / dep.per_b_cols;
        for (int64_t b = b_lo; b <= b_hi; ++b) warp_publish(dep.mix_done + b, lane);
      }
      // every MMA of tile t is done: its 128-column group of Sbuf (read exactly
      // once, by this CTA) leaves L2 without a write-back when the caller allows
      if (discard_s) {
        const uint8_t* grp = reinterpret_cast<const uint8_t*>(discard_s + t * static_cast<int64_t>(M) * 128);
        for (int e = (warp - 2) * 32 + lane; e < 2 * M; e += 256) discard_l2_line(grp + e * 128);
      }
    }
  }
}

// ============================================================================
// readout
// Work item = (b, i, h) with the head fastest, so neighbouring CTAs read the
// neighbouring 128-byte head rows of the same tokens at about the same time.
// One MMA per 16 channels gives numerator and denominator together:
//   D[t][0..d)  = phi(q_t) S~_i                   (B columns 0..d-1: S~_i)
//   D[t][d]     = phi(q_t) . hi(z~_i)             (B column d:   z~_i rounded to bf16)
//   D[t][d+1]   = phi(q_t) . (z~_i - hi(z~_i))    (B column d+1: the rounding remainder)
// so the float32 denominator keeps about 16 bits more than a bf16 z~ would.
//
// The pipeline streams q at the rate HBM allows only if enough loads are in
// flight: under full load a q chunk takes several microseconds to arrive, so
// shared memory goes almost entirely to q stages.  The output of a chunk is
// written back into its own q stage (the MMA has consumed it by then) and
// stored from there; the S~_i tiles, one per work item, have their own small
// ring fed by a second producer warp.  Roles: warp 0 q producer, warp 1 MMA
// issuer, warps 2-5 phi on q (and the z~ columns of B), warps 6-13 two
// epilogue warpgroups taking alternate chunks, warp 14 S~ producer, warp 15
// store issuer.
//
// PAIR (D = 64 only): each 64-channel row is two adjacent heads of 32 channels
// (heads 2h', 2h' + 1 as one "head" h' of the TMA view), so q and o move in
// 128-byte rows; the B operand is block-diagonal, [S~_a 0; 0 S~_b], with z~_a
// hi, lo in columns 64, 65 for the rows of head a and z~_b in 66, 67 for the rows
// of head b, and each half of the output row takes its own denominator.
// ============================================================================
template <int D>
struct OutCfg {
  static constexpr int C = 128;                 // tokens per chunk = MMA M
  static constexpr int N = D + 16;              // S~ columns + the two z~ columns (+ 14 unused)
  static constexpr int ROWB = D * 2;
  static constexpr int QT = C * ROWB;           // q tile, then the output tile of the chunk
  static constexpr int KG = D / 8;              // core matrices along K (= rows of S~)
  static constexpr int B_SBO = KG * 128;        // bytes between column groups of 8
  static constexpr int ST_BYTES = D * D * 2;    // S~_i tile as written by the mixing step
  static constexpr int BOPS = (N / 8) * B_SBO;  // B operand: S~ columns and the z~ column groups
  static constexpr int ZRAW = D * 4;              // z~_i in float32, copied in after the operand
  static constexpr int BT = (BOPS + ZRAW + 1023) / 1024 * 1024;
  static constexpr int NQ = D == 64 ? 9 : 16;   // q stages
  static constexpr int NB = D == 64 ? 6 : 10;   // B slots (one per work item)
  static constexpr uint32_t A_SBO = 8 * ROWB;
  static constexpr uint32_t A_LAYOUT = D == 64 ? 2u : 4u;
  static constexpr int ACC_STRIDE = D == 64 ? 128 : 64;
  static constexpr int TMEM_COLS = 2 * ACC_STRIDE;
  static constexpr size_t DATA = static_cast<size_t>(NQ) * QT + static_cast<size_t>(NB) * BT;
  static constexpr int WARPS = 16;
};
constexpr int kOutStoresInFlight = 3;   // TMA stores allowed to be reading shared memory at once
constexpr int kItemRing = 16;           // work items handed from the q producer to the other roles
constexpr int kItemRingReaders = 15;    // warps 1-15 read every item

struct OutBars {
  uint64_t *qfull, *phid, *ostore, *qempty, *bfull, *bempty, *tfull, *tempty, *fin, *ifull, *iempty;
  int32_t* ids;
};

template <int D>
__device__ __forceinline__ OutBars out_bars(uint8_t* ctrl) {
  using Cfg = OutCfg<D>;
  OutBars b;
  b.qfull = reinterpret_cast<uint64_t*>(ctrl);
  b.phid = b.qfull + Cfg::NQ;
  b.ostore = b.phid + Cfg::NQ;
  b.qempty = b.ostore + Cfg::NQ;
  b.bfull = b.qempty + Cfg::NQ;
  b.bempty = b.bfull + Cfg::NB;
  b.tfull = b.bempty + Cfg::NB;
  b.tempty = b.tfull + 2;
  b.fin = b.tempty + 2;
  b.ifull = b.fin + 1;
  b.iempty = b.ifull + kItemRing;
  b.ids = reinterpret_cast<int32_t*>(b.iempty + kItemRing);
  return b;
}
// bytes of the control region out_bars carves (barriers and the item ring)
template <int D>
constexpr int out_ctrl_bytes() {
  return (4 * OutCfg<D>::NQ + 2 * OutCfg<D>::NB + 5 + 2 * kItemRing) * 8 + kItemRing * 4;
}

template <int D>
__device__ __forceinline__ void out_init(const OutBars& b) {
  using Cfg = OutCfg<D>;
  for (int s = 0; s < Cfg::NQ; ++s) {
    mbar_init(b.qfull + s, 1);
    mbar_init(b.phid + s, 128);
    mbar_init(b.ostore + s, 128);
    mbar_init(b.qempty + s, 1);
  }
  for (int k = 0; k < Cfg::NB; ++k) {
    mbar_init(b.bfull + k, 1);
    mbar_init(b.bempty + k, 1);
  }
  for (int a = 0; a < 2; ++a) {
    mbar_init(b.tfull + a, 1);
    mbar_init(b.tempty + a, 128);
  }
  mbar_init(b.fin, 1);
  for (int r = 0; r < kItemRing; ++r) {
    mbar_init(b.ifull + r, 1);
    mbar_init(b.iempty + r, kItemRingReaders);
  }
}

// PAIR: the off-diagonal 32 x 32 blocks of every slot's S~ operand stay zero.
template <int D, bool PAIR>
__device__ __forceinline__ void out_zero_offdiag(uint8_t* bslot, int tid, int nthreads) {
  using Cfg = OutCfg<D>;
  if constexpr (PAIR) {
    for (int e = tid; e < Cfg::NB * 8 * 32; e += nthreads) {
      const int kb = e / 256, grp = (e / 32) % 8, r = e % 32;
      const int row = grp < 4 ? 32 + r : r;
      *reinterpret_cast<uint4*>(bslot + kb * Cfg::BT + grp * Cfg::B_SBO + row * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// Where the readout's items come from.  queue == null: first, first + stride,
// ... below n_items (a separate launch).  Otherwise the q producer takes the
// next item from the global queue counter and hands it to the other roles
// through the ring; a negative id ends the sequence.  mix_done (with queue):
// per batch counter of the mixing step, raised by each of its 8 epilogue warps
// for every 128-column tile that touches the batch's per_b_cols columns.
struct OutSched {
  int64_t first, stride, n_items;
  uint32_t* queue;
  const uint32_t* mix_done;
  int64_t per_b_cols;
};

// Value mix_done[b] reaches once every mixing tile of batch b is stored.
static __device__ __forceinline__ uint32_t mix_target(int64_t b, int64_t per_b_cols) {
  const int64_t t_lo = b * per_b_cols / 128, t_hi = ((b + 1) * per_b_cols - 1) / 128;
  return static_cast<uint32_t>(8 * (t_hi - t_lo + 1));
}

// Role-local cursor over the item sequence.
struct ItemCursor {
  int64_t next;
  uint32_t k;                   // ring position (items popped or pushed)
};

// The next item for a reading role: lane-0-only roles pass warp_wide = false.
static __device__ __forceinline__ bool next_item(const OutSched& sc, const OutBars& bars, ItemCursor& cur,
                                                 int64_t& item, bool warp_wide, volatile uint32_t* abortf,
                                                 unsigned int* err) {
  if (!sc.queue) {
    if (cur.next >= sc.n_items) return false;
    item = cur.next;
    cur.next += sc.stride;
    return true;
  }
  const uint32_t slot = cur.k % kItemRing, par = (cur.k / kItemRing) & 1u;
  ++cur.k;
  const bool ok = warp_wide ? warp_wait_on(bars.ifull + slot, par, abortf, err)
                            : wait_bounded_on(bars.ifull + slot, par, abortf, err);
  if (!ok) return false;
  const int32_t id = *reinterpret_cast<volatile int32_t*>(bars.ids + slot);
  if (warp_wide) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bars.iempty + slot);
  } else {
    mbar_arrive(bars.iempty + slot);
  }
  item = id;
  return id >= 0;
}

// The q producer's next item: from the queue (then handed on through the ring)
// or from the static sequence.
static __device__ __forceinline__ bool produce_item(const OutSched& sc, const OutBars& bars, ItemCursor& cur,
                                                    int64_t& item, volatile uint32_t* abortf, unsigned int* err) {
  if (!sc.queue) {
    if (cur.next >= sc.n_items) return false;
    item = cur.next;
    cur.next += sc.stride;
    return true;
  }
  const uint32_t got = atomicAdd(sc.queue, 1u);
  const int32_t id = got < static_cast<uint64_t>(sc.n_items) ? static_cast<int32_t>(got) : -1;
  const uint32_t slot = cur.k % kItemRing, par = (cur.k / kItemRing) & 1u;
  ++cur.k;
  if (!wait_bounded_on(bars.iempty + slot, par ^ 1u, abortf, err)) return false;
  bars.ids[slot] = id;
  mbar_arrive(bars.ifull + slot);
  item = id;
  return id >= 0;
}

template <int D, bool PAIR>
__device__ __forceinline__ void output_roles(const CUtensorMap* tm_q, const CUtensorMap* tm_o,
                                             const CUtensorMap* tm_st, const TcGeom& g, const OutSched& sc,
                                             int phi_kind, float eps, const float* __restrict__ zt,
                                             const __nv_bfloat16* St, uint8_t* smem, const OutBars& bars,
                                             uint32_t tmem, volatile uint32_t* abortf, unsigned int* err) {
  static_assert(!PAIR || D == 64, "head pairs form 64-channel rows");
  using Cfg = OutCfg<D>;
  uint8_t* qst = smem;                                   // [NQ] q / output tiles
  uint8_t* bslot = smem + Cfg::NQ * Cfg::QT;             // [NB] S~ tiles + z~ columns
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  ItemCursor cur{sc.first, 0};
  int64_t item = 0;

  if (warp == 0) {
    // ------------------------------------------- q producer
    if (lane == 0) {
      const uint64_t pol_q = policy_evict_first();
      int s = 0;
      uint32_t ph = 0;
      uint64_t fills = 0;
      bool ok = true;
      while (ok && produce_item(sc, bars, cur, item, abortf, err)) {
        const uint32_t it32 = static_cast<uint32_t>(item), rest = it32 / static_cast<uint32_t>(g.H);
        const int32_t h = static_cast<int32_t>(it32 - rest * static_cast<uint32_t>(g.H));
        const int32_t i = static_cast<int32_t>(rest % static_cast<uint32_t>(g.M));
        const int32_t b = static_cast<int32_t>(rest / static_cast<uint32_t>(g.M));
        for (int c = 0; c < g.chunks; ++c) {
          if (!wait_bounded_on(bars.qempty + s, ph ^ 1u, abortf, err)) { ok = false; break; }
          mbar_arrive_expect_tx(bars.qfull + s, Cfg::QT);
          int32_t x, y, z;
          chunk_coords(g, i, c, b, x, y, z);
          tma_load_5d(qst + s * Cfg::QT, tm_q, bars.qfull + s, 0, h, x, y, z, pol_q);
          ++fills;
          if (++s == Cfg::NQ) { s = 0; ph ^= 1u; }
        }
      }
      for (int st = 0; st < Cfg::NQ; ++st) {
        const uint64_t n = fills / Cfg::NQ + (static_cast<uint64_t>(st) < fills % Cfg::NQ ? 1 : 0);
        if (n > 0) drain_wait_on(bars.qfull + st, static_cast<uint32_t>((n - 1) & 1), err);
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
      if (!sc.queue) grid_dep_wait();   // separate launch: S~ and z~ come from the mixing launch
      const uint64_t pol_s = policy_evict_last();
      int kb = 0;
      uint32_t bph = 0;
      uint64_t fills = 0;
      int64_t ready_to = -1;            // mixing of batches <= ready_to is complete
      while (next_item(sc, bars, cur, item, false, abortf, err)) {
        const uint32_t it32 = static_cast<uint32_t>(item), rest = it32 / static_cast<uint32_t>(g.H);
        const int64_t h = it32 - rest * static_cast<uint32_t>(g.H);
        const int64_t i = rest % static_cast<uint32_t>(g.M), b = rest / static_cast<uint32_t>(g.M);
        if (sc.mix_done && b > ready_to) {
          if (!wait_counter_on(sc.mix_done + b, mix_target(b, sc.per_b_cols), abortf, err)) break;
          ready_to = b;
        }
        const int64_t tile = (b * g.H + h) * g.M + i;
        if (!wait_bounded_on(bars.bempty + kb, bph ^ 1u, abortf, err)) break;
        uint8_t* slot = bslot + kb * Cfg::BT;
        if constexpr (PAIR) {
          // heads 2h and 2h + 1 (32 x 32 tiles): one (8, 32) box per column group onto the diagonal
          mbar_arrive_expect_tx(bars.bfull + kb, 8 * 512 + Cfg::ZRAW);
          for (int e = 0; e < 2; ++e) {
            const int64_t t2 = (b * 2 * g.H + 2 * h + e) * g.M + i;
            for (int gq = 0; gq < 4; ++gq)
              tma_load_4d(slot + (4 * e + gq) * Cfg::B_SBO + 32 * e * 16, tm_st, bars.bfull + kb, 0, 0, gq,
                          static_cast<int32_t>(t2), pol_s);
            bulk_load(slot + Cfg::BOPS + e * 128, zt + t2 * 32, 128, bars.bfull + kb, pol_s);
          }
        } else {
          mbar_arrive_expect_tx(bars.bfull + kb, Cfg::ST_BYTES + Cfg::ZRAW);
          tma_load_4d(slot, tm_st, bars.bfull + kb, 0, 0, 0, static_cast<int32_t>(tile), pol_s);
          bulk_load(slot + Cfg::BOPS, zt + tile * D, Cfg::ZRAW, bars.bfull + kb, pol_s);
        }
        ++fills;
        if (++kb == Cfg::NB) { kb = 0; bph ^= 1u; }
      }
      for (int st = 0; st < Cfg::NB; ++st) {
        const uint64_t n = fills / Cfg::NB + (static_cast<uint64_t>(st) < fills % Cfg::NB ? 1 : 0);
        if (n > 0) drain_wait_on(bars.bfull + st, static_cast<uint32_t>((n - 1) & 1), err);
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
      while (ok && next_item(sc, bars, cur, item, false, abortf, err)) {
        const uint32_t it32 = static_cast<uint32_t>(item), rest = it32 / static_cast<uint32_t>(g.H);
        const int32_t h = static_cast<int32_t>(it32 - rest * static_cast<uint32_t>(g.H));
        const int32_t i = static_cast<int32_t>(rest % static_cast<uint32_t>(g.M));
        const int32_t b = static_cast<int32_t>(rest / static_cast<uint32_t>(g.M));
        for (int c = 0; c < g.chunks; ++c) {
          if (!wait_bounded_on(bars.ostore + s, ph, abortf, err)) { ok = false; break; }
          int32_t x, y, z;
          chunk_coords(g, i, c, b, x, y, z);
          // d = 64: the output leaves L2 early (evict-first); measured slower at d = 32
          if constexpr (D == 64) {
            tma_store_5d_hint(tm_o, qst + s * Cfg::QT, 0, h, x, y, z, policy_evict_first());
          } else {
            tma_store_5d(tm_o, qst + s * Cfg::QT, 0, h, x, y, z);
          }
          bulk_commit_group();
          pend[npend++] = s;
          if (npend > kOutStoresInFlight) {
            bulk_wait_group_read<kOutStoresInFlight>();   // the oldest store has read its tile
            mbar_arrive(bars.qempty + pend[0]);
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
      while (ok && next_item(sc, bars, cur, item, false, abortf, err)) {
        // the slot of this item: S~ copy landed and z~ columns written
        if (!wait_bounded_on(bars.bfull + kb, bph, abortf, err)) break;
        const uint32_t bbase = smem_u32(bslot + kb * Cfg::BT);
        for (int c = 0; c < g.chunks; ++c, ++cnt) {
          const uint32_t acc = cnt & 1u, aph = (cnt >> 1) & 1u;
          if (!wait_bounded_on(bars.tempty + acc, aph ^ 1u, abortf, err)) { ok = false; break; }
          if (!wait_bounded_on(bars.phid + s, ph, abortf, err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t base = smem_u32(qst + s * Cfg::QT);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint64_t a = smem_desc(base + ks * 32, 16, Cfg::A_SBO, Cfg::A_LAYOUT);
            const uint64_t b = smem_desc(bbase + ks * 256, 128, Cfg::B_SBO, 0);
            mma_bf16(tmem + acc * Cfg::ACC_STRIDE, a, b, idesc, ks != 0 ? 1u : 0u);
          }
          mma_commit(bars.tfull + acc);
          if (++s == Cfg::NQ) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        mma_commit(bars.bempty + kb);              // slot reusable once this item's MMAs are done
        if (++kb == Cfg::NB) { kb = 0; bph ^= 1u; }
      }
      mma_commit(bars.fin);
      drain_wait_on(bars.fin, 0, err);
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
    while (ok && next_item(sc, bars, cur, item, true, abortf, err)) {
      // the item's slot: S~_i and the float32 z~_i have landed (the producer runs ahead)
      if (!warp_wait_on(bars.bfull + kb, bph, abortf, err)) break;
      if (rt < D) {
        uint8_t* slot = bslot + kb * Cfg::BT;
        const float zv = *reinterpret_cast<const float*>(slot + Cfg::BOPS + rt * 4);
        const __nv_bfloat16 hi = __float2bfloat16_rn(zv);
        const __nv_bfloat16 lo = __float2bfloat16_rn(zv - __bfloat162float(hi));
        const uint32_t hl =
            static_cast<uint32_t>(__bfloat16_as_ushort(hi)) | (static_cast<uint32_t>(__bfloat16_as_ushort(lo)) << 16);
        if constexpr (PAIR) {   // row rt belongs to head rt / 32: columns 64, 65 or 66, 67
          *reinterpret_cast<uint2*>(slot + zoff) = rt < 32 ? make_uint2(hl, 0u) : make_uint2(0u, hl);
        } else {
          *reinterpret_cast<uint32_t*>(slot + zoff) = hl;
        }
      }
      if (++kb == Cfg::NB) { kb = 0; bph ^= 1u; }
      for (int c = 0; c < g.chunks; ++c) {
        if (!warp_wait_on(bars.qfull + s, ph, abortf, err)) { ok = false; break; }
        uint8_t* tile = qst + s * Cfg::QT;
#pragma unroll
        for (int m = 0; m < Cfg::C / RP; ++m) {
          uint4* ptr = reinterpret_cast<uint4*>(tile + (rg + RP * m) * Cfg::ROWB + p * 16);
          *ptr = phi8_packed(*ptr, add_eps, eps2);
        }
        // also publishes this item's z~ columns to the MMA (first chunk)
        fence_proxy_async_smem();
        mbar_arrive(bars.phid + s);
        if (++s == Cfg::NQ) { s = 0; ph ^= 1u; }
      }
    }
  } else if (warp < 14) {
    // ------------------------------------------- epilogue: scale and write back
    // Warpgroup wg (warps 6-9 or 10-13) takes the chunks with cnt % 2 == wg, which
    // are exactly the chunks accumulated in TMEM accumulator wg.
    const int wg = (warp - 6) >> 2;
    const int q4 = warp & 3;
    const int row = 32 * q4 + lane;      // token row of the chunk
    int s = 0;
    uint32_t ph = 0, cnt = 0;
    bool ok = true;
    while (ok && next_item(sc, bars, cur, item, true, abortf, err)) {
      for (int c = 0; c < g.chunks; ++c, ++cnt) {
        const int cs = s;
        if (++s == Cfg::NQ) { s = 0; ph ^= 1u; }
        if (static_cast<int>(cnt & 1u) != wg) continue;
        const uint32_t acc = wg, aph = (cnt >> 1) & 1u;
        if (!warp_wait_on(bars.tfull + acc, aph, abortf, err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tb = tmem + acc * Cfg::ACC_STRIDE + (static_cast<uint32_t>(32 * q4) << 16);
        uint32_t v0[32], v1[32], vz[16];
        tmem_ld_x32(tb, v0);
        if (D == 64) tmem_ld_x32(tb + 32, v1);
        tmem_ld_x16(tb + D, vz);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(bars.tempty + acc);
        const float inv0 = 1.0f / (__uint_as_float(vz[0]) + __uint_as_float(vz[1]) + eps);
        const float inv1 = PAIR ? 1.0f / (__uint_as_float(vz[2]) + __uint_as_float(vz[3]) + eps) : inv0;
        // the MMA has finished reading the q tile: the output row goes in its place
        uint8_t* orow = qst + cs * Cfg::QT + row * Cfg::ROWB;
#pragma unroll
        for (int q = 0; q < D / 8; ++q) {
          const uint32_t* src = (q < 4) ? (v0 + 8 * q) : (v1 + 8 * (q - 4));
          const float inv = q < 4 ? inv0 : inv1;
          const uint4 packed = make_uint4(
              pack_bf16(__uint_as_float(src[0]) * inv, __uint_as_float(src[1]) * inv),
              pack_bf16(__uint_as_float(src[2]) * inv, __uint_as_float(src[3]) * inv),
              pack_bf16(__uint_as_float(src[4]) * inv, __uint_as_float(src[5]) * inv),
              pack_bf16(__uint_as_float(src[6]) * inv, __uint_as_float(src[7]) * inv));
          *reinterpret_cast<uint4*>(orow + ((q ^ swz<D>(row)) * 16)) = packed;
        }
        fence_proxy_async_smem();
        mbar_arrive(bars.ostore + cs);
        if (D == 64 && !PAIR && c + 1 == g.chunks) {
          // the item's last MMA has read its S~ tile and z~ (each read once, by this
          // CTA): their lines leave L2 without a write-back (measured slower at d = 32)
          const uint32_t it32 = static_cast<uint32_t>(item), rest = it32 / static_cast<uint32_t>(g.H);
          const uint32_t hh = it32 - rest * static_cast<uint32_t>(g.H);
          const uint32_t bb = rest / static_cast<uint32_t>(g.M), ii = rest - bb * static_cast<uint32_t>(g.M);
          const int64_t tile = (static_cast<int64_t>(bb) * g.H + hh) * g.M + ii;
          const int e = 32 * q4 + lane;
          if (e < D * D * 2 / 128) discard_l2_line(reinterpret_cast<const uint8_t*>(St + tile * D * D) + e * 128);
          else if (e < D * D * 2 / 128 + D * 4 / 128)
            discard_l2_line(reinterpret_cast<const uint8_t*>(zt + tile * D) + (e - D * D * 2 / 128) * 128);
        }
      }
    }
  }
}

}  // namespace tc
}  // namespace mhla
