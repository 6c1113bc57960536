// Fused tensor-core path of the MHLA forward for short sequences (N <= 256
// tokens per image, M <= 96 blocks): one launch, no workspace.
//
// When all keys of an image fit one 256-column tile, the block summaries and
// the mixed summaries need not be materialised.  Substituting
// S~_i = sum_j W[i][j] S_j and z~_i = sum_j W[i][j] z_j, S_j = sum_{s in j}
// phi(k_s) v_s^T, into the readout o_t = phi(q_t) S~_b(t) / (phi(q_t) . z~_b(t)
// + eps) gives the two-stage form of the same quantity:
//
//   P[t][s] = W[b(t)][b(s)] * (phi(q_t) . phi(k_s))
//   o_t     = sum_s P[t][s] v_s / (sum_s P[t][s] + eps)
//
// ([P2] "MHLA: Restoring Expressivity of Linear Attention via Token-Level
// Multi-Head", section 4 "Multi-Head Mixing" and "Token-Level Adaptivity";
// [P1] 171host.com/767426.html, section 5(4), the two-stage selection).  Per
// block count this is cheaper than the three-launch path whenever M^2 is not
// small next to N (DeiT-T: N = 196, M = 49).
//
// One work unit = (b, h, 128 query tokens).  Persistent CTAs of nine warps:
//   warp 8   (control) TMA of the q tile (128 x d) and of all keys and values
//            (KR x d, KR = N rounded up to 32, rows past N zero-filled) through
//            4-D maps (d, H, N, B); issues both MMAs;
//   warps 0-7 (workers, two warpgroups):
//            phi in place on the q and k tiles in shared memory;
//            after MMA 1 (scores phi(Q) phi(K)^T, 128 x KR, float32 in tensor
//            memory) each thread owns one query row and half of the key
//            columns: P = score * W[b(t)][b(s)] rounded to bf16, written
//            K-major (128-byte swizzle) as the A operand of MMA 2, 64 keys at
//            a time; the control warp starts MMA 2 on each 64-key chunk as
//            soon as both warpgroups have written it;
//            MMA 2 = P [V | 1]: the value tile as it landed (MN-major B) plus a
//            constant ones column, so the tensor core also sums the rounded P
//            into the denominator; each warpgroup scales half of the output
//            columns by 1 / (den + eps), rounds to bf16 and stores them.
// The next unit's q and k tiles load once MMA 1 has read the current ones, its
// values once MMA 2 has; the first unit's loads overlap the set-up of W.  The
// workers apply phi to the next unit between forming P and writing the output,
// so that phi runs under MMA 2 and the next unit's MMA 1 under the output.
//
// Every wait is bounded (2 s of %globaltimer, 2^28 polls); a wait that gives
// up sets bit 0 of this file's device error word and a per-CTA abort flag so
// the other roles stop waiting too; copies and MMAs in flight are drained
// (bit 1 if that drain gives up) and tensor memory is released.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "mhla_internal.h"
#include "ptx.cuh"
#include "stall_hook.cuh"
#include "tma_host.h"

namespace mhla {

__device__ unsigned int g_small_error = 0;

namespace {

using namespace ptx;

constexpr uint64_t kSmallWaitNs = 2000000000ull;   // 2 s
constexpr uint32_t kSmallWaitPolls = 1u << 28;
constexpr uint64_t kSmallDrainNs = 50000000ull;    // 50 ms for work already in flight
constexpr int kWorkers = 256;                      // warps 0-7
constexpr int kSmallThreads = kWorkers + 32;       // + the control warp
constexpr int kQRows = 128;      // query tokens per unit: MMA M, one TMEM lane each
constexpr int kMaxKeys = 256;    // keys per image: MMA N of the score product
constexpr int kMaxBlocks = 96;   // W is held in shared memory as float32
constexpr int kTmemCols = 512;   // scores in [0, 256), P [V | 1] in [256, 256 + d + 16)

template <int D>
struct SmallCfg {
  static constexpr int ROWB = D * 2;                 // bytes per token row
  static constexpr int Q_BYTES = kQRows * ROWB;
  static constexpr int KV_BYTES = kMaxKeys * ROWB;
  static constexpr int P_CHUNK = kQRows * 128;       // 64 keys of P: 128 rows of 128 bytes
  static constexpr int P_BYTES = (kMaxKeys / 64) * P_CHUNK;
  static constexpr int W_BYTES = kMaxBlocks * (kMaxBlocks + 1) * 4;   // rows of M + 1 (zero sentinel)
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + Q_BYTES;      // k directly after q: phi runs over both
  static constexpr int V_OFF = K_OFF + KV_BYTES;
  static constexpr int ONES_OFF = V_OFF + KV_BYTES;  // second N atom of MMA 2's B operand
  static constexpr int P_OFF = ONES_OFF + KV_BYTES;
  static constexpr int W_OFF = P_OFF + P_BYTES;
  static constexpr int BLK_OFF = W_OFF + (W_BYTES + 15) / 16 * 16;   // byte offset of W[.][b(s)] per key
  static constexpr int CTRL_OFF = BLK_OFF + kMaxKeys * 2;
  static constexpr size_t SMEM = CTRL_OFF + 128 + 1024;
  static constexpr uint32_t SBO = 8 * ROWB;          // 8-row groups of a token tile
  static constexpr uint32_t LAYOUT = D == 64 ? 2u : 4u;   // 128- or 64-byte swizzle
  static constexpr int NO = D + 16;                  // MMA 2 columns: d values, the ones block
};

struct SmallGeom {
  int32_t N, H, M, KR, nqt;          // tokens, heads, blocks, key rows loaded, query tiles
  int32_t X, Y, bx, by, bt, nbx, nby;
  int64_t osb, osn, osh;             // output strides, elements
};

__device__ __noinline__ bool small_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  // diagnostic hook (stall_hook.cuh), looked at only once a wait has to poll
  if (stall_this_warp()) {
    stalled_wait(abort_flag);
    *abort_flag = 1u;
    atomicOr(&g_small_error, 1u);
    return false;
  }
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1; it < kSmallWaitPolls; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > kSmallWaitNs) break;
    }
  }
  *abort_flag = 1u;
  atomicOr(&g_small_error, 1u);
  return false;
}

// Every lane waits, then the warp agrees, so warp-collective tcgen05.ld that
// follows runs on all lanes or on none.
__device__ __forceinline__ bool small_warp_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag) {
  return __all_sync(0xffffffffu, small_wait(bar, parity, abort_flag));
}

__device__ __noinline__ void small_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 0; it < kSmallWaitPolls; ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 63u) == 63u && globaltimer() - t0 > kSmallDrainNs) {
      atomicOr(&g_small_error, 2u);
      return;
    }
  }
}

__device__ __forceinline__ uint4 phi8(uint4 raw, bool add_eps, __nv_bfloat162 eps2) {
  const __nv_bfloat162 zero = __float2bfloat162_rn(0.0f);
  uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&w[e]);
    v = __hmax2(v, zero);
    if (add_eps) v = __hadd2(v, eps2);
    w[e] = *reinterpret_cast<uint32_t*>(&v);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

template <int D>
__global__ void __launch_bounds__(kSmallThreads, 1)
tc_small(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
         const __grid_constant__ CUtensorMap tm_v, SmallGeom g, int64_t n_units, int phi_kind, float eps,
         const float* __restrict__ W, __nv_bfloat16* __restrict__ out) {
  using Cfg = SmallCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  uint8_t* sq = smem + Cfg::Q_OFF;
  uint8_t* sk = smem + Cfg::K_OFF;
  uint8_t* sv = smem + Cfg::V_OFF;
  uint8_t* sones = smem + Cfg::ONES_OFF;
  uint8_t* sp = smem + Cfg::P_OFF;
  float* sw = reinterpret_cast<float*>(smem + Cfg::W_OFF);
  uint16_t* soff = reinterpret_cast<uint16_t*>(smem + Cfg::BLK_OFF);
  uint64_t* full_qk = reinterpret_cast<uint64_t*>(smem + Cfg::CTRL_OFF);
  uint64_t* full_v = full_qk + 1;
  uint64_t* phid = full_qk + 2;     // workers: phi applied
  uint64_t* done1 = full_qk + 3;    // MMA 1 complete
  uint64_t* done2 = full_qk + 4;    // MMA 2 complete
  uint64_t* odone = full_qk + 5;    // workers: MMA 2 result read from tensor memory
  uint64_t* chunk = full_qk + 6;    // [4] workers: 64 keys of P written
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(full_qk + 10);
  volatile uint32_t* abortf = tmem_slot + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_chunks = (g.KR + 63) / 64;

  if (tid == kWorkers) {
    mbar_init(full_qk, 1);
    mbar_init(full_v, 1);
    mbar_init(phid, kWorkers / 32);
    mbar_init(done1, 1);
    mbar_init(done2, 1);
    mbar_init(odone, kWorkers / 32);
    for (int c = 0; c < 4; ++c) mbar_init(chunk + c, kWorkers / 32);
    *abortf = 0u;
    fence_mbar_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  __syncthreads();

  const uint64_t pol_q = policy_evict_first();
  const uint64_t pol_kv = policy_evict_last();   // every query tile of (b, h) reads them
  // unit -> (b, h, query tile) in 32-bit arithmetic (units < 2^31, checked on the host)
  auto issue_qk = [&](int64_t u) {
    const uint32_t uu = static_cast<uint32_t>(u);
    const int32_t qt = static_cast<int32_t>(uu % static_cast<uint32_t>(g.nqt));
    const uint32_t bh = uu / static_cast<uint32_t>(g.nqt);
    const int32_t h = static_cast<int32_t>(bh % static_cast<uint32_t>(g.H));
    const int32_t b = static_cast<int32_t>(bh / static_cast<uint32_t>(g.H));
    mbar_arrive_expect_tx(full_qk, static_cast<uint32_t>((kQRows + g.KR) * Cfg::ROWB));
    tma_load_4d(sq, &tm_q, full_qk, 0, h, qt * kQRows, b, pol_q);
    tma_load_4d(sk, &tm_k, full_qk, 0, h, 0, b, pol_kv);
  };
  auto issue_v = [&](int64_t u) {
    const uint32_t bh = static_cast<uint32_t>(u) / static_cast<uint32_t>(g.nqt);
    const int32_t h = static_cast<int32_t>(bh % static_cast<uint32_t>(g.H));
    const int32_t b = static_cast<int32_t>(bh / static_cast<uint32_t>(g.H));
    mbar_arrive_expect_tx(full_v, static_cast<uint32_t>(g.KR * Cfg::ROWB));
    tma_load_4d(sv, &tm_v, full_v, 0, h, 0, b, pol_kv);
  };
  uint32_t n_qk = 0, n_v = 0, n_m1 = 0, n_m2 = 0;   // phases issued (control lane)
  if (tid == kWorkers && static_cast<int64_t>(blockIdx.x) < n_units) {
    issue_qk(blockIdx.x);
    issue_v(blockIdx.x);
    n_qk = n_v = 1;
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (tid < kWorkers) {
    // W with a zero column M appended to every row (the block of padded keys),
    // every element copied asynchronously so all of them are in flight at once.
    const int M = g.M, nW = M * M;
    for (int e = tid; e < nW; e += kWorkers) cp_async_4(sw + (e / M) * (M + 1) + e % M, W + e);
    for (int i = tid; i < M; i += kWorkers) sw[i * (M + 1) + M] = 0.0f;
    // Byte offset of W[.][b(s)] for key s: blocks row-major over (nbt, nby,
    // nbx), tokens raster over (T, Y, X); keys past N point at the zero column.
    for (int n = tid; n < kMaxKeys; n += kWorkers) {
      int id = M;
      if (n < g.N) {
        const int x = n % g.X, r = n / g.X, y = r % g.Y, t = r / g.Y;
        id = ((t / g.bt) * g.nby + y / g.by) * g.nbx + x / g.bx;
      }
      soff[n] = static_cast<uint16_t>(id * 4);
    }
    // Constant ones block of MMA 2's B operand: row s holds (1, 0, ..., 0) in
    // the swizzled layout, so output column d sums P over the keys.
    for (int idx = tid; idx < kMaxKeys * (D / 8); idx += kWorkers) {
      const int row = idx / (D / 8), phys = idx % (D / 8);
      const int logical = phys ^ (D == 64 ? (row & 7) : ((row >> 1) & 3));
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (logical == 0) v.x = 0x3F80u;   // bf16 1.0 in the low half
      *reinterpret_cast<uint4*>(sones + row * Cfg::ROWB + phys * 16) = v;
    }
    fence_proxy_async_smem();
    cp_async_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWorkers / 32) {
    // ------------------------------------------------------------ control
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      // MMA 1 (scores) of the unit whose phi the workers have just applied
      auto issue_mma1 = [&]() {
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(128, g.KR, /*a K-major*/ false, /*b K-major*/ false);
        const uint32_t qa = smem_u32(sq), ka = smem_u32(sk);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_bf16(tmem, smem_desc(qa + ks * 32, 16, Cfg::SBO, Cfg::LAYOUT),
                   smem_desc(ka + ks * 32, 16, Cfg::SBO, Cfg::LAYOUT), idesc, ks > 0 ? 1u : 0u);
        mma_commit(done1);
        ++n_m1;
      };
      if (static_cast<int64_t>(blockIdx.x) < n_units) {
        if (small_wait(phid, 0u, abortf)) issue_mma1();
        else ok = false;
      }
      for (int64_t u = blockIdx.x; ok && u < n_units; u += gridDim.x, ++it) {
        const uint32_t par = it & 1u;
        const int64_t next = u + gridDim.x;
        if (!small_wait(done1, par, abortf)) break;
        if (next < n_units) {   // q and k consumed: the next unit's may land
          issue_qk(next);
          ++n_qk;
        }
        // The previous unit's result must be out of tensor memory before
        // MMA 2 overwrites it, and this unit's values must have landed.
        if (it > 0 && !small_wait(odone, par ^ 1u, abortf)) break;
        if (!small_wait(full_v, par, abortf)) break;
        const uint32_t idesc2 = idesc_bf16_f32(128, Cfg::NO, /*a K-major*/ false, /*b MN-major*/ true);
        const uint32_t pa = smem_u32(sp), va = smem_u32(sv);
        for (int c = 0; c < n_chunks; ++c) {
          if (!small_wait(chunk + c, par, abortf)) { ok = false; break; }
          tc_fence_after();
          const int ks_end = min(4 * c + 4, g.KR / 16);
          for (int ks = 4 * c; ks < ks_end; ++ks)
            mma_bf16(tmem + 256, smem_desc(pa + c * Cfg::P_CHUNK + (ks & 3) * 32, 16, 1024, 2),
                     smem_desc(va + ks * 2 * Cfg::SBO, Cfg::ONES_OFF - Cfg::V_OFF, Cfg::SBO, Cfg::LAYOUT), idesc2,
                     ks > 0 ? 1u : 0u);
        }
        if (!ok) break;
        mma_commit(done2);
        ++n_m2;
        // The next unit's scores go in behind MMA 2 as soon as its phi is
        // applied: the workers have read this unit's scores before that.
        if (next < n_units) {
          if (!small_wait(phid, par ^ 1u, abortf)) break;
          issue_mma1();
        }
        if (!small_wait(done2, par, abortf)) break;
        if (next < n_units) {   // values consumed
          issue_v(next);
          ++n_v;
        }
      }
      // Copies and MMAs issued must finish before shared and tensor memory go
      // away (a phase already complete returns at once).
      if (n_qk) small_drain(full_qk, (n_qk - 1) & 1u);
      if (n_v) small_drain(full_v, (n_v - 1) & 1u);
      if (n_m1) small_drain(done1, (n_m1 - 1) & 1u);
      if (n_m2) small_drain(done2, (n_m2 - 1) & 1u);
    }
  } else {
    // ------------------------------------------------------------ workers
    const int row = tid & 127;              // query row = TMEM lane
    const int half = tid >> 7;              // key columns and output columns of this warpgroup
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const bool add_eps = phi_kind == MHLA_PHI_RELU_EPS;
    const __nv_bfloat162 eps2 = __float2bfloat162_rn(eps);
    const int swr = row & 7;                // 128-byte swizzle phase of this thread's P row
    const int n16 = (kQRows + g.KR) * Cfg::ROWB / 16;
    // phi in place over the q and k tiles (contiguous) of the unit with
    // copy phase par; false when the wait gives up
    auto apply_phi = [&](uint32_t par) {
      if (!small_warp_wait(full_qk, par, abortf)) return false;
      uint4* base = reinterpret_cast<uint4*>(sq);
      for (int e = tid; e < n16; e += kWorkers) base[e] = phi8(base[e], add_eps, eps2);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(phid);
      return true;
    };
    // Per unit: P, then phi of the next unit (under MMA 2), then the output
    // (under the next unit's MMA 1).
    uint32_t it = 0;
    bool live = static_cast<int64_t>(blockIdx.x) >= n_units || apply_phi(0u);
    for (int64_t u = blockIdx.x; live && u < n_units; u += gridDim.x, ++it) {
      const uint32_t par = it & 1u;
      const uint32_t uu = static_cast<uint32_t>(u);
      const int32_t qt = static_cast<int32_t>(uu % static_cast<uint32_t>(g.nqt));
      const uint32_t bh = uu / static_cast<uint32_t>(g.nqt);
      const int32_t h = static_cast<int32_t>(bh % static_cast<uint32_t>(g.H));
      const int32_t b = static_cast<int32_t>(bh / static_cast<uint32_t>(g.H));

      // ---- P[t][s] = score * W[b(t)][b(s)], bf16, K-major SW128, 64 keys per chunk
      if (!small_warp_wait(done1, par, abortf)) break;
      tc_fence_after();
      const int32_t nq = qt * kQRows + row;
      const uint8_t* wrow =
          reinterpret_cast<const uint8_t*>(sw) + (nq < g.N ? soff[nq] / 4 : 0) * (g.M + 1) * 4;
      // two score buffers: the tensor-memory load of chunk c + 1 is in flight
      // while chunk c is weighted (n_chunks <= 4, so the loop unrolls fully)
      const int mlim = g.KR / 32;
      uint32_t r[2][32];
      if (half < mlim) tmem_ld_x32(lane_base + half * 32, r[0]);
#pragma unroll
      for (int c = 0; c < kMaxKeys / 64; ++c) {
        if (c >= n_chunks) break;
        const int m = 2 * c + half;         // 32 keys of this warpgroup in chunk c
        uint4 offs[4];
        if (m < mlim) {
#pragma unroll
          for (int i = 0; i < 4; ++i) offs[i] = reinterpret_cast<const uint4*>(soff + m * 32)[i];
        }
        tmem_ld_wait();                     // chunk c's scores (the only load in flight)
        if (c + 1 < kMaxKeys / 64 && c + 1 < n_chunks && m + 2 < mlim)
          tmem_ld_x32(lane_base + (m + 2) * 32, r[(c + 1) & 1]);
        if (m < mlim) {
          const uint32_t* ow = reinterpret_cast<const uint32_t*>(offs);
          const uint32_t* rc = r[c & 1];
          uint32_t packed[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const uint32_t o2 = ow[e >> 1];
            const float w0 = *reinterpret_cast<const float*>(wrow + (o2 & 0xFFFFu));
            const float w1 = *reinterpret_cast<const float*>(wrow + (o2 >> 16));
            packed[e >> 1] = pack2(__uint_as_float(rc[e]) * w0, __uint_as_float(rc[e + 1]) * w1);
          }
          uint8_t* prow = sp + c * Cfg::P_CHUNK + row * 128;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4*>(prow + (((half * 4 + q) ^ swr) * 16)) =
                make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(chunk + c);
      }
      tmem_ld_wait();                       // nothing left in flight (no-op when none was issued)

      // ---- the next unit's phi, while MMA 2 of this one runs
      if (u + gridDim.x < n_units && !apply_phi(par ^ 1u)) break;

      // ---- output: o_t = (P V)_t / (P 1)_t + eps), this warpgroup's half of the columns
      if (!small_warp_wait(done2, par, abortf)) break;
      tc_fence_after();
      constexpr int HC = D / 2;
      uint32_t o[HC], dn;
      if constexpr (HC == 32) {
        tmem_ld_x32(lane_base + 256 + half * HC, o);
      } else {
        tmem_ld_x16(lane_base + 256 + half * HC, o);
      }
      tmem_ld_x1(lane_base + 256 + D, dn);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(odone);
      if (nq < g.N) {
        const float inv = 1.0f / (__uint_as_float(dn) + eps);
        uint4* dst = reinterpret_cast<uint4*>(out + b * g.osb + static_cast<int64_t>(nq) * g.osn + h * g.osh +
                                              half * HC);
#pragma unroll
        for (int q = 0; q < HC / 8; ++q)
          dst[q] = make_uint4(pack2(__uint_as_float(o[8 * q]) * inv, __uint_as_float(o[8 * q + 1]) * inv),
                              pack2(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv),
                              pack2(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv),
                              pack2(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ----------------------------------------------------------------- host side

bool small_operand_ok(const Problem& p, const Operand& o) {
  if (reinterpret_cast<uintptr_t>(o.data) % 16 != 0) return false;
  if (o.sb % 8 != 0 || o.sn % 8 != 0 || o.sh % 8 != 0) return false;
  if ((p.H > 1 && o.sh <= 0) || (p.N > 1 && o.sn <= 0) || (p.B > 1 && o.sb <= 0)) return false;
  const int64_t lim = int64_t{1} << 39;   // byte strides of a tensor map stay below 2^40
  return o.sb < lim && o.sn < lim && o.sh < lim;
}

// (d, H, N, B) view of a [B, N, H, d] operand; a box of `rows` tokens of one head.
bool small_map(const Problem& p, const Operand& o, int rows, CUtensorMap* m) {
  const int64_t sh = p.H > 1 ? o.sh : p.d;
  const int64_t sn = p.N > 1 ? o.sn : p.H * p.d;
  const int64_t sb = p.B > 1 ? o.sb : p.N * p.H * p.d;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(p.d), static_cast<cuuint64_t>(p.H),
                              static_cast<cuuint64_t>(p.N), static_cast<cuuint64_t>(p.B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(sh * 2), static_cast<cuuint64_t>(sn * 2),
                                 static_cast<cuuint64_t>(sb * 2)};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(p.d), 1u, static_cast<cuuint32_t>(rows), 1u};
  return encode_tensor_map(m, 4, o.data, dims, strides, box,
                           p.d == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}

template <int D>
int launch_small_d(const Problem& p, const float* W, cudaStream_t stream) {
  using Cfg = SmallCfg<D>;
  const int32_t KR = static_cast<int32_t>((p.N + 31) / 32 * 32);
  CUtensorMap tq, tk, tv;
  if (!small_map(p, p.q, kQRows, &tq) || !small_map(p, p.k, KR, &tk) || !small_map(p, p.v, KR, &tv))
    return MHLA_ERR_CUDA;
  SmallGeom g;
  g.N = static_cast<int32_t>(p.N);
  g.H = static_cast<int32_t>(p.H);
  g.M = static_cast<int32_t>(p.M);
  g.KR = KR;
  g.nqt = static_cast<int32_t>((p.N + kQRows - 1) / kQRows);
  g.X = static_cast<int32_t>(p.X);
  g.Y = static_cast<int32_t>(p.Y);
  g.bx = static_cast<int32_t>(p.bx);
  g.by = static_cast<int32_t>(p.by);
  g.bt = static_cast<int32_t>(p.bt);
  g.nbx = static_cast<int32_t>(p.nbx);
  g.nby = static_cast<int32_t>(p.nby);
  g.osb = p.o.sb;
  g.osn = p.o.sn;
  g.osh = p.o.sh;
  const int64_t n_units = p.B * p.H * g.nqt;
  const int sms = device_sm_count();
  if (sms <= 0) return MHLA_ERR_CUDA;
  if (cudaFuncSetAttribute(tc_small<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(Cfg::SMEM)) != cudaSuccess)
    return MHLA_ERR_CUDA;
  const int grid = static_cast<int>(std::min<int64_t>(n_units, sms));
  KernelTimer timer("tc_small", stream);
  tc_small<D><<<grid, kSmallThreads, Cfg::SMEM, stream>>>(tq, tk, tv, g, n_units, p.phi_kind, p.eps, W,
                                                           static_cast<__nv_bfloat16*>(p.o.data));
  return cudaGetLastError() == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
}

}  // namespace

bool small_eligible(const Problem& p) {
  if (p.dtype != MHLA_BF16 || (p.d != 32 && p.d != 64)) return false;
  if (p.B < 1 || p.H < 1 || p.N > kMaxKeys || p.M > kMaxBlocks) return false;
  for (const Operand* o : {&p.q, &p.k, &p.v, &p.o})
    if (!small_operand_ok(p, *o)) return false;
  const int64_t lim32 = int64_t{1} << 31;
  return p.B < lim32 && p.H < lim32 && p.B * p.H * ((p.N + kQRows - 1) / kQRows) < lim32;
}

int launch_small(const Problem& p, const float* W, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.d == 64) return launch_small_d<64>(p, W, s);
  return launch_small_d<32>(p, W, s);
}

int read_and_clear_small_error(void* stream, uint32_t* flags) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int host = 0;
  if (cudaMemcpyFromSymbolAsync(&host, g_small_error, sizeof(host), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MHLA_ERR_CUDA;
  const unsigned int zero = 0;
  if (cudaMemcpyToSymbolAsync(g_small_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return MHLA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MHLA_ERR_CUDA;
  *flags = host;
  return host ? MHLA_ERR_TIMEOUT : MHLA_OK;
}

MHLA_DEFINE_STALL_SETTER(set_stall_small)

}  // namespace mhla
