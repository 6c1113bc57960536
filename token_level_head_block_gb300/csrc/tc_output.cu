// tc_output: the readout step of the tensor-core path, per (b, h, block i),
// 128 tokens at a time: o_t = phi(q_t) S~_i / (phi(q_t) . z~_i + eps)
// ([P2] "MHLA: Restoring Expressivity of Linear Attention via Token-Level
// Multi-Head", section 4 "Token-Level Adaptivity"; [P1] 171host.com/767426.html,
// section 5(4) and section 7, MHLA.forward).

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

__device__ unsigned int g_out_error = 0;

namespace {

using namespace ptx;
using namespace tc;

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag) {
  return wait_bounded_on(bar, parity, abort_flag, &g_out_error);
}
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag) {
  return warp_wait_on(bar, parity, abort_flag, &g_out_error);
}
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) { drain_wait_on(bar, parity, &g_out_error); }

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

// PAIR (D = 64 only): each 64-channel row is two adjacent heads of 32 channels
// (heads 2h', 2h' + 1 as one "head" h' of the TMA view), so q and o move in
// 128-byte rows; the B operand is block-diagonal, [S~_a 0; 0 S~_b], with z~_a
// hi, lo in columns 64, 65 for the rows of head a and z~_b in 66, 67 for the rows
// of head b, and each half of the output row takes its own denominator.
template <int D, bool PAIR>
__global__ void __launch_bounds__(kOutThreadsTC, 1)
tc_output(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_o,
          const __grid_constant__ CUtensorMap tm_st, TcGeom g, int64_t n_items, int phi_kind, float eps,
          const float* __restrict__ zt, const __nv_bfloat16* St) {
  static_assert(!PAIR || D == 64, "head pairs form 64-channel rows");
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
  if (PAIR) {   // the off-diagonal 32 x 32 blocks of every slot's S~ operand stay zero
    for (int e = threadIdx.x; e < Cfg::NB * 8 * 32; e += kOutThreadsTC) {
      const int kb = e / 256, grp = (e / 32) % 8, r = e % 32;
      const int row = grp < 4 ? 32 + r : r;
      *reinterpret_cast<uint4*>(bslot + kb * Cfg::BT + grp * Cfg::B_SBO + row * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
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
      grid_dep_wait();   // S~ and z~ come from the mixing launch
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
        if constexpr (PAIR) {
          // heads 2h and 2h + 1 (32 x 32 tiles): one (8, 32) box per column group onto the diagonal
          mbar_arrive_expect_tx(bfull + kb, 8 * 512 + Cfg::ZRAW);
          for (int e = 0; e < 2; ++e) {
            const int64_t t2 = (b * 2 * g.H + 2 * h + e) * g.M + i;
            for (int gq = 0; gq < 4; ++gq)
              tma_load_4d(slot + (4 * e + gq) * Cfg::B_SBO + 32 * e * 16, &tm_st, bfull + kb, 0, 0, gq,
                          static_cast<int32_t>(t2), pol_s);
            bulk_load(slot + Cfg::BOPS + e * 128, zt + t2 * 32, 128, bfull + kb, pol_s);
          }
        } else {
          mbar_arrive_expect_tx(bfull + kb, Cfg::ST_BYTES + Cfg::ZRAW);
          tma_load_4d(slot, &tm_st, bfull + kb, 0, 0, 0, static_cast<int32_t>(tile), pol_s);
          bulk_load(slot + Cfg::BOPS, zt + tile * D, Cfg::ZRAW, bfull + kb, pol_s);
        }
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
          // d = 64: the output leaves L2 early (evict-first); measured slower at d = 32
          if constexpr (D == 64) {
            tma_store_5d_hint(&tm_o, qst + s * Cfg::QT, 0, h, x, y, z, policy_evict_first());
          } else {
            tma_store_5d(&tm_o, qst + s * Cfg::QT, 0, h, x, y, z);
          }
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
        mbar_arrive(ostore + cs);
        if (D == 64 && !PAIR && c + 1 == g.chunks) {
          // the item's last MMA has read its S~ tile and z~ (each read once, by this
          // CTA): their lines leave L2 without a write-back (measured slower at d = 32)
          const int64_t tile = ((item / g.H) / g.M * g.H + item % g.H) * g.M + (item / g.H) % g.M;
          const int e = 32 * q4 + lane;
          if (e < D * D * 2 / 128) discard_l2_line(reinterpret_cast<const uint8_t*>(St + tile * D * D) + e * 128);
          else if (e < D * D * 2 / 128 + D * 4 / 128)
            discard_l2_line(reinterpret_cast<const uint8_t*>(zt + tile * D) + (e - D * D * 2 / 128) * 128);
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

// ----------------------------------------------------------------- host side

template <int D, bool PAIR>
int run_output(const Problem& p, const __nv_bfloat16* St, const float* zt, cudaStream_t stream) {
  using Cfg = OutCfg<D>;
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
                           static_cast<int>(Cfg::SMEM)) != cudaSuccess)
    return MHLA_ERR_CUDA;
  const int per_sm =
      std::max(1, std::min(occupancy(tc_output<D, PAIR>, kOutThreadsTC, Cfg::SMEM), 512 / Cfg::TMEM_COLS));
  const int grid = static_cast<int>(std::min<int64_t>(n_items, static_cast<int64_t>(sms) * per_sm));
  KernelTimer timer("tc_output", stream);
  const cudaError_t e = launch_dependent(tc_output<D, PAIR>, dim3(grid), dim3(kOutThreadsTC), Cfg::SMEM, stream, tq,
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

}  // namespace mhla
