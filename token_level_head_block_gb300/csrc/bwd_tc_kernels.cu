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
//                 MMA A   num = phi(Q) S~
//                 epilogue den = phi(q) . z~ + eps, dnum = g / den,
//                          dden = -(g . o) / den (CUDA cores)
//                 MMA B   dnum S~^T
//                 MMA C   [dS~ | dz~] += phi(Q)^T [dnum | dden], over the block
//                 dq = (dnum S~^T + dden z~) * [q > 0]; the next chunk's MMA A
//                 runs under MMAs B and C; dS~, dz~ go to a buffer laid out like
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
__device__ __forceinline__ bool bwarp_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abortf) {
  return warp_wait_on(bar, parity, abortf, &g_bwd_error);
}
__device__ __forceinline__ void bdrain(uint64_t* bar, uint32_t parity) { drain_wait_on(bar, parity, &g_bwd_error); }

// 16-byte unit of a row in a 128-byte-swizzled tile (rows of 128 bytes).
__device__ __forceinline__ int swz128(int row) { return row & 7; }

// ============================================================================
// tc_bwd_query
// Work item = (b, query block i, head group of 128 / d heads), head group
// fastest; 128-token chunks.  Per chunk n:
//   MMA A   num = phi(Q) S~                               (accumulator n % 2)
//   epi 1   den = phi(q) . z~ + eps (CUDA cores), dnum = g / den written over
//           g, dden = -(g . num) / den^2
//   MMA B   dnum S~^T                                      (accumulator n % 2)
//   MMA C   [dS~ | dz~] += phi(Q)^T [dnum | dden]          (one accumulator per item)
//   epi 2   dq = (dnum S~^T + dden z~) * [q > 0] written over dnum, stored by TMA
//   epi 3   after the item's last chunk: dS~, dz~ to a buffer laid out like the
//           forward's summaries, so the forward's mixing GEMM with W^T turns
//           them into dS, dz
// Roles (24 warps): q and S~ producer, MMA issuer, dq store issuer, dout
// producer, a phi warpgroup, two epilogue-1 and two epilogue-2 warpgroups
// (each pair splits the heads of the item).  Every hand-off is an mbarrier, so the phases of neighbouring
// chunks overlap: MMA A of chunk n + 1 runs under epilogue 1 of chunk n, and
// epilogue 2 of chunk n under epilogue 1 of chunk n + 1.
// ============================================================================
template <int D>
struct BqCfg {
  static constexpr int HP = 128 / D;              // heads per work item
  static constexpr int C = 128;                   // tokens per chunk (MMA M)
  static constexpr int ROWB = D * 2;
  static constexpr int TILE = C * ROWB;           // one head's [128][D] token tile
  static constexpr int HT = HP * TILE;            // all heads of a chunk (32 KB)
  static constexpr uint32_t SBO = 8 * ROWB;
  static constexpr uint32_t LAYOUT = D == 64 ? 2u : 4u;
  static constexpr int ST = D * D * 2;            // one S~ tile (row-major, swizzled like a token tile)
  static constexpr int NQ = 3;                    // q stages
  static constexpr int NG = 2;                    // dout stages: dout, then dnum, then dq
  static constexpr int MASKB = HP * C * (D / 8);  // q > 0 bits of a chunk
  static constexpr int DDB = 2 * C * 16;          // dden operand: 2 groups of 8 columns, unswizzled MN-major
  static constexpr int Q_OFF = 0;
  static constexpr int G_OFF = Q_OFF + NQ * HT;
  static constexpr int SZ_OFF = G_OFF + NG * HT;             // [2] slots of HP S~ tiles
  static constexpr int ZRAW_OFF = SZ_OFF + 2 * HP * ST;      // [2][HP][D] z~ float32
  static constexpr int DDB_OFF = ZRAW_OFF + 2 * HP * D * 4;  // [NG] dden operands
  static constexpr int DDS_OFF = DDB_OFF + NG * DDB;         // [NG][HP][C] dden float32
  static constexpr int MASK_OFF = DDS_OFF + NG * HP * C * 4; // [NG] q > 0 bits
  static constexpr int CTRL_OFF = MASK_OFF + NG * MASKB;
  static constexpr size_t SMEM = CTRL_OFF + 512 + 1024;
  static constexpr int CCOL = 256;                // [dS~ | dz~]: 128 + 16 columns
  static constexpr int TMEM_COLS = 512;           // accumulators 0 and 1 at 0 and 128
};
constexpr int kBqThreads = 768;

// q > 0 bits of the eight bf16 values of a 16-byte unit (bit e for element e).
// Per 16-bit half: adding 0x7FFF to the magnitude sets the half's top bit
// exactly when the magnitude is non-zero (no carry reaches the next half); the
// sign bit then clears it for negative values.
__device__ __forceinline__ uint32_t positive_bits(uint4 q) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  uint32_t p[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) p[k] = ((w[k] & 0x7FFF7FFFu) + 0x7FFF7FFFu) & ~w[k] & 0x80008000u;
  // word k: low half to bit 2k, high half to bit 2k + 16, then folded to 2k + 1
  const uint32_t c = (p[0] >> 15) | (p[1] >> 13) | (p[2] >> 11) | (p[3] >> 9);
  return (c | (c >> 15)) & 0xFFu;
}

template <int D>
__global__ void __launch_bounds__(kBqThreads, 1)
tc_bwd_query(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_g,
             const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_st, TcGeom g,
             int32_t G, int64_t n_items, int phi_kind, float eps, const float* __restrict__ zt,
             __nv_bfloat16* __restrict__ dSbuf) {
  using Cfg = BqCfg<D>;
  constexpr int HP = Cfg::HP, NQ = Cfg::NQ, NG = Cfg::NG;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  uint8_t* qst = smem + Cfg::Q_OFF;
  uint8_t* gst = smem + Cfg::G_OFF;
  uint8_t* sz = smem + Cfg::SZ_OFF;
  float* zraw = reinterpret_cast<float*>(smem + Cfg::ZRAW_OFF);
  uint8_t* ddb = smem + Cfg::DDB_OFF;
  float* dds = reinterpret_cast<float*>(smem + Cfg::DDS_OFF);
  uint8_t* masks = smem + Cfg::MASK_OFF;
  uint64_t* qfull = reinterpret_cast<uint64_t*>(smem + Cfg::CTRL_OFF);
  uint64_t* qempty = qfull + NQ;     // MMA C of the chunk done
  uint64_t* phid = qempty + NQ;      // phi applied (128 arrivals)
  uint64_t* gfull = phid + NQ;
  uint64_t* gempty = gfull + NG;     // the dq store has read the stage
  uint64_t* mfull = gempty + NG;     // q > 0 bits written (128)
  uint64_t* mempty = mfull + NG;     // q > 0 bits read by epilogue 2 (256)
  uint64_t* dqready = mempty + NG;   // dq written over the stage (256)
  uint64_t* sfull = dqready + NG;    // [2] S~ tiles and z~ of an item landed
  uint64_t* sempty = sfull + 2;      // [2] the item's last chunk is through epilogue 2 (256)
  uint64_t* tfullA = sempty + 2;     // [2] MMA A done
  uint64_t* e1done = tfullA + 2;     // [2] epilogue 1 done (256)
  uint64_t* mmadone = e1done + 2;    // [2] MMAs B and C done
  uint64_t* accfree = mmadone + 2;   // [2] epilogue 2 has read the accumulator (256)
  uint64_t* cfree = accfree + 2;     // epilogue 3 has read [dS~ | dz~] (256)
  uint64_t* fin = cfree + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fin + 1);
  volatile uint32_t* abortf = tmem_slot + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NQ; ++s) {
      mbar_init(qfull + s, 1);
      mbar_init(qempty + s, 1);
      mbar_init(phid + s, 128);
    }
    for (int s = 0; s < NG; ++s) {
      mbar_init(gfull + s, 1);
      mbar_init(gempty + s, 1);
      mbar_init(mfull + s, 128);
      mbar_init(mempty + s, 256);
      mbar_init(dqready + s, 256);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(sfull + s, 1);
      mbar_init(sempty + s, 256);
      mbar_init(tfullA + s, 1);
      mbar_init(e1done + s, 256);
      mbar_init(mmadone + s, 1);
      mbar_init(accfree + s, 256);
    }
    mbar_init(cfree, 256);
    mbar_init(fin, 1);
    *abortf = 0u;
    fence_mbar_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_g);
    prefetch_tmap(&tm_dq);
    prefetch_tmap(&tm_st);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  // the dden operands: only their first HP columns are ever written
  for (int e = threadIdx.x; e < NG * Cfg::DDB / 16; e += kBqThreads)
    reinterpret_cast<uint4*>(ddb)[e] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // item -> (grp, i, b), head group fastest
  auto item_coords = [&](int64_t item, int32_t& grp, int32_t& i, int32_t& b) {
    grp = static_cast<int32_t>(item % G);
    const int64_t rest = item / G;
    i = static_cast<int32_t>(rest % g.M);
    b = static_cast<int32_t>(rest / g.M);
  };

  if (warp == 0) {
    // ------------------------------------------- q and S~ producer
    if (lane == 0) {
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_s = policy_evict_last();
      uint32_t qfills[NQ] = {}, sfills[2] = {};
      int qs = 0;
      uint32_t qph = 0, k = 0;
      bool ok = true;
      for (int64_t item = blockIdx.x; ok && item < n_items; item += gridDim.x, ++k) {
        int32_t grp, i, b;
        item_coords(item, grp, i, b);
        const int sl = static_cast<int>(k & 1u);
        if (!bwait(sempty + sl, ((k >> 1) & 1u) ^ 1u, abortf)) break;
        uint32_t bytes = 0;
        for (int hh = 0; hh < HP; ++hh)
          if (grp * HP + hh < g.H) bytes += Cfg::ST + D * 4;
        mbar_arrive_expect_tx(sfull + sl, bytes);
        for (int hh = 0; hh < HP; ++hh) {
          const int32_t h = grp * HP + hh;
          if (h >= g.H) continue;
          const int64_t tile = (static_cast<int64_t>(b) * g.H + h) * g.M + i;
          tma_load_2d(sz + (sl * HP + hh) * Cfg::ST, &tm_st, sfull + sl, 0, static_cast<int32_t>(tile * D), pol_s);
          bulk_load(zraw + (sl * HP + hh) * D, zt + tile * D, D * 4, sfull + sl, pol_s);
        }
        ++sfills[sl];
        for (int c = 0; c < g.chunks; ++c) {
          if (!bwait(qempty + qs, qph ^ 1u, abortf)) { ok = false; break; }
          int32_t x, y, z;
          chunk_coords(g, i, c, b, x, y, z);
          mbar_arrive_expect_tx(qfull + qs, Cfg::HT);
#pragma unroll
          for (int hh = 0; hh < HP; ++hh)   // heads >= H read zeros
            tma_load_5d(qst + qs * Cfg::HT + hh * Cfg::TILE, &tm_q, qfull + qs, 0, grp * HP + hh, x, y, z, pol_q);
          ++qfills[qs];
          if (++qs == NQ) { qs = 0; qph ^= 1u; }
        }
      }
      for (int s = 0; s < NQ; ++s)
        if (qfills[s]) bdrain(qfull + s, (qfills[s] - 1) & 1u);
      for (int s = 0; s < 2; ++s)
        if (sfills[s]) bdrain(sfull + s, (sfills[s] - 1) & 1u);
    }
  } else if (warp == 3) {
    // ------------------------------------------- dout producer
    if (lane == 0) {
      const uint64_t pol_g = policy_evict_first();
      uint32_t gfills[NG] = {};
      int gs = 0;
      uint32_t gph = 0;
      bool ok = true;
      for (int64_t item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        int32_t grp, i, b;
        item_coords(item, grp, i, b);
        for (int c = 0; c < g.chunks; ++c) {
          if (!bwait(gempty + gs, gph ^ 1u, abortf)) { ok = false; break; }
          int32_t x, y, z;
          chunk_coords(g, i, c, b, x, y, z);
          mbar_arrive_expect_tx(gfull + gs, Cfg::HT);
#pragma unroll
          for (int hh = 0; hh < HP; ++hh)
            tma_load_5d(gst + gs * Cfg::HT + hh * Cfg::TILE, &tm_g, gfull + gs, 0, grp * HP + hh, x, y, z, pol_g);
          ++gfills[gs];
          if (++gs == NG) { gs = 0; gph ^= 1u; }
        }
      }
      for (int s = 0; s < NG; ++s)
        if (gfills[s]) bdrain(gfull + s, (gfills[s] - 1) & 1u);
    }
  } else if (warp == 2) {
    // ------------------------------------------- dq store issuer
    if (lane == 0) {
      int gs = 0;
      uint32_t gph = 0;
      bool ok = true;
      for (int64_t item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        int32_t grp, i, b;
        item_coords(item, grp, i, b);
        for (int c = 0; c < g.chunks; ++c) {
          if (!bwait(dqready + gs, gph, abortf)) { ok = false; break; }
          int32_t x, y, z;
          chunk_coords(g, i, c, b, x, y, z);
          for (int hh = 0; hh < HP; ++hh)
            if (grp * HP + hh < g.H)
              tma_store_5d_hint(&tm_dq, gst + gs * Cfg::HT + hh * Cfg::TILE, 0, grp * HP + hh, x, y, z,
                                policy_evict_first());
          bulk_commit_group();
          bulk_wait_group_read<0>();      // the stage has been read: back to the dout producer
          mbar_arrive(gempty + gs);
          if (++gs == NG) { gs = 0; gph ^= 1u; }
        }
      }
      bulk_wait_group0();
    }
  } else if (warp == 1) {
    // ------------------------------------------- MMA issuer
    // Two streams in chunk order, issued as their inputs become ready: MMA A
    // of chunk nA (q stage phi'd, S~ landed, accumulator nA % 2 read out by
    // epilogue 2 of chunk nA - 2) and MMAs B, C of chunk nB < nA (epilogue 1
    // done; for an item's first chunk also [dS~ | dz~] read out).
    if (lane == 0) {
      constexpr uint32_t idA = idesc_bf16_f32(128, D, /*a K-major*/ false, /*b MN-major*/ true);
      constexpr uint32_t idB = idesc_bf16_f32(128, D, /*a K-major*/ false, /*b K-major*/ false);
      constexpr uint32_t idC = idesc_bf16_f32(128, 128, /*a MN-major*/ true, /*b MN-major*/ true);
      constexpr uint32_t idZ = idesc_bf16_f32(128, 16, /*a MN-major*/ true, /*b MN-major*/ true);
      int64_t itemA = blockIdx.x, itemB = blockIdx.x;
      int cA = 0, cB = 0;
      uint32_t nA = 0, nB = 0, kA = 0, kB = 0;
      uint64_t t0 = globaltimer();
      uint32_t idle = 0;
      // diagnostic hook (stall_hook.cuh): this issuer sees no completion at all
      const bool stalled = stall_this_warp();
      const uint64_t limit_ns = stalled ? c_stall_ns : kWaitLimitNs;
      while (itemB < n_items) {
        bool prog = false;
        if (!stalled && itemA < n_items && nA < nB + 2) {
          const uint32_t s = nA % NQ, acc = nA & 1u, sl = kA & 1u;
          if ((cA != 0 || mbar_test_wait(sfull + sl, (kA >> 1) & 1u)) &&
              mbar_test_wait(phid + s, (nA / NQ) & 1u) && mbar_test_wait(accfree + acc, ((nA >> 1) & 1u) ^ 1u)) {
            tc_fence_after();
#pragma unroll
            for (int hh = 0; hh < HP; ++hh) {
              const uint32_t qa = smem_u32(qst + s * Cfg::HT + hh * Cfg::TILE);
              const uint32_t sb = smem_u32(sz + (sl * HP + hh) * Cfg::ST);
#pragma unroll
              for (int ks = 0; ks < D / 16; ++ks)
                mma_bf16(tmem + acc * 128 + hh * D, smem_desc(qa + ks * 32, 16, Cfg::SBO, Cfg::LAYOUT),
                         smem_desc(sb + ks * 2 * Cfg::SBO, Cfg::ST, Cfg::SBO, Cfg::LAYOUT), idA, ks > 0 ? 1u : 0u);
            }
            mma_commit(tfullA + acc);
            ++nA;
            if (++cA == g.chunks) { cA = 0; itemA += gridDim.x; ++kA; }
            prog = true;
          }
        }
        if (nB < nA) {
          const uint32_t acc = nB & 1u, sl = kB & 1u, s = nB % NQ, gs = nB % NG;
          if (mbar_test_wait(e1done + acc, (nB >> 1) & 1u) && (cB != 0 || mbar_test_wait(cfree, (kB & 1u) ^ 1u))) {
            tc_fence_after();
#pragma unroll
            for (int hh = 0; hh < HP; ++hh) {
              const uint32_t da = smem_u32(gst + gs * Cfg::HT + hh * Cfg::TILE);
              const uint32_t sb = smem_u32(sz + (sl * HP + hh) * Cfg::ST);
#pragma unroll
              for (int ks = 0; ks < D / 16; ++ks)
                mma_bf16(tmem + acc * 128 + hh * D, smem_desc(da + ks * 32, 16, Cfg::SBO, Cfg::LAYOUT),
                         smem_desc(sb + ks * 32, 16, Cfg::SBO, Cfg::LAYOUT), idB, ks > 0 ? 1u : 0u);
            }
            const uint32_t qa = smem_u32(qst + s * Cfg::HT), da = smem_u32(gst + gs * Cfg::HT);
            const uint32_t zb = smem_u32(ddb + gs * Cfg::DDB);
#pragma unroll
            for (int ks = 0; ks < Cfg::C / 16; ++ks) {
              const uint64_t adesc = smem_desc(qa + ks * 2 * Cfg::SBO, Cfg::TILE, Cfg::SBO, Cfg::LAYOUT);
              const uint32_t accum = (cB > 0 || ks > 0) ? 1u : 0u;
              mma_bf16(tmem + Cfg::CCOL, adesc, smem_desc(da + ks * 2 * Cfg::SBO, Cfg::TILE, Cfg::SBO, Cfg::LAYOUT),
                       idC, accum);
              mma_bf16(tmem + Cfg::CCOL + 128, adesc, smem_desc(zb + ks * 256, 128, Cfg::C * 16, 0), idZ, accum);
            }
            mma_commit(mmadone + acc);
            mma_commit(qempty + s);
            ++nB;
            if (++cB == g.chunks) { cB = 0; itemB += gridDim.x; ++kB; }
            prog = true;
          }
        }
        if (prog) {
          idle = 0;
          t0 = globaltimer();
        } else if ((++idle & 63u) == 0) {
          if (*abortf) break;
          if (globaltimer() - t0 > limit_ns || idle >= kWaitLimitPolls) {
            *abortf = 1u;
            atomicOr(&g_bwd_error, 1u);
            break;
          }
        }
      }
      mma_commit(fin);
      bdrain(fin, 0);
    }
  } else if (warp < 8) {
    // ------------------------------------------- phi on q, and the q > 0 bits
    const int t4 = threadIdx.x - 128;
    const bool add_eps = phi_kind == MHLA_PHI_RELU_EPS;
    const __nv_bfloat162 eps2 = __float2bfloat162_rn(eps);
    int qs = 0, gs = 0;
    uint32_t qph = 0, gph = 0;
    bool ok = true;
    for (int64_t item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      for (int c = 0; c < g.chunks; ++c) {
        if (!bwarp_wait(qfull + qs, qph, abortf) || !bwarp_wait(mempty + gs, gph ^ 1u, abortf)) { ok = false; break; }
        uint8_t* qs_base = qst + qs * Cfg::HT;
        uint8_t* mk = masks + gs * Cfg::MASKB;
#pragma unroll 4
        for (int e = t4; e < Cfg::HT / 16; e += 128) {
          const int hh = e / (Cfg::TILE / 16), rem = e % (Cfg::TILE / 16);
          const int t = rem / (D / 8), p = rem % (D / 8);
          uint4* ptr = reinterpret_cast<uint4*>(qs_base) + e;
          const uint4 raw = *ptr;
          mk[(hh * Cfg::C + t) * (D / 8) + (p ^ swz<D>(t))] = static_cast<uint8_t>(positive_bits(raw));
          *ptr = phi8_packed(raw, add_eps, eps2);
        }
        fence_proxy_async_smem();
        mbar_arrive(phid + qs);
        mbar_arrive(mfull + gs);
        if (++qs == NQ) { qs = 0; qph ^= 1u; }
        if (++gs == NG) { gs = 0; gph ^= 1u; }
      }
    }
  } else {
    const int q4 = warp & 3;
    const int ew = (warp >> 2) & 1;                 // warpgroup of the pair: heads ew, ew + 2, ...
    const int row = 32 * q4 + lane;                 // token row of the chunk = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * q4) << 16);
    int qs = 0, gs = 0;
    uint32_t qph = 0, gph = 0, n = 0, k = 0;
    bool ok = true;
    if (warp < 16) {
      // ----------------------------------------- epilogue 1: den, dnum, dden
      for (int64_t item = blockIdx.x; ok && item < n_items; item += gridDim.x, ++k) {
        const int32_t grp = static_cast<int32_t>(item % G);
        const int sl = static_cast<int>(k & 1u);
        for (int c = 0; c < g.chunks; ++c, ++n) {
          const uint32_t acc = n & 1u;
          if (!bwarp_wait(tfullA + acc, (n >> 1) & 1u, abortf) || !bwarp_wait(gfull + gs, gph, abortf) ||
              !bwarp_wait(phid + qs, qph, abortf) || !bwarp_wait(sfull + sl, (k >> 1) & 1u, abortf)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int hh = ew; hh < HP; hh += 2) {
            uint32_t nv[32];
            tmem_ld_x32(lane_base + acc * 128 + hh * D, nv);
            // den = phi(q_t) . z~ + eps on the CUDA cores, from this row of the q tile
            const uint8_t* qrow = qst + qs * Cfg::HT + hh * Cfg::TILE + row * Cfg::ROWB;
            const float* zr = zraw + (sl * HP + hh) * D;
            float dpart[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int u = 0; u < D / 8; ++u) {
              const uint4 qv = *reinterpret_cast<const uint4*>(qrow + ((u ^ swz<D>(row)) * 16));
              const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
              const float4 za = *reinterpret_cast<const float4*>(zr + 8 * u);
              const float4 zb = *reinterpret_cast<const float4*>(zr + 8 * u + 4);
              const float zz[8] = {za.x, za.y, za.z, za.w, zb.x, zb.y, zb.z, zb.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 q2 = *reinterpret_cast<const __nv_bfloat162*>(&qw[e]);
                dpart[e] = fmaf(__low2float(q2), zz[2 * e], dpart[e]);
                dpart[e] = fmaf(__high2float(q2), zz[2 * e + 1], dpart[e]);
              }
            }
            const bool valid = grp * HP + hh < g.H;
            // heads past H (zero inputs, no S~ loaded) give exact zeros
            const float inv = valid ? 1.0f / ((dpart[0] + dpart[1]) + (dpart[2] + dpart[3]) + eps) : 0.0f;
            uint8_t* grow = gst + gs * Cfg::HT + hh * Cfg::TILE + row * Cfg::ROWB;
            float gpart[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int h2 = 0; h2 < D / 32; ++h2) {
              if (h2 > 0) tmem_ld_x32(lane_base + acc * 128 + hh * D + 32 * h2, nv);
              tmem_ld_wait();
#pragma unroll
              for (int u4 = 0; u4 < 4; ++u4) {
                const int u = 4 * h2 + u4;
                uint4* gp = reinterpret_cast<uint4*>(grow + ((u ^ swz<D>(row)) * 16));
                const uint4 gr = *gp;
                const uint32_t gw[4] = {gr.x, gr.y, gr.z, gr.w};
                uint32_t ow[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const __nv_bfloat162 g2 = *reinterpret_cast<const __nv_bfloat162*>(&gw[e]);
                  const float g0 = __low2float(g2), g1 = __high2float(g2);
                  gpart[e] = fmaf(g0, __uint_as_float(nv[8 * u4 + 2 * e]), gpart[e]);
                  gpart[e] = fmaf(g1, __uint_as_float(nv[8 * u4 + 2 * e + 1]), gpart[e]);
                  ow[e] = pack_bf16(g0 * inv, g1 * inv);
                }
                *gp = make_uint4(ow[0], ow[1], ow[2], ow[3]);   // dnum over g (this row is this thread's)
              }
            }
            const float go = (gpart[0] + gpart[1]) + (gpart[2] + gpart[3]);
            const float dden = valid ? -go * inv * inv : 0.0f;   // -(g . num / den) / den
            dds[(gs * HP + hh) * Cfg::C + row] = dden;
            // column hh of the dden operand (token row, unswizzled MN-major)
            *reinterpret_cast<__nv_bfloat16*>(ddb + gs * Cfg::DDB + row * 16 + hh * 2) = __float2bfloat16_rn(dden);
          }
          fence_proxy_async_smem();
          tc_fence_before();
          mbar_arrive(e1done + acc);
          if (++qs == NQ) { qs = 0; qph ^= 1u; }
          if (++gs == NG) { gs = 0; gph ^= 1u; }
        }
      }
    } else {
      // ----------------------------------------- epilogue 2: dq; epilogue 3: dS~, dz~
      for (int64_t item = blockIdx.x; ok && item < n_items; item += gridDim.x, ++k) {
        int32_t grp, i, b;
        item_coords(item, grp, i, b);
        const int sl = static_cast<int>(k & 1u);
        for (int c = 0; c < g.chunks; ++c, ++n) {
          const uint32_t acc = n & 1u, aph = (n >> 1) & 1u;
          if (!bwarp_wait(mmadone + acc, aph, abortf) || !bwarp_wait(e1done + acc, aph, abortf) ||
              !bwarp_wait(mfull + gs, gph, abortf) || !bwarp_wait(sfull + sl, (k >> 1) & 1u, abortf)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int hh = ew; hh < HP; hh += 2) {
            uint32_t v[32];
            tmem_ld_x32(lane_base + acc * 128 + hh * D, v);
            const float* zr = zraw + (sl * HP + hh) * D;
            const float ddv = dds[(gs * HP + hh) * Cfg::C + row];
            const uint8_t* mrow = masks + gs * Cfg::MASKB + (hh * Cfg::C + row) * (D / 8);
            uint64_t mbits;
            if constexpr (D == 64) {
              mbits = *reinterpret_cast<const uint64_t*>(mrow);
            } else {
              mbits = *reinterpret_cast<const uint32_t*>(mrow);
            }
            uint8_t* orow = gst + gs * Cfg::HT + hh * Cfg::TILE + row * Cfg::ROWB;
#pragma unroll
            for (int h2 = 0; h2 < D / 32; ++h2) {
              if (h2 > 0) tmem_ld_x32(lane_base + acc * 128 + hh * D + 32 * h2, v);
              tmem_ld_wait();
#pragma unroll
              for (int u4 = 0; u4 < 4; ++u4) {
                const int u = 4 * h2 + u4;
                const uint32_t bits = static_cast<uint32_t>(mbits >> (8 * u)) & 0xFFu;
                const float4 za = *reinterpret_cast<const float4*>(zr + 8 * u);
                const float4 zb = *reinterpret_cast<const float4*>(zr + 8 * u + 4);
                const float zz[8] = {za.x, za.y, za.z, za.w, zb.x, zb.y, zb.z, zb.w};
                uint32_t ow[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int c0 = 8 * u4 + 2 * e;
                  const float a0 = (bits >> (2 * e)) & 1u ? fmaf(ddv, zz[2 * e], __uint_as_float(v[c0])) : 0.0f;
                  const float a1 = (bits >> (2 * e + 1)) & 1u ? fmaf(ddv, zz[2 * e + 1], __uint_as_float(v[c0 + 1])) : 0.0f;
                  ow[e] = pack_bf16(a0, a1);
                }
                *reinterpret_cast<uint4*>(orow + ((u ^ swz<D>(row)) * 16)) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
              }
            }
          }
          tc_fence_before();
          mbar_arrive(accfree + acc);
          fence_proxy_async_smem();
          mbar_arrive(dqready + gs);
          mbar_arrive(mempty + gs);
          if (c + 1 == g.chunks) {
            // ---- epilogue 3: row = (head hh, channel r) of phi(Q)^T
            const int hh = row / D, r = row % D;
            const int32_t h = grp * HP + hh;
            constexpr int32_t PER_BH = (D + 1) * D;
            const int64_t col = (static_cast<int64_t>(b) * g.H + h) * PER_BH + r * D + ew * (D / 2);
            uint4* drow = reinterpret_cast<uint4*>(dSbuf + ((col >> 7) * g.M + i) * 128 + (col & 127));
            uint32_t vz = 0;
            tmem_ld_x1(lane_base + Cfg::CCOL + 128 + hh, vz);
            uint32_t v[D / 2];
            if constexpr (D == 64) {
              tmem_ld_x32(lane_base + Cfg::CCOL + hh * D + ew * 32, v);
            } else {
              tmem_ld_x16(lane_base + Cfg::CCOL + hh * D + ew * 16, v);
            }
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(cfree);
            if (h < g.H) {
#pragma unroll
              for (int q = 0; q < D / 16; ++q)
                drow[q] = make_uint4(pack_bf16(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
                                     pack_bf16(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                                     pack_bf16(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                                     pack_bf16(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
            }
            if (h < g.H && ew == 0) {
              const int64_t zcol = (static_cast<int64_t>(b) * g.H + h) * PER_BH + D * D + r;
              dSbuf[((zcol >> 7) * g.M + i) * 128 + (zcol & 127)] = __float2bfloat16_rn(__uint_as_float(vz));
            }
            mbar_arrive(sempty + sl);
          }
          if (++gs == NG) { gs = 0; gph ^= 1u; }
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
constexpr int kBkThreads = 256;                 // warps 0-7: phi, MMA issue (thread 0), epilogue
constexpr int kBkAll = kBkThreads + 32;          // + warp 8: stores and k, v loads
constexpr uint32_t kBkBar = 1;                   // named barrier of warps 0-7

// Warps 0-7 take every chunk through phi, the MMAs and the epilogue; warp 8
// stores a chunk's dk, dv as soon as its epilogue is written and loads the
// chunk two ahead into the stage once the stores have read it, so each load
// has a whole chunk of work to land under.
template <int D>
__global__ void __launch_bounds__(kBkAll, 1)
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
  uint64_t* be = bl + 4;                                               // [2] dk, dv of the stage written
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bl + 6);
  volatile uint32_t* abortf = tmem_slot + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(bl, 1);
    mbar_init(bl + 1, 1);
    mbar_init(bs, 1);
    mbar_init(bm, 1);
    mbar_init(be, 1);
    mbar_init(be + 1, 1);
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
  for (int e = tid; e < Cfg::EXT / 16; e += kBkAll) {
    const int r = e / 8, p = e % 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if ((p ^ swz128(r)) == 0) v.x = 0x3F803F80u;   // bf16 1.0, 1.0
    reinterpret_cast<uint4*>(ones)[e] = v;
  }
  for (int e = tid; e < HP * Cfg::ZB / 16; e += kBkAll)
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

  if (warp == kBkThreads / 32) {
    // ------------------------------------------------ stores and k, v loads
    if (lane == 0) {
      uint32_t n_l[2] = {0, 0};
      // the chunk sequence of this CTA: (item, c) in order, k = position
      int64_t l_item = blockIdx.x;     // next chunk to load
      int l_c = 0;
      auto load_next = [&](int st) {
        if (l_item >= n_items) return;
        issue_kv(st, l_item, l_c);
        ++n_l[st];
        if (++l_c == g.chunks) { l_c = 0; l_item += gridDim.x; }
      };
      load_next(0);
      load_next(1);
      uint32_t k = 0;
      for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
        int32_t grp, j, b;
        item_coords(item, grp, j, b);
        bool ok = true;
        for (int c = 0; c < g.chunks; ++c, ++k) {
          const int st = static_cast<int>(k & 1u);
          if (!bwait(be + st, (k >> 1) & 1u, abortf)) { ok = false; break; }
          uint8_t* kt = stages + st * Cfg::STAGE;
          uint8_t* vt = kt + Cfg::HT;
          int32_t x, y, z;
          chunk_coords(g, j, c, b, x, y, z);
          for (int hh = 0; hh < HP; ++hh) {
            if (grp * HP + hh >= g.H) continue;
            tma_store_5d_hint(&tm_dk, kt + hh * Cfg::TILE, 0, grp * HP + hh, x, y, z, policy_evict_first());
            tma_store_5d_hint(&tm_dv, vt + hh * Cfg::TILE, 0, grp * HP + hh, x, y, z, policy_evict_first());
          }
          bulk_commit_group();
          if (l_item < n_items) {
            bulk_wait_group_read<0>();   // the stores have read the stage: the chunk two ahead loads into it
            load_next(st);
          }
        }
        if (!ok) break;
      }
      bulk_wait_group0();
      for (int st = 0; st < 2; ++st)
        if (n_l[st]) bdrain(bl + st, (n_l[st] - 1) & 1u);
    }
  } else {
    // ------------------------------------------------ warps 0-7
    uint32_t n_s = 0, n_m = 0, c_s = 0, c_m = 0;
    uint32_t c_l[2] = {0, 0};
    uint32_t chunk_no = 0;   // chunks processed by this CTA (stage = chunk_no & 1)
    if (tid == 0 && static_cast<int64_t>(blockIdx.x) < n_items) {
      issue_ds(blockIdx.x);
      n_s = 1;
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
      if (!named_bar_and(kBkBar, kBkThreads, bwait(bs, c_s & 1u, abortf))) break;
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
      named_bar_sync(kBkBar, kBkThreads);

      for (int c = 0; c < g.chunks; ++c, ++chunk_no) {
        const int st = chunk_no & 1;
        uint8_t* kt = stages + st * Cfg::STAGE;
        uint8_t* vt = kt + Cfg::HT;
        uint8_t* mask = masks + st * Cfg::MASK_BYTES;
        const bool last = c + 1 == g.chunks;
        const int64_t nitem = item + gridDim.x;
        if (!named_bar_and(kBkBar, kBkThreads, bwait(bl + st, c_l[st] & 1u, abortf))) { ok = false; break; }
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
        named_bar_sync(kBkBar, kBkThreads);

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
            mma_bf16(dkc, smem_desc(smem_u32(ones), 16, 1024, 2),
                     smem_desc(smem_u32(zb + hh * Cfg::ZB), 16, 1024, 2), ide, 1u);
          }
          mma_commit(bm);
          ++n_m;
        }
        if (!named_bar_and(kBkBar, kBkThreads, bwait(bm, c_m & 1u, abortf))) { ok = false; break; }
        ++c_m;
        tc_fence_after();
        if (tid == 0 && last && nitem < n_items) {   // dS, dz consumed by this item's last MMAs
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
        named_bar_sync(kBkBar, kBkThreads);
        if (tid == 0) mbar_arrive(be + st);   // warp 8 stores the stage, then reloads it
      }
    }
    if (tid == 0) {
      if (n_s > c_s) bdrain(bs, (n_s - 1) & 1u);
      if (n_m > c_m) bdrain(bm, (n_m - 1) & 1u);
    }
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
// One CTA per (i tile of 256 as two 128-row MMA halves, so each j row of S is
// read once for both; j tile of up to 256; split of the column groups).  Warp 0
// loads 64-column halves of a group into a 3-stage ring, warp 1 issues the MMAs,
// warps 4-7 write the float32 tile with 16-byte stores.
// ============================================================================
struct DwCfg {
  static constexpr int IT = 256;                  // rows i per tile (two MMA M halves)
  static constexpr int JT = 256;                  // rows j per tile (MMA N, at most)
  static constexpr int A_BYTES = IT * 128;        // [256][64] K-major, 128-byte swizzle
  static constexpr int B_BYTES = JT * 128;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int NS = 3;
  static constexpr size_t SMEM = static_cast<size_t>(NS) * STAGE + 256 + 1024;
  static constexpr int TMEM_COLS = 512;           // the two halves' accumulators at 0 and 256
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
        tma_load_3d(base, &tm_a, full + s, half * 64, i0, grp, pol);            // 256 rows; i >= M read zeros
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
        for (int mh = 0; mh < 2; ++mh)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tmem + mh * 256, smem_desc(base + mh * 128 * 128 + ks * 32, 16, 1024, 2),
                     smem_desc(base + Cfg::A_BYTES + ks * 32, 16, 1024, 2), idesc, (st > 0 || ks > 0) ? 1u : 0u);
        mma_commit(empty + s);
        if (++s == Cfg::NS) { s = 0; ph ^= 1u; }
      }
      mma_commit(done);
      bdrain(done, 0);
    }
  } else if (warp >= 4) {
    // warp 4 + q4 reads TMEM lanes 32 q4 .. 32 q4 + 31 of both halves
    const int q4 = warp & 3;
    const bool ok = __all_sync(0xffffffffu, bwait(done, 0, abortf));
    if (ok) {
      tc_fence_after();
      for (int mh = 0; mh < 2; ++mh) {
        const int32_t i = i0 + mh * 128 + 32 * q4 + lane;
        const uint32_t tb = tmem + mh * 256 + (static_cast<uint32_t>(32 * q4) << 16);
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
            if (j0 + cc + 32 <= M && M % 4 == 0) {   // 16-byte stores: each lane writes 128 contiguous bytes
              float4* dst = reinterpret_cast<float4*>(prow + j0 + cc);
#pragma unroll
              for (int e = 0; e < 8; ++e)
                dst[e] = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                     __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (j0 + cc + e < M) prow[j0 + cc + e] = __uint_as_float(v[e]);
            }
          }
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

// dW = the partial products summed over the splits in a fixed order: 64
// outputs per CTA, four threads per output each summing a fixed quarter of
// the splits in order, then the quarters added in order (deterministic; four
// loads in flight per output instead of one).
constexpr int kDwrOut = 64;
__global__ void __launch_bounds__(256) tc_dw_reduce(const float* __restrict__ part, float* __restrict__ dW,
                                                    int64_t MM, int32_t nsplit) {
  __shared__ float quarter[4][kDwrOut];
  const int o = threadIdx.x % kDwrOut, q = threadIdx.x / kDwrOut;
  const int64_t x = static_cast<int64_t>(blockIdx.x) * kDwrOut + o;
  const int32_t k0 = nsplit * q / 4, k1 = nsplit * (q + 1) / 4;
  float s = 0.0f;
  if (x < MM) {
#pragma unroll 4
    for (int32_t k = k0; k < k1; ++k) s += part[k * MM + x];
  }
  quarter[q][o] = s;
  __syncthreads();
  if (q == 0 && x < MM) dW[x] = ((quarter[0][o] + quarter[1][o]) + quarter[2][o]) + quarter[3][o];
}

// ----------------------------------------------------------------- host side

struct BwdLayout {
  size_t wb_off, wbt_off, sbuf_off, dsbuf_off, st_off, zt_off, part_off, total;
  int64_t Mp, ngroups;
  int32_t n_it, n_jt, JN, nsplit;
};

// CTAs the dW product is split over: every split writes an M x M float32 tile
// that the reduction reads back, so large tiles take about two thirds of a
// GB300's SMs (M = 256, DiT-S/2: 152 splits 46 us, 100: 40, 38: 49) and small ones
// one per SM (M = 64: 152 splits 27 us, 100: 30); constants, so that the workspace
// size does not depend on the device.
inline int64_t dw_target_ctas(int64_t M) { return M >= 192 ? 100 : 152; }

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
      std::max<int64_t>(1, std::min<int64_t>(L.ngroups, (dw_target_ctas(p.M) + tiles - 1) / tiles)));
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
      tc_dw_reduce<<<static_cast<unsigned>((MM + kDwrOut - 1) / kDwrOut), 256, 0, stream>>>(part, bo.dW, MM,
                                                                                            L.nsplit);
      if (cudaGetLastError() != cudaSuccess) return MHLA_ERR_CUDA;
    }
    rc = tc_run_mix(p, WbT, L.Mp, dSbuf, St, zt, stream, /*discard_input=*/true);   // dS~ is not read again
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
    tc_bwd_key<D><<<grid, kBkAll, Cfg::SMEM, stream>>>(tk, tv, tdk, tdv, tds, geo, G, n_items, p.phi_kind, p.eps,
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

int64_t tc_dw_part_floats(const Problem& p) {
  const BwdLayout L = bwd_layout(p);
  return static_cast<int64_t>(L.nsplit) * p.M * p.M;
}

int tc_run_dw(const Problem& p, const void* dSbuf, const void* Sbuf, float* part, float* dW, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const BwdLayout L = bwd_layout(p);
  CUtensorMap ta, tb;
  const cuuint64_t dims[3] = {128u, static_cast<cuuint64_t>(p.M), static_cast<cuuint64_t>(L.ngroups)};
  const cuuint64_t strides[2] = {256u, static_cast<cuuint64_t>(p.M * 256)};
  const cuuint32_t abox[3] = {64u, static_cast<cuuint32_t>(DwCfg::IT), 1u};
  const cuuint32_t bbox[3] = {64u, static_cast<cuuint32_t>(L.JN), 1u};
  if (!encode_tensor_map(&ta, 3, const_cast<void*>(dSbuf), dims, strides, abox, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tensor_map(&tb, 3, const_cast<void*>(Sbuf), dims, strides, bbox, CU_TENSOR_MAP_SWIZZLE_128B))
    return MHLA_ERR_CUDA;
  if (cudaFuncSetAttribute(tc_dw, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(DwCfg::SMEM)) !=
      cudaSuccess)
    return MHLA_ERR_CUDA;
  const int64_t ctas = static_cast<int64_t>(L.n_it) * L.n_jt * L.nsplit;
  KernelTimer timer("tc_dw", s);
  tc_dw<<<static_cast<unsigned>(ctas), kDwThreads, DwCfg::SMEM, s>>>(ta, tb, static_cast<int32_t>(p.M), L.n_jt, L.JN,
                                                                     L.ngroups, L.nsplit, part);
  if (cudaGetLastError() != cudaSuccess) return MHLA_ERR_CUDA;
  const int64_t MM = p.M * p.M;
  tc_dw_reduce<<<static_cast<unsigned>((MM + kDwrOut - 1) / kDwrOut), 256, 0, s>>>(part, dW, MM, L.nsplit);
  return cudaGetLastError() == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
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

MHLA_DEFINE_STALL_SETTER(set_stall_bwd)

}  // namespace mhla
