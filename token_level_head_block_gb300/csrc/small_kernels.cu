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
// One work unit = (b, h, 128 query tokens).  Persistent CTAs of four warps:
//   TMA      q tile (128 x d) and all keys and values (KR x d, KR = N rounded
//            up to 32, rows past N zero-filled) through 4-D maps (d, H, N, B);
//   phi      in place on the q and k tiles in shared memory;
//   MMA 1    scores phi(Q) phi(K)^T, 128 x KR, float32 in tensor memory;
//   weights  every thread owns one query row: P = score * W[b(t)][b(s)],
//            rounded to bf16 and written K-major (128-byte swizzle) as the next
//            MMA's A operand; the denominator sums the rounded P in float32;
//   MMA 2    P V, 128 x d, from the value tile as it landed (MN-major B);
//   output   scale by 1 / (den + eps), round to bf16, 16-byte stores.
// The next unit's q and k tiles load while the weights and the output of the
// current one are formed; its value tile once MMA 2 has read the current one.
//
// Every wait is bounded (2 s of %globaltimer, 2^28 polls); a wait that gives
// up sets bit 0 of this file's device error word, all threads of the CTA agree
// to stop, copies and MMAs in flight are drained (bit 1 if that drain gives up)
// and tensor memory is released.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "mhla_internal.h"
#include "ptx.cuh"
#include "tma_host.h"

namespace mhla {

__device__ unsigned int g_small_error = 0;

namespace {

using namespace ptx;

constexpr uint64_t kSmallWaitNs = 2000000000ull;   // 2 s
constexpr uint32_t kSmallWaitPolls = 1u << 28;
constexpr uint64_t kSmallDrainNs = 50000000ull;    // 50 ms for work already in flight
constexpr int kSmallThreads = 128;
constexpr int kQRows = 128;      // query tokens per unit: MMA M, one TMEM lane each
constexpr int kMaxKeys = 256;    // keys per image: MMA N of the score product
constexpr int kMaxBlocks = 96;   // W is held in shared memory as float32
constexpr int kTmemCols = 512;   // scores in [0, 256), P V in [256, 256 + d)

template <int D>
struct SmallCfg {
  static constexpr int ROWB = D * 2;                 // bytes per token row
  static constexpr int Q_BYTES = kQRows * ROWB;
  static constexpr int KV_BYTES = kMaxKeys * ROWB;
  static constexpr int P_CHUNK = kQRows * 128;       // 64 keys of P: 128 rows of 128 bytes
  static constexpr int P_BYTES = (kMaxKeys / 64) * P_CHUNK;
  static constexpr int W_BYTES = kMaxBlocks * kMaxBlocks * 4;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + Q_BYTES;      // k directly after q: phi runs over both
  static constexpr int V_OFF = K_OFF + KV_BYTES;
  static constexpr int P_OFF = V_OFF + KV_BYTES;
  static constexpr int W_OFF = P_OFF + P_BYTES;
  static constexpr int BLK_OFF = W_OFF + W_BYTES;    // block id of every token, one byte each
  static constexpr int CTRL_OFF = BLK_OFF + kMaxKeys;
  static constexpr size_t SMEM = CTRL_OFF + 64 + 1024;
  static constexpr uint32_t SBO = 8 * ROWB;          // 8-row groups of a token tile
  static constexpr uint32_t LAYOUT = D == 64 ? 2u : 4u;   // 128- or 64-byte swizzle
};

struct SmallGeom {
  int32_t N, H, M, KR, nqt;          // tokens, heads, blocks, key rows loaded, query tiles
  int32_t X, Y, bx, by, bt, nbx, nby;
  int64_t osb, osn, osh;             // output strides, elements
};

__device__ __noinline__ bool small_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1; it < kSmallWaitPolls; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0 && globaltimer() - t0 > kSmallWaitNs) break;
  }
  atomicOr(&g_small_error, 1u);
  return false;
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
  uint8_t* sp = smem + Cfg::P_OFF;
  float* sw = reinterpret_cast<float*>(smem + Cfg::W_OFF);
  uint8_t* sblk = smem + Cfg::BLK_OFF;
  uint64_t* full_qk = reinterpret_cast<uint64_t*>(smem + Cfg::CTRL_OFF);
  uint64_t* full_v = full_qk + 1;
  uint64_t* done1 = full_qk + 2;
  uint64_t* done2 = full_qk + 3;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(full_qk + 4);

  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t qk_bytes = static_cast<uint32_t>((kQRows + g.KR) * Cfg::ROWB);
  const uint32_t v_bytes = static_cast<uint32_t>(g.KR * Cfg::ROWB);

  if (tid == 0) {
    mbar_init(full_qk, 1);
    mbar_init(full_v, 1);
    mbar_init(done1, 1);
    mbar_init(done2, 1);
    fence_mbar_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  for (int e = tid; e < g.M * g.M; e += kSmallThreads) sw[e] = W[e];
  // Block id of token n: blocks row-major over (nbt, nby, nbx), tokens raster
  // over (T, Y, X).
  for (int n = tid; n < kMaxKeys; n += kSmallThreads) {
    int id = 0;
    if (n < g.N) {
      const int x = n % g.X, r = n / g.X, y = r % g.Y, t = r / g.Y;
      id = ((t / g.bt) * g.nby + y / g.by) * g.nbx + x / g.bx;
    }
    sblk[n] = static_cast<uint8_t>(id);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const uint64_t pol_q = policy_evict_first();
  const uint64_t pol_kv = policy_evict_last();   // every query tile of (b, h) reads them
  auto issue_qk = [&](int64_t u) {
    const int32_t qt = static_cast<int32_t>(u % g.nqt);
    const int64_t bh = u / g.nqt;
    const int32_t h = static_cast<int32_t>(bh % g.H), b = static_cast<int32_t>(bh / g.H);
    mbar_arrive_expect_tx(full_qk, qk_bytes);
    tma_load_4d(sq, &tm_q, full_qk, 0, h, qt * kQRows, b, pol_q);
    tma_load_4d(sk, &tm_k, full_qk, 0, h, 0, b, pol_kv);
  };
  auto issue_v = [&](int64_t u) {
    const int64_t bh = u / g.nqt;
    const int32_t h = static_cast<int32_t>(bh % g.H), b = static_cast<int32_t>(bh / g.H);
    mbar_arrive_expect_tx(full_v, v_bytes);
    tma_load_4d(sv, &tm_v, full_v, 0, h, 0, b, pol_kv);
  };

  // Issued (thread 0) and consumed (all threads) counts of each barrier's phases.
  uint32_t n_qk = 0, n_v = 0, n_m1 = 0, n_m2 = 0;
  uint32_t c_qk = 0, c_v = 0, c_m1 = 0, c_m2 = 0;
  if (tid == 0 && static_cast<int64_t>(blockIdx.x) < n_units) {
    issue_qk(blockIdx.x);
    issue_v(blockIdx.x);
    n_qk = n_v = 1;
  }
  const bool add_eps = phi_kind == MHLA_PHI_RELU_EPS;
  const __nv_bfloat162 eps2 = __float2bfloat162_rn(eps);
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  const int swr = tid & 7;   // 128-byte swizzle phase of this thread's P row

  for (int64_t u = blockIdx.x; u < n_units; u += gridDim.x) {
    const int32_t qt = static_cast<int32_t>(u % g.nqt);
    const int64_t bh = u / g.nqt;
    const int32_t h = static_cast<int32_t>(bh % g.H), b = static_cast<int32_t>(bh / g.H);
    const int64_t next = u + gridDim.x;

    // ---- q and k tiles landed: phi in place over both (contiguous)
    if (!__syncthreads_and(small_wait(full_qk, c_qk & 1u))) break;
    ++c_qk;
    {
      uint4* base = reinterpret_cast<uint4*>(sq);
      const int n16 = (kQRows + g.KR) * Cfg::ROWB / 16;
      for (int e = tid; e < n16; e += kSmallThreads) base[e] = phi8(base[e], add_eps, eps2);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- MMA 1: scores = phi(Q) phi(K)^T, 128 x KR, TMEM columns [0, KR)
    if (tid == 0) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16_f32(128, g.KR, /*a K-major*/ false, /*b K-major*/ false);
      const uint32_t qa = smem_u32(sq), ka = smem_u32(sk);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        mma_bf16(tmem, smem_desc(qa + ks * 32, 16, Cfg::SBO, Cfg::LAYOUT),
                 smem_desc(ka + ks * 32, 16, Cfg::SBO, Cfg::LAYOUT), idesc, ks > 0 ? 1u : 0u);
      mma_commit(done1);
      ++n_m1;
    }
    if (!__syncthreads_and(small_wait(done1, c_m1 & 1u))) break;
    ++c_m1;
    tc_fence_after();
    // q and k of this unit are consumed: the next unit's may land meanwhile.
    if (tid == 0 && next < n_units) {
      fence_proxy_async_smem();
      issue_qk(next);
      ++n_qk;
    }

    // ---- weights: P[t][s] = score * W[b(t)][b(s)], bf16, K-major SW128
    const int32_t nq = qt * kQRows + tid;
    const float* wrow = sw + (nq < g.N ? sblk[nq] : 0) * g.M;
    float den = 0.0f;
    for (int m = 0; m < g.KR / 32; ++m) {
      uint32_t r[32];
      tmem_ld_x32(lane_base + m * 32, r);
      const uint4 id0 = *reinterpret_cast<const uint4*>(sblk + m * 32);
      const uint4 id1 = *reinterpret_cast<const uint4*>(sblk + m * 32 + 16);
      tmem_ld_wait();
      const uint32_t ids[8] = {id0.x, id0.y, id0.z, id0.w, id1.x, id1.y, id1.z, id1.w};
      uint32_t packed[16];
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        const int s = m * 32 + e;
        const uint32_t j0 = (ids[e >> 2] >> (8 * (e & 3))) & 0xFFu;
        const uint32_t j1 = (ids[e >> 2] >> (8 * ((e + 1) & 3))) & 0xFFu;
        const float p0 = s < g.N ? __uint_as_float(r[e]) * wrow[j0] : 0.0f;
        const float p1 = s + 1 < g.N ? __uint_as_float(r[e + 1]) * wrow[j1] : 0.0f;
        packed[e >> 1] = pack2(p0, p1);
        const float2 pr = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&packed[e >> 1]));
        den += pr.x + pr.y;
      }
      uint8_t* prow = sp + (m >> 1) * Cfg::P_CHUNK + tid * 128;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int unit = (m & 1) * 4 + q;
        *reinterpret_cast<uint4*>(prow + ((unit ^ swr) * 16)) =
            make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();

    // ---- MMA 2: P V, 128 x d, TMEM columns [256, 256 + d)
    bool vok = true;
    if (tid == 0) vok = small_wait(full_v, c_v & 1u);
    if (!__syncthreads_and(vok)) break;
    ++c_v;
    if (tid == 0) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16_f32(128, D, /*a K-major*/ false, /*b MN-major*/ true);
      const uint32_t pa = smem_u32(sp), va = smem_u32(sv);
      for (int ks = 0; ks < g.KR / 16; ++ks)
        mma_bf16(tmem + 256, smem_desc(pa + (ks >> 2) * Cfg::P_CHUNK + (ks & 3) * 32, 16, 1024, 2),
                 smem_desc(va + ks * 2 * Cfg::SBO, Cfg::KV_BYTES, Cfg::SBO, Cfg::LAYOUT), idesc,
                 ks > 0 ? 1u : 0u);
      mma_commit(done2);
      ++n_m2;
    }
    if (!__syncthreads_and(small_wait(done2, c_m2 & 1u))) break;
    ++c_m2;
    tc_fence_after();
    if (tid == 0 && next < n_units) {
      issue_v(next);
      ++n_v;
    }

    // ---- output: o_t = (P V)_t / (den_t + eps)
    uint32_t o0[32], o1[32];
    tmem_ld_x32(lane_base + 256, o0);
    if (D == 64) tmem_ld_x32(lane_base + 288, o1);
    tmem_ld_wait();
    tc_fence_before();
    if (nq < g.N) {
      const float inv = 1.0f / (den + eps);
      uint4* dst = reinterpret_cast<uint4*>(out + b * g.osb + static_cast<int64_t>(nq) * g.osn + h * g.osh);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        dst[q] = make_uint4(pack2(__uint_as_float(o0[8 * q]) * inv, __uint_as_float(o0[8 * q + 1]) * inv),
                            pack2(__uint_as_float(o0[8 * q + 2]) * inv, __uint_as_float(o0[8 * q + 3]) * inv),
                            pack2(__uint_as_float(o0[8 * q + 4]) * inv, __uint_as_float(o0[8 * q + 5]) * inv),
                            pack2(__uint_as_float(o0[8 * q + 6]) * inv, __uint_as_float(o0[8 * q + 7]) * inv));
      if (D == 64) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          dst[4 + q] =
              make_uint4(pack2(__uint_as_float(o1[8 * q]) * inv, __uint_as_float(o1[8 * q + 1]) * inv),
                         pack2(__uint_as_float(o1[8 * q + 2]) * inv, __uint_as_float(o1[8 * q + 3]) * inv),
                         pack2(__uint_as_float(o1[8 * q + 4]) * inv, __uint_as_float(o1[8 * q + 5]) * inv),
                         pack2(__uint_as_float(o1[8 * q + 6]) * inv, __uint_as_float(o1[8 * q + 7]) * inv));
      }
    }
  }

  // Copies and MMAs issued but never waited for (a wait gave up) must finish
  // before shared and tensor memory go away.
  if (tid == 0) {
    if (n_qk > c_qk) small_drain(full_qk, (n_qk - 1) & 1u);
    if (n_v > c_v) small_drain(full_v, (n_v - 1) & 1u);
    if (n_m1 > c_m1) small_drain(done1, (n_m1 - 1) & 1u);
    if (n_m2 > c_m2) small_drain(done2, (n_m2 - 1) & 1u);
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

}  // namespace mhla
