// mhla_gemm: the two projections of the MHLA module ([P1] "MHLA：通过令牌级多头
// 机制恢复线性注意力机制的表达能力", 171host.com/767426.html, section 7, class
// MHLA: to_qkv = nn.Linear(dim, 3 inner_dim), to_out = nn.Linear(inner_dim,
// dim)) as a hand-written tcgen05 GEMM with the bias in its epilogue:
//
//   y[r][n] = sum_k x[r][k] w[n][k] + bias[n]     (bf16 x, w, bias, y; float32
//                                                   accumulation, one rounding)
//
// x is [rows][K] and w [n_out][K], both row-major (K contiguous), the layout of
// the activations and of nn.Linear's weight, so both MMA operands are K-major.
//
// Persistent CTAs, one per SM, walk 128 x 256 output tiles, the 256 columns
// fastest, so the CTAs working on the same rows of x run side by side and share
// them in L2 (w, at most a few MB, stays in L2 throughout); with more than one
// row tile, CTAs work in clusters of two that share the w chunks (below).  Roles: warp 0
// issues TMA loads of 64-wide K chunks of x and w into a 4-stage ring; warp 1
// issues one 128 x 256 x 16 MMA per 16 of K into one of two tensor-memory
// accumulators; warps 2-5 drain the other accumulator: each thread owns an
// output row, adds the bias, rounds to bf16 and writes 64-column groups into
// its warp's 128-byte-swizzled staging tile, which the warp's lane 0 stores by
// TMA (two staging tiles per warp alternate, so a store overlaps the next
// group's rounding).
//
// Measured on GB300 (the module's DiT-S/2 shapes, rows = 262144, K = 384): a
// tile takes about 3.3 us against 2 us of MMA work.  Within a tile the MMA
// waits for loads: four 48 KB stages hold about 1.3 us of MMA work, less than
// the 1.5 us a load takes to land under full load; the epilogue needs about
// 2.4 us per tile.  Neither the pair's multicast (fewer bytes fetched per SM,
// the same stage footprint) nor a w slice kept resident (room for fewer x
// stages) nor eight epilogue warps shortened it.  Rows past
// `rows`, columns past n_out and K past its end are zero-filled on load and
// clipped on store by the tensor maps.
//
// Every mbarrier wait is bounded (time and poll count); a wait that gives up
// raises a per-CTA abort flag so the other roles stop waiting too, sets bit 0
// of this file's device error word, and the CTA drains its copies, releases
// tensor memory and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "mhla_internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"
#include "tma_host.h"

namespace mhla {

__device__ unsigned int g_gemm_error = 0;

namespace {

using namespace ptx;
using namespace tc;

// Two variants of one pipeline:
//   single  one CTA per tile; every stage holds a 64-wide K chunk of x (its 128
//           rows) and of w (its BN = 256 or 192 columns).
//   pair    a cluster of two CTAs computes two vertically adjacent tiles (rows
//           m0 and m0 + 128, the same columns): each CTA loads its own x chunk
//           and one half of the w chunk, which TMA multicasts into both CTAs'
//           stages, so per tile an SM fetches 128 + BN / 2 instead of 128 + BN
//           rows of operands.  The pipeline is bound by the bytes an
//           SM keeps in flight (about 190 KB of stages against an L2 latency of
//           a few microseconds under load), so fewer bytes per tile is more
//           tiles per second.  A stage is refilled only when both CTAs' MMAs
//           are done with it: every MMA commit arrives on the stage's empty
//           barrier in both CTAs.
template <bool PAIR, int BN_>
struct GemmCfg {
  static constexpr int BM = 128;                 // rows per tile (MMA M, TMEM lanes)
  static constexpr int BN = BN_;                 // columns per tile (MMA N): 256 or 192
  static constexpr int BK = 64;                  // K per stage: one 128-byte swizzled row
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;    // one K chunk of w (both halves)
  static constexpr int B_LOAD = PAIR ? BN / 2 : BN;   // rows of w one CTA loads per chunk
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int NS = 4;
  static constexpr int OUT_GROUP = 64;           // columns per staging tile (128-byte rows)
  static constexpr int WARP_OUT = 32 * OUT_GROUP * 2;   // one epilogue warp's staging tile: 32 rows
  static constexpr int OUT_BYTES = 8 * WARP_OUT;        // four epilogue warps, two tiles each
  static constexpr int TMEM_COLS = 512;          // two accumulators of BN <= 256 columns
  static constexpr int CTRL = 1024;
  static constexpr size_t SMEM = static_cast<size_t>(NS) * STAGE + OUT_BYTES + CTRL + 1024;
};
constexpr int kGemmThreads = 192;   // producer, MMA, four epilogue warps

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag) {
  return wait_bounded_on(bar, parity, abort_flag, &g_gemm_error);
}
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag) {
  return warp_wait_on(bar, parity, abort_flag, &g_gemm_error);
}
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  drain_wait_on(bar, parity, &g_gemm_error);
}

// Tile coordinates of unit u.  single: tile (u / n_tiles_n, u % n_tiles_n).
// pair: the pair of row tiles 2 (u / n_tiles_n) + rank, columns u % n_tiles_n.
template <bool PAIR, int BN>
__device__ __forceinline__ void tile_coords(int64_t u, int32_t n_tiles_n, uint32_t rank, int32_t& m0, int32_t& n0) {
  using Cfg = GemmCfg<PAIR, BN>;
  const int64_t mt = PAIR ? 2 * (u / n_tiles_n) + rank : u / n_tiles_n;
  m0 = static_cast<int32_t>(mt) * Cfg::BM;
  n0 = static_cast<int32_t>(u % n_tiles_n) * Cfg::BN;
}

template <bool PAIR, int BN>
__global__ void __launch_bounds__(kGemmThreads, 1)
mhla_gemm(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
          const __grid_constant__ CUtensorMap tm_y, const __nv_bfloat16* __restrict__ bias, int32_t rows,
          int32_t n_out, int32_t k_chunks, int32_t n_tiles_n, int64_t n_units) {
  using Cfg = GemmCfg<PAIR, BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  uint8_t* stages = smem;
  uint8_t* staging = stages + Cfg::NS * Cfg::STAGE;
  uint8_t* ctrl = staging + Cfg::OUT_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + Cfg::NS;
  uint64_t* tfull = empty + Cfg::NS;
  uint64_t* tempty = tfull + 2;
  uint64_t* fin = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 512);
  volatile uint32_t* abortf = tmem_slot + 1;

  // single: units blockIdx.x, + gridDim.x, ...; pair: units of the cluster
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int64_t first = PAIR ? blockIdx.x / 2 : blockIdx.x;
  const int64_t stride = PAIR ? gridDim.x / 2 : gridDim.x;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::NS; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, PAIR ? 2 : 1);   // pair: both CTAs' MMAs release a stage
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
    prefetch_tmap(&tm_x);
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_y);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  if (PAIR) cluster_sync();   // both CTAs' barriers exist before either multicasts into the other
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_x = policy_evict_first();   // x is read by the few CTAs of one row block, close in time
      const uint64_t pol_w = policy_evict_last();    // w is read by every tile
      int s = 0;
      uint32_t ph = 0;
      uint64_t fills = 0;
      bool ok = true;
      for (int64_t u = first; ok && u < n_units; u += stride) {
        int32_t m0, n0;
        tile_coords<PAIR, BN>(u, n_tiles_n, rank, m0, n0);
        for (int kc = 0; kc < k_chunks; ++kc) {
          if (!wait_bounded(empty + s, ph ^ 1u, abortf)) { ok = false; break; }
          mbar_arrive_expect_tx(full + s, Cfg::STAGE);
          uint8_t* st = stages + s * Cfg::STAGE;
          tma_load_2d(st, &tm_x, full + s, kc * Cfg::BK, m0, pol_x);
          if (PAIR) {
            const int32_t half = static_cast<int32_t>(rank) * Cfg::B_LOAD;
            tma_load_2d_multicast(st + Cfg::A_BYTES + half * 128, &tm_w, full + s, kc * Cfg::BK, n0 + half, 0x3,
                                  pol_w);
          } else {
            tma_load_2d(st + Cfg::A_BYTES, &tm_w, full + s, kc * Cfg::BK, n0, pol_w);
          }
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
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(Cfg::BM, Cfg::BN, /*a K-major*/ false, /*b K-major*/ false);
      int s = 0;
      uint32_t ph = 0, local = 0;
      bool ok = true;
      for (int64_t u = first; ok && u < n_units; u += stride, ++local) {
        const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
        if (!wait_bounded(tempty + acc, aph ^ 1u, abortf)) break;
        tc_fence_after();
        const uint32_t dt = tmem + acc * Cfg::BN;
        for (int kc = 0; kc < k_chunks; ++kc) {
          if (!wait_bounded(full + s, ph, abortf)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_base = smem_u32(stages + s * Cfg::STAGE);
          const uint32_t b_base = a_base + Cfg::A_BYTES;
#pragma unroll
          for (int ks = 0; ks < Cfg::BK / 16; ++ks) {
            const uint64_t a = smem_desc(a_base + ks * 32, 16, 1024, 2);
            const uint64_t b = smem_desc(b_base + ks * 32, 16, 1024, 2);
            mma_bf16(dt, a, b, idesc, (kc | ks) != 0 ? 1u : 0u);
          }
          if (PAIR) mma_commit_multicast(empty + s, 0x3);
          else mma_commit(empty + s);
          if (++s == Cfg::NS) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        mma_commit(tfull + acc);
      }
      mma_commit(fin);
      drain_wait(fin, 0);
    }
  } else {
    // ------------------------------------------------ epilogue (warps 2-5)
    // Each warp owns 32 output rows (its TMEM lane quarter) and its own pair of
    // 4 KB staging tiles, so no barrier spans the epilogue warps.
    const int q4 = warp & 3;                 // TMEM lane quarter this warp may read
    uint8_t* my_staging = staging + q4 * 2 * Cfg::WARP_OUT;
    constexpr int G = Cfg::BN / Cfg::OUT_GROUP;   // 64-column groups per tile
    uint32_t local = 0;
    int group = 0;                           // staging tiles this warp used so far
    for (int64_t u = first; u < n_units; u += stride, ++local) {
      const uint32_t acc = local & 1u, aph = (local >> 1) & 1u;
      if (!warp_wait(tfull + acc, aph, abortf)) break;
      tc_fence_after();
      int32_t m0, n0;
      tile_coords<PAIR, BN>(u, n_tiles_n, rank, m0, n0);
      const uint32_t tb = tmem + acc * Cfg::BN + (static_cast<uint32_t>(32 * q4) << 16);
      const int n_groups = min(Cfg::BN, n_out - n0 + Cfg::OUT_GROUP - 1) / Cfg::OUT_GROUP;
#pragma unroll 1
      for (int gi = 0; gi < G; ++gi) {
        uint32_t v0[32], v1[32];
        tmem_ld_x32(tb + gi * Cfg::OUT_GROUP, v0);
        tmem_ld_x32(tb + gi * Cfg::OUT_GROUP + 32, v1);
        tmem_ld_wait();
        if (gi + 1 == G) {                        // the accumulator is read out: the MMA may reuse it
          tc_fence_before();
          mbar_arrive(tempty + acc);
        }
        if (gi >= n_groups) continue;             // columns past n_out (the same for every warp)
        // this warp's staging tile of two groups ago has been read by its store
        if (lane == 0) bulk_wait_group_read<1>();
        __syncwarp();
        uint8_t* sb = my_staging + (group & 1) * Cfg::WARP_OUT;
        const int c0 = n0 + gi * Cfg::OUT_GROUP;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t* src = q < 4 ? v0 + 8 * q : v1 + 8 * (q - 4);
          float bb[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          if (bias && c0 + 8 * q < n_out) {   // n_out % 8 == 0: a unit is wholly in or out
            const uint4 raw = *reinterpret_cast<const uint4*>(bias + c0 + 8 * q);
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&w[e]);
              bb[2 * e] = __low2float(b2);
              bb[2 * e + 1] = __high2float(b2);
            }
          }
          const uint4 packed = make_uint4(pack_bf16(__uint_as_float(src[0]) + bb[0], __uint_as_float(src[1]) + bb[1]),
                                          pack_bf16(__uint_as_float(src[2]) + bb[2], __uint_as_float(src[3]) + bb[3]),
                                          pack_bf16(__uint_as_float(src[4]) + bb[4], __uint_as_float(src[5]) + bb[5]),
                                          pack_bf16(__uint_as_float(src[6]) + bb[6], __uint_as_float(src[7]) + bb[7]));
          *reinterpret_cast<uint4*>(sb + lane * 128 + ((q ^ (lane & 7)) * 16)) = packed;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && m0 + 32 * q4 < rows) {   // a box wholly past the last row stores nothing
          tma_store_2d(&tm_y, sb, c0, m0 + 32 * q4);
          bulk_commit_group();
        }
        ++group;
      }
    }
    if (lane == 0) bulk_wait_group0();
  }
  tc_fence_before();
  // pair: neither CTA leaves while the other's MMA commits or multicasts may
  // still target its shared memory
  if (PAIR) cluster_sync();
  else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::TMEM_COLS);
  }
}

bool encode_2d(CUtensorMap* m, const void* base, int64_t inner, int64_t outer, int64_t row_elems, uint32_t box_in,
               uint32_t box_out) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_elems * 2)};
  const cuuint32_t box[2] = {box_in, box_out};
  return encode_tensor_map(m, 2, const_cast<void*>(base), dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <bool PAIR, int BN>
int run_gemm(const char* name, const void* x, const void* w, const void* bias, void* y, int64_t rows, int64_t k,
             int64_t n_out, int sms, cudaStream_t stream) {
  using Cfg = GemmCfg<PAIR, BN>;
  CUtensorMap tx, tw, ty;
  if (!encode_2d(&tx, x, k, rows, k, Cfg::BK, Cfg::BM) || !encode_2d(&tw, w, k, n_out, k, Cfg::BK, Cfg::B_LOAD) ||
      !encode_2d(&ty, y, n_out, rows, n_out, Cfg::OUT_GROUP, 32))
    return MHLA_ERR_CUDA;
  const int32_t k_chunks = static_cast<int32_t>((k + Cfg::BK - 1) / Cfg::BK);
  const int32_t n_tiles_n = static_cast<int32_t>((n_out + Cfg::BN - 1) / Cfg::BN);
  const int64_t m_tiles = (rows + Cfg::BM - 1) / Cfg::BM;
  const int64_t n_units = (PAIR ? (m_tiles + 1) / 2 : m_tiles) * n_tiles_n;
  auto kernel = mhla_gemm<PAIR, BN>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(Cfg::SMEM)) !=
      cudaSuccess)
    return MHLA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = Cfg::SMEM;
  cfg.stream = stream;
  int64_t grid = std::min<int64_t>(n_units, sms);
  if (PAIR) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    cfg.gridDim = dim3(2);
    if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess || clusters < 1)
      return MHLA_ERR_UNSUPPORTED;
    grid = 2 * std::min<int64_t>(n_units, clusters);
  }
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  KernelTimer timer(name, stream);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, tx, tw, ty, static_cast<const __nv_bfloat16*>(bias),
                                           static_cast<int32_t>(rows), static_cast<int32_t>(n_out), k_chunks,
                                           n_tiles_n, n_units);
  if (e != cudaSuccess) return MHLA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
}

template <int BN>
int gemm_dispatch(const char* name, const void* x, const void* w, const void* bias, void* y, int64_t rows, int64_t k,
                  int64_t n_out, int sms, cudaStream_t s) {
  // one row tile: nothing to pair with
  if (rows <= 128) return run_gemm<false, BN>(name, x, w, bias, y, rows, k, n_out, sms, s);
  const int rc = run_gemm<true, BN>(name, x, w, bias, y, rows, k, n_out, sms, s);
  return rc == MHLA_ERR_UNSUPPORTED ? run_gemm<false, BN>(name, x, w, bias, y, rows, k, n_out, sms, s) : rc;
}

}  // namespace

bool gemm_supported(int64_t rows, int64_t k, int64_t n_out) {
  return rows >= 1 && k >= 8 && n_out >= 8 && k % 8 == 0 && n_out % 8 == 0 && rows < (int64_t{1} << 31) &&
         k < (int64_t{1} << 20) && n_out < (int64_t{1} << 20);
}

int launch_gemm(const char* name, const void* x, const void* w, const void* bias, void* y, int64_t rows, int64_t k,
                int64_t n_out, void* stream) {
  if (!gemm_supported(rows, k, n_out)) return MHLA_ERR_UNSUPPORTED;
  const int sms = device_sm_count();
  if (sms <= 0) return MHLA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // column tiles of 192 where they need no more tiles than tiles of 256 (fewer
  // MMA columns wasted at the edge, e.g. n_out = 384: 2 x 192 rather than
  // 256 + a half-empty 256); otherwise 256 (n_out = 1152: 5 tiles rather than 6
  // measured faster, each extra tile re-reading x)
  if ((n_out + 191) / 192 <= (n_out + 255) / 256) return gemm_dispatch<192>(name, x, w, bias, y, rows, k, n_out, sms, s);
  return gemm_dispatch<256>(name, x, w, bias, y, rows, k, n_out, sms, s);
}

int read_and_clear_gemm_error(void* stream, uint32_t* flags) { return read_and_clear_word(g_gemm_error, stream, flags); }

MHLA_DEFINE_STALL_SETTER(set_stall_gemm)

}  // namespace mhla
