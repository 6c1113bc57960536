// tc_mix: the mixing step of the tensor-core path, S~ = W . S as one GEMM over
// the source blocks for every (b, h) at once ([P2] "MHLA: Restoring
// Expressivity of Linear Attention via Token-Level Multi-Head", section 4
// "Multi-Head Mixing"; [P1] 171host.com/767426.html, section 7: piece_attn, a
// 1x1 convolution over the block axis).  The backward pass runs it with W^T.

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
#include "tc_fwd_bodies.cuh"
#include "tma_host.h"

namespace mhla {

__device__ unsigned int g_mix_error = 0;

namespace {

using namespace ptx;
using namespace tc;

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag) {
  return wait_bounded_on(bar, parity, abort_flag, &g_mix_error);
}
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag) {
  return warp_wait_on(bar, parity, abort_flag, &g_mix_error);
}
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) { drain_wait_on(bar, parity, &g_mix_error); }

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
      grid_dep_wait();   // W in bf16 and Sbuf come from the summary launch
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
// tc_mix_resident: the M <= 256 mixing pipeline (tc_fwd_bodies.cuh: W resident
// in shared memory, transposed GEMM with the Sbuf columns on the TMEM lanes) in
// a launch of its own, W loaded by TMA from its bf16 copy.
// ============================================================================
constexpr int kMixResStages = 6;
using MixRes = MixResCfg<kMixResStages>;
constexpr size_t kMixResSmem = MixRes::DATA + 1024 + 1024;

template <int D>
__global__ void __launch_bounds__(kMixThreadsTC, 1)
tc_mix_resident(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_s, int32_t M,
                int32_t NP, int64_t ncols, int32_t n_tiles, __nv_bfloat16* __restrict__ St, float* __restrict__ zt,
                const __nv_bfloat16* discard_s) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  uint8_t* ctrl = smem + MixRes::DATA;
  const MixBars bars = mix_bars<kMixResStages>(ctrl);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 512);
  volatile uint32_t* abortf = tmem_slot + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mix_init<kMixResStages>(bars);
    *abortf = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_s);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, MixRes::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const MixDeps none{nullptr, 0u, nullptr, 1};
  mix_roles<kMixResStages, D>(&tm_w, &tm_s, M, NP, ncols, blockIdx.x, gridDim.x, n_tiles, St, zt, discard_s, smem,
                              bars, tmem, abortf, &g_mix_error, none);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, MixRes::TMEM_COLS);
  }
}

// D[i, col] = sum_j Wm[i][j] Sbuf[j][col] for the ncols = BH (d + 1) d columns:
// S~ (row-major [BH][M][d][d]) and z~ (float32 [BH][M][d]).
template <int D>
int run_mix(const Problem& p, const __nv_bfloat16* Wm, int64_t Mp, const __nv_bfloat16* Sbuf, __nv_bfloat16* St,
            float* zt, bool discard_input, cudaStream_t stream) {
  const int sms = device_sm_count();
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
    const cuuint32_t wbox[2] = {static_cast<cuuint32_t>(MixRes::KC), static_cast<cuuint32_t>(NP)};
    const cuuint32_t sbox[3] = {64u, static_cast<cuuint32_t>(MixRes::KC), 1u};
    if (!encode_tensor_map(&tw, 2, wptr, wdims, wstrides, wbox, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map(&ts, 3, sptr, sdims, sstrides, sbox, CU_TENSOR_MAP_SWIZZLE_128B))
      return MHLA_ERR_CUDA;
    const int32_t n_tiles = static_cast<int32_t>((ncols + MixRes::COLS - 1) / MixRes::COLS);
    if (cudaFuncSetAttribute(tc_mix_resident<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kMixResSmem)) != cudaSuccess)
      return MHLA_ERR_CUDA;
    const int grid = static_cast<int>(std::min<int64_t>(n_tiles, sms));
    KernelTimer timer("tc_mix", stream);
    const cudaError_t e = launch_dependent(tc_mix_resident<D>, dim3(grid), dim3(kMixThreadsTC), kMixResSmem,
                                           stream, tw, ts, static_cast<int32_t>(p.M), NP, ncols, n_tiles, St, zt,
                                           discard_input ? Sbuf : static_cast<const __nv_bfloat16*>(nullptr));
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
  }
  CUtensorMap tw, ts;
  const cuuint32_t wbox[2] = {static_cast<cuuint32_t>(MixCfg::KC), static_cast<cuuint32_t>(MixCfg::ROWS)};
  const cuuint32_t sbox[3] = {64u, static_cast<cuuint32_t>(MixCfg::KC), 1u};
  if (!encode_tensor_map(&tw, 2, wptr, wdims, wstrides, wbox, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tensor_map(&ts, 3, sptr, sdims, sstrides, sbox, CU_TENSOR_MAP_SWIZZLE_128B))
    return MHLA_ERR_CUDA;
  const int32_t n_col_tiles = static_cast<int32_t>((ncols + MixCfg::COLS - 1) / MixCfg::COLS);
  const int32_t n_i_tiles = static_cast<int32_t>((p.M + MixCfg::ROWS - 1) / MixCfg::ROWS);
  if (cudaFuncSetAttribute(tc_mix<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(MixCfg::SMEM)) !=
      cudaSuccess)
    return MHLA_ERR_CUDA;
  const int64_t n_tiles = static_cast<int64_t>(n_col_tiles) * n_i_tiles;
  const int grid = static_cast<int>(std::min<int64_t>(n_tiles, sms));
  KernelTimer timer("tc_mix", stream);
  const cudaError_t e = launch_dependent(tc_mix<D>, dim3(grid), dim3(kMixThreadsTC), MixCfg::SMEM, stream, tw, ts,
                                         static_cast<int32_t>(p.M), ncols, n_col_tiles, n_i_tiles, St, zt);
  if (e != cudaSuccess) return MHLA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
}

}  // namespace

int tc_run_mix(const Problem& p, const void* Wm, int64_t Mp, const void* Sbuf, void* St, float* zt, void* stream,
               bool discard_input) {
  auto* wm = static_cast<const __nv_bfloat16*>(Wm);
  auto* sb = static_cast<const __nv_bfloat16*>(Sbuf);
  auto* st = static_cast<__nv_bfloat16*>(St);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return p.d == 64 ? run_mix<64>(p, wm, Mp, sb, st, zt, discard_input, s)
                   : run_mix<32>(p, wm, Mp, sb, st, zt, discard_input, s);
}

int read_and_clear_mix_error(void* stream, uint32_t* flags) { return read_and_clear_word(g_mix_error, stream, flags); }

MHLA_DEFINE_STALL_SETTER(set_stall_mix)

}  // namespace mhla
