// tc_fused: the whole tensor-core MHLA forward in one persistent launch, one CTA
// per SM, for problems whose mixing matrix fits in shared memory (M <= 256):
//
//   phase 1  CTAs [0, n_stream) form the block summaries S_j, z_j (HBM-bound:
//            they stream K and V once), while the other CTAs run the mixing
//            GEMM S~ = W . S batch by batch, each batch as soon as its
//            summaries are stored (a per-batch counter);
//   phase 2  every CTA turns to the readout, taking (b, i, h) items in order
//            from a global queue; an item's S~ tile is loaded once the mixing
//            of its batch is stored (a second per-batch counter).
//
// The three steps are those of the separate launches ([P2] "MHLA: Restoring
// Expressivity of Linear Attention via Token-Level Multi-Head", section 4
// "Architecture", "Multi-Head Mixing", "Token-Level Adaptivity"; [P1]
// 171host.com/767426.html, section 7, MHLA.forward) and run the same pipelines
// (tc_fwd_bodies.cuh).  What the fusion buys: the mixing GEMM, which moves no
// input or output bytes, overlaps the summaries' streaming instead of running
// between two HBM-bound launches, and the readout starts on each SM as soon as
// that SM is free, with no launch boundaries and their tails in between.
//
// Measured on GB300 (DiT-S/2 4096 px): 185 us against 160 us for the three
// launches, so the library's AUTO path does not take it.  The summaries are
// HBM-bound only when every SM streams (each CTA keeps about 33 GB/s in
// flight); with 29 SMs mixing they took 104 us instead of 79, more than the
// 22 us of mixing the overlap hides.  It stays as an explicit path
// (MHLA_PATH_TC_FUSED) that gives the same bits as the three launches.
//
// The mixing CTAs build the bf16 copy of W directly in shared memory from the
// float32 W.  The counters live in the workspace and are zeroed on the stream
// before the launch.  Every CTA of the grid must be resident at once (one per
// SM, grid = SM count): a wait on another CTA's counter is bounded like every
// other wait, so a CTA that cannot become resident costs a timeout
// (MHLA_ERR_TIMEOUT from mhla_device_status), never a hang.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "mhla_internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"
#include "tc_fwd_bodies.cuh"
#include "tma_host.h"

namespace mhla {

__device__ unsigned int g_fused_error = 0;

namespace {

using namespace ptx;
using namespace tc;

constexpr int kFusedThreads = 512;            // the readout's 16 warps; phase 1 uses the first 10
constexpr int kFusedMixStages = 5;
using FMix = MixResCfg<kFusedMixStages>;
constexpr int kCtrl1 = 1024;                  // phase-1 barriers
constexpr int kCtrl2 = 2048;                  // phase-2 barriers and the item ring

template <int D, int DO>
constexpr size_t fused_data() {
  return std::max(std::max(SumCfg<D>::DATA, FMix::DATA), OutCfg<DO>::DATA);
}

template <int D, int DO>
constexpr size_t fused_smem() {
  return fused_data<D, DO>() + kCtrl1 + kCtrl2 + 256 + 1024;
}

struct FusedArgs {
  TcGeom gs;             // summaries: 64-token chunks of the [B, N, H, d] view
  TcGeom go;             // readout: 128-token chunks (heads paired when PAIR)
  int32_t G;             // head groups of the summary items
  int32_t n_stream;      // CTAs [0, n_stream) summarise, the others mix
  int64_t n_sum;         // summary items
  int32_t M, NP;         // blocks; MMA N of the mixing GEMM (M rounded up to 16)
  int64_t ncols;         // Sbuf columns: B H (d + 1) d
  int64_t n_tiles;       // mixing tiles of 128 columns
  int64_t per_b_cols;    // Sbuf columns of one batch
  int64_t n_out;         // readout items
  int phi_kind;
  float eps;
  const float* W;        // float32 M x M
  __nv_bfloat16* Sbuf;
  __nv_bfloat16* St;
  float* zt;
  uint32_t* ctr;         // [B] summaries stored, [B] mixing stored, [1] readout queue
  int32_t B;
};

template <int D, int DO, bool PAIR>
__global__ void __launch_bounds__(kFusedThreads, 1)
tc_fused(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
         const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_q,
         const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_st, const FusedArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  uint8_t* ctrl1 = smem + fused_data<D, DO>();
  uint8_t* ctrl2 = ctrl1 + kCtrl1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl2 + kCtrl2);
  volatile uint32_t* abortf = tmem_slot + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool streaming = static_cast<int32_t>(blockIdx.x) < a.n_stream;
  const SumBars sb = sum_bars<D>(ctrl1);
  const MixBars mb = mix_bars<kFusedMixStages>(ctrl1);
  const OutBars ob = out_bars<DO>(ctrl2);
  uint32_t* sum_done = a.ctr;
  uint32_t* mix_done = a.ctr + a.B;
  uint32_t* queue = a.ctr + 2 * a.B;

  if (threadIdx.x == 0) {
    if (streaming) sum_init<D>(sb);
    else mix_init<kFusedMixStages>(mb);
    out_init<DO>(ob);
    *abortf = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_s);
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_o);
    prefetch_tmap(&tm_st);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (streaming) sum_fill_ones<D>(smem, threadIdx.x, kFusedThreads);
  else mix_fill_w<kFusedMixStages>(smem, a.W, a.M, a.NP, threadIdx.x, kFusedThreads);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // ------------------------------------------------ phase 1
  if (streaming) {
    summary_roles<D>(&tm_k, &tm_v, a.gs, a.G, blockIdx.x, a.n_stream, a.n_sum, a.phi_kind, a.eps, a.Sbuf, smem, sb,
                     tmem, abortf, &g_fused_error, sum_done);
  } else {
    const MixDeps dep{sum_done, static_cast<uint32_t>(4 * a.M * a.G), mix_done, a.per_b_cols};
    mix_roles<kFusedMixStages, D>(nullptr, &tm_s, a.M, a.NP, a.ncols, blockIdx.x - a.n_stream,
                                  gridDim.x - a.n_stream, a.n_tiles, a.St, a.zt, a.Sbuf, smem, mb, tmem, abortf,
                                  &g_fused_error, dep);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ------------------------------------------------ phase 2
  if (!*abortf) {
    if (PAIR) {
      out_zero_offdiag<DO, PAIR>(smem + OutCfg<DO>::NQ * OutCfg<DO>::QT, threadIdx.x, kFusedThreads);
      fence_proxy_async_smem();
      __syncthreads();
    }
    const OutSched sc{0, 1, a.n_out, queue, mix_done, a.per_b_cols};
    output_roles<DO, PAIR>(&tm_q, &tm_o, &tm_st, a.go, sc, a.phi_kind, a.eps, a.zt, a.St, smem, ob, tmem, abortf,
                           &g_fused_error);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// How many of the CTAs mix: the split that lets the mixing of the last batch
// finish about when the summaries do.  Rates measured on GB300: a streaming CTA
// keeps about 33 GB/s of K and V in flight (HBM caps the sum near 6 TB/s), and
// a mixing tile takes about 0.5 us plus 0.5 us per 64 source blocks on one SM.
int mixing_ctas(const Problem& p, int sms, int64_t n_tiles) {
  const double kv_bytes = 2.0 * p.B * p.N * p.H * p.d * 2.0;
  const double nk = static_cast<double>((p.M + 63) / 64);
  const double mix_work = static_cast<double>(n_tiles) * (0.5 + 0.5 * nk);   // SM-microseconds
  int best = 1;
  double best_t = 1e300;
  for (int x = 1; x <= sms / 2; ++x) {
    const double t_sum = std::max(kv_bytes / 6.0e6, kv_bytes / ((sms - x) * 3.3e4));
    const double t = std::max(t_sum, mix_work / x + t_sum / static_cast<double>(p.B));
    if (t < best_t) {
      best_t = t;
      best = x;
    }
  }
  return best;
}

template <int D, int DO, bool PAIR>
int run_fused(const Problem& p, const float* W, __nv_bfloat16* Sbuf, __nv_bfloat16* St, float* zt, uint32_t* ctr,
              cudaStream_t stream) {
  constexpr size_t SMEM = fused_smem<D, DO>();
  const int sms = device_sm_count();
  if (sms < 2) return MHLA_ERR_CUDA;
  ChunkPlan c64, c128;
  Problem v = p;   // the readout's view: PAIR sees heads of 64 channels, two real heads each
  if (PAIR) {
    v.d = 64;
    v.H = p.H / 2;
    v.q.sh = 2 * p.q.sh;
    v.o.sh = 2 * p.o.sh;
  }
  if (!chunk_plan(p, 64, &c64) || !chunk_plan(v, 128, &c128)) return MHLA_ERR_UNSUPPORTED;
  CUtensorMap tk, tv, ts, tq, to, tst;
  if (!operand_map(p, p.k, c64.box_y, c64.box_t, &tk) || !operand_map(p, p.v, c64.box_y, c64.box_t, &tv) ||
      !operand_map(v, v.q, c128.box_y, c128.box_t, &tq) || !operand_map(v, v.o, c128.box_y, c128.box_t, &to))
    return MHLA_ERR_CUDA;
  const int64_t ncols = p.BH() * (p.d + 1) * p.d;
  const int64_t ngroups = (ncols + 127) / 128;
  {
    // Sbuf as (128 columns, M source blocks, G groups), 64 x 64 boxes, 128-byte swizzle
    const cuuint64_t dims[3] = {128u, static_cast<cuuint64_t>(p.M), static_cast<cuuint64_t>(ngroups)};
    const cuuint64_t strides[2] = {256u, static_cast<cuuint64_t>(p.M * 256)};
    const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(FMix::KC), 1u};
    if (!encode_tensor_map(&ts, 3, Sbuf, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return MHLA_ERR_CUDA;
  }
  {
    // S~ tiles (row-major [BH*M][d][d]) seen as (c % 8, r, c / 8, tile): the
    // unswizzled MN-major operand layout of the readout's B operand
    const cuuint64_t dims[4] = {8u, static_cast<cuuint64_t>(p.d), static_cast<cuuint64_t>(p.d / 8),
                                static_cast<cuuint64_t>(p.BH() * p.M)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(p.d * 2), 16u, static_cast<cuuint64_t>(p.d * p.d * 2)};
    const cuuint32_t box[4] = {8u, static_cast<cuuint32_t>(p.d), PAIR ? 1u : static_cast<cuuint32_t>(p.d / 8), 1u};
    if (!encode_tensor_map(&tst, 4, St, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE)) return MHLA_ERR_CUDA;
  }
  FusedArgs a;
  a.gs = make_geom(p, c64);
  a.go = make_geom(v, c128);
  a.G = static_cast<int32_t>((p.H + SumCfg<D>::HP - 1) / SumCfg<D>::HP);
  a.n_sum = p.B * a.G * p.M;
  a.M = static_cast<int32_t>(p.M);
  a.NP = static_cast<int32_t>((p.M + 15) / 16 * 16);
  a.ncols = ncols;
  a.n_tiles = ngroups;
  a.per_b_cols = p.H * (p.d + 1) * p.d;
  a.n_out = v.BH() * v.M;
  a.phi_kind = p.phi_kind;
  a.eps = p.eps;
  a.W = W;
  a.Sbuf = Sbuf;
  a.St = St;
  a.zt = zt;
  a.ctr = ctr;
  a.B = static_cast<int32_t>(p.B);
  a.n_stream = sms - mixing_ctas(p, sms, a.n_tiles);
  if (cudaFuncSetAttribute(tc_fused<D, DO, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(SMEM)) != cudaSuccess)
    return MHLA_ERR_CUDA;
  if (occupancy(tc_fused<D, DO, PAIR>, kFusedThreads, SMEM) < 1) return MHLA_ERR_UNSUPPORTED;
  if (cudaMemsetAsync(ctr, 0, static_cast<size_t>(2 * p.B + 1) * sizeof(uint32_t), stream) != cudaSuccess)
    return MHLA_ERR_CUDA;
  KernelTimer timer("tc_fused", stream);
  tc_fused<D, DO, PAIR><<<sms, kFusedThreads, SMEM, stream>>>(tk, tv, ts, tq, to, tst, a);
  return cudaGetLastError() == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
}

}  // namespace

bool output_pairs_heads(const Problem& p);

bool tc_fused_eligible(const Problem& p) {
  if (!tc_rows_eligible(p) || p.M > 256) return false;
  const int64_t lim32 = int64_t{1} << 30;
  return p.B < lim32 && p.BH() * p.M < lim32;
}

size_t tc_fused_counter_bytes(const Problem& p) { return static_cast<size_t>(2 * p.B + 1) * sizeof(uint32_t); }

int launch_tc_fused(const Problem& p, const float* W, void* Sbuf, void* St, float* zt, void* ctr, void* stream) {
  auto* sb = static_cast<__nv_bfloat16*>(Sbuf);
  auto* st = static_cast<__nv_bfloat16*>(St);
  auto* c = static_cast<uint32_t*>(ctr);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.d == 64) return run_fused<64, 64, false>(p, W, sb, st, zt, c, s);
  return output_pairs_heads(p) ? run_fused<32, 64, true>(p, W, sb, st, zt, c, s)
                               : run_fused<32, 32, false>(p, W, sb, st, zt, c, s);
}

int read_and_clear_fused_error(void* stream, uint32_t* flags) {
  return read_and_clear_word(g_fused_error, stream, flags);
}

MHLA_DEFINE_STALL_SETTER(set_stall_fused)

}  // namespace mhla
