// Shared pieces of the tensor-core kernels (forward and backward): bounded
// mbarrier waits, the token-chunk geometry of a block, phi on packed bf16,
// swizzle phases, and the host side of the TMA maps over [B, N, H, d] operands.
// Every translation unit that includes it passes its own device error word to
// the waits.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <utility>

#include "mhla_internal.h"
#include "ptx.cuh"
#include "stall_hook.cuh"
#include "tma_host.h"

namespace mhla {
namespace tc {

using namespace ptx;

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr uint32_t kWaitLimitPolls = 1u << 28;
constexpr uint64_t kDrainLimitNs = 50000000ull;   // 50 ms for copies already in flight

static __device__ __noinline__ bool wait_bounded_on(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag,
                                                    unsigned int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  // diagnostic hook (stall_hook.cuh), looked at only once a wait has to poll:
  // for the chosen warp the completion never comes
  if (stall_this_warp()) {
    stalled_wait(abort_flag);
    *abort_flag = 1u;
    atomicOr(err, 1u);
    return false;
  }
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1; it < kWaitLimitPolls; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > kWaitLimitNs) break;
    }
  }
  *abort_flag = 1u;
  atomicOr(err, 1u);
  return false;
}

// Every lane waits, then the warp agrees: warp-collective instructions that
// follow (shuffles, tcgen05.ld) run either on all lanes or on none.
static __device__ __forceinline__ bool warp_wait_on(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag,
                                                    unsigned int* err) {
  const bool ok = wait_bounded_on(bar, parity, abort_flag, err);
  return __all_sync(0xffffffffu, ok);
}

// Wait for a phase that must already be under way (copies or MMAs in flight),
// without consulting the abort flag.
static __device__ __noinline__ void drain_wait_on(uint64_t* bar, uint32_t parity, unsigned int* err) {
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 0; it < kWaitLimitPolls; ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 63u) == 63u && globaltimer() - t0 > kDrainLimitNs) {
      atomicOr(err, 2u);
      return;
    }
  }
}

// Waits until a global counter another CTA of the same grid raises reaches
// target (acquire), bounded like the mbarrier waits; on success the data it
// publishes may be read by this thread's TMA and bulk copies too.
static __device__ __noinline__ bool wait_counter_on(const uint32_t* ctr, uint32_t target,
                                                    volatile uint32_t* abort_flag, unsigned int* err) {
  if (ld_acquire_gpu(ctr) >= target) {
    fence_proxy_async_global();
    return true;
  }
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1; it < kWaitLimitPolls; ++it) {
    __nanosleep(128);
    if (ld_acquire_gpu(ctr) >= target) {
      fence_proxy_async_global();
      return true;
    }
    if ((it & 15u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > kWaitLimitNs) break;
    }
  }
  *abort_flag = 1u;
  atomicOr(err, 1u);
  return false;
}

// Token-grid geometry of one launch (all int32: checked on the host).
struct TcGeom {
  int32_t M, nbx, nby;     // block grid, x fastest
  int32_t bx, by, bt, T;   // block extents; frames per batch image (1 for 2-D)
  int32_t box_y, box_t;    // TMA box of one chunk along y and t (x: whole block rows)
  int32_t nyc;             // chunks stacked along y inside one frame of a block
  int32_t chunks;          // chunks per block
  int32_t H, B;
};

// Coordinates (x, y, z = b*T + t) of chunk c of block j of batch b.
static __device__ __forceinline__ void chunk_coords(const TcGeom& g, int32_t j, int32_t c, int32_t b, int32_t& x,
                                             int32_t& y, int32_t& z) {
  const int32_t jx = j % g.nbx, jr = j / g.nbx;
  const int32_t jy = jr % g.nby, jt = jr / g.nby;
  x = jx * g.bx;
  y = jy * g.by + (c % g.nyc) * g.box_y;
  z = b * g.T + jt * g.bt + (c / g.nyc) * g.box_t;
}

// phi on eight bf16 values in place with packed bf16 arithmetic (no float32
// round trip): max(x, 0), then + eps under MHLA_PHI_RELU_EPS.
static __device__ __forceinline__ uint4 phi8_packed(uint4 raw, bool add_eps, __nv_bfloat162 eps2) {
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

static __device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// LayerNorm of a row of C bf16 values held by one warp, lane holding the
// 16-byte units lane, lane + 32, ... (zeros past C): the mean, then the biased
// variance from the deviations, both reduced in the same order by every
// kernel that normalises, so they agree bit for bit.  Returns (mean, rstd).
template <int NV>
static __device__ __forceinline__ float2 ln_row_stats(const uint4 (&v)[NV], int32_t C, float eps, int lane) {
  const int nu = C / 8;
  float s = 0.0f;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&w[e]);
      s += __low2float(b2) + __high2float(b2);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const float mean = s / static_cast<float>(C);
  float q = 0.0f;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    if (lane + 32 * k >= nu) continue;
    const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&w[e]);
      const float a = __low2float(b2) - mean, b = __high2float(b2) - mean;
      q = fmaf(a, a, q);
      q = fmaf(b, b, q);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
  return make_float2(mean, rsqrtf(q / static_cast<float>(C) + eps));
}

// Eight bf16 values of a row normalised, scaled and shifted, rounded once to
// bf16: y = (x - mean) rstd g + b.  Every LayerNorm in the library applies it
// through this function, so a fused normalisation equals the stand-alone one.
static __device__ __forceinline__ uint4 ln_apply8(uint4 raw, float mean, float rstd, const float (&g)[8],
                                                  const float (&bt)[8]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  uint32_t out[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&w[e]);
    const float a = (__low2float(b2) - mean) * rstd * g[2 * e] + bt[2 * e];
    const float b = (__high2float(b2) - mean) * rstd * g[2 * e + 1] + bt[2 * e + 1];
    const __nv_bfloat162 r = __floats2bfloat162_rn(a, b);
    out[e] = *reinterpret_cast<const uint32_t*>(&r);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// 16-byte chunk position inside a swizzled row: 128-byte swizzle for d = 64
// (row r XORs chunk bits with r mod 8), 64-byte swizzle for d = 32.
template <int D>
static __device__ __forceinline__ int swz(int row) {
  return D == 64 ? (row & 7) : ((row >> 1) & 3);
}

// ----------------------------------------------------------------- host side

// Launch with programmatic stream serialization: the grid may start while the
// previous kernel on the stream drains (its CTAs take SMs as they free up); the
// threads that read the previous kernel's results call grid_dep_wait() first.
template <typename... Params, typename... Args>
static cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename K>
int occupancy(K kernel, int threads, size_t smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess) return 0;
  return n;
}

// Copies a translation unit's device error word to *flags and clears it
// (synchronises stream); MHLA_ERR_TIMEOUT when it was set.
template <typename Word>
int read_and_clear_word(Word& word, void* stream, uint32_t* flags) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int host = 0;
  if (cudaMemcpyFromSymbolAsync(&host, word, sizeof(host), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MHLA_ERR_CUDA;
  const unsigned int zero = 0;
  if (cudaMemcpyToSymbolAsync(word, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return MHLA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MHLA_ERR_CUDA;
  *flags = host;
  return host ? MHLA_ERR_TIMEOUT : MHLA_OK;
}

struct ChunkPlan {
  int64_t box_y, box_t, nyc, chunks;
};

// Split every block into chunks of C tokens made of whole block rows (and,
// where a frame holds fewer than C tokens, whole frames).
inline bool chunk_plan(const Problem& p, int64_t C, ChunkPlan* cp) {
  if (p.w % C != 0 || C % p.bx != 0 || p.bx > 256) return false;
  const int64_t rows = C / p.bx;
  if (rows <= p.by) {
    if (p.by % rows != 0) return false;
    cp->box_y = rows;
    cp->box_t = 1;
    cp->nyc = p.by / rows;
  } else {
    if (rows % p.by != 0) return false;
    const int64_t frames = rows / p.by;
    if (p.bt % frames != 0) return false;
    cp->box_y = p.by;
    cp->box_t = frames;
    cp->nyc = 1;
  }
  if (cp->box_y > 256 || cp->box_t > 256) return false;
  cp->chunks = p.w / C;
  return true;
}

inline bool operand_tma_ok(const Problem& p, const Operand& o) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(o.data);
  if (a % 16 != 0) return false;
  if (o.sh % 8 != 0 || o.sn % 8 != 0 || o.sb % 8 != 0) return false;
  if ((p.H > 1 && o.sh <= 0) || o.sn <= 0) return false;
  if (p.T > 1 && o.sb != p.T * p.Y * p.X * o.sn) return false;   // (b, t) fold into one dimension
  const int64_t zstride = p.T > 1 ? p.Y * p.X * o.sn : o.sb;
  if (p.B > 1 && zstride <= 0) return false;
  const int64_t lim = int64_t{1} << 39;   // strides in bytes below 2^40
  return o.sh < lim && o.sn * p.X < lim && zstride < lim;
}

inline bool operand_map(const Problem& p, const Operand& o, int64_t box_y, int64_t box_t, CUtensorMap* m) {
  const int64_t zstride = p.T > 1 ? p.Y * p.X * o.sn : (p.B > 1 ? o.sb : p.Y * p.X * o.sn);
  const int64_t sh = p.H > 1 ? o.sh : p.d;
  const cuuint64_t dims[5] = {static_cast<cuuint64_t>(p.d), static_cast<cuuint64_t>(p.H),
                              static_cast<cuuint64_t>(p.X), static_cast<cuuint64_t>(p.Y),
                              static_cast<cuuint64_t>(p.B * p.T)};
  const cuuint64_t strides[4] = {static_cast<cuuint64_t>(sh * 2), static_cast<cuuint64_t>(o.sn * 2),
                                 static_cast<cuuint64_t>(p.X * o.sn * 2), static_cast<cuuint64_t>(zstride * 2)};
  const cuuint32_t box[5] = {static_cast<cuuint32_t>(p.d), 1u, static_cast<cuuint32_t>(p.bx),
                             static_cast<cuuint32_t>(box_y), static_cast<cuuint32_t>(box_t)};
  return encode_tensor_map(m, 5, o.data, dims, strides, box,
                           p.d == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}

inline TcGeom make_geom(const Problem& p, const ChunkPlan& cp) {
  TcGeom g;
  g.M = static_cast<int32_t>(p.M);
  g.nbx = static_cast<int32_t>(p.nbx);
  g.nby = static_cast<int32_t>(p.nby);
  g.bx = static_cast<int32_t>(p.bx);
  g.by = static_cast<int32_t>(p.by);
  g.bt = static_cast<int32_t>(p.bt);
  g.T = static_cast<int32_t>(p.T);
  g.box_y = static_cast<int32_t>(cp.box_y);
  g.box_t = static_cast<int32_t>(cp.box_t);
  g.nyc = static_cast<int32_t>(cp.nyc);
  g.chunks = static_cast<int32_t>(cp.chunks);
  g.H = static_cast<int32_t>(p.H);
  g.B = static_cast<int32_t>(p.B);
  return g;
}

}  // namespace tc
}  // namespace mhla
