// The MHLA module around the core ([P1] "MHLA：通过令牌级多头机制恢复线性注意力
// 机制的表达能力", 171host.com/767426.html, section 7, class MHLA: norm,
// to_qkv, lepe, to_out and forward):
//
//   xn = LayerNorm(x)                       mhla_ln_rows (one warp per token)
//   qkv = xn W_qkv^T (+ b_qkv)              mhla_gemm (gemm_kernels.cu), bias in its epilogue
//   o = MHLA(q, k, v)                       the core, reading q, k, v in place
//                                           from the qkv rows (strided views)
//   o += lepe(v) = dwconv5x5(v) + b_lepe    mhla_lepe_add (one pass over v and o)
//   y = o W_out^T (+ b_out)                 mhla_gemm, bias in its epilogue
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "mhla_internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"
#include "tma_host.h"

namespace mhla {

__device__ unsigned int g_module_error = 0;

namespace {

using namespace tc;

// ------------------------------------------------------------------ LayerNorm

// One warp per token row of C bf16 values (C % 8 == 0, C <= 32 * 8 * NV):
// mean, then the biased variance from the row held in registers, then
// (x - mean) / sqrt(var + eps) * weight + bias rounded to bf16.
template <int NV>
__global__ void __launch_bounds__(256) mhla_ln_rows(const __nv_bfloat16* __restrict__ x, __nv_bfloat16* __restrict__ y,
                                                    int64_t rows, int32_t C, const float* __restrict__ weight,
                                                    const float* __restrict__ bias, float eps) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int nu = C / 8;   // 16-byte units per row
  const uint4* src = reinterpret_cast<const uint4*>(x + row * C);
  uint4 v[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int u = lane + 32 * k;
    v[k] = u < nu ? src[u] : make_uint4(0u, 0u, 0u, 0u);
  }
  const float2 st = ln_row_stats<NV>(v, C, eps, lane);
  uint4* dst = reinterpret_cast<uint4*>(y + row * C);
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int u = lane + 32 * k;
    if (u >= nu) continue;
    const float4 ga = reinterpret_cast<const float4*>(weight)[2 * u], gb = reinterpret_cast<const float4*>(weight)[2 * u + 1];
    const float4 ba = reinterpret_cast<const float4*>(bias)[2 * u], bb = reinterpret_cast<const float4*>(bias)[2 * u + 1];
    const float g[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
    const float bt[8] = {ba.x, ba.y, ba.z, ba.w, bb.x, bb.y, bb.z, bb.w};
    dst[u] = ln_apply8(v[k], st.x, st.y, g, bt);
  }
}

// Rows of C <= 512: one row per half warp (16 lanes, NU 16-byte units each), so
// an SM keeps twice as many rows in flight as with a warp per row; the same
// statistics (mean, then the biased variance from the deviations) reduced
// within the half warp.
template <int NU>
__global__ void __launch_bounds__(256) mhla_ln_rows_half(const __nv_bfloat16* __restrict__ x,
                                                         __nv_bfloat16* __restrict__ y, int64_t rows, int32_t C,
                                                         const float* __restrict__ weight,
                                                         const float* __restrict__ bias, float eps) {
  const int lane = threadIdx.x & 15;
  const unsigned mask = 0xFFFFu << (threadIdx.x & 16);   // this half warp's lanes
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 4) + (threadIdx.x >> 4);
  if (row >= rows) return;
  const int nu = C / 8;
  const uint4* src = reinterpret_cast<const uint4*>(x + row * C);
  uint4 v[NU];
#pragma unroll
  for (int k = 0; k < NU; ++k) {
    const int u = lane + 16 * k;
    v[k] = u < nu ? src[u] : make_uint4(0u, 0u, 0u, 0u);
  }
  float s = 0.0f;
#pragma unroll
  for (int k = 0; k < NU; ++k) {
    const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&w[e]);
      s += __low2float(b2) + __high2float(b2);
    }
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) s += __shfl_xor_sync(mask, s, o, 16);
  const float mean = s / static_cast<float>(C);
  float q = 0.0f;
#pragma unroll
  for (int k = 0; k < NU; ++k) {
    if (lane + 16 * k >= nu) continue;
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
  for (int o = 8; o > 0; o >>= 1) q += __shfl_xor_sync(mask, q, o, 16);
  const float rstd = rsqrtf(q / static_cast<float>(C) + eps);
  uint4* dst = reinterpret_cast<uint4*>(y + row * C);
#pragma unroll
  for (int k = 0; k < NU; ++k) {
    const int u = lane + 16 * k;
    if (u >= nu) continue;
    const float4 ga = reinterpret_cast<const float4*>(weight)[2 * u], gb = reinterpret_cast<const float4*>(weight)[2 * u + 1];
    const float4 ba = reinterpret_cast<const float4*>(bias)[2 * u], bb = reinterpret_cast<const float4*>(bias)[2 * u + 1];
    const float g[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
    const float bt[8] = {ba.x, ba.y, ba.z, ba.w, bb.x, bb.y, bb.z, bb.w};
    dst[u] = ln_apply8(v[k], mean, rstd, g, bt);
  }
}

// ------------------------------------------------------- LePE (5 x 5 depthwise)

// Persistent CTAs each walk one contiguous run of 8 x 16 token patches of one
// frame and 64 channels (32 pairs), channel chunk slowest, so a CTA changes
// chunk (and reloads the 5 x 5 weights) at most a few times and its
// neighbouring patches share their halos in L2.  Per patch two TMA loads land in one of two
// stage buffers: v with its 2-token halo, [12][20][64] bf16, whose out-of-frame
// elements read as zero (the convolution's padding), and the o tile,
// [8][16][64] bf16.  Eight compute warps: thread (pair q = lane, row y, strip s)
// convolves kLpSX tokens of its row for its two channels with packed float32
// FMAs and adds them into the o tile in place (the 32 lanes of a warp touch 128
// contiguous bytes, no bank conflicts), then reports the stage done.  A ninth
// warp stores each finished o tile by TMA (clipped at the frame and channel
// edges); the v patch two ahead loads into the stage at once (the store does not
// read it), that patch's o tile once the store has read the old one, so the
// compute warps never wait on a store.
constexpr int kLpTY = 8, kLpTX = 16, kLpHY = kLpTY + 4, kLpHX = kLpTX + 4;
constexpr int kLpV = kLpHY * kLpHX * 128;                     // v patch bytes
constexpr int kLpO = kLpTY * kLpTX * 128;                     // o tile bytes
constexpr int kLpStage = kLpV + kLpO;
constexpr int kLpSX = 16;                                     // tokens of a row one thread convolves
constexpr int kLpWorkers = 32 * kLpTY * (kLpTX / kLpSX);      // 256: warp = (row, strip)
constexpr int kLpThreads = kLpWorkers + 32;                   // + the store / load warp
constexpr uint32_t kLpBar = 1;                                // named barrier of the compute warps
constexpr size_t kLpSmem = 2 * kLpStage + 25 * 64 * 4 + 64 * 4 + 4 * 8 + 8 + 128;

struct LpGeom {
  uint32_t ntiles;                  // below 2^31 (checked on the host)
  int32_t C, B, T, Y, X, ntx, nty;
};

// acc += w * v on two float32 lanes (each lane rounds like fmaf)
__device__ __forceinline__ uint64_t fma2(uint64_t w, uint64_t v, uint64_t acc) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(w), "l"(v), "l"(acc));
  return d;
}

__global__ void __launch_bounds__(kLpThreads, 2) mhla_lepe_add(const __grid_constant__ CUtensorMap tm_v,
                                                               const __grid_constant__ CUtensorMap tm_o, LpGeom g,
                                                               const float* __restrict__ weight,
                                                               const float* __restrict__ bias) {
  extern __shared__ uint8_t lp_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(lp_raw) + 127) & ~uintptr_t{127});
  uint8_t* stage = smem;                                              // [2] (v patch, o tile)
  float* wsm = reinterpret_cast<float*>(smem + 2 * kLpStage);         // [25 taps][64 channels]
  float* bsm = wsm + 25 * 64;                                         // [64]
  uint64_t* full = reinterpret_cast<uint64_t*>(bsm + 64);             // [2] patch and o tile landed
  uint64_t* done = full + 2;                                          // [2] compute warps finished the o tile
  volatile uint32_t* abortf = reinterpret_cast<volatile uint32_t*>(full + 4);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t frames = static_cast<uint32_t>(g.B) * static_cast<uint32_t>(g.T);
  // this CTA's tiles [t_lo, t_hi)
  const uint32_t t_lo = static_cast<uint32_t>(static_cast<uint64_t>(g.ntiles) * blockIdx.x / gridDim.x);
  const uint32_t t_hi = static_cast<uint32_t>(static_cast<uint64_t>(g.ntiles) * (blockIdx.x + 1) / gridDim.x);

  // tile -> (chunk, frame, ty, tx), tx fastest (32-bit arithmetic)
  auto decode = [&](uint32_t t, int& chunk, int64_t& frame, int& ty, int& tx) {
    tx = static_cast<int>(t % static_cast<uint32_t>(g.ntx));
    uint32_t r = t / static_cast<uint32_t>(g.ntx);
    ty = static_cast<int>(r % static_cast<uint32_t>(g.nty));
    r /= static_cast<uint32_t>(g.nty);
    frame = r % frames;
    chunk = static_cast<int>(r / frames);
  };
  if (tid == kLpWorkers) {
    for (int st = 0; st < 2; ++st) {
      mbar_init(full + st, 2);            // the v patch and the o tile, loaded separately
      mbar_init(done + st, kLpWorkers / 32);
    }
    *abortf = 0u;
    fence_mbar_init();
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_o);
  }
  __syncthreads();

  if (warp == kLpWorkers / 32) {
    // ------------------------------------------------------------ stores and loads
    if (lane == 0) {
      uint32_t issued[2] = {0u, 0u};
      auto issue = [&](int st, uint32_t t, bool v_part) {
        int chunk, ty, tx;
        int64_t frame;
        decode(t, chunk, frame, ty, tx);
        const int32_t tf = static_cast<int32_t>(frame % g.T), b = static_cast<int32_t>(frame / g.T);
        const uint64_t pol = policy_evict_first();
        if (v_part) {
          mbar_arrive_expect_tx(full + st, kLpV);
          tma_load_5d(stage + st * kLpStage, &tm_v, full + st, chunk * 64, tx * kLpTX - 2, ty * kLpTY - 2, tf, b,
                      pol);
        } else {
          mbar_arrive_expect_tx(full + st, kLpO);
          tma_load_5d(stage + st * kLpStage + kLpV, &tm_o, full + st, chunk * 64, tx * kLpTX, ty * kLpTY, tf, b,
                      pol);
          ++issued[st];
        }
      };
      for (int st = 0; st < 2; ++st)
        if (t_lo + st < t_hi) {
          issue(st, t_lo + st, true);
          issue(st, t_lo + st, false);
        }
      uint32_t k = 0;
      for (uint32_t t = t_lo; t < t_hi; ++t, ++k) {
        const int st = static_cast<int>(k & 1u);
        if (!wait_bounded_on(done + st, (k >> 1) & 1u, abortf, &g_module_error)) break;
        int chunk, ty, tx;
        int64_t frame;
        decode(t, chunk, frame, ty, tx);
        const int32_t tf = static_cast<int32_t>(frame % g.T), b = static_cast<int32_t>(frame / g.T);
        tma_store_5d(&tm_o, stage + st * kLpStage + kLpV, chunk * 64, tx * kLpTX, ty * kLpTY, tf, b);
        bulk_commit_group();
        if (t + 2 < t_hi) {
          issue(st, t + 2, true);                 // the compute warps are done with the patch
          bulk_wait_group_read<0>();              // the store has read the o tile: reload it
          issue(st, t + 2, false);
        }
      }
      bulk_wait_group0();
      for (int st = 0; st < 2; ++st)
        if (issued[st]) drain_wait_on(full + st, (issued[st] - 1) & 1u, &g_module_error);
    }
  } else {
    // ------------------------------------------------------------ compute warps
    const int y = warp % kLpTY, s = warp / kLpTY;   // output row, strip of kLpSX tokens
    const int ch = 2 * lane;
    int cur_chunk = -1;
    uint32_t k = 0;
    for (uint32_t t = t_lo; t < t_hi; ++t, ++k) {
      int chunk, ty, tx;
      int64_t frame;
      decode(t, chunk, frame, ty, tx);
      const int c0 = chunk * 64;
      const int pairs = min(32, (g.C - c0) / 2);   // a multiple of 4
      if (chunk != cur_chunk) {
        // the chunk's 64 x 25 weights and 64 biases: every load in flight at once
        constexpr int kPer = (64 * 25 + kLpWorkers - 1) / kLpWorkers;
        float wv[kPer];
#pragma unroll
        for (int r = 0; r < kPer; ++r) {
          const int e = tid + r * kLpWorkers;
          wv[r] = e < pairs * 2 * 25 ? __ldg(weight + static_cast<int64_t>(c0) * 25 + e) : 0.0f;
        }
        const float bv = tid < pairs * 2 ? __ldg(bias + c0 + tid) : 0.0f;
        // every compute warp is done with the previous chunk's weights (the
        // chunk sequence and every exit below are the same for all of them)
        named_bar_sync(kLpBar, kLpWorkers);
#pragma unroll
        for (int r = 0; r < kPer; ++r) {
          const int e = tid + r * kLpWorkers;   // = channel * 25 + tap
          if (e < pairs * 2 * 25) wsm[(e % 25) * 64 + e / 25] = wv[r];
        }
        if (tid < pairs * 2) bsm[tid] = bv;
        cur_chunk = chunk;
      }
      const int st = static_cast<int>(k & 1u);
      const bool ok = warp_wait_on(full + st, (k >> 1) & 1u, abortf, &g_module_error);
      // one verdict for all compute warps; also orders the weights before their use
      if (!named_bar_and(kLpBar, kLpWorkers, ok)) break;

      if (lane < pairs) {
        const uint8_t* pl = stage + st * kLpStage + (y * kLpHX + s * kLpSX) * 128 + lane * 4;
        uint32_t* ot =
            reinterpret_cast<uint32_t*>(stage + st * kLpStage + kLpV + (y * kLpTX + s * kLpSX) * 128) + lane;
        uint64_t acc[kLpSX];
        const uint64_t bias2 = *reinterpret_cast<const uint64_t*>(bsm + ch);
#pragma unroll
        for (int x = 0; x < kLpSX; ++x) acc[x] = bias2;
#pragma unroll
        for (int i = 0; i < 5; ++i) {
          uint64_t vv[kLpSX + 4];
#pragma unroll
          for (int c = 0; c < kLpSX + 4; ++c) {   // bf16 pair -> float32 pair (exact)
            const uint32_t w = *reinterpret_cast<const uint32_t*>(pl + (i * kLpHX + c) * 128);
            vv[c] = static_cast<uint64_t>(w << 16) | (static_cast<uint64_t>(w & 0xFFFF0000u) << 32);
          }
#pragma unroll
          for (int j = 0; j < 5; ++j) {
            const uint64_t w2 = *reinterpret_cast<const uint64_t*>(wsm + (i * 5 + j) * 64 + ch);
#pragma unroll
            for (int x = 0; x < kLpSX; ++x) acc[x] = fma2(w2, vv[x + j], acc[x]);
          }
        }
        // o + (bias + conv), rounded once, in place in the o tile
#pragma unroll
        for (int x = 0; x < kLpSX; ++x) {
          const uint32_t ow = ot[x * 32];
          const __nv_bfloat162 o2 = *reinterpret_cast<const __nv_bfloat162*>(&ow);
          const __nv_bfloat162 r =
              __floats2bfloat162_rn(__low2float(o2) + __uint_as_float(static_cast<uint32_t>(acc[x])),
                                    __high2float(o2) + __uint_as_float(static_cast<uint32_t>(acc[x] >> 32)));
          ot[x * 32] = *reinterpret_cast<const uint32_t*>(&r);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(done + st);
    }
  }
}

}  // namespace

// ------------------------------------------------------------- host entries

int launch_layer_norm(const void* x, void* y, int64_t rows, int32_t C, const float* weight, const float* bias,
                      float eps, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const unsigned grid = static_cast<unsigned>((rows + 7) / 8);
  const auto* xi = static_cast<const __nv_bfloat16*>(x);
  auto* yo = static_cast<__nv_bfloat16*>(y);
  KernelTimer timer("mhla_ln_rows", stream);
  const int nv = (C / 8 + 31) / 32;
  const unsigned grid_half = static_cast<unsigned>((rows + 15) / 16);
  const int nu16 = (C / 8 + 15) / 16;   // units per lane of a half warp
  if (nu16 <= 1) mhla_ln_rows_half<1><<<grid_half, 256, 0, s>>>(xi, yo, rows, C, weight, bias, eps);
  else if (nu16 <= 2) mhla_ln_rows_half<2><<<grid_half, 256, 0, s>>>(xi, yo, rows, C, weight, bias, eps);
  else if (nu16 <= 3) mhla_ln_rows_half<3><<<grid_half, 256, 0, s>>>(xi, yo, rows, C, weight, bias, eps);
  else if (nu16 <= 4) mhla_ln_rows_half<4><<<grid_half, 256, 0, s>>>(xi, yo, rows, C, weight, bias, eps);
  else if (nv <= 4) mhla_ln_rows<4><<<grid, 256, 0, s>>>(xi, yo, rows, C, weight, bias, eps);
  else mhla_ln_rows<8><<<grid, 256, 0, s>>>(xi, yo, rows, C, weight, bias, eps);
  return cudaGetLastError() == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
}

int launch_lepe_add(const LepeArgs& a, void* stream) {
  // v and o as 5-D tensors (channel, x, y, frame, batch); their heads are adjacent
  auto map = [&](const void* base, int64_t sn, int64_t sb, uint32_t bx, uint32_t by, CUtensorMap* m) {
    const int64_t frame_stride = static_cast<int64_t>(a.Y) * a.X * sn;
    const int64_t bstride = a.B > 1 ? sb : frame_stride * a.T;
    const cuuint64_t dims[5] = {static_cast<cuuint64_t>(a.C), static_cast<cuuint64_t>(a.X),
                                static_cast<cuuint64_t>(a.Y), static_cast<cuuint64_t>(a.T),
                                static_cast<cuuint64_t>(a.B)};
    const cuuint64_t strides[4] = {static_cast<cuuint64_t>(sn * 2), static_cast<cuuint64_t>(a.X * sn * 2),
                                   static_cast<cuuint64_t>(frame_stride * 2), static_cast<cuuint64_t>(bstride * 2)};
    const cuuint32_t box[5] = {64u, bx, by, 1u, 1u};
    return encode_tensor_map(m, 5, const_cast<void*>(base), dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
  };
  CUtensorMap tv, to;
  if (!map(a.v, a.vsn, a.vsb, kLpHX, kLpHY, &tv) || !map(a.o, a.osn, a.osb, kLpTX, kLpTY, &to)) return MHLA_ERR_CUDA;
  LpGeom g;
  g.C = a.C; g.B = static_cast<int32_t>(a.B); g.T = a.T; g.Y = a.Y; g.X = a.X;
  g.ntx = (a.X + kLpTX - 1) / kLpTX;
  g.nty = (a.Y + kLpTY - 1) / kLpTY;
  const int64_t ntiles = static_cast<int64_t>((a.C + 63) / 64) * a.B * a.T * g.nty * g.ntx;
  if (ntiles >= (int64_t{1} << 31)) return MHLA_ERR_UNSUPPORTED;
  g.ntiles = static_cast<uint32_t>(ntiles);
  // a per-device setting: made on every call, for whichever device is current
  if (cudaFuncSetAttribute(mhla_lepe_add, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kLpSmem)) !=
      cudaSuccess)
    return MHLA_ERR_CUDA;
  const int sms = device_sm_count();
  if (sms <= 0) return MHLA_ERR_CUDA;
  const int grid = static_cast<int>(std::min<int64_t>(ntiles, 2 * static_cast<int64_t>(sms)));
  KernelTimer timer("mhla_lepe_add", stream);
  mhla_lepe_add<<<grid, kLpThreads, kLpSmem, static_cast<cudaStream_t>(stream)>>>(tv, to, g, a.weight, a.bias);
  return cudaGetLastError() == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
}

int read_and_clear_module_error(void* stream, uint32_t* flags) {
  return read_and_clear_word(g_module_error, stream, flags);
}

MHLA_DEFINE_STALL_SETTER(set_stall_module)

}  // namespace mhla
