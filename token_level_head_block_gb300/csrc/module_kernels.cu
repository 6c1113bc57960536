// The MHLA module around the core ([P1] "MHLA：通过令牌级多头机制恢复线性注意力
// 机制的表达能力", 171host.com/767426.html, section 7, class MHLA: norm,
// to_qkv, lepe, to_out and forward):
//
//   xn = LayerNorm(x)                       mhla_ln_rows (one warp per token)
//   qkv = xn W_qkv^T (+ b_qkv)              cuBLASLt GEMM, bias in its epilogue
//   o = MHLA(q, k, v)                       the core, reading q, k, v in place
//                                           from the qkv rows (strided views)
//   o += lepe(v) = dwconv5x5(v) + b_lepe    mhla_lepe_add (one pass over v and o)
//   y = o W_out^T (+ b_out)                 cuBLASLt GEMM, bias in its epilogue
//
// The projections are plain GEMMs and go to cuBLASLt, which is loaded at run
// time (dlopen), so the library loads on machines without it and only the
// module call reports MHLA_ERR_UNSUPPORTED there.
#include <cublasLt.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <dlfcn.h>

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
  float s = 0.0f;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int u = lane + 32 * k;
    v[k] = u < nu ? src[u] : make_uint4(0u, 0u, 0u, 0u);
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
  const float rstd = rsqrtf(q / static_cast<float>(C) + eps);
  uint4* dst = reinterpret_cast<uint4*>(y + row * C);
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int u = lane + 32 * k;
    if (u >= nu) continue;
    const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
    const float4 ga = reinterpret_cast<const float4*>(weight)[2 * u], gb = reinterpret_cast<const float4*>(weight)[2 * u + 1];
    const float4 ba = reinterpret_cast<const float4*>(bias)[2 * u], bb = reinterpret_cast<const float4*>(bias)[2 * u + 1];
    const float g[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
    const float bt[8] = {ba.x, ba.y, ba.z, ba.w, bb.x, bb.y, bb.z, bb.w};
    uint32_t out[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&w[e]);
      const float a = (__low2float(b2) - mean) * rstd * g[2 * e] + bt[2 * e];
      const float b = (__high2float(b2) - mean) * rstd * g[2 * e + 1] + bt[2 * e + 1];
      const __nv_bfloat162 r = __floats2bfloat162_rn(a, b);
      out[e] = *reinterpret_cast<const uint32_t*>(&r);
    }
    dst[u] = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

// ------------------------------------------------------- LePE (5 x 5 depthwise)

// Persistent CTAs walk 8 x 16 token patches of one frame and 64 channels (32
// pairs), channel chunk slowest.  Per patch two TMA loads land in one of two
// stage buffers: v with its 2-token halo, [12][20][64] bf16, whose out-of-frame
// elements read as zero (the convolution's padding), and the o tile,
// [8][16][64] bf16.  Thread (pair q = lane, row y, strip s) convolves 8 tokens
// of its row for its two channels with packed float32 FMAs and adds them into
// the o tile in place (the 32 lanes of a warp touch 128 contiguous bytes, no
// bank conflicts); one TMA store then writes the tile back, clipped at the
// frame and channel edges.  The next patch's loads run while this one is
// convolved; the 5 x 5 weights are reloaded only when the chunk changes.
constexpr int kLpTY = 8, kLpTX = 16, kLpHY = kLpTY + 4, kLpHX = kLpTX + 4;
constexpr int kLpV = kLpHY * kLpHX * 128;                     // v patch bytes
constexpr int kLpO = kLpTY * kLpTX * 128;                     // o tile bytes
constexpr int kLpStage = kLpV + kLpO;
constexpr int kLpThreads = 32 * kLpTY * (kLpTX / 8);          // 512: warp = (row, strip)
constexpr size_t kLpSmem = 2 * kLpStage + 25 * 64 * 4 + 64 * 4 + 64 + 128;

struct LpGeom {
  int64_t ntiles;
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
  uint64_t* full = reinterpret_cast<uint64_t*>(bsm + 64);             // [2]
  volatile uint32_t* abortf = reinterpret_cast<volatile uint32_t*>(full + 2);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t frames = static_cast<int64_t>(g.B) * g.T;

  // tile -> (chunk, frame, ty, tx), tx fastest
  auto decode = [&](int64_t t, int& chunk, int64_t& frame, int& ty, int& tx) {
    tx = static_cast<int>(t % g.ntx);
    int64_t r = t / g.ntx;
    ty = static_cast<int>(r % g.nty);
    r /= g.nty;
    frame = r % frames;
    chunk = static_cast<int>(r / frames);
  };
  uint32_t issued[2] = {0u, 0u};
  auto issue = [&](int st, int64_t t) {
    int chunk, ty, tx;
    int64_t frame;
    decode(t, chunk, frame, ty, tx);
    const int32_t tf = static_cast<int32_t>(frame % g.T), b = static_cast<int32_t>(frame / g.T);
    const uint64_t pol = policy_evict_first();
    mbar_arrive_expect_tx(full + st, kLpStage);
    tma_load_5d(stage + st * kLpStage, &tm_v, full + st, chunk * 64, tx * kLpTX - 2, ty * kLpTY - 2, tf, b, pol);
    tma_load_5d(stage + st * kLpStage + kLpV, &tm_o, full + st, chunk * 64, tx * kLpTX, ty * kLpTY, tf, b, pol);
    ++issued[st];
  };
  if (tid == 0) {
    mbar_init(full, 1);
    mbar_init(full + 1, 1);
    *abortf = 0u;
    fence_mbar_init();
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_o);
    for (int st = 0; st < 2; ++st)
      if (static_cast<int64_t>(blockIdx.x) + st * gridDim.x < g.ntiles) issue(st, blockIdx.x + st * gridDim.x);
  }
  __syncthreads();

  const int y = warp % kLpTY, s = warp / kLpTY;   // output row, 8-token strip
  const int ch = 2 * lane;
  int cur_chunk = -1;
  uint32_t k = 0;
  for (int64_t t = blockIdx.x; t < g.ntiles; t += gridDim.x, ++k) {
    int chunk, ty, tx;
    int64_t frame;
    decode(t, chunk, frame, ty, tx);
    const int c0 = chunk * 64;
    const int pairs = min(32, (g.C - c0) / 2);   // a multiple of 4
    if (chunk != cur_chunk) {                    // the previous patch is done (barrier below)
      for (int e = tid; e < pairs * 2 * 25; e += kLpThreads) {
        const int c = e / 25, tap = e % 25;
        wsm[tap * 64 + c] = weight[static_cast<int64_t>(c0 + c) * 25 + tap];
      }
      for (int e = tid; e < pairs * 2; e += kLpThreads) bsm[e] = bias[c0 + e];
      cur_chunk = chunk;
    }
    const int st = static_cast<int>(k & 1u);
    const bool ok = warp_wait_on(full + st, (k >> 1) & 1u, abortf, &g_module_error);
    if (!__syncthreads_and(ok)) break;

    if (lane < pairs) {
      const uint8_t* pl = stage + st * kLpStage + (y * kLpHX + s * 8) * 128 + lane * 4;
      uint32_t* ot = reinterpret_cast<uint32_t*>(stage + st * kLpStage + kLpV + (y * kLpTX + s * 8) * 128) + lane;
      uint64_t acc[8];
      const uint64_t bias2 = *reinterpret_cast<const uint64_t*>(bsm + ch);
#pragma unroll
      for (int x = 0; x < 8; ++x) acc[x] = bias2;
#pragma unroll
      for (int i = 0; i < 5; ++i) {
        uint64_t vv[12];
#pragma unroll
        for (int c = 0; c < 12; ++c) {   // bf16 pair -> float32 pair (exact)
          const uint32_t w = *reinterpret_cast<const uint32_t*>(pl + (i * kLpHX + c) * 128);
          vv[c] = static_cast<uint64_t>(w << 16) | (static_cast<uint64_t>(w & 0xFFFF0000u) << 32);
        }
#pragma unroll
        for (int j = 0; j < 5; ++j) {
          const uint64_t w2 = *reinterpret_cast<const uint64_t*>(wsm + (i * 5 + j) * 64 + ch);
#pragma unroll
          for (int x = 0; x < 8; ++x) acc[x] = fma2(w2, vv[x + j], acc[x]);
        }
      }
      // o + (bias + conv), rounded once, in place in the o tile
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        const uint32_t ow = ot[x * 32];
        const __nv_bfloat162 o2 = *reinterpret_cast<const __nv_bfloat162*>(&ow);
        const __nv_bfloat162 r =
            __floats2bfloat162_rn(__low2float(o2) + __uint_as_float(static_cast<uint32_t>(acc[x])),
                                  __high2float(o2) + __uint_as_float(static_cast<uint32_t>(acc[x] >> 32)));
        ot[x * 32] = *reinterpret_cast<const uint32_t*>(&r);
      }
    }
    fence_proxy_async_smem();
    __syncthreads();                             // the o tile is complete; the weights are free
    if (tid == 0) {
      const int32_t tf = static_cast<int32_t>(frame % g.T), b = static_cast<int32_t>(frame / g.T);
      tma_store_5d(&tm_o, stage + st * kLpStage + kLpV, c0, tx * kLpTX, ty * kLpTY, tf, b);
      bulk_commit_group();
      if (t + 2 * static_cast<int64_t>(gridDim.x) < g.ntiles) {
        bulk_wait_group_read<0>();               // the store has read the stage: reload it
        issue(st, t + 2 * gridDim.x);
      }
    }
  }
  if (tid == 0) {
    bulk_wait_group0();
    for (int st = 0; st < 2; ++st)
      if (issued[st]) drain_wait_on(full + st, (issued[st] - 1) & 1u, &g_module_error);
  }
}

// ------------------------------------------------------------ cuBLASLt loader

struct LtApi {
  decltype(&cublasLtCreate) create = nullptr;
  decltype(&cublasLtMatmulDescCreate) desc_create = nullptr;
  decltype(&cublasLtMatmulDescSetAttribute) desc_set = nullptr;
  decltype(&cublasLtMatmulDescDestroy) desc_destroy = nullptr;
  decltype(&cublasLtMatrixLayoutCreate) layout_create = nullptr;
  decltype(&cublasLtMatrixLayoutDestroy) layout_destroy = nullptr;
  decltype(&cublasLtMatmulPreferenceCreate) pref_create = nullptr;
  decltype(&cublasLtMatmulPreferenceSetAttribute) pref_set = nullptr;
  decltype(&cublasLtMatmulPreferenceDestroy) pref_destroy = nullptr;
  decltype(&cublasLtMatmulAlgoGetHeuristic) heuristic = nullptr;
  decltype(&cublasLtMatmul) matmul = nullptr;
  bool ok = false;   // every entry point found
};

const LtApi& lt_api() {
  static LtApi api;
  static std::once_flag once;
  std::call_once(once, [] {
    const char* names[] = {"libcublasLt.so.13", "libcublasLt.so", "/usr/local/cuda/lib64/libcublasLt.so.13",
                           "/usr/local/cuda/targets/sbsa-linux/lib/libcublasLt.so.13",
                           "/usr/local/cuda/targets/x86_64-linux/lib/libcublasLt.so.13"};
    void* h = nullptr;
    for (const char* n : names)
      if ((h = dlopen(n, RTLD_NOW | RTLD_LOCAL)) != nullptr) break;
    if (!h) return;
    auto sym = [&](auto& fn, const char* name) {
      fn = reinterpret_cast<std::remove_reference_t<decltype(fn)>>(dlsym(h, name));
      return fn != nullptr;
    };
    bool all = sym(api.create, "cublasLtCreate") && sym(api.desc_create, "cublasLtMatmulDescCreate") &&
               sym(api.desc_set, "cublasLtMatmulDescSetAttribute") &&
               sym(api.desc_destroy, "cublasLtMatmulDescDestroy") &&
               sym(api.layout_create, "cublasLtMatrixLayoutCreate") &&
               sym(api.layout_destroy, "cublasLtMatrixLayoutDestroy") &&
               sym(api.pref_create, "cublasLtMatmulPreferenceCreate") &&
               sym(api.pref_set, "cublasLtMatmulPreferenceSetAttribute") &&
               sym(api.pref_destroy, "cublasLtMatmulPreferenceDestroy") &&
               sym(api.heuristic, "cublasLtMatmulAlgoGetHeuristic") && sym(api.matmul, "cublasLtMatmul");
    api.ok = all;
  });
  return api;
}

// One cuBLASLt handle per device, created on first use with that device
// current; null when the device cannot be used.
cublasLtHandle_t lt_handle() {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static cublasLtHandle_t handles[kMaxDevices] = {};
  const LtApi& lt = lt_api();
  int dev = -1;
  if (!lt.ok || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!handles[dev] && lt.create(&handles[dev]) != CUBLAS_STATUS_SUCCESS) handles[dev] = nullptr;
  return handles[dev];
}

constexpr size_t kLtWorkspace = size_t{32} << 20;

// y[rows][n_out] = x[rows][k] W^T (+ bias[n_out]), W [n_out][k], all bf16 and
// row-major, float32 accumulation.  In cuBLASLt's column-major terms:
// y^T (n_out x rows) = op_T(W stored k x n_out) * x^T (k x rows).
int linear_bf16(const char* name, const void* x, const void* W, const void* bias, void* y, int64_t rows, int64_t k,
                int64_t n_out, void* lt_ws, cudaStream_t stream) {
  const LtApi& lt = lt_api();
  const cublasLtHandle_t handle = lt_handle();
  if (!handle) return MHLA_ERR_UNSUPPORTED;
  cublasLtMatmulDesc_t op = nullptr;
  cublasLtMatrixLayout_t la = nullptr, lb = nullptr, lc = nullptr;
  cublasLtMatmulPreference_t pref = nullptr;
  int rc = MHLA_ERR_CUDA;
  do {
    if (lt.desc_create(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F) != CUBLAS_STATUS_SUCCESS) break;
    const cublasOperation_t ta = CUBLAS_OP_T, tb = CUBLAS_OP_N;
    if (lt.desc_set(op, CUBLASLT_MATMUL_DESC_TRANSA, &ta, sizeof(ta)) != CUBLAS_STATUS_SUCCESS) break;
    if (lt.desc_set(op, CUBLASLT_MATMUL_DESC_TRANSB, &tb, sizeof(tb)) != CUBLAS_STATUS_SUCCESS) break;
    if (bias) {
      const cublasLtEpilogue_t epi = CUBLASLT_EPILOGUE_BIAS;
      if (lt.desc_set(op, CUBLASLT_MATMUL_DESC_EPILOGUE, &epi, sizeof(epi)) != CUBLAS_STATUS_SUCCESS) break;
      if (lt.desc_set(op, CUBLASLT_MATMUL_DESC_BIAS_POINTER, &bias, sizeof(bias)) != CUBLAS_STATUS_SUCCESS) break;
    }
    if (lt.layout_create(&la, CUDA_R_16BF, static_cast<uint64_t>(k), static_cast<uint64_t>(n_out), k) !=
            CUBLAS_STATUS_SUCCESS ||
        lt.layout_create(&lb, CUDA_R_16BF, static_cast<uint64_t>(k), static_cast<uint64_t>(rows), k) !=
            CUBLAS_STATUS_SUCCESS ||
        lt.layout_create(&lc, CUDA_R_16BF, static_cast<uint64_t>(n_out), static_cast<uint64_t>(rows), n_out) !=
            CUBLAS_STATUS_SUCCESS)
      break;
    if (lt.pref_create(&pref) != CUBLAS_STATUS_SUCCESS) break;
    const uint64_t wsb = kLtWorkspace;
    if (lt.pref_set(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &wsb, sizeof(wsb)) != CUBLAS_STATUS_SUCCESS) break;
    cublasLtMatmulHeuristicResult_t res{};
    int found = 0;
    if (lt.heuristic(handle, op, la, lb, lc, lc, pref, 1, &res, &found) != CUBLAS_STATUS_SUCCESS || found < 1) {
      rc = MHLA_ERR_UNSUPPORTED;
      break;
    }
    const float alpha = 1.0f, beta = 0.0f;
    KernelTimer timer(name, stream);
    if (lt.matmul(handle, op, &alpha, W, la, x, lb, &beta, y, lc, y, lc, &res.algo, lt_ws, kLtWorkspace, stream) !=
        CUBLAS_STATUS_SUCCESS)
      break;
    rc = MHLA_OK;
  } while (false);
  if (pref) lt.pref_destroy(pref);
  if (lc) lt.layout_destroy(lc);
  if (lb) lt.layout_destroy(lb);
  if (la) lt.layout_destroy(la);
  if (op) lt.desc_destroy(op);
  return rc;
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
  if (nv <= 1) mhla_ln_rows<1><<<grid, 256, 0, s>>>(xi, yo, rows, C, weight, bias, eps);
  else if (nv <= 2) mhla_ln_rows<2><<<grid, 256, 0, s>>>(xi, yo, rows, C, weight, bias, eps);
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
  g.ntiles = static_cast<int64_t>((a.C + 63) / 64) * a.B * a.T * g.nty * g.ntx;
  // a per-device setting: made on every call, for whichever device is current
  if (cudaFuncSetAttribute(mhla_lepe_add, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kLpSmem)) !=
      cudaSuccess)
    return MHLA_ERR_CUDA;
  const int sms = device_sm_count();
  if (sms <= 0) return MHLA_ERR_CUDA;
  const int grid = static_cast<int>(std::min<int64_t>(g.ntiles, 2 * static_cast<int64_t>(sms)));
  KernelTimer timer("mhla_lepe_add", stream);
  mhla_lepe_add<<<grid, kLpThreads, kLpSmem, static_cast<cudaStream_t>(stream)>>>(tv, to, g, a.weight, a.bias);
  return cudaGetLastError() == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
}

int read_and_clear_module_error(void* stream, uint32_t* flags) {
  return read_and_clear_word(g_module_error, stream, flags);
}

int launch_linear(const char* name, const void* x, const void* W, const void* bias, void* y, int64_t rows, int64_t k,
                  int64_t n_out, void* lt_ws, void* stream) {
  return linear_bf16(name, x, W, bias, y, rows, k, n_out, lt_ws, static_cast<cudaStream_t>(stream));
}

bool linear_available() { return lt_handle() != nullptr; }

size_t linear_workspace_bytes() { return kLtWorkspace; }

}  // namespace mhla
