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

namespace mhla {
namespace {

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

// One CTA: a 16 x 16 token patch of one frame and 64 channels (8 units of 8).
// The v patch with its 2-token halo is staged in shared memory, one plane per
// channel unit (plane stride padded by 16 bytes, so the 8 units of a token land
// in different banks).  Thread (unit u, row y, strip s) owns 8 tokens of row y
// and the 8 channels of unit u: it reads their o units, convolves two channels
// at a time with packed float32 FMAs, and writes the units back, so the 8
// threads of a token move its 128 contiguous bytes.
constexpr int kLpTY = 16, kLpTX = 16, kLpHY = kLpTY + 4, kLpHX = kLpTX + 4, kLpUnits = 8;
constexpr int kLpPlane = kLpHY * kLpHX * 16 + 16;   // bytes per channel-unit plane
constexpr int kLpThreads = kLpUnits * kLpTY * (kLpTX / 8);   // 256
constexpr size_t kLpSmem = static_cast<size_t>(kLpUnits) * kLpPlane + 25 * 64 * 4 + 64 * 4;

struct LpView {
  const __nv_bfloat16* v;
  __nv_bfloat16* o;
  int64_t vsb, vsn, vsh, osb, osn, osh;   // elements
  int32_t d, C, T, Y, X;
};

__device__ __forceinline__ int64_t unit_offset(int32_t c, int32_t d, int64_t sh) {
  return static_cast<int64_t>(c / d) * sh + (c % d);
}

// acc += w * v on two float32 lanes (each lane rounds like fmaf)
__device__ __forceinline__ uint64_t fma2(uint64_t w, uint64_t v, uint64_t acc) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(w), "l"(v), "l"(acc));
  return d;
}

__device__ __forceinline__ uint64_t pack_f2(float lo, float hi) {
  return static_cast<uint64_t>(__float_as_uint(lo)) | (static_cast<uint64_t>(__float_as_uint(hi)) << 32);
}

// the two bf16 values of a 32-bit word as a float32 pair (exact)
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t w) {
  return static_cast<uint64_t>(w << 16) | (static_cast<uint64_t>(w & 0xFFFF0000u) << 32);
}

__global__ void __launch_bounds__(kLpThreads, 3) mhla_lepe_add(LpView L, const float* __restrict__ weight,
                                                            const float* __restrict__ bias) {
  extern __shared__ __align__(16) uint8_t lp_smem[];
  uint8_t* planes = lp_smem;
  float* wsm = reinterpret_cast<float*>(lp_smem + kLpUnits * kLpPlane);   // [25 taps][64 channels]
  float* bsm = wsm + 25 * 64;                                              // [64]
  const int tid = threadIdx.x;
  const int nchunks = (L.C + 63) / 64;
  const int chunk = static_cast<int>(blockIdx.z % nchunks);
  const int64_t frame = blockIdx.z / nchunks;                               // b * T + t
  const int64_t b = frame / L.T, t = frame % L.T;
  const int y0 = blockIdx.y * kLpTY, x0 = blockIdx.x * kLpTX;
  const int c0 = chunk * 64;
  const int units = min(kLpUnits, (L.C - c0) / 8);
  const int64_t tok0 = t * static_cast<int64_t>(L.Y) * L.X;                 // first token of the frame

  for (int e = tid; e < units * 8 * 25; e += kLpThreads) {
    const int c = e / 25, tap = e % 25;
    wsm[tap * 64 + c] = weight[static_cast<int64_t>(c0 + c) * 25 + tap];
  }
  for (int e = tid; e < units * 8; e += kLpThreads) bsm[e] = bias[c0 + e];
  // v patch with halo, zero outside the frame
  for (int e = tid; e < kLpHY * kLpHX * kLpUnits; e += kLpThreads) {
    const int u = e % kLpUnits, pos = e / kLpUnits;
    const int hy = pos / kLpHX, hx = pos % kLpHX;
    const int gy = y0 + hy - 2, gx = x0 + hx - 2;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (u < units && gy >= 0 && gy < L.Y && gx >= 0 && gx < L.X) {
      const int64_t n = tok0 + static_cast<int64_t>(gy) * L.X + gx;
      val = *reinterpret_cast<const uint4*>(L.v + b * L.vsb + n * L.vsn + unit_offset(c0 + 8 * u, L.d, L.vsh));
    }
    *reinterpret_cast<uint4*>(planes + u * kLpPlane + pos * 16) = val;
  }
  __syncthreads();

  const int u = tid % kLpUnits, rest = tid / kLpUnits;
  const int y = rest % kLpTY, s = rest / kLpTY;   // output row, 8-token strip
  const int gy = y0 + y;
  if (u >= units || gy >= L.Y) return;
  const int xs = x0 + s * 8;
  const int nx = min(8, L.X - xs);                // tokens of the strip inside the frame
  if (nx <= 0) return;
  __nv_bfloat16* obase = L.o + b * L.osb + unit_offset(c0 + 8 * u, L.d, L.osh);
  const int64_t nrow = tok0 + static_cast<int64_t>(gy) * L.X + xs;
  uint4 ov[8];
#pragma unroll
  for (int x = 0; x < 8; ++x)
    ov[x] = x < nx ? *reinterpret_cast<const uint4*>(obase + (nrow + x) * L.osn) : make_uint4(0u, 0u, 0u, 0u);
  const uint8_t* pl = planes + u * kLpPlane;
#pragma unroll
  for (int p = 0; p < 4; ++p) {                   // channels 8u + 2p, 8u + 2p + 1
    const int ch = 8 * u + 2 * p;
    uint64_t acc[8];
    const uint64_t bias2 = pack_f2(bsm[ch], bsm[ch + 1]);
#pragma unroll
    for (int x = 0; x < 8; ++x) acc[x] = bias2;
#pragma unroll 1
    for (int i = 0; i < 5; ++i) {
      uint64_t vv[12];
#pragma unroll
      for (int c = 0; c < 12; ++c)
        vv[c] = bf2_to_f2(*reinterpret_cast<const uint32_t*>(pl + ((y + i) * kLpHX + s * 8 + c) * 16 + p * 4));
#pragma unroll
      for (int j = 0; j < 5; ++j) {
        const uint64_t w2 = *reinterpret_cast<const uint64_t*>(wsm + (i * 5 + j) * 64 + ch);
#pragma unroll
        for (int x = 0; x < 8; ++x) acc[x] = fma2(w2, vv[x + j], acc[x]);
      }
    }
    // o + (bias + conv), rounded once
#pragma unroll
    for (int x = 0; x < 8; ++x) {
      uint32_t* wd = reinterpret_cast<uint32_t*>(&ov[x]) + p;
      const __nv_bfloat162 o2 = *reinterpret_cast<const __nv_bfloat162*>(wd);
      const float lo = __low2float(o2) + __uint_as_float(static_cast<uint32_t>(acc[x]));
      const float hi = __high2float(o2) + __uint_as_float(static_cast<uint32_t>(acc[x] >> 32));
      const __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
      *wd = *reinterpret_cast<const uint32_t*>(&r);
    }
  }
#pragma unroll
  for (int x = 0; x < 8; ++x)
    if (x < nx) *reinterpret_cast<uint4*>(obase + (nrow + x) * L.osn) = ov[x];
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
  cublasLtHandle_t handle = nullptr;
  bool ok = false;
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
    if (!all) return;
    api.ok = api.create(&api.handle) == CUBLAS_STATUS_SUCCESS;
  });
  return api;
}

constexpr size_t kLtWorkspace = size_t{32} << 20;

// y[rows][n_out] = x[rows][k] W^T (+ bias[n_out]), W [n_out][k], all bf16 and
// row-major, float32 accumulation.  In cuBLASLt's column-major terms:
// y^T (n_out x rows) = op_T(W stored k x n_out) * x^T (k x rows).
int linear_bf16(const char* name, const void* x, const void* W, const void* bias, void* y, int64_t rows, int64_t k,
                int64_t n_out, void* lt_ws, cudaStream_t stream) {
  const LtApi& lt = lt_api();
  if (!lt.ok) return MHLA_ERR_UNSUPPORTED;
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
    if (lt.heuristic(lt.handle, op, la, lb, lc, lc, pref, 1, &res, &found) != CUBLAS_STATUS_SUCCESS || found < 1) {
      rc = MHLA_ERR_UNSUPPORTED;
      break;
    }
    const float alpha = 1.0f, beta = 0.0f;
    KernelTimer timer(name, stream);
    if (lt.matmul(lt.handle, op, &alpha, W, la, x, lb, &beta, y, lc, y, lc, &res.algo, lt_ws, kLtWorkspace, stream) !=
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
  LpView L;
  L.v = static_cast<const __nv_bfloat16*>(a.v);
  L.o = static_cast<__nv_bfloat16*>(a.o);
  L.vsb = a.vsb; L.vsn = a.vsn; L.vsh = a.vsh;
  L.osb = a.osb; L.osn = a.osn; L.osh = a.osh;
  L.d = a.d; L.C = a.C; L.T = a.T; L.Y = a.Y; L.X = a.X;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(mhla_lepe_add, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kLpSmem)) !=
        cudaSuccess)
      return MHLA_ERR_CUDA;
    attr = true;
  }
  const int64_t nchunks = (a.C + 63) / 64;
  const dim3 grid(static_cast<unsigned>((a.X + kLpTX - 1) / kLpTX), static_cast<unsigned>((a.Y + kLpTY - 1) / kLpTY),
                  static_cast<unsigned>(a.B * a.T * nchunks));
  KernelTimer timer("mhla_lepe_add", stream);
  mhla_lepe_add<<<grid, kLpThreads, kLpSmem, static_cast<cudaStream_t>(stream)>>>(L, a.weight, a.bias);
  return cudaGetLastError() == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
}

int launch_linear(const char* name, const void* x, const void* W, const void* bias, void* y, int64_t rows, int64_t k,
                  int64_t n_out, void* lt_ws, void* stream) {
  return linear_bf16(name, x, W, bias, y, rows, k, n_out, lt_ws, static_cast<cudaStream_t>(stream));
}

bool linear_available() { return lt_api().ok; }

size_t linear_workspace_bytes() { return kLtWorkspace; }

}  // namespace mhla
