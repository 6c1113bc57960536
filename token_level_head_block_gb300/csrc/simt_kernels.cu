// CUDA-core path of the MHLA forward: any d <= 128, any block shape, bf16 or
// float32 inputs, float32 arithmetic throughout.
//
// Three kernels, the three steps of the method ([P2] "MHLA: Restoring
// Expressivity of Linear Attention via Token-Level Multi-Head", section 4;
// [P1] 171host.com/767426.html, section 7, MHLA.forward):
//   simt_summary  S_j = phi(K_j)^T V_j and z_j = sum phi(k) per (b, h, block j)
//   simt_mix      S~_i = sum_j W[i][j] S_j and z~_i likewise, per (b, h)
//   simt_output   o_t = phi(q_t) S~_i / (phi(q_t) . z~_i + eps)
// Workspace: two float32 buffers [BH][M][d*(d+1)] (S_j row-major, then z_j).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "mhla_internal.h"

namespace mhla {
namespace {

__device__ __forceinline__ float load_f(const float* p) { return __ldg(p); }
__device__ __forceinline__ float load_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void store_f(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_f(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ float phi_f(float x, int kind, float eps) {
  const float r = fmaxf(x, 0.0f);
  return kind == MHLA_PHI_RELU_EPS ? r + eps : r;
}

// Token index n of in-block slot s of block j.
__device__ __forceinline__ int64_t token_of(const TokenGeom& g, int64_t j, int64_t s) {
  const int64_t jx = j % g.nbx, jr = j / g.nbx;
  const int64_t jy = jr % g.nby, jt = jr / g.nby;
  const int64_t sx = s % g.bx, sr = s / g.bx;
  const int64_t sy = sr % g.by, st = sr / g.by;
  const int64_t t = jt * g.bt + st, y = jy * g.by + sy, x = jx * g.bx + sx;
  return (t * g.Y + y) * g.X + x;
}

constexpr int kSumThreads = 256;
constexpr int kSumChunk = 32;   // tokens staged in shared memory per step

// One CTA per (b, h, j).  ENT = ceil(d*d / 256) accumulators per thread.
template <typename T, int ENT>
__global__ void __launch_bounds__(kSumThreads)
simt_summary(const T* __restrict__ k, const T* __restrict__ v, Operand ko, Operand vo, TokenGeom g,
             int64_t H, int d, int phi_kind, float eps, float* __restrict__ Sz) {
  extern __shared__ float sm[];
  float* sk = sm;                    // [kSumChunk][d]  phi(k)
  float* sv = sm + kSumChunk * d;    // [kSumChunk][d]  v
  const int64_t item = blockIdx.x;
  const int64_t j = item % g.M, bh = item / g.M;
  const int64_t b = bh / H, h = bh % H;
  const int tid = threadIdx.x;
  const int E = d * d;
  const T* kb = k + b * ko.sb + h * ko.sh;
  const T* vb = v + b * vo.sb + h * vo.sh;

  float acc[ENT];
#pragma unroll
  for (int m = 0; m < ENT; ++m) acc[m] = 0.0f;
  float zacc = 0.0f;

  for (int64_t s0 = 0; s0 < g.w; s0 += kSumChunk) {
    const int cnt = static_cast<int>(g.w - s0 < kSumChunk ? g.w - s0 : kSumChunk);
    for (int e = tid; e < cnt * d; e += kSumThreads) {
      const int sl = e / d, c = e % d;
      const int64_t n = token_of(g, j, s0 + sl);
      sk[sl * d + c] = phi_f(load_f(kb + n * ko.sn + c), phi_kind, eps);
      sv[sl * d + c] = load_f(vb + n * vo.sn + c);
    }
    __syncthreads();
#pragma unroll
    for (int m = 0; m < ENT; ++m) {
      const int e = tid + m * kSumThreads;
      if (e < E) {
        const int r = e / d, c = e % d;
        float a = acc[m];
        for (int sl = 0; sl < cnt; ++sl) a = fmaf(sk[sl * d + r], sv[sl * d + c], a);
        acc[m] = a;
      }
    }
    if (tid < d)
      for (int sl = 0; sl < cnt; ++sl) zacc += sk[sl * d + tid];
    __syncthreads();
  }
  float* out = Sz + (bh * g.M + j) * static_cast<int64_t>(E + d);
#pragma unroll
  for (int m = 0; m < ENT; ++m) {
    const int e = tid + m * kSumThreads;
    if (e < E) out[e] = acc[m];
  }
  if (tid < d) out[E + tid] = zacc;
}

constexpr int kMixThreads = 128;
constexpr int kMixRows = 8;     // query blocks i per thread

// S~ = W . S per (b, h), treating the d*(d+1) entries of every block as columns.
__global__ void __launch_bounds__(kMixThreads)
simt_mix(const float* __restrict__ W, const float* __restrict__ Sz, float* __restrict__ Szt,
         int64_t M, int64_t E, int64_t BH) {
  const int64_t e = static_cast<int64_t>(blockIdx.x) * kMixThreads + threadIdx.x;
  const int64_t i0 = static_cast<int64_t>(blockIdx.y) * kMixRows;
  if (e >= E) return;
  for (int64_t bh = blockIdx.z; bh < BH; bh += gridDim.z) {
    float acc[kMixRows];
#pragma unroll
    for (int u = 0; u < kMixRows; ++u) acc[u] = 0.0f;
    const float* src = Sz + bh * M * E + e;
    for (int64_t j = 0; j < M; ++j) {
      const float s = src[j * E];
#pragma unroll
      for (int u = 0; u < kMixRows; ++u)
        if (i0 + u < M) acc[u] = fmaf(__ldg(W + (i0 + u) * M + j), s, acc[u]);
    }
#pragma unroll
    for (int u = 0; u < kMixRows; ++u)
      if (i0 + u < M) Szt[(bh * M + i0 + u) * E + e] = acc[u];
  }
}

constexpr int kOutThreads = 256;
constexpr int kOutWarps = kOutThreads / 32;

// One CTA per (b, h, i): S~_i and z~_i in shared memory, one warp per token.
template <typename T>
__global__ void __launch_bounds__(kOutThreads)
simt_output(const T* __restrict__ q, Operand qo, T* __restrict__ o, Operand oo, TokenGeom g,
            int64_t H, int d, int phi_kind, float eps, const float* __restrict__ Szt) {
  extern __shared__ float sm[];
  const int E = d * d;
  float* st = sm;                          // [d][d] S~_i
  float* zt = sm + E;                      // [d]    z~_i
  float* qrow = sm + E + d;                // [kOutWarps][d] phi(q_t)
  const int64_t item = blockIdx.x;
  const int64_t i = item % g.M, bh = item / g.M;
  const int64_t b = bh / H, h = bh % H;
  const float* src = Szt + (bh * g.M + i) * static_cast<int64_t>(E + d);
  for (int e = threadIdx.x; e < E + d; e += kOutThreads) sm[e] = src[e];
  __syncthreads();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  float* myq = qrow + warp * d;
  const T* qb = q + b * qo.sb + h * qo.sh;
  T* ob = o + b * oo.sb + h * oo.sh;
  for (int64_t s = warp; s < g.w; s += kOutWarps) {
    const int64_t n = token_of(g, i, s);
    float den = 0.0f;
    for (int r = lane; r < d; r += 32) {
      const float x = phi_f(load_f(qb + n * qo.sn + r), phi_kind, eps);
      myq[r] = x;
      den = fmaf(x, zt[r], den);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
    __syncwarp();
    const float denom = den + eps;
    for (int c = lane; c < d; c += 32) {
      float num = 0.0f;
      for (int r = 0; r < d; ++r) num = fmaf(myq[r], st[r * d + c], num);
      store_f(ob + n * oo.sn + c, num / denom);
    }
    __syncwarp();
  }
}

template <typename T>
int launch_simt_typed(const Problem& p, const float* W, const SimtWorkspace& ws, cudaStream_t stream) {
  const TokenGeom g = token_geom(p);
  const int d = static_cast<int>(p.d);
  const int64_t BH = p.BH();
  const int64_t items = BH * p.M;
  if (items > 0x7fffffffLL) return MHLA_ERR_UNSUPPORTED;
  const size_t sum_smem = 2 * kSumChunk * d * sizeof(float);
  const T* qp = static_cast<const T*>(p.q.data);
  const T* kp = static_cast<const T*>(p.k.data);
  const T* vp = static_cast<const T*>(p.v.data);
  T* op = static_cast<T*>(p.o.data);
  {
    KernelTimer timer("simt_summary", stream);
    if (d <= 16)
      simt_summary<T, 1><<<static_cast<unsigned>(items), kSumThreads, sum_smem, stream>>>(
          kp, vp, p.k, p.v, g, p.H, d, p.phi_kind, p.eps, ws.Sz);
    else if (d <= 32)
      simt_summary<T, 4><<<static_cast<unsigned>(items), kSumThreads, sum_smem, stream>>>(
          kp, vp, p.k, p.v, g, p.H, d, p.phi_kind, p.eps, ws.Sz);
    else if (d <= 64)
      simt_summary<T, 16><<<static_cast<unsigned>(items), kSumThreads, sum_smem, stream>>>(
          kp, vp, p.k, p.v, g, p.H, d, p.phi_kind, p.eps, ws.Sz);
    else
      simt_summary<T, 64><<<static_cast<unsigned>(items), kSumThreads, sum_smem, stream>>>(
          kp, vp, p.k, p.v, g, p.H, d, p.phi_kind, p.eps, ws.Sz);
    if (cudaGetLastError() != cudaSuccess) return MHLA_ERR_CUDA;
  }

  const int64_t E = p.d * (p.d + 1);
  const dim3 mix_grid(static_cast<unsigned>((E + kMixThreads - 1) / kMixThreads),
                      static_cast<unsigned>((p.M + kMixRows - 1) / kMixRows),
                      static_cast<unsigned>(std::min<int64_t>(BH, 65535)));
  if (mix_grid.y > 65535) return MHLA_ERR_UNSUPPORTED;
  {
    KernelTimer timer("simt_mix", stream);
    simt_mix<<<mix_grid, kMixThreads, 0, stream>>>(W, ws.Sz, ws.Szt, p.M, E, BH);
    if (cudaGetLastError() != cudaSuccess) return MHLA_ERR_CUDA;
  }

  const size_t out_smem = (E + p.d + kOutWarps * p.d) * sizeof(float);
  if (out_smem > 48 * 1024) {
    if (cudaFuncSetAttribute(simt_output<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(out_smem)) != cudaSuccess)
      return MHLA_ERR_CUDA;
  }
  {
    KernelTimer timer("simt_output", stream);
    simt_output<T><<<static_cast<unsigned>(items), kOutThreads, out_smem, stream>>>(
        qp, p.q, op, p.o, g, p.H, d, p.phi_kind, p.eps, ws.Szt);
    if (cudaGetLastError() != cudaSuccess) return MHLA_ERR_CUDA;
  }
  return MHLA_OK;
}

}  // namespace

size_t simt_workspace_bytes(const Problem& p) {
  const size_t per = static_cast<size_t>(p.BH()) * p.M * p.d * (p.d + 1) * sizeof(float);
  return 2 * align_up(per);
}

SimtWorkspace simt_carve(const Problem& p, void* base) {
  const size_t per = static_cast<size_t>(p.BH()) * p.M * p.d * (p.d + 1) * sizeof(float);
  char* c = static_cast<char*>(base);
  return SimtWorkspace{reinterpret_cast<float*>(c), reinterpret_cast<float*>(c + align_up(per))};
}

int launch_simt(const Problem& p, const float* W, void* workspace, void* stream) {
  const SimtWorkspace ws = simt_carve(p, workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.dtype == MHLA_BF16) return launch_simt_typed<__nv_bfloat16>(p, W, ws, s);
  return launch_simt_typed<float>(p, W, ws, s);
}

}  // namespace mhla
