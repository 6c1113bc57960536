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
// The backward pass (below) reuses the summary and mixing kernels.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <type_traits>

#include "mhla_internal.h"

namespace mhla {
namespace {

__device__ __forceinline__ float load_f(const float* p) { return __ldg(p); }
__device__ __forceinline__ float load_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void store_f(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_f(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// Asynchronous 4-byte global -> shared copies (any alignment); a copy with
// full = false reads nothing and writes zero.  wait<N> returns once at most N
// of this thread's committed groups are still in flight.
__device__ __forceinline__ void cp_async_f32(float* dst, const float* src, bool full) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src), "r"(full ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

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
constexpr int kSumLanes = kSumThreads / kSumChunk;   // threads staging one token row

// One CTA per (b, h, j).  Thread (ty, tx) = (tid / 16, tid % 16) accumulates
// the TB x TB tile of S_j at rows TB ty.., columns TB tx.. (16 TB >= d): per
// token, TB values of phi(k) and TB of v feed TB * TB products.  Every entry
// sums its tokens in slot order.
template <typename T, int TB>
__global__ void __launch_bounds__(kSumThreads)
simt_summary(const T* __restrict__ k, const T* __restrict__ v, Operand ko, Operand vo, TokenGeom g,
             int64_t H, int d, int phi_kind, float eps, float* __restrict__ Sz) {
  extern __shared__ __align__(16) float sum_sm[];
  float* sk = sum_sm;                    // [kSumChunk][d]  phi(k)
  float* sv = sum_sm + kSumChunk * d;    // [kSumChunk][d]  v, then 16 TB floats of slack
  const int64_t item = blockIdx.x;
  const int64_t j = item % g.M, bh = item / g.M;
  const int64_t b = bh / H, h = bh % H;
  const int tid = threadIdx.x;
  const int E = d * d;
  const T* kb = k + b * ko.sb + h * ko.sh;
  const T* vb = v + b * vo.sb + h * vo.sh;
  const int r0 = TB * (tid / 16), c0 = TB * (tid % 16);
  const int srow = tid / kSumLanes, spart = tid % kSumLanes;

  float acc[TB * TB];
#pragma unroll
  for (int m = 0; m < TB * TB; ++m) acc[m] = 0.0f;
  float zacc = 0.0f;

  for (int64_t s0 = 0; s0 < g.w; s0 += kSumChunk) {
    const int cnt = static_cast<int>(g.w - s0 < kSumChunk ? g.w - s0 : kSumChunk);
    if (srow < cnt) {
      const int64_t n = token_of(g, j, s0 + srow);
      for (int c = spart; c < d; c += kSumLanes) {
        sk[srow * d + c] = phi_f(load_f(kb + n * ko.sn + c), phi_kind, eps);
        sv[srow * d + c] = load_f(vb + n * vo.sn + c);
      }
    }
    __syncthreads();
    auto scalar_steps = [&]() {
      for (int sl = 0; sl < cnt; ++sl) {
        float kr[TB], vc[TB];
#pragma unroll
        for (int u = 0; u < TB; ++u) {
          kr[u] = sk[sl * d + r0 + u];
          vc[u] = sv[sl * d + c0 + u];
        }
#pragma unroll
        for (int u = 0; u < TB; ++u)
#pragma unroll
          for (int w = 0; w < TB; ++w) acc[u * TB + w] = fmaf(kr[u], vc[w], acc[u * TB + w]);
      }
    };
    if constexpr (TB % 4 == 0) {
      if (d % 4 == 0) {
        for (int sl = 0; sl < cnt; ++sl) {
          float kr[TB], vc[TB];
#pragma unroll
          for (int u = 0; u < TB; u += 4) {
            const float4 a = *reinterpret_cast<const float4*>(sk + sl * d + r0 + u);
            const float4 c = *reinterpret_cast<const float4*>(sv + sl * d + c0 + u);
            kr[u] = a.x, kr[u + 1] = a.y, kr[u + 2] = a.z, kr[u + 3] = a.w;
            vc[u] = c.x, vc[u + 1] = c.y, vc[u + 2] = c.z, vc[u + 3] = c.w;
          }
#pragma unroll
          for (int u = 0; u < TB; ++u)
#pragma unroll
            for (int w = 0; w < TB; ++w) acc[u * TB + w] = fmaf(kr[u], vc[w], acc[u * TB + w]);
        }
      } else {
        scalar_steps();
      }
    } else {
      scalar_steps();
    }
    if (tid < d)
      for (int sl = 0; sl < cnt; ++sl) zacc += sk[sl * d + tid];
    __syncthreads();
  }
  float* out = Sz + (bh * g.M + j) * static_cast<int64_t>(E + d);
#pragma unroll
  for (int m = 0; m < TB * TB; ++m) {
    const int r = r0 + m / TB, c = c0 + m % TB;
    if (r < d && c < d) out[r * d + c] = acc[m];
  }
  if (tid < d) out[E + tid] = zacc;
}

// S_j, z_j of every (b, h, j) into Sz.
template <typename T>
int launch_summary(const Problem& p, const TokenGeom& g, float* Sz, cudaStream_t stream) {
  const int d = static_cast<int>(p.d);
  const int64_t items = p.BH() * p.M;
  const size_t smem = (2 * kSumChunk * d + 16 * 8) * sizeof(float);
  const T* kp = static_cast<const T*>(p.k.data);
  const T* vp = static_cast<const T*>(p.v.data);
  auto launch = [&](auto kern) -> int {
    KernelTimer timer("simt_summary", stream);
    kern<<<static_cast<unsigned>(items), kSumThreads, smem, stream>>>(kp, vp, p.k, p.v, g, p.H, d, p.phi_kind,
                                                                      p.eps, Sz);
    return cudaGetLastError() == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
  };
  return d <= 16   ? launch(simt_summary<T, 1>)
         : d <= 32 ? launch(simt_summary<T, 2>)
         : d <= 64 ? launch(simt_summary<T, 4>)
                   : launch(simt_summary<T, 8>);
}

constexpr int kMixThreads = 256;
constexpr int kMixTileI = 64;    // output blocks per CTA, 8 per warp
constexpr int kMixTileE = 128;   // entries per CTA, 4 per lane (stride 32)
constexpr int kMixK = 16;        // source blocks per slab
constexpr int kMixStages = 3;    // slabs in flight (within 48 KB of shared memory)
constexpr int kMixWRow = kMixTileI + 4;
constexpr int kMixStage = kMixK * kMixWRow + kMixK * kMixTileE;   // floats per stage
constexpr size_t kMixSmem = static_cast<size_t>(kMixStages) * kMixStage * sizeof(float);

// S~ = W . S per (b, h), treating the d*(d+1) entries of every block as columns
// (TRANS: W^T . S, the mixing step of the backward pass).
// (PAST: only source blocks j < i, the mixed past summaries of causal MHLA;
// with TRANS, only i > j: the reverse of that mixing in the causal backward.)
// A CTA holds a 64-block x 128-entry tile of the output; W's 64 x 16 slabs and
// the sources' 16 x 128 slabs go through shared memory in a three-stage cp.async
// ring, and each thread keeps 8 x 4 sums.  Every output sums its sources in
// ascending order, skipping the ones that PAST excludes.
template <bool TRANS, bool PAST = false>
__global__ void __launch_bounds__(kMixThreads)
simt_mix(const float* __restrict__ W, const float* __restrict__ Sz, float* __restrict__ Szt,
         int64_t M, int64_t E, int64_t BH) {
  extern __shared__ __align__(16) float mix_sm[];   // [stage]: W slab [jj][kMixWRow], then source slab [jj][128]
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int64_t e0 = static_cast<int64_t>(blockIdx.x) * kMixTileE;
  const int64_t i0 = static_cast<int64_t>(blockIdx.y) * kMixTileI;
  const int64_t ia = i0 + 8 * warp;   // this warp's first output block
  // sources that reach some row of the tile
  const int64_t jb = PAST && TRANS ? i0 + 1 : 0;
  const int64_t je = PAST && !TRANS ? std::min<int64_t>(M, i0 + kMixTileI - 1) : M;
  const int64_t nslab = je > jb ? (je - jb + kMixK - 1) / kMixK : 0;
  for (int64_t bh = blockIdx.z; bh < BH; bh += gridDim.z) {
    const float* src = Sz + bh * M * E;
    // slab n into stage n % kMixStages (nothing past the last slab; the commit
    // keeps one group per slot either way)
    auto stage = [&](int64_t n) {
      if (n < nslab) {
        float* ws = mix_sm + (n % kMixStages) * kMixStage;
        float* ss = ws + kMixK * kMixWRow;
        const int64_t j0 = jb + n * kMixK;
        for (int x = tid; x < kMixK * kMixTileI; x += kMixThreads) {
          const int jj = TRANS ? x / kMixTileI : x % kMixK;
          const int r = TRANS ? x % kMixTileI : x / kMixK;
          const int64_t i = i0 + r, j = j0 + jj;
          const bool in = i < M && j < je;
          cp_async_f32(ws + jj * kMixWRow + r, in ? (TRANS ? W + j * M + i : W + i * M + j) : W, in);
        }
        for (int x = tid; x < kMixK * kMixTileE; x += kMixThreads) {
          const int jj = x / kMixTileE, c = x % kMixTileE;
          const int64_t j = j0 + jj, e = e0 + c;
          const bool in = j < je && e < E;
          cp_async_f32(ss + jj * kMixTileE + c, in ? src + j * E + e : src, in);
        }
      }
      cp_async_commit();
    };
    float acc[8][4];
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int w = 0; w < 4; ++w) acc[u][w] = 0.0f;
    __syncthreads();   // the previous (b, h) has finished with every stage
#pragma unroll
    for (int n = 0; n < kMixStages - 1; ++n) stage(n);
    for (int64_t n = 0; n < nslab; ++n) {
      cp_async_wait<kMixStages - 2>();   // slab n has landed (this thread's copies)
      __syncthreads();                   // everyone's copies, and slab n - 1's stage is free
      stage(n + kMixStages - 1);
      const float* ws = mix_sm + (n % kMixStages) * kMixStage;
      const float* ss = ws + kMixK * kMixWRow;
      const int64_t j0 = jb + n * kMixK;
      const int cnt = static_cast<int>(je - j0 < kMixK ? je - j0 : kMixK);
      for (int jj = 0; jj < cnt; ++jj) {
        const int64_t j = j0 + jj;
        const float4 wa = *reinterpret_cast<const float4*>(ws + jj * kMixWRow + 8 * warp);
        const float4 wb = *reinterpret_cast<const float4*>(ws + jj * kMixWRow + 8 * warp + 4);
        const float wr[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
        float sc[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) sc[w] = ss[jj * kMixTileE + lane + 32 * w];
        if (!PAST || (TRANS ? j > ia + 7 : j < ia)) {
#pragma unroll
          for (int u = 0; u < 8; ++u)
#pragma unroll
            for (int w = 0; w < 4; ++w) acc[u][w] = fmaf(wr[u], sc[w], acc[u][w]);
        } else if (TRANS ? j > ia : j < ia + 7) {
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (TRANS ? j > ia + u : j < ia + u)
#pragma unroll
              for (int w = 0; w < 4; ++w) acc[u][w] = fmaf(wr[u], sc[w], acc[u][w]);
        }
      }
    }
    cp_async_wait<0>();   // only empty groups remain; nothing may land after the next (b, h) starts
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const int64_t i = ia + u, e = e0 + lane + 32 * w;
        if (i < M && e < E) Szt[(bh * M + i) * E + e] = acc[u][w];
      }
  }
}

// dst = W . src (TRANS: W^T . src), PAST as simt_mix, per (b, h).
template <bool TRANS, bool PAST>
int launch_mix(const float* W, const float* src, float* dst, int64_t M, int64_t E, int64_t BH,
               cudaStream_t stream) {
  const int64_t gx = (E + kMixTileE - 1) / kMixTileE, gy = (M + kMixTileI - 1) / kMixTileI;
  if (gx > 0x7fffffffLL || gy > 65535) return MHLA_ERR_UNSUPPORTED;
  const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy),
                  static_cast<unsigned>(std::min<int64_t>(BH, 65535)));
  static_assert(kMixSmem <= 48 * 1024, "no opt-in attribute needed");
  KernelTimer timer("simt_mix", stream);
  simt_mix<TRANS, PAST><<<grid, kMixThreads, kMixSmem, stream>>>(W, src, dst, M, E, BH);
  return cudaGetLastError() == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
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

// ============================================================================
// Causal MHLA ([P2] "MHLA: Restoring Expressivity of Linear Attention via
// Token-Level Multi-Head", App. B "Causal MHLA": block-specific mixed summaries,
// causal, at the cost of chunkwise linear attention).  Blocks are contiguous
// token ranges; for token t of query block i
//   o_t = phi(q_t) (S<_i + W[i][i] P_t) / (phi(q_t) . (z<_i + W[i][i] y_t) + eps)
// with S<_i = sum_{j < i} W[i][j] S_j (simt_mix<false, true>) and P_t, y_t the
// running sums of phi(k_s) v_s^T, phi(k_s) over the block's tokens s <= t.
// simt_causal_output walks the block in chunks of kCausalChunk tokens: the
// running state starts at S<_i, z<_i; inside a chunk each token adds the
// W[i][i]-weighted causal scores against the chunk's earlier tokens, then the
// state absorbs W[i][i] times the chunk's summary.
// ============================================================================
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

constexpr int kCausalThreads = 256;
constexpr int kCausalWarps = kCausalThreads / 32;
constexpr int kCausalChunk = 32;   // one key per lane in the score step

template <typename T, int ENT>
__global__ void __launch_bounds__(kCausalThreads)
simt_causal_output(const T* __restrict__ q, Operand qo, const T* __restrict__ k, Operand ko,
                   const T* __restrict__ v, Operand vo, T* __restrict__ o, Operand oo, TokenGeom g, int64_t H, int d,
                   int phi_kind, float eps, const float* __restrict__ W, const float* __restrict__ Szt) {
  extern __shared__ float sm[];
  const int E = d * d, P = d + 1;
  float* st = sm;                          // [d][d] running state S<_i + W_ii P
  float* zs = st + E;                      // [d]    running z<_i + W_ii y
  float* sq = zs + d;                      // [chunk][d]     phi(q)
  float* sk = sq + kCausalChunk * d;       // [chunk][d + 1] phi(k), rows padded (lanes walk keys)
  float* sv = sk + kCausalChunk * P;       // [chunk][d]     v
  float* sa = sv + kCausalChunk * d;       // [warps][chunk] causal scores of the warp's token
  const int64_t item = blockIdx.x;
  const int64_t i = item % g.M, bh = item / g.M;
  const int64_t b = bh / H, h = bh % H;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const float wii = __ldg(W + i * g.M + i);
  const float* src = Szt + (bh * g.M + i) * static_cast<int64_t>(E + d);
  for (int e = tid; e < E + d; e += kCausalThreads) sm[e] = src[e];
  const T* qb = q + b * qo.sb + h * qo.sh;
  const T* kb = k + b * ko.sb + h * ko.sh;
  const T* vb = v + b * vo.sb + h * vo.sh;
  T* ob = o + b * oo.sb + h * oo.sh;
  for (int64_t s0 = 0; s0 < g.w; s0 += kCausalChunk) {
    const int cnt = static_cast<int>(g.w - s0 < kCausalChunk ? g.w - s0 : kCausalChunk);
    __syncthreads();   // the state is complete (and the previous chunk's rows are free)
    for (int e = tid; e < cnt * d; e += kCausalThreads) {
      const int sl = e / d, c = e % d;
      const int64_t n = token_of(g, i, s0 + sl);   // contiguous blocks: n increases with s
      sq[sl * d + c] = phi_f(load_f(qb + n * qo.sn + c), phi_kind, eps);
      sk[sl * P + c] = phi_f(load_f(kb + n * ko.sn + c), phi_kind, eps);
      sv[sl * d + c] = load_f(vb + n * vo.sn + c);
    }
    __syncthreads();
    for (int sl = warp; sl < cnt; sl += kCausalWarps) {
      const float* myq = sq + sl * d;
      // lane = key s of the chunk: a_s = W_ii phi(q_t) . phi(k_s) for s <= t
      float a = 0.0f;
      if (lane <= sl) {
        for (int r = 0; r < d; ++r) a = fmaf(myq[r], sk[lane * P + r], a);
        a *= wii;
      }
      float* mya = sa + warp * kCausalChunk;
      mya[lane] = a;
      float den = 0.0f;
      for (int r = lane; r < d; r += 32) den = fmaf(myq[r], zs[r], den);
      den = warp_sum(den + a) + eps;
      __syncwarp();
      const int64_t n = token_of(g, i, s0 + sl);
      for (int c = lane; c < d; c += 32) {
        float num = 0.0f;
        for (int r = 0; r < d; ++r) num = fmaf(myq[r], st[r * d + c], num);
        for (int s2 = 0; s2 <= sl; ++s2) num = fmaf(mya[s2], sv[s2 * d + c], num);
        store_f(ob + n * oo.sn + c, num / den);
      }
      __syncwarp();
    }
    __syncthreads();
    // state += W_ii * (the chunk's summary)
#pragma unroll
    for (int m = 0; m < ENT; ++m) {
      const int e = tid + m * kCausalThreads;
      if (e < E) {
        const int r = e / d, c = e % d;
        float acc = 0.0f;
        for (int sl = 0; sl < cnt; ++sl) acc = fmaf(sk[sl * P + r], sv[sl * d + c], acc);
        st[e] = fmaf(wii, acc, st[e]);
      }
    }
    if (tid < d) {
      float acc = 0.0f;
      for (int sl = 0; sl < cnt; ++sl) acc += sk[sl * P + tid];
      zs[tid] = fmaf(wii, acc, zs[tid]);
    }
  }
}

// ============================================================================
// Backward pass.  The pages print none; these kernels follow the chain rule
// through the three forward steps in reverse (the derivation is in the
// header, next to mhla_backward):
//   simt_bwd_query  per (b, h, query block i): dq, dS~_i = sum_t phi(q_t) dnum_t^T,
//                   dz~_i = sum_t dden_t phi(q_t), with dnum_t = g_t / den_t and
//                   dden_t = -(g_t . o_t) / den_t recomputed from S~_i, z~_i
//   simt_mix<true>  dS_j = sum_i W[i][j] dS~_i, dz_j likewise
//   simt_dw_*       dW[i][j] = sum_{b,h} <dS~_i, S_j> + dz~_i . z_j
//   simt_bwd_key    per (b, h, source block j): dv_s = dS_j^T phi(k_s),
//                   dk_s = (dS_j v_s + dz_j) * [k_s > 0]
// ============================================================================
constexpr int kBwdThreads = 256;
constexpr int kBwdWarps = kBwdThreads / 32;
constexpr int kBwdChunk = 32;   // tokens staged per accumulation step

// One CTA per (b, h, i).  S~_i in shared memory with rows padded to d + 1 so
// that lanes walking a column and lanes walking a row both avoid bank conflicts.
template <typename T, int ENT>
__global__ void __launch_bounds__(kBwdThreads)
simt_bwd_query(const T* __restrict__ q, Operand qo, const T* __restrict__ g_out, Operand go, T* __restrict__ dq,
               Operand dqo, TokenGeom g, int64_t H, int d, int phi_kind, float eps, const float* __restrict__ Szt,
               float* __restrict__ dSzt) {
  extern __shared__ float sm[];
  const int E = d * d, P = d + 1;
  float* st = sm;                          // [d][d + 1] S~_i
  float* zt = st + d * P;                  // [d]        z~_i
  float* sq = zt + d;                      // [kBwdChunk][d] phi(q_t)
  float* sdn = sq + kBwdChunk * d;         // [kBwdChunk][d] dnum_t
  float* sdd = sdn + kBwdChunk * d;        // [kBwdChunk]    dden_t
  const int64_t item = blockIdx.x;
  const int64_t i = item % g.M, bh = item / g.M;
  const int64_t b = bh / H, h = bh % H;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const float* src = Szt + (bh * g.M + i) * static_cast<int64_t>(E + d);
  for (int e = tid; e < E; e += kBwdThreads) st[(e / d) * P + e % d] = src[e];
  for (int r = tid; r < d; r += kBwdThreads) zt[r] = src[E + r];
  const T* qb = q + b * qo.sb + h * qo.sh;
  const T* gb = g_out + b * go.sb + h * go.sh;
  T* dqb = dq + b * dqo.sb + h * dqo.sh;

  float acc[ENT];
#pragma unroll
  for (int m = 0; m < ENT; ++m) acc[m] = 0.0f;
  float zacc = 0.0f;
  __syncthreads();

  for (int64_t s0 = 0; s0 < g.w; s0 += kBwdChunk) {
    const int cnt = static_cast<int>(g.w - s0 < kBwdChunk ? g.w - s0 : kBwdChunk);
    for (int sl = warp; sl < cnt; sl += kBwdWarps) {
      const int64_t n = token_of(g, i, s0 + sl);
      float* myq = sq + sl * d;
      float* mydn = sdn + sl * d;
      float den = 0.0f;
      for (int r = lane; r < d; r += 32) {
        const float x = phi_f(load_f(qb + n * qo.sn + r), phi_kind, eps);
        myq[r] = x;
        den = fmaf(x, zt[r], den);
      }
      den = warp_sum(den) + eps;
      __syncwarp();
      // num_c = sum_r phi(q)_r S~[r][c];  g . o = sum_c g_c num_c / den
      float go_dot = 0.0f;
      for (int c = lane; c < d; c += 32) {
        float num = 0.0f;
        for (int r = 0; r < d; ++r) num = fmaf(myq[r], st[r * P + c], num);
        const float gc = load_f(gb + n * go.sn + c);
        go_dot = fmaf(gc, num, go_dot);
        mydn[c] = gc / den;
      }
      go_dot = warp_sum(go_dot) / den;
      const float dden = -go_dot / den;
      if (lane == 0) sdd[sl] = dden;
      __syncwarp();
      // dphi(q)_r = sum_c S~[r][c] dnum_c + dden z~_r, masked by phi'
      for (int r = lane; r < d; r += 32) {
        float x = dden * zt[r];
        for (int c = 0; c < d; ++c) x = fmaf(st[r * P + c], mydn[c], x);
        const float qr = load_f(qb + n * qo.sn + r);
        store_f(dqb + n * dqo.sn + r, qr > 0.0f ? x : 0.0f);
      }
    }
    __syncthreads();
#pragma unroll
    for (int m = 0; m < ENT; ++m) {
      const int e = tid + m * kBwdThreads;
      if (e < E) {
        const int r = e / d, c = e % d;
        float a = acc[m];
        for (int sl = 0; sl < cnt; ++sl) a = fmaf(sq[sl * d + r], sdn[sl * d + c], a);
        acc[m] = a;
      }
    }
    if (tid < d)
      for (int sl = 0; sl < cnt; ++sl) zacc = fmaf(sq[sl * d + tid], sdd[sl], zacc);
    __syncthreads();
  }
  float* out = dSzt + (bh * g.M + i) * static_cast<int64_t>(E + d);
#pragma unroll
  for (int m = 0; m < ENT; ++m) {
    const int e = tid + m * kBwdThreads;
    if (e < E) out[e] = acc[m];
  }
  if (tid < d) out[E + tid] = zacc;
}

// One CTA per (b, h, j): dS_j (rows padded to d + 1) and dz_j in shared
// memory, one warp per token.
template <typename T>
__global__ void __launch_bounds__(kBwdThreads)
simt_bwd_key(const T* __restrict__ k, Operand ko, const T* __restrict__ v, Operand vo, T* __restrict__ dk,
             Operand dko, T* __restrict__ dv, Operand dvo, TokenGeom g, int64_t H, int d, int phi_kind, float eps,
             const float* __restrict__ dSz) {
  extern __shared__ float sm[];
  const int E = d * d, P = d + 1;
  float* ds = sm;                          // [d][d + 1] dS_j
  float* dz = ds + d * P;                  // [d]        dz_j
  float* rows = dz + d;                    // [kBwdWarps][2 d] phi(k_s), v_s
  const int64_t item = blockIdx.x;
  const int64_t j = item % g.M, bh = item / g.M;
  const int64_t b = bh / H, h = bh % H;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const float* src = dSz + (bh * g.M + j) * static_cast<int64_t>(E + d);
  for (int e = tid; e < E; e += kBwdThreads) ds[(e / d) * P + e % d] = src[e];
  for (int r = tid; r < d; r += kBwdThreads) dz[r] = src[E + r];
  __syncthreads();
  const T* kb = k + b * ko.sb + h * ko.sh;
  const T* vb = v + b * vo.sb + h * vo.sh;
  T* dkb = dk + b * dko.sb + h * dko.sh;
  T* dvb = dv + b * dvo.sb + h * dvo.sh;
  float* myk = rows + warp * 2 * d;
  float* myv = myk + d;
  for (int64_t s = warp; s < g.w; s += kBwdWarps) {
    const int64_t n = token_of(g, j, s);
    for (int r = lane; r < d; r += 32) {
      myk[r] = phi_f(load_f(kb + n * ko.sn + r), phi_kind, eps);
      myv[r] = load_f(vb + n * vo.sn + r);
    }
    __syncwarp();
    for (int c = lane; c < d; c += 32) {     // dv_c = sum_r phi(k)_r dS[r][c]
      float x = 0.0f;
      for (int r = 0; r < d; ++r) x = fmaf(myk[r], ds[r * P + c], x);
      store_f(dvb + n * dvo.sn + c, x);
    }
    for (int r = lane; r < d; r += 32) {     // dphi(k)_r = sum_c dS[r][c] v_c + dz_r
      float x = dz[r];
      for (int c = 0; c < d; ++c) x = fmaf(ds[r * P + c], myv[c], x);
      const float kr = load_f(kb + n * ko.sn + r);
      store_f(dkb + n * dko.sn + r, kr > 0.0f ? x : 0.0f);
    }
    __syncwarp();
  }
}

constexpr int kDwTile = 64;     // 64 x 64 outputs per CTA, 4 x 4 per thread
constexpr int kDwK = 32;        // entries of the contraction staged per step

// Contraction splits of the dW partial products: about one wave of CTAs at
// four per SM of a 152-SM part, each split at least 256 entries long.
int64_t dw_splits(const Problem& p) {
  const int64_t tiles = (p.M + kDwTile - 1) / kDwTile;
  const int64_t ctas = tiles * tiles * p.BH();
  const int64_t E = p.d * (p.d + 1);
  const int64_t want = 608 / ctas;
  return std::max<int64_t>(1, std::min<int64_t>(want, std::max<int64_t>(1, E / 256)));
}

// part[bh][ks][i][j] = sum over e in split ks of dSzt[bh][i][e] * Sz[bh][j][e]
// (z index = bh * KS + ks; the KS splits of the contraction cut E into equal
// column ranges so that a small M still spreads over many CTAs).  The 32-entry
// slabs of both operands are double-buffered: cp.async fills the next slab
// while the current one is multiplied.
__global__ void __launch_bounds__(256)
simt_dw_partial(const float* __restrict__ dSzt, const float* __restrict__ Sz, float* __restrict__ part, int64_t M,
                int64_t E, int32_t KS) {
  __shared__ __align__(16) float sa[2][kDwK][kDwTile + 4];
  __shared__ __align__(16) float sb[2][kDwK][kDwTile + 4];
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kDwTile, j0 = static_cast<int64_t>(blockIdx.y) * kDwTile;
  const int64_t bh = blockIdx.z / KS, ks = blockIdx.z % KS;
  const int64_t e_lo = E * ks / KS, e_hi = E * (ks + 1) / KS;
  const float* A = dSzt + bh * M * E;
  const float* Bm = Sz + bh * M * E;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  auto stage = [&](int buf, int64_t e0) {
    for (int x = threadIdx.x; x < kDwK * kDwTile; x += 256) {
      const int row = x / kDwK, kk = x % kDwK;
      const int64_t e = e0 + kk;
      const bool ina = i0 + row < M && e < e_hi, inb = j0 + row < M && e < e_hi;
      cp_async_f32(&sa[buf][kk][row], ina ? A + (i0 + row) * E + e : A, ina);
      cp_async_f32(&sb[buf][kk][row], inb ? Bm + (j0 + row) * E + e : Bm, inb);
    }
    cp_async_commit();
  };
  float acc[4][4] = {};
  if (e_lo < e_hi) stage(0, e_lo);
  int buf = 0;
  for (int64_t e0 = e_lo; e0 < e_hi; e0 += kDwK, buf ^= 1) {
    if (e0 + kDwK < e_hi) {
      stage(buf ^ 1, e0 + kDwK);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kDwK; ++kk) {
      const float4 a4 = *reinterpret_cast<const float4*>(&sa[buf][kk][ty * 4]);
      const float4 b4 = *reinterpret_cast<const float4*>(&sb[buf][kk][tx * 4]);
      const float a[4] = {a4.x, a4.y, a4.z, a4.w}, bb[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int w = 0; w < 4; ++w) acc[u][w] = fmaf(a[u], bb[w], acc[u][w]);
    }
    __syncthreads();   // the next iteration refills this buffer's partner, then this one
  }
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const int64_t ii = i0 + ty * 4 + u, jj = j0 + tx * 4 + w;
      if (ii < M && jj < M) part[(static_cast<int64_t>(blockIdx.z) * M + ii) * M + jj] = acc[u][w];
    }
}

constexpr int kDwrWarps = 8;

// dW = sum over (b, h) and the contraction splits of the partials (NP = BH *
// KS of them), in a fixed order (deterministic): a CTA owns 32 consecutive
// outputs, warp w sums partials w, w + 8, ... of output x0 + lane, then the
// eight warp sums are added in warp order.
__global__ void __launch_bounds__(kDwrWarps * 32)
simt_dw_reduce(const float* __restrict__ part, float* __restrict__ dW, int64_t MM, int64_t NP) {
  __shared__ float red[kDwrWarps][32];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t x = static_cast<int64_t>(blockIdx.x) * 32 + lane;
  float s = 0.0f;
  if (x < MM)
    for (int64_t n = warp; n < NP; n += kDwrWarps) s += part[n * MM + x];
  red[warp][lane] = s;
  __syncthreads();
  if (warp == 0 && x < MM) {
    float r = 0.0f;
    for (int w = 0; w < kDwrWarps; ++w) r += red[w][lane];
    dW[x] = r;
  }
}

// ============================================================================
// Causal backward.  The pages print none; [P2] App. B "Causal MHLA" trains
// with the chunkwise causal form and section 4 makes W learnable, so these are
// the chain-rule derivatives of simt_causal_output's arithmetic.  Per (b, h)
// and token t of query block i, with C_t = S<_i + W_ii P_t, c_t = z<_i + W_ii y_t
// (P_t, y_t the block's prefix sums of phi(k_s) v_s^T and phi(k_s), s <= t):
//   dnum_t = g_t / den_t,  dden_t = -(g_t . o_t) / den_t
//   dphi(q_t) = C_t dnum_t + dden_t c_t
//   dS<_i = sum_t phi(q_t) dnum_t^T,  dz<_i = sum_t dden_t phi(q_t)
//   dW_ii = sum_t sum_{s <= t} (phi(q_t) . phi(k_s)) (v_s . dnum_t + dden_t)
//   dW_ij = <dS<_i, S_j> + dz<_i . z_j  (j < i),   0 above the diagonal
//   dS_j  = sum_{i > j} W_ij dS<_i,  dz_j likewise
//   dv_s  = dS_j^T phi(k_s) + W_jj sum_{t >= s} (phi(q_t) . phi(k_s)) dnum_t
//   dphi(k_s) = dS_j v_s + dz_j + W_jj sum_{t >= s} phi(q_t) (dnum_t . v_s + dden_t)
// (t and s range over the block).  Kernels, in launch order:
//   simt_summary, simt_mix<false, true>   S_j and the mixed past S<_i, z<_i
//   simt_causal_bwd_query  per (b, h, i), 32-token chunks in order, the running
//                          state C in shared memory, each chunk in phases of
//                          register tiles: dq, dS<_i, dz<_i, the (b, h) share of
//                          dW_ii, and dnum_t, dden_t to scratch
//   simt_dw_partial, simt_dw_reduce_causal   dW below the diagonal, plus dW_ii
//   simt_mix<true, true>   dS_j, dz_j
//   simt_causal_bwd_key    per (b, h, j), chunks in reverse, the running
//                          suffix state dS_j + W_jj sum_{later t} phi(q_t) dnum_t^T,
//                          each chunk in phases of register tiles
// ============================================================================
constexpr int kCbThreads = 256;
constexpr int kCbWarps = kCbThreads / 32;
constexpr int kCbChunk = 32;    // one chunk token per lane in the score steps
constexpr int kCbRowLanes = kCbThreads / kCbChunk;   // threads staging one token row

// ENT = ceil(d*d / 256) state entries per thread (P_t and dS<_i in registers);
// DB = ceil(d / 16) columns per thread in the token x column phases.
//
// Per chunk of up to 32 tokens, in phases separated by block barriers, each
// thread computing a small register tile (2 tokens x DB columns, or a 2 x 2
// block of the 32 x 32 token pairs) so that every shared-memory operand it
// loads serves several FMAs:
//   1  scores a_ts = phi(q_t) . phi(k_s) (s <= t, same chunk) and P = W_ii a
//   2  den_t = phi(q_t) . c + sum_s P_ts + eps
//   3  num_t = phi(q_t)^T C + sum_s P_ts v_s; dnum_t = g_t / den_t,
//      dden_t = -(g_t . num_t) / den_t^2 (a 16-lane reduction per token)
//   4  b_ts = v_s . dnum_t + dden_t (s <= t); dW_ii += a_ts b_ts
//   5  dq_t = (C dnum_t + dden_t c + W_ii sum_s b_ts phi(k_s)) * [q_t > 0]
//   6  the chunk into the running state, dS<_i and dW_ii (as before)
template <typename T, int ENT, int DB>
__global__ void __launch_bounds__(kCbThreads)
simt_causal_bwd_query(const T* __restrict__ q, Operand qo, const T* __restrict__ k, Operand ko,
                      const T* __restrict__ v, Operand vo, const T* __restrict__ g_out, Operand go,
                      T* __restrict__ dq, Operand dqo, TokenGeom g, int64_t H, int d, int phi_kind, float eps,
                      const float* __restrict__ W, const float* __restrict__ Sp, float* __restrict__ dSp,
                      float* __restrict__ diag, float* __restrict__ dn) {
  extern __shared__ float sm[];
  constexpr int CP = kCbChunk + 1;         // padded row of a 32 x 32 token-pair matrix
  const int E = d * d, P = d + 1;
  float* st = sm;                          // [d][d + 1] C = S<_i + W_ii P before the chunk
  float* zs = st + d * P;                  // [d]        c = z<_i + W_ii y before the chunk
  float* sq = zs + d;                      // [chunk][d + 1] phi(q_t)
  float* sk = sq + kCbChunk * P;           // [chunk][d + 1] phi(k_s)
  float* sv = sk + kCbChunk * P;           // [chunk][d + 1] v_s
  float* sg = sv + kCbChunk * P;           // [chunk][d + 1] g_t
  float* sdn = sg + kCbChunk * P;          // [chunk][d + 1] dnum_t
  float* sdd = sdn + kCbChunk * P;         // [chunk]        dden_t
  float* sden = sdd + kCbChunk;            // [chunk]        den_t
  float* sa = sden + kCbChunk;             // [chunk][CP]    a_ts (s <= t, else 0)
  float* sb = sa + kCbChunk * CP;          // [chunk][CP]    b_ts (s <= t, else 0)
  float* red = sb + kCbChunk * CP;         // [warps]
  const int64_t item = blockIdx.x;
  const int64_t i = item % g.M, bh = item / g.M;
  const int64_t b = bh / H, h = bh % H;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const float wii = __ldg(W + i * g.M + i);
  const float* src = Sp + (bh * g.M + i) * static_cast<int64_t>(E + d);
  for (int e = tid; e < E; e += kCbThreads) st[(e / d) * P + e % d] = src[e];
  for (int r = tid; r < d; r += kCbThreads) zs[r] = src[E + r];
  const T* qb = q + b * qo.sb + h * qo.sh;
  const T* kb = k + b * ko.sb + h * ko.sh;
  const T* vb = v + b * vo.sb + h * vo.sh;
  const T* gb = g_out + b * go.sb + h * go.sh;
  T* dqb = dq + b * dqo.sb + h * dqo.sh;
  float* dnb = dn + (bh * g.M + i) * g.w * P;   // token rows: dnum_t (d), dden_t
  float pr[ENT], acc[ENT];
#pragma unroll
  for (int m = 0; m < ENT; ++m) pr[m] = acc[m] = 0.0f;
  float yr = 0.0f, zacc = 0.0f, dw = 0.0f;
  // token x column tiles: tokens 2 tt, 2 tt + 1 (a half-warp shares them), columns cc + 16 j
  const int tt = tid / 16, cc = tid % 16;
  const int t0 = 2 * tt, t1 = t0 + 1;
  // token-pair tiles: rows 2 pi, 2 pi + 1 and columns 2 pj, 2 pj + 1
  const int pi = tid / 16, pj = tid % 16;
  // state-entry tiles (phase 6 and the outputs): TB x TB entries per thread
  constexpr int TB = ENT == 1 ? 1 : ENT == 4 ? 2 : ENT == 16 ? 4 : 8;
  static_assert(TB * TB == ENT, "ENT is a square");
  const int r0 = TB * (tid / 16), c0 = TB * (tid % 16);
  // staging: one token row per kCbRowLanes threads; the blocks are contiguous
  // token ranges, so slot s of the block is token nb + s
  const int srow = tid / kCbRowLanes, spart = tid % kCbRowLanes;
  const int64_t nb = token_of(g, i, 0);
  for (int64_t s0 = 0; s0 < g.w; s0 += kCbChunk) {
    const int cnt = static_cast<int>(g.w - s0 < kCbChunk ? g.w - s0 : kCbChunk);
    __syncthreads();   // the state is complete and the previous chunk's rows are free
    if (srow < cnt) {
      const int64_t n = nb + s0 + srow;
      for (int c = spart; c < d; c += kCbRowLanes) {
        sq[srow * P + c] = phi_f(load_f(qb + n * qo.sn + c), phi_kind, eps);
        sk[srow * P + c] = phi_f(load_f(kb + n * ko.sn + c), phi_kind, eps);
        sv[srow * P + c] = load_f(vb + n * vo.sn + c);
        sg[srow * P + c] = load_f(gb + n * go.sn + c);
      }
    }
    __syncthreads();
    // ---- 1: a_ts for every pair of the chunk, a 2 x 2 block per thread (rows
    // past cnt hold stale values; the select below discards them)
    {
      const int ra = 2 * pi, rb = ra + 1, ca = 2 * pj, cb = ca + 1;
      float x00 = 0.0f, x01 = 0.0f, x10 = 0.0f, x11 = 0.0f;
      for (int r = 0; r < d; ++r) {
        const float qa = sq[ra * P + r], qb2 = sq[rb * P + r];
        const float ka = sk[ca * P + r], kb2 = sk[cb * P + r];
        x00 = fmaf(qa, ka, x00);
        x01 = fmaf(qa, kb2, x01);
        x10 = fmaf(qb2, ka, x10);
        x11 = fmaf(qb2, kb2, x11);
      }
      sa[ra * CP + ca] = (ra < cnt && ca <= ra) ? x00 : 0.0f;
      sa[ra * CP + cb] = (ra < cnt && cb <= ra) ? x01 : 0.0f;
      sa[rb * CP + ca] = (rb < cnt && ca <= rb) ? x10 : 0.0f;
      sa[rb * CP + cb] = (rb < cnt && cb <= rb) ? x11 : 0.0f;
    }
    __syncthreads();
    // ---- 2: den_t, eight threads per token (strided parts, then a fixed-order
    // shuffle sum over the eight)
    {
      const int tok = tid / 8, part = tid % 8;
      float den = 0.0f, own = 0.0f;
      for (int r = part; r < d; r += 8) den = fmaf(sq[tok * P + r], zs[r], den);
      for (int s2 = part; s2 < kCbChunk; s2 += 8) own += sa[tok * CP + s2];
#pragma unroll
      for (int off = 4; off > 0; off >>= 1) {
        den += __shfl_xor_sync(0xffffffffu, den, off);
        own += __shfl_xor_sync(0xffffffffu, own, off);
      }
      if (part == 0) sden[tok] = fmaf(wii, own, den) + eps;
    }
    __syncthreads();
    // ---- 3: num, dnum, dden (tokens t0, t1; columns cc + 16 j)
    {
      float n0[DB], n1[DB], o0[DB], o1[DB];
#pragma unroll
      for (int j = 0; j < DB; ++j) n0[j] = n1[j] = o0[j] = o1[j] = 0.0f;
      for (int r = 0; r < d; ++r) {
        const float q0 = sq[t0 * P + r], q1 = sq[t1 * P + r];
#pragma unroll
        for (int j = 0; j < DB; ++j) {
          const float cv = st[r * P + cc + 16 * j];   // columns past d read other data, discarded below
          n0[j] = fmaf(q0, cv, n0[j]);
          n1[j] = fmaf(q1, cv, n1[j]);
        }
      }
      for (int s2 = 0; s2 < cnt; ++s2) {
        const float p0 = sa[t0 * CP + s2], p1 = sa[t1 * CP + s2];
#pragma unroll
        for (int j = 0; j < DB; ++j) {
          const float vv = sv[s2 * P + cc + 16 * j];
          o0[j] = fmaf(p0, vv, o0[j]);
          o1[j] = fmaf(p1, vv, o1[j]);
        }
      }
      const float den0 = sden[t0], den1 = sden[t1];
      float go0 = 0.0f, go1 = 0.0f;
#pragma unroll
      for (int j = 0; j < DB; ++j) {
        const int c = cc + 16 * j;
        if (c < d) {
          const float g0 = sg[t0 * P + c], g1 = sg[t1 * P + c];
          go0 = fmaf(g0, fmaf(wii, o0[j], n0[j]), go0);
          go1 = fmaf(g1, fmaf(wii, o1[j], n1[j]), go1);
          const float dn0 = g0 / den0, dn1 = g1 / den1;
          sdn[t0 * P + c] = dn0;
          sdn[t1 * P + c] = dn1;
          if (t0 < cnt) dnb[(s0 + t0) * P + c] = dn0;
          if (t1 < cnt) dnb[(s0 + t1) * P + c] = dn1;
        }
      }
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) {   // the 16 lanes of this half-warp share t0, t1
        go0 += __shfl_xor_sync(0xffffffffu, go0, off);
        go1 += __shfl_xor_sync(0xffffffffu, go1, off);
      }
      if (cc == 0) {
        const float dd0 = -(go0 / den0) / den0, dd1 = -(go1 / den1) / den1;
        sdd[t0] = dd0;
        sdd[t1] = dd1;
        if (t0 < cnt) dnb[(s0 + t0) * P + d] = dd0;
        if (t1 < cnt) dnb[(s0 + t1) * P + d] = dd1;
      }
    }
    __syncthreads();
    // ---- 4: b_ts = v_s . dnum_t + dden_t (s <= t), dW_ii's own-chunk part
    {
      const int ra = 2 * pi, rb = ra + 1, ca = 2 * pj, cb = ca + 1;
      float x00 = 0.0f, x01 = 0.0f, x10 = 0.0f, x11 = 0.0f;
      for (int c = 0; c < d; ++c) {
        const float na = sdn[ra * P + c], nb = sdn[rb * P + c];
        const float va = sv[ca * P + c], vb2 = sv[cb * P + c];
        x00 = fmaf(na, va, x00);
        x01 = fmaf(na, vb2, x01);
        x10 = fmaf(nb, va, x10);
        x11 = fmaf(nb, vb2, x11);
      }
      const float da = sdd[ra], db = sdd[rb];
      const float b00 = (ra < cnt && ca <= ra) ? x00 + da : 0.0f;
      const float b01 = (ra < cnt && cb <= ra) ? x01 + da : 0.0f;
      const float b10 = (rb < cnt && ca <= rb) ? x10 + db : 0.0f;
      const float b11 = (rb < cnt && cb <= rb) ? x11 + db : 0.0f;
      sb[ra * CP + ca] = b00;
      sb[ra * CP + cb] = b01;
      sb[rb * CP + ca] = b10;
      sb[rb * CP + cb] = b11;
      // a is zero wherever b is (the same mask)
      dw = fmaf(sa[ra * CP + ca], b00, dw);
      dw = fmaf(sa[ra * CP + cb], b01, dw);
      dw = fmaf(sa[rb * CP + ca], b10, dw);
      dw = fmaf(sa[rb * CP + cb], b11, dw);
    }
    __syncthreads();
    // ---- 5: dq (tokens t0, t1; rows r = cc + 16 j)
    {
      float x0[DB], x1[DB], w0[DB], w1[DB];
#pragma unroll
      for (int j = 0; j < DB; ++j) x0[j] = x1[j] = w0[j] = w1[j] = 0.0f;
      for (int c = 0; c < d; ++c) {
        const float n0 = sdn[t0 * P + c], n1 = sdn[t1 * P + c];
#pragma unroll
        for (int j = 0; j < DB; ++j) {
          const float cv = st[(cc + 16 * j) * P + c];   // rows past d read other data, discarded below
          x0[j] = fmaf(cv, n0, x0[j]);
          x1[j] = fmaf(cv, n1, x1[j]);
        }
      }
      for (int s2 = 0; s2 < cnt; ++s2) {
        const float b0 = sb[t0 * CP + s2], b1 = sb[t1 * CP + s2];
#pragma unroll
        for (int j = 0; j < DB; ++j) {
          const float kv = sk[s2 * P + cc + 16 * j];
          w0[j] = fmaf(kv, b0, w0[j]);
          w1[j] = fmaf(kv, b1, w1[j]);
        }
      }
      const float dd0 = sdd[t0], dd1 = sdd[t1];
      const int64_t n0t = t0 < cnt ? nb + s0 + t0 : 0;
      const int64_t n1t = t1 < cnt ? nb + s0 + t1 : 0;
#pragma unroll
      for (int j = 0; j < DB; ++j) {
        const int r = cc + 16 * j;
        if (r < d) {
          const float zr = zs[r];
          if (t0 < cnt) {
            const float x = fmaf(wii, w0[j], fmaf(dd0, zr, x0[j]));
            store_f(dqb + n0t * dqo.sn + r, load_f(qb + n0t * qo.sn + r) > 0.0f ? x : 0.0f);
          }
          if (t1 < cnt) {
            const float x = fmaf(wii, w1[j], fmaf(dd1, zr, x1[j]));
            store_f(dqb + n1t * dqo.sn + r, load_f(qb + n1t * qo.sn + r) > 0.0f ? x : 0.0f);
          }
        }
      }
    }
    __syncthreads();   // phase 6 rewrites the state phase 5 has read
    // ---- 6: dS<_i += X (the chunk's sum of phi(q_t) dnum_t^T); dW_ii += <P, X>; then
    // P and the state advance by the chunk's phi(k_s) v_s^T.  Each thread owns a
    // TB x TB tile of the entries (rows TB (tid / 16) + u, columns TB (tid % 16) + w).
    {
      // the X terms go straight into dS<_i and dW_ii (P is this chunk's old value
      // throughout the loop); the state increments wait in dps
      float dps[ENT];
#pragma unroll
      for (int m = 0; m < ENT; ++m) dps[m] = 0.0f;
      for (int sl = 0; sl < cnt; ++sl) {
        float qr[TB], kr[TB], nc[TB], vc[TB];
#pragma unroll
        for (int u = 0; u < TB; ++u) {
          qr[u] = sq[sl * P + r0 + u];   // rows and columns past d read other data, discarded below
          kr[u] = sk[sl * P + r0 + u];
          nc[u] = sdn[sl * P + c0 + u];
          vc[u] = sv[sl * P + c0 + u];
        }
#pragma unroll
        for (int u = 0; u < TB; ++u)
#pragma unroll
          for (int w = 0; w < TB; ++w) {
            const float x = qr[u] * nc[w];
            acc[u * TB + w] += x;
            dw = fmaf(pr[u * TB + w], x, dw);
            dps[u * TB + w] = fmaf(kr[u], vc[w], dps[u * TB + w]);
          }
      }
#pragma unroll
      for (int m = 0; m < ENT; ++m) {
        const int r = r0 + m / TB, c = c0 + m % TB;
        pr[m] += dps[m];
        if (r < d && c < d) st[r * P + c] = fmaf(wii, dps[m], st[r * P + c]);
      }
    }
    if (tid < d) {
      float x = 0.0f, dy = 0.0f;
      for (int sl = 0; sl < cnt; ++sl) {
        x = fmaf(sq[sl * P + tid], sdd[sl], x);
        dy += sk[sl * P + tid];
      }
      dw = fmaf(yr, x, dw);
      zacc += x;
      yr += dy;
      zs[tid] = fmaf(wii, dy, zs[tid]);
    }
  }
  float* out = dSp + (bh * g.M + i) * static_cast<int64_t>(E + d);
#pragma unroll
  for (int m = 0; m < ENT; ++m) {
    const int r = r0 + m / TB, c = c0 + m % TB;
    if (r < d && c < d) out[r * d + c] = acc[m];
  }
  if (tid < d) out[E + tid] = zacc;
  dw = warp_sum(dw);
  if (lane == 0) red[warp] = dw;
  __syncthreads();
  if (tid == 0) {
    float s = 0.0f;
    for (int w = 0; w < kCbWarps; ++w) s += red[w];
    diag[bh * g.M + i] = s;
  }
}

// One CTA per (b, h, j), chunks of the block in reverse, each chunk in phases of
// register tiles (DB = ceil(d / 16) columns per thread; TB x TB state entries):
//   1  a_st = phi(k_s) . phi(q_t) and b_st = v_s . dnum_t + dden_t for t >= s
//   2  dv_s = G^T phi(k_s) + W_jj sum_t a_st dnum_t
//      dphi(k_s) = G v_s + gz + W_jj sum_t b_st phi(q_t), masked by [k_s > 0]
//   3  G += W_jj sum_t phi(q_t) dnum_t^T, gz += W_jj sum_t dden_t phi(q_t)
// with G = dS_j + W_jj sum over later chunks of phi(q_t) dnum_t^T (gz likewise).
template <typename T, int DB, int TB>
__global__ void __launch_bounds__(kCbThreads)
simt_causal_bwd_key(const T* __restrict__ q, Operand qo, const T* __restrict__ k, Operand ko,
                    const T* __restrict__ v, Operand vo, T* __restrict__ dk, Operand dko, T* __restrict__ dv,
                    Operand dvo, TokenGeom g, int64_t H, int d, int phi_kind, float eps, const float* __restrict__ W,
                    const float* __restrict__ dS, const float* __restrict__ dn) {
  extern __shared__ float sm[];
  constexpr int CP = kCbChunk + 1;
  const int E = d * d, P = d + 1;
  float* gs = sm;                          // [d][d + 1] G
  float* gz = gs + d * P;                  // [d]        gz
  float* sq = gz + d;                      // [chunk][d + 1] phi(q_t)
  float* sdn = sq + kCbChunk * P;          // [chunk][d + 1] dnum_t
  float* sk = sdn + kCbChunk * P;          // [chunk][d + 1] phi(k_s)
  float* sv = sk + kCbChunk * P;           // [chunk][d + 1] v_s
  float* sdd = sv + kCbChunk * P;          // [chunk]        dden_t
  float* sa = sdd + kCbChunk;              // [chunk][CP]    a_st (t >= s, else 0)
  float* sb = sa + kCbChunk * CP;          // [chunk][CP]    b_st (t >= s, else 0)
  const int64_t item = blockIdx.x;
  const int64_t j = item % g.M, bh = item / g.M;
  const int64_t b = bh / H, h = bh % H;
  const int tid = threadIdx.x;
  const float wjj = __ldg(W + j * g.M + j);
  const float* src = dS + (bh * g.M + j) * static_cast<int64_t>(E + d);
  for (int e = tid; e < E; e += kCbThreads) gs[(e / d) * P + e % d] = src[e];
  for (int r = tid; r < d; r += kCbThreads) gz[r] = src[E + r];
  const T* qb = q + b * qo.sb + h * qo.sh;
  const T* kb = k + b * ko.sb + h * ko.sh;
  const T* vb = v + b * vo.sb + h * vo.sh;
  T* dkb = dk + b * dko.sb + h * dko.sh;
  T* dvb = dv + b * dvo.sb + h * dvo.sh;
  const float* dnb = dn + (bh * g.M + j) * g.w * P;
  const int tt = tid / 16, cc = tid % 16;          // sources 2 tt, 2 tt + 1; columns cc + 16 j
  const int s0t = 2 * tt, s1t = s0t + 1;
  const int pi = tid / 16, pj = tid % 16;          // pair tiles: sources 2 pi (+1), queries 2 pj (+1)
  const int r0 = TB * (tid / 16), c0 = TB * (tid % 16);   // state tile
  const int srow = tid / kCbRowLanes, spart = tid % kCbRowLanes;   // staging, as in the query kernel
  const int64_t nb = token_of(g, j, 0);
  const int64_t nch = (g.w + kCbChunk - 1) / kCbChunk;
  for (int64_t ci = nch - 1; ci >= 0; --ci) {
    const int64_t s0 = ci * kCbChunk;
    const int cnt = static_cast<int>(g.w - s0 < kCbChunk ? g.w - s0 : kCbChunk);
    __syncthreads();   // the suffix state is complete and the later chunk's rows are free
    if (srow < cnt) {
      const int64_t n = nb + s0 + srow;
      for (int c = spart; c < d; c += kCbRowLanes) {
        sq[srow * P + c] = phi_f(load_f(qb + n * qo.sn + c), phi_kind, eps);
        sdn[srow * P + c] = dnb[(s0 + srow) * P + c];
        sk[srow * P + c] = phi_f(load_f(kb + n * ko.sn + c), phi_kind, eps);
        sv[srow * P + c] = load_f(vb + n * vo.sn + c);
      }
    }
    for (int sl = tid; sl < cnt; sl += kCbThreads) sdd[sl] = dnb[(s0 + sl) * P + d];
    __syncthreads();
    // ---- 1: a_st and b_st, 2 x 2 blocks (sources ra, rb; queries ca, cb)
    {
      const int ra = 2 * pi, rb = ra + 1, ca = 2 * pj, cb = ca + 1;
      float a00 = 0.0f, a01 = 0.0f, a10 = 0.0f, a11 = 0.0f;
      float b00 = 0.0f, b01 = 0.0f, b10 = 0.0f, b11 = 0.0f;
      for (int r = 0; r < d; ++r) {
        const float ka = sk[ra * P + r], kb2 = sk[rb * P + r], qa = sq[ca * P + r], qb2 = sq[cb * P + r];
        const float va = sv[ra * P + r], vb2 = sv[rb * P + r], na = sdn[ca * P + r], nb = sdn[cb * P + r];
        a00 = fmaf(ka, qa, a00);
        a01 = fmaf(ka, qb2, a01);
        a10 = fmaf(kb2, qa, a10);
        a11 = fmaf(kb2, qb2, a11);
        b00 = fmaf(va, na, b00);
        b01 = fmaf(va, nb, b01);
        b10 = fmaf(vb2, na, b10);
        b11 = fmaf(vb2, nb, b11);
      }
      const float dda = sdd[ca], ddb = sdd[cb];
      const bool m00 = ca < cnt && ca >= ra, m01 = cb < cnt && cb >= ra;
      const bool m10 = ca < cnt && ca >= rb, m11 = cb < cnt && cb >= rb;
      sa[ra * CP + ca] = m00 ? a00 : 0.0f;
      sa[ra * CP + cb] = m01 ? a01 : 0.0f;
      sa[rb * CP + ca] = m10 ? a10 : 0.0f;
      sa[rb * CP + cb] = m11 ? a11 : 0.0f;
      sb[ra * CP + ca] = m00 ? b00 + dda : 0.0f;
      sb[ra * CP + cb] = m01 ? b01 + ddb : 0.0f;
      sb[rb * CP + ca] = m10 ? b10 + dda : 0.0f;
      sb[rb * CP + cb] = m11 ? b11 + ddb : 0.0f;
    }
    __syncthreads();
    // ---- 2: dv and dk of sources s0t, s1t (columns / rows cc + 16 j)
    {
      float v0[DB], v1[DB], w0[DB], w1[DB];
#pragma unroll
      for (int jj = 0; jj < DB; ++jj) v0[jj] = v1[jj] = w0[jj] = w1[jj] = 0.0f;
      // G^T phi(k_s) (column c of G) and G v_s (row r of G): one pass over the inner index
      for (int x = 0; x < d; ++x) {
        const float k0 = sk[s0t * P + x], k1 = sk[s1t * P + x];
        const float e0 = sv[s0t * P + x], e1 = sv[s1t * P + x];
#pragma unroll
        for (int jj = 0; jj < DB; ++jj) {
          const float gcol = gs[x * P + cc + 16 * jj];    // G[x][c]   (past d: other data, discarded)
          const float grow = gs[(cc + 16 * jj) * P + x];  // G[r][x]
          v0[jj] = fmaf(k0, gcol, v0[jj]);
          v1[jj] = fmaf(k1, gcol, v1[jj]);
          w0[jj] = fmaf(grow, e0, w0[jj]);
          w1[jj] = fmaf(grow, e1, w1[jj]);
        }
      }
      float ov0[DB], ov1[DB], ok0[DB], ok1[DB];
#pragma unroll
      for (int jj = 0; jj < DB; ++jj) ov0[jj] = ov1[jj] = ok0[jj] = ok1[jj] = 0.0f;
      for (int t = 0; t < cnt; ++t) {
        const float a0 = sa[s0t * CP + t], a1 = sa[s1t * CP + t];
        const float b0 = sb[s0t * CP + t], b1 = sb[s1t * CP + t];
#pragma unroll
        for (int jj = 0; jj < DB; ++jj) {
          const float nv = sdn[t * P + cc + 16 * jj];
          const float qv = sq[t * P + cc + 16 * jj];
          ov0[jj] = fmaf(a0, nv, ov0[jj]);
          ov1[jj] = fmaf(a1, nv, ov1[jj]);
          ok0[jj] = fmaf(b0, qv, ok0[jj]);
          ok1[jj] = fmaf(b1, qv, ok1[jj]);
        }
      }
      const int64_t n0t = s0t < cnt ? nb + s0 + s0t : 0;
      const int64_t n1t = s1t < cnt ? nb + s0 + s1t : 0;
#pragma unroll
      for (int jj = 0; jj < DB; ++jj) {
        const int c = cc + 16 * jj;
        if (c < d) {
          const float zr = gz[c];
          if (s0t < cnt) {
            store_f(dvb + n0t * dvo.sn + c, fmaf(wjj, ov0[jj], v0[jj]));
            const float x = fmaf(wjj, ok0[jj], w0[jj] + zr);
            store_f(dkb + n0t * dko.sn + c, load_f(kb + n0t * ko.sn + c) > 0.0f ? x : 0.0f);
          }
          if (s1t < cnt) {
            store_f(dvb + n1t * dvo.sn + c, fmaf(wjj, ov1[jj], v1[jj]));
            const float x = fmaf(wjj, ok1[jj], w1[jj] + zr);
            store_f(dkb + n1t * dko.sn + c, load_f(kb + n1t * ko.sn + c) > 0.0f ? x : 0.0f);
          }
        }
      }
    }
    __syncthreads();   // phase 3 rewrites G, which phase 2 has read
    // ---- 3: G += W_jj sum_t phi(q_t) dnum_t^T (a TB x TB tile per thread), gz likewise
    {
      float x[TB * TB];
#pragma unroll
      for (int m = 0; m < TB * TB; ++m) x[m] = 0.0f;
      for (int t = 0; t < cnt; ++t) {
        float qr[TB], nc[TB];
#pragma unroll
        for (int u = 0; u < TB; ++u) {
          qr[u] = sq[t * P + r0 + u];
          nc[u] = sdn[t * P + c0 + u];
        }
#pragma unroll
        for (int u = 0; u < TB; ++u)
#pragma unroll
          for (int w = 0; w < TB; ++w) x[u * TB + w] = fmaf(qr[u], nc[w], x[u * TB + w]);
      }
#pragma unroll
      for (int m = 0; m < TB * TB; ++m) {
        const int r = r0 + m / TB, c = c0 + m % TB;
        if (r < d && c < d) gs[r * P + c] = fmaf(wjj, x[m], gs[r * P + c]);
      }
    }
    if (tid < d) {
      float x = 0.0f;
      for (int t = 0; t < cnt; ++t) x = fmaf(sdd[t], sq[t * P + tid], x);
      gz[tid] = fmaf(wjj, x, gz[tid]);
    }
  }
}

// Vector loads and stores of V consecutive floats (V = 1, 2 or 4; the address
// aligned to V floats).
template <int V>
__device__ __forceinline__ void ldv(const float* p, float (&x)[V]) {
  if constexpr (V == 4) {
    const float4 t = *reinterpret_cast<const float4*>(p);
    x[0] = t.x, x[1] = t.y, x[2] = t.z, x[3] = t.w;
  } else if constexpr (V == 2) {
    const float2 t = *reinterpret_cast<const float2*>(p);
    x[0] = t.x, x[1] = t.y;
  } else {
    x[0] = *p;
  }
}
template <int V>
__device__ __forceinline__ void stv(float* p, const float (&x)[V]) {
  if constexpr (V == 4) {
    *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
  } else if constexpr (V == 2) {
    *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]);
  } else {
    *p = x[0];
  }
}

// The causal backward's query side for d = D in {32, 64}, laid out for 16-byte
// shared-memory vectors (token and state rows padded to D + 4 floats) and
// rearranged so that one product of the state serves two terms: with
// u_t = C g_t,
//   C dnum_t = u_t / den_t   and   g_t . num_t = phi(q_t) . u_t + W_ii sum_s a_ts e_ts,
// e_ts = g_t . v_s, so b_ts = e_ts / den_t + dden_t needs no second pass over the
// columns.  Only C^T is kept (u reads it by rows).  Per 32-token chunk:
//   1  a_ts = phi(q_t) . phi(k_s) and e_ts (s <= t), pair tiles {p, p + 16} x {q, q + 16}
//   2  per token, over the 16 lanes of a half-warp (V = D / 16 columns each):
//      u_t, den_t, g_t . num_t, dnum_t, dden_t, b_ts, dW_ii's own-chunk part
//   3  dq_t = u_t / den_t + dden_t c + W_ii sum_s b_ts phi(k_s), masked by [q_t > 0]
//   4  X = sum_t phi(q_t) dnum_t^T over V x V entries per thread: dS<_i += X,
//      dW_ii += <P, X>; then (unless the block ends here) P and C^T advance by
//      the chunk's phi(k_s) v_s^T
// Chunk rows past the block's end are zero, so every loop runs the full 32 tokens.
template <typename T, int D>
__global__ void __launch_bounds__(kCbThreads, 2)
simt_causal_bwd_query_v(const T* __restrict__ q, Operand qo, const T* __restrict__ k, Operand ko,
                        const T* __restrict__ v, Operand vo, const T* __restrict__ g_out, Operand go,
                        T* __restrict__ dq, Operand dqo, TokenGeom g, int64_t H, int phi_kind, float eps,
                        const float* __restrict__ W, const float* __restrict__ Sp, float* __restrict__ dSp,
                        float* __restrict__ diag, float* __restrict__ dn, const __nv_bfloat16* __restrict__ Stb,
                        const float* __restrict__ ztb) {
  constexpr int V = D / 16;
  constexpr int P = D + 4;                 // padded token / state row
  constexpr int CP = kCbChunk + 4;         // padded row of a 32 x 32 token-pair matrix
  constexpr int E = D * D, PD = D + 1;     // PD: the dnum / dden scratch row
  extern __shared__ __align__(16) float cbq_sm[];
  float* stT = cbq_sm;                     // [D][P] C^T, C = S<_i + W_ii P before the chunk
  float* zs = stT + D * P;                 // [D]    c = z<_i + W_ii y before the chunk
  float* sq = zs + D;                      // [chunk][P] phi(q_t)
  float* sk = sq + kCbChunk * P;           // [chunk][P] phi(k_s)
  float* sv = sk + kCbChunk * P;           // [chunk][P] v_s
  float* sg = sv + kCbChunk * P;           // [chunk][P] g_t
  float* sdn = sg + kCbChunk * P;          // [chunk][P] dnum_t
  float* sdd = sdn + kCbChunk * P;         // [chunk]    dden_t
  float* sa = sdd + kCbChunk;              // [chunk][CP] a_ts (s <= t, else 0)
  float* se = sa + kCbChunk * CP;          // [chunk][CP] e_ts, then b_ts (s <= t, else 0)
  float* red = se + kCbChunk * CP;         // [warps]
  const int64_t item = blockIdx.x;
  const int64_t i = item % g.M, bh = item / g.M;
  const int64_t b = bh / H, h = bh % H;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const float wii = __ldg(W + i * g.M + i);
  // S<_i and z<_i: float32 rows of Sp, or (Stb non-null) the tensor-core states
  // (bf16 row-major S<_i, float32 z<_i)
  const int64_t si = bh * g.M + i;
  if (Stb) {
    for (int e = tid; e < E; e += kCbThreads) stT[(e % D) * P + e / D] = __bfloat162float(Stb[si * E + e]);
    for (int r = tid; r < D; r += kCbThreads) zs[r] = ztb[si * D + r];
  } else {
    const float* src = Sp + si * static_cast<int64_t>(E + D);
    for (int e = tid; e < E; e += kCbThreads) stT[(e % D) * P + e / D] = src[e];
    for (int r = tid; r < D; r += kCbThreads) zs[r] = src[E + r];
  }
  const T* qb = q + b * qo.sb + h * qo.sh;
  const T* kb = k + b * ko.sb + h * ko.sh;
  const T* vb = v + b * vo.sb + h * vo.sh;
  const T* gb = g_out + b * go.sb + h * go.sh;
  T* dqb = dq + b * dqo.sb + h * dqo.sh;
  float* dnb = dn + (bh * g.M + i) * g.w * PD;   // token rows: dnum_t (D), dden_t
  float pr[V * V], acc[V * V];
#pragma unroll
  for (int m = 0; m < V * V; ++m) pr[m] = acc[m] = 0.0f;
  float yr = 0.0f, zacc = 0.0f, dw = 0.0f;
  const int tt = tid / 16, cc = tid % 16;
  const int t0 = 2 * tt, t1 = t0 + 1;      // per-token steps: tokens t0, t1; columns c0 ..
  const int c0 = V * cc;
  const int r0 = V * tt;                   // state tile: rows r0 .., columns c0 ..
  const int pi = tid / 16, pj = tid % 16;  // pair tiles: tokens pi, pi + 16; sources pj, pj + 16
  const int srow = tid / kCbRowLanes, spart = tid % kCbRowLanes;
  const int64_t nb = token_of(g, i, 0);    // contiguous blocks: slot s is token nb + s
  for (int64_t s0 = 0; s0 < g.w; s0 += kCbChunk) {
    const int cnt = static_cast<int>(g.w - s0 < kCbChunk ? g.w - s0 : kCbChunk);
    const bool more = s0 + kCbChunk < g.w;   // a later chunk of the block reads the advanced state
    __syncthreads();   // the state is complete and the previous chunk's rows are free
    {
      const bool live = srow < cnt;
      const int64_t n = nb + s0 + srow;
#pragma unroll
      for (int c = 4 * spart; c < D; c += 4 * kCbRowLanes) {
        float xq[4], xk[4], xv[4], xg[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          xq[u] = live ? phi_f(load_f(qb + n * qo.sn + c + u), phi_kind, eps) : 0.0f;
          xk[u] = live ? phi_f(load_f(kb + n * ko.sn + c + u), phi_kind, eps) : 0.0f;
          xv[u] = live ? load_f(vb + n * vo.sn + c + u) : 0.0f;
          xg[u] = live ? load_f(gb + n * go.sn + c + u) : 0.0f;
        }
        stv<4>(sq + srow * P + c, xq);
        stv<4>(sk + srow * P + c, xk);
        stv<4>(sv + srow * P + c, xv);
        stv<4>(sg + srow * P + c, xg);
      }
    }
    __syncthreads();
    // ---- 1: a_ts and e_ts (s <= t); the block (pi, pj + 16) lies above the diagonal
    {
      const int ra = pi, rb = pi + 16, ca = pj, cb = pj + 16;
      float a00 = 0.0f, a10 = 0.0f, a11 = 0.0f, e00 = 0.0f, e10 = 0.0f, e11 = 0.0f;
#pragma unroll 2
      for (int r = 0; r < D; r += V) {
        float qa[V], qc[V], ka[V], kc[V], ga[V], gc[V], va[V], vc[V];
        ldv<V>(sq + ra * P + r, qa);
        ldv<V>(sq + rb * P + r, qc);
        ldv<V>(sk + ca * P + r, ka);
        ldv<V>(sk + cb * P + r, kc);
        ldv<V>(sg + ra * P + r, ga);
        ldv<V>(sg + rb * P + r, gc);
        ldv<V>(sv + ca * P + r, va);
        ldv<V>(sv + cb * P + r, vc);
#pragma unroll
        for (int u = 0; u < V; ++u) {
          a00 = fmaf(qa[u], ka[u], a00);
          a10 = fmaf(qc[u], ka[u], a10);
          a11 = fmaf(qc[u], kc[u], a11);
          e00 = fmaf(ga[u], va[u], e00);
          e10 = fmaf(gc[u], va[u], e10);
          e11 = fmaf(gc[u], vc[u], e11);
        }
      }
      const bool m00 = ra < cnt && ca <= ra, m10 = rb < cnt, m11 = rb < cnt && cb <= rb;
      sa[ra * CP + ca] = m00 ? a00 : 0.0f;
      sa[ra * CP + cb] = 0.0f;
      sa[rb * CP + ca] = m10 ? a10 : 0.0f;
      sa[rb * CP + cb] = m11 ? a11 : 0.0f;
      se[ra * CP + ca] = m00 ? e00 : 0.0f;
      se[ra * CP + cb] = 0.0f;
      se[rb * CP + ca] = m10 ? e10 : 0.0f;
      se[rb * CP + cb] = m11 ? e11 : 0.0f;
    }
    __syncthreads();
    // ---- 2: per token (t0, t1 on the 16 lanes of a half-warp; columns / rows c0 ..)
    float x0[V], x1[V];   // C dnum_t + dden_t c, this lane's rows
    {
      float u0[V], u1[V];
#pragma unroll
      for (int w = 0; w < V; ++w) u0[w] = u1[w] = 0.0f;
#pragma unroll 2
      for (int c = 0; c < D; c += V) {
        float ga[V], gc[V];
        ldv<V>(sg + t0 * P + c, ga);
        ldv<V>(sg + t1 * P + c, gc);
#pragma unroll
        for (int u = 0; u < V; ++u) {
          float cv[V];
          ldv<V>(stT + (c + u) * P + c0, cv);   // C[c0 + w][c + u]
#pragma unroll
          for (int w = 0; w < V; ++w) {
            u0[w] = fmaf(cv[w], ga[u], u0[w]);
            u1[w] = fmaf(cv[w], gc[u], u1[w]);
          }
        }
      }
      float qa[V], qc[V], zv[V], gva[V], gvc[V];
      ldv<V>(sq + t0 * P + c0, qa);
      ldv<V>(sq + t1 * P + c0, qc);
      ldv<V>(zs + c0, zv);
      ldv<V>(sg + t0 * P + c0, gva);
      ldv<V>(sg + t1 * P + c0, gvc);
      float den0 = 0.0f, den1 = 0.0f, go0 = 0.0f, go1 = 0.0f;
#pragma unroll
      for (int w = 0; w < V; ++w) {
        den0 = fmaf(qa[w], zv[w], den0);
        den1 = fmaf(qc[w], zv[w], den1);
        go0 = fmaf(qa[w], u0[w], go0);
        go1 = fmaf(qc[w], u1[w], go1);
      }
      // this lane's own-chunk sources s = cc, cc + 16
      const float a0a = sa[t0 * CP + cc], a0b = sa[t0 * CP + cc + 16];
      const float a1a = sa[t1 * CP + cc], a1b = sa[t1 * CP + cc + 16];
      const float e0a = se[t0 * CP + cc], e0b = se[t0 * CP + cc + 16];
      const float e1a = se[t1 * CP + cc], e1b = se[t1 * CP + cc + 16];
      den0 = fmaf(wii, a0a + a0b, den0);
      den1 = fmaf(wii, a1a + a1b, den1);
      go0 = fmaf(wii, fmaf(a0a, e0a, a0b * e0b), go0);
      go1 = fmaf(wii, fmaf(a1a, e1a, a1b * e1b), go1);
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) {   // the 16 lanes of this half-warp share t0, t1
        den0 += __shfl_xor_sync(0xffffffffu, den0, off);
        den1 += __shfl_xor_sync(0xffffffffu, den1, off);
        go0 += __shfl_xor_sync(0xffffffffu, go0, off);
        go1 += __shfl_xor_sync(0xffffffffu, go1, off);
      }
      den0 += eps;
      den1 += eps;
      const bool l0 = t0 < cnt, l1 = t1 < cnt;   // rows past the block stay zero
      const float dd0 = l0 ? -(go0 / den0) / den0 : 0.0f;
      const float dd1 = l1 ? -(go1 / den1) / den1 : 0.0f;
      float dn0[V], dn1[V];
#pragma unroll
      for (int w = 0; w < V; ++w) {
        dn0[w] = l0 ? gva[w] / den0 : 0.0f;
        dn1[w] = l1 ? gvc[w] / den1 : 0.0f;
        x0[w] = fmaf(dd0, zv[w], u0[w] / den0);
        x1[w] = fmaf(dd1, zv[w], u1[w] / den1);
      }
      stv<V>(sdn + t0 * P + c0, dn0);
      stv<V>(sdn + t1 * P + c0, dn1);
#pragma unroll
      for (int w = 0; w < V; ++w) {
        if (l0) dnb[(s0 + t0) * PD + c0 + w] = dn0[w];
        if (l1) dnb[(s0 + t1) * PD + c0 + w] = dn1[w];
      }
      if (cc == 0) {
        sdd[t0] = dd0;
        sdd[t1] = dd1;
        if (l0) dnb[(s0 + t0) * PD + D] = dd0;
        if (l1) dnb[(s0 + t1) * PD + D] = dd1;
      }
      // b_ts = e_ts / den_t + dden_t (s <= t) in place of e_ts; dW_ii's own-chunk part
      const float b0a = (l0 && cc <= t0) ? e0a / den0 + dd0 : 0.0f;
      const float b0b = (l0 && cc + 16 <= t0) ? e0b / den0 + dd0 : 0.0f;
      const float b1a = (l1 && cc <= t1) ? e1a / den1 + dd1 : 0.0f;
      const float b1b = (l1 && cc + 16 <= t1) ? e1b / den1 + dd1 : 0.0f;
      se[t0 * CP + cc] = b0a;
      se[t0 * CP + cc + 16] = b0b;
      se[t1 * CP + cc] = b1a;
      se[t1 * CP + cc + 16] = b1b;
      dw = fmaf(a0a, b0a, dw);
      dw = fmaf(a0b, b0b, dw);
      dw = fmaf(a1a, b1a, dw);
      dw = fmaf(a1b, b1b, dw);
    }
    __syncthreads();
    // ---- 3: dq (tokens t0, t1; rows c0 ..)
    {
      float w0[V], w1[V];
#pragma unroll
      for (int w = 0; w < V; ++w) w0[w] = w1[w] = 0.0f;
#pragma unroll 2
      for (int s = 0; s < kCbChunk; s += V) {
        float ba[V], bc[V];
        ldv<V>(se + t0 * CP + s, ba);
        ldv<V>(se + t1 * CP + s, bc);
#pragma unroll
        for (int u = 0; u < V; ++u) {
          float kv[V];
          ldv<V>(sk + (s + u) * P + c0, kv);
#pragma unroll
          for (int w = 0; w < V; ++w) {
            w0[w] = fmaf(kv[w], ba[u], w0[w]);
            w1[w] = fmaf(kv[w], bc[u], w1[w]);
          }
        }
      }
      const int64_t n0t = nb + s0 + t0, n1t = nb + s0 + t1;
#pragma unroll
      for (int w = 0; w < V; ++w) {
        const int r = c0 + w;
        if (t0 < cnt) {
          const float x = fmaf(wii, w0[w], x0[w]);
          store_f(dqb + n0t * dqo.sn + r, load_f(qb + n0t * qo.sn + r) > 0.0f ? x : 0.0f);
        }
        if (t1 < cnt) {
          const float x = fmaf(wii, w1[w], x1[w]);
          store_f(dqb + n1t * dqo.sn + r, load_f(qb + n1t * qo.sn + r) > 0.0f ? x : 0.0f);
        }
      }
    }
    // ---- 4: X and, unless the block ends here, the chunk's phi(k_s) v_s^T over this
    // thread's V x V entries (no barrier before: steps 2 and 3 are done with C^T)
    {
      float X[V * V], dps[V * V];
#pragma unroll
      for (int m = 0; m < V * V; ++m) X[m] = dps[m] = 0.0f;
      if (more) {
#pragma unroll 4
        for (int sl = 0; sl < kCbChunk; ++sl) {
          float qr[V], kr[V], nc[V], vc[V];
          ldv<V>(sq + sl * P + r0, qr);
          ldv<V>(sk + sl * P + r0, kr);
          ldv<V>(sdn + sl * P + c0, nc);
          ldv<V>(sv + sl * P + c0, vc);
#pragma unroll
          for (int u = 0; u < V; ++u)
#pragma unroll
            for (int w = 0; w < V; ++w) {
              X[u * V + w] = fmaf(qr[u], nc[w], X[u * V + w]);
              dps[u * V + w] = fmaf(kr[u], vc[w], dps[u * V + w]);
            }
        }
      } else {
#pragma unroll 4
        for (int sl = 0; sl < kCbChunk; ++sl) {
          float qr[V], nc[V];
          ldv<V>(sq + sl * P + r0, qr);
          ldv<V>(sdn + sl * P + c0, nc);
#pragma unroll
          for (int u = 0; u < V; ++u)
#pragma unroll
            for (int w = 0; w < V; ++w) X[u * V + w] = fmaf(qr[u], nc[w], X[u * V + w]);
        }
      }
#pragma unroll
      for (int m = 0; m < V * V; ++m) {
        dw = fmaf(pr[m], X[m], dw);
        acc[m] += X[m];
        pr[m] += dps[m];
      }
      if (more) {
#pragma unroll
        for (int w = 0; w < V; ++w) {
          float cur[V];
          ldv<V>(stT + (c0 + w) * P + r0, cur);
#pragma unroll
          for (int u = 0; u < V; ++u) cur[u] = fmaf(wii, dps[u * V + w], cur[u]);
          stv<V>(stT + (c0 + w) * P + r0, cur);
        }
      }
    }
    if (tid < D) {
      float x = 0.0f, dy = 0.0f;
      for (int sl = 0; sl < kCbChunk; ++sl) {
        x = fmaf(sq[sl * P + tid], sdd[sl], x);
        dy += sk[sl * P + tid];
      }
      dw = fmaf(yr, x, dw);
      zacc += x;
      yr += dy;
      zs[tid] = fmaf(wii, dy, zs[tid]);
    }
  }
  float* out = dSp + (bh * g.M + i) * static_cast<int64_t>(E + D);
#pragma unroll
  for (int u = 0; u < V; ++u) {
    float row[V];
#pragma unroll
    for (int w = 0; w < V; ++w) row[w] = acc[u * V + w];
    stv<V>(out + (r0 + u) * D + c0, row);
  }
  if (tid < D) out[E + tid] = zacc;
  dw = warp_sum(dw);
  if (lane == 0) red[warp] = dw;
  __syncthreads();
  if (tid == 0) {
    float s = 0.0f;
    for (int w = 0; w < kCbWarps; ++w) s += red[w];
    diag[bh * g.M + i] = s;
  }
}

// Four consecutive bf16 from global memory (8-byte aligned) as floats: a bf16 is
// the upper half of the float with the same bits.
__device__ __forceinline__ void ld4_bf16(const __nv_bfloat16* p, float (&x)[4]) {
  const uint2 r = *reinterpret_cast<const uint2*>(p);
  x[0] = __uint_as_float(r.x << 16);
  x[1] = __uint_as_float(r.x & 0xffff0000u);
  x[2] = __uint_as_float(r.y << 16);
  x[3] = __uint_as_float(r.y & 0xffff0000u);
}

// Warp-level bf16 tensor-core products for the causal backward's per-chunk
// steps (PTX mma.sync m16n8k16, float32 accumulation).  Fragments are built from
// float32 shared memory, rounded to bf16 (round to nearest even): with
// g = lane / 4 and t = lane % 4, A holds rows g, g + 8 at columns 2t, 2t + 1 and
// 2t + 8, 2t + 9; B holds column g at rows 2t, 2t + 1 and 2t + 8, 2t + 9; the
// accumulator holds rows g, g + 8 at columns 2t, 2t + 1.
__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ void mma_m16n8k16(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// A[m][k] = s[(m0 + m) ld + k0 + k]: rows of A, k contiguous (ld even)
__device__ __forceinline__ void frag_a_rows(const float* s, int ld, int m0, int k0, int lane, uint32_t (&a)[4]) {
  const int g = lane >> 2, t = lane & 3;
  const float* p = s + (m0 + g) * ld + k0 + 2 * t;
  const float2 x0 = *reinterpret_cast<const float2*>(p);
  const float2 x1 = *reinterpret_cast<const float2*>(p + 8 * ld);
  const float2 x2 = *reinterpret_cast<const float2*>(p + 8);
  const float2 x3 = *reinterpret_cast<const float2*>(p + 8 * ld + 8);
  a[0] = bf16x2(x0.x, x0.y);
  a[1] = bf16x2(x1.x, x1.y);
  a[2] = bf16x2(x2.x, x2.y);
  a[3] = bf16x2(x3.x, x3.y);
}
// A[m][k] = s[(k0 + k) ld + m0 + m]: the transpose of rows of k, m contiguous
__device__ __forceinline__ void frag_a_cols(const float* s, int ld, int m0, int k0, int lane, uint32_t (&a)[4]) {
  const int g = lane >> 2, t = lane & 3;
  const float* p = s + (k0 + 2 * t) * ld + m0 + g;
  a[0] = bf16x2(p[0], p[ld]);
  a[1] = bf16x2(p[8], p[ld + 8]);
  a[2] = bf16x2(p[8 * ld], p[9 * ld]);
  a[3] = bf16x2(p[8 * ld + 8], p[9 * ld + 8]);
}
// B[k][n] = s[(n0 + n) ld + k0 + k]: rows of n, k contiguous (ld even)
__device__ __forceinline__ void frag_b_rows(const float* s, int ld, int n0, int k0, int lane, uint32_t (&b)[2]) {
  const int g = lane >> 2, t = lane & 3;
  const float* p = s + (n0 + g) * ld + k0 + 2 * t;
  const float2 x0 = *reinterpret_cast<const float2*>(p);
  const float2 x1 = *reinterpret_cast<const float2*>(p + 8);
  b[0] = bf16x2(x0.x, x0.y);
  b[1] = bf16x2(x1.x, x1.y);
}
// B[k][n] = s[(k0 + k) ld + n0 + n]: rows of k, n contiguous
__device__ __forceinline__ void frag_b_cols(const float* s, int ld, int n0, int k0, int lane, uint32_t (&b)[2]) {
  const int g = lane >> 2, t = lane & 3;
  const float* p = s + (k0 + 2 * t) * ld + n0 + g;
  b[0] = bf16x2(p[0], p[ld]);
  b[1] = bf16x2(p[8 * ld], p[9 * ld]);
}

// The causal backward's query side for bf16 inputs and d = D in {32, 64}: the
// arithmetic of simt_causal_bwd_query_v with its products on warp-level tensor
// cores (operands rounded to bf16 from the float32 rows in shared memory,
// float32 accumulation): the pair dots a = phi(Q) phi(K)^T and e = G V^T,
// u = G C^T, the b sum B phi(K), and per chunk X = phi(Q)^T dnum and
// phi(K)^T V.  The per-token steps (den, g . num, dnum, dden, b, dq) stay on CUDA
// cores between them; the state C is kept row-major, and each warp owns a fixed
// set of 16 x 8 tiles of X, of dS<_i and of the prefix state P.
template <int D>
__global__ void __launch_bounds__(kCbThreads, 3)
simt_causal_bwd_query_mma(const __nv_bfloat16* __restrict__ q, Operand qo, const __nv_bfloat16* __restrict__ k,
                          Operand ko, const __nv_bfloat16* __restrict__ v, Operand vo,
                          const __nv_bfloat16* __restrict__ g_out, Operand go, __nv_bfloat16* __restrict__ dq,
                          Operand dqo, TokenGeom g, int64_t H, int phi_kind, float eps, const float* __restrict__ W,
                          const float* __restrict__ Sp, float* __restrict__ dSp, float* __restrict__ diag,
                          float* __restrict__ dn, const __nv_bfloat16* __restrict__ Stb,
                          const float* __restrict__ ztb) {
  constexpr int V = D / 16;
  constexpr int P = D + 4;                 // padded token / state row (even: 8-byte fragment loads)
  constexpr int CP = kCbChunk + 4;         // padded row of a 32 x 32 token-pair matrix
  constexpr int E = D * D, PD = D + 4;     // PD: the dnum / dden scratch row (16-byte aligned)
  constexpr int NMT = D / 16, NNT = D / 8; // 16 x 8 tiles of a D x D state
  constexpr int WPM = kCbWarps / NMT;      // warps per row tile of the state
  constexpr int NPW = NNT / WPM;           // state tiles per warp (D = 64: 4, D = 32: 1)
  constexpr int TPW = NNT / 4;             // chunk x D tiles per warp (2 row tiles x NNT over 8 warps)
  extern __shared__ __align__(16) float cbm_sm[];
  float* st = cbm_sm;                      // [D][P] C = S<_i + W_ii P before the chunk, row-major
  float* zs = st + D * P;                  // [D]    c = z<_i + W_ii y before the chunk
  float* sq = zs + D;                      // [chunk][P] phi(q_t)
  float* sk = sq + kCbChunk * P;           // [chunk][P] phi(k_s)
  float* sv = sk + kCbChunk * P;           // [chunk][P] v_s
  float* sg = sv + kCbChunk * P;           // [chunk][P] g_t, then dnum_t: each lane of the
  float* sdn = sg;                         //   per-token step reads its own g_t entries first
  float* su = sg + kCbChunk * P;           // [chunk][P] u_t = C g_t, then (B phi(K))_t
  float* sdd = su + kCbChunk * P;          // [chunk]    dden_t
  float* sa = sdd + kCbChunk;              // [chunk][CP] a_ts (s <= t, else 0)
  float* se = sa + kCbChunk * CP;          // [chunk][CP] e_ts, then b_ts (s <= t, else 0)
  float* red = se + kCbChunk * CP;         // [warps]
  uint32_t* qpos = reinterpret_cast<uint32_t*>(red + kCbWarps);   // [chunk][D / 32] bits [q_t > 0]
  const int64_t item = blockIdx.x;
  const int64_t i = item % g.M, bh = item / g.M;
  const int64_t b = bh / H, h = bh % H;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const float wii = __ldg(W + i * g.M + i);
  // S<_i and z<_i: float32 rows of Sp, or (Stb non-null) the tensor-core states
  const int64_t si = bh * g.M + i;
  if (Stb) {
    for (int e = tid; e < E; e += kCbThreads) st[(e / D) * P + e % D] = __bfloat162float(Stb[si * E + e]);
    for (int r = tid; r < D; r += kCbThreads) zs[r] = ztb[si * D + r];
  } else {
    const float* src = Sp + si * static_cast<int64_t>(E + D);
    for (int e = tid; e < E; e += kCbThreads) st[(e / D) * P + e % D] = src[e];
    for (int r = tid; r < D; r += kCbThreads) zs[r] = src[E + r];
  }
  const __nv_bfloat16* qb = q + b * qo.sb + h * qo.sh;
  const __nv_bfloat16* kb = k + b * ko.sb + h * ko.sh;
  const __nv_bfloat16* vb = v + b * vo.sb + h * vo.sh;
  const __nv_bfloat16* gb = g_out + b * go.sb + h * go.sh;
  __nv_bfloat16* dqb = dq + b * dqo.sb + h * dqo.sh;
  float* dnb = dn + (bh * g.M + i) * g.w * PD;   // token rows: dnum_t (D), dden_t
  const int g8 = lane >> 2, t4 = lane & 3;      // accumulator rows g8, g8 + 8; columns 2 t4, 2 t4 + 1
  const int smt = warp / WPM, snt0 = (warp % WPM) * NPW;   // this warp's state tiles
  float pr[NPW][4], acc[NPW][4];
#pragma unroll
  for (int j = 0; j < NPW; ++j)
#pragma unroll
    for (int e4 = 0; e4 < 4; ++e4) pr[j][e4] = acc[j][e4] = 0.0f;
  float yr = 0.0f, zacc = 0.0f, dw = 0.0f;
  const int tt = tid / 16, cc = tid % 16;
  const int t0 = 2 * tt, t1 = t0 + 1;      // per-token steps: tokens t0, t1; columns c0 ..
  const int c0 = V * cc;
  const int srow = tid / kCbRowLanes, spart = tid % kCbRowLanes;
  const int64_t nb = token_of(g, i, 0);    // contiguous blocks: slot s is token nb + s
  // rows that start on 8-byte boundaries load four bf16 at a time
  const bool vec = ((reinterpret_cast<uintptr_t>(qb) | reinterpret_cast<uintptr_t>(kb) |
                     reinterpret_cast<uintptr_t>(vb) | reinterpret_cast<uintptr_t>(gb)) & 7) == 0 &&
                   ((qo.sn | ko.sn | vo.sn | go.sn) & 3) == 0;
  // a chunk x D product of this warp's tiles (rows 16 (warp & 1) .., columns
  // 8 ((warp >> 1) TPW + j)) into rows of dst
  // (scale != 0: dst += scale * product, else dst = product)
  auto chunk_by_d = [&](const float* A, int lda, int kdim, auto load_b, float* dst, float scale) {
    const int mt = warp & 1, ntb = (warp >> 1) * TPW;
    float cf[TPW][4];
#pragma unroll
    for (int j = 0; j < TPW; ++j)
#pragma unroll
      for (int e4 = 0; e4 < 4; ++e4) cf[j][e4] = 0.0f;
    for (int ks = 0; ks < kdim / 16; ++ks) {
      uint32_t af[4];
      frag_a_rows(A, lda, 16 * mt, 16 * ks, lane, af);
#pragma unroll
      for (int j = 0; j < TPW; ++j) {
        uint32_t bf[2];
        load_b(8 * (ntb + j), 16 * ks, bf);
        mma_m16n8k16(cf[j], af, bf);
      }
    }
#pragma unroll
    for (int j = 0; j < TPW; ++j)
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        float2* o2 = reinterpret_cast<float2*>(dst + (16 * mt + g8 + 8 * h2) * P + 8 * (ntb + j) + 2 * t4);
        if (scale != 0.0f) {
          const float2 x = *o2;
          *o2 = make_float2(fmaf(scale, cf[j][2 * h2], x.x), fmaf(scale, cf[j][2 * h2 + 1], x.y));
        } else {
          *o2 = make_float2(cf[j][2 * h2], cf[j][2 * h2 + 1]);
        }
      }
  };
  for (int64_t s0 = 0; s0 < g.w; s0 += kCbChunk) {
    const int cnt = static_cast<int>(g.w - s0 < kCbChunk ? g.w - s0 : kCbChunk);
    const bool more = s0 + kCbChunk < g.w;   // a later chunk of the block reads the advanced state
    __syncthreads();   // the state is complete and the previous chunk's rows are free
    {
      const bool live = srow < cnt;
      const int64_t n = nb + s0 + srow;
#pragma unroll
      for (int c = 4 * spart; c < D; c += 4 * kCbRowLanes) {
        float xq[4], xk[4], xv[4], xg[4];
        if (!live) {
#pragma unroll
          for (int u = 0; u < 4; ++u) xq[u] = xk[u] = xv[u] = xg[u] = 0.0f;
        } else if (vec) {
          ld4_bf16(qb + n * qo.sn + c, xq);
          ld4_bf16(kb + n * ko.sn + c, xk);
          ld4_bf16(vb + n * vo.sn + c, xv);
          ld4_bf16(gb + n * go.sn + c, xg);
        } else {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            xq[u] = load_f(qb + n * qo.sn + c + u);
            xk[u] = load_f(kb + n * ko.sn + c + u);
            xv[u] = load_f(vb + n * vo.sn + c + u);
            xg[u] = load_f(gb + n * go.sn + c + u);
          }
        }
        uint32_t pos = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          pos |= (xq[u] > 0.0f ? 1u : 0u) << u;
          xq[u] = live ? phi_f(xq[u], phi_kind, eps) : 0.0f;
          xk[u] = live ? phi_f(xk[u], phi_kind, eps) : 0.0f;
        }
        // the eight lanes of this row hold columns c % 32 = 4 spart .. of one word
        pos <<= (c & 31);
#pragma unroll
        for (int off = 1; off < kCbRowLanes; off <<= 1) pos |= __shfl_xor_sync(0xffffffffu, pos, off);
        if (spart == 0) qpos[srow * (D / 32) + c / 32] = pos;
        stv<4>(sq + srow * P + c, xq);
        stv<4>(sk + srow * P + c, xk);
        stv<4>(sv + srow * P + c, xv);
        stv<4>(sg + srow * P + c, xg);
      }
    }
    __syncthreads();
    // ---- 1: a = phi(Q) phi(K)^T (warps 0-3) and e = G V^T (warps 4-7), kept for s <= t
    {
      const int mat = warp >> 2, mt = (warp >> 1) & 1, nt0 = (warp & 1) * 2;
      const float* A = mat ? sg : sq;
      const float* Bm = mat ? sv : sk;
      float* dst = mat ? se : sa;
      float cf[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4) cf[j][e4] = 0.0f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t af[4];
        frag_a_rows(A, P, 16 * mt, 16 * ks, lane, af);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          uint32_t bf[2];
          frag_b_rows(Bm, P, 8 * (nt0 + j), 16 * ks, lane, bf);
          mma_m16n8k16(cf[j], af, bf);
        }
      }
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4) {
          const int row = 16 * mt + g8 + 8 * (e4 >> 1), col = 8 * (nt0 + j) + 2 * t4 + (e4 & 1);
          dst[row * CP + col] = (row < cnt && col <= row) ? cf[j][e4] : 0.0f;
        }
    }
    __syncthreads();
    // ---- 2: u = G C^T into su (B[c][r] = C[r][c], rows of C)
    chunk_by_d(sg, P, D, [&](int n0, int k0, uint32_t(&bf)[2]) { frag_b_rows(st, P, n0, k0, lane, bf); }, su,
               0.0f);
    __syncthreads();
    // ---- 3: per token (tokens t0, t1 in turn on the 16 lanes of a half-warp; columns /
    // rows c0 ..): den_t, g_t . num_t, dnum_t, dden_t, b_ts, dW_ii's own-chunk part; the
    // lane's entries of u_t are replaced by those of C dnum_t + dden_t c, and of g_t by
    // those of dnum_t
    {
      float zv[V];
      ldv<V>(zs + c0, zv);
#pragma unroll 1
      for (int tk = 0; tk < 2; ++tk) {
        const int tq = t0 + tk;
        float uu[V], qv[V], gv[V];
        ldv<V>(su + tq * P + c0, uu);
        ldv<V>(sq + tq * P + c0, qv);
        ldv<V>(sg + tq * P + c0, gv);
        float den = 0.0f, gov = 0.0f;
#pragma unroll
        for (int w = 0; w < V; ++w) {
          den = fmaf(qv[w], zv[w], den);
          gov = fmaf(qv[w], uu[w], gov);
        }
        // this lane's own-chunk sources s = cc, cc + 16
        const float aa = sa[tq * CP + cc], ab = sa[tq * CP + cc + 16];
        const float ea = se[tq * CP + cc], eb = se[tq * CP + cc + 16];
        den = fmaf(wii, aa + ab, den);
        gov = fmaf(wii, fmaf(aa, ea, ab * eb), gov);
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) {   // the 16 lanes of this half-warp share the token
          den += __shfl_xor_sync(0xffffffffu, den, off);
          gov += __shfl_xor_sync(0xffffffffu, gov, off);
        }
        den += eps;
        const bool live = tq < cnt;   // rows past the block stay zero
        const float rd = 1.0f / den;  // one division per token
        const float dd = live ? -(gov * rd) * rd : 0.0f;
        float dnv[V], xv[V];
#pragma unroll
        for (int w = 0; w < V; ++w) {
          dnv[w] = live ? gv[w] * rd : 0.0f;
          xv[w] = fmaf(dd, zv[w], uu[w] * rd);
        }
        stv<V>(sdn + tq * P + c0, dnv);
        stv<V>(su + tq * P + c0, xv);
        if (live) stv<V>(dnb + (s0 + tq) * PD + c0, dnv);
        if (cc == 0) {
          sdd[tq] = dd;
          if (live) dnb[(s0 + tq) * PD + D] = dd;
        }
        // b_ts = e_ts / den_t + dden_t (s <= t) in place of e_ts; dW_ii's own-chunk part
        const float ba = (live && cc <= tq) ? fmaf(ea, rd, dd) : 0.0f;
        const float bb = (live && cc + 16 <= tq) ? fmaf(eb, rd, dd) : 0.0f;
        se[tq * CP + cc] = ba;
        se[tq * CP + cc + 16] = bb;
        dw = fmaf(aa, ba, dw);
        dw = fmaf(ab, bb, dw);
      }
    }
    __syncthreads();
    // ---- 4: su += W_ii B phi(K) (B[s][r] = phi(k_s)[r], rows of phi(K)): dq before its mask
    chunk_by_d(se, CP, kCbChunk, [&](int n0, int k0, uint32_t(&bf)[2]) { frag_b_cols(sk, P, n0, k0, lane, bf); },
               su, wii);
    __syncthreads();
    // ---- 5: dq_t = (u_t / den_t + dden_t c + W_ii Y_t) [q_t > 0] (tokens t0, t1; rows c0 ..)
    {
      float w0[V], w1[V];
      ldv<V>(su + t0 * P + c0, w0);
      ldv<V>(su + t1 * P + c0, w1);
      const int64_t n0t = nb + s0 + t0, n1t = nb + s0 + t1;
#pragma unroll
      for (int w = 0; w < V; ++w) {
        const int r = c0 + w;
        if (t0 < cnt)
          store_f(dqb + n0t * dqo.sn + r, (qpos[t0 * (D / 32) + r / 32] >> (r & 31)) & 1u ? w0[w] : 0.0f);
        if (t1 < cnt)
          store_f(dqb + n1t * dqo.sn + r, (qpos[t1 * (D / 32) + r / 32] >> (r & 31)) & 1u ? w1[w] : 0.0f);
      }
    }
    // ---- 6: X = phi(Q)^T dnum over this warp's state tiles (no barrier before: steps 2
    // to 5 are done with C): dS<_i += X, dW_ii += <P, X>; then, unless the block ends
    // here, phi(K)^T V: P and C advance
    {
      float X[NPW][4];
#pragma unroll
      for (int j = 0; j < NPW; ++j)
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4) X[j][e4] = 0.0f;
#pragma unroll
      for (int ks = 0; ks < kCbChunk / 16; ++ks) {
        uint32_t aq[4];
        frag_a_cols(sq, P, 16 * smt, 16 * ks, lane, aq);   // A[r][t] = phi(q_t)[r]
#pragma unroll
        for (int j = 0; j < NPW; ++j) {
          uint32_t bn[2];
          frag_b_cols(sdn, P, 8 * (snt0 + j), 16 * ks, lane, bn);   // B[t][c] = dnum_t[c]
          mma_m16n8k16(X[j], aq, bn);
        }
      }
#pragma unroll
      for (int j = 0; j < NPW; ++j)
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4) {
          dw = fmaf(pr[j][e4], X[j][e4], dw);
          acc[j][e4] += X[j][e4];
        }
    }
    if (more) {
      float dps[NPW][4];
#pragma unroll
      for (int j = 0; j < NPW; ++j)
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4) dps[j][e4] = 0.0f;
#pragma unroll
      for (int ks = 0; ks < kCbChunk / 16; ++ks) {
        uint32_t ak[4];
        frag_a_cols(sk, P, 16 * smt, 16 * ks, lane, ak);   // A[r][s] = phi(k_s)[r]
#pragma unroll
        for (int j = 0; j < NPW; ++j) {
          uint32_t bv[2];
          frag_b_cols(sv, P, 8 * (snt0 + j), 16 * ks, lane, bv);   // B[s][c] = v_s[c]
          mma_m16n8k16(dps[j], ak, bv);
        }
      }
#pragma unroll
      for (int j = 0; j < NPW; ++j)
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4) {
          pr[j][e4] += dps[j][e4];
          float* cs = st + (16 * smt + g8 + 8 * (e4 >> 1)) * P + 8 * (snt0 + j) + 2 * t4 + (e4 & 1);
          *cs = fmaf(wii, dps[j][e4], *cs);
        }
    }
    if (tid < D) {
      float x = 0.0f, dy = 0.0f;
      for (int sl = 0; sl < kCbChunk; ++sl) {
        x = fmaf(sq[sl * P + tid], sdd[sl], x);
        dy += sk[sl * P + tid];
      }
      dw = fmaf(yr, x, dw);
      zacc += x;
      yr += dy;
      zs[tid] = fmaf(wii, dy, zs[tid]);
    }
  }
  float* out = dSp + (bh * g.M + i) * static_cast<int64_t>(E + D);
#pragma unroll
  for (int j = 0; j < NPW; ++j)
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2)
      *reinterpret_cast<float2*>(out + (16 * smt + g8 + 8 * h2) * D + 8 * (snt0 + j) + 2 * t4) =
          make_float2(acc[j][2 * h2], acc[j][2 * h2 + 1]);
  if (tid < D) out[E + tid] = zacc;
  dw = warp_sum(dw);
  if (lane == 0) red[warp] = dw;
  __syncthreads();
  if (tid == 0) {
    float s = 0.0f;
    for (int w = 0; w < kCbWarps; ++w) s += red[w];
    diag[bh * g.M + i] = s;
  }
}

// The same arithmetic as simt_causal_bwd_key for d = D in {32, 64}, laid out as
// simt_causal_bwd_query_v: padded rows, 16-byte vectors, G kept row-major and
// transposed (G feeds dv, G^T feeds dk), token-pair tiles {p, p + 16} x
// {q, q + 16}, zero rows past the block's end; the block's first chunk (the
// last one taken) skips the update of G.
template <typename T, int D>
__global__ void __launch_bounds__(kCbThreads, 2)
simt_causal_bwd_key_v(const T* __restrict__ q, Operand qo, const T* __restrict__ k, Operand ko,
                      const T* __restrict__ v, Operand vo, T* __restrict__ dk, Operand dko, T* __restrict__ dv,
                      Operand dvo, TokenGeom g, int64_t H, int phi_kind, float eps, const float* __restrict__ W,
                      const float* __restrict__ dS, const float* __restrict__ dn,
                      const __nv_bfloat16* __restrict__ Stb, const float* __restrict__ ztb) {
  constexpr int V = D / 16;
  constexpr int P = D + 4;
  constexpr int CP = kCbChunk + 4;
  constexpr int E = D * D, PD = D + 1;
  extern __shared__ __align__(16) float cbk_sm[];
  float* gs = cbk_sm;                      // [D][P] G
  float* gsT = gs + D * P;                 // [D][P] G^T
  float* gz = gsT + D * P;                 // [D]    gz
  float* sq = gz + D;                      // [chunk][P] phi(q_t)
  float* sdn = sq + kCbChunk * P;          // [chunk][P] dnum_t
  float* sk = sdn + kCbChunk * P;          // [chunk][P] phi(k_s)
  float* sv = sk + kCbChunk * P;           // [chunk][P] v_s
  float* sdd = sv + kCbChunk * P;          // [chunk]    dden_t
  float* sa = sdd + kCbChunk;              // [chunk][CP] a_st (t >= s, else 0)
  float* sb = sa + kCbChunk * CP;          // [chunk][CP] b_st (t >= s, else 0)
  const int64_t item = blockIdx.x;
  const int64_t j = item % g.M, bh = item / g.M;
  const int64_t b = bh / H, h = bh % H;
  const int tid = threadIdx.x;
  const float wjj = __ldg(W + j * g.M + j);
  // dS_j and dz_j: float32 rows of dS, or (Stb non-null) the tensor-core mixing's
  // output (bf16 row-major dS_j, float32 dz_j)
  const int64_t sj = bh * g.M + j;
  const float* src = dS + sj * static_cast<int64_t>(E + D);
  for (int e = tid; e < E; e += kCbThreads) {
    const int r = e / D, c = e % D;
    const float x = Stb ? __bfloat162float(Stb[sj * E + e]) : src[e];
    gs[r * P + c] = x;
    gsT[c * P + r] = x;
  }
  for (int r = tid; r < D; r += kCbThreads) gz[r] = Stb ? ztb[sj * D + r] : src[E + r];
  const T* qb = q + b * qo.sb + h * qo.sh;
  const T* kb = k + b * ko.sb + h * ko.sh;
  const T* vb = v + b * vo.sb + h * vo.sh;
  T* dkb = dk + b * dko.sb + h * dko.sh;
  T* dvb = dv + b * dvo.sb + h * dvo.sh;
  const float* dnb = dn + (bh * g.M + j) * g.w * PD;
  const int tt = tid / 16, cc = tid % 16;
  const int c0 = V * cc;                   // columns c0 .. of the dv / dk and state steps
  const int r0 = V * tt;                   // state tile: rows r0 .., columns c0 ..
  const int pi = tid / 16, pj = tid % 16;  // pair tiles: sources pi, pi + 16; queries pj, pj + 16
  const int srow = tid / kCbRowLanes, spart = tid % kCbRowLanes;
  const int64_t nb = token_of(g, j, 0);
  const int64_t nch = (g.w + kCbChunk - 1) / kCbChunk;
  for (int64_t ci = nch - 1; ci >= 0; --ci) {
    const int64_t s0 = ci * kCbChunk;
    const int cnt = static_cast<int>(g.w - s0 < kCbChunk ? g.w - s0 : kCbChunk);
    __syncthreads();   // the suffix state is complete and the later chunk's rows are free
    {
      const bool live = srow < cnt;
      const int64_t n = nb + s0 + srow;
#pragma unroll
      for (int c = 4 * spart; c < D; c += 4 * kCbRowLanes) {
        float xq[4], xn[4], xk[4], xv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          xq[u] = live ? phi_f(load_f(qb + n * qo.sn + c + u), phi_kind, eps) : 0.0f;
          xn[u] = live ? dnb[(s0 + srow) * PD + c + u] : 0.0f;
          xk[u] = live ? phi_f(load_f(kb + n * ko.sn + c + u), phi_kind, eps) : 0.0f;
          xv[u] = live ? load_f(vb + n * vo.sn + c + u) : 0.0f;
        }
        stv<4>(sq + srow * P + c, xq);
        stv<4>(sdn + srow * P + c, xn);
        stv<4>(sk + srow * P + c, xk);
        stv<4>(sv + srow * P + c, xv);
      }
    }
    if (tid < kCbChunk) sdd[tid] = tid < cnt ? dnb[(s0 + tid) * PD + D] : 0.0f;
    __syncthreads();
    // ---- 1: a_st and b_st (t >= s); the block (pi + 16, pj) lies below the diagonal
    {
      const int ra = pi, rb = pi + 16, ca = pj, cb = pj + 16;
      float a00 = 0.0f, a01 = 0.0f, a11 = 0.0f, b00 = 0.0f, b01 = 0.0f, b11 = 0.0f;
#pragma unroll 2
      for (int r = 0; r < D; r += V) {
        float ka[V], kc[V], qa[V], qc[V], va[V], vc[V], na[V], nc[V];
        ldv<V>(sk + ra * P + r, ka);
        ldv<V>(sk + rb * P + r, kc);
        ldv<V>(sq + ca * P + r, qa);
        ldv<V>(sq + cb * P + r, qc);
        ldv<V>(sv + ra * P + r, va);
        ldv<V>(sv + rb * P + r, vc);
        ldv<V>(sdn + ca * P + r, na);
        ldv<V>(sdn + cb * P + r, nc);
#pragma unroll
        for (int u = 0; u < V; ++u) {
          a00 = fmaf(ka[u], qa[u], a00);
          a01 = fmaf(ka[u], qc[u], a01);
          a11 = fmaf(kc[u], qc[u], a11);
          b00 = fmaf(va[u], na[u], b00);
          b01 = fmaf(va[u], nc[u], b01);
          b11 = fmaf(vc[u], nc[u], b11);
        }
      }
      const float dda = sdd[ca], ddc = sdd[cb];
      const bool m00 = ca < cnt && ca >= ra, m01 = cb < cnt, m11 = cb < cnt && cb >= rb;
      sa[ra * CP + ca] = m00 ? a00 : 0.0f;
      sa[ra * CP + cb] = m01 ? a01 : 0.0f;
      sa[rb * CP + ca] = 0.0f;
      sa[rb * CP + cb] = m11 ? a11 : 0.0f;
      sb[ra * CP + ca] = m00 ? b00 + dda : 0.0f;
      sb[ra * CP + cb] = m01 ? b01 + ddc : 0.0f;
      sb[rb * CP + ca] = 0.0f;
      sb[rb * CP + cb] = m11 ? b11 + ddc : 0.0f;
    }
    __syncthreads();
    // ---- 2: warps 0-3 form dv, warps 4-7 dk; a thread takes 4 sources x V columns:
    //   dv_s[c] = sum_x phi(k_s)[x] G[x][c] + W_jj sum_t a_st dnum_t[c]
    //   dk_s[r] = (sum_x G[r][x] v_s[x] + gz[r] + W_jj sum_t b_st phi(q_t)[r]) [k_s > 0]
    {
      const bool kside = tid >= kCbThreads / 2;
      const int sb4 = 4 * ((tid % (kCbThreads / 2)) / 16);   // sources sb4 .. sb4 + 3
      const float* opd = kside ? sv : sk;
      const float* gm = kside ? gsT : gs;                    // gm[x][c0 + w]: G[x][c] or G[r][x]
      const float* pm = kside ? sb : sa;
      const float* tm = kside ? sq : sdn;
      float ga[4][V], pa[4][V];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj)
#pragma unroll
        for (int w = 0; w < V; ++w) ga[jj][w] = pa[jj][w] = 0.0f;
#pragma unroll 2
      for (int x = 0; x < D; x += V) {
        float o[4][V];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) ldv<V>(opd + (sb4 + jj) * P + x, o[jj]);
#pragma unroll
        for (int u = 0; u < V; ++u) {
          float gv[V];
          ldv<V>(gm + (x + u) * P + c0, gv);
#pragma unroll
          for (int jj = 0; jj < 4; ++jj)
#pragma unroll
            for (int w = 0; w < V; ++w) ga[jj][w] = fmaf(o[jj][u], gv[w], ga[jj][w]);
        }
      }
#pragma unroll 2
      for (int t = 0; t < kCbChunk; t += V) {
        float pv[4][V];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) ldv<V>(pm + (sb4 + jj) * CP + t, pv[jj]);
#pragma unroll
        for (int u = 0; u < V; ++u) {
          float tv[V];
          ldv<V>(tm + (t + u) * P + c0, tv);
#pragma unroll
          for (int jj = 0; jj < 4; ++jj)
#pragma unroll
            for (int w = 0; w < V; ++w) pa[jj][w] = fmaf(pv[jj][u], tv[w], pa[jj][w]);
        }
      }
      float zv[V];
      ldv<V>(gz + c0, zv);
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int s = sb4 + jj;
        if (s < cnt) {
          const int64_t n = nb + s0 + s;
#pragma unroll
          for (int w = 0; w < V; ++w) {
            const int c = c0 + w;
            if (kside) {
              const float x = fmaf(wjj, pa[jj][w], ga[jj][w] + zv[w]);
              store_f(dkb + n * dko.sn + c, load_f(kb + n * ko.sn + c) > 0.0f ? x : 0.0f);
            } else {
              store_f(dvb + n * dvo.sn + c, fmaf(wjj, pa[jj][w], ga[jj][w]));
            }
          }
        }
      }
    }
    if (ci == 0) break;   // the block's first chunk: nothing reads the suffix state after it
    __syncthreads();      // phase 3 rewrites G, which phase 2 has read
    // ---- 3: G += W_jj sum_t phi(q_t) dnum_t^T (V x V entries per thread), gz likewise
    {
      float X[V * V];
#pragma unroll
      for (int m = 0; m < V * V; ++m) X[m] = 0.0f;
#pragma unroll 4
      for (int t = 0; t < kCbChunk; ++t) {
        float qr[V], nc[V];
        ldv<V>(sq + t * P + r0, qr);
        ldv<V>(sdn + t * P + c0, nc);
#pragma unroll
        for (int u = 0; u < V; ++u)
#pragma unroll
          for (int w = 0; w < V; ++w) X[u * V + w] = fmaf(qr[u], nc[w], X[u * V + w]);
      }
#pragma unroll
      for (int u = 0; u < V; ++u) {
        float cur[V];
        ldv<V>(gs + (r0 + u) * P + c0, cur);
#pragma unroll
        for (int w = 0; w < V; ++w) cur[w] = fmaf(wjj, X[u * V + w], cur[w]);
        stv<V>(gs + (r0 + u) * P + c0, cur);
      }
#pragma unroll
      for (int w = 0; w < V; ++w) {
        float cur[V];
        ldv<V>(gsT + (c0 + w) * P + r0, cur);
#pragma unroll
        for (int u = 0; u < V; ++u) cur[u] = fmaf(wjj, X[u * V + w], cur[u]);
        stv<V>(gsT + (c0 + w) * P + r0, cur);
      }
    }
    if (tid < D) {
      float x = 0.0f;
      for (int t = 0; t < kCbChunk; ++t) x = fmaf(sdd[t], sq[t * P + tid], x);
      gz[tid] = fmaf(wjj, x, gz[tid]);
    }
  }
}

// The causal backward's key side for bf16 inputs and d = D in {32, 64}: the
// arithmetic of simt_causal_bwd_key_v with its products on warp-level tensor
// cores (operands rounded to bf16 from the float32 rows in shared memory,
// float32 accumulation): the pair dots a = phi(K) phi(Q)^T and b = V dnum^T
// (+ dden_t), kept scaled by W_jj, dv = phi(K) G + (W_jj a) dnum and
// dk = V G^T + (W_jj b) phi(Q) (G row-major serves both; each in one
// accumulator), and the suffix-state update phi(Q)^T dnum.  dv and dk go from
// the accumulators to global memory.
template <int D>
__global__ void __launch_bounds__(kCbThreads, 3)
simt_causal_bwd_key_mma(const __nv_bfloat16* __restrict__ q, Operand qo, const __nv_bfloat16* __restrict__ k,
                        Operand ko, const __nv_bfloat16* __restrict__ v, Operand vo, __nv_bfloat16* __restrict__ dk,
                        Operand dko, __nv_bfloat16* __restrict__ dv, Operand dvo, TokenGeom g, int64_t H, int phi_kind,
                        float eps, const float* __restrict__ W, const float* __restrict__ dS,
                        const float* __restrict__ dn, const __nv_bfloat16* __restrict__ Stb,
                        const float* __restrict__ ztb) {
  constexpr int P = D + 4;
  constexpr int CP = kCbChunk + 4;
  constexpr int E = D * D, PD = D + 4;     // the dnum / dden scratch row (16-byte aligned)
  constexpr int NMT = D / 16, NNT = D / 8; // 16 x 8 tiles of a D x D state
  constexpr int WPM = kCbWarps / NMT;      // warps per row tile of the state
  constexpr int NPW = NNT / WPM;           // state tiles per warp
  constexpr int OPW = NNT / 2;             // chunk x D tiles per warp of a warp half (2 row tiles x NNT over 4)
  extern __shared__ __align__(16) float ckm_sm[];
  float* gs = ckm_sm;                      // [D][P] G = dS_j + W_jj sum over later chunks, row-major
  float* gz = gs + D * P;                  // [D]    gz
  float* sq = gz + D;                      // [chunk][P] phi(q_t)
  float* sdn = sq + kCbChunk * P;          // [chunk][P] dnum_t
  float* sk = sdn + kCbChunk * P;          // [chunk][P] phi(k_s)
  float* sv = sk + kCbChunk * P;           // [chunk][P] v_s
  float* sdd = sv + kCbChunk * P;          // [chunk]    dden_t
  float* sa = sdd + kCbChunk;              // [chunk][CP] W_jj a_st (t >= s, else 0)
  float* sb = sa + kCbChunk * CP;          // [chunk][CP] W_jj b_st (t >= s, else 0)
  uint32_t* kpos = reinterpret_cast<uint32_t*>(sb + kCbChunk * CP);   // [chunk][D / 32] bits [k_s > 0]
  const int64_t item = blockIdx.x;
  const int64_t j = item % g.M, bh = item / g.M;
  const int64_t b = bh / H, h = bh % H;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const float wjj = __ldg(W + j * g.M + j);
  // dS_j and dz_j: float32 rows of dS, or (Stb non-null) the tensor-core mixing's
  // output (bf16 row-major dS_j, float32 dz_j)
  const int64_t sj = bh * g.M + j;
  const float* src = dS + sj * static_cast<int64_t>(E + D);
  for (int e = tid; e < E; e += kCbThreads)
    gs[(e / D) * P + e % D] = Stb ? __bfloat162float(Stb[sj * E + e]) : src[e];
  for (int r = tid; r < D; r += kCbThreads) gz[r] = Stb ? ztb[sj * D + r] : src[E + r];
  const __nv_bfloat16* qb = q + b * qo.sb + h * qo.sh;
  const __nv_bfloat16* kb = k + b * ko.sb + h * ko.sh;
  const __nv_bfloat16* vb = v + b * vo.sb + h * vo.sh;
  __nv_bfloat16* dkb = dk + b * dko.sb + h * dko.sh;
  __nv_bfloat16* dvb = dv + b * dvo.sb + h * dvo.sh;
  const float* dnb = dn + (bh * g.M + j) * g.w * PD;
  const int g8 = lane >> 2, t4 = lane & 3;
  const int smt = warp / WPM, snt0 = (warp % WPM) * NPW;   // this warp's state tiles
  const int srow = tid / kCbRowLanes, spart = tid % kCbRowLanes;
  const int64_t nb = token_of(g, j, 0);
  const int64_t nch = (g.w + kCbChunk - 1) / kCbChunk;
  // rows that start on 8-byte boundaries load four bf16 at a time
  const bool vec = ((reinterpret_cast<uintptr_t>(qb) | reinterpret_cast<uintptr_t>(kb) |
                     reinterpret_cast<uintptr_t>(vb)) & 7) == 0 &&
                   ((qo.sn | ko.sn | vo.sn) & 3) == 0;
  for (int64_t ci = nch - 1; ci >= 0; --ci) {
    const int64_t s0 = ci * kCbChunk;
    const int cnt = static_cast<int>(g.w - s0 < kCbChunk ? g.w - s0 : kCbChunk);
    __syncthreads();   // the suffix state is complete and the later chunk's rows are free
    {
      const bool live = srow < cnt;
      const int64_t n = nb + s0 + srow;
#pragma unroll
      for (int c = 4 * spart; c < D; c += 4 * kCbRowLanes) {
        float xq[4], xn[4], xk[4], xv[4];
        if (!live) {
#pragma unroll
          for (int u = 0; u < 4; ++u) xq[u] = xn[u] = xk[u] = xv[u] = 0.0f;
        } else {
          ldv<4>(dnb + (s0 + srow) * PD + c, xn);
          if (vec) {
            ld4_bf16(qb + n * qo.sn + c, xq);
            ld4_bf16(kb + n * ko.sn + c, xk);
            ld4_bf16(vb + n * vo.sn + c, xv);
          } else {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              xq[u] = load_f(qb + n * qo.sn + c + u);
              xk[u] = load_f(kb + n * ko.sn + c + u);
              xv[u] = load_f(vb + n * vo.sn + c + u);
            }
          }
        }
        uint32_t pos = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          pos |= (xk[u] > 0.0f ? 1u : 0u) << u;
          xq[u] = live ? phi_f(xq[u], phi_kind, eps) : 0.0f;
          xk[u] = live ? phi_f(xk[u], phi_kind, eps) : 0.0f;
        }
        pos <<= (c & 31);   // one word's columns over the eight lanes of this row
#pragma unroll
        for (int off = 1; off < kCbRowLanes; off <<= 1) pos |= __shfl_xor_sync(0xffffffffu, pos, off);
        if (spart == 0) kpos[srow * (D / 32) + c / 32] = pos;
        stv<4>(sq + srow * P + c, xq);
        stv<4>(sdn + srow * P + c, xn);
        stv<4>(sk + srow * P + c, xk);
        stv<4>(sv + srow * P + c, xv);
      }
    }
    if (tid < kCbChunk) sdd[tid] = tid < cnt ? dnb[(s0 + tid) * PD + D] : 0.0f;
    __syncthreads();
    // ---- 1: a = phi(K) phi(Q)^T (warps 0-3) and b = V dnum^T + dden_t (warps 4-7), kept for t >= s
    {
      const int mat = warp >> 2, mt = (warp >> 1) & 1, nt0 = (warp & 1) * 2;
      const float* A = mat ? sv : sk;
      const float* Bm = mat ? sdn : sq;
      float* dst = mat ? sb : sa;
      float cf[2][4];
#pragma unroll
      for (int jj = 0; jj < 2; ++jj)
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4) cf[jj][e4] = 0.0f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t af[4];
        frag_a_rows(A, P, 16 * mt, 16 * ks, lane, af);
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          uint32_t bf[2];
          frag_b_rows(Bm, P, 8 * (nt0 + jj), 16 * ks, lane, bf);
          mma_m16n8k16(cf[jj], af, bf);
        }
      }
#pragma unroll
      for (int jj = 0; jj < 2; ++jj)
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4) {
          const int row = 16 * mt + g8 + 8 * (e4 >> 1), col = 8 * (nt0 + jj) + 2 * t4 + (e4 & 1);
          const bool keep = col < cnt && col >= row;   // source row s, query col t >= s
          dst[row * CP + col] = keep ? wjj * (cf[jj][e4] + (mat ? sdd[col] : 0.0f)) : 0.0f;
        }
    }
    __syncthreads();
    // ---- 2: dv (warps 0-3) and dk (warps 4-7) of this warp's tiles, straight to memory:
    //   dv_s = sum_x phi(k_s)[x] G[x][.] + W_jj sum_t a_st dnum_t
    //   dk_s = (sum_x G[.][x] v_s[x] + gz + W_jj sum_t b_st phi(q_t)) [k_s > 0]
    {
      const bool kside = warp >= kCbWarps / 2;
      const int mt = warp & 1, ntb = ((warp >> 1) & 1) * OPW;
      float c1[OPW][4];   // both products (the pair matrices carry W_jj) in one accumulator
#pragma unroll
      for (int jj = 0; jj < OPW; ++jj)
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4) c1[jj][e4] = 0.0f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t af[4];
        frag_a_rows(kside ? sv : sk, P, 16 * mt, 16 * ks, lane, af);
#pragma unroll
        for (int jj = 0; jj < OPW; ++jj) {
          uint32_t bf[2];
          if (kside)
            frag_b_rows(gs, P, 8 * (ntb + jj), 16 * ks, lane, bf);   // B[x][r] = G[r][x]
          else
            frag_b_cols(gs, P, 8 * (ntb + jj), 16 * ks, lane, bf);   // B[x][c] = G[x][c]
          mma_m16n8k16(c1[jj], af, bf);
        }
      }
#pragma unroll
      for (int ks = 0; ks < kCbChunk / 16; ++ks) {
        uint32_t af[4];
        frag_a_rows(kside ? sb : sa, CP, 16 * mt, 16 * ks, lane, af);
#pragma unroll
        for (int jj = 0; jj < OPW; ++jj) {
          uint32_t bf[2];
          frag_b_cols(kside ? sq : sdn, P, 8 * (ntb + jj), 16 * ks, lane, bf);   // B[t][.] = row t
          mma_m16n8k16(c1[jj], af, bf);
        }
      }
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int s = 16 * mt + g8 + 8 * h2;
        if (s < cnt) {
          const int64_t n = nb + s0 + s;
#pragma unroll
          for (int jj = 0; jj < OPW; ++jj) {
            const int c = 8 * (ntb + jj) + 2 * t4;
            float x0 = c1[jj][2 * h2], x1 = c1[jj][2 * h2 + 1];
            if (kside) {
              const uint32_t word = kpos[s * (D / 32) + c / 32] >> (c & 31);
              x0 = word & 1u ? x0 + gz[c] : 0.0f;
              x1 = word & 2u ? x1 + gz[c + 1] : 0.0f;
              store_f(dkb + n * dko.sn + c, x0);
              store_f(dkb + n * dko.sn + c + 1, x1);
            } else {
              store_f(dvb + n * dvo.sn + c, x0);
              store_f(dvb + n * dvo.sn + c + 1, x1);
            }
          }
        }
      }
    }
    if (ci == 0) break;   // the block's first chunk: nothing reads the suffix state after it
    __syncthreads();      // the G update below rewrites G, which step 2 has read
    // ---- 3: G += W_jj phi(Q)^T dnum over this warp's state tiles, gz likewise
    {
      float X[NPW][4];
#pragma unroll
      for (int jj = 0; jj < NPW; ++jj)
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4) X[jj][e4] = 0.0f;
#pragma unroll
      for (int ks = 0; ks < kCbChunk / 16; ++ks) {
        uint32_t aq[4];
        frag_a_cols(sq, P, 16 * smt, 16 * ks, lane, aq);   // A[r][t] = phi(q_t)[r]
#pragma unroll
        for (int jj = 0; jj < NPW; ++jj) {
          uint32_t bn[2];
          frag_b_cols(sdn, P, 8 * (snt0 + jj), 16 * ks, lane, bn);   // B[t][c] = dnum_t[c]
          mma_m16n8k16(X[jj], aq, bn);
        }
      }
#pragma unroll
      for (int jj = 0; jj < NPW; ++jj)
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4) {
          float* gp = gs + (16 * smt + g8 + 8 * (e4 >> 1)) * P + 8 * (snt0 + jj) + 2 * t4 + (e4 & 1);
          *gp = fmaf(wjj, X[jj][e4], *gp);
        }
    }
    if (tid < D) {
      float x = 0.0f;
      for (int t = 0; t < kCbChunk; ++t) x = fmaf(sdd[t], sq[t * P + tid], x);
      gz[tid] = fmaf(wjj, x, gz[tid]);
    }
  }
}

// Shared memory of the vector-layout causal backward kernels, d = D.
constexpr size_t cbv_query_smem(int D) {
  return static_cast<size_t>(D * (D + 4) + D + 5 * kCbChunk * (D + 4) + kCbChunk + 2 * kCbChunk * (kCbChunk + 4) +
                             kCbWarps) *
         sizeof(float);
}
constexpr size_t cbm_query_smem(int D) {
  return static_cast<size_t>(D * (D + 4) + D + 5 * kCbChunk * (D + 4) + kCbChunk + 2 * kCbChunk * (kCbChunk + 4) +
                             kCbWarps + kCbChunk * (D / 32)) *
         sizeof(float);
}
constexpr size_t cbm_key_smem(int D) {
  return static_cast<size_t>(D * (D + 4) + D + 4 * kCbChunk * (D + 4) + kCbChunk + 2 * kCbChunk * (kCbChunk + 4) +
                             kCbChunk * (D / 32)) *
         sizeof(float);
}
constexpr size_t cbv_key_smem(int D) {
  return static_cast<size_t>(2 * D * (D + 4) + D + 4 * kCbChunk * (D + 4) + kCbChunk +
                             2 * kCbChunk * (kCbChunk + 4)) *
         sizeof(float);
}

// Causal dW: the partials below the diagonal, the query kernel's W_ii shares
// on it, zero above it; summed in a fixed order, laid out as simt_dw_reduce.
__global__ void __launch_bounds__(kDwrWarps * 32)
simt_dw_reduce_causal(const float* __restrict__ part, const float* __restrict__ diag, float* __restrict__ dW,
                      int64_t M, int64_t BH, int64_t KS) {
  __shared__ float red[kDwrWarps][32];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t MM = M * M;
  const int64_t x = static_cast<int64_t>(blockIdx.x) * 32 + lane;
  const int64_t i = x / M, j = x % M;
  float s = 0.0f;
  if (x < MM && j < i)
    for (int64_t n = warp; n < BH * KS; n += kDwrWarps) s += part[n * MM + x];
  else if (x < MM && j == i)
    for (int64_t bh = warp; bh < BH; bh += kDwrWarps) s += diag[bh * M + i];
  red[warp][lane] = s;
  __syncthreads();
  if (warp == 0 && x < MM) {
    float r = 0.0f;
    for (int w = 0; w < kDwrWarps; ++w) r += red[w][lane];
    dW[x] = r;
  }
}

template <typename T>
int launch_simt_typed(const Problem& p, const float* W, const SimtWorkspace& ws, cudaStream_t stream) {
  const TokenGeom g = token_geom(p);
  const int d = static_cast<int>(p.d);
  const int64_t BH = p.BH();
  const int64_t items = BH * p.M;
  if (items > 0x7fffffffLL) return MHLA_ERR_UNSUPPORTED;
  const T* qp = static_cast<const T*>(p.q.data);
  T* op = static_cast<T*>(p.o.data);
  if (const int rc = launch_summary<T>(p, g, ws.Sz, stream); rc != MHLA_OK) return rc;

  const int64_t E = p.d * (p.d + 1);
  if (const int rc = launch_mix<false, false>(W, ws.Sz, ws.Szt, p.M, E, BH, stream); rc != MHLA_OK)
    return rc;

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

template <typename T>
int launch_simt_bwd_typed(const Problem& p, const float* W, const BwdOperands& bo, const SimtBwdWorkspace& ws,
                          cudaStream_t stream) {
  const TokenGeom g = token_geom(p);
  const int d = static_cast<int>(p.d);
  const int64_t BH = p.BH();
  const int64_t items = BH * p.M;
  if (items > 0x7fffffffLL || BH > 65535) return MHLA_ERR_UNSUPPORTED;
  const T* qp = static_cast<const T*>(p.q.data);
  const T* kp = static_cast<const T*>(p.k.data);
  const T* vp = static_cast<const T*>(p.v.data);
  const T* gp = static_cast<const T*>(bo.dout.data);
  T* dqp = static_cast<T*>(bo.dq.data);
  T* dkp = static_cast<T*>(bo.dk.data);
  T* dvp = static_cast<T*>(bo.dv.data);
  const int64_t E = p.d * (p.d + 1);

  // forward summaries and mixing, recomputed
  if (const int rc = launch_summary<T>(p, g, ws.Sz, stream); rc != MHLA_OK) return rc;
  if (const int rc = launch_mix<false, false>(W, ws.Sz, ws.Szt, p.M, E, BH, stream); rc != MHLA_OK)
    return rc;
  // query blocks: dq, dS~, dz~
  {
    const size_t smem = (d * (d + 1) + d + 2 * kBwdChunk * d + kBwdChunk) * sizeof(float);
    auto launch = [&](auto kern) -> int {
      if (smem > 48 * 1024 && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem)) != cudaSuccess)
        return MHLA_ERR_CUDA;
      KernelTimer timer("simt_bwd_query", stream);
      kern<<<static_cast<unsigned>(items), kBwdThreads, smem, stream>>>(qp, p.q, gp, bo.dout, dqp, bo.dq, g, p.H, d,
                                                                          p.phi_kind, p.eps, ws.Szt, ws.dSzt);
      return cudaGetLastError() == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
    };
    const int rc = d <= 16   ? launch(simt_bwd_query<T, 1>)
                   : d <= 32 ? launch(simt_bwd_query<T, 4>)
                   : d <= 64 ? launch(simt_bwd_query<T, 16>)
                             : launch(simt_bwd_query<T, 64>);
    if (rc != MHLA_OK) return rc;
  }
  // dW (before the transposed mixing overwrites S~ with dS)
  {
    const int64_t KS = dw_splits(p);
    const dim3 grid(static_cast<unsigned>((p.M + kDwTile - 1) / kDwTile),
                    static_cast<unsigned>((p.M + kDwTile - 1) / kDwTile), static_cast<unsigned>(BH * KS));
    if (grid.x > 65535 || BH * KS > 65535) return MHLA_ERR_UNSUPPORTED;
    KernelTimer timer("simt_dw", stream);
    simt_dw_partial<<<grid, 256, 0, stream>>>(ws.dSzt, ws.Sz, ws.part, p.M, E, static_cast<int32_t>(KS));
    if (cudaGetLastError() != cudaSuccess) return MHLA_ERR_CUDA;
    const int64_t MM = p.M * p.M;
    simt_dw_reduce<<<static_cast<unsigned>((MM + 31) / 32), kDwrWarps * 32, 0, stream>>>(ws.part, bo.dW, MM,
                                                                                         BH * KS);
    if (cudaGetLastError() != cudaSuccess) return MHLA_ERR_CUDA;
  }
  // dS = W^T dS~ into the S~ buffer
  if (const int rc = launch_mix<true, false>(W, ws.dSzt, ws.Szt, p.M, E, BH, stream); rc != MHLA_OK)
    return rc;
  // source blocks: dk, dv
  {
    const size_t smem = (d * (d + 1) + d + 2 * kBwdWarps * d) * sizeof(float);
    if (smem > 48 * 1024 && cudaFuncSetAttribute(simt_bwd_key<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem)) != cudaSuccess)
      return MHLA_ERR_CUDA;
    KernelTimer timer("simt_bwd_key", stream);
    simt_bwd_key<T><<<static_cast<unsigned>(items), kBwdThreads, smem, stream>>>(
        kp, p.k, vp, p.v, dkp, bo.dk, dvp, bo.dv, g, p.H, d, p.phi_kind, p.eps, ws.Szt);
    if (cudaGetLastError() != cudaSuccess) return MHLA_ERR_CUDA;
  }
  return MHLA_OK;
}

template <typename T>
int launch_simt_causal_typed(const Problem& p, const float* W, const SimtWorkspace& ws, cudaStream_t stream) {
  const TokenGeom g = token_geom(p);
  const int d = static_cast<int>(p.d);
  const int64_t BH = p.BH();
  const int64_t items = BH * p.M;
  if (items > 0x7fffffffLL) return MHLA_ERR_UNSUPPORTED;
  const T* qp = static_cast<const T*>(p.q.data);
  const T* kp = static_cast<const T*>(p.k.data);
  const T* vp = static_cast<const T*>(p.v.data);
  T* op = static_cast<T*>(p.o.data);
  if (const int rc = launch_summary<T>(p, g, ws.Sz, stream); rc != MHLA_OK) return rc;
  const int64_t E = p.d * (p.d + 1);
  if (const int rc = launch_mix<false, true>(W, ws.Sz, ws.Szt, p.M, E, BH, stream); rc != MHLA_OK)
    return rc;
  {
    const size_t smem = (d * d + d + kCausalChunk * (3 * d + 1) + kCausalWarps * kCausalChunk) * sizeof(float);
    auto launch = [&](auto kern) -> int {
      if (smem > 48 * 1024 && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem)) != cudaSuccess)
        return MHLA_ERR_CUDA;
      KernelTimer timer("simt_causal_output", stream);
      kern<<<static_cast<unsigned>(items), kCausalThreads, smem, stream>>>(qp, p.q, kp, p.k, vp, p.v, op, p.o, g, p.H,
                                                                             d, p.phi_kind, p.eps, W, ws.Szt);
      return cudaGetLastError() == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
    };
    return d <= 16   ? launch(simt_causal_output<T, 1>)
           : d <= 32 ? launch(simt_causal_output<T, 4>)
           : d <= 64 ? launch(simt_causal_output<T, 16>)
                     : launch(simt_causal_output<T, 64>);
  }
}

// Helpers of the causal backward's TC path, between the float32 [BH][M][d(d+1)]
// rows of the token kernels and the tensor-core causal forward's summary layout
// (Sbuf: bf16, the (b, h, entry) columns in groups of 128, one row per block).
// One CTA per (b, h, block), eight consecutive entries per thread: for d in
// {32, 64}, d(d+1) is a multiple of 8, so a run stays inside one 128-column group.
constexpr int kStThreads = 256;

// Two floats rounded to bf16 (round to nearest even), packed low then high.
__device__ __forceinline__ uint32_t pack_bf16_rn(float a, float b) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(a))) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(b))) << 16);
}

// dSbuf (summary layout) = dSp rounded to bf16; the padding columns of the last
// group (past BH d(d+1)) are zeroed in dSbuf and in the forward's Sbuf, whose
// whole groups the dW product reads.
__global__ void __launch_bounds__(kStThreads)
simt_ds_to_summary(const float* __restrict__ dSp, __nv_bfloat16* __restrict__ dSbuf, __nv_bfloat16* __restrict__ Sbuf,
                   int64_t M, int d, int64_t BH, int64_t ngroups) {
  const int E1 = d * d + d;
  const int64_t items = BH * M;
  for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
    const int64_t bh = it / M, i = it % M;
    for (int e = 8 * threadIdx.x; e < E1; e += 8 * kStThreads) {
      const int64_t col = bh * E1 + e;
      const float4* src = reinterpret_cast<const float4*>(dSp + it * E1 + e);
      const float4 lo = src[0], hi = src[1];
      uint4 o;
      o.x = pack_bf16_rn(lo.x, lo.y), o.y = pack_bf16_rn(lo.z, lo.w);
      o.z = pack_bf16_rn(hi.x, hi.y), o.w = pack_bf16_rn(hi.z, hi.w);
      *reinterpret_cast<uint4*>(dSbuf + ((col >> 7) * M + i) * 128 + (col & 127)) = o;
    }
    if (bh == BH - 1) {
      const int64_t c0 = BH * E1, c1 = ngroups * 128;
      for (int64_t col = c0 + threadIdx.x; col < c1; col += kStThreads) {
        const int64_t at = ((col >> 7) * M + i) * 128 + (col & 127);
        dSbuf[at] = __float2bfloat16_rn(0.0f);
        Sbuf[at] = __float2bfloat16_rn(0.0f);
      }
    }
  }
}

// Between the dW product and the mixing of dS, one pass over M x M:
//   dW made causal: zero above the diagonal (the product below it stays), and on
//   it the query kernel's W_ii shares summed over (b, h) by one warp per
//   diagonal entry (lane-strided, then a fixed-order shuffle sum);
//   Wm[j][i] = W[i][j] for i > j, else 0 (bf16 [M][Mp]), so that
//   dS_j = sum_{i > j} W[i][j] dS<_i is one mixing GEMM.
// The grid covers max(M Mp, 32 M) threads in whole warps.
__global__ void simt_dw_causal_and_wt(float* __restrict__ dW, const float* __restrict__ diag,
                                      const float* __restrict__ W, __nv_bfloat16* __restrict__ Wm, int64_t M,
                                      int64_t Mp, int64_t BH) {
  const int64_t x = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (x < M * Mp) {
    const int64_t r = x / Mp, c = x % Mp;
    Wm[x] = __float2bfloat16_rn(c < M && c > r ? W[c * M + r] : 0.0f);
    if (c < M && c > r) dW[r * M + c] = 0.0f;
  }
  if (x < 32 * M) {   // whole warps: 32 M is a multiple of the warp
    const int64_t r = x / 32;
    const int lane = static_cast<int>(x % 32);
    float s = 0.0f;
    for (int64_t bh = lane; bh < BH; bh += 32) s += diag[bh * M + r];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) dW[r * M + r] = s;
  }
}

struct SimtCausalBwdWorkspace {
  float* Sz;     // [BH][M][d*(d+1)] S_j, z_j
  float* Sp;     // [BH][M][d*(d+1)] S<_i, z<_i, later dS_j, dz_j
  float* dSp;    // [BH][M][d*(d+1)] dS<_i, dz<_i
  float* part;   // [BH][M][M]       <dS<_i, S_j> + dz<_i . z_j
  float* diag;   // [BH][M]          the (b, h) share of dW_ii
  float* dn;     // [BH][N][d + 1]   dnum_t, dden_t in block-slot order
  void* tc;      // the region of launch_tc_causal_states (tensor-core summaries and mixing), or null
  float* tcpart; // the tensor-core dW product's split partials (path TC)
};

SimtCausalBwdWorkspace simt_causal_bwd_carve(const Problem& p, void* base) {
  const size_t per = static_cast<size_t>(p.BH()) * p.M * p.d * (p.d + 1) * sizeof(float);
  const size_t part = static_cast<size_t>(p.BH()) * dw_splits(p) * p.M * p.M * sizeof(float);
  const size_t diag = static_cast<size_t>(p.BH()) * p.M * sizeof(float);
  char* c = static_cast<char*>(base);
  SimtCausalBwdWorkspace ws;
  ws.Sz = reinterpret_cast<float*>(c);
  ws.Sp = reinterpret_cast<float*>(c + align_up(per));
  ws.dSp = reinterpret_cast<float*>(c + 2 * align_up(per));
  ws.part = reinterpret_cast<float*>(c + 3 * align_up(per));
  ws.diag = reinterpret_cast<float*>(c + 3 * align_up(per) + align_up(part));
  ws.dn = reinterpret_cast<float*>(c + 3 * align_up(per) + align_up(part) + align_up(diag));
  ws.tc = nullptr;
  ws.tcpart = nullptr;
  return ws;
}

template <typename T>
int launch_simt_causal_bwd_typed(const Problem& p, const float* W, const BwdOperands& bo,
                                 const SimtCausalBwdWorkspace& ws, cudaStream_t stream) {
  const TokenGeom g = token_geom(p);
  const int d = static_cast<int>(p.d);
  const int64_t BH = p.BH();
  const int64_t items = BH * p.M;
  if (items > 0x7fffffffLL || BH > 65535) return MHLA_ERR_UNSUPPORTED;
  const T* qp = static_cast<const T*>(p.q.data);
  const T* kp = static_cast<const T*>(p.k.data);
  const T* vp = static_cast<const T*>(p.v.data);
  const T* gp = static_cast<const T*>(bo.dout.data);
  T* dqp = static_cast<T*>(bo.dq.data);
  T* dkp = static_cast<T*>(bo.dk.data);
  T* dvp = static_cast<T*>(bo.dv.data);
  const int64_t E = p.d * (p.d + 1);
  // path TC: S_j (kept in the summary layout) and S<_i from the tensor-core causal
  // forward's summary and mixing kernels; later the dW product and the mixing of
  // dS on the tensor cores as well
  CausalStates cs{};
  if (ws.tc) {   // the token kernels read S<_i (later dS_j) from the tensor-core layout
    if (const int rc = launch_tc_causal_states(p, W, ws.tc, stream, &cs); rc != MHLA_OK) return rc;
  } else {
    if (const int rc = launch_summary<T>(p, g, ws.Sz, stream); rc != MHLA_OK) return rc;
    if (const int rc = launch_mix<false, true>(W, ws.Sz, ws.Sp, p.M, E, BH, stream); rc != MHLA_OK)
      return rc;
  }
  {
    const size_t smem = (d * (d + 1) + d + 5 * kCbChunk * (d + 1) + 2 * kCbChunk + 2 * kCbChunk * (kCbChunk + 1) +
                         kCbWarps) * sizeof(float);
    auto launch = [&](auto kern) -> int {
      if (smem > 48 * 1024 && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem)) != cudaSuccess)
        return MHLA_ERR_CUDA;
      KernelTimer timer("simt_causal_bwd_query", stream);
      kern<<<static_cast<unsigned>(items), kCbThreads, smem, stream>>>(
          qp, p.q, kp, p.k, vp, p.v, gp, bo.dout, dqp, bo.dq, g, p.H, d, p.phi_kind, p.eps, W, ws.Sp, ws.dSp,
          ws.diag, ws.dn);
      return cudaGetLastError() == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
    };
    // d = 32, 64: the vector layout
    auto launch_v = [&](auto kern, size_t vsmem) -> int {
      if (vsmem > 48 * 1024 && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                    static_cast<int>(vsmem)) != cudaSuccess)
        return MHLA_ERR_CUDA;
      KernelTimer timer("simt_causal_bwd_query", stream);
      kern<<<static_cast<unsigned>(items), kCbThreads, vsmem, stream>>>(
          qp, p.q, kp, p.k, vp, p.v, gp, bo.dout, dqp, bo.dq, g, p.H, p.phi_kind, p.eps, W, ws.Sp, ws.dSp,
          ws.diag, ws.dn, static_cast<const __nv_bfloat16*>(cs.St), cs.zt);
      return cudaGetLastError() == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
    };
    int rc = -1;
    if constexpr (std::is_same_v<T, __nv_bfloat16>) {   // bf16: the products on warp-level tensor cores
      if (d == 64) rc = launch_v(simt_causal_bwd_query_mma<64>, cbm_query_smem(64));
      if (d == 32) rc = launch_v(simt_causal_bwd_query_mma<32>, cbm_query_smem(32));
    } else {                                            // float32: every product on CUDA cores
      if (d == 64) rc = launch_v(simt_causal_bwd_query_v<T, 64>, cbv_query_smem(64));
      if (d == 32) rc = launch_v(simt_causal_bwd_query_v<T, 32>, cbv_query_smem(32));
    }
    if (rc == -1)
      rc = d <= 16   ? launch(simt_causal_bwd_query<T, 1, 1>)
         : d <= 32 ? launch(simt_causal_bwd_query<T, 4, 2>)
         : d <= 64 ? launch(simt_causal_bwd_query<T, 16, 4>)
                   : launch(simt_causal_bwd_query<T, 64, 8>);
    if (rc != MHLA_OK) return rc;
  }
  const int64_t MM = p.M * p.M;
  if (ws.tc) {
    // dS<_i into the summary layout (over the float32 S_j buffer, unused on this
    // path); dW = <dS<_i, S_j> for every (i, j) on the tensor cores, then made
    // causal; dS_j = sum_{i > j} W[i][j] dS<_i as a mixing GEMM with W's strict
    // lower triangle transposed (in the states' matrix slot), back to float32
    auto* dSbuf = reinterpret_cast<__nv_bfloat16*>(ws.Sz);
    const int64_t ngroups = (BH * E + 127) / 128;
    {
      KernelTimer timer("simt_ds_to_summary", stream);
      simt_ds_to_summary<<<static_cast<unsigned>(items), kStThreads, 0, stream>>>(
          ws.dSp, dSbuf, static_cast<__nv_bfloat16*>(cs.Sbuf), p.M, d, BH, ngroups);
      if (cudaGetLastError() != cudaSuccess) return MHLA_ERR_CUDA;
    }
    if (const int rc = tc_run_dw(p, dSbuf, cs.Sbuf, ws.tcpart, bo.dW, stream); rc != MHLA_OK) return rc;
    {
      const int64_t n = std::max<int64_t>(p.M * cs.Mp, 32 * p.M);
      if ((n + 255) / 256 > 0x7fffffffLL) return MHLA_ERR_UNSUPPORTED;
      KernelTimer timer("simt_dw_causal_and_wt", stream);
      simt_dw_causal_and_wt<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(
          bo.dW, ws.diag, W, static_cast<__nv_bfloat16*>(cs.Wu), p.M, cs.Mp, BH);
      if (cudaGetLastError() != cudaSuccess) return MHLA_ERR_CUDA;
    }
    if (const int rc = launch_tc_causal_mix(p, cs.Wu, cs.Mp, dSbuf, cs.St, cs.zt, stream); rc != MHLA_OK) return rc;
  } else {
    {
      const int64_t KS = dw_splits(p);
      const dim3 grid(static_cast<unsigned>((p.M + kDwTile - 1) / kDwTile),
                      static_cast<unsigned>((p.M + kDwTile - 1) / kDwTile), static_cast<unsigned>(BH * KS));
      if (grid.x > 65535 || BH * KS > 65535) return MHLA_ERR_UNSUPPORTED;
      KernelTimer timer("simt_dw", stream);
      simt_dw_partial<<<grid, 256, 0, stream>>>(ws.dSp, ws.Sz, ws.part, p.M, E, static_cast<int32_t>(KS));
      if (cudaGetLastError() != cudaSuccess) return MHLA_ERR_CUDA;
      simt_dw_reduce_causal<<<static_cast<unsigned>((MM + 31) / 32), kDwrWarps * 32, 0, stream>>>(
          ws.part, ws.diag, bo.dW, p.M, BH, KS);
      if (cudaGetLastError() != cudaSuccess) return MHLA_ERR_CUDA;
    }
    if (const int rc = launch_mix<true, true>(W, ws.dSp, ws.Sp, p.M, E, BH, stream); rc != MHLA_OK)
      return rc;
  }
  {
    const size_t smem = (d * (d + 1) + d + 4 * kCbChunk * (d + 1) + kCbChunk + 2 * kCbChunk * (kCbChunk + 1)) *
                        sizeof(float);
    auto launch = [&](auto kern) -> int {
      if (smem > 48 * 1024 && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem)) != cudaSuccess)
        return MHLA_ERR_CUDA;
      KernelTimer timer("simt_causal_bwd_key", stream);
      kern<<<static_cast<unsigned>(items), kCbThreads, smem, stream>>>(
          qp, p.q, kp, p.k, vp, p.v, dkp, bo.dk, dvp, bo.dv, g, p.H, d, p.phi_kind, p.eps, W, ws.Sp, ws.dn);
      return cudaGetLastError() == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
    };
    auto launch_v = [&](auto kern, size_t vsmem) -> int {
      if (vsmem > 48 * 1024 && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                    static_cast<int>(vsmem)) != cudaSuccess)
        return MHLA_ERR_CUDA;
      KernelTimer timer("simt_causal_bwd_key", stream);
      kern<<<static_cast<unsigned>(items), kCbThreads, vsmem, stream>>>(
          qp, p.q, kp, p.k, vp, p.v, dkp, bo.dk, dvp, bo.dv, g, p.H, p.phi_kind, p.eps, W, ws.Sp, ws.dn,
          static_cast<const __nv_bfloat16*>(cs.St), cs.zt);
      return cudaGetLastError() == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
    };
    if constexpr (std::is_same_v<T, __nv_bfloat16>) {   // bf16: the products on warp-level tensor cores
      if (d == 64) return launch_v(simt_causal_bwd_key_mma<64>, cbm_key_smem(64));
      if (d == 32) return launch_v(simt_causal_bwd_key_mma<32>, cbm_key_smem(32));
    } else {                                            // float32: every product on CUDA cores
      if (d == 64) return launch_v(simt_causal_bwd_key_v<T, 64>, cbv_key_smem(64));
      if (d == 32) return launch_v(simt_causal_bwd_key_v<T, 32>, cbv_key_smem(32));
    }
    return d <= 16   ? launch(simt_causal_bwd_key<T, 1, 1>)
           : d <= 32 ? launch(simt_causal_bwd_key<T, 2, 2>)
           : d <= 64 ? launch(simt_causal_bwd_key<T, 4, 4>)
                     : launch(simt_causal_bwd_key<T, 8, 8>);
  }
}

}  // namespace

int launch_simt_causal(const Problem& p, const float* W, void* workspace, void* stream) {
  const SimtWorkspace ws = simt_carve(p, workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.dtype == MHLA_BF16) return launch_simt_causal_typed<__nv_bfloat16>(p, W, ws, s);
  return launch_simt_causal_typed<float>(p, W, ws, s);
}

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

size_t simt_bwd_workspace_bytes(const Problem& p) {
  const size_t per = static_cast<size_t>(p.BH()) * p.M * p.d * (p.d + 1) * sizeof(float);
  const size_t part = static_cast<size_t>(p.BH()) * dw_splits(p) * p.M * p.M * sizeof(float);
  return 3 * align_up(per) + align_up(part);
}

int launch_simt_bwd(const Problem& p, const float* W, const BwdOperands& bo, void* workspace, void* stream) {
  const size_t per = static_cast<size_t>(p.BH()) * p.M * p.d * (p.d + 1) * sizeof(float);
  char* c = static_cast<char*>(workspace);
  SimtBwdWorkspace ws;
  ws.Sz = reinterpret_cast<float*>(c);
  ws.Szt = reinterpret_cast<float*>(c + align_up(per));
  ws.dSzt = reinterpret_cast<float*>(c + 2 * align_up(per));
  ws.part = reinterpret_cast<float*>(c + 3 * align_up(per));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.dtype == MHLA_BF16) return launch_simt_bwd_typed<__nv_bfloat16>(p, W, bo, ws, s);
  return launch_simt_bwd_typed<float>(p, W, bo, ws, s);
}

namespace {
size_t simt_causal_bwd_own_bytes(const Problem& p) {
  const size_t per = static_cast<size_t>(p.BH()) * p.M * p.d * (p.d + 1) * sizeof(float);
  const size_t part = static_cast<size_t>(p.BH()) * dw_splits(p) * p.M * p.M * sizeof(float);
  const size_t diag = static_cast<size_t>(p.BH()) * p.M * sizeof(float);
  // dnum / dden rows of d + 1 floats, at a stride of d + 4 on the bf16 warp-MMA kernels
  const size_t dn = static_cast<size_t>(p.BH()) * p.M * p.w * (p.d + 4) * sizeof(float);
  return 3 * align_up(per) + align_up(part) + align_up(diag) + align_up(dn);
}
}  // namespace

size_t simt_causal_bwd_workspace_bytes(const Problem& p, bool tc_states) {
  return simt_causal_bwd_own_bytes(p) +
         (tc_states ? align_up(tc_causal_states_bytes(p)) + align_up(tc_dw_part_floats(p) * sizeof(float)) : 0);
}

int launch_simt_causal_bwd(const Problem& p, const float* W, const BwdOperands& bo, void* workspace, void* stream,
                           bool tc_states) {
  SimtCausalBwdWorkspace ws = simt_causal_bwd_carve(p, workspace);
  if (tc_states) {
    ws.tc = static_cast<char*>(workspace) + simt_causal_bwd_own_bytes(p);
    ws.tcpart = reinterpret_cast<float*>(static_cast<char*>(ws.tc) + align_up(tc_causal_states_bytes(p)));
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.dtype == MHLA_BF16) return launch_simt_causal_bwd_typed<__nv_bfloat16>(p, W, bo, ws, s);
  return launch_simt_causal_bwd_typed<float>(p, W, bo, ws, s);
}

}  // namespace mhla
