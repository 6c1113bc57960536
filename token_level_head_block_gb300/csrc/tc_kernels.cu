// Tensor-core path of the MHLA forward on sm_103a: TMA-fed, tcgen05 MMAs with
// float32 accumulators in tensor memory, persistent warp-specialised CTAs.
//
// The three steps of the method ([P2] "MHLA: Restoring Expressivity of Linear
// Attention via Token-Level Multi-Head", section 4 "Architecture", "Multi-Head
// Mixing", "Token-Level Adaptivity"; [P1] 171host.com/767426.html, section 7,
// MHLA.forward):
//
//   tc_summary  per (b, head group, block j): [S_j | z_j] = phi(K_j)^T [V_j | 1]
//               (its prologue also rounds W to bf16 for the mixing GEMM)
//               K and V chunks of 64 tokens arrive by 5-D TMA (d, H, X, Y, B*T);
//               phi is applied in shared memory; 128/d heads share one
//               128 x (128+16) MMA whose diagonal d x d blocks are the S_j and
//               whose column 128 (a constant "ones" operand) is z_j.
//   tc_mix      S~ = W . S as one GEMM over the source blocks j:
//               D[i, col] = sum_j W[i][j] Sbuf[j][col], col = (b, h, row, c).
//   tc_output   per (b, h, block i), 128 tokens at a time:
//               o_t = phi(q_t) S~_i / (phi(q_t) . z~_i + eps); numerator and
//               denominator from one MMA (z~_i rides as two extra B columns),
//               the result scaled, rounded and stored by TMA in the input layout.
//
// The kernels live in tc_summary.cu, tc_mix.cu and tc_output.cu; this file
// holds the host side they share: tensor-map encoding, the workspace layout,
// eligibility, the launch sequence and the device error words.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "mhla_internal.h"
#include "tc_common.cuh"
#include "tma_host.h"

namespace mhla {
namespace {

using namespace tc;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool encode(CUtensorMap* m, int rank, void* base, const cuuint64_t* dims, const cuuint64_t* strides_bytes,
            const cuuint32_t* box, CUtensorMapSwizzle swz, CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return fn(m, dt, static_cast<cuuint32_t>(rank), base, dims, strides_bytes, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct TcLayout {
  size_t wb_off, sbuf_off, st_off, zt_off, ctr_off, total;
  int64_t Mp, ncols, ngroups;
};

TcLayout tc_layout(const Problem& p) {
  TcLayout L;
  L.Mp = (p.M + 7) / 8 * 8;
  L.ncols = p.BH() * (p.d + 1) * p.d;
  L.ngroups = (L.ncols + 127) / 128;                    // Sbuf column groups of 128
  size_t off = 0;
  L.wb_off = off;
  off += align_up(static_cast<size_t>(p.M) * L.Mp * 2);
  L.sbuf_off = off;
  off += align_up(static_cast<size_t>(p.M) * L.ngroups * 128 * 2);
  L.st_off = off;
  off += align_up(static_cast<size_t>(p.BH()) * p.M * p.d * p.d * 2);
  L.zt_off = off;
  off += align_up(static_cast<size_t>(p.BH()) * p.M * p.d * 4);
  L.ctr_off = off;
  off += align_up(tc_fused_counter_bytes(p));
  L.total = off;
  return L;
}

int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

}  // namespace

bool encode_tensor_map(CUtensorMap* m, int rank, void* base, const cuuint64_t* dims,
                       const cuuint64_t* strides_bytes, const cuuint32_t* box, CUtensorMapSwizzle swz) {
  return encode(m, rank, base, dims, strides_bytes, box, swz);
}

int device_sm_count() { return device_sms(); }

// The three-launch tensor-core forward: tokens per block a multiple of 128 in
// whole block rows, or contiguous 64-token blocks (the tile readout).
bool tc_rows_eligible(const Problem& p) {
  if (p.dtype != MHLA_BF16) return false;
  if (p.d != 32 && p.d != 64) return false;
  if (p.B < 1 || p.H < 1) return false;
  ChunkPlan cp;
  if (!chunk_plan(p, 64, &cp) || !chunk_plan(p, 128, &cp)) return false;
  for (const Operand* o : {&p.q, &p.k, &p.v, &p.o})
    if (!operand_tma_ok(p, *o)) return false;
  const int64_t lim32 = int64_t{1} << 31;
  const int64_t ncols = p.BH() * (p.d + 1) * p.d;
  if (p.BH() * p.M * p.d >= lim32 || ncols >= lim32 || p.M >= (int64_t{1} << 16)) return false;
  if (p.X >= lim32 || p.Y >= lim32 || p.B * p.T >= lim32 || p.H >= lim32) return false;
  if (p.B * ((p.H + 1) / 2) * p.M >= lim32) return false;
  return true;
}

bool tc_eligible(const Problem& p) { return tc_rows_eligible(p) || tc_tile_eligible(p); }

size_t tc_workspace_bytes(const Problem& p) { return tc_layout(p).total; }

int launch_tc(const Problem& p, const float* W, void* workspace, void* stream, bool fused) {
  const TcLayout L = tc_layout(p);
  char* ws = static_cast<char*>(workspace);
  if (!tc_rows_eligible(p))
    return launch_tc_tile_forward(p, W, ws + L.wb_off, L.Mp, ws + L.sbuf_off, ws + L.st_off,
                                  reinterpret_cast<float*>(ws + L.zt_off), stream);
  if (fused)
    return launch_tc_fused(p, W, ws + L.sbuf_off, ws + L.st_off, reinterpret_cast<float*>(ws + L.zt_off),
                           ws + L.ctr_off, stream);
  int rc = tc_run_summary(p, W, ws + L.wb_off, nullptr, L.Mp, ws + L.sbuf_off, stream);
  if (rc == MHLA_OK)
    rc = tc_run_mix(p, ws + L.wb_off, L.Mp, ws + L.sbuf_off, ws + L.st_off, reinterpret_cast<float*>(ws + L.zt_off),
                    stream, /*discard_input=*/true);
  if (rc == MHLA_OK) rc = tc_run_output(p, ws + L.st_off, reinterpret_cast<float*>(ws + L.zt_off), stream);
  return rc;
}

int read_and_clear_device_error(void* stream, uint32_t* flags) {
  uint32_t a = 0, b = 0, c = 0, f = 0;
  const int ra = read_and_clear_summary_error(stream, &a);
  const int rb = read_and_clear_mix_error(stream, &b);
  const int rc = read_and_clear_output_error(stream, &c);
  const int rf = read_and_clear_fused_error(stream, &f);
  if (ra == MHLA_ERR_CUDA || rb == MHLA_ERR_CUDA || rc == MHLA_ERR_CUDA || rf == MHLA_ERR_CUDA) return MHLA_ERR_CUDA;
  *flags = a | b | c | f;
  return *flags ? MHLA_ERR_TIMEOUT : MHLA_OK;
}

}  // namespace mhla
