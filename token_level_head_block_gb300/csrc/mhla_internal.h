// Internal host/device descriptors shared by the C ABI and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>

#include "../../include/mhla.h"

namespace mhla {

// One [B, N, H, d] operand: base pointer and element strides.
struct Operand {
  void* data;
  int64_t sb, sn, sh;
};

// Everything a launch needs about the token geometry, resolved on the host.
struct Problem {
  int64_t B, N, H, d;
  int dtype;            // mhla_dtype_t
  int ndim;             // 2 or 3
  int64_t T, Y, X;      // grid (T = 1 for 2-D)
  int64_t bt, by, bx;   // block (bt = 1 for 2-D)
  int64_t nbt, nby, nbx;
  int64_t M, w;         // blocks, tokens per block
  int phi_kind;
  float eps;
  Operand q, k, v, o;
  int64_t BH() const { return B * H; }
};

// Block j (row-major over (nbt, nby, nbx)) and in-block slot s (raster over
// (bt, by, bx)) -> token index n (raster over (T, Y, X)).
struct TokenGeom {
  int64_t Y, X, bt, by, bx, nby, nbx, M, w;
};

inline TokenGeom token_geom(const Problem& p) {
  return TokenGeom{p.Y, p.X, p.bt, p.by, p.bx, p.nby, p.nbx, p.M, p.w};
}

// Workspace layout of the CUDA-core path (float32):
//   Sz  [BH][M][d*(d+1)]  per block: S_j row-major then z_j
//   Szt [BH][M][d*(d+1)]  mixed:     S~_i row-major then z~_i
struct SimtWorkspace {
  float* Sz;
  float* Szt;
};
size_t simt_workspace_bytes(const Problem& p);
SimtWorkspace simt_carve(const Problem& p, void* base);
int launch_simt(const Problem& p, const float* W, void* workspace, void* stream);
// Causal MHLA on CUDA cores (contiguous blocks); same workspace as the forward,
// Szt holding the mixed past summaries.
int launch_simt_causal(const Problem& p, const float* W, void* workspace, void* stream);
// Causal MHLA on tensor cores (bf16, d in {32, 64}, contiguous blocks of 64
// tokens or a multiple of 128, N a multiple of 128).  Workspace: the unit-level
// W' (bf16), unit summaries (Sbuf layout), unit states (St, zt layouts).
bool tc_causal_eligible(const Problem& p);
size_t tc_causal_workspace_bytes(const Problem& p);
int launch_tc_causal(const Problem& p, const float* W, void* workspace, void* stream);
int read_and_clear_causal_error(void* stream, uint32_t* flags);
// The forward's tensor-core path for contiguous 64-token blocks (N a multiple
// of 128): summaries and mixing as usual, then per 128-token tile one MMA per
// block of the tile against that block's rows.  Workspace as tc_layout.
bool tc_tile_eligible(const Problem& p);
int launch_tc_tile_forward(const Problem& p, const float* W, void* Wb, int64_t Mp, void* Sbuf, void* St, float* zt,
                           void* stream);

// Backward pass operands (dout read; dq, dk, dv, dW written) and the CUDA-core
// backward's workspace (float32):
//   Sz   [BH][M][d*(d+1)]  S_j, z_j (recomputed)
//   Szt  [BH][M][d*(d+1)]  S~_i, z~_i; later overwritten with dS_j, dz_j
//   dSzt [BH][M][d*(d+1)]  dS~_i, dz~_i
//   part [BH][M][M]        per-(b, h) partial sums of dW
struct BwdOperands {
  Operand dout, dq, dk, dv;
  float* dW;
};
struct SimtBwdWorkspace {
  float *Sz, *Szt, *dSzt, *part;
};
size_t simt_bwd_workspace_bytes(const Problem& p);
int launch_simt_bwd(const Problem& p, const float* W, const BwdOperands& bo, void* workspace, void* stream);
// Causal backward on CUDA cores (contiguous blocks, any d <= 128).  Workspace:
// S_j, the mixed past S<_i (later dS_j), dS<_i, the dW partials and diagonal
// shares, and dnum_t, dden_t per token (float32); with tc_states, then the
// region of launch_tc_causal_states, whose summaries and states replace the
// CUDA-core summary and mixing steps.
size_t simt_causal_bwd_workspace_bytes(const Problem& p, bool tc_states);
int launch_simt_causal_bwd(const Problem& p, const float* W, const BwdOperands& bo, void* workspace, void* stream,
                           bool tc_states);
// The tensor-core causal forward's first two steps kept for the backward when
// every block is one unit (w = 64 or 128, and tc_causal_eligible): the block
// summaries S_j (Sbuf: bf16, the (b, h, entry) columns in groups of 128, one
// row of each group per block, entries S_j row-major then z_j) and the mixed
// past S<_i (St: bf16 [BH][M][d][d] row-major; zt: float32 [BH][M][d]).
struct CausalStates {
  void* Sbuf;
  void* St;
  float* zt;
  void* Wu;      // bf16 [M][Mp]: the mixing matrix of the states, free for reuse after them
  int64_t Mp;
};
// dW[i][j] = sum over every summary column of dSbuf[i] . Sbuf[j] (both in the
// summary layout above, padding columns zero), by the tensor-core backward's
// dW kernel; part holds tc_dw_part_floats(p) floats.
int64_t tc_dw_part_floats(const Problem& p);
int tc_run_dw(const Problem& p, const void* dSbuf, const void* Sbuf, float* part, float* dW, void* stream);
bool tc_causal_states_eligible(const Problem& p);
size_t tc_causal_states_bytes(const Problem& p);
int launch_tc_causal_states(const Problem& p, const float* W, void* region, void* stream, CausalStates* out);
// One mixing GEMM of the tensor-core causal forward on the same problem:
// [St | zt] (its layout) = Wm (bf16 [M][Mp]) times the summary-layout Sbuf.
int launch_tc_causal_mix(const Problem& p, const void* Wm, int64_t Mp, const void* Sbuf, void* St, float* zt,
                         void* stream);

// Tensor-core backward (bf16, d in {32, 64}, the forward tensor-core path's
// token geometry, TMA-friendly strides on every operand).  Workspace: Wb and
// W^T in bf16 [M][Mp]; Sbuf and dSbuf as the forward's Sbuf; St, zt as the
// forward's (S~, z~, later overwritten with dS, dz); float32 dW partials.
bool tc_bwd_eligible(const Problem& p, const BwdOperands& bo);
size_t tc_bwd_workspace_bytes(const Problem& p);
int launch_tc_bwd(const Problem& p, const float* W, const BwdOperands& bo, void* workspace, void* stream);
int read_and_clear_bwd_error(void* stream, uint32_t* flags);

// Workspace layout of the tensor-core path:
//   Wb   bf16 [M][Mp]                  W rounded to bf16, Mp = round_up(M, 8)
//   Sbuf bf16 [G][M][128]               columns col = (b,h) then the d rows of S_j
//                                       then the row z_j, blocked by G groups of
//                                       128 columns: (col/128, j, col%128)
//   St   bf16 [BH][M][d][d]             S~_i row-major (r, c)
//   zt   f32  [BH][M][d]                z~_i
//   ctr  u32  [2B + 1]                  counters of the fused launch (zeroed per call)
size_t tc_workspace_bytes(const Problem& p);
bool tc_eligible(const Problem& p);
// The three-launch path's own condition (tokens per block a multiple of 128 in
// whole block rows); tc_eligible also admits the tile readout's contiguous
// 64-token blocks.
bool tc_rows_eligible(const Problem& p);
// fused: the single persistent launch (tc_fused.cu; the caller checked
// tc_fused_eligible); otherwise the summary, mixing and readout launches.
int launch_tc(const Problem& p, const float* W, void* workspace, void* stream, bool fused = false);

// The fused launch: tc_rows_eligible and M <= 256.  Sbuf, St, zt as above; ctr
// holds 2B + 1 counters the launch zeroes on the stream first.
bool tc_fused_eligible(const Problem& p);
size_t tc_fused_counter_bytes(const Problem& p);
int launch_tc_fused(const Problem& p, const float* W, void* Sbuf, void* St, float* zt, void* ctr, void* stream);
int read_and_clear_fused_error(void* stream, uint32_t* flags);
// d = 32 with an even number of adjacent heads: the readout pairs heads into
// 64-channel rows.
bool output_pairs_heads(const Problem& p);

// Fused short-sequence path (N <= 256 tokens, M <= 96 blocks, bf16, d in
// {32, 64}): one launch that forms the two-stage N x N product; no workspace.
bool small_eligible(const Problem& p);
int launch_small(const Problem& p, const float* W, void* stream);

// Steps of the tensor-core path on caller-given buffers (layouts as above):
// tc_run_summary writes Wb (and W^T into WbT when WbT is not null) and Sbuf;
// with upb > 0 the problem's blocks are causal units, upb per block of the
// Mw x Mw matrix W, and Wb receives the unit-level causal matrix instead;
// tc_run_mix computes St, zt = Wm . Sbuf for the bf16 [M][Mp] matrix Wm; with
// discard_input its M <= 256 kernel drops Sbuf's L2 lines once read (no
// write-back): only for callers that do not read Sbuf afterwards.
int tc_run_summary(const Problem& p, const float* W, void* Wb, void* WbT, int64_t Mp, void* Sbuf, void* stream,
                   int32_t Mw = 0, int32_t upb = 0);
int tc_run_mix(const Problem& p, const void* Wm, int64_t Mp, const void* Sbuf, void* St, float* zt, void* stream,
               bool discard_input = false);
int tc_run_output(const Problem& p, const void* St, const float* zt, void* stream);
int read_and_clear_summary_error(void* stream, uint32_t* flags);
int read_and_clear_mix_error(void* stream, uint32_t* flags);
int read_and_clear_output_error(void* stream, uint32_t* flags);

// Device error words of the tensor-core and fused kernels (bounded waits).
int read_and_clear_device_error(void* stream, uint32_t* flags);
int read_and_clear_small_error(void* stream, uint32_t* flags);

// Each file's copy of the diagnostic stall hook (stall_hook.cuh): the warp
// index + 1 whose bounded waits stall (0: off) and how long they last.
int set_stall_summary(uint32_t warp_plus_1, uint64_t ns);
int set_stall_mix(uint32_t warp_plus_1, uint64_t ns);
int set_stall_output(uint32_t warp_plus_1, uint64_t ns);
int set_stall_fused(uint32_t warp_plus_1, uint64_t ns);
int set_stall_small(uint32_t warp_plus_1, uint64_t ns);
int set_stall_bwd(uint32_t warp_plus_1, uint64_t ns);
int set_stall_causal(uint32_t warp_plus_1, uint64_t ns);
int set_stall_module(uint32_t warp_plus_1, uint64_t ns);
int set_stall_gemm(uint32_t warp_plus_1, uint64_t ns);

// Brackets one kernel launch with CUDA events on its stream while
// mhla_profile_begin/end collection is active, and always with an NVTX range
// named after the kernel (free when no profiler is attached).
class KernelTimer {
 public:
  KernelTimer(const char* name, void* stream);
  ~KernelTimer();
  KernelTimer(const KernelTimer&) = delete;
  KernelTimer& operator=(const KernelTimer&) = delete;

 private:
  const char* name_;
  void* stream_;
  void* start_;
};

// Every block a contiguous range of raster-order tokens: for some axis a, the
// block is one unit on every slower axis and the whole grid on every faster one.
inline bool blocks_contiguous(const Problem& p) {
  const int64_t g[3] = {p.T, p.Y, p.X}, b[3] = {p.bt, p.by, p.bx};
  for (int a = 0; a < 3; ++a) {
    bool ok = true;
    for (int s = 0; s < a; ++s) ok = ok && b[s] == 1;
    for (int f = a + 1; f < 3; ++f) ok = ok && b[f] == g[f];
    if (ok) return true;
  }
  return false;
}

// Module around the core: LayerNorm rows, the 5 x 5 depthwise positional term
// added into the core's output, and the bf16 linear layers (launch_gemm).
struct LepeArgs {
  const void* v;
  void* o;
  int64_t vsb, vsn, vsh, osb, osn, osh;   // elements
  int64_t B;
  int32_t d, C, T, Y, X;
  const float* weight;   // [C][5][5]
  const float* bias;     // [C]
};
int launch_layer_norm(const void* x, void* y, int64_t rows, int32_t C, const float* weight, const float* bias,
                      float eps, void* stream);
int launch_lepe_add(const LepeArgs& a, void* stream);
int read_and_clear_module_error(void* stream, uint32_t* flags);
// y[rows][n_out] = x[rows][k] w^T (+ bias), bf16, w [n_out][k] (nn.Linear's
// layout); tcgen05 GEMM (gemm_kernels.cu).  k % 8 == 0, n_out % 8 == 0, x, w,
// bias and y 16-byte aligned; name labels the launch for the kernel timer.
bool gemm_supported(int64_t rows, int64_t k, int64_t n_out);
int launch_gemm(const char* name, const void* x, const void* w, const void* bias, void* y, int64_t rows, int64_t k,
                int64_t n_out, void* stream);
int read_and_clear_gemm_error(void* stream, uint32_t* flags);

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }

}  // namespace mhla
