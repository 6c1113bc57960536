// extern "C" entry points of libmhla: argument validation, problem
// construction, path selection and workspace handling.  Every check runs on the
// host before anything is queued on the stream.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "mhla_internal.h"

namespace mhla {
namespace {

int64_t elem_bytes(int dtype) { return dtype == MHLA_BF16 ? 2 : 4; }

bool valid_dtype(int dtype) { return dtype == MHLA_BF16 || dtype == MHLA_F32; }

// Byte span [lo, hi) a [B, N, H, d] tensor can touch.
void span(const mhla_tensor_t* t, uintptr_t* lo, uintptr_t* hi) {
  const int64_t e = elem_bytes(t->dtype);
  const int64_t last = (t->B - 1) * t->stride_b + (t->N - 1) * t->stride_n + (t->H - 1) * t->stride_h + t->d;
  *lo = reinterpret_cast<uintptr_t>(t->data);
  *hi = *lo + static_cast<uintptr_t>(last * e);
}

bool overlaps(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) { return a0 < b1 && b0 < a1; }

// No two (b, n, h, c) index tuples of an output may share an address: sort the
// three outer dimensions by stride and require each stride to clear the extent
// of everything inside it.
bool non_overlapping(const mhla_tensor_t* t) {
  struct Dim { int64_t stride, extent; } dims[3] = {
      {t->stride_b, t->B}, {t->stride_n, t->N}, {t->stride_h, t->H}};
  std::sort(dims, dims + 3, [](const Dim& a, const Dim& b) { return a.stride < b.stride; });
  int64_t inner = t->d;   // elements spanned so far
  for (const Dim& dm : dims) {
    if (dm.extent <= 1) continue;
    if (dm.stride < inner) return false;
    inner = dm.stride * (dm.extent - 1) + inner;
  }
  return true;
}

int check_tensor(const mhla_tensor_t* t) {
  if (!t) return MHLA_ERR_INVALID_ARG;
  if (!valid_dtype(t->dtype)) return MHLA_ERR_INVALID_ARG;
  if (t->B < 0 || t->N < 1 || t->H < 0 || t->d < 1 || t->d > 128) return MHLA_ERR_INVALID_ARG;
  if (t->stride_b < 0 || t->stride_n < 0 || t->stride_h < 0) return MHLA_ERR_INVALID_ARG;
  if (t->B > 0 && t->H > 0 && !t->data) return MHLA_ERR_INVALID_ARG;
  return MHLA_OK;
}

bool same_shape(const mhla_tensor_t* a, const mhla_tensor_t* b) {
  return a->B == b->B && a->N == b->N && a->H == b->H && a->d == b->d && a->dtype == b->dtype;
}

int build_problem(const mhla_tensor_t* q, const mhla_tensor_t* k, const mhla_tensor_t* v,
                  const mhla_tensor_t* o, const mhla_shape3_t* grid, const mhla_shape3_t* block,
                  const mhla_phi_t* phi, bool check_alias, Problem* p) {
  for (const mhla_tensor_t* t : {q, k, v, o}) {
    const int rc = check_tensor(t);
    if (rc != MHLA_OK) return rc;
  }
  if (!same_shape(q, k) || !same_shape(q, v) || !same_shape(q, o)) return MHLA_ERR_SHAPE;
  if (!grid || !block) return MHLA_ERR_INVALID_ARG;
  const int64_t M = mhla_num_blocks(grid, block);
  if (M < 0) return static_cast<int>(-M);
  int64_t n_grid = 1;
  for (int a = 0; a < grid->ndim; ++a) n_grid *= grid->extent[a];
  if (n_grid != q->N) return MHLA_ERR_SHAPE;
  if (phi) {
    if (phi->kind != MHLA_PHI_RELU && phi->kind != MHLA_PHI_RELU_EPS) return MHLA_ERR_INVALID_ARG;
    if (!(phi->eps >= 0.0f) || !std::isfinite(phi->eps)) return MHLA_ERR_INVALID_ARG;
  }
  Problem& P = *p;
  P.B = q->B; P.N = q->N; P.H = q->H; P.d = q->d; P.dtype = q->dtype;
  P.ndim = grid->ndim;
  if (grid->ndim == 2) {
    P.T = 1; P.Y = grid->extent[0]; P.X = grid->extent[1];
    P.bt = 1; P.by = block->extent[0]; P.bx = block->extent[1];
  } else {
    P.T = grid->extent[0]; P.Y = grid->extent[1]; P.X = grid->extent[2];
    P.bt = block->extent[0]; P.by = block->extent[1]; P.bx = block->extent[2];
  }
  P.nbt = P.T / P.bt; P.nby = P.Y / P.by; P.nbx = P.X / P.bx;
  P.M = M; P.w = P.N / M;
  P.phi_kind = phi ? phi->kind : MHLA_PHI_RELU;
  P.eps = phi ? phi->eps : 1e-6f;
  P.q = Operand{q->data, q->stride_b, q->stride_n, q->stride_h};
  P.k = Operand{k->data, k->stride_b, k->stride_n, k->stride_h};
  P.v = Operand{v->data, v->stride_b, v->stride_n, v->stride_h};
  P.o = Operand{o->data, o->stride_b, o->stride_n, o->stride_h};
  if (check_alias && P.B > 0 && P.H > 0) {
    if (!non_overlapping(o)) return MHLA_ERR_INVALID_ARG;
    uintptr_t o0, o1;
    span(o, &o0, &o1);
    for (const mhla_tensor_t* t : {q, k, v}) {
      uintptr_t t0, t1;
      span(t, &t0, &t1);
      if (overlaps(o0, o1, t0, t1)) return MHLA_ERR_INVALID_ARG;
    }
  }
  return MHLA_OK;
}

// W (M x M float32) must not overlap the output the call writes.
bool w_overlaps_out(const mhla_tensor_t* out, const float* W, int64_t M) {
  uintptr_t o0, o1;
  span(out, &o0, &o1);
  const uintptr_t w0 = reinterpret_cast<uintptr_t>(W);
  return overlaps(o0, o1, w0, w0 + static_cast<uintptr_t>(M * M) * sizeof(float));
}

// AUTO: the fused short-sequence kernel, else the three tensor-core launches,
// else the CUDA cores.
int auto_path(const Problem& p) {
  if (small_eligible(p)) return MHLA_PATH_FUSED;
  if (tc_eligible(p)) return MHLA_PATH_TC;
  return MHLA_PATH_SIMT;
}

int resolve_path(const Problem& p, int32_t path, int* sel) {
  if (path == MHLA_PATH_AUTO) {
    *sel = auto_path(p);
    return MHLA_OK;
  }
  if (path == MHLA_PATH_SIMT) { *sel = MHLA_PATH_SIMT; return MHLA_OK; }
  if (path == MHLA_PATH_TC) {
    if (!tc_eligible(p)) return MHLA_ERR_UNSUPPORTED;
    *sel = MHLA_PATH_TC;
    return MHLA_OK;
  }
  if (path == MHLA_PATH_TC_FUSED) {
    if (!tc_fused_eligible(p)) return MHLA_ERR_UNSUPPORTED;
    *sel = MHLA_PATH_TC_FUSED;
    return MHLA_OK;
  }
  if (path == MHLA_PATH_FUSED) {
    if (!small_eligible(p)) return MHLA_ERR_UNSUPPORTED;
    *sel = MHLA_PATH_FUSED;
    return MHLA_OK;
  }
  return MHLA_ERR_INVALID_ARG;
}

size_t workspace_for(const Problem& p, int sel) {
  if (sel == MHLA_PATH_FUSED) return 0;
  return (sel == MHLA_PATH_TC || sel == MHLA_PATH_TC_FUSED) ? tc_workspace_bytes(p) : simt_workspace_bytes(p);
}

}  // namespace
}  // namespace mhla

using namespace mhla;

extern "C" mhla_status_t mhla_workspace_size(const mhla_tensor_t* q, const mhla_shape3_t* grid,
                                             const mhla_shape3_t* block, int32_t path, size_t* bytes) {
  if (!bytes) return MHLA_ERR_INVALID_ARG;
  Problem p;
  const int rc = build_problem(q, q, q, q, grid, block, nullptr, /*check_alias=*/false, &p);
  if (rc != MHLA_OK) return static_cast<mhla_status_t>(rc);
  if (p.B == 0 || p.H == 0) { *bytes = 0; return MHLA_OK; }
  int sel = 0;
  const int rp = resolve_path(p, path, &sel);
  if (rp != MHLA_OK) return static_cast<mhla_status_t>(rp);
  *bytes = workspace_for(p, sel);
  return MHLA_OK;
}

extern "C" int32_t mhla_select_path(const mhla_tensor_t* q, const mhla_tensor_t* k, const mhla_tensor_t* v,
                                    const mhla_tensor_t* out, const mhla_shape3_t* grid,
                                    const mhla_shape3_t* block) {
  Problem p;
  const int rc = build_problem(q, k, v, out, grid, block, nullptr, true, &p);
  if (rc != MHLA_OK) return -rc;
  return auto_path(p);
}

extern "C" mhla_status_t mhla_forward(const mhla_tensor_t* q, const mhla_tensor_t* k, const mhla_tensor_t* v,
                                      const float* W, const mhla_shape3_t* grid, const mhla_shape3_t* block,
                                      const mhla_phi_t* phi, const mhla_tensor_t* out, void* workspace,
                                      size_t workspace_bytes, void* stream, int32_t path) {
  if (!phi) return MHLA_ERR_INVALID_ARG;
  Problem p;
  const int rc = build_problem(q, k, v, out, grid, block, phi, true, &p);
  if (rc != MHLA_OK) return static_cast<mhla_status_t>(rc);
  int sel = 0;
  const int rp = resolve_path(p, path, &sel);
  if (rp != MHLA_OK) return static_cast<mhla_status_t>(rp);
  if (p.B == 0 || p.H == 0) return MHLA_OK;
  if (!W) return MHLA_ERR_INVALID_ARG;
  if (w_overlaps_out(out, W, p.M)) return MHLA_ERR_INVALID_ARG;
  const size_t need = workspace_for(p, sel);
  void* ws = workspace;
  if (!ws && workspace_bytes != 0) return MHLA_ERR_WORKSPACE;
  if (ws && (workspace_bytes < need || reinterpret_cast<uintptr_t>(ws) % kAlign != 0)) return MHLA_ERR_WORKSPACE;
  if (sel == MHLA_PATH_FUSED) return static_cast<mhla_status_t>(launch_small(p, W, stream));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bool owned = false;
  if (!ws) {
    if (cudaMallocAsync(&ws, need, s) != cudaSuccess) return MHLA_ERR_CUDA;
    owned = true;
  }
  const int lr = sel == MHLA_PATH_SIMT ? launch_simt(p, W, ws, stream)
                                      : launch_tc(p, W, ws, stream, /*fused=*/sel == MHLA_PATH_TC_FUSED);
  if (owned && cudaFreeAsync(ws, s) != cudaSuccess && lr == MHLA_OK) return MHLA_ERR_CUDA;
  return static_cast<mhla_status_t>(lr);
}

namespace mhla {
namespace {

// AUTO takes the tensor-core backward whenever every operand qualifies.
int resolve_bwd_path(const Problem& p, const BwdOperands& bo, int32_t path, int* sel) {
  if (path == MHLA_PATH_AUTO) {
    *sel = tc_bwd_eligible(p, bo) ? MHLA_PATH_TC : MHLA_PATH_SIMT;
    return MHLA_OK;
  }
  if (path == MHLA_PATH_SIMT) { *sel = MHLA_PATH_SIMT; return MHLA_OK; }
  if (path == MHLA_PATH_TC) {
    if (!tc_bwd_eligible(p, bo)) return MHLA_ERR_UNSUPPORTED;
    *sel = MHLA_PATH_TC;
    return MHLA_OK;
  }
  if (path == MHLA_PATH_FUSED || path == MHLA_PATH_TC_FUSED) return MHLA_ERR_UNSUPPORTED;
  return MHLA_ERR_INVALID_ARG;
}

size_t bwd_workspace_for(const Problem& p, int sel) {
  return sel == MHLA_PATH_TC ? tc_bwd_workspace_bytes(p) : simt_bwd_workspace_bytes(p);
}

}  // namespace
}  // namespace mhla

extern "C" mhla_status_t mhla_backward_workspace_size(const mhla_tensor_t* q, const mhla_shape3_t* grid,
                                                      const mhla_shape3_t* block, int32_t path, size_t* bytes) {
  if (!bytes) return MHLA_ERR_INVALID_ARG;
  Problem p;
  const int rc = build_problem(q, q, q, q, grid, block, nullptr, /*check_alias=*/false, &p);
  if (rc != MHLA_OK) return static_cast<mhla_status_t>(rc);
  // Only q is known here: the operands of the later call take q's strides.
  BwdOperands bo;
  bo.dout = bo.dq = bo.dk = bo.dv = p.q;
  bo.dW = nullptr;
  int sel = 0;
  const int rp = resolve_bwd_path(p, bo, path, &sel);
  if (rp != MHLA_OK) return static_cast<mhla_status_t>(rp);
  if (p.B == 0 || p.H == 0) {
    *bytes = 0;
  } else if (path == MHLA_PATH_AUTO && sel == MHLA_PATH_TC) {
    // enough for either path, whichever AUTO takes for the actual operands
    *bytes = std::max(tc_bwd_workspace_bytes(p), simt_bwd_workspace_bytes(p));
  } else {
    *bytes = bwd_workspace_for(p, sel);
  }
  return MHLA_OK;
}

namespace mhla {
namespace {

// The operand checks both backward entries share: dq, dk, dv shaped like q
// (check_bwd_operands); every written tensor free of self-overlap and disjoint
// from everything else (check_bwd_overlaps).
int check_bwd_operands(const mhla_tensor_t* q, const mhla_tensor_t* dout, const mhla_tensor_t* dq,
                       const mhla_tensor_t* dk, const mhla_tensor_t* dv, float* dW, BwdOperands* bo) {
  for (const mhla_tensor_t* t : {dq, dk, dv}) {
    const int rt = check_tensor(t);
    if (rt != MHLA_OK) return rt;
    if (!same_shape(q, t)) return MHLA_ERR_SHAPE;
  }
  bo->dout = Operand{dout->data, dout->stride_b, dout->stride_n, dout->stride_h};
  bo->dq = Operand{dq->data, dq->stride_b, dq->stride_n, dq->stride_h};
  bo->dk = Operand{dk->data, dk->stride_b, dk->stride_n, dk->stride_h};
  bo->dv = Operand{dv->data, dv->stride_b, dv->stride_n, dv->stride_h};
  bo->dW = dW;
  return MHLA_OK;
}

int check_bwd_overlaps(const Problem& p, const mhla_tensor_t* q, const mhla_tensor_t* k, const mhla_tensor_t* v,
                       const float* W, const mhla_tensor_t* dout, const mhla_tensor_t* dq, const mhla_tensor_t* dk,
                       const mhla_tensor_t* dv, const float* dW) {
  if (!W || !dW) return MHLA_ERR_INVALID_ARG;
  const uintptr_t w_bytes = static_cast<uintptr_t>(p.M * p.M) * sizeof(float);
  const uintptr_t dw0 = reinterpret_cast<uintptr_t>(dW), dw1 = dw0 + w_bytes;
  const uintptr_t wi0 = reinterpret_cast<uintptr_t>(W), wi1 = wi0 + w_bytes;
  if (overlaps(dw0, dw1, wi0, wi1)) return MHLA_ERR_INVALID_ARG;
  if (p.B > 0 && p.H > 0) {
    uintptr_t lo[7], hi[7];
    const mhla_tensor_t* all[7] = {dq, dk, dv, q, k, v, dout};
    for (int a = 0; a < 7; ++a) span(all[a], &lo[a], &hi[a]);
    for (int a = 0; a < 3; ++a) {
      if (!non_overlapping(all[a])) return MHLA_ERR_INVALID_ARG;
      for (int b = 0; b < 7; ++b)
        if (b != a && overlaps(lo[a], hi[a], lo[b], hi[b])) return MHLA_ERR_INVALID_ARG;
      if (overlaps(lo[a], hi[a], dw0, dw1) || overlaps(lo[a], hi[a], wi0, wi1)) return MHLA_ERR_INVALID_ARG;
    }
    for (int b = 3; b < 7; ++b)
      if (overlaps(lo[b], hi[b], dw0, dw1)) return MHLA_ERR_INVALID_ARG;
  }
  return MHLA_OK;
}

// Runs a backward launcher with the caller's workspace or a stream-ordered
// allocation; B == 0 or H == 0 only zeroes dW.
template <typename Launch>
int run_bwd(const Problem& p, float* dW, size_t need, void* workspace, size_t workspace_bytes, void* stream,
            Launch launch) {
  void* ws = workspace;
  if (!ws && workspace_bytes != 0) return MHLA_ERR_WORKSPACE;
  if (ws && (workspace_bytes < need || reinterpret_cast<uintptr_t>(ws) % kAlign != 0)) return MHLA_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.B == 0 || p.H == 0)   // no (b, h) contributes: dW is zero
    return cudaMemsetAsync(dW, 0, static_cast<size_t>(p.M * p.M) * sizeof(float), s) == cudaSuccess ? MHLA_OK
                                                                                                    : MHLA_ERR_CUDA;
  bool owned = false;
  if (!ws) {
    if (cudaMallocAsync(&ws, need, s) != cudaSuccess) return MHLA_ERR_CUDA;
    owned = true;
  }
  const int lr = launch(ws);
  if (owned && cudaFreeAsync(ws, s) != cudaSuccess && lr == MHLA_OK) return MHLA_ERR_CUDA;
  return lr;
}

}  // namespace
}  // namespace mhla

extern "C" mhla_status_t mhla_backward(const mhla_tensor_t* q, const mhla_tensor_t* k, const mhla_tensor_t* v,
                                       const float* W, const mhla_shape3_t* grid, const mhla_shape3_t* block,
                                       const mhla_phi_t* phi, const mhla_tensor_t* dout, const mhla_tensor_t* dq,
                                       const mhla_tensor_t* dk, const mhla_tensor_t* dv, float* dW,
                                       void* workspace, size_t workspace_bytes, void* stream, int32_t path) {
  if (!phi) return MHLA_ERR_INVALID_ARG;
  Problem p;
  const int rc = build_problem(q, k, v, dout, grid, block, phi, /*check_alias=*/false, &p);
  if (rc != MHLA_OK) return static_cast<mhla_status_t>(rc);
  BwdOperands bo;
  const int ro = check_bwd_operands(q, dout, dq, dk, dv, dW, &bo);
  if (ro != MHLA_OK) return static_cast<mhla_status_t>(ro);
  int sel = 0;
  const int rp = resolve_bwd_path(p, bo, path, &sel);
  if (rp != MHLA_OK) return static_cast<mhla_status_t>(rp);
  const int rv = check_bwd_overlaps(p, q, k, v, W, dout, dq, dk, dv, dW);
  if (rv != MHLA_OK) return static_cast<mhla_status_t>(rv);
  const size_t need = (p.B == 0 || p.H == 0) ? 0 : bwd_workspace_for(p, sel);
  return static_cast<mhla_status_t>(run_bwd(p, dW, need, workspace, workspace_bytes, stream, [&](void* ws) {
    return sel == MHLA_PATH_TC ? launch_tc_bwd(p, W, bo, ws, stream) : launch_simt_bwd(p, W, bo, ws, stream);
  }));
}

namespace mhla {
namespace {

// The causal backward's token kernels run on CUDA cores.  TC: the summaries and
// the mixing come from the tensor-core causal forward's kernels (every block one
// unit of its tiling); AUTO takes that whenever it applies.  SIMT: CUDA cores
// throughout.
int resolve_causal_bwd_path(const Problem& p, int32_t path, int* sel) {
  if (path == MHLA_PATH_AUTO) {
    *sel = tc_causal_states_eligible(p) ? MHLA_PATH_TC : MHLA_PATH_SIMT;
    return MHLA_OK;
  }
  if (path == MHLA_PATH_SIMT) { *sel = MHLA_PATH_SIMT; return MHLA_OK; }
  if (path == MHLA_PATH_TC) {
    if (!tc_causal_states_eligible(p)) return MHLA_ERR_UNSUPPORTED;
    *sel = MHLA_PATH_TC;
    return MHLA_OK;
  }
  if (path == MHLA_PATH_FUSED || path == MHLA_PATH_TC_FUSED) return MHLA_ERR_UNSUPPORTED;
  return MHLA_ERR_INVALID_ARG;
}

}  // namespace
}  // namespace mhla

extern "C" mhla_status_t mhla_backward_causal_workspace_size(const mhla_tensor_t* q, const mhla_shape3_t* grid,
                                                             const mhla_shape3_t* block, int32_t path,
                                                             size_t* bytes) {
  if (!bytes) return MHLA_ERR_INVALID_ARG;
  Problem p;
  const int rc = build_problem(q, q, q, q, grid, block, nullptr, /*check_alias=*/false, &p);
  if (rc != MHLA_OK) return static_cast<mhla_status_t>(rc);
  if (!blocks_contiguous(p)) return MHLA_ERR_SHAPE;
  int sel = 0;
  const int rp = resolve_causal_bwd_path(p, path, &sel);
  if (rp != MHLA_OK) return static_cast<mhla_status_t>(rp);
  *bytes = (p.B == 0 || p.H == 0) ? 0 : simt_causal_bwd_workspace_bytes(p, sel == MHLA_PATH_TC);
  return MHLA_OK;
}

extern "C" mhla_status_t mhla_backward_causal(const mhla_tensor_t* q, const mhla_tensor_t* k,
                                              const mhla_tensor_t* v, const float* W, const mhla_shape3_t* grid,
                                              const mhla_shape3_t* block, const mhla_phi_t* phi,
                                              const mhla_tensor_t* dout, const mhla_tensor_t* dq,
                                              const mhla_tensor_t* dk, const mhla_tensor_t* dv, float* dW,
                                              void* workspace, size_t workspace_bytes, void* stream, int32_t path) {
  if (!phi) return MHLA_ERR_INVALID_ARG;
  Problem p;
  const int rc = build_problem(q, k, v, dout, grid, block, phi, /*check_alias=*/false, &p);
  if (rc != MHLA_OK) return static_cast<mhla_status_t>(rc);
  if (!blocks_contiguous(p)) return MHLA_ERR_SHAPE;
  BwdOperands bo;
  const int ro = check_bwd_operands(q, dout, dq, dk, dv, dW, &bo);
  if (ro != MHLA_OK) return static_cast<mhla_status_t>(ro);
  int sel = 0;
  const int rp = resolve_causal_bwd_path(p, path, &sel);
  if (rp != MHLA_OK) return static_cast<mhla_status_t>(rp);
  const int rv = check_bwd_overlaps(p, q, k, v, W, dout, dq, dk, dv, dW);
  if (rv != MHLA_OK) return static_cast<mhla_status_t>(rv);
  const bool tc_states = sel == MHLA_PATH_TC;
  const size_t need = (p.B == 0 || p.H == 0) ? 0 : simt_causal_bwd_workspace_bytes(p, tc_states);
  return static_cast<mhla_status_t>(run_bwd(p, dW, need, workspace, workspace_bytes, stream, [&](void* ws) {
    return launch_simt_causal_bwd(p, W, bo, ws, stream, tc_states);
  }));
}

namespace mhla {
namespace {

int resolve_causal_path(const Problem& p, int32_t path, int* sel) {
  if (path == MHLA_PATH_AUTO) {
    *sel = tc_causal_eligible(p) ? MHLA_PATH_TC : MHLA_PATH_SIMT;
    return MHLA_OK;
  }
  if (path == MHLA_PATH_SIMT) { *sel = MHLA_PATH_SIMT; return MHLA_OK; }
  if (path == MHLA_PATH_TC) {
    if (!tc_causal_eligible(p)) return MHLA_ERR_UNSUPPORTED;
    *sel = MHLA_PATH_TC;
    return MHLA_OK;
  }
  if (path == MHLA_PATH_FUSED || path == MHLA_PATH_TC_FUSED) return MHLA_ERR_UNSUPPORTED;
  return MHLA_ERR_INVALID_ARG;
}

size_t causal_workspace_for(const Problem& p, int sel) {
  return sel == MHLA_PATH_TC ? tc_causal_workspace_bytes(p) : simt_workspace_bytes(p);
}

}  // namespace
}  // namespace mhla

extern "C" mhla_status_t mhla_causal_workspace_size(const mhla_tensor_t* q, const mhla_shape3_t* grid,
                                                    const mhla_shape3_t* block, int32_t path, size_t* bytes) {
  if (!bytes) return MHLA_ERR_INVALID_ARG;
  Problem p;
  const int rc = build_problem(q, q, q, q, grid, block, nullptr, /*check_alias=*/false, &p);
  if (rc != MHLA_OK) return static_cast<mhla_status_t>(rc);
  if (!blocks_contiguous(p)) return MHLA_ERR_SHAPE;
  int sel = 0;
  const int rp = resolve_causal_path(p, path, &sel);
  if (rp != MHLA_OK) return static_cast<mhla_status_t>(rp);
  if (p.B == 0 || p.H == 0) {
    *bytes = 0;
  } else if (path == MHLA_PATH_AUTO && sel == MHLA_PATH_TC) {
    // only q is known here: enough for either path, whichever AUTO takes
    *bytes = std::max(tc_causal_workspace_bytes(p), simt_workspace_bytes(p));
  } else {
    *bytes = causal_workspace_for(p, sel);
  }
  return MHLA_OK;
}

extern "C" mhla_status_t mhla_forward_causal(const mhla_tensor_t* q, const mhla_tensor_t* k, const mhla_tensor_t* v,
                                             const float* W, const mhla_shape3_t* grid, const mhla_shape3_t* block,
                                             const mhla_phi_t* phi, const mhla_tensor_t* out, void* workspace,
                                             size_t workspace_bytes, void* stream, int32_t path) {
  if (!phi) return MHLA_ERR_INVALID_ARG;
  Problem p;
  const int rc = build_problem(q, k, v, out, grid, block, phi, true, &p);
  if (rc != MHLA_OK) return static_cast<mhla_status_t>(rc);
  if (!blocks_contiguous(p)) return MHLA_ERR_SHAPE;
  int sel = 0;
  const int rp = resolve_causal_path(p, path, &sel);
  if (rp != MHLA_OK) return static_cast<mhla_status_t>(rp);
  if (p.B == 0 || p.H == 0) return MHLA_OK;
  if (!W) return MHLA_ERR_INVALID_ARG;
  if (w_overlaps_out(out, W, p.M)) return MHLA_ERR_INVALID_ARG;
  const size_t need = causal_workspace_for(p, sel);
  void* ws = workspace;
  if (!ws && workspace_bytes != 0) return MHLA_ERR_WORKSPACE;
  if (ws && (workspace_bytes < need || reinterpret_cast<uintptr_t>(ws) % kAlign != 0)) return MHLA_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bool owned = false;
  if (!ws) {
    if (cudaMallocAsync(&ws, need, s) != cudaSuccess) return MHLA_ERR_CUDA;
    owned = true;
  }
  const int lr = sel == MHLA_PATH_TC ? launch_tc_causal(p, W, ws, stream) : launch_simt_causal(p, W, ws, stream);
  if (owned && cudaFreeAsync(ws, s) != cudaSuccess && lr == MHLA_OK) return MHLA_ERR_CUDA;
  return static_cast<mhla_status_t>(lr);
}

extern "C" mhla_status_t mhla_device_status(void* stream, uint32_t* flags) {
  if (!flags) return MHLA_ERR_INVALID_ARG;
  uint32_t tc = 0, small = 0, bwd = 0, causal = 0, module = 0, gemm = 0;
  const int a = read_and_clear_device_error(stream, &tc);
  const int b = read_and_clear_small_error(stream, &small);
  const int c = read_and_clear_bwd_error(stream, &bwd);
  const int e = read_and_clear_causal_error(stream, &causal);
  const int f = read_and_clear_module_error(stream, &module);
  const int g = read_and_clear_gemm_error(stream, &gemm);
  if (a == MHLA_ERR_CUDA || b == MHLA_ERR_CUDA || c == MHLA_ERR_CUDA || e == MHLA_ERR_CUDA || f == MHLA_ERR_CUDA ||
      g == MHLA_ERR_CUDA)
    return MHLA_ERR_CUDA;
  *flags = tc | small | bwd | causal | module | gemm;
  return *flags ? MHLA_ERR_TIMEOUT : MHLA_OK;
}

extern "C" mhla_status_t mhla_debug_stall_waits(int32_t warp, uint64_t limit_ns) {
  if (warp < -1 || warp >= 32) return MHLA_ERR_INVALID_ARG;
  if (warp >= 0 && (limit_ns < 1000 || limit_ns > 1000000000ull)) return MHLA_ERR_INVALID_ARG;
  const uint32_t w = warp < 0 ? 0u : static_cast<uint32_t>(warp) + 1u;
  const uint64_t ns = warp < 0 ? 0 : limit_ns;
  int (*const setters[])(uint32_t, uint64_t) = {set_stall_summary, set_stall_mix, set_stall_output,
                                                set_stall_fused,   set_stall_small, set_stall_bwd,
                                                set_stall_causal,  set_stall_module, set_stall_gemm};
  for (auto set : setters)
    if (set(w, ns) != MHLA_OK) return MHLA_ERR_CUDA;
  return MHLA_OK;
}

extern "C" const char* mhla_status_string(int32_t status) {
  switch (status) {
    case MHLA_OK: return "ok";
    case MHLA_ERR_INVALID_ARG: return "invalid argument";
    case MHLA_ERR_SHAPE: return "shape mismatch";
    case MHLA_ERR_UNSUPPORTED: return "unsupported by the selected path";
    case MHLA_ERR_CUDA: return "CUDA error";
    case MHLA_ERR_TIMEOUT: return "device wait timed out";
    case MHLA_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    default: return "unknown status";
  }
}

extern "C" const char* mhla_version(void) { return "mhla-gb300 0.1.0 sm_103a"; }

// ----------------------------------------------------------------- module

namespace mhla {
namespace {

bool aligned16(const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

int check_grid_tokens(const mhla_shape3_t* grid, int64_t N, int64_t* T, int64_t* Y, int64_t* X) {
  if (!grid || (grid->ndim != 2 && grid->ndim != 3)) return MHLA_ERR_INVALID_ARG;
  int64_t n = 1;
  for (int a = 0; a < grid->ndim; ++a) {
    if (grid->extent[a] < 1) return MHLA_ERR_SHAPE;
    n *= grid->extent[a];
  }
  if (n != N) return MHLA_ERR_SHAPE;
  *T = grid->ndim == 3 ? grid->extent[0] : 1;
  *Y = grid->extent[grid->ndim - 2];
  *X = grid->extent[grid->ndim - 1];
  return MHLA_OK;
}

bool lepe_view_ok(const mhla_tensor_t* t) {
  return t->dtype == MHLA_BF16 && t->d % 8 == 0 && t->stride_b % 8 == 0 && t->stride_n % 8 == 0 &&
         t->stride_h % 8 == 0 && aligned16(t->data);
}

// v and out move by TMA as (channel, x, y, frame, batch): heads adjacent.
bool lepe_tma_ok(const mhla_tensor_t* v, int64_t T, int64_t Y, int64_t X) {
  if (v->H > 1 && v->stride_h != v->d) return false;
  if (v->stride_n < v->H * v->d) return false;
  const int64_t lim = int64_t{1} << 39;   // bytes / 2
  return v->stride_n * X * Y * T < lim && v->stride_b < lim && v->H * v->d < (int64_t{1} << 31);
}

int lepe_args(const mhla_tensor_t* v, const mhla_tensor_t* out, const mhla_shape3_t* grid, const float* weight,
              const float* bias, LepeArgs* a) {
  for (const mhla_tensor_t* t : {v, out}) {
    const int rc = check_tensor(t);
    if (rc != MHLA_OK) return rc;
  }
  if (!same_shape(v, out)) return MHLA_ERR_SHAPE;
  int64_t T, Y, X;
  const int rg = check_grid_tokens(grid, v->N, &T, &Y, &X);
  if (rg != MHLA_OK) return rg;
  if (!lepe_view_ok(v) || !lepe_view_ok(out) || !lepe_tma_ok(v, T, Y, X) || !lepe_tma_ok(out, T, Y, X))
    return MHLA_ERR_UNSUPPORTED;
  if (v->B > 0 && v->H > 0) {
    if (!weight || !bias) return MHLA_ERR_INVALID_ARG;
    if (!non_overlapping(out)) return MHLA_ERR_INVALID_ARG;
    uintptr_t o0, o1, v0, v1;
    span(out, &o0, &o1);
    span(v, &v0, &v1);
    if (overlaps(o0, o1, v0, v1)) return MHLA_ERR_INVALID_ARG;
  }
  // The kernel keeps channels, frames, rows and columns in 32 bits (TMA
  // coordinates) and the tile index in 64.
  const int64_t lim32 = int64_t{1} << 30;
  if (v->H * v->d > lim32 || v->B >= lim32 || T >= lim32 || Y >= lim32 || X >= lim32) return MHLA_ERR_UNSUPPORTED;
  a->v = v->data;
  a->o = out->data;
  a->vsb = v->stride_b; a->vsn = v->stride_n; a->vsh = v->stride_h;
  a->osb = out->stride_b; a->osn = out->stride_n; a->osh = out->stride_h;
  a->B = v->B;
  a->d = static_cast<int32_t>(v->d);
  a->C = static_cast<int32_t>(v->H * v->d);
  a->T = static_cast<int32_t>(T); a->Y = static_cast<int32_t>(Y); a->X = static_cast<int32_t>(X);
  a->weight = weight;
  a->bias = bias;
  return MHLA_OK;
}

// Buffers of the module inside its workspace.
struct ModuleLayout {
  size_t a_off, qkv_off, core_off, total;
};

// The core's [B, N, heads, d] views of the projection and of the output buffer.
void module_views(void* qkv, void* obuf, int64_t B, int64_t N, int64_t C, int32_t heads, mhla_tensor_t* q,
                  mhla_tensor_t* k, mhla_tensor_t* v, mhla_tensor_t* o) {
  const int64_t d = C / heads;
  auto* base = static_cast<uint16_t*>(qkv);
  mhla_tensor_t* views[3] = {q, k, v};
  for (int s = 0; s < 3; ++s) {
    mhla_tensor_t& t = *views[s];
    t.data = qkv ? base + s * C : nullptr;
    t.dtype = MHLA_BF16;
    t.pad_ = 0;
    t.B = B; t.N = N; t.H = heads; t.d = d;
    t.stride_b = N * 3 * C; t.stride_n = 3 * C; t.stride_h = d;
  }
  o->data = obuf;
  o->dtype = MHLA_BF16;
  o->pad_ = 0;
  o->B = B; o->N = N; o->H = heads; o->d = d;
  o->stride_b = N * C; o->stride_n = C; o->stride_h = d;
}

int module_check(int64_t B, int64_t N, int64_t C, int32_t heads, const mhla_shape3_t* grid,
                 const mhla_shape3_t* block) {
  if (B < 0 || N < 1 || C < 8 || heads < 1 || C % heads != 0) return MHLA_ERR_INVALID_ARG;
  if (C % 8 != 0 || C > 2048 || (C / heads) % 8 != 0 || C / heads > 128) return MHLA_ERR_UNSUPPORTED;
  if (!grid || !block) return MHLA_ERR_INVALID_ARG;
  int64_t T, Y, X;
  const int rg = check_grid_tokens(grid, N, &T, &Y, &X);
  if (rg != MHLA_OK) return rg;
  const int64_t M = mhla_num_blocks(grid, block);
  if (M < 0) return static_cast<int>(-M);
  if (B * N >= (int64_t{1} << 31)) return MHLA_ERR_UNSUPPORTED;   // the projections' row coordinate
  return MHLA_OK;
}

int module_layout(int64_t B, int64_t N, int64_t C, int32_t heads, const mhla_shape3_t* grid,
                  const mhla_shape3_t* block, ModuleLayout* L) {
  const int64_t R = B * N;
  mhla_tensor_t q, k, v, o;
  // a 256-byte aligned stand-in address: the core's path choice depends on alignment, not on the value
  module_views(reinterpret_cast<void*>(uintptr_t{1} << 20), reinterpret_cast<void*>(uintptr_t{1} << 21), B, N, C,
               heads, &q, &k, &v, &o);
  size_t core = 0;
  const mhla_status_t rc = mhla_workspace_size(&q, grid, block, MHLA_PATH_AUTO, &core);
  if (rc != MHLA_OK) return rc;
  size_t off = 0;
  L->a_off = off;
  off += align_up(static_cast<size_t>(R) * C * 2);
  L->qkv_off = off;
  off += align_up(static_cast<size_t>(R) * 3 * C * 2);
  L->core_off = off;
  off += align_up(core);
  L->total = off;
  return MHLA_OK;
}

}  // namespace
}  // namespace mhla

extern "C" mhla_status_t mhla_layer_norm(const void* x, void* y, int64_t rows, int64_t C, const float* weight,
                                         const float* bias, float eps, void* stream) {
  if (rows < 0 || C < 8) return MHLA_ERR_INVALID_ARG;
  if (C % 8 != 0 || C > 2048) return MHLA_ERR_UNSUPPORTED;
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return MHLA_ERR_INVALID_ARG;
  if (rows == 0) return MHLA_OK;
  if (!x || !y || !weight || !bias) return MHLA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || !aligned16(weight) || !aligned16(bias)) return MHLA_ERR_INVALID_ARG;
  const uintptr_t x0 = reinterpret_cast<uintptr_t>(x), y0 = reinterpret_cast<uintptr_t>(y);
  const uintptr_t n = static_cast<uintptr_t>(rows * C * 2);
  if (x0 != y0 && overlaps(x0, x0 + n, y0, y0 + n)) return MHLA_ERR_INVALID_ARG;
  if ((rows + 7) / 8 >= (int64_t{1} << 31)) return MHLA_ERR_UNSUPPORTED;
  return static_cast<mhla_status_t>(
      launch_layer_norm(x, y, rows, static_cast<int32_t>(C), weight, bias, eps, stream));
}

extern "C" mhla_status_t mhla_linear(const void* x, const void* w, const void* bias, void* y, int64_t rows, int64_t k,
                                     int64_t n_out, void* stream) {
  if (rows < 0 || k < 1 || n_out < 1) return MHLA_ERR_INVALID_ARG;
  if (!gemm_supported(rows == 0 ? 1 : rows, k, n_out)) return MHLA_ERR_UNSUPPORTED;
  if (rows == 0) return MHLA_OK;
  if (!x || !w || !y) return MHLA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (bias && !aligned16(bias))) return MHLA_ERR_INVALID_ARG;
  const uintptr_t y0 = reinterpret_cast<uintptr_t>(y), y1 = y0 + static_cast<uintptr_t>(rows * n_out * 2);
  const uintptr_t x0 = reinterpret_cast<uintptr_t>(x), w0 = reinterpret_cast<uintptr_t>(w);
  if (overlaps(y0, y1, x0, x0 + static_cast<uintptr_t>(rows * k * 2)) ||
      overlaps(y0, y1, w0, w0 + static_cast<uintptr_t>(n_out * k * 2)))
    return MHLA_ERR_INVALID_ARG;
  if (bias) {
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(bias);
    if (overlaps(y0, y1, b0, b0 + static_cast<uintptr_t>(n_out * 2))) return MHLA_ERR_INVALID_ARG;
  }
  return static_cast<mhla_status_t>(launch_gemm("mhla_gemm", x, w, bias, y, rows, k, n_out, stream));
}

extern "C" mhla_status_t mhla_lepe_add(const mhla_tensor_t* v, const mhla_tensor_t* out, const mhla_shape3_t* grid,
                                       const float* weight, const float* bias, void* stream) {
  LepeArgs a = {};
  const int rc = lepe_args(v, out, grid, weight, bias, &a);
  if (rc != MHLA_OK) return static_cast<mhla_status_t>(rc);
  if (v->B == 0 || v->H == 0) return MHLA_OK;
  return static_cast<mhla_status_t>(launch_lepe_add(a, stream));
}

extern "C" mhla_status_t mhla_module_workspace_size(int64_t B, int64_t N, int64_t C, int32_t heads,
                                                    const mhla_shape3_t* grid, const mhla_shape3_t* block,
                                                    size_t* bytes) {
  if (!bytes) return MHLA_ERR_INVALID_ARG;
  const int rc = module_check(B, N, C, heads, grid, block);
  if (rc != MHLA_OK) return static_cast<mhla_status_t>(rc);
  if (B == 0) { *bytes = 0; return MHLA_OK; }
  ModuleLayout L;
  const int rl = module_layout(B, N, C, heads, grid, block, &L);
  if (rl != MHLA_OK) return static_cast<mhla_status_t>(rl);
  *bytes = L.total;
  return MHLA_OK;
}

extern "C" mhla_status_t mhla_module_forward(const void* x, void* y, int64_t B, int64_t N, int64_t C,
                                             const mhla_module_params_t* params, const float* W,
                                             const mhla_shape3_t* grid, const mhla_shape3_t* block,
                                             const mhla_phi_t* phi, void* workspace, size_t workspace_bytes,
                                             void* stream) {
  if (!params || !phi) return MHLA_ERR_INVALID_ARG;
  const int rc = module_check(B, N, C, params->heads, grid, block);
  if (rc != MHLA_OK) return static_cast<mhla_status_t>(rc);
  if (B == 0) return MHLA_OK;
  if (!x || !y || !W || !params->ln_weight || !params->ln_bias || !params->qkv_weight || !params->out_weight)
    return MHLA_ERR_INVALID_ARG;
  if (params->lepe_weight && !params->lepe_bias) return MHLA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || !aligned16(params->ln_weight) || !aligned16(params->ln_bias) ||
      !aligned16(params->qkv_weight) || !aligned16(params->out_weight))
    return MHLA_ERR_INVALID_ARG;
  if (!(params->ln_eps >= 0.0f) || !std::isfinite(params->ln_eps)) return MHLA_ERR_INVALID_ARG;
  if ((params->qkv_bias && !aligned16(params->qkv_bias)) || (params->out_bias && !aligned16(params->out_bias)))
    return MHLA_ERR_INVALID_ARG;
  ModuleLayout L;
  const int rl = module_layout(B, N, C, params->heads, grid, block, &L);
  if (rl != MHLA_OK) return static_cast<mhla_status_t>(rl);
  void* ws = workspace;
  if (!ws && workspace_bytes != 0) return MHLA_ERR_WORKSPACE;
  if (ws && (workspace_bytes < L.total || reinterpret_cast<uintptr_t>(ws) % kAlign != 0)) return MHLA_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bool owned = false;
  if (!ws) {
    if (cudaMallocAsync(&ws, L.total, s) != cudaSuccess) return MHLA_ERR_CUDA;
    owned = true;
  }
  char* base = static_cast<char*>(ws);
  void* abuf = base + L.a_off;
  void* qkv = base + L.qkv_off;
  const int64_t R = B * N;
  mhla_tensor_t q, k, v, o;
  module_views(qkv, abuf, B, N, C, params->heads, &q, &k, &v, &o);
  // The core's and the positional term's checks run on these views before the
  // first launch, so a request either of them refuses queues nothing.
  Problem core;
  int r = build_problem(&q, &k, &v, &o, grid, block, phi, /*check_alias=*/true, &core);
  if (r == MHLA_OK && w_overlaps_out(&o, W, core.M)) r = MHLA_ERR_INVALID_ARG;
  LepeArgs lepe = {};
  if (r == MHLA_OK && params->lepe_weight)
    r = lepe_args(&v, &o, grid, params->lepe_weight, params->lepe_bias, &lepe);
  if (r == MHLA_OK)
    r = launch_layer_norm(x, abuf, R, static_cast<int32_t>(C), params->ln_weight, params->ln_bias, params->ln_eps,
                          stream);
  if (r == MHLA_OK)
    r = launch_gemm("mhla_gemm_qkv", abuf, params->qkv_weight, params->qkv_bias, qkv, R, C, 3 * C, stream);
  if (r == MHLA_OK)
    r = mhla_forward(&q, &k, &v, W, grid, block, phi, &o, base + L.core_off, L.total - L.core_off, stream,
                     MHLA_PATH_AUTO);
  if (r == MHLA_OK && params->lepe_weight) r = launch_lepe_add(lepe, stream);
  if (r == MHLA_OK) r = launch_gemm("mhla_gemm_out", abuf, params->out_weight, params->out_bias, y, R, C, C, stream);
  if (owned && cudaFreeAsync(ws, s) != cudaSuccess && r == MHLA_OK) return MHLA_ERR_CUDA;
  return static_cast<mhla_status_t>(r);
}
