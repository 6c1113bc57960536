/*
 * mhla.h -- C ABI of the MHLA forward pass (Multi-Head Linear Attention with the
 * heads taken along the token dimension) for NVIDIA GB300 (sm_103a).
 *
 * Sources of the operation (web pages, cited by title and section):
 *   [P1] "MHLA：通过令牌级多头机制恢复线性注意力机制的表达能力" module walkthrough,
 *        171host.com/767426.html, section 5 (principle) and section 7 (the
 *        plug-and-play BlockDistanceConv / MHLA PyTorch module).
 *   [P2] "MHLA: Restoring Expressivity of Linear Attention via Token-Level
 *        Multi-Head", paperlayer.ai summary of arXiv 2601.07832v2, sections 3-4.
 *
 * What one forward computes, per batch b and head h (notation of [P2] section 4):
 *   1. split the N tokens of a 2-D (Y, X) or 3-D (T, Y, X) grid into M
 *      non-overlapping blocks and form every block's summary
 *        S_j = sum_{s in j} phi(k_s) v_s^T   (d x d),   z_j = sum_{s in j} phi(k_s);
 *   2. mix the summaries per query block with the M x M matrix W
 *        S~_i = sum_j W[i][j] S_j,   z~_i = sum_j W[i][j] z_j;
 *   3. read out every token t of query block i
 *        o_t = phi(q_t)^T S~_i / (phi(q_t) . z~_i + eps).
 *   phi is ReLU ([P1] section 7, MHLA._process_qkv_impl), optionally ReLU + eps.
 *
 * Conventions shared by every call:
 *   - Tensors q, k, v, out are [B, N, H, d] with d contiguous (stride 1) and
 *     the N tokens in raster order over the grid (last grid axis fastest).
 *     Strides are in ELEMENTS.  Pointers are borrowed, never freed or kept.
 *   - Block ids are row-major over the block grid, slowest axis first; W is
 *     row-major float32, W[i * M + j], i = query (output) block, j = source
 *     block -- the weight[out][in] of the 1x1 convolution in [P1] section 7.
 *   - Nothing throws across the ABI; every call returns an mhla_status_t.
 *     Validation happens before any GPU work is queued.
 */
#ifndef MHLA_H
#define MHLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mhla_status {
    MHLA_OK = 0,
    MHLA_ERR_INVALID_ARG = 1,  /* null pointer, bad enum, negative or inconsistent size */
    MHLA_ERR_SHAPE = 2,        /* grid does not match N, block does not tile grid, ... */
    MHLA_ERR_UNSUPPORTED = 3,  /* valid request the selected path cannot run */
    MHLA_ERR_CUDA = 4,         /* a CUDA runtime call or a launch failed */
    MHLA_ERR_TIMEOUT = 5,      /* a device-side wait gave up (see mhla_device_status) */
    MHLA_ERR_WORKSPACE = 6     /* workspace missing, too small or misaligned */
} mhla_status_t;

typedef enum mhla_dtype { MHLA_BF16 = 0, MHLA_F32 = 1 } mhla_dtype_t;

/* Distance -> weight transforms of [P1] section 7, BlockDistanceConv._apply_transform. */
typedef enum mhla_transform {
    MHLA_TRANSFORM_LINEAR = 0,    /* 1 - D / max D                         */
    MHLA_TRANSFORM_COS = 1,       /* cos(D / max D * pi / 4)               */
    MHLA_TRANSFORM_EXP = 2,       /* exp(-D / exp_sigma)                   */
    MHLA_TRANSFORM_GAUSSIAN = 3,  /* exp(-D^2 / (2 s^2)), s = max D / 3    */
    MHLA_TRANSFORM_LOCAL = 4      /* 1 if D <= local_thres else 0          */
} mhla_transform_t;

typedef enum mhla_phi_kind {
    MHLA_PHI_RELU = 0,      /* phi(x) = max(x, 0)                               */
    MHLA_PHI_RELU_EPS = 1   /* phi(x) = max(x, 0) + eps, as the [P1] module does */
} mhla_phi_kind_t;

/* Which kernels run.  AUTO takes, in this order, the first path the request is
 * eligible for:
 *   FUSED  one tensor-core launch for short sequences: bf16, d in {32, 64},
 *          N <= 256 tokens, M <= 96 blocks, strides multiples of 8 elements,
 *          16-byte aligned bases.  It forms the same result through the
 *          two-stage form o_t = sum_s P[t][s] v_s / (sum_s P[t][s] + eps),
 *          P[t][s] = W[b(t)][b(s)] phi(q_t) . phi(k_s) ([P2] section 4
 *          "Multi-Head Mixing"; [P1] section 5(4)), needs no workspace and
 *          suits grids with many small blocks (M^2 comparable to N).
 *   TC     three tensor-core launches (summaries, mixing GEMM, readout): bf16,
 *          d in {32, 64}, tokens per block a multiple of 128 in whole block
 *          rows (or contiguous 64-token blocks), TMA friendly strides.
 *   SIMT   CUDA cores, any supported request (float32 included).
 * TC_FUSED, never taken by AUTO, runs TC's three pipelines in one persistent
 * launch (M <= 256, tokens per block a multiple of 128 in whole block rows):
 * some CTAs form the block summaries while the others run the mixing GEMM
 * batch by batch as the summaries arrive, then every CTA reads out.  It gives
 * TC's results bit for bit; on GB300 it is slower than TC (the summaries need
 * every SM to draw full HBM bandwidth), so it is kept for measurement. */
typedef enum mhla_path {
    MHLA_PATH_AUTO = 0,
    MHLA_PATH_SIMT = 1,
    MHLA_PATH_TC = 2,
    MHLA_PATH_FUSED = 3,
    MHLA_PATH_TC_FUSED = 4
} mhla_path_t;

/* Token grid or block shape, slowest axis first: (Y, X) when ndim == 2,
 * (T, Y, X) when ndim == 3.  Unused extents are ignored. */
typedef struct mhla_shape3 {
    int32_t ndim;
    int32_t pad_;
    int64_t extent[3];
} mhla_shape3_t;

typedef struct mhla_phi {
    int32_t kind;   /* mhla_phi_kind_t */
    float eps;      /* added to the denominator; also to phi under MHLA_PHI_RELU_EPS */
} mhla_phi_t;

/* A [B, N, H, d] tensor.  data is device memory for mhla_forward. */
typedef struct mhla_tensor {
    void* data;
    int32_t dtype;  /* mhla_dtype_t */
    int32_t pad_;
    int64_t B, N, H, d;
    int64_t stride_b, stride_n, stride_h;   /* elements; d has stride 1 */
} mhla_tensor_t;

/* Number of token blocks M for a grid and block shape, or -MHLA_ERR_SHAPE /
 * -MHLA_ERR_INVALID_ARG when the block does not tile the grid. */
int64_t mhla_num_blocks(const mhla_shape3_t* grid, const mhla_shape3_t* block);

/* Builds the M x M mixing matrix from block-centre distances: centres at
 * (index + 0.5) per axis in block units, Euclidean distance, the transform,
 * then every column divided by its sum ([P1] section 7,
 * BlockDistanceConv._compute_block_distances and _apply_transform; [P2]
 * section 5 "locality-biased initialization").  Computed in double and rounded
 * once to float32; a single block gives W = [[1]].
 *   W_host      host memory the caller owns, room for W_capacity floats;
 *               receives W[i * M + j].
 * Returns MHLA_ERR_INVALID_ARG for a null pointer, unknown transform, a
 * non-positive exp_sigma or W_capacity < M * M; MHLA_ERR_SHAPE when the block
 * does not tile the grid.  Host only; touches no GPU. */
mhla_status_t mhla_init_mixing(const mhla_shape3_t* grid, const mhla_shape3_t* block,
                               int32_t transform, double local_thres, double exp_sigma,
                               float* W_host, int64_t W_capacity);

/* Device workspace mhla_forward needs for this problem and path (bytes, a
 * multiple of 256).  q gives B, N, H, d and the dtype.  Host only. */
mhla_status_t mhla_workspace_size(const mhla_tensor_t* q, const mhla_shape3_t* grid,
                                  const mhla_shape3_t* block, int32_t path, size_t* bytes);

/* The path AUTO would take for this problem (MHLA_PATH_SIMT, MHLA_PATH_TC or
 * MHLA_PATH_FUSED), or a negative status when the problem is invalid.  Host
 * only. */
int32_t mhla_select_path(const mhla_tensor_t* q, const mhla_tensor_t* k,
                         const mhla_tensor_t* v, const mhla_tensor_t* out,
                         const mhla_shape3_t* grid, const mhla_shape3_t* block);

/* The MHLA forward pass ([P2] section 4 "Architecture", "Multi-Head Mixing",
 * "Token-Level Adaptivity"; [P1] section 7, MHLA.forward with the normaliser
 * read as phi(q_t) . z~_i + eps).
 *   q, k, v     device tensors [B, N, H, d], all the same shape and dtype.
 *   W           device float32, M x M row-major, shared by every batch and head.
 *   grid, block token grid and block shape; prod(grid) == N, block tiles grid.
 *   phi         feature map and eps (eps >= 0, finite).
 *   out         device tensor, same shape and dtype as q; must not overlap
 *               q, k, v or W.  Written in the input dtype (round to nearest even).
 *   workspace   device memory of at least mhla_workspace_size() bytes, 256-byte
 *               aligned, owned by the caller and not used by anything else
 *               until the work queued on stream has finished.  Passing NULL
 *               with workspace_bytes == 0 makes the call take it with
 *               cudaMallocAsync / cudaFreeAsync on the stream.
 *   stream      cudaStream_t (NULL = legacy default stream).
 *   path        mhla_path_t; AUTO unless a test wants one path.
 * Asynchronous: queues kernels on stream and returns; never synchronises.
 * Returns MHLA_ERR_INVALID_ARG / SHAPE / WORKSPACE before queuing anything
 * when the request is malformed, MHLA_ERR_UNSUPPORTED when an explicit path
 * cannot take it, MHLA_ERR_CUDA when a launch fails.  A device-side wait that
 * gives up is reported later by mhla_device_status.
 * B == 0 or H == 0 is a valid empty call that queues nothing. */
mhla_status_t mhla_forward(const mhla_tensor_t* q, const mhla_tensor_t* k,
                           const mhla_tensor_t* v, const float* W,
                           const mhla_shape3_t* grid, const mhla_shape3_t* block,
                           const mhla_phi_t* phi, const mhla_tensor_t* out,
                           void* workspace, size_t workspace_bytes, void* stream,
                           int32_t path);

/* Device workspace mhla_backward needs for this problem and path (bytes, a
 * multiple of 256).  q gives B, N, H, d and the dtype.  Host only. */
mhla_status_t mhla_backward_workspace_size(const mhla_tensor_t* q, const mhla_shape3_t* grid,
                                           const mhla_shape3_t* block, int32_t path, size_t* bytes);

/* Gradients of the MHLA forward for training: given dout = dL/d(out) of a
 * forward with the same q, k, v, W, grid, block and phi, writes dq, dk, dv and
 * dW = dL/dW.  The pages print no backward pass; they make the mixing
 * coefficients learnable ([P2] section 4 "Multi-Head Mixing": learned,
 * initialised from block distances; [P1] section 7: W is a 1x1 convolution's
 * weight), so these are the chain-rule derivatives of the three forward steps
 * taken in reverse:
 *   dnum_t = dout_t / den_t,   dden_t = -(dout_t . o_t) / den_t
 *   dq_t   = (S~_i dnum_t + dden_t z~_i) * [q_t > 0]
 *   dS~_i  = sum_{t in i} phi(q_t) dnum_t^T,  dz~_i = sum_{t in i} dden_t phi(q_t)
 *   dS_j   = sum_i W[i][j] dS~_i,             dz_j  = sum_i W[i][j] dz~_i
 *   dW[i][j] = sum_{b,h} <dS~_i, S_j> + dz~_i . z_j
 *   dv_s   = dS_j^T phi(k_s),  dk_s = (dS_j v_s + dz_j) * [k_s > 0]
 * phi'(x) is 1 for x > 0 and 0 otherwise in both phi modes.  The summaries and
 * the mixing are recomputed from k, v and W (nothing is kept from the forward).
 *   q, k, v, dout  device tensors [B, N, H, d], same shape and dtype.
 *   dq, dk, dv     device tensors, same shape and dtype, written in that dtype;
 *                  none may overlap another tensor argument, W or dW.
 *   W              device float32 M x M, as for mhla_forward.
 *   dW             device float32 M x M, overwritten with the sum over every
 *                  batch and head (one W is shared by all); must not overlap W.
 *   workspace      at least mhla_backward_workspace_size() bytes, 256-byte
 *                  aligned, or NULL with workspace_bytes == 0 (stream-ordered
 *                  cudaMallocAsync / cudaFreeAsync).
 *   path           AUTO takes TC whenever every operand qualifies, else SIMT.
 *                  TC: tensor cores, bf16 with float32 accumulation, d in
 *                  {32, 64}, the forward TC path's token geometry and TMA
 *                  friendly strides on q, k, v, dout, dq, dk, dv; SIMT: CUDA
 *                  cores, float32 arithmetic, any d <= 128 and block shape.
 *                  FUSED and TC_FUSED return MHLA_ERR_UNSUPPORTED.
 * With AUTO, mhla_backward_workspace_size returns enough for either path.
 * Asynchronous on stream; statuses as for mhla_forward.  B == 0 or H == 0
 * writes dW = 0 and nothing else. */
mhla_status_t mhla_backward(const mhla_tensor_t* q, const mhla_tensor_t* k,
                            const mhla_tensor_t* v, const float* W,
                            const mhla_shape3_t* grid, const mhla_shape3_t* block,
                            const mhla_phi_t* phi, const mhla_tensor_t* dout,
                            const mhla_tensor_t* dq, const mhla_tensor_t* dk,
                            const mhla_tensor_t* dv, float* dW,
                            void* workspace, size_t workspace_bytes, void* stream,
                            int32_t path);

/* Device workspace mhla_forward_causal needs (bytes, a multiple of 256).  Host
 * only; MHLA_ERR_SHAPE when the blocks are not contiguous token ranges. */
mhla_status_t mhla_causal_workspace_size(const mhla_tensor_t* q, const mhla_shape3_t* grid,
                                         const mhla_shape3_t* block, int32_t path, size_t* bytes);

/* Causal (chunkwise) MHLA for autoregressive models ([P2] App. B "Causal MHLA":
 * block-specific mixed summaries, reusing each block's mixture, causal at the
 * cost of chunkwise linear attention).  The page gives no formula; this is the
 * causal restriction of the two-stage form: token t of query block i sees
 * every past block j < i through W[i][j] and the tokens s <= t of its own
 * block through W[i][i]:
 *   o_t = phi(q_t)^T (S<_i + W[i][i] P_t) / (phi(q_t) . (z<_i + W[i][i] y_t) + eps)
 *   S<_i = sum_{j<i} W[i][j] S_j,  P_t = sum_{s in i, s <= t} phi(k_s) v_s^T,
 * z<_i and y_t likewise.  Entries W[i][j] with j > i are never read.
 *   Arguments as for mhla_forward.  The blocks must be contiguous ranges of
 *   raster-order tokens (a 1-D sequence grid (1, N) in blocks (1, w), or whole
 *   rows or frames), else MHLA_ERR_SHAPE.
 *   path: AUTO takes TC whenever the request qualifies, else SIMT.
 *     TC: tensor cores, bf16 with float32 accumulation, d in {32, 64},
 *     N a multiple of 128, blocks of 64 tokens or a multiple of 128, strides
 *     multiples of 8 elements; the sequence is cut into units of min(w, 128)
 *     tokens whose causal states come from one mixing GEMM with the unit-level
 *     matrix W'[u][u'] (W[b(u)][b(u')] for a past block, W[b(u)][b(u)] for an
 *     earlier unit of the same block, 0 otherwise), then every 128-token tile
 *     forms its causal scores and its state term in one accumulator.
 *     SIMT: CUDA cores, float32 arithmetic, any d <= 128, bf16 or float32.
 *     FUSED and TC_FUSED return MHLA_ERR_UNSUPPORTED.
 *   With AUTO, mhla_causal_workspace_size returns enough for either path. */
mhla_status_t mhla_forward_causal(const mhla_tensor_t* q, const mhla_tensor_t* k,
                                  const mhla_tensor_t* v, const float* W,
                                  const mhla_shape3_t* grid, const mhla_shape3_t* block,
                                  const mhla_phi_t* phi, const mhla_tensor_t* out,
                                  void* workspace, size_t workspace_bytes, void* stream,
                                  int32_t path);

/* Device workspace mhla_backward_causal needs (bytes, a multiple of 256).  Host
 * only; MHLA_ERR_SHAPE when the blocks are not contiguous token ranges. */
mhla_status_t mhla_backward_causal_workspace_size(const mhla_tensor_t* q, const mhla_shape3_t* grid,
                                                  const mhla_shape3_t* block, int32_t path, size_t* bytes);

/* Gradients of mhla_forward_causal for chunkwise training ([P2] App. B "Causal
 * MHLA" trains autoregressive models with the causal form; section 4 "Multi-Head
 * Mixing" makes W learnable).  The pages print no backward pass; these are the
 * chain-rule derivatives of the causal form above, for token t of query block
 * i with C_t = S<_i + W[i][i] P_t and c_t = z<_i + W[i][i] y_t:
 *   dnum_t = dout_t / den_t,   dden_t = -(dout_t . o_t) / den_t
 *   dq_t   = (C_t dnum_t + dden_t c_t) * [q_t > 0]
 *   dS<_i  = sum_{t in i} phi(q_t) dnum_t^T,  dz<_i = sum_{t in i} dden_t phi(q_t)
 *   dW[i][i] = sum_{t in i} sum_{s in i, s <= t} (phi(q_t) . phi(k_s)) (v_s . dnum_t + dden_t)
 *   dW[i][j] = <dS<_i, S_j> + dz<_i . z_j for j < i, 0 for j > i (summed over b, h)
 *   dS_j   = sum_{i > j} W[i][j] dS<_i,       dz_j likewise
 *   dv_s   = dS_j^T phi(k_s) + W[j][j] sum_{t in j, t >= s} (phi(q_t) . phi(k_s)) dnum_t
 *   dk_s   = (dS_j v_s + dz_j + W[j][j] sum_{t in j, t >= s} phi(q_t) (dnum_t . v_s + dden_t))
 *            * [k_s > 0]
 * The forward's states are recomputed from k, v and W.
 *   Arguments, aliasing rules and statuses as for mhla_backward; the blocks must
 *   be contiguous ranges of raster-order tokens as for mhla_forward_causal, else
 *   MHLA_ERR_SHAPE.  Entries W[i][j] with j > i are never read.
 *   path: the per-token steps run on CUDA cores (float32 arithmetic, any
 *   d <= 128, bf16 or float32).  SIMT: the recomputed summaries S_j and mixed
 *   past S<_i too.  TC: those two steps on the tensor-core causal forward's
 *   summary and mixing kernels (bf16 MMA operands, float32 accumulation), when
 *   that path takes the problem and every block is one of its units (w = 64 or
 *   128 tokens), else MHLA_ERR_UNSUPPORTED.  AUTO: TC when it applies, else
 *   SIMT.  FUSED and TC_FUSED return MHLA_ERR_UNSUPPORTED.
 *   workspace: at least mhla_backward_causal_workspace_size() bytes for the same
 *   path (about 3 B H M d (d + 1) + B H N (d + 1) floats, plus the tensor-core
 *   summaries and states for TC), 256-byte aligned, or NULL with
 *   workspace_bytes == 0 (stream-ordered allocation).
 * B == 0 or H == 0 writes dW = 0 and nothing else. */
mhla_status_t mhla_backward_causal(const mhla_tensor_t* q, const mhla_tensor_t* k,
                                   const mhla_tensor_t* v, const float* W,
                                   const mhla_shape3_t* grid, const mhla_shape3_t* block,
                                   const mhla_phi_t* phi, const mhla_tensor_t* dout,
                                   const mhla_tensor_t* dq, const mhla_tensor_t* dk,
                                   const mhla_tensor_t* dv, float* dW,
                                   void* workspace, size_t workspace_bytes, void* stream,
                                   int32_t path);

/* mhla_forward for callers that must not allocate device memory -- the paper
 * has no counterpart to this; it is a property of the library, not the method.
 * Who needs it: code that runs the forward where device allocation is not
 * allowed, such as a plugin executing inside an inference engine's enqueue
 * step (the engine owns all device memory) or a serving loop that plans its
 * memory once at start-up (cudaFree synchronises the device; an allocation can
 * fail under fragmentation).  The caller still passes q, k, v, W and out; the
 * scratch comes from one array of MHLA_NOALLOC_SCRATCH_BYTES (64 MiB) compiled
 * into the library, which every GPU that loads the library holds until the
 * process exits.  After its set-up call (below) the call allocates nothing:
 * no cudaMalloc, cudaMallocAsync, cudaFree or allocating library routine.
 *   Arguments as for mhla_forward, without workspace and workspace_bytes.
 *   Returns MHLA_ERR_WORKSPACE, before touching the GPU, when the problem needs
 *   more scratch than the array holds (mhla_workspace_size says how much it
 *   needs); other statuses as for mhla_forward.
 *   Set-up: the first call in a CUDA context (per device, and again after a
 *   device reset, which creates a new context) looks up the array's device
 *   address there (cudaGetSymbolAddress, with the caller's device current).
 *   That first lookup loads the library's device code into the context, and
 *   the driver allocates the array's 64 MiB at that moment -- so the first
 *   call can fail with MHLA_ERR_CUDA under memory pressure, and it is the one
 *   call that does allocate, implicitly.  Make it at start-up, before any
 *   stream capture: a call with B == 0 does the set-up, queues nothing and
 *   returns MHLA_OK.  Every later call in that context allocates nothing.
 *   Every call on a device shares the one array and leaves its contents
 *   behind; no part of it needs to start at zero: a call writes every scratch
 *   byte whose value reaches its results before reading it (padding it reads
 *   unwritten only feeds outputs it discards).  Calls whose work overlaps on
 *   the GPU (two streams, or two threads) race on the array: order them on one
 *   stream. */
#define MHLA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
mhla_status_t mhla_forward_noalloc(const mhla_tensor_t* q, const mhla_tensor_t* k,
                                   const mhla_tensor_t* v, const float* W,
                                   const mhla_shape3_t* grid, const mhla_shape3_t* block,
                                   const mhla_phi_t* phi, const mhla_tensor_t* out,
                                   void* stream, int32_t path);

/* ---------------------------------------------------------------------------
 * The module around the core ([P1] section 7, class MHLA: norm, to_qkv, lepe,
 * to_out and forward), for a [B, N, C] bf16 token array x with C = heads * d:
 *
 *   xn      = LayerNorm(x)                        (mhla_layer_norm)
 *   q, k, v = split(xn W_qkv^T + b_qkv, 3)        (mhla_linear; q, k, v are read
 *             in place as [B, N, heads, d] views of its [B, N, 3C] result)
 *   o       = MHLA(q, k, v)                       (mhla_forward, path AUTO)
 *   o      += lepe(v)                             (mhla_lepe_add)
 *   y       = o W_out^T + b_out                   (mhla_linear)
 *
 * Every step runs in this library's own kernels (the projections on the
 * tensor cores, tcgen05).  Dropout is the identity (inference); q_norm /
 * k_norm are identities (the listing's default).
 * ------------------------------------------------------------------------ */

/* A linear layer y = x w^T + bias in bf16 with float32 accumulation, rounded
 * once to bf16: the module's to_qkv and to_out ([P1] section 7, nn.Linear).
 *   x      device [rows][k] bf16, row-major;  w  device [n_out][k] bf16
 *          (nn.Linear's [out][in] layout);  bias  device [n_out] bf16 or NULL;
 *   y      device [rows][n_out] bf16; must not overlap x, w or bias.
 * k and n_out multiples of 8, every pointer 16-byte aligned, rows < 2^31
 * (MHLA_ERR_UNSUPPORTED otherwise); rows == 0 queues nothing.  Asynchronous on
 * stream; tensor-core GEMM in 128 x 256 output tiles. */
mhla_status_t mhla_linear(const void* x, const void* w, const void* bias, void* y, int64_t rows, int64_t k,
                          int64_t n_out, void* stream);

/* LayerNorm over the last axis of a row-major [rows, C] bf16 device array:
 * y = (x - mean) / sqrt(var + eps) * weight + bias with the biased variance and
 * float32 statistics, rounded to bf16 ([P1] section 7, MHLA.norm, an
 * nn.LayerNorm(dim)).  C % 8 == 0 and C <= 2048; x, y, weight and bias (float32
 * [C]) 16-byte aligned device memory; y may equal x, other overlaps are
 * invalid.  Asynchronous on stream. */
mhla_status_t mhla_layer_norm(const void* x, void* y, int64_t rows, int64_t C, const float* weight,
                              const float* bias, float eps, void* stream);

/* out += lepe(v): the locally-enhanced positional term of [P1] section 7
 * (MHLA.lepe, a depthwise nn.Conv2d with 5 x 5 kernels and padding 2, and
 * "out = out + lepe" in MHLA.forward):
 *   out[b, (y, x), c] += bias[c] + sum_{i, j < 5} weight[c][i][j] * v[b, (y + i - 2, x + j - 2), c]
 * with zero outside the frame, over the (Y, X) axes of the grid (each frame of
 * a 3-D grid on its own).  Channel c is h * d + j of a [B, N, H, d] view.
 *   v, out   bf16 device views of the same shape; d % 8 == 0, every stride a
 *            multiple of 8 elements, 16-byte aligned bases; heads adjacent
 *            (stride_h == d), as in a projection's [B, N, 3C] rows or a
 *            contiguous [B, N, H, d] tensor; out must not overlap v.
 *   weight   device float32 [H * d][5][5];  bias  device float32 [H * d].
 * Rounds o + (bias + conv) once to bf16.  Asynchronous on stream. */
mhla_status_t mhla_lepe_add(const mhla_tensor_t* v, const mhla_tensor_t* out, const mhla_shape3_t* grid,
                            const float* weight, const float* bias, void* stream);

/* Parameters of the module; every pointer is device memory the caller owns. */
typedef struct mhla_module_params {
    const float* ln_weight;    /* [C] float32 */
    const float* ln_bias;      /* [C] float32 */
    const void* qkv_weight;    /* [3C][C] bf16, nn.Linear layout [out][in]; rows q, then k, then v,
                                  each (head, d) with the head slower */
    const void* qkv_bias;      /* [3C] bf16 or NULL */
    const float* lepe_weight;  /* [C][5][5] float32, or NULL for no positional term */
    const float* lepe_bias;    /* [C] float32; required with lepe_weight */
    const void* out_weight;    /* [C][C] bf16, [out][in] */
    const void* out_bias;      /* [C] bf16 or NULL */
    float ln_eps;              /* LayerNorm eps (1e-5 in the listing) */
    int32_t heads;             /* C = heads * d */
} mhla_module_params_t;

/* Device workspace mhla_module_forward needs (bytes): the normalised input and
 * the core's output (one buffer), the [B, N, 3C] projection and the core's own
 * workspace.  Host only. */
mhla_status_t mhla_module_workspace_size(int64_t B, int64_t N, int64_t C, int32_t heads,
                                         const mhla_shape3_t* grid, const mhla_shape3_t* block,
                                         size_t* bytes);

/* The module forward on x [B, N, C] (bf16, row-major, 16-byte aligned; tokens in
 * raster order over grid) into y of the same layout (y may equal x).  W, grid,
 * block and phi are those of mhla_forward (the listing uses
 * MHLA_PHI_RELU_EPS).  C % 8 == 0, C <= 2048, d = C / heads with d % 8 == 0,
 * B * N < 2^31; the projection biases, when given, 16-byte aligned.
 * workspace as for mhla_forward (NULL with workspace_bytes == 0: stream-ordered
 * allocation).  Asynchronous on stream.  The argument checks of every step (the
 * core's and the positional term's included) run before the first launch; only
 * a failed launch can return after earlier steps were queued. */
mhla_status_t mhla_module_forward(const void* x, void* y, int64_t B, int64_t N, int64_t C,
                                  const mhla_module_params_t* params, const float* W,
                                  const mhla_shape3_t* grid, const mhla_shape3_t* block,
                                  const mhla_phi_t* phi, void* workspace, size_t workspace_bytes,
                                  void* stream);

/* Reads and clears the device error words the tensor-core and fused kernels
 * set when one of their bounded waits gives up (bit 0: pipeline wait timeout;
 * bit 1: a copy or MMA still in flight when the kernel gave up did not finish
 * within its drain limit).  Synchronises stream.  *flags receives the word; returns MHLA_ERR_TIMEOUT when it was
 * non-zero, MHLA_ERR_CUDA when the copy failed. */
mhla_status_t mhla_device_status(void* stream, uint32_t* flags);

/* Diagnostic hook for testing the timeout path of the device-side waits (no
 * counterpart in the method).  With warp >= 0, every bounded mbarrier wait made
 * by warp index `warp` of any kernel of this library that does not find its
 * phase complete at the first poll behaves as if the completion it waits for
 * never came: it gives up after limit_ns nanoseconds
 * (1 us .. 1 s), the kernel's other roles stop, copies already in flight are
 * drained, tensor memory is released, and the next mhla_device_status reports
 * MHLA_ERR_TIMEOUT (bit 0).  The outputs of calls made meanwhile are undefined.
 * warp == -1 turns it off (the default).  Synchronous; call it only while no
 * work of this library is queued or running.  Returns MHLA_ERR_INVALID_ARG for
 * a warp outside -1 .. 31 or a limit outside the range, MHLA_ERR_CUDA when a
 * copy to the device failed. */
mhla_status_t mhla_debug_stall_waits(int32_t warp, uint64_t limit_ns);

/* Per-kernel timing.  Between mhla_profile_begin and mhla_profile_end every
 * kernel the library launches is bracketed by a pair of CUDA events recorded on
 * its launch stream.  mhla_profile_end waits for those events, writes one entry
 * per kernel name (launch count and summed duration in milliseconds) into out
 * (room for capacity entries; *count receives the number of names) and stops
 * collecting.  Host only apart from the event records; thread safe. */
typedef struct mhla_kernel_time {
    char name[32];
    int32_t launches;
    float total_ms;
} mhla_kernel_time_t;

mhla_status_t mhla_profile_begin(void);
mhla_status_t mhla_profile_end(mhla_kernel_time_t* out, int32_t capacity, int32_t* count);

/* Static description of a status code (never NULL). */
const char* mhla_status_string(int32_t status);

/* Library version, e.g. "mhla-gb300 0.1.0 sm_103a". */
const char* mhla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MHLA_H */
