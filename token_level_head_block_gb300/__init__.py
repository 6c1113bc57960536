"""MHLA forward pass (token-level multi-head linear attention) on GB300, sm_103a.

Thin Python binding of the C ABI in ``include/mhla.h`` (``lib/libmhla.so``):
argument marshalling only.  Every step of the forward pass runs in the
library's CUDA kernels; PyTorch supplies device memory and streams.  There is
no CPU fallback: calls raise when the library is missing or a call fails.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

__all__ = [
    "MhlaError", "lib", "library_path", "num_blocks", "init_mixing", "workspace_size",
    "select_path", "forward", "forward_causal", "causal_workspace_size", "backward", "backward_workspace_size",
    "backward_causal", "backward_causal_workspace_size",
    "device_status", "profile_begin", "layer_norm", "lepe_add", "module_forward",
    "module_workspace_size",
    "profile_end", "tensor_desc", "shape3",
    "PATHS", "TRANSFORMS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "lib", "libmhla.so")

PATHS = {"auto": 0, "simt": 1, "tc": 2, "fused": 3, "tc_fused": 4}
TRANSFORMS = {"linear": 0, "cos": 1, "exp": 2, "gaussian": 3, "local": 4}
PHIS = {"relu": 0, "relu_eps": 1}
DTYPES = {"bf16": 0, "f32": 1}

STATUS = {
    0: "ok", 1: "invalid argument", 2: "shape mismatch", 3: "unsupported by the selected path",
    4: "CUDA error", 5: "device wait timed out", 6: "workspace missing, too small or misaligned",
}


class MhlaError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = int(status)
        super().__init__(f"{what}: {STATUS.get(self.status, 'unknown status')} ({self.status})")


class Shape3(ctypes.Structure):
    _fields_ = [("ndim", ctypes.c_int32), ("pad_", ctypes.c_int32), ("extent", ctypes.c_int64 * 3)]


class Phi(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("eps", ctypes.c_float)]


class KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int32), ("total_ms", ctypes.c_float)]


class Tensor(ctypes.Structure):
    _fields_ = [
        ("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("pad_", ctypes.c_int32),
        ("B", ctypes.c_int64), ("N", ctypes.c_int64), ("H", ctypes.c_int64), ("d", ctypes.c_int64),
        ("stride_b", ctypes.c_int64), ("stride_n", ctypes.c_int64), ("stride_h", ctypes.c_int64),
    ]


class ModuleParams(ctypes.Structure):
    """mhla_module_params_t: device pointers of the module's parameters."""
    _fields_ = [
        ("ln_weight", ctypes.c_void_p), ("ln_bias", ctypes.c_void_p),
        ("qkv_weight", ctypes.c_void_p), ("qkv_bias", ctypes.c_void_p),
        ("lepe_weight", ctypes.c_void_p), ("lepe_bias", ctypes.c_void_p),
        ("out_weight", ctypes.c_void_p), ("out_bias", ctypes.c_void_p),
        ("ln_eps", ctypes.c_float), ("heads", ctypes.c_int32),
    ]


_lib = None


def library_path():
    return _LIB_PATH


def lib():
    """The loaded libmhla (raises when it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise MhlaError(4, f"{_LIB_PATH} is missing; build it with "
                           "`python -m token_level_head_block_gb300.build`")
    L = ctypes.CDLL(_LIB_PATH)
    P = ctypes.POINTER
    L.mhla_num_blocks.argtypes = [P(Shape3), P(Shape3)]
    L.mhla_num_blocks.restype = ctypes.c_int64
    L.mhla_init_mixing.argtypes = [P(Shape3), P(Shape3), ctypes.c_int32, ctypes.c_double, ctypes.c_double,
                                   P(ctypes.c_float), ctypes.c_int64]
    L.mhla_init_mixing.restype = ctypes.c_int
    L.mhla_workspace_size.argtypes = [P(Tensor), P(Shape3), P(Shape3), ctypes.c_int32, P(ctypes.c_size_t)]
    L.mhla_workspace_size.restype = ctypes.c_int
    L.mhla_select_path.argtypes = [P(Tensor), P(Tensor), P(Tensor), P(Tensor), P(Shape3), P(Shape3)]
    L.mhla_select_path.restype = ctypes.c_int32
    L.mhla_forward.argtypes = [P(Tensor), P(Tensor), P(Tensor), ctypes.c_void_p, P(Shape3), P(Shape3), P(Phi),
                               P(Tensor), ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int32]
    L.mhla_forward.restype = ctypes.c_int
    L.mhla_causal_workspace_size.argtypes = [P(Tensor), P(Shape3), P(Shape3), ctypes.c_int32, P(ctypes.c_size_t)]
    L.mhla_causal_workspace_size.restype = ctypes.c_int
    L.mhla_forward_causal.argtypes = [P(Tensor), P(Tensor), P(Tensor), ctypes.c_void_p, P(Shape3), P(Shape3),
                                      P(Phi), P(Tensor), ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                      ctypes.c_int32]
    L.mhla_forward_causal.restype = ctypes.c_int
    L.mhla_backward_workspace_size.argtypes = [P(Tensor), P(Shape3), P(Shape3), ctypes.c_int32,
                                               P(ctypes.c_size_t)]
    L.mhla_backward_workspace_size.restype = ctypes.c_int
    L.mhla_backward.argtypes = [P(Tensor), P(Tensor), P(Tensor), ctypes.c_void_p, P(Shape3), P(Shape3), P(Phi),
                                P(Tensor), P(Tensor), P(Tensor), P(Tensor), ctypes.c_void_p, ctypes.c_void_p,
                                ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int32]
    L.mhla_backward.restype = ctypes.c_int
    L.mhla_backward_causal_workspace_size.argtypes = [P(Tensor), P(Shape3), P(Shape3), ctypes.c_int32,
                                                      P(ctypes.c_size_t)]
    L.mhla_backward_causal_workspace_size.restype = ctypes.c_int
    L.mhla_backward_causal.argtypes = L.mhla_backward.argtypes
    L.mhla_backward_causal.restype = ctypes.c_int
    L.mhla_layer_norm.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                  ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p]
    L.mhla_layer_norm.restype = ctypes.c_int
    L.mhla_lepe_add.argtypes = [P(Tensor), P(Tensor), P(Shape3), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    L.mhla_lepe_add.restype = ctypes.c_int
    L.mhla_linear.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                              ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
    L.mhla_linear.restype = ctypes.c_int
    L.mhla_module_workspace_size.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                             P(Shape3), P(Shape3), P(ctypes.c_size_t)]
    L.mhla_module_workspace_size.restype = ctypes.c_int
    L.mhla_module_forward.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                      ctypes.c_int64, P(ModuleParams), ctypes.c_void_p, P(Shape3), P(Shape3),
                                      P(Phi), ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    L.mhla_module_forward.restype = ctypes.c_int
    L.mhla_debug_stall_waits.argtypes = [ctypes.c_int32, ctypes.c_uint64]
    L.mhla_debug_stall_waits.restype = ctypes.c_int
    L.mhla_device_status.argtypes = [ctypes.c_void_p, P(ctypes.c_uint32)]
    L.mhla_device_status.restype = ctypes.c_int
    L.mhla_status_string.argtypes = [ctypes.c_int32]
    L.mhla_status_string.restype = ctypes.c_char_p
    L.mhla_profile_begin.argtypes = []
    L.mhla_profile_begin.restype = ctypes.c_int
    L.mhla_profile_end.argtypes = [P(KernelTime), ctypes.c_int32, P(ctypes.c_int32)]
    L.mhla_profile_end.restype = ctypes.c_int
    L.mhla_version.argtypes = []
    L.mhla_version.restype = ctypes.c_char_p
    _lib = L
    return L


def shape3(ext):
    ext = tuple(int(e) for e in ext)
    s = Shape3()
    s.ndim = len(ext)
    for a, e in enumerate(ext[:3]):
        s.extent[a] = e
    return s


def tensor_desc(ptr, dtype, shape, strides):
    """mhla_tensor_t for a [B, N, H, d] operand given its address and element strides."""
    t = Tensor()
    t.data = ctypes.c_void_p(int(ptr)) if ptr else None
    t.dtype = DTYPES[dtype] if isinstance(dtype, str) else int(dtype)
    t.B, t.N, t.H, t.d = (int(x) for x in shape)
    t.stride_b, t.stride_n, t.stride_h = (int(x) for x in strides[:3])
    return t


def _desc(x):
    import torch
    if x.dim() != 4:
        raise ValueError("expected a [B, N, H, d] tensor")
    if x.shape[3] > 1 and x.stride(3) != 1:
        raise ValueError("the d dimension must be contiguous")
    if x.dtype == torch.bfloat16:
        dt = "bf16"
    elif x.dtype == torch.float32:
        dt = "f32"
    else:
        raise ValueError(f"unsupported dtype {x.dtype}")
    return tensor_desc(x.data_ptr(), dt, tuple(x.shape), (x.stride(0), x.stride(1), x.stride(2)))


def _check(status, what):
    if status != 0:
        raise MhlaError(status, what)


def num_blocks(grid, block):
    m = lib().mhla_num_blocks(ctypes.byref(shape3(grid)), ctypes.byref(shape3(block)))
    if m < 0:
        raise MhlaError(-m, "mhla_num_blocks")
    return int(m)


def init_mixing(grid, block, transform="linear", local_thres=1.5, exp_sigma=3.0):
    """M x M float32 mixing matrix from block-centre distances (host computation)."""
    M = num_blocks(grid, block)
    W = np.empty((M, M), dtype=np.float32)
    st = lib().mhla_init_mixing(ctypes.byref(shape3(grid)), ctypes.byref(shape3(block)),
                                TRANSFORMS[transform], float(local_thres), float(exp_sigma),
                                W.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), W.size)
    _check(st, "mhla_init_mixing")
    return W


def workspace_size(q, grid, block, path="auto"):
    n = ctypes.c_size_t(0)
    _check(lib().mhla_workspace_size(ctypes.byref(_desc(q) if not isinstance(q, Tensor) else q),
                                     ctypes.byref(shape3(grid)), ctypes.byref(shape3(block)), PATHS[path],
                                     ctypes.byref(n)), "mhla_workspace_size")
    return int(n.value)


def select_path(q, k, v, out, grid, block):
    r = lib().mhla_select_path(ctypes.byref(_desc(q)), ctypes.byref(_desc(k)), ctypes.byref(_desc(v)),
                               ctypes.byref(_desc(out)), ctypes.byref(shape3(grid)), ctypes.byref(shape3(block)))
    if r < 0:
        raise MhlaError(-r, "mhla_select_path")
    return {1: "simt", 2: "tc", 3: "fused"}[r]


def forward(q, k, v, W, grid, block, phi="relu", eps=1e-6, out=None, workspace=None, stream=None,
            path="auto"):
    """MHLA forward of device tensors q, k, v [B, N, H, d]; returns ``out``.

    W is a float32 CUDA tensor (M x M, contiguous), shared by all batches and
    heads.  ``workspace`` is an optional uint8 CUDA tensor of at least
    ``workspace_size`` bytes; without it the call takes stream-ordered memory.
    Asynchronous on ``stream`` (default: torch's current stream).
    """
    import torch
    if out is None:
        out = torch.empty_like(q)
    if not W.is_contiguous() or W.dtype != torch.float32:
        raise ValueError("W must be a contiguous float32 tensor")
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sptr = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(), workspace.numel() *
                                                            workspace.element_size())
    st = lib().mhla_forward(ctypes.byref(_desc(q)), ctypes.byref(_desc(k)), ctypes.byref(_desc(v)),
                            ctypes.c_void_p(W.data_ptr()), ctypes.byref(shape3(grid)),
                            ctypes.byref(shape3(block)), ctypes.byref(Phi(PHIS[phi], float(eps))),
                            ctypes.byref(_desc(out)), ctypes.c_void_p(ws_ptr) if ws_ptr else None,
                            ws_bytes, ctypes.c_void_p(sptr) if sptr else None, PATHS[path])
    _check(st, "mhla_forward")
    return out


def causal_workspace_size(q, grid, block, path="auto"):
    n = ctypes.c_size_t(0)
    _check(lib().mhla_causal_workspace_size(ctypes.byref(_desc(q) if not isinstance(q, Tensor) else q),
                                            ctypes.byref(shape3(grid)), ctypes.byref(shape3(block)), PATHS[path],
                                            ctypes.byref(n)), "mhla_causal_workspace_size")
    return int(n.value)


def forward_causal(q, k, v, W, grid, block, phi="relu", eps=1e-6, out=None, workspace=None, stream=None,
                   path="auto"):
    """Causal (chunkwise) MHLA of device tensors [B, N, H, d]; blocks must be
    contiguous token ranges (e.g. grid (1, N), block (1, w)).  Returns ``out``."""
    import torch
    if out is None:
        out = torch.empty_like(q)
    if not W.is_contiguous() or W.dtype != torch.float32:
        raise ValueError("W must be a contiguous float32 tensor")
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sptr = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(), workspace.numel() *
                                                            workspace.element_size())
    st = lib().mhla_forward_causal(ctypes.byref(_desc(q)), ctypes.byref(_desc(k)), ctypes.byref(_desc(v)),
                                   ctypes.c_void_p(W.data_ptr()), ctypes.byref(shape3(grid)),
                                   ctypes.byref(shape3(block)), ctypes.byref(Phi(PHIS[phi], float(eps))),
                                   ctypes.byref(_desc(out)), ctypes.c_void_p(ws_ptr) if ws_ptr else None,
                                   ws_bytes, ctypes.c_void_p(sptr) if sptr else None, PATHS[path])
    _check(st, "mhla_forward_causal")
    return out


def backward_workspace_size(q, grid, block, path="auto"):
    n = ctypes.c_size_t(0)
    _check(lib().mhla_backward_workspace_size(ctypes.byref(_desc(q) if not isinstance(q, Tensor) else q),
                                              ctypes.byref(shape3(grid)), ctypes.byref(shape3(block)),
                                              PATHS[path], ctypes.byref(n)), "mhla_backward_workspace_size")
    return int(n.value)


def backward(q, k, v, W, dout, grid, block, phi="relu", eps=1e-6, dq=None, dk=None, dv=None, dW=None,
             workspace=None, stream=None, path="auto"):
    """Gradients (dq, dk, dv, dW) of the MHLA forward given dout = dL/d(out).

    Device tensors [B, N, H, d] like ``forward``; dW is a float32 M x M CUDA
    tensor (allocated when not given) holding the sum over batches and heads.
    Asynchronous on ``stream`` (default: torch's current stream).
    """
    import torch
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if dW is None:
        dW = torch.empty_like(W)
    for name, x in (("W", W), ("dW", dW)):
        if not x.is_contiguous() or x.dtype != torch.float32:
            raise ValueError(f"{name} must be a contiguous float32 tensor")
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sptr = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(), workspace.numel() *
                                                            workspace.element_size())
    st = lib().mhla_backward(ctypes.byref(_desc(q)), ctypes.byref(_desc(k)), ctypes.byref(_desc(v)),
                             ctypes.c_void_p(W.data_ptr()), ctypes.byref(shape3(grid)),
                             ctypes.byref(shape3(block)), ctypes.byref(Phi(PHIS[phi], float(eps))),
                             ctypes.byref(_desc(dout)), ctypes.byref(_desc(dq)), ctypes.byref(_desc(dk)),
                             ctypes.byref(_desc(dv)), ctypes.c_void_p(dW.data_ptr()),
                             ctypes.c_void_p(ws_ptr) if ws_ptr else None, ws_bytes,
                             ctypes.c_void_p(sptr) if sptr else None, PATHS[path])
    _check(st, "mhla_backward")
    return dq, dk, dv, dW


def backward_causal_workspace_size(q, grid, block, path="auto"):
    n = ctypes.c_size_t(0)
    _check(lib().mhla_backward_causal_workspace_size(ctypes.byref(_desc(q) if not isinstance(q, Tensor) else q),
                                                     ctypes.byref(shape3(grid)), ctypes.byref(shape3(block)),
                                                     PATHS[path], ctypes.byref(n)),
           "mhla_backward_causal_workspace_size")
    return int(n.value)


def backward_causal(q, k, v, W, dout, grid, block, phi="relu", eps=1e-6, dq=None, dk=None, dv=None, dW=None,
                    workspace=None, stream=None, path="auto"):
    """Gradients (dq, dk, dv, dW) of ``forward_causal`` given dout = dL/d(out).

    Arguments as for ``backward``; the blocks must be contiguous token ranges
    as for ``forward_causal``.  dW is zero above the diagonal."""
    import torch
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if dW is None:
        dW = torch.empty_like(W)
    for name, x in (("W", W), ("dW", dW)):
        if not x.is_contiguous() or x.dtype != torch.float32:
            raise ValueError(f"{name} must be a contiguous float32 tensor")
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sptr = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(), workspace.numel() *
                                                            workspace.element_size())
    st = lib().mhla_backward_causal(ctypes.byref(_desc(q)), ctypes.byref(_desc(k)), ctypes.byref(_desc(v)),
                                    ctypes.c_void_p(W.data_ptr()), ctypes.byref(shape3(grid)),
                                    ctypes.byref(shape3(block)), ctypes.byref(Phi(PHIS[phi], float(eps))),
                                    ctypes.byref(_desc(dout)), ctypes.byref(_desc(dq)), ctypes.byref(_desc(dk)),
                                    ctypes.byref(_desc(dv)), ctypes.c_void_p(dW.data_ptr()),
                                    ctypes.c_void_p(ws_ptr) if ws_ptr else None, ws_bytes,
                                    ctypes.c_void_p(sptr) if sptr else None, PATHS[path])
    _check(st, "mhla_backward_causal")
    return dq, dk, dv, dW


def _stream_ptr(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    sptr = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    return ctypes.c_void_p(sptr) if sptr else None


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def layer_norm(x, weight, bias, eps=1e-5, out=None, stream=None):
    """LayerNorm over the last axis of a contiguous bf16 CUDA tensor (float32
    weight and bias of that size); returns ``out`` (may be ``x``)."""
    import torch
    out = torch.empty_like(x) if out is None else out
    C = x.shape[-1]
    st = lib().mhla_layer_norm(_ptr(x), _ptr(out), x.numel() // C, C, _ptr(weight), _ptr(bias), float(eps),
                               _stream_ptr(stream, x.device))
    _check(st, "mhla_layer_norm")
    return out


def linear(x, w, bias=None, out=None, stream=None):
    """y = x w^T (+ bias) for a contiguous bf16 CUDA tensor x [..., k] and an
    nn.Linear-layout weight w [n_out, k] (bias [n_out] or None); returns ``out``."""
    import torch
    k = x.shape[-1]
    n_out = w.shape[0]
    rows = x.numel() // k if k else 0
    if out is None:
        out = torch.empty(*x.shape[:-1], n_out, dtype=x.dtype, device=x.device)
    st = lib().mhla_linear(_ptr(x), _ptr(w), _ptr(bias), _ptr(out), rows, k, n_out, _stream_ptr(stream, x.device))
    _check(st, "mhla_linear")
    return out


def lepe_add(v, out, grid, weight, bias, stream=None):
    """out += 5 x 5 depthwise convolution of v (+ bias) over the token image, for
    bf16 [B, N, H, d] CUDA views; weight float32 [H * d, 5, 5], bias [H * d]."""
    st = lib().mhla_lepe_add(ctypes.byref(_desc(v)), ctypes.byref(_desc(out)), ctypes.byref(shape3(grid)),
                             _ptr(weight), _ptr(bias), _stream_ptr(stream, v.device))
    _check(st, "mhla_lepe_add")
    return out


def module_workspace_size(B, N, C, heads, grid, block):
    n = ctypes.c_size_t(0)
    _check(lib().mhla_module_workspace_size(B, N, C, heads, ctypes.byref(shape3(grid)), ctypes.byref(shape3(block)),
                                            ctypes.byref(n)), "mhla_module_workspace_size")
    return int(n.value)


def module_forward(x, params, W, grid, block, heads, phi="relu_eps", eps=1e-6, ln_eps=1e-5, out=None,
                   workspace=None, stream=None):
    """The MHLA module (LayerNorm, qkv projection, MHLA, 5 x 5 positional term,
    output projection) on a contiguous bf16 CUDA tensor x [B, N, C].

    ``params``: CUDA tensors ln_weight, ln_bias (float32 [C]); qkv_weight (bf16
    [3C, C]) and optional qkv_bias (bf16 [3C]); optional lepe_weight (float32
    [C, 5, 5]) with lepe_bias (float32 [C]); out_weight (bf16 [C, C]) and
    optional out_bias (bf16 [C]).  Returns ``out`` ([B, N, C], bf16).
    """
    import torch
    B, N, C = x.shape
    out = torch.empty_like(x) if out is None else out
    p = ModuleParams(_ptr(params["ln_weight"]), _ptr(params["ln_bias"]), _ptr(params["qkv_weight"]),
                     _ptr(params.get("qkv_bias")), _ptr(params.get("lepe_weight")), _ptr(params.get("lepe_bias")),
                     _ptr(params["out_weight"]), _ptr(params.get("out_bias")), float(ln_eps), int(heads))
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(), workspace.numel() *
                                                            workspace.element_size())
    st = lib().mhla_module_forward(_ptr(x), _ptr(out), B, N, C, ctypes.byref(p), _ptr(W),
                                   ctypes.byref(shape3(grid)), ctypes.byref(shape3(block)),
                                   ctypes.byref(Phi(PHIS[phi], float(eps))),
                                   ctypes.c_void_p(ws_ptr) if ws_ptr else None, ws_bytes,
                                   _stream_ptr(stream, x.device))
    _check(st, "mhla_module_forward")
    return out


def profile_begin():
    """Start bracketing every kernel launch with CUDA events on its stream."""
    _check(lib().mhla_profile_begin(), "mhla_profile_begin")


def profile_end():
    """Stop collecting; {kernel name: (launches, total milliseconds)}."""
    buf = (KernelTime * 32)()
    n = ctypes.c_int32(0)
    _check(lib().mhla_profile_end(buf, 32, ctypes.byref(n)), "mhla_profile_end")
    return {buf[i].name.decode(): (int(buf[i].launches), float(buf[i].total_ms)) for i in range(min(n.value, 32))}


def debug_stall_waits(warp, limit_ns=1_000_000):
    """Diagnostic hook of the timeout path: warp >= 0 makes every bounded wait
    of that warp index give up after limit_ns (the kernels then stop and report
    MHLA_ERR_TIMEOUT through device_status); warp = -1 turns it off."""
    _check(lib().mhla_debug_stall_waits(int(warp), int(limit_ns)), "mhla_debug_stall_waits")


def device_status(stream=None):
    """Reads and clears the device error word; raises MhlaError on a timeout flag."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    flags = ctypes.c_uint32(0)
    st = lib().mhla_device_status(ctypes.c_void_p(sptr) if sptr else None, ctypes.byref(flags))
    _check(st, f"mhla_device_status (flags={flags.value:#x})")
    return int(flags.value)
