"""ctypes binding of liblisa.so (C ABI in include/lisa.h).

Argument marshalling only: torch supplies device memory and the current CUDA
stream, every step of the layer runs in the library's kernels.  There is no
CPU path: a missing library, a CPU tensor or a non-zero status raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liblisa.so")

LISA_OK = 0
LISA_ERR_INVALID_ARG = 1
LISA_ERR_UNSUPPORTED = 2
LISA_ERR_WORKSPACE = 3
LISA_ERR_CUDA = 4
LISA_ERR_TIMEOUT = 5

LISA_F32 = 0
LISA_BF16 = 1

LISA_W_GEOMETRIC = 0
LISA_W_FIXED = 1
LISA_W_MLP = 2

LISA_MAX_T = 16
LISA_MAX_T_MLP = 8
LISA_MAX_HIDDEN = 64

EXPORTED = ("lisa_workspace_bytes", "lisa_forward", "lisa_forward_host", "lisa_num_stages",
            "lisa_stage_name", "lisa_forward_stage", "lisa_forward_noalloc", "lisa_backward_workspace_bytes",
            "lisa_backward", "lisa_backward_mlp_workspace_bytes", "lisa_backward_mlp", "lisa_status_string",
            "lisa_abi_version", "lisa_query_status", "lisa_selftest_wait_timeout",
            "lisa_forward_resident")

LISA_NOALLOC_SCRATCH_BYTES = 32 << 20


class lisa_weights(ctypes.Structure):
    _fields_ = [
        ("mode", ctypes.c_int),
        ("beta", ctypes.c_float),
        ("w", ctypes.POINTER(ctypes.c_float)),
        ("W1", ctypes.c_void_p),
        ("b1", ctypes.c_void_p),
        ("W2", ctypes.c_void_p),
        ("b2", ctypes.c_void_p),
        ("hidden", ctypes.c_int),
    ]


class lisa_mlp_grads(ctypes.Structure):
    _fields_ = [("dW1", ctypes.c_void_p), ("db1", ctypes.c_void_p), ("dW2", ctypes.c_void_p),
                ("db2", ctypes.c_void_p)]


class LisaError(RuntimeError):
    def __init__(self, status: int):
        self.status = status
        super().__init__(lisa_status_string(status))


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load liblisa.so (built by hop_stochastic_vision_gb300.build); raise if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError("liblisa.so is not built (%s); run hop_stochastic_vision_gb300.build" % path)
        lib = ctypes.CDLL(path)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        wp = ctypes.POINTER(lisa_weights)
        lib.lisa_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i]
        lib.lisa_workspace_bytes.restype = sz
        lib.lisa_forward.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, wp, vp, f, i, i, vp, sz, vp]
        lib.lisa_forward.restype = i
        lib.lisa_forward_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, wp, vp,
                                          f, i, i, vp, sz, vp]
        lib.lisa_forward_host.restype = i
        lib.lisa_num_stages.argtypes = [i, i, i, i, i, i, i, wp]
        lib.lisa_num_stages.restype = i
        lib.lisa_stage_name.argtypes = [i, i, i, i, i, i, i, wp, i]
        lib.lisa_stage_name.restype = ctypes.c_char_p
        lib.lisa_forward_stage.argtypes = [i] + lib.lisa_forward.argtypes
        lib.lisa_forward_stage.restype = i
        lib.lisa_forward_noalloc.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, wp, vp, f, i, i, vp]
        lib.lisa_forward_noalloc.restype = i
        lib.lisa_backward_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i]
        lib.lisa_backward_workspace_bytes.restype = sz
        lib.lisa_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, wp, vp, f, i, i,
                                      vp, sz, vp]
        lib.lisa_backward.restype = i
        lib.lisa_backward_mlp_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i, i]
        lib.lisa_backward_mlp_workspace_bytes.restype = sz
        lib.lisa_backward_mlp.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ctypes.POINTER(lisa_mlp_grads), i, i, i,
                                          i, i, i, i, wp, vp, f, i, i, vp, sz, vp]
        lib.lisa_backward_mlp.restype = i
        lib.lisa_status_string.argtypes = [i]
        lib.lisa_status_string.restype = ctypes.c_char_p
        lib.lisa_abi_version.argtypes = []
        lib.lisa_abi_version.restype = i
        lib.lisa_query_status.argtypes = [vp, vp]
        lib.lisa_query_status.restype = i
        lib.lisa_selftest_wait_timeout.argtypes = [ctypes.c_longlong, vp, sz, vp]
        lib.lisa_selftest_wait_timeout.restype = i
        lib.lisa_forward_resident.argtypes = lib.lisa_forward.argtypes
        lib.lisa_forward_resident.restype = i
        _lib = lib
        return lib


# -- the C entry points under their own names ---------------------------------------

def lisa_status_string(status: int) -> str:
    return load().lisa_status_string(int(status)).decode()


def lisa_abi_version() -> int:
    return int(load().lisa_abi_version())


def lisa_query_status(workspace, stream) -> int:
    return int(load().lisa_query_status(workspace, stream))


def lisa_selftest_wait_timeout(cycles, workspace, workspace_bytes, stream) -> int:
    return int(load().lisa_selftest_wait_timeout(cycles, workspace, workspace_bytes, stream))


def lisa_forward_resident(Q, K, V, O, B, heads, H, W, d_h, d_v, T, wts, alpha, eps, relu_inputs, dtype,
                          workspace, workspace_bytes, stream) -> int:
    """Test hook: lisa_forward's raw call through the single-kernel
    tensor-core path (LISA_ERR_UNSUPPORTED where it does not apply)."""
    return int(load().lisa_forward_resident(Q, K, V, O, B, heads, H, W, d_h, d_v, T, ctypes.byref(wts),
                                            alpha, eps, relu_inputs, dtype, workspace, workspace_bytes,
                                            stream))


def lisa_workspace_bytes(B, heads, H, W, d_h, d_v, T, dtype) -> int:
    return int(load().lisa_workspace_bytes(B, heads, H, W, d_h, d_v, T, dtype))


def lisa_forward(Q, K, V, O, B, heads, H, W, d_h, d_v, T, wts, alpha, eps, relu_inputs, dtype,
                 workspace, workspace_bytes, stream) -> int:
    """Raw call: pointers are ints (device addresses), wts a lisa_weights."""
    return int(load().lisa_forward(Q, K, V, O, B, heads, H, W, d_h, d_v, T, ctypes.byref(wts), alpha,
                                   eps, relu_inputs, dtype, workspace, workspace_bytes, stream))


def lisa_num_stages(B, heads, H, W, d_h, T, dtype, wts) -> int:
    return int(load().lisa_num_stages(B, heads, H, W, d_h, T, dtype, ctypes.byref(wts)))


def lisa_stage_name(B, heads, H, W, d_h, T, dtype, wts, stage):
    r = load().lisa_stage_name(B, heads, H, W, d_h, T, dtype, ctypes.byref(wts), stage)
    return None if r is None else r.decode()


def lisa_forward_stage(stage, Q, K, V, O, B, heads, H, W, d_h, d_v, T, wts, alpha, eps, relu_inputs,
                       dtype, workspace, workspace_bytes, stream) -> int:
    return int(load().lisa_forward_stage(stage, Q, K, V, O, B, heads, H, W, d_h, d_v, T,
                                         ctypes.byref(wts), alpha, eps, relu_inputs, dtype,
                                         workspace, workspace_bytes, stream))


def lisa_forward_noalloc(Q, K, V, O, B, heads, H, W, d_h, d_v, T, wts, alpha, eps, relu_inputs, dtype,
                         stream) -> int:
    """lisa_forward for callers that cannot allocate device memory: the
    library's own fixed scratch array replaces the workspace (see lisa.h)."""
    return int(load().lisa_forward_noalloc(Q, K, V, O, B, heads, H, W, d_h, d_v, T, ctypes.byref(wts),
                                           alpha, eps, relu_inputs, dtype, stream))


def lisa_backward_workspace_bytes(B, heads, H, W, d_h, d_v, T, dtype) -> int:
    return int(load().lisa_backward_workspace_bytes(B, heads, H, W, d_h, d_v, T, dtype))


def lisa_backward(Q, K, V, dO, dQ, dK, dV, dalpha, B, heads, H, W, d_h, d_v, T, wts, alpha, eps, relu_inputs,
                  dtype, workspace, workspace_bytes, stream) -> int:
    return int(load().lisa_backward(Q, K, V, dO, dQ, dK, dV, dalpha, B, heads, H, W, d_h, d_v, T,
                                    ctypes.byref(wts), alpha, eps, relu_inputs, dtype, workspace,
                                    workspace_bytes, stream))


def lisa_backward_mlp_workspace_bytes(B, heads, H, W, d_h, d_v, T, hidden, dtype) -> int:
    return int(load().lisa_backward_mlp_workspace_bytes(B, heads, H, W, d_h, d_v, T, hidden, dtype))


def lisa_backward_mlp(Q, K, V, dO, dQ, dK, dV, dalpha, mgrads, B, heads, H, W, d_h, d_v, T, wts, alpha, eps,
                      relu_inputs, dtype, workspace, workspace_bytes, stream) -> int:
    """mgrads: a lisa_mlp_grads (or None for a null pointer)."""
    return int(load().lisa_backward_mlp(Q, K, V, dO, dQ, dK, dV, dalpha,
                                        None if mgrads is None else ctypes.byref(mgrads), B, heads, H, W, d_h,
                                        d_v, T, ctypes.byref(wts), alpha, eps, relu_inputs, dtype, workspace,
                                        workspace_bytes, stream))


def lisa_forward_host(hQ, hK, hV, hO, dQ, dK, dV, dO, B, heads, H, W, d_h, d_v, T, wts, alpha, eps,
                      relu_inputs, dtype, workspace, workspace_bytes, stream) -> int:
    return int(load().lisa_forward_host(hQ, hK, hV, hO, dQ, dK, dV, dO, B, heads, H, W, d_h, d_v, T,
                                        ctypes.byref(wts), alpha, eps, relu_inputs, dtype, workspace,
                                        workspace_bytes, stream))


# -- tensor-level convenience ---------------------------------------------------------

_DTYPES = {torch.float32: LISA_F32, torch.bfloat16: LISA_BF16}

# relu_inputs codes: the feature map applied to Q and K on load
_FEATURE_MAPS = {False: 0, True: 1, "none": 0, "relu": 1, "elu1": 2}


def feature_map_code(relu) -> int:
    """relu=True (ReLU, the default), False (the inputs are the features) or
    "elu1" (ELU(x) + 1) as the C ABI's relu_inputs value."""
    if relu not in _FEATURE_MAPS:
        raise ValueError("relu must be True, False, 'none', 'relu' or 'elu1'")
    return _FEATURE_MAPS[relu]


def make_weights(T: int, beta=None, w=None, mlp=None):
    """Build the lisa_weights struct.  Returns (struct, keepalive) -- keep the
    second item alive for as long as the struct is used."""
    wt = lisa_weights()
    keep = []
    if w is not None:
        arr = (ctypes.c_float * T)(*[float(x) for x in w])
        keep.append(arr)
        wt.mode = LISA_W_FIXED
        wt.w = ctypes.cast(arr, ctypes.POINTER(ctypes.c_float))
    elif mlp is not None:
        W1, b1, W2, b2 = mlp
        for t in (W1, b1, W2, b2):
            if not (t.is_cuda and t.dtype == torch.float32 and t.is_contiguous()):
                raise ValueError("MLP parameters must be contiguous fp32 CUDA tensors")
        keep.extend((W1, b1, W2, b2))
        wt.mode = LISA_W_MLP
        wt.W1, wt.b1, wt.W2, wt.b2 = W1.data_ptr(), b1.data_ptr(), W2.data_ptr(), b2.data_ptr()
        wt.hidden = int(W1.shape[0])
    elif beta is not None:
        wt.mode = LISA_W_GEOMETRIC
        wt.beta = float(beta)
    else:
        raise ValueError("give beta, w or mlp")
    return wt, keep


def workspace_for(q: torch.Tensor, T: int) -> torch.Tensor:
    B, heads, n, d = q.shape
    nbytes = lisa_workspace_bytes(B, heads, n, 1, d, d, T, _DTYPES[q.dtype])
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)


def forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, grid, T: int, *, alpha: torch.Tensor,
            beta=None, w=None, mlp=None, eps: float = 1e-6, relu: bool = True, out=None,
            workspace=None, stream=None) -> torch.Tensor:
    """LiSA forward on CUDA tensors [B, heads, H*W, d] (fp32 or bf16).
    Returns O (a new tensor unless ``out`` is given)."""
    if not (q.is_cuda and k.is_cuda and v.is_cuda and alpha.is_cuda):
        raise ValueError("lisa.forward runs on CUDA tensors only")
    if q.dtype not in _DTYPES or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share dtype float32 or bfloat16")
    if alpha.dtype != torch.float32:
        raise ValueError("alpha must be fp32")
    for t in (q, k, v, alpha):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    B, heads, n, d = q.shape
    H, W = grid
    dv = v.shape[-1]
    O = torch.empty_like(v) if out is None else out
    wt, keep = make_weights(T, beta=beta, w=w, mlp=mlp)
    dt = _DTYPES[q.dtype]
    nbytes = lisa_workspace_bytes(B, heads, H, W, d, dv, T, dt)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    st = torch.cuda.current_stream(q.device).cuda_stream if stream is None else stream
    status = lisa_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), O.data_ptr(), B, heads, H, W, d,
                          dv, T, wt, alpha.data_ptr(), float(eps), feature_map_code(relu), dt,
                          workspace.data_ptr(), workspace.numel(), st)
    del keep
    if status != LISA_OK:
        raise LisaError(status)
    return O


def backward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, dO: torch.Tensor, grid, T: int, *,
             alpha: torch.Tensor, beta=None, w=None, mlp=None, eps: float = 1e-6, relu: bool = True,
             workspace=None, stream=None):
    """Gradients of the LiSA forward on CUDA tensors [B, heads, H*W, d]
    (fp32 or bf16) for the upstream gradient ``dO``: returns
    (dq, dk, dv, dalpha), dalpha fp32 [heads] summed over the batch.  With
    ``mlp`` = (W1, b1, W2, b2) (adaptive weights) it returns a fifth item,
    (dW1, db1, dW2, db2), the parameters' gradients summed over every slice."""
    for t in (q, k, v, dO, alpha):
        if not t.is_cuda:
            raise ValueError("lisa.backward runs on CUDA tensors only")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    if q.dtype not in _DTYPES or k.dtype != q.dtype or v.dtype != q.dtype or dO.dtype != q.dtype:
        raise ValueError("q, k, v, dO must share dtype float32 or bfloat16")
    if alpha.dtype != torch.float32:
        raise ValueError("alpha must be fp32")
    B, heads, n, d = q.shape
    H, W = grid
    dv = v.shape[-1]
    dq, dk, dvv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dalpha = torch.empty(heads, dtype=torch.float32, device=q.device)
    wt, keep = make_weights(T, beta=beta, w=w, mlp=mlp)
    dt = _DTYPES[q.dtype]
    st = torch.cuda.current_stream(q.device).cuda_stream if stream is None else stream
    if mlp is None:
        nbytes = lisa_backward_workspace_bytes(B, heads, H, W, d, dv, T, dt)
    else:
        hidden = int(mlp[0].shape[0])
        nbytes = lisa_backward_mlp_workspace_bytes(B, heads, H, W, d, dv, T, hidden, dt)
        pg = tuple(torch.empty_like(x) for x in mlp)
        mg = lisa_mlp_grads(pg[0].data_ptr(), pg[1].data_ptr(), pg[2].data_ptr(), pg[3].data_ptr())
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    if mlp is None:
        status = lisa_backward(q.data_ptr(), k.data_ptr(), v.data_ptr(), dO.data_ptr(), dq.data_ptr(),
                               dk.data_ptr(), dvv.data_ptr(), dalpha.data_ptr(), B, heads, H, W, d, dv, T, wt,
                               alpha.data_ptr(), float(eps), feature_map_code(relu), dt, workspace.data_ptr(),
                               workspace.numel(), st)
    else:
        status = lisa_backward_mlp(q.data_ptr(), k.data_ptr(), v.data_ptr(), dO.data_ptr(), dq.data_ptr(),
                                   dk.data_ptr(), dvv.data_ptr(), dalpha.data_ptr(), mg, B, heads, H, W, d, dv, T,
                                   wt, alpha.data_ptr(), float(eps), feature_map_code(relu), dt, workspace.data_ptr(),
                                   workspace.numel(), st)
    del keep
    if status != LISA_OK:
        raise LisaError(status)
    if mlp is not None:
        return dq, dk, dvv, dalpha, pg
    return dq, dk, dvv, dalpha
