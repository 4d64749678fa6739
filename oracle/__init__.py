"""Double-precision CPU oracle of the LiSA layer: forward and backward.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The product path (the CUDA library and
its Python binding) never imports this package, and this package imports
nothing from the product path.

The arithmetic lives in ``lisa_oracle.c`` (plain C, double precision, loops
written from "LiSA: Linear Stochastic Attention for Long-Range Visual
Modeling", reading note of arXiv 2611.04216v2); this module only compiles it
with gcc and marshals numpy float64 arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lisa_oracle.c")
_LIB = os.path.join(_HERE, "liblisa_oracle.so")
_lock = threading.Lock()
_lib = None

EXPLICIT = 0
LOWRANK = 1
W_GEOMETRIC = 0
W_FIXED = 1
W_MLP = 2


def build(force: bool = False) -> str:
    """Compile ``lisa_oracle.c`` into ``liblisa_oracle.so`` next to it.

    -O2 without -ffast-math keeps the C evaluation order; OpenMP only spreads
    independent outputs (query rows, matrix entries, tokens) over threads, so
    every sum keeps its serial order and the result does not depend on the
    thread count.
    """
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        dp = ctypes.POINTER(ctypes.c_double)
        i, d = ctypes.c_int, ctypes.c_double
        lib.lisa_oracle_forward.argtypes = [dp, dp, dp, dp, dp, dp, i, i, i, i, i, i, i, i, d,
                                            dp, dp, dp, dp, dp, i, dp, d, i, i, i]
        lib.lisa_oracle_forward.restype = i
        lib.lisa_oracle_geometric_weights.argtypes = [d, i, dp]
        lib.lisa_oracle_geometric_weights.restype = i
        lib.lisa_oracle_transition.argtypes = [dp, dp, i, i, d, i, dp]
        lib.lisa_oracle_transition.restype = i
        lib.lisa_oracle_step_weights.argtypes = [dp, dp, i, i, i, dp, dp, dp, dp, i, i, dp]
        lib.lisa_oracle_step_weights.restype = i
        lib.lisa_oracle_backward.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, i, i, i, i, i, i, i, i, d,
                                             dp, dp, dp, dp, dp, i, dp, dp, dp, dp, dp, d, i]
        lib.lisa_oracle_backward.restype = i
        lib.lisa_oracle_max_threads.argtypes = []
        lib.lisa_oracle_max_threads.restype = i
        _lib = lib
        return lib


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


FEATURE_MAPS = {False: 0, True: 1, "none": 0, "relu": 1, "elu1": 2}


def _fmap(relu):
    """The feature-map code: relu=True (ReLU, the default), False (inputs are
    the features), or "elu1" for phi(x) = ELU(x) + 1."""
    if relu not in FEATURE_MAPS:
        raise ValueError("relu must be True, False, 'none', 'relu' or 'elu1'")
    return FEATURE_MAPS[relu]


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def max_threads() -> int:
    return int(_load().lisa_oracle_max_threads())


def geometric_weights(beta: float, T: int) -> np.ndarray:
    """w_k = (1-beta) beta^k / (1-beta^T), k = 0..T-1 (paper Eq. 4)."""
    out = np.empty(T, dtype=np.float64)
    if _load().lisa_oracle_geometric_weights(float(beta), int(T), _ptr(out)) != 0:
        raise ValueError("geometric weights need T >= 1 and 0 <= beta < 1")
    return out


def forward(xq, xk, v, grid, T, *, alpha, beta=None, w=None, mlp=None, eps=1e-6,
            relu=True, mode=LOWRANK, nthreads=0, branches=False):
    """LiSA forward in double precision.

    xq, xk: [B, heads, n, d_h]; v: [B, heads, n, d_v]; grid = (H, W), n = H*W.
    Exactly one of ``beta`` (geometric weights), ``w`` (fixed weights, length
    T) or ``mlp`` = (W1 [hidden, 2 d_h], b1 [hidden], W2 [T, hidden], b2 [T])
    selects the walk weights.  ``T = 0`` with ``beta`` is the untruncated
    geometric walk, g = (1 - beta) (I - beta S)^-1 V.  ``alpha`` is a scalar
    or [heads].  ``relu``: the feature map -- True (ReLU, the paper's
    default), False (the inputs are the features) or "elu1" (ELU(x) + 1).
    Returns O, or (O, G, L) with the global and local branches when
    ``branches`` is set.
    """
    xq, xk, v = _f64(xq), _f64(xk), _f64(v)
    if xq.ndim != 4 or xk.shape != xq.shape or v.ndim != 4 or v.shape[:3] != xq.shape[:3]:
        raise ValueError("expected xq, xk [B, heads, n, d_h] and v [B, heads, n, d_v]")
    B, heads, n, dh = xq.shape
    dv = v.shape[3]
    H, W = grid
    if H * W != n:
        raise ValueError("grid does not match n")
    alpha = np.broadcast_to(np.asarray(alpha, dtype=np.float64), (heads,)).copy()
    wmode, wv, W1 = W_GEOMETRIC, None, None
    b1 = W2 = b2 = None
    hidden = 0
    if T == 0 and (beta is None or w is not None or mlp is not None):
        raise ValueError("T = 0 (untruncated walk) needs geometric weights (beta)")
    if w is not None:
        wmode, wv = W_FIXED, _f64(w)
        if wv.shape != (T,):
            raise ValueError("fixed weights need length T")
    elif mlp is not None:
        wmode = W_MLP
        W1, b1, W2, b2 = (_f64(x) for x in mlp)
        hidden = W1.shape[0]
        if W1.shape != (hidden, 2 * dh) or b1.shape != (hidden,) or W2.shape != (T, hidden) or b2.shape != (T,):
            raise ValueError("bad MLP parameter shapes")
    elif beta is None:
        raise ValueError("give beta, w or mlp")
    O = np.empty((B, heads, n, dv))
    G = np.empty_like(O) if branches else None
    L = np.empty_like(O) if branches else None
    rc = _load().lisa_oracle_forward(
        _ptr(xq), _ptr(xk), _ptr(v), _ptr(O), _ptr(G), _ptr(L), B, heads, H, W, dh, dv, int(T),
        wmode, float(beta if beta is not None else 0.0), _ptr(wv), _ptr(W1), _ptr(b1), _ptr(W2),
        _ptr(b2), hidden, _ptr(alpha), float(eps), _fmap(relu), int(mode), int(nthreads))
    if rc != 0:
        raise ValueError("lisa_oracle_forward failed with code %d" % rc)
    return (O, G, L) if branches else O


def backward(xq, xk, v, dO, grid, T, *, alpha, beta=None, w=None, mlp=None, eps=1e-6, relu=True):
    """Gradients of the LiSA forward for the upstream gradient ``dO``:
    returns (dXq, dXk, dV, dalpha), dalpha summed over the batch per head.
    Weights as for ``forward`` (T = 0 with ``beta``: the untruncated walk).
    With ``mlp`` = (W1, b1, W2, b2) it returns a fifth item, (dW1, db1, dW2,
    db2), the parameter gradients summed over every slice."""
    xq, xk, v, dO = _f64(xq), _f64(xk), _f64(v), _f64(dO)
    B, heads, n, dh = xq.shape
    dv = v.shape[3]
    H, W = grid
    if H * W != n or dO.shape != v.shape or xk.shape != xq.shape:
        raise ValueError("bad shapes")
    alpha = np.broadcast_to(np.asarray(alpha, dtype=np.float64), (heads,)).copy()
    W1 = b1 = W2 = b2 = gW1 = gb1 = gW2 = gb2 = None
    hidden = 0
    if w is not None:
        wmode, wv = W_FIXED, _f64(w)
        if T == 0 or wv.shape != (T,):
            raise ValueError("fixed weights need length T >= 1")
    elif mlp is not None:
        wmode, wv = W_MLP, None
        W1, b1, W2, b2 = (_f64(x) for x in mlp)
        hidden = W1.shape[0]
        if T < 1 or W1.shape != (hidden, 2 * dh) or b1.shape != (hidden,) or W2.shape != (T, hidden) or \
                b2.shape != (T,):
            raise ValueError("bad MLP parameter shapes")
        gW1, gb1, gW2, gb2 = np.empty_like(W1), np.empty_like(b1), np.empty_like(W2), np.empty_like(b2)
    elif beta is not None:
        wmode, wv = W_GEOMETRIC, None
    else:
        raise ValueError("give beta, w or mlp")
    dXq, dXk, dV = np.empty_like(xq), np.empty_like(xk), np.empty_like(v)
    da = np.empty(heads)
    rc = _load().lisa_oracle_backward(
        _ptr(xq), _ptr(xk), _ptr(v), _ptr(dO), _ptr(dXq), _ptr(dXk), _ptr(dV), _ptr(da), B, heads, H, W,
        dh, dv, int(T), wmode, float(beta if beta is not None else 0.0), _ptr(wv), _ptr(W1), _ptr(b1),
        _ptr(W2), _ptr(b2), hidden, _ptr(gW1), _ptr(gb1), _ptr(gW2), _ptr(gb2), _ptr(alpha), float(eps),
        _fmap(relu))
    if rc != 0:
        raise ValueError("lisa_oracle_backward failed with code %d" % rc)
    if mlp is not None:
        return dXq, dXk, dV, da, (gW1, gb1, gW2, gb2)
    return dXq, dXk, dV, da


def transition(xq, xk, eps=1e-6, relu=True):
    """Dense n x n transition S = Q~ K^T of one slice (xq, xk: [n, d_h])."""
    xq, xk = _f64(xq), _f64(xk)
    n, dh = xq.shape
    S = np.empty((n, n))
    if _load().lisa_oracle_transition(_ptr(xq), _ptr(xk), n, dh, float(eps), _fmap(relu), _ptr(S)):
        raise ValueError("lisa_oracle_transition failed")
    return S


def step_weights(xq, xk, mlp, T, relu=True):
    """Adaptive walk weights [n, T] of one slice (xq, xk: [n, d_h])."""
    xq, xk = _f64(xq), _f64(xk)
    n, dh = xq.shape
    W1, b1, W2, b2 = (_f64(x) for x in mlp)
    out = np.empty((n, T))
    rc = _load().lisa_oracle_step_weights(_ptr(xq), _ptr(xk), n, dh, int(T), _ptr(W1), _ptr(b1),
                                          _ptr(W2), _ptr(b2), W1.shape[0], _fmap(relu), _ptr(out))
    if rc:
        raise ValueError("lisa_oracle_step_weights failed")
    return out
