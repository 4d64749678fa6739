"""Shared helpers of the GPU parity tests: run the CUDA path and the oracle
on the same seeded inputs and measure the normwise error the tolerances are
stated in (max over (batch, head) slices of ||x - y||_inf / ||y||_inf)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from lisa_synth import to_f64

TOL = {"f32": 1e-4, "bf16": 2e-2}


def max_rel_err(x: np.ndarray, y: np.ndarray) -> float:
    """x, y: [B, heads, n, d]; y is the oracle."""
    x = x.reshape(x.shape[0] * x.shape[1], -1)
    y = y.reshape(y.shape[0] * y.shape[1], -1)
    if x.shape[1] == 0:
        return 0.0
    num = np.abs(x - y).max(axis=1)
    den = np.abs(y).max(axis=1)
    den = np.where(den > 0, den, 1.0)
    return float((num / den).max())


def oracle_weights_kwargs(inp: dict, weights: str, beta: float = 0.5, w=None):
    if w is not None:
        return {"w": np.asarray(w, dtype=np.float64)}
    if weights == "mlp":
        return {"mlp": tuple(inp[k].double().numpy() for k in ("W1", "b1", "W2", "b2"))}
    return {"beta": beta}


def run_oracle(inp: dict, grid, T: int, weights: str, *, beta=0.5, w=None, eps=1e-6, relu=True,
               mode=oracle.LOWRANK, branches=False, nthreads=0):
    return oracle.forward(to_f64(inp["xq"]), to_f64(inp["xk"]), to_f64(inp["v"]), grid, T,
                          alpha=inp["alpha"].double().numpy(), eps=eps, relu=relu, mode=mode,
                          branches=branches, nthreads=nthreads,
                          **oracle_weights_kwargs(inp, weights, beta, w))


def to_device(inp: dict, device="cuda") -> dict:
    return {k: v.to(device).contiguous() for k, v in inp.items()}


def run_gpu(dinp: dict, grid, T: int, weights: str, *, beta=0.5, w=None, eps=1e-6, relu=True,
            sync=True):
    from hop_stochastic_vision_gb300 import lisa
    kw = {}
    if w is not None:
        kw["w"] = list(w)
    elif weights == "mlp":
        kw["mlp"] = tuple(dinp[k] for k in ("W1", "b1", "W2", "b2"))
    else:
        kw["beta"] = beta
    out = lisa.forward(dinp["xq"], dinp["xk"], dinp["v"], grid, T, alpha=dinp["alpha"], eps=eps,
                       relu=relu, **kw)
    if sync:
        torch.cuda.synchronize()
    return out
