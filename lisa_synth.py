"""Seeded synthetic inputs for the LiSA forward layer, shared by the tests and
the benchmark.

This module holds no arithmetic of the method: it only draws random tensors
(torch CPU generator, fixed seed, fixed draw order Xq, Xk, V, alpha, W1, b1,
W2, b2) in the shapes of the vision-transformer layers the LiSA paper plugs
into, and lists those layer shapes.  Both the CUDA path and the oracle
consume what it returns; neither is imported here.

The real workloads are DeiT / PVT attention layers on ImageNet images; no
dataset or trained weight is available, so i.i.d. N(0, 1) projections stand
in for them (plus a structured variant whose transition matrix is close to
block-diagonal, so the multi-hop terms are not washed out by averaging).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class LayerShape:
    """One LiSA layer workload: B x heads slices on an H x W token grid."""
    name: str
    dtype: str            # "f32" or "bf16"
    B: int
    heads: int
    H: int
    W: int
    d: int                # d_h = d_v
    T: int                # walk truncation depth; 0 = untruncated (geometric weights only)
    weights: str          # "geometric" or "mlp"
    beta: float = 0.5
    alpha: str = "0.5"    # "0.5" or "uniform(0.3,0.7)" (one value per head)
    hidden: int = 32

    @property
    def n(self) -> int:
        return self.H * self.W

    @property
    def slices(self) -> int:
        return self.B * self.heads


# The layer shapes the paper's backbones give (patch grid only, no CLS token).
SHAPES = {
    "tiny_f32_14x14_d16": LayerShape("tiny_f32_14x14_d16", "f32", 1, 1, 14, 14, 16, 3, "geometric"),
    "deit_t_14x14": LayerShape("deit_t_14x14", "bf16", 64, 3, 14, 14, 64, 3, "geometric",
                               alpha="uniform(0.3,0.7)"),
    "deit_t384_24x24_mlp": LayerShape("deit_t384_24x24_mlp", "bf16", 64, 3, 24, 24, 64, 3, "mlp"),
    "pvt_t_s1_56x56_T3": LayerShape("pvt_t_s1_56x56_T3", "bf16", 32, 1, 56, 56, 64, 3, "geometric"),
    "pvt_t_s1_56x56_T5": LayerShape("pvt_t_s1_56x56_T5", "bf16", 32, 1, 56, 56, 64, 5, "geometric"),
    # the same layer with the untruncated geometric walk (T = 0)
    "pvt_t_s1_56x56_untruncated": LayerShape("pvt_t_s1_56x56_untruncated", "bf16", 32, 1, 56, 56, 64, 0,
                                             "geometric"),
}
for _g in (64, 128, 256):
    for _T in (3, 5):
        _k = "long_%dx%d_T%d_mlp" % (_g, _g, _T)
        SHAPES[_k] = LayerShape(_k, "bf16", 1, 4, _g, _g, 64, _T, "mlp")

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def make_inputs(shape: LayerShape, seed: int = 0, B: Optional[int] = None,
                heads: Optional[int] = None, structured: bool = False) -> dict:
    """Draw one batch of inputs for ``shape`` (optionally with a smaller B or
    head count).  Returns CPU tensors: xq, xk [B, heads, n, d] and v
    [B, heads, n, d] in the layer dtype; alpha [heads] fp32; and, for MLP
    weights, W1 [hidden, 2d], b1 [hidden], W2 [T, hidden], b2 [T] fp32."""
    B = shape.B if B is None else B
    heads = shape.heads if heads is None else heads
    g = torch.Generator("cpu").manual_seed(seed)
    n, d = shape.n, shape.d
    if structured:
        xq, xk, v = _structured(shape, B, heads, g)
    else:
        xq = torch.randn(B, heads, n, d, generator=g)
        xk = torch.randn(B, heads, n, d, generator=g)
        v = torch.randn(B, heads, n, d, generator=g)
    if shape.alpha == "0.5":
        alpha = torch.full((heads,), 0.5)
    else:
        alpha = 0.3 + 0.4 * torch.rand(heads, generator=g)
    out = {"xq": xq, "xk": xk, "v": v, "alpha": alpha}
    if shape.weights == "mlp":
        out["W1"] = 0.02 * torch.randn(shape.hidden, 2 * d, generator=g)
        out["b1"] = 0.02 * torch.randn(shape.hidden, generator=g)
        out["W2"] = 0.02 * torch.randn(shape.T, shape.hidden, generator=g)
        out["b2"] = 0.02 * torch.randn(shape.T, generator=g)
    dt = TORCH_DTYPE[shape.dtype]
    for key in ("xq", "xk", "v"):
        out[key] = out[key].to(dt).contiguous()
    return out


def _structured(shape: LayerShape, B: int, heads: int, g: torch.Generator):
    """Tokens fall in four spatial quadrants; queries and keys are close to a
    one-hot code of their quadrant, values are a smooth field plus noise.
    The resulting transition matrix is nearly block-diagonal, so S^2 V, S^3 V
    differ visibly from the mean of V."""
    H, W, d = shape.H, shape.W, shape.d
    r = torch.arange(H).view(H, 1).expand(H, W)
    c = torch.arange(W).view(1, W).expand(H, W)
    quad = ((r >= (H + 1) // 2).long() * 2 + (c >= (W + 1) // 2).long()).reshape(-1)
    code = torch.zeros(H * W, d)
    code[torch.arange(H * W), quad % d] = 3.0
    xq = code + 0.3 * torch.randn(B, heads, H * W, d, generator=g)
    xk = code + 0.3 * torch.randn(B, heads, H * W, d, generator=g)
    yy = (r.float() / max(H - 1, 1)).reshape(-1, 1)
    xx = (c.float() / max(W - 1, 1)).reshape(-1, 1)
    freq = torch.arange(1, d + 1).float().view(1, d)
    field = torch.sin(3.0 * yy * freq / d * 4.0) + torch.cos(2.0 * xx * freq / d * 4.0)
    v = field + 0.2 * torch.randn(B, heads, H * W, d, generator=g)
    return xq, xk, v


def to_f64(t: torch.Tensor):
    """The exact values a kernel sees (after the dtype cast), widened to
    float64 numpy for the oracle."""
    return t.detach().to("cpu").to(torch.float64).numpy()
