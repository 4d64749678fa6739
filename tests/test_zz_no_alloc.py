"""lisa_forward_noalloc: the LiSA layer for callers that cannot allocate
device memory while they run it (an operator inside an engine that owns all
device memory through its own planned pool, a serving loop that cannot take
the synchronisation of cudaFree).  It runs in a fixed scratch array compiled
into the library instead of a caller workspace.

Each case calls it twice in a row through the C ABI and compares both
outputs with lisa_forward's (caller-allocated workspace), within the parity
tolerance of the other GPU tests.  The file name makes pytest collect it
last; it builds and loads the library itself, so it also runs alone in a
fresh process."""
import pytest
import torch

from lisa_synth import SHAPES, make_inputs, to_f64

from helpers import TOL, max_rel_err, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lisa():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from hop_stochastic_vision_gb300 import build, lisa as binding
    build.build()
    binding.load()
    return binding


def _weights(binding, shape, d):
    if shape.weights == "mlp":
        return binding.make_weights(shape.T, mlp=tuple(d[k] for k in ("W1", "b1", "W2", "b2")))
    return binding.make_weights(shape.T, beta=shape.beta)


@pytest.mark.parametrize("name,B", [("deit_t_14x14", 8), ("deit_t384_24x24_mlp", 4),
                                    ("pvt_t_s1_56x56_T5", 4), ("tiny_f32_14x14_d16", 1)])
def test_noalloc_matches_lisa_forward_twice(lisa, name, B):
    shape = SHAPES[name]
    inp = make_inputs(shape, B=B)
    d = to_device(inp)
    heads, n, D = shape.heads, shape.n, shape.d
    dt = lisa.LISA_BF16 if shape.dtype == "bf16" else lisa.LISA_F32
    assert 0 < lisa.lisa_workspace_bytes(B, heads, shape.H, shape.W, D, D, shape.T, dt) \
        <= lisa.LISA_NOALLOC_SCRATCH_BYTES
    wt, keep = _weights(lisa, shape, d)
    kw = {"mlp": tuple(d[k] for k in ("W1", "b1", "W2", "b2"))} if shape.weights == "mlp" \
        else {"beta": shape.beta}
    ref = lisa.forward(d["xq"], d["xk"], d["v"], (shape.H, shape.W), shape.T, alpha=d["alpha"], **kw)
    stream = torch.cuda.current_stream().cuda_stream
    outs = []
    for _ in range(2):
        o = torch.full_like(d["v"], float("nan"))
        rc = lisa.lisa_forward_noalloc(d["xq"].data_ptr(), d["xk"].data_ptr(), d["v"].data_ptr(),
                                       o.data_ptr(), B, heads, shape.H, shape.W, D, D, shape.T, wt,
                                       d["alpha"].data_ptr(), 1e-6, 1, dt, stream)
        assert rc == lisa.LISA_OK, lisa.lisa_status_string(rc)
        outs.append(o)
    torch.cuda.synchronize()
    want = to_f64(ref)
    for o in outs:
        assert max_rel_err(to_f64(o), want) <= TOL[shape.dtype]


def test_noalloc_rejects_problems_beyond_its_scratch(lisa):
    B, heads, H, W, D, T = 4096, 1, 14, 14, 64, 16
    dt = lisa.LISA_BF16
    assert lisa.lisa_workspace_bytes(B, heads, H, W, D, D, T, dt) > lisa.LISA_NOALLOC_SCRATCH_BYTES
    q = torch.zeros(B, heads, H * W, D, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros_like(q)
    alpha = torch.full((heads,), 0.5, device="cuda")
    wt, keep = lisa.make_weights(T, beta=0.5)
    rc = lisa.lisa_forward_noalloc(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), B, heads, H,
                                   W, D, D, T, wt, alpha.data_ptr(), 1e-6, 1, dt,
                                   torch.cuda.current_stream().cuda_stream)
    assert rc == lisa.LISA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert int(o.abs().sum()) == 0          # nothing was launched
