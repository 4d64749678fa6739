"""Device-side failure reporting: a bounded wait that gives up reaches the
caller through lisa_query_status, and every forward call starts with a
clean error word.

No test here faults, traps or hangs the GPU.  (a) The host writes the
timeout bits into a workspace's error word and the query must report them.
(b) The library's self-test kernel waits, with a limit of 2e5 SM cycles
(about 0.1 ms), on an mbarrier nothing arrives on -- through the same
bounded wait the tensor-core kernels use, with no TMA or tensor-core work in
flight -- and the query must return LISA_ERR_TIMEOUT; the context stays
usable, so a forward on the same workspace afterwards runs, reports
LISA_OK and matches the oracle."""
import pytest
import torch

from lisa_synth import SHAPES, make_inputs, to_f64

from helpers import TOL, max_rel_err, run_oracle, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lisa():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from hop_stochastic_vision_gb300 import build, lisa as binding
    build.build()
    binding.load()
    return binding


def _forward_into(lisa, d, shape, B, ws):
    dt = lisa.LISA_BF16 if shape.dtype == "bf16" else lisa.LISA_F32
    wt, keep = lisa.make_weights(shape.T, beta=shape.beta)
    o = torch.empty_like(d["v"])
    stream = torch.cuda.current_stream().cuda_stream
    rc = lisa.lisa_forward(d["xq"].data_ptr(), d["xk"].data_ptr(), d["v"].data_ptr(), o.data_ptr(), B,
                           shape.heads, shape.H, shape.W, shape.d, shape.d, shape.T, wt, d["alpha"].data_ptr(),
                           1e-6, 1, dt, ws.data_ptr(), ws.numel(), stream)
    assert rc == lisa.LISA_OK, lisa.lisa_status_string(rc)
    return o


@pytest.mark.parametrize("name,B", [("pvt_t_s1_56x56_T3", 2), ("tiny_f32_14x14_d16", 1)])
def test_error_word_is_reported_and_cleared_by_the_next_call(lisa, name, B):
    shape = SHAPES[name]
    dt = lisa.LISA_BF16 if shape.dtype == "bf16" else lisa.LISA_F32
    nbytes = lisa.lisa_workspace_bytes(B, shape.heads, shape.H, shape.W, shape.d, shape.d, shape.T, dt)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert lisa.lisa_query_status(ws.data_ptr(), stream) == lisa.LISA_OK
    ws[:4].copy_(torch.tensor([3, 0, 0, 0], dtype=torch.uint8))      # both timeout bits, set by the host
    assert lisa.lisa_query_status(ws.data_ptr(), stream) == lisa.LISA_ERR_TIMEOUT
    inp = make_inputs(shape, B=B)
    o = _forward_into(lisa, to_device(inp), shape, B, ws)
    assert lisa.lisa_query_status(ws.data_ptr(), stream) == lisa.LISA_OK
    assert max_rel_err(to_f64(o), run_oracle(inp, (shape.H, shape.W), shape.T, "geometric")) <= TOL[shape.dtype]


def test_a_wait_that_runs_out_is_reported_and_the_context_stays_usable(lisa):
    shape = SHAPES["pvt_t_s1_56x56_T3"]
    B = 2
    nbytes = lisa.lisa_workspace_bytes(B, 1, 56, 56, 64, 64, 3, lisa.LISA_BF16)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        assert lisa.lisa_selftest_wait_timeout(200000, ws.data_ptr(), nbytes, stream) == lisa.LISA_OK
        assert lisa.lisa_query_status(ws.data_ptr(), stream) == lisa.LISA_ERR_TIMEOUT
    inp = make_inputs(shape, B=B)
    o = _forward_into(lisa, to_device(inp), shape, B, ws)
    assert lisa.lisa_query_status(ws.data_ptr(), stream) == lisa.LISA_OK
    torch.cuda.synchronize()
    assert max_rel_err(to_f64(o), run_oracle(inp, (56, 56), 3, "geometric")) <= TOL["bf16"]
