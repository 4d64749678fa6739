"""The C ABI of liblisa.so on the host: the library loads without a GPU,
exports every function include/lisa.h declares, and rejects bad arguments
with a status code before anything is launched (no test here reaches a
kernel launch, so none needs a GPU)."""
import ctypes
import os
import re

import pytest

from hop_stochastic_vision_gb300 import build as lisa_build
from hop_stochastic_vision_gb300 import lisa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    lisa_build.build()
    lisa.load()


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"\b(lisa_\w+)\s*\(", text)
    return sorted(set(names))


def test_exports_every_declared_function():
    names = _declared_functions()
    assert "lisa_forward" in names and "lisa_workspace_bytes" in names
    lib = ctypes.CDLL(lisa.LIB_PATH)
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) <= set(lisa.EXPORTED) | set(names)
    for name in lisa.EXPORTED:
        assert name in names


def test_status_strings_and_version():
    assert lisa.lisa_abi_version() >= 100
    for st in range(6):
        assert lisa.lisa_status_string(st).startswith("LISA_")
    assert "unknown" in lisa.lisa_status_string(99)


def test_workspace_bytes():
    ws = lisa.lisa_workspace_bytes
    assert ws(32, 1, 56, 56, 64, 64, 3, lisa.LISA_BF16) > 0
    assert ws(32, 1, 56, 56, 64, 64, 5, lisa.LISA_BF16) >= ws(32, 1, 56, 56, 64, 64, 3, lisa.LISA_BF16)
    assert ws(0, 1, 56, 56, 64, 64, 3, lisa.LISA_BF16) == 0          # empty problem
    assert ws(1, 1, 4, 4, 48, 48, 3, lisa.LISA_BF16) == 0            # unsupported d
    assert ws(1, 1, 4, 4, 64, 32, 3, lisa.LISA_BF16) == 0            # d_v != d_h
    assert ws(1, 1, 4, 4, 64, 64, -1, lisa.LISA_BF16) == 0           # T < 0
    assert ws(1, 1, 4, 4, 64, 64, 0, lisa.LISA_BF16) > 0             # T = 0: untruncated walk
    assert ws(1, 1, 4, 4, 16, 16, 0, lisa.LISA_F32) == ws(1, 1, 4, 4, 16, 16, 2, lisa.LISA_F32)
    assert ws(1, 1, 4, 4, 64, 64, 3, 7) == 0                         # bad dtype
    assert ws(-1, 1, 4, 4, 64, 64, 3, lisa.LISA_F32) == 0
    assert ws(1, 1, 4, 4, 16, 16, 16, lisa.LISA_F32) > 0
    assert ws(1, 1, 4, 4, 16, 16, 17, lisa.LISA_F32) == 0


FAKE = 1 << 20          # a 16-byte aligned address; never dereferenced (checks fail first)


def _call(**over):
    args = dict(Q=FAKE, K=FAKE + 4096, V=FAKE + 8192, O=FAKE + 12288, B=1, heads=1, H=4, W=4, d_h=16,
                d_v=16, T=3, alpha=FAKE + 16384, eps=1e-6, relu=1, dtype=lisa.LISA_F32,
                workspace=FAKE + 32768, wbytes=1 << 30, beta=0.5)
    args.update(over)
    wt, keep = lisa.make_weights(args["T"] if args["T"] > 0 else 1, beta=args["beta"]) \
        if "wt" not in args else (args["wt"], None)
    return lisa.lisa_forward(args["Q"], args["K"], args["V"], args["O"], args["B"], args["heads"],
                             args["H"], args["W"], args["d_h"], args["d_v"], args["T"], wt,
                             args["alpha"], args["eps"], args["relu"], args["dtype"],
                             args["workspace"], args["wbytes"], 0)


@pytest.mark.parametrize("over,status", [
    (dict(Q=0), lisa.LISA_ERR_INVALID_ARG),
    (dict(K=0), lisa.LISA_ERR_INVALID_ARG),
    (dict(V=0), lisa.LISA_ERR_INVALID_ARG),
    (dict(O=0), lisa.LISA_ERR_INVALID_ARG),
    (dict(alpha=0), lisa.LISA_ERR_INVALID_ARG),
    (dict(Q=FAKE + 8), lisa.LISA_ERR_INVALID_ARG),                  # misaligned
    (dict(O=FAKE + 4), lisa.LISA_ERR_INVALID_ARG),
    (dict(O=FAKE + 4096), lisa.LISA_ERR_INVALID_ARG),               # O overlaps K
    (dict(B=-1), lisa.LISA_ERR_INVALID_ARG),
    (dict(H=-2), lisa.LISA_ERR_INVALID_ARG),
    (dict(T=-1), lisa.LISA_ERR_INVALID_ARG),
    (dict(T=0, beta=1.0), lisa.LISA_ERR_INVALID_ARG),              # untruncated needs beta < 1
    (dict(T=0, wbytes=16), lisa.LISA_ERR_WORKSPACE),
    (dict(T=17), lisa.LISA_ERR_UNSUPPORTED),
    (dict(d_h=48, d_v=48), lisa.LISA_ERR_UNSUPPORTED),
    (dict(d_h=128, d_v=128), lisa.LISA_ERR_UNSUPPORTED),
    (dict(d_v=32), lisa.LISA_ERR_UNSUPPORTED),
    (dict(d_h=0), lisa.LISA_ERR_INVALID_ARG),
    (dict(eps=0.0), lisa.LISA_ERR_INVALID_ARG),
    (dict(eps=-1e-6), lisa.LISA_ERR_INVALID_ARG),
    (dict(eps=float("nan")), lisa.LISA_ERR_INVALID_ARG),
    (dict(eps=float("inf")), lisa.LISA_ERR_INVALID_ARG),
    (dict(beta=1.0), lisa.LISA_ERR_INVALID_ARG),
    (dict(beta=-0.1), lisa.LISA_ERR_INVALID_ARG),
    (dict(relu=3), lisa.LISA_ERR_INVALID_ARG),
    (dict(relu=-1), lisa.LISA_ERR_INVALID_ARG),
    (dict(relu=2, wbytes=16), lisa.LISA_ERR_WORKSPACE),            # ELU + 1: a valid feature map
    (dict(dtype=5), lisa.LISA_ERR_INVALID_ARG),
    (dict(workspace=0), lisa.LISA_ERR_WORKSPACE),
    (dict(wbytes=16), lisa.LISA_ERR_WORKSPACE),
    (dict(workspace=FAKE + 32776), lisa.LISA_ERR_INVALID_ARG),      # misaligned workspace
])
def test_forward_rejects_before_launch(over, status):
    assert _call(**over) == status


def test_weight_struct_checks():
    wt = lisa.lisa_weights()
    wt.mode = 9
    assert _call(wt=wt) == lisa.LISA_ERR_INVALID_ARG
    wt = lisa.lisa_weights()
    wt.mode = lisa.LISA_W_FIXED                      # w missing
    assert _call(wt=wt) == lisa.LISA_ERR_INVALID_ARG
    arr = (ctypes.c_float * 3)(0.5, float("nan"), 0.5)
    wt.w = ctypes.cast(arr, ctypes.POINTER(ctypes.c_float))
    assert _call(wt=wt) == lisa.LISA_ERR_INVALID_ARG
    wt = lisa.lisa_weights()
    wt.mode = lisa.LISA_W_MLP                        # MLP pointers missing
    assert _call(wt=wt) == lisa.LISA_ERR_INVALID_ARG
    wt.W1 = wt.b1 = wt.W2 = wt.b2 = FAKE
    wt.hidden = 0
    assert _call(wt=wt) == lisa.LISA_ERR_INVALID_ARG
    wt.hidden = 65
    assert _call(wt=wt) == lisa.LISA_ERR_UNSUPPORTED
    wt.hidden = 32
    assert _call(wt=wt, T=9) == lisa.LISA_ERR_UNSUPPORTED
    assert _call(wt=wt, T=0) == lisa.LISA_ERR_INVALID_ARG      # untruncated walk: geometric only
    wt = lisa.lisa_weights()
    wt.mode = lisa.LISA_W_FIXED
    wt.w = ctypes.cast(arr, ctypes.POINTER(ctypes.c_float))
    assert _call(wt=wt, T=0) == lisa.LISA_ERR_INVALID_ARG
    # a null weight struct
    lib = lisa.load()
    rc = lib.lisa_forward(FAKE, FAKE, FAKE, FAKE, 1, 1, 4, 4, 16, 16, 3, None, FAKE, 1e-6, 1, 0,
                          FAKE, 1 << 30, None)
    assert rc == lisa.LISA_ERR_INVALID_ARG


def test_empty_problem_launches_nothing():
    # zero slices or zero tokens: OK with null buffers, nothing to do
    assert _call(B=0, Q=0, K=0, V=0, O=0, workspace=0) == lisa.LISA_OK
    assert _call(heads=0, Q=0, K=0, V=0, O=0, workspace=0) == lisa.LISA_OK
    assert _call(H=0, Q=0, K=0, V=0, O=0, workspace=0) == lisa.LISA_OK


def test_forward_host_checks_before_copies():
    wt, _ = lisa.make_weights(3, beta=0.5)
    dev = [FAKE + 4096 * i for i in range(4)]
    args = [FAKE] * 4 + dev + [1, 1, 4, 4, 16, 16, 3, wt, FAKE, 1e-6, 1, lisa.LISA_F32, FAKE, 16, 0]
    assert lisa.lisa_forward_host(*args) == lisa.LISA_ERR_WORKSPACE
    args[0] = 0
    args[-3], args[-2] = FAKE, 1 << 30
    assert lisa.lisa_forward_host(*args) == lisa.LISA_ERR_INVALID_ARG


def _bwd(**over):
    args = dict(Q=FAKE, K=FAKE + 4096, V=FAKE + 8192, dO=FAKE + 12288, dQ=FAKE + 16384, dK=FAKE + 20480,
                dV=FAKE + 24576, dalpha=FAKE + 28672, B=1, heads=1, H=4, W=4, d_h=16, d_v=16, T=3,
                alpha=FAKE + 28688, eps=1e-6, relu=1, dtype=lisa.LISA_F32, workspace=FAKE + 65536,
                wbytes=1 << 30, beta=0.5)
    args.update(over)
    wt = args.get("wt") or lisa.make_weights(max(args["T"], 1), beta=args["beta"])[0]
    return lisa.lisa_backward(args["Q"], args["K"], args["V"], args["dO"], args["dQ"], args["dK"], args["dV"],
                              args["dalpha"], args["B"], args["heads"], args["H"], args["W"], args["d_h"],
                              args["d_v"], args["T"], wt, args["alpha"], args["eps"], args["relu"],
                              args["dtype"], args["workspace"], args["wbytes"], 0)


def test_backward_workspace_bytes():
    ws = lisa.lisa_backward_workspace_bytes
    assert ws(32, 1, 56, 56, 64, 64, 3, lisa.LISA_BF16) > ws(1, 1, 56, 56, 64, 64, 3, lisa.LISA_BF16) > 0
    assert ws(1, 1, 4, 4, 64, 64, 0, lisa.LISA_BF16) > 0
    assert ws(0, 1, 4, 4, 64, 64, 3, lisa.LISA_BF16) == 0
    assert ws(1, 1, 4, 4, 48, 48, 3, lisa.LISA_BF16) == 0
    assert ws(1, 1, 4, 4, 64, 64, 17, lisa.LISA_BF16) == 0


@pytest.mark.parametrize("over,status", [
    (dict(dO=0), lisa.LISA_ERR_INVALID_ARG),
    (dict(dQ=0), lisa.LISA_ERR_INVALID_ARG),
    (dict(dalpha=0), lisa.LISA_ERR_INVALID_ARG),
    (dict(dK=FAKE + 8), lisa.LISA_ERR_INVALID_ARG),                 # misaligned
    (dict(dV=FAKE + 8192), lisa.LISA_ERR_INVALID_ARG),              # dV overlaps V
    (dict(dK=FAKE + 16384), lisa.LISA_ERR_INVALID_ARG),             # dK overlaps dQ
    (dict(dalpha=FAKE + 28688), lisa.LISA_ERR_INVALID_ARG),         # dalpha overlaps alpha
    (dict(T=-1), lisa.LISA_ERR_INVALID_ARG),
    (dict(T=17), lisa.LISA_ERR_UNSUPPORTED),
    (dict(d_h=48, d_v=48), lisa.LISA_ERR_UNSUPPORTED),
    (dict(eps=0.0), lisa.LISA_ERR_INVALID_ARG),
    (dict(beta=1.0), lisa.LISA_ERR_INVALID_ARG),
    (dict(relu=3), lisa.LISA_ERR_INVALID_ARG),
    (dict(workspace=0), lisa.LISA_ERR_WORKSPACE),
    (dict(wbytes=1024), lisa.LISA_ERR_WORKSPACE),
    (dict(T=0, wbytes=1024), lisa.LISA_ERR_WORKSPACE),
])
def test_backward_rejects_before_launch(over, status):
    assert _bwd(**over) == status


def test_backward_weight_modes():
    wt = lisa.lisa_weights()
    wt.mode = lisa.LISA_W_MLP
    wt.W1 = wt.b1 = wt.W2 = wt.b2 = FAKE
    wt.hidden = 32
    assert _bwd(wt=wt) == lisa.LISA_ERR_UNSUPPORTED             # adaptive weights: not covered
    wt = lisa.lisa_weights()
    wt.mode = lisa.LISA_W_FIXED
    arr = (ctypes.c_float * 3)(0.5, 0.25, 0.25)
    wt.w = ctypes.cast(arr, ctypes.POINTER(ctypes.c_float))
    assert _bwd(wt=wt, T=0) == lisa.LISA_ERR_INVALID_ARG        # untruncated: geometric only
    assert _bwd(wt=wt, wbytes=16) == lisa.LISA_ERR_WORKSPACE


def _bwd_mlp(wt=None, mg=True, **over):
    args = dict(Q=FAKE, K=FAKE + 4096, V=FAKE + 8192, dO=FAKE + 12288, dQ=FAKE + 16384, dK=FAKE + 20480,
                dV=FAKE + 24576, dalpha=FAKE + 28672, B=1, heads=1, H=4, W=4, d_h=16, d_v=16, T=3,
                alpha=FAKE + 28688, eps=1e-6, relu=1, dtype=lisa.LISA_F32, workspace=FAKE + 65536,
                wbytes=1 << 30, hidden=32)
    args.update(over)
    if wt is None:
        wt = lisa.lisa_weights()
        wt.mode = lisa.LISA_W_MLP
        wt.W1 = wt.b1 = wt.W2 = wt.b2 = FAKE + 40960
        wt.hidden = args["hidden"]
    grads = lisa.lisa_mlp_grads(FAKE + 49152, FAKE + 50176, FAKE + 51200, FAKE + 52224) if mg is True else mg
    return lisa.lisa_backward_mlp(args["Q"], args["K"], args["V"], args["dO"], args["dQ"], args["dK"], args["dV"],
                                  args["dalpha"], grads, args["B"], args["heads"], args["H"], args["W"],
                                  args["d_h"], args["d_v"], args["T"], wt, args["alpha"], args["eps"],
                                  args["relu"], args["dtype"], args["workspace"], args["wbytes"], 0)


def test_backward_mlp_workspace_bytes():
    ws = lisa.lisa_backward_mlp_workspace_bytes
    assert ws(8, 3, 24, 24, 64, 64, 3, 32, lisa.LISA_BF16) > lisa.lisa_backward_workspace_bytes(
        8, 3, 24, 24, 64, 64, 3, lisa.LISA_BF16)
    assert ws(1, 1, 4, 4, 64, 64, 9, 32, lisa.LISA_BF16) == 0        # T > LISA_MAX_T_MLP
    assert ws(1, 1, 4, 4, 64, 64, 0, 32, lisa.LISA_BF16) == 0        # no untruncated adaptive walk
    assert ws(1, 1, 4, 4, 64, 64, 3, 65, lisa.LISA_BF16) == 0        # hidden too wide
    assert ws(1, 1, 4, 4, 64, 64, 3, 0, lisa.LISA_BF16) == 0
    # the adaptive weights' own buffers include the bf16 operand images of the
    # tensor path: per slice and walk length U_k as hi + lo rows and alpha U_k^T
    # (72-wide rows), and W1 as hi + lo rows (136 wide)
    S, T, hidden, n = 8 * 3, 3, 32, 24 * 24
    images = S * (T - 1) * (2 * 64 * 72 + 64 * 72) * 2 + 2 * 64 * 136 * 2
    per_token = S * n * 4 * (2 * T + 2 * hidden + 2 * 64)   # w, dz, h, da and the MLP's share of dq, dk
    extra = ws(8, 3, 24, 24, 64, 64, T, hidden, lisa.LISA_BF16) - lisa.lisa_backward_workspace_bytes(
        8, 3, 24, 24, 64, 64, T, lisa.LISA_BF16)
    assert extra >= images + per_token


def test_backward_mlp_rejects_before_launch():
    assert _bwd_mlp(wbytes=1024) == lisa.LISA_ERR_WORKSPACE
    assert _bwd_mlp(mg=None) == lisa.LISA_ERR_INVALID_ARG
    assert _bwd_mlp(mg=lisa.lisa_mlp_grads(FAKE, 0, FAKE, FAKE)) == lisa.LISA_ERR_INVALID_ARG
    assert _bwd_mlp(T=9) == lisa.LISA_ERR_UNSUPPORTED
    assert _bwd_mlp(hidden=65) == lisa.LISA_ERR_UNSUPPORTED
    assert _bwd_mlp(hidden=0) == lisa.LISA_ERR_INVALID_ARG
    assert _bwd_mlp(dO=0) == lisa.LISA_ERR_INVALID_ARG
    assert _bwd_mlp(eps=0.0) == lisa.LISA_ERR_INVALID_ARG
    geo, _ = lisa.make_weights(3, beta=0.5)
    assert _bwd_mlp(wt=geo) == lisa.LISA_ERR_INVALID_ARG         # adaptive weights only


def test_untruncated_walk_runs_the_T2_chain():
    """T = 0 (untruncated) runs the kernels of a T = 2 fixed-weight walk."""
    for args in ((32, 1, 56, 56, 64), (1, 4, 128, 128, 64), (2, 2, 11, 13, 16)):
        for dt in (lisa.LISA_BF16, lisa.LISA_F32):
            wt, _ = lisa.make_weights(1, beta=0.5)
            n0 = lisa.lisa_num_stages(*args, 0, dt, wt)
            assert n0 == lisa.lisa_num_stages(*args, 2, dt, wt) > 0
            assert [lisa.lisa_stage_name(*args, 0, dt, wt, i) for i in range(n0)] == \
                [lisa.lisa_stage_name(*args, 2, dt, wt, i) for i in range(n0)]
            assert lisa.lisa_workspace_bytes(*args[:4], args[4], args[4], 0, dt) == \
                lisa.lisa_workspace_bytes(*args[:4], args[4], args[4], 2, dt)


def test_backward_workspaces_and_version():
    assert lisa.lisa_abi_version() >= 102
    for B, heads, H, W, d in ((32, 1, 56, 56, 64), (2, 3, 9, 11, 16)):
        plain = lisa.lisa_backward_workspace_bytes(B, heads, H, W, d, d, 3, lisa.LISA_BF16)
        for hidden in (1, 32, 64):
            assert lisa.lisa_backward_mlp_workspace_bytes(B, heads, H, W, d, d, 3, hidden, lisa.LISA_BF16) > plain
        assert lisa.lisa_backward_mlp_workspace_bytes(B, heads, H, W, d, d, 5, 32, lisa.LISA_BF16) > \
            lisa.lisa_backward_mlp_workspace_bytes(B, heads, H, W, d, d, 3, 32, lisa.LISA_BF16)


def test_elu_feature_map_host_side():
    """relu_inputs = 2 (ELU + 1) runs the SIMT chain for every dtype, so the
    workspace covers that chain too; the per-kernel access refuses it."""
    B, heads, H, W, d = 32, 1, 56, 56, 64
    wt, _ = lisa.make_weights(3, beta=0.5)
    need = lisa.lisa_workspace_bytes(B, heads, H, W, d, d, 3, lisa.LISA_BF16)
    assert need >= lisa.lisa_workspace_bytes(B, heads, H, W, d, d, 3, lisa.LISA_F32)
    lib = lisa.load()
    rc = lib.lisa_forward_stage(0, FAKE, FAKE + 4096, FAKE + 8192, FAKE + 12288, 1, 1, 4, 4, 16, 16, 3,
                                ctypes.byref(wt), FAKE + 16384, 1e-6, 2, lisa.LISA_F32, FAKE + 32768, 1 << 30, None)
    assert rc == lisa.LISA_ERR_INVALID_ARG
    assert lisa.feature_map_code("elu1") == 2 and lisa.feature_map_code(True) == 1
    with pytest.raises(ValueError):
        lisa.feature_map_code("elu")


def test_status_query_and_wait_selftest_reject_before_any_cuda_call():
    """lisa_query_status and the bounded-wait self-test check their arguments
    on the host: a null or misaligned workspace, a negative limit or a
    workspace too small for the error word return LISA_ERR_INVALID_ARG."""
    assert lisa.lisa_query_status(None, None) == lisa.LISA_ERR_INVALID_ARG
    assert lisa.lisa_query_status(FAKE + 4, None) == lisa.LISA_ERR_INVALID_ARG
    assert lisa.lisa_selftest_wait_timeout(-1, FAKE, 256, None) == lisa.LISA_ERR_INVALID_ARG
    assert lisa.lisa_selftest_wait_timeout(1000, None, 256, None) == lisa.LISA_ERR_INVALID_ARG
    assert lisa.lisa_selftest_wait_timeout(1000, FAKE + 8, 256, None) == lisa.LISA_ERR_INVALID_ARG
    assert lisa.lisa_selftest_wait_timeout(1000, FAKE, 2, None) == lisa.LISA_ERR_INVALID_ARG
