"""The MLP entry point that allocates nothing (tpl_tp_mlp_forward_static_ws).

It exists for callers that cannot hand the library a device workspace: a
serving loop whose HBM is all in its own pool, code that must not call
cudaMalloc (it synchronises the device and breaks a stream capture in
progress), or a host without an allocator of its own.  It runs the same
kernels as tpl_tp_mlp_forward with scratch from a static device array inside
the library, so its results must match the workspace entry point's, call
after call: the array keeps the previous call's contents, and nothing in it
may leak into the next result.

This file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

import synthetic_inputs as si
from tests.helpers import BF16_REL, assert_close, to_np

pytestmark = pytest.mark.gpu
tpl = pytest.importorskip("mlp_megatron_tp_layer_b300")


@pytest.fixture(autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    torch.cuda.synchronize()
    assert tpl.device_status() == 0


def _call_static(X, Wg, Wu, Wd, tp, Y, P):
    """One call straight through the C ABI; returns the status code."""
    B, D = X.shape
    F = Wg.shape[0]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return tpl.lib.tpl_tp_mlp_forward_static_ws(ptr(X), ptr(Wg), ptr(Wu), ptr(Wd), ptr(Y), ptr(P), B, D, F, tp,
                                                tpl.BF16, tpl.F32 if Y.dtype == torch.float32 else tpl.BF16, stream)


# Qwen2.5-1.5B-shaped MLP at decode batch sizes: B = 1 runs the CUDA-core
# kernel with split-K partials in the scratch, B = 8 and 32 the swapped
# tensor-core GEMM with its split partials, B = 200 the tensor-core GEMM with H
# in scratch.
@pytest.mark.parametrize("B", [1, 8, 32, 200])
def test_static_scratch_matches_workspace_entry_point(B):
    D, F, tp = 1536, 8960, 2
    Wg = si.normal((F, D), 0.02, 11, "na.Wg", device="cuda")
    Wu = si.normal((F, D), 0.02, 11, "na.Wu", device="cuda")
    Wd = si.normal((D, F), 0.02, 11, "na.Wd", device="cuda")
    for call in range(2):   # two calls in a row, different inputs
        X = si.normal((B, D), 1.0, 100 + call, "na.X", device="cuda")
        ref32, ref_p = tpl.tp_mlp_forward(X, Wg, Wu, Wd, tp, out_dtype=torch.float32, partials=True)
        ref_b = tpl.tp_mlp_forward(X, Wg, Wu, Wd, tp)
        Y32 = torch.full((B, D), float("nan"), dtype=torch.float32, device="cuda")
        P = torch.full((tp, B, D), float("nan"), dtype=torch.float32, device="cuda")
        assert _call_static(X, Wg, Wu, Wd, tp, Y32, P) == 0
        Yb = torch.full((B, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _call_static(X, Wg, Wu, Wd, tp, Yb, None) == 0
        torch.cuda.synchronize()
        r = to_np(ref32)
        assert_close(Y32, r, rel=BF16_REL, what=f"call {call}: Y fp32")
        for s in range(tp):
            assert_close(P[s], to_np(ref_p[s]), rel=BF16_REL, what=f"call {call}: P_{s}")
        assert_close(Yb, to_np(ref_b), rel=BF16_REL, bf16_out=True, what=f"call {call}: Y bf16")


def test_static_scratch_llama_shaped_mlp_at_its_largest_batch():
    """The Llama-3.1-70B-shaped MLP (D 8192, F 28672, tp 8) at B = 32, the
    largest decode batch whose scratch fits the static array, against the
    workspace entry point, two calls in a row."""
    B, D, F, tp = 32, 8192, 28672, 8
    assert tpl.mlp_workspace_bytes(B, D, F, tp) <= tpl.STATIC_WS_BYTES
    Wg = si.normal((F, D), 0.02, 12, "na.Wg70", device="cuda")
    Wu = si.normal((F, D), 0.02, 12, "na.Wu70", device="cuda")
    Wd = si.normal((D, F), 0.02, 12, "na.Wd70", device="cuda")
    for call in range(2):
        X = si.normal((B, D), 1.0, 200 + call, "na.X70", device="cuda")
        ref32, ref_p = tpl.tp_mlp_forward(X, Wg, Wu, Wd, tp, out_dtype=torch.float32, partials=True)
        Y32 = torch.full((B, D), float("nan"), dtype=torch.float32, device="cuda")
        P = torch.full((tp, B, D), float("nan"), dtype=torch.float32, device="cuda")
        assert _call_static(X, Wg, Wu, Wd, tp, Y32, P) == 0
        torch.cuda.synchronize()
        assert_close(Y32, to_np(ref32), rel=BF16_REL, what=f"call {call}: Y fp32")
        for s in (0, tp - 1):
            assert_close(P[s], to_np(ref_p[s]), rel=BF16_REL, what=f"call {call}: P_{s}")
    del Wg, Wu, Wd
    torch.cuda.empty_cache()


def test_static_scratch_rejects_problems_beyond_its_size():
    # Llama-3.1-70B-shaped prefill MLP: 352 MiB of workspace > 32 MiB
    B, D, F, tp = 4096, 8192, 28672, 8
    need = tpl.mlp_workspace_bytes(B, D, F, tp)
    assert need > tpl.STATIC_WS_BYTES
    X = torch.zeros((B, D), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((16, 16), dtype=torch.bfloat16, device="cuda")   # never read: rejected before launch
    Y = torch.zeros((B, D), dtype=torch.bfloat16, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = tpl.lib.tpl_tp_mlp_forward_static_ws(ctypes.c_void_p(X.data_ptr()), ctypes.c_void_p(W.data_ptr()),
                                              ctypes.c_void_p(W.data_ptr()), ctypes.c_void_p(W.data_ptr()),
                                              ctypes.c_void_p(Y.data_ptr()), None, B, D, F, tp, tpl.BF16, tpl.BF16,
                                              stream)
    assert tpl.STATUS[st] == "TPL_ERR_STATIC_LIMIT"
    assert "static" in tpl.lib.tpl_status_string(st).decode()
    assert not Y.any()
