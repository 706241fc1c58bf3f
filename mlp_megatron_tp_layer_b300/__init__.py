"""Megatron tensor-parallel layer forward on one B300: Python binding.

Thin ctypes binding of ``libtpl.so`` (declared in ``include/tpl.h``): it only
checks and marshals arguments (pointers, sizes, the current CUDA stream); every
step of the computation runs in the library's CUDA kernels.  PyTorch supplies
device memory and streams.

The library must be built (``python mlp_megatron_tp_layer_b300/build.py``);
importing this package without it raises ImportError -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# TPL_LIBRARY selects another build of the same library, e.g. the instrumented
# libtpl_trace.so (build.py --trace) for phase traces.
LIB_PATH = os.environ.get("TPL_LIBRARY") or os.path.join(_HERE, "libtpl.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "tpl.h")

F32, BF16 = 0, 1
ALLREDUCE, REDUCE_SCATTER = 0, 1
GATHER_B, GATHER_A = 0, 1
PATH_AUTO, PATH_UNFUSED, PATH_FUSED = 0, 1, 2
BLOCK_SERIAL, BLOCK_PARALLEL = 0, 1
STATUS = {0: "TPL_OK", 1: "TPL_ERR_NULL", 2: "TPL_ERR_SHAPE", 3: "TPL_ERR_ALIGN", 4: "TPL_ERR_DTYPE",
          5: "TPL_ERR_WORKSPACE", 6: "TPL_ERR_UNSUPPORTED", 7: "TPL_ERR_CUDA", 8: "TPL_ERR_TIMEOUT",
          9: "TPL_ERR_ALIAS", 10: "TPL_ERR_STATIC_LIMIT"}
STATIC_WS_BYTES = 32 << 20

_vp, _i64, _i32, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
_SIGS = {
    "tpl_status_string": (ctypes.c_char_p, [_i32]),
    "tpl_version": (_i32, []),
    "tpl_device_status": (_i32, [ctypes.POINTER(ctypes.c_uint), _vp]),
    "tpl_shard_reduce": (_i32, [_vp, _vp, _i64, _i64, _i32, _i32, _i32, _vp]),
    "tpl_tp_mlp_forward_workspace": (_i32, [_i64, _i64, _i64, _i32, _i32, ctypes.POINTER(_sz)]),
    "tpl_tp_mlp_forward": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _i32, _i32,
                                  _vp, _sz, _vp]),
    "tpl_tp_mlp_forward_static_ws": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _i32, _i32,
                                            _vp]),
    "tpl_tp_attn_proj_workspace": (_i32, [_i64, _i64, _i32, _i32, _i32, _i32, _i32, ctypes.POINTER(_sz)]),
    "tpl_tp_attn_proj": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i32, _i32, _i32, _i32, _i32,
                                _i32, _vp, _sz, _vp]),
    "tpl_sharded_matmul_workspace": (_i32, [_i32, _i32, _i64, _i64, _i64, _i32, _i32, ctypes.POINTER(_sz)]),
    "tpl_sharded_matmul": (_i32, [_i32, _i32, _i32, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _i32, _i32,
                                  _vp, _sz, _vp]),
    "tpl_profile_enable": (_i32, [_i32]),
    "tpl_profile_count": (_i32, []),
    "tpl_profile_read": (_i32, [_i32, ctypes.c_char_p, _sz, ctypes.POINTER(ctypes.c_float)]),
    "tpl_test_fused_fault": (_i32, [_i32, _i32, _i64]),
    "tpl_fused_trace_read": (_i32, [_vp, _sz]),
    "tpl_tp_decoder_workspace": (_i32, [_i64, _i64, _i64, _i32, _i32, _i32, _i32, ctypes.POINTER(_sz)]),
    "tpl_tp_decoder_stack_path": (_i32, [_vp, _vp, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                         ctypes.POINTER(_vp), ctypes.POINTER(_vp), _i32, _i64, _i64, _i64, _i32,
                                         _i32, _i32, _i32, _vp, _sz, _i32, _vp]),
    "tpl_tp_decoder_stack_ex": (_i32, [_vp, _vp, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                       ctypes.POINTER(_vp), ctypes.POINTER(_vp), _i32, _i64, _i64, _i64, _i32,
                                       _i32, _i32, _i32, _vp, _sz, _i32, _i32, _vp]),
    "tpl_tp_decoder_layer": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _i32, _i32,
                                    _i32, _vp, _sz, _vp]),
    "tpl_tp_decoder_stack": (_i32, [_vp, _vp, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                    ctypes.POINTER(_vp), ctypes.POINTER(_vp), _i32, _i64, _i64, _i64, _i32,
                                    _i32, _i32, _i32, _vp, _sz, _vp]),
    "tpl_quantize_w8": (_i32, [_vp, _i64, _i64, _i32, _vp, _vp, _vp]),
    "tpl_tp_mlp_forward_w8_workspace": (_i32, [_i64, _i64, _i64, _i32, ctypes.POINTER(_sz)]),
    "tpl_tp_mlp_forward_w8": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _i32,
                                     _vp, _sz, _vp]),
    "tpl_vocab_parallel_topk_workspace": (_i32, [_i64, _i64, _i32, _i32, ctypes.POINTER(_sz)]),
    "tpl_vocab_parallel_topk": (_i32, [_vp, _vp, _i64, _i64, _i64, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp,
                                       _sz, _vp]),
}


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python mlp_megatron_tp_layer_b300/build.py`")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def header_functions() -> list[str]:
    """Names of the functions include/tpl.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+char\*|tpl_status|int)\s+(tpl_\w+)\s*\(", text, re.M)))


class TplError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = lib.tpl_status_string(status).decode()
        super().__init__(f"{what}: {STATUS.get(status, status)} ({msg})")


def _check(status: int, what: str):
    if status != 0:
        raise TplError(status, what)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _tdt(code: int):
    return torch.bfloat16 if code == BF16 else torch.float32


def _out_code(dt: int, out, out_dtype) -> int:
    """Output element type: the given out tensor's, else out_dtype, else the input's."""
    if out is not None:
        code = _dt(out)
        if out_dtype is not None and _dt(torch.empty(0, dtype=out_dtype)) != code:
            raise ValueError("out and out_dtype disagree")
        return code
    return dt if out_dtype is None else _dt(torch.empty(0, dtype=out_dtype))


def _contig(*ts):
    for t in ts:
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors must be contiguous (row-major)")


def _need(t, shape, dtype, what: str):
    """The library reads or writes exactly shape x dtype at t's address: reject
    a tensor of another shape or type, or not contiguous, before the call (a
    wrong size would become an out-of-bounds device access)."""
    if t is None:
        return
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{what} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{what} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous (row-major)")


def _same_device(ref, *ts):
    """Every tensor the call passes lives in ref's CUDA device memory."""
    if not ref.is_cuda:
        raise ValueError("tensors must be CUDA tensors")
    for t in ts:
        if t is not None and t.device != ref.device:
            raise ValueError(f"every tensor must be on {ref.device}, got one on {t.device}")


def _mlp_args(X, Wg, Wu, Wd, tp, out, partials, out_dtype):
    """Shape, type and device checks shared by the bf16/fp32 MLP wrappers;
    returns (B, D, F, dt, odt, out, partials, want_partials)."""
    _contig(X)
    if X.dim() != 2 or Wg.dim() != 2:
        raise ValueError("X must be [B, D] and Wg [F, D]")
    B, D = X.shape
    F = Wg.shape[0]
    dt = _dt(X)
    for t, shape, name in ((Wg, (F, D), "Wg"), (Wu, (F, D), "Wu"), (Wd, (D, F), "Wd")):
        _need(t, shape, X.dtype, name)
    odt = _out_code(dt, out, out_dtype)
    if out is None:
        out = torch.empty((B, D), dtype=_tdt(odt), device=X.device)
    _need(out, (B, D), _tdt(odt), "out")
    want = partials is not None and partials is not False
    if partials is True:
        partials = torch.empty((tp, B, D), dtype=torch.float32, device=X.device)
    elif not want:
        partials = None
    _need(partials, (tp, B, D), torch.float32, "partials")
    _same_device(X, Wg, Wu, Wd, out, partials)
    return B, D, F, dt, odt, out, partials, want


_ws_cache: dict = {}


def workspace(nbytes: int, device) -> torch.Tensor:
    """A cached scratch buffer of at least nbytes on device (grown on demand)."""
    dev = torch.device(device)
    key = (dev.type, dev.index)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
        _ws_cache[key] = buf
    return buf


def device_status(stream=None) -> int:
    """Synchronise and return (and clear) the device error word."""
    flags = ctypes.c_uint(0)
    st = lib.tpl_device_status(ctypes.byref(flags), _stream(stream))
    if st not in (0, 8):
        raise TplError(st, "tpl_device_status")
    return flags.value


# ------------------------------------------------------------------- calls

def shard_reduce(partials: torch.Tensor, mode: int = ALLREDUCE, out_dtype=torch.bfloat16, out=None, stream=None):
    """Sum fp32 partials [tp, rows, cols] over shards in ascending order."""
    _contig(partials)
    tp, rows, cols = partials.shape
    if out is None:
        shape = (rows, cols) if mode == ALLREDUCE else (tp, rows, cols // tp)
        out = torch.empty(shape, dtype=out_dtype, device=partials.device)
    _contig(out)
    _check(lib.tpl_shard_reduce(_p(partials), _p(out), rows, cols, tp, mode, _dt(out), _stream(stream)),
           "tpl_shard_reduce")
    return out


def mlp_workspace_bytes(B, D, F, tp, dtype=BF16) -> int:
    n = ctypes.c_size_t(0)
    _check(lib.tpl_tp_mlp_forward_workspace(B, D, F, tp, dtype, ctypes.byref(n)), "tpl_tp_mlp_forward_workspace")
    return n.value


def tp_mlp_forward(X, Wg, Wu, Wd, tp: int, out=None, partials=None, out_dtype=None, ws=None, stream=None):
    """Y = sum_s (silu(X Wg_s^T) * (X Wu_s^T)) Wd_s^T over tp logical shards.

    ``partials``: None (reduction fused), True (allocate) or an fp32 [tp, B, D] tensor.
    Returns Y, or (Y, partials) when partials were requested.
    """
    B, D, F, dt, odt, out, partials, want = _mlp_args(X, Wg, Wu, Wd, tp, out, partials, out_dtype)
    nbytes = mlp_workspace_bytes(B, D, F, tp, dt)
    ws = workspace(nbytes, X.device) if ws is None else ws
    _check(lib.tpl_tp_mlp_forward(_p(X), _p(Wg), _p(Wu), _p(Wd), _p(out), _p(partials), B, D, F, tp, dt, odt,
                                  _p(ws), ws.numel() * ws.element_size(), _stream(stream)), "tpl_tp_mlp_forward")
    return (out, partials) if want else out


def tp_mlp_forward_static_ws(X, Wg, Wu, Wd, tp: int, out=None, partials=None, out_dtype=None, stream=None):
    """tp_mlp_forward with the library's static device scratch instead of a
    workspace: for callers that cannot allocate device memory (see
    tpl_tp_mlp_forward_static_ws in include/tpl.h for the limit and sharing).
    The call is made with X's device current, since the scratch array the
    library picks is the current device's."""
    B, D, F, dt, odt, out, partials, want = _mlp_args(X, Wg, Wu, Wd, tp, out, partials, out_dtype)
    with torch.cuda.device(X.device):
        _check(lib.tpl_tp_mlp_forward_static_ws(_p(X), _p(Wg), _p(Wu), _p(Wd), _p(out), _p(partials), B, D, F, tp,
                                                dt, odt, _stream(stream)), "tpl_tp_mlp_forward_static_ws")
    return (out, partials) if want else out


def attn_workspace_bytes(B, D, n_q, n_kv, head_dim, tp, dtype=BF16) -> int:
    n = ctypes.c_size_t(0)
    _check(lib.tpl_tp_attn_proj_workspace(B, D, n_q, n_kv, head_dim, tp, dtype, ctypes.byref(n)),
           "tpl_tp_attn_proj_workspace")
    return n.value


def qkv_shard_width(n_q, n_kv, head_dim, tp) -> int:
    kv_s = n_kv // tp if tp <= n_kv else 1
    return (n_q // tp + 2 * kv_s) * head_dim


def tp_attn_proj(X, Wqkv, Wo, n_q, n_kv, head_dim, tp, out=None, qkv_out=None, partials=None, out_dtype=None,
                 ws=None, stream=None):
    """Head-partitioned QKV projection, context-1 attention stand-in, row-parallel o_proj.

    ``qkv_out``: None, True (allocate [tp, B, W_s]) or a tensor.  ``partials`` as in
    tp_mlp_forward.  Returns Y, plus qkv_out / partials when requested (in that order).
    """
    _contig(X)
    B, D = X.shape
    dt = _dt(X)
    _need(Wqkv, ((n_q + 2 * n_kv) * head_dim, D), X.dtype, "Wqkv")
    _need(Wo, (D, n_q * head_dim), X.dtype, "Wo")
    odt = _out_code(dt, out, out_dtype)
    if out is None:
        out = torch.empty((B, D), dtype=_tdt(odt), device=X.device)
    _need(out, (B, D), _tdt(odt), "out")
    want_qkv = qkv_out is not None and qkv_out is not False
    if qkv_out is True:
        qkv_out = torch.empty((tp, B, qkv_shard_width(n_q, n_kv, head_dim, tp)), dtype=X.dtype, device=X.device)
    elif not want_qkv:
        qkv_out = None
    if qkv_out is not None and tp > 0 and n_q % tp == 0:
        _need(qkv_out, (tp, B, qkv_shard_width(n_q, n_kv, head_dim, tp)), X.dtype, "qkv_out")
    want_p = partials is not None and partials is not False
    if partials is True:
        partials = torch.empty((tp, B, D), dtype=torch.float32, device=X.device)
    elif not want_p:
        partials = None
    _need(partials, (tp, B, D), torch.float32, "partials")
    _same_device(X, Wqkv, Wo, out, qkv_out, partials)
    nbytes = attn_workspace_bytes(B, D, n_q, n_kv, head_dim, tp, dt)
    ws = workspace(nbytes, X.device) if ws is None else ws
    _check(lib.tpl_tp_attn_proj(_p(X), _p(Wqkv), _p(Wo), _p(qkv_out), _p(out), _p(partials), B, D, n_q, n_kv,
                                head_dim, tp, dt, odt, _p(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "tpl_tp_attn_proj")
    res = [out]
    if want_qkv:
        res.append(qkv_out)
    if want_p:
        res.append(partials)
    return res[0] if len(res) == 1 else tuple(res)


def case_workspace_bytes(case, mode, I, J, K, X, dtype=BF16) -> int:
    n = ctypes.c_size_t(0)
    _check(lib.tpl_sharded_matmul_workspace(case, mode, I, J, K, X, dtype, ctypes.byref(n)),
           "tpl_sharded_matmul_workspace")
    return n.value


def sharded_matmul(case: int, A, Bt, X: int, mode: int = ALLREDUCE, gather: int = GATHER_B, out=None,
                   partials=None, out_dtype=None, ws=None, stream=None):
    """C = A B (B stored as Bt[K, J]) in one of the four sharding cases over X devices.

    K-sharded results (case 3 reduce-scatter, case 4 gather-A) are [X, I, K/X].
    """
    _contig(A)
    I, J = A.shape
    K = Bt.shape[0]
    dt = _dt(A)
    _need(Bt, (K, J), A.dtype, "Bt")
    odt = _out_code(dt, out, out_dtype)
    k_sharded = (case == 3 and mode == REDUCE_SCATTER) or (case == 4 and gather == GATHER_A)
    shape = (X, I, K // X) if k_sharded else (I, K)
    if out is None:
        out = torch.empty(shape, dtype=_tdt(odt), device=A.device)
    if X > 0 and K % X == 0:
        _need(out, shape, _tdt(odt), "out")
    want_p = partials is not None and partials is not False
    if partials is True:
        partials = torch.empty((X, I, K), dtype=torch.float32, device=A.device)
    elif not want_p:
        partials = None
    _need(partials, (X, I, K), torch.float32, "partials")
    _same_device(A, Bt, out, partials)
    nbytes = case_workspace_bytes(case, mode, I, J, K, X, dt)
    ws = workspace(nbytes, A.device) if ws is None else ws
    _check(lib.tpl_sharded_matmul(case, mode, gather, _p(A), _p(Bt), _p(out), _p(partials), I, J, K, X, dt, odt,
                                  _p(ws), ws.numel() * ws.element_size(), _stream(stream)), "tpl_sharded_matmul")
    return (out, partials) if want_p else out


def decoder_workspace_bytes(B, D, F, n_q, n_kv, head_dim, tp) -> int:
    n = ctypes.c_size_t(0)
    _check(lib.tpl_tp_decoder_workspace(B, D, F, n_q, n_kv, head_dim, tp, ctypes.byref(n)),
           "tpl_tp_decoder_workspace")
    return n.value


def _layer_args(W, D, F, n_q, n_kv, head_dim, dtype):
    """Every weight of one decoder layer has the shape the library reads."""
    for name, shape in (("Wqkv", ((n_q + 2 * n_kv) * head_dim, D)), ("Wo", (D, n_q * head_dim)),
                        ("Wg", (F, D)), ("Wu", (F, D)), ("Wd", (D, F))):
        _need(W[name], shape, dtype, name)


def _ptr_array(ts):
    arr = (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])
    return arr


def tp_decoder_stack(x, layers, n_q, n_kv, head_dim, tp, out=None, ws=None, stream=None, path=PATH_AUTO,
                     block=BLOCK_SERIAL):
    """Decoder layers; ``layers`` is a list of dicts with Wqkv, Wo, Wg, Wu, Wd.
    ``path``: PATH_AUTO (fused where it applies), PATH_UNFUSED or PATH_FUSED.
    ``block``: BLOCK_SERIAL (pre-norm) or BLOCK_PARALLEL (x + Attn(RMSNorm x) + MLP(RMSNorm x))."""
    _contig(x)
    B, D = x.shape
    F = layers[0]["Wg"].shape[0]
    for W in layers:
        _layer_args(W, D, F, n_q, n_kv, head_dim, x.dtype)
    if out is None:
        out = torch.empty_like(x)
    _need(out, (B, D), x.dtype, "out")
    _same_device(x, out, *[W[k] for W in layers for k in ("Wqkv", "Wo", "Wg", "Wu", "Wd")])
    nbytes = decoder_workspace_bytes(B, D, F, n_q, n_kv, head_dim, tp)
    ws = workspace(nbytes, x.device) if ws is None else ws
    arrs = [_ptr_array([L[k] for L in layers]) for k in ("Wqkv", "Wo", "Wg", "Wu", "Wd")]
    _check(lib.tpl_tp_decoder_stack_ex(_p(x), _p(out), *arrs, len(layers), B, D, F, n_q, n_kv, head_dim, tp,
                                       _p(ws), ws.numel() * ws.element_size(), path, block, _stream(stream)),
           "tpl_tp_decoder_stack_ex")
    return out


def tp_decoder_layer(x, W, n_q, n_kv, head_dim, tp, out=None, ws=None, stream=None):
    """One serial pre-norm decoder layer (see tp_decoder_stack)."""
    _contig(x)
    B, D = x.shape
    F = W["Wg"].shape[0]
    _layer_args(W, D, F, n_q, n_kv, head_dim, x.dtype)
    if out is None:
        out = torch.empty_like(x)
    _need(out, (B, D), x.dtype, "out")
    _same_device(x, out, *W.values())
    nbytes = decoder_workspace_bytes(B, D, F, n_q, n_kv, head_dim, tp)
    ws = workspace(nbytes, x.device) if ws is None else ws
    _check(lib.tpl_tp_decoder_layer(_p(x), _p(out), _p(W["Wqkv"]), _p(W["Wo"]), _p(W["Wg"]), _p(W["Wu"]),
                                    _p(W["Wd"]), B, D, F, n_q, n_kv, head_dim, tp, _p(ws),
                                    ws.numel() * ws.element_size(), _stream(stream)), "tpl_tp_decoder_layer")
    return out


def test_fused_fault(cta: int = -1, phase: int = 1, wait_limit_ns: int = 0):
    """Test hook (tpl_test_fused_fault): make CTA `cta` of the next fused-stack
    launches leave out its first ticket arrival of `phase`, with every wait
    limited to wait_limit_ns; test_fused_fault() restores the defaults."""
    _check(lib.tpl_test_fused_fault(cta, phase, wait_limit_ns), "tpl_test_fused_fault")


FUSED_TRACE_SHAPE = (148, 129, 12)    # CTAs, phases, events (see tpl_fused_trace_read)


def fused_trace():
    """Per-CTA, per-phase event stamps (ns) of the last fused-stack launch of an
    instrumented build, as an int64 array FUSED_TRACE_SHAPE (0: not reached)."""
    import numpy as np
    buf = np.zeros(FUSED_TRACE_SHAPE, dtype=np.uint64)
    _check(lib.tpl_fused_trace_read(ctypes.c_void_p(buf.ctypes.data), buf.nbytes), "tpl_fused_trace_read")
    return buf.astype(np.int64)


def profile_enable(max_launches: int = 4096):
    """Start recording per-launch device times (see tpl_profile_enable)."""
    _check(lib.tpl_profile_enable(max_launches), "tpl_profile_enable")


def profile_disable():
    _check(lib.tpl_profile_enable(0), "tpl_profile_enable")


def profile_records():
    """[(tag, ms)] for every launch recorded since profile_enable."""
    out = []
    buf = ctypes.create_string_buffer(64)
    ms = ctypes.c_float(0.0)
    for i in range(lib.tpl_profile_count()):
        _check(lib.tpl_profile_read(i, buf, 64, ctypes.byref(ms)), "tpl_profile_read")
        out.append((buf.value.decode(), float(ms.value)))
    return out


def vocab_topk_workspace_bytes(B, V, tp, k) -> int:
    n = ctypes.c_size_t(0)
    _check(lib.tpl_vocab_parallel_topk_workspace(B, V, tp, k, ctypes.byref(n)),
           "tpl_vocab_parallel_topk_workspace")
    return n.value


def vocab_parallel_topk(x, W, tp: int, k: int = 1, shard_outputs: bool = False, out=None, ws=None,
                        stream=None):
    """Top-k next-token candidates of the vocabulary-parallel lm_head.

    x [B, D] and W [V, D] bf16; shard s owns rows [s V/tp, (s+1) V/tp) of W.
    Returns (idx [B, k] int32, val [B, k] fp32); with ``shard_outputs`` also
    each shard's own top-k (sidx, sval), both [tp, B, k].  ``out`` may supply
    the (idx, val) tensors."""
    _contig(x, W)
    B, D = x.shape
    V = W.shape[0]
    if W.shape[1] != D:
        raise ValueError("W must be [V, D]")
    dev = x.device
    if out is None:
        idx = torch.empty(B, k, dtype=torch.int32, device=dev)
        val = torch.empty(B, k, dtype=torch.float32, device=dev)
    else:
        idx, val = out
        if (idx.dtype != torch.int32 or val.dtype != torch.float32 or tuple(idx.shape) != (B, k)
                or tuple(val.shape) != (B, k)):
            raise ValueError("out must be (int32 [B, k], float32 [B, k])")
        _contig(idx, val)
    sidx = sval = None
    if shard_outputs:
        sidx = torch.empty(tp, B, k, dtype=torch.int32, device=dev)
        sval = torch.empty(tp, B, k, dtype=torch.float32, device=dev)
    nbytes = vocab_topk_workspace_bytes(B, V, tp, k)
    ws = workspace(nbytes, dev) if ws is None else ws
    _check(lib.tpl_vocab_parallel_topk(_p(x), _p(W), B, D, V, tp, k, _dt(x), _p(idx), _p(val), _p(sidx), _p(sval),
                                       _p(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "tpl_vocab_parallel_topk")
    return (idx, val, sidx, sval) if shard_outputs else (idx, val)


def quantize_w8(W, groups: int = 1, stream=None):
    """Symmetric int8 codes of a bf16 matrix W [rows, cols], one float32 scale
    per row and column group: returns (Q int8 [rows, cols], scale [rows, groups])."""
    _contig(W)
    rows, cols = W.shape
    Q = torch.empty(rows, cols, dtype=torch.int8, device=W.device)
    scale = torch.empty(rows, groups, dtype=torch.float32, device=W.device)
    _check(lib.tpl_quantize_w8(_p(W), rows, cols, groups, _p(Q), _p(scale), _stream(stream)), "tpl_quantize_w8")
    return Q, scale


def mlp_w8_workspace_bytes(B, D, F, tp) -> int:
    n = ctypes.c_size_t(0)
    _check(lib.tpl_tp_mlp_forward_w8_workspace(B, D, F, tp, ctypes.byref(n)), "tpl_tp_mlp_forward_w8_workspace")
    return n.value


def tp_mlp_forward_w8(X, Qg, sg, Qu, su, Qd, sd, tp: int, out=None, partials=None, out_dtype=None, ws=None,
                      stream=None):
    """tp_mlp_forward with int8 weights (codes and scales from quantize_w8:
    groups 1 for Qg/Qu [F, D], groups tp for Qd [D, F]); X is bf16."""
    _contig(X, Qg, sg, Qu, su, Qd, sd)
    B, D = X.shape
    F = Qg.shape[0]
    # the library reads exactly these many codes and scales
    if Qg.shape != (F, D) or Qu.shape != (F, D) or Qd.shape != (D, F):
        raise ValueError("codes must be Qg, Qu [F, D] and Qd [D, F]")
    if sg.numel() != F or su.numel() != F or sd.numel() != D * tp:
        raise ValueError("scales must be sg, su [F] (one group) and sd [D, tp] (one per shard)")
    if any(t.dtype != torch.int8 for t in (Qg, Qu, Qd)) or any(t.dtype != torch.float32 for t in (sg, su, sd)):
        raise TypeError("codes are int8 and scales float32")
    odt = _out_code(BF16, out, out_dtype)
    if out is None:
        out = torch.empty(B, D, dtype=_tdt(odt), device=X.device)
    want_p = partials is True or isinstance(partials, torch.Tensor)
    if partials is True:
        partials = torch.empty(tp, B, D, dtype=torch.float32, device=X.device)
    elif not want_p:
        partials = None
    nbytes = mlp_w8_workspace_bytes(B, D, F, tp)
    ws = workspace(nbytes, X.device) if ws is None else ws
    _check(lib.tpl_tp_mlp_forward_w8(_p(X), _p(Qg), _p(sg), _p(Qu), _p(su), _p(Qd), _p(sd), _p(out), _p(partials),
                                     B, D, F, tp, odt, _p(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "tpl_tp_mlp_forward_w8")
    return (out, partials) if want_p else out
