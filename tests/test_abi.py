"""Host-side checks of the C-ABI library that need no GPU: it loads, exports
every function include/tpl.h declares, and rejects bad arguments with the
documented status codes before touching any device."""
import ctypes

import pytest

tpl = pytest.importorskip("mlp_megatron_tp_layer_b300")
lib = tpl.lib
NULL = None


def test_every_declared_symbol_is_exported():
    names = tpl.header_functions()
    assert len(names) >= 24
    missing = [n for n in names if not hasattr(lib, n)]
    assert missing == []


def test_binding_declares_every_header_function_with_its_arity():
    """The ctypes table covers the whole header, argument count for argument
    count, so no call goes through ctypes' default int conversion."""
    import re
    text = open(tpl.HEADER).read()
    for name in tpl.header_functions():
        assert name in tpl._SIGS, name
        m = re.search(r"\b%s\s*\(([^;]*?)\)\s*;" % name, text, re.S)
        assert m, name
        params = m.group(1).strip()
        n = 0 if params in ("", "void") else params.count(",") + 1
        assert len(tpl._SIGS[name][1]) == n, (name, n, len(tpl._SIGS[name][1]))


def test_status_strings_and_version():
    for code in range(10):
        assert lib.tpl_status_string(code)
    assert lib.tpl_status_string(12345) == b"unknown status"
    assert lib.tpl_version() >> 16 == 1


def _ws(fn, *args):
    n = ctypes.c_size_t(0)
    st = fn(*args, ctypes.byref(n))
    return st, n.value


def test_workspace_queries_and_shape_errors():
    st, n = _ws(lib.tpl_tp_mlp_forward_workspace, 64, 1536, 8960, 2, tpl.BF16)
    assert st == 0 and n >= 64 * 8960 * 2
    assert _ws(lib.tpl_tp_mlp_forward_workspace, 64, 1536, 8960, 3, tpl.BF16)[0] == 2      # F % tp
    assert _ws(lib.tpl_tp_mlp_forward_workspace, 0, 1536, 8960, 2, tpl.BF16)[0] == 2       # B <= 0
    assert _ws(lib.tpl_tp_mlp_forward_workspace, 4, 1532, 8960, 2, tpl.BF16)[0] == 3       # D row not 16 B
    assert _ws(lib.tpl_tp_mlp_forward_workspace, 4, 1536, 8960, 2, 7)[0] == 4              # dtype
    assert lib.tpl_tp_mlp_forward_workspace(4, 1536, 8960, 2, 1, None) == 1                # null out
    st, n = _ws(lib.tpl_tp_attn_proj_workspace, 8, 1536, 12, 2, 128, 2, tpl.BF16)
    assert st == 0 and n > 0
    assert _ws(lib.tpl_tp_attn_proj_workspace, 8, 1536, 12, 2, 128, 5, tpl.BF16)[0] == 2   # n_q % tp
    assert _ws(lib.tpl_tp_attn_proj_workspace, 8, 1536, 12, 4, 128, 6, tpl.BF16)[0] == 2   # tp > n_kv, tp % n_kv
    assert _ws(lib.tpl_tp_attn_proj_workspace, 8, 1536, 12, 2, 128, 4, tpl.BF16)[0] == 0   # replicated KV ok
    assert _ws(lib.tpl_sharded_matmul_workspace, 3, 0, 512, 8192, 28672, 8, tpl.BF16)[0] == 0
    assert _ws(lib.tpl_sharded_matmul_workspace, 1, 0, 500, 8192, 28672, 8, tpl.BF16)[0] == 2   # I % X case 1
    assert _ws(lib.tpl_sharded_matmul_workspace, 3, 0, 500, 8192, 28672, 8, tpl.BF16)[0] == 0   # I free in case 3
    assert _ws(lib.tpl_sharded_matmul_workspace, 5, 0, 512, 8192, 28672, 8, tpl.BF16)[0] == 6   # no case 5
    assert _ws(lib.tpl_tp_decoder_workspace, 8, 8192, 28672, 64, 8, 128, 8)[0] == 0


def test_calls_reject_null_and_misaligned_pointers_without_launching():
    s = ctypes.c_void_p(0)
    good = ctypes.c_void_p(1 << 20)
    bad = ctypes.c_void_p((1 << 20) + 8)
    # null pointers
    assert lib.tpl_shard_reduce(NULL, good, 4, 8, 2, 0, 1, s) == 1
    assert lib.tpl_tp_mlp_forward(good, good, NULL, good, good, NULL, 8, 256, 1024, 2, 1, 1, good, 1 << 30, s) == 1
    assert lib.tpl_tp_attn_proj(NULL, good, good, NULL, good, NULL, 8, 256, 4, 2, 64, 2, 1, 1, good, 1 << 30, s) == 1
    assert lib.tpl_sharded_matmul(1, 0, 0, good, NULL, good, NULL, 8, 64, 64, 2, 1, 1, good, 1 << 30, s) == 1
    # misaligned pointers
    assert lib.tpl_shard_reduce(bad, good, 4, 8, 2, 0, 1, s) == 3
    assert lib.tpl_tp_mlp_forward(good, good, good, bad, ctypes.c_void_p(2 << 20), NULL, 8, 256, 1024, 2, 1, 1,
                                  ctypes.c_void_p(3 << 20), 1 << 30, s) == 3
    # bad dtype combination: fp32 inputs with a bf16 output
    assert lib.tpl_tp_mlp_forward(good, good, good, good, good, NULL, 8, 256, 1024, 2, 0, 1, good, 1 << 30, s) == 4
    # shape errors come before anything else that needs a device
    assert lib.tpl_shard_reduce(good, ctypes.c_void_p(2 << 20), 4, 9, 2, 1, 1, s) == 2   # RS needs cols % tp
    assert lib.tpl_shard_reduce(good, ctypes.c_void_p(2 << 20), 4, 8, 2, 9, 1, s) == 6   # bad mode


def test_overlapping_output_is_rejected():
    s = ctypes.c_void_p(0)
    base = 1 << 24
    # Y overlaps X
    st = lib.tpl_tp_mlp_forward(ctypes.c_void_p(base), ctypes.c_void_p(2 * base), ctypes.c_void_p(3 * base),
                                ctypes.c_void_p(4 * base), ctypes.c_void_p(base + 256), None, 8, 256, 1024, 2, 1,
                                1, ctypes.c_void_p(5 * base), 1 << 30, s)
    assert st == 9
    # workspace too small
    st = lib.tpl_tp_mlp_forward(ctypes.c_void_p(base), ctypes.c_void_p(2 * base), ctypes.c_void_p(3 * base),
                                ctypes.c_void_p(4 * base), ctypes.c_void_p(6 * base), None, 8, 256, 1024, 2, 1,
                                1, ctypes.c_void_p(5 * base), 16, s)
    assert st == 5


def test_decoder_stack_rejects_bad_path_and_block_before_any_launch():
    """Path / block checks run before anything touches a device: the parallel
    block exists only on the fused implementation."""
    one = (ctypes.c_void_p * 1)(16)
    fake = ctypes.c_void_p(256)
    args = [fake, fake, one, one, one, one, one, 1, 8, 1536, 8960, 12, 2, 128, 2, fake, 1 << 30]
    unsupported = 6
    assert lib.tpl_tp_decoder_stack_ex(*args, tpl.PATH_UNFUSED, tpl.BLOCK_PARALLEL, None) == unsupported
    assert lib.tpl_tp_decoder_stack_ex(*args, 7, tpl.BLOCK_SERIAL, None) == unsupported
    assert lib.tpl_tp_decoder_stack_ex(*args, tpl.PATH_AUTO, 5, None) == unsupported
    assert lib.tpl_tp_decoder_stack_path(*args, 9, None) == unsupported


def test_vocab_topk_rejects_bad_arguments_before_any_launch():
    s = ctypes.c_void_p(0)
    x, w, ws = ctypes.c_void_p(1 << 24), ctypes.c_void_p(2 << 24), ctypes.c_void_p(3 << 24)
    idx, val = ctypes.c_void_p(4 << 24), ctypes.c_void_p(5 << 24)
    big = 1 << 30

    def call(*, x=x, w=w, B=4, D=256, V=1000, tp=4, k=2, dtype=tpl.BF16, idx=idx, val=val, sidx=None, sval=None,
             ws=ws, nbytes=big):
        return lib.tpl_vocab_parallel_topk(x, w, B, D, V, tp, k, dtype, idx, val, sidx, sval, ws, nbytes, s)

    st, n = _ws(lib.tpl_vocab_parallel_topk_workspace, 4, 1000, 4, 2)
    assert st == 0 and n > 0
    assert _ws(lib.tpl_vocab_parallel_topk_workspace, 4, 1000, 3, 2)[0] == 2     # V % tp
    assert _ws(lib.tpl_vocab_parallel_topk_workspace, 4, 1000, 4, 9)[0] == 2     # k > 8
    assert _ws(lib.tpl_vocab_parallel_topk_workspace, 4, 16, 4, 5)[0] == 2       # k > V / tp
    assert _ws(lib.tpl_vocab_parallel_topk_workspace, 0, 1000, 4, 1)[0] == 2     # no tokens
    assert call(x=None) == 1 and call(idx=None) == 1
    assert call(D=100) == 2                                   # D % 8
    assert call(dtype=tpl.F32) == 4
    assert call(x=ctypes.c_void_p((1 << 24) + 8)) == 3       # X not 16-byte aligned
    assert call(val=ctypes.c_void_p((5 << 24) + 2)) == 3     # output not 4-byte aligned
    assert call(nbytes=16) == 5 and call(ws=None) == 5
    assert call(idx=ctypes.c_void_p((1 << 24) + 64)) == 9    # top_idx inside X
    assert call(val=ctypes.c_void_p((4 << 24) + 16)) == 9    # top_val overlaps top_idx
    assert call(sidx=ctypes.c_void_p((3 << 24) + 256)) == 9  # shard output inside the workspace


def test_int8_binding_checks_code_and_scale_shapes_before_calling():
    """Scales are read by index from the shapes the call implies, so the binding
    refuses mismatched arrays before anything reaches the library (CPU tensors
    suffice: nothing is launched)."""
    import torch
    B, D, F, tp = 2, 64, 128, 2
    x = torch.zeros(B, D, dtype=torch.bfloat16)
    q = lambda r, c: torch.zeros(r, c, dtype=torch.int8)  # noqa: E731
    f = lambda *s: torch.zeros(*s, dtype=torch.float32)  # noqa: E731
    good = (q(F, D), f(F, 1), q(F, D), f(F, 1), q(D, F), f(D, tp))
    with pytest.raises(ValueError):
        tpl.tp_mlp_forward_w8(x, *good[:5], f(D, 1), tp)           # down scales for one group, not tp
    with pytest.raises(ValueError):
        tpl.tp_mlp_forward_w8(x, q(F, D + 64), *good[1:], tp)      # codes wider than X
    with pytest.raises(TypeError):
        tpl.tp_mlp_forward_w8(x, good[0].float(), *good[1:], tp)   # codes not int8


def test_lm_head_binding_checks_given_outputs():
    import torch
    x = torch.zeros(3, 64, dtype=torch.bfloat16)
    W = torch.zeros(256, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        tpl.vocab_parallel_topk(x, W, 2, 2, out=(torch.zeros(3, 1, dtype=torch.int32), torch.zeros(3, 1)))
    with pytest.raises(ValueError):
        tpl.vocab_parallel_topk(x, W, 2, 2, out=(torch.zeros(3, 2), torch.zeros(3, 2)))


# ------------------------------------------------ binding argument checks
# The library reads and writes as much as the sizes imply, so the wrappers
# reject any tensor of another shape or type before the call.  These checks
# run before any device is touched, so CPU tensors suffice.

def _t(*shape, dtype=None):
    import torch
    return torch.zeros(shape, dtype=dtype or torch.bfloat16)


def _mlp(B=4, D=64, F=128):
    return _t(B, D), _t(F, D), _t(F, D), _t(D, F)


def test_mlp_wrappers_reject_wrong_weight_shapes_and_types():
    import torch
    for fn in (tpl.tp_mlp_forward, tpl.tp_mlp_forward_static_ws):
        X, Wg, Wu, Wd = _mlp()
        with pytest.raises(ValueError, match="Wd"):
            fn(X, Wg, Wu, _t(128, 64), 2)                      # Wd transposed
        with pytest.raises(ValueError, match="Wu"):
            fn(X, Wg, _t(128, 32), Wd, 2)
        with pytest.raises(TypeError, match="Wg"):
            fn(X, Wg.float(), Wu, Wd, 2)                       # fp32 weights, bf16 X
        with pytest.raises(ValueError, match="contiguous"):
            fn(X, Wg, _t(64, 128).t(), Wd, 2)


def test_mlp_wrappers_reject_wrong_outputs():
    import torch
    for fn in (tpl.tp_mlp_forward, tpl.tp_mlp_forward_static_ws):
        X, Wg, Wu, Wd = _mlp()
        with pytest.raises(ValueError, match="out"):
            fn(X, Wg, Wu, Wd, 2, out=_t(2, 64))                # smaller than [B, D]
        with pytest.raises(ValueError, match="partials"):
            fn(X, Wg, Wu, Wd, 2, partials=_t(2, 4, 32, dtype=torch.float32))
        with pytest.raises(TypeError, match="partials"):
            fn(X, Wg, Wu, Wd, 2, partials=_t(2, 4, 64))        # bf16 partials
        with pytest.raises(ValueError, match="CUDA"):
            fn(X, Wg, Wu, Wd, 2)                               # host tensors


def test_attn_case_and_decoder_wrappers_reject_wrong_shapes():
    import torch
    X = _t(4, 256)
    with pytest.raises(ValueError, match="Wo"):
        tpl.tp_attn_proj(X, _t(512, 256), _t(256, 128), 4, 2, 64, 2)        # Wo must be [256, 256]
    with pytest.raises(ValueError, match="Wqkv"):
        tpl.tp_attn_proj(X, _t(256, 256), _t(256, 256), 4, 2, 64, 2)       # Wqkv must be [512, 256]
    with pytest.raises(ValueError, match="qkv_out"):
        tpl.tp_attn_proj(X, _t(512, 256), _t(256, 256), 4, 2, 64, 2, qkv_out=_t(2, 4, 128))
    with pytest.raises(TypeError, match="Bt"):
        tpl.sharded_matmul(1, _t(16, 64), _t(32, 64, dtype=torch.float32), 2)
    with pytest.raises(ValueError, match="out"):
        tpl.sharded_matmul(3, _t(16, 64), _t(32, 64), 2, mode=tpl.REDUCE_SCATTER, out=_t(16, 32))
    W = {"Wqkv": _t(512, 256), "Wo": _t(256, 256), "Wg": _t(512, 256), "Wu": _t(512, 256), "Wd": _t(256, 512)}
    bad = dict(W, Wd=_t(512, 256))
    with pytest.raises(ValueError, match="Wd"):
        tpl.tp_decoder_stack(X, [W, bad], 4, 2, 64, 2)
    with pytest.raises(ValueError, match="out"):
        tpl.tp_decoder_layer(X, W, 4, 2, 64, 2, out=_t(4, 128))


def test_static_scratch_limit_uses_the_calls_own_plan_and_dtype_comes_first():
    """tpl_tp_mlp_forward_static_ws: the Llama-3.1-70B-shaped MLP (D 8192,
    F 28672, tp 8) fits the static scratch up to B = 32 and not at B = 64;
    the size check runs before any device is touched, after the dtype check."""
    s = ctypes.c_void_p(0)
    p = [ctypes.c_void_p((i + 1) << 24) for i in range(6)]
    D, F, tp = 8192, 28672, 8
    # without partials, then with: both plans exceed 32 MiB at B = 64
    for part in (NULL, p[5]):
        st = lib.tpl_tp_mlp_forward_static_ws(p[0], p[1], p[2], p[3], p[4], part, 64, D, F, tp, tpl.BF16,
                                              tpl.BF16, s)
        assert tpl.STATUS[st] == "TPL_ERR_STATIC_LIMIT"
    # an output type tp_mlp_forward rejects is reported as such, not as a size problem
    st = lib.tpl_tp_mlp_forward_static_ws(p[0], p[1], p[2], p[3], p[4], NULL, 64, D, F, tp, tpl.F32, tpl.BF16, s)
    assert tpl.STATUS[st] == "TPL_ERR_DTYPE"
    # the plan for the call's own partials argument decides, not the larger of the two
    assert lib.tpl_tp_mlp_forward_workspace(32, D, F, tp, tpl.BF16, ctypes.byref(ctypes.c_size_t())) == 0
    n = ctypes.c_size_t(0)
    lib.tpl_tp_mlp_forward_workspace(32, D, F, tp, tpl.BF16, ctypes.byref(n))
    assert n.value <= tpl.STATIC_WS_BYTES


def test_fused_fault_hook_checks_its_arguments():
    assert lib.tpl_test_fused_fault(-1, 1, 0) == 0                       # defaults
    assert tpl.STATUS[lib.tpl_test_fused_fault(3, 0, 0)] == "TPL_ERR_UNSUPPORTED"        # phase 0 has no units
    assert tpl.STATUS[lib.tpl_test_fused_fault(148, 1, 0)] == "TPL_ERR_UNSUPPORTED"      # beyond the grid
    assert tpl.STATUS[lib.tpl_test_fused_fault(-1, 1, 5000)] == "TPL_ERR_UNSUPPORTED"    # under 10 us
    assert tpl.STATUS[lib.tpl_test_fused_fault(-1, 1, 3_000_000_000)] == "TPL_ERR_UNSUPPORTED"
    assert lib.tpl_test_fused_fault(-1, 1, 0) == 0
