"""Out-of-bounds guards, in place of a memory checker: every output and the
workspace of a call are views into larger device buffers whose 4 KiB borders
(and the padding up to the next 256 bytes) hold a canary byte pattern.  After
each call at ragged sizes -- token counts that leave partial tiles, widths
that are not multiples of 128, shard counts that do not divide 128 -- every
canary byte must be unchanged.  The workspace is given at exactly the size the
library's query returns, so a write past any region the library plans inside
it (the fused stack's control words, tile sums, activations, partial tiles)
lands in the guard."""
import math

import pytest
import torch

import synthetic_inputs as si
from tests.helpers import assert_close, to_np

pytestmark = pytest.mark.gpu
tpl = pytest.importorskip("mlp_megatron_tp_layer_b300")

GUARD = 4096          # bytes on each side; keeps the view 256-byte aligned
CANARY = 0xA5


@pytest.fixture(autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    torch.cuda.synchronize()
    assert tpl.device_status() == 0


class Guarded:
    """A tensor of `shape` x `dtype` (NaN-filled if floating) inside a buffer
    whose surrounding bytes hold the canary."""

    def __init__(self, shape, dtype, nbytes=None):
        elem = torch.empty(0, dtype=dtype).element_size()
        self.n = nbytes if nbytes is not None else math.prod(shape) * elem
        self.span = (self.n + 255) // 256 * 256
        self.raw = torch.full((GUARD + self.span + GUARD,), CANARY, dtype=torch.uint8, device="cuda")
        body = self.raw[GUARD:GUARD + self.n]
        self.t = body.view(dtype).view(shape) if nbytes is None else body
        if nbytes is None and dtype.is_floating_point:
            self.t.fill_(float("nan"))

    def check(self, what):
        torch.cuda.synchronize()
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.n:]
        bad_h = int((head != CANARY).sum())
        bad_t = int((tail != CANARY).sum())
        assert bad_h == 0 and bad_t == 0, f"{what}: {bad_h} bytes before and {bad_t} after the buffer were written"


def _ws(nbytes):
    return Guarded(None, torch.uint8, nbytes=max(int(nbytes), 1))


def _mlp_w(D, F, seed):
    Wg = si.normal((F, D), 0.05, seed, "g.Wg", device="cuda")
    Wu = si.normal((F, D), 0.05, seed, "g.Wu", device="cuda")
    Wd = si.normal((D, F), 0.05, seed, "g.Wd", device="cuda")
    return Wg, Wu, Wd


# ragged MLP: D = 448 (3.5 tiles of 128), F = 1152, tp 3 (F/tp = 384); B = 1
# runs the CUDA-core kernel, 13 the swapped tensor-core GEMM, 300 the GEMM
@pytest.mark.parametrize("B", [1, 13, 300])
@pytest.mark.parametrize("want_partials", [False, True])
def test_mlp_writes_nothing_outside_its_buffers(B, want_partials):
    D, F, tp = 448, 1152, 3
    Wg, Wu, Wd = _mlp_w(D, F, 21)
    X = si.normal((B, D), 1.0, 21, "g.X", device="cuda")
    out = Guarded((B, D), torch.float32)
    P = Guarded((tp, B, D), torch.float32) if want_partials else None
    ws = _ws(tpl.mlp_workspace_bytes(B, D, F, tp))
    res = tpl.tp_mlp_forward(X, Wg, Wu, Wd, tp, out=out.t, partials=P.t if P else None, ws=ws.t)
    out.check("out")
    ws.check("workspace")
    if P:
        P.check("partials")
    ref = tpl.tp_mlp_forward(X, Wg, Wu, Wd, tp, out_dtype=torch.float32)
    y = res[0] if want_partials else res
    assert_close(y, to_np(ref), rel=1e-5, what="guarded vs plain call")


@pytest.mark.parametrize("B", [5, 13, 136])
def test_attn_proj_writes_nothing_outside_its_buffers(B):
    # 7 Q heads, 1 KV group replicated over tp 7, D 448
    D, n_q, n_kv, hd, tp = 448, 7, 1, 64, 7
    Wqkv = si.normal(((n_q + 2 * n_kv) * hd, D), 0.05, 22, "g.Wqkv", device="cuda")
    Wo = si.normal((D, n_q * hd), 0.05, 22, "g.Wo", device="cuda")
    X = si.normal((B, D), 1.0, 22, "g.Xa", device="cuda")
    out = Guarded((B, D), torch.bfloat16)
    qkv = Guarded((tp, B, tpl.qkv_shard_width(n_q, n_kv, hd, tp)), torch.bfloat16)
    P = Guarded((tp, B, D), torch.float32)
    ws = _ws(tpl.attn_workspace_bytes(B, D, n_q, n_kv, hd, tp))
    tpl.tp_attn_proj(X, Wqkv, Wo, n_q, n_kv, hd, tp, out=out.t, qkv_out=qkv.t, partials=P.t, ws=ws.t)
    for g, what in ((out, "out"), (qkv, "qkv_out"), (P, "partials"), (ws, "workspace")):
        g.check(what)
    assert torch.isfinite(out.t.float()).all()


# the fused stack's hand-computed workspace plan: 16/32/64/128-column
# instantiations at ragged batch sizes, serial and parallel blocks
@pytest.mark.parametrize("B", [3, 13, 24, 50, 100])
@pytest.mark.parametrize("block", [tpl.BLOCK_SERIAL, tpl.BLOCK_PARALLEL])
def test_fused_stack_writes_nothing_outside_its_buffers(B, block):
    D, F, n_q, n_kv, hd, tp, L = 448, 1344, 7, 1, 64, 7, 3
    layers = [si.layer_weights(D, F, n_q, n_kv, hd, seed=23, layer=l, sigma=0.05, device="cuda")
              for l in range(L)]
    x = si.activations(B, D, seed=23, device="cuda")
    y = Guarded((B, D), torch.bfloat16)
    ws = _ws(tpl.decoder_workspace_bytes(B, D, F, n_q, n_kv, hd, tp))
    tpl.tp_decoder_stack(x, layers, n_q, n_kv, hd, tp, out=y.t, ws=ws.t, path=tpl.PATH_FUSED, block=block)
    y.check("y")
    ws.check("workspace")
    ref = tpl.tp_decoder_stack(x, layers, n_q, n_kv, hd, tp, path=tpl.PATH_FUSED, block=block)
    assert torch.equal(y.t, ref), "guarded call differs from a plain one"


@pytest.mark.parametrize("B", [13, 160])
def test_unfused_stack_writes_nothing_outside_its_buffers(B):
    D, F, n_q, n_kv, hd, tp, L = 448, 1344, 7, 1, 64, 7, 2
    layers = [si.layer_weights(D, F, n_q, n_kv, hd, seed=24, layer=l, sigma=0.05, device="cuda")
              for l in range(L)]
    x = si.activations(B, D, seed=24, device="cuda")
    y = Guarded((B, D), torch.bfloat16)
    ws = _ws(tpl.decoder_workspace_bytes(B, D, F, n_q, n_kv, hd, tp))
    tpl.tp_decoder_stack(x, layers, n_q, n_kv, hd, tp, out=y.t, ws=ws.t, path=tpl.PATH_UNFUSED)
    y.check("y")
    ws.check("workspace")


@pytest.mark.parametrize("case,mode,gather", [(1, 0, 0), (3, 0, 0), (3, 1, 0), (4, 0, 1)])
def test_sharded_matmul_writes_nothing_outside_its_buffers(case, mode, gather):
    I, J, K, X = 26, 448, 1152, 2
    A = si.normal((I, J), 1.0, 25, "g.A", device="cuda")
    Bt = si.normal((K, J), 0.05, 25, "g.Bt", device="cuda")
    k_sharded = (case == 3 and mode == 1) or (case == 4 and gather == 1)
    out = Guarded((X, I, K // X) if k_sharded else (I, K), torch.float32)
    P = Guarded((X, I, K), torch.float32) if case == 3 else None
    ws = _ws(tpl.case_workspace_bytes(case, mode, I, J, K, X))
    tpl.sharded_matmul(case, A, Bt, X, mode, gather, out=out.t, partials=P.t if P else None, ws=ws.t)
    out.check("C")
    ws.check("workspace")
    if P:
        P.check("partials")


def test_shard_reduce_and_lm_head_write_nothing_outside_their_buffers():
    tp, rows, cols = 3, 13, 456
    parts = si.normal((tp, rows, cols), 1.0, 26, "g.P", dtype=torch.float32, device="cuda")
    for mode, shape in ((tpl.ALLREDUCE, (rows, cols)), (tpl.REDUCE_SCATTER, (tp, rows, cols // tp))):
        out = Guarded(shape, torch.bfloat16)
        tpl.shard_reduce(parts, mode, torch.bfloat16, out=out.t)
        out.check(f"shard_reduce mode {mode}")
    B, D, V, tp, k = 13, 448, 1000, 4, 5
    x, W = si.lm_head(B, D, V, seed=26, device="cuda")
    idx = Guarded((B, k), torch.int32)
    val = Guarded((B, k), torch.float32)
    ws = _ws(tpl.vocab_topk_workspace_bytes(B, V, tp, k))
    tpl.vocab_parallel_topk(x, W, tp, k, out=(idx.t, val.t), ws=ws.t)
    for g, what in ((idx, "top-k indices"), (val, "top-k values"), (ws, "workspace")):
        g.check(what)


@pytest.mark.parametrize("B", [1, 13])
def test_int8_mlp_writes_nothing_outside_its_buffers(B):
    D, F, tp = 448, 1152, 3
    Wg, Wu, Wd = _mlp_w(D, F, 27)
    qg, sg = tpl.quantize_w8(Wg)
    qu, su = tpl.quantize_w8(Wu)
    qd, sd = tpl.quantize_w8(Wd, groups=tp)
    X = si.normal((B, D), 1.0, 27, "g.X8", device="cuda")
    out = Guarded((B, D), torch.float32)
    P = Guarded((tp, B, D), torch.float32)
    ws = _ws(tpl.mlp_w8_workspace_bytes(B, D, F, tp))
    tpl.tp_mlp_forward_w8(X, qg, sg, qu, su, qd, sd, tp, out=out.t, partials=P.t, ws=ws.t)
    for g, what in ((out, "out"), (P, "partials"), (ws, "workspace")):
        g.check(what)
