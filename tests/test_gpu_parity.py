"""Parity of the CUDA path (through the C ABI) with the oracle, on the same
seeded inputs, at sizes the oracle finishes in seconds that still span several
tiles and ragged tails, and on every kernel path (CUDA-core row-dot for one bf16
token and for fp32, swapped tensor-core GEMM for 2..128 bf16 tokens, tensor-core
GEMM above)."""
import numpy as np
import pytest
import torch

import synthetic_inputs as si
from oracle import tp_layer as O
from tests.helpers import F32_REL, assert_close, assert_equal, assert_within, stack_allowance, to_np

pytestmark = pytest.mark.gpu
tpl = pytest.importorskip("mlp_megatron_tp_layer_b300")


@pytest.fixture(autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.synchronize()
    yield
    torch.cuda.synchronize()
    assert tpl.device_status() == 0, "a device-side wait timed out"


def nan_like(shape, dtype):
    return torch.full(shape, float("nan"), dtype=dtype, device="cuda")


# --------------------------------------------------------------- tiny fp32

def test_tiny_fp32_mlp_partials_sum_to_unsharded():
    d = si.tiny_mlp(seed=0, device="cuda")
    X, Wg, Wu, Wd, tp = d["X"], d["Wg"], d["Wu"], d["Wd"], d["tp"]
    Xn, Wgn, Wun, Wdn = map(to_np, (X, Wg, Wu, Wd))
    Y_ref = O.mlp_unsharded(Xn, Wgn, Wun, Wdn, bf16=False)
    _, P_ref, _ = O.mlp_sharded(Xn, Wgn, Wun, Wdn, tp, bf16=False)
    Y, P = tpl.tp_mlp_forward(X, Wg, Wu, Wd, tp, out=nan_like((8, 256), torch.float32),
                              partials=nan_like((tp, 8, 256), torch.float32))
    assert_close(Y, Y_ref, rel=F32_REL, what="Y")
    for s in range(tp):
        assert_close(P[s], P_ref[s], rel=F32_REL, what=f"P_{s}")
    # the spec check: the sum of the row-parallel partials is the unsharded Y
    assert_close(to_np(P).sum(axis=0), Y_ref, rel=F32_REL, what="sum of partials")
    Yf = tpl.tp_mlp_forward(X, Wg, Wu, Wd, tp)
    assert_close(Yf, Y_ref, rel=F32_REL, what="fused Y")


# --------------------------------------------------------------- bf16 MLP

def _mlp_inputs(B, D, F, seed=0):
    X = si.normal((B, D), 1.0, seed, "t.X", device="cuda")
    Wg = si.normal((F, D), 0.05, seed, "t.Wg", device="cuda")
    Wu = si.normal((F, D), 0.05, seed, "t.Wu", device="cuda")
    Wd = si.normal((D, F), 0.05, seed, "t.Wd", device="cuda")
    return X, Wg, Wu, Wd


@pytest.mark.parametrize("B", [1, 3, 8, 13, 64, 128, 200, 300])
def test_mlp_bf16_all_paths(B):
    D, F, tp = 448, 1408, 2          # D spans 3.5 tiles of 128; F/tp = 704 = 11 K blocks of 64
    X, Wg, Wu, Wd = _mlp_inputs(B, D, F)
    Xn, Wgn, Wun, Wdn = map(to_np, (X, Wg, Wu, Wd))
    Y_ref, P_ref, _ = O.mlp_sharded(Xn, Wgn, Wun, Wdn, tp, bf16=True)
    y_unrounded = O.shard_reduce(P_ref)
    # unrounded fp32 result against the stated tolerance
    Y32, P = tpl.tp_mlp_forward(X, Wg, Wu, Wd, tp, out=nan_like((B, D), torch.float32),
                                partials=nan_like((tp, B, D), torch.float32))
    assert_close(Y32, y_unrounded, what="Y fp32 (partials path)")
    for s in range(tp):
        assert_close(P[s], P_ref[s], what=f"P_{s}")
    Y32f = tpl.tp_mlp_forward(X, Wg, Wu, Wd, tp, out=nan_like((B, D), torch.float32))
    assert_close(Y32f, y_unrounded, what="Y fp32 (fused)")
    # bf16 output
    Yb = tpl.tp_mlp_forward(X, Wg, Wu, Wd, tp, out=nan_like((B, D), torch.bfloat16))
    assert_close(Yb, y_unrounded, bf16_out=True, what="Y bf16")


@pytest.mark.parametrize("tp", [1, 4, 8])
def test_mlp_bf16_shard_counts(tp):
    B, D, F = 40, 256, 2048
    X, Wg, Wu, Wd = _mlp_inputs(B, D, F, seed=3)
    Xn, Wgn, Wun, Wdn = map(to_np, (X, Wg, Wu, Wd))
    _, P_ref, _ = O.mlp_sharded(Xn, Wgn, Wun, Wdn, tp, bf16=True)
    Y32, P = tpl.tp_mlp_forward(X, Wg, Wu, Wd, tp, out=nan_like((B, D), torch.float32), partials=True)
    assert_close(Y32, O.shard_reduce(P_ref), what="Y")
    for s in range(tp):
        assert_close(P[s], P_ref[s], what=f"P_{s}")


# ---------------------------------------------------------- attention

def _attn_inputs(B, D, n_q, n_kv, hd, seed=0, integer=False):
    nqkv = (n_q + 2 * n_kv) * hd
    if integer:
        X = si.small_integers((B, D), seed, "a.X", -2, 2, device="cuda")
        Wqkv = si.small_integers((nqkv, D), seed, "a.Wqkv", -1, 1, device="cuda", zero_frac_num=8)
        Wo = si.small_integers((D, n_q * hd), seed, "a.Wo", -1, 1, device="cuda", zero_frac_num=8)
    else:
        X = si.normal((B, D), 1.0, seed, "a.X", device="cuda")
        Wqkv = si.normal((nqkv, D), 0.05, seed, "a.Wqkv", device="cuda")
        Wo = si.normal((D, n_q * hd), 0.05, seed, "a.Wo", device="cuda")
    return X, Wqkv, Wo


@pytest.mark.parametrize("tp", [1, 2, 4, 8])
@pytest.mark.parametrize("B", [1, 5, 40, 160])
def test_attn_proj_bf16(tp, B):
    D, n_q, n_kv, hd = 512, 8, 2, 64
    X, Wqkv, Wo = _attn_inputs(B, D, n_q, n_kv, hd, seed=tp)
    Xn, Wq, Won = map(to_np, (X, Wqkv, Wo))
    _, QKV_ref, _, P_ref = O.attn_proj_sharded(Xn, Wq, Won, n_q, n_kv, hd, tp, bf16=True)
    Y32, qkv, P = tpl.tp_attn_proj(X, Wqkv, Wo, n_q, n_kv, hd, tp, out=nan_like((B, D), torch.float32),
                                   qkv_out=True, partials=True)
    for s in range(tp):
        assert_close(qkv[s], QKV_ref[s], bf16_out=True, what=f"QKV_{s}")
        assert_close(P[s], P_ref[s], what=f"P_{s}")
    assert_close(Y32, O.shard_reduce(P_ref), what="Y fp32")
    Yb = tpl.tp_attn_proj(X, Wqkv, Wo, n_q, n_kv, hd, tp)
    assert_close(Yb, O.shard_reduce(P_ref), bf16_out=True, what="Y bf16")


@pytest.mark.parametrize("tp", [1, 2, 4, 8])
@pytest.mark.parametrize("B", [2, 24, 136])
def test_attn_head_layout_bit_exact(tp, B):
    """Integer-valued data: every product and sum is exact, so the shard
    blocks of QKV, the partials and Y must match the oracle bit for bit."""
    D, n_q, n_kv, hd = 256, 8, 2, 64
    X, Wqkv, Wo = _attn_inputs(B, D, n_q, n_kv, hd, seed=7, integer=True)
    Xn, Wq, Won = map(to_np, (X, Wqkv, Wo))
    Y_ref, QKV_ref, _, P_ref = O.attn_proj_sharded(Xn, Wq, Won, n_q, n_kv, hd, tp, bf16=True)
    Y, qkv, P = tpl.tp_attn_proj(X, Wqkv, Wo, n_q, n_kv, hd, tp, qkv_out=True, partials=True)
    for s in range(tp):
        assert_equal(qkv[s], QKV_ref[s], what=f"QKV_{s}")
        assert_equal(P[s], P_ref[s], what=f"P_{s}")
    assert_equal(Y, Y_ref, what="Y")


# -------------------------------------------------------- four cases

CASES = [(1, tpl.ALLREDUCE, tpl.GATHER_B), (2, tpl.ALLREDUCE, tpl.GATHER_B), (3, tpl.ALLREDUCE, tpl.GATHER_B),
         (3, tpl.REDUCE_SCATTER, tpl.GATHER_B), (4, tpl.ALLREDUCE, tpl.GATHER_B), (4, tpl.ALLREDUCE, tpl.GATHER_A)]


def _oracle_case(case, mode, gather, An, Btn, X, bf16):
    return O.sharded_matmul(case, An, Btn, X, mode="allreduce" if mode == tpl.ALLREDUCE else "reducescatter",
                            gather="A" if gather == tpl.GATHER_A else "B", bf16=bf16)


@pytest.mark.parametrize("I", [8, 64, 256])
@pytest.mark.parametrize("case,mode,gather", CASES)
def test_sharded_matmul_cases(I, case, mode, gather):
    J, K, X = 1024, 2048, 8
    A = si.normal((I, J), 1.0, 0, "c.A", device="cuda")
    Bt = si.normal((K, J), 1.0 / np.sqrt(J), 0, "c.Bt", device="cuda")
    An, Btn = to_np(A), to_np(Bt)
    C_ref, P_ref = _oracle_case(case, mode, gather, An, Btn, X, bf16=False)
    C32 = tpl.sharded_matmul(case, A, Bt, X, mode, gather, out_dtype=torch.float32)
    assert_close(C32, C_ref, what="C fp32")
    Cb = tpl.sharded_matmul(case, A, Bt, X, mode, gather)
    assert_close(Cb, C_ref, bf16_out=True, what="C bf16")
    if case == 3:
        C2, P = tpl.sharded_matmul(case, A, Bt, X, mode, gather, out_dtype=torch.float32, partials=True)
        assert_close(C2, C_ref, what="C via partials")
        for s in range(X):
            assert_close(P[s], P_ref[s], what=f"P_{s}")


@pytest.mark.parametrize("I", [8, 64, 256])
@pytest.mark.parametrize("case,mode,gather", CASES)
def test_sharded_matmul_layout_bit_exact(I, case, mode, gather):
    J, K, X = 512, 1024, 4
    A = si.small_integers((I, J), 1, "ci.A", -2, 2, device="cuda")
    Bt = si.small_integers((K, J), 1, "ci.Bt", -1, 1, device="cuda", zero_frac_num=8)
    C_ref, _ = _oracle_case(case, mode, gather, to_np(A), to_np(Bt), X, bf16=True)
    C = tpl.sharded_matmul(case, A, Bt, X, mode, gather)
    assert_equal(C, C_ref, what="C")


# 2 x 80 output tiles of 128 x 256 = 160 tiles on 148 SMs: the GEMM runs one
# full wave and splits the 12 tiles of its last wave along K (8 chunks each),
# then sums each tile's chunk partials in k order
@pytest.mark.parametrize("case,mode,gather", CASES)
def test_sharded_matmul_split_last_wave(case, mode, gather):
    I, J, K, X = 256, 512, 20480, 4
    if torch.cuda.get_device_properties(0).multi_processor_count == 148:
        assert tpl.case_workspace_bytes(case, mode, I, J, K, X) > 0 or case == 3
    A = si.normal((I, J), 1.0, 3, "cw.A", device="cuda")
    Bt = si.normal((K, J), 1.0 / np.sqrt(J), 3, "cw.Bt", device="cuda")
    C_ref, _ = _oracle_case(case, mode, gather, to_np(A), to_np(Bt), X, bf16=False)
    C32 = tpl.sharded_matmul(case, A, Bt, X, mode, gather, out_dtype=torch.float32)
    assert_close(C32, C_ref, what="C fp32")
    Cb = tpl.sharded_matmul(case, A, Bt, X, mode, gather)
    assert_close(Cb, C_ref, bf16_out=True, what="C bf16")
    # integer data: every order of the sums is exact, so the layout is checked bit for bit
    Ai = si.small_integers((I, J), 4, "cwi.A", -2, 2, device="cuda")
    Bi = si.small_integers((K, J), 4, "cwi.Bt", -1, 1, device="cuda", zero_frac_num=8)
    C_int, _ = _oracle_case(case, mode, gather, to_np(Ai), to_np(Bi), X, bf16=True)
    assert_equal(tpl.sharded_matmul(case, Ai, Bi, X, mode, gather), C_int, what="C integer data")
    # deterministic: a second call gives the same bits
    assert torch.equal(tpl.sharded_matmul(case, A, Bt, X, mode, gather, out_dtype=torch.float32), C32)


# ------------------------------------------------------ shard_reduce

@pytest.mark.parametrize("tp", [1, 2, 3, 8])
@pytest.mark.parametrize("mode", [tpl.ALLREDUCE, tpl.REDUCE_SCATTER])
def test_shard_reduce(tp, mode):
    rows, cols = 37, 8 * 24
    P = si.normal((tp, rows, cols), 1.0, tp, "r.P", torch.float32, device="cuda")
    Pn = to_np(P)
    ref = O.shard_reduce(list(Pn))
    if mode == tpl.REDUCE_SCATTER:
        ref = O.reduce_scatter_blocks(ref, tp)
    out32 = tpl.shard_reduce(P, mode, torch.float32)
    # same precision, same order: a float32 left-to-right sum on the host
    acc = Pn[0].astype(np.float32)
    for s in range(1, tp):
        acc = acc + Pn[s].astype(np.float32)
    host = acc.astype(np.float64)
    if mode == tpl.REDUCE_SCATTER:
        host = O.reduce_scatter_blocks(host, tp)
    assert_equal(out32, host, what="fp32 sum in shard order")
    assert_close(out32, ref, rel=1e-6, what="vs oracle")
    outb = tpl.shard_reduce(P, mode, torch.bfloat16)
    assert_equal(outb, O.bf16_round(host), what="bf16 output")


# --------------------------------------------------------- decoder stack

@pytest.mark.parametrize("B", [1, 16, 160])
def test_decoder_stack_small(B):
    D, F, n_q, n_kv, hd, tp, L = 256, 512, 4, 2, 64, 2, 3
    x = si.activations(B, D, seed=5, device="cuda")
    layers = [si.layer_weights(D, F, n_q, n_kv, hd, seed=5, layer=l, sigma=0.05, device="cuda") for l in range(L)]
    trace = []
    ref = O.decoder_stack(to_np(x), [{k: to_np(v) for k, v in W.items()} for W in layers], n_q, n_kv, hd, tp,
                          trace=trace)
    y = tpl.tp_decoder_stack(x, layers, n_q, n_kv, hd, tp)
    # one layer: the stated bar plus the bf16 roundings of h and y
    y1 = tpl.tp_decoder_stack(x, layers[:1], n_q, n_kv, hd, tp)
    assert_within(y1, trace[1], stack_allowance(trace[:2], trace[1]), what="first layer")
    assert_within(y, ref, stack_allowance(trace, ref), what="stack output")
    # the stack equals the layer-by-layer composition bit for bit
    z = x
    for W in layers:
        z = tpl.tp_decoder_layer(z, W, n_q, n_kv, hd, tp)
    assert_equal(y, to_np(z), what="stack vs layers")


# ------------------------------------------------ fused decode stack

# every instantiation of the fused kernel (16, 32, 64 and 128 token columns),
# at full and ragged batch sizes
@pytest.mark.parametrize("B", [1, 5, 16, 17, 24, 32, 40, 64, 100, 128])
@pytest.mark.parametrize("path", [tpl.PATH_FUSED, tpl.PATH_UNFUSED])
def test_decoder_stack_paths(B, path):
    """Both implementations of the stack against the oracle; each deterministic."""
    D, F, n_q, n_kv, hd, tp, L = 256, 512, 4, 2, 64, 2, 3
    x = si.activations(B, D, seed=6, device="cuda")
    layers = [si.layer_weights(D, F, n_q, n_kv, hd, seed=6, layer=l, sigma=0.05, device="cuda") for l in range(L)]
    trace = []
    ref = O.decoder_stack(to_np(x), [{k: to_np(v) for k, v in W.items()} for W in layers], n_q, n_kv, hd, tp,
                          trace=trace)
    y1 = tpl.tp_decoder_stack(x, layers[:1], n_q, n_kv, hd, tp, path=path)
    assert_within(y1, trace[1], stack_allowance(trace[:2], trace[1]), what="first layer")
    y = tpl.tp_decoder_stack(x, layers, n_q, n_kv, hd, tp, path=path)
    assert_within(y, ref, stack_allowance(trace, ref), what="stack output")
    y2 = tpl.tp_decoder_stack(x, layers, n_q, n_kv, hd, tp, path=path)
    assert_equal(y2, to_np(y), what="second run")


@pytest.mark.parametrize("B", [3, 64])
def test_decoder_stack_fused_in_place_and_gqa_shapes(B):
    """Fused stack with y == x, tp > n_kv (replicated KV groups) and hd 128."""
    D, F, n_q, n_kv, hd, tp, L = 512, 1024, 8, 2, 128, 4, 2
    x = si.activations(B, D, seed=8, device="cuda")
    layers = [si.layer_weights(D, F, n_q, n_kv, hd, seed=8, layer=l, sigma=0.04, device="cuda") for l in range(L)]
    trace = []
    ref = O.decoder_stack(to_np(x), [{k: to_np(v) for k, v in W.items()} for W in layers], n_q, n_kv, hd, tp,
                          trace=trace)
    y = x.clone()
    tpl.tp_decoder_stack(y, layers, n_q, n_kv, hd, tp, out=y, path=tpl.PATH_FUSED)
    assert_within(y, ref, stack_allowance(trace, ref), what="in-place fused stack")


# gate/up with at least one 128-row tile per CTA (149 tiles): CTA c takes tile c
# whole and applies SwiGLU from TMEM; the remaining tile is split over the grid
# (the 32- and 128-column builds; the others split every tile)
@pytest.mark.parametrize("B", [1, 24, 40, 128])
@pytest.mark.parametrize("block", ["serial", "parallel"])
def test_decoder_stack_fused_whole_gateup_tiles(B, block):
    D, F, n_q, n_kv, hd, tp, L = 256, 19072, 2, 1, 128, 2, 2
    x = si.activations(B, D, seed=12, device="cuda")
    layers = [si.layer_weights(D, F, n_q, n_kv, hd, seed=12, layer=l, sigma=0.03, device="cuda") for l in range(L)]
    trace = []
    ref = O.decoder_stack(to_np(x), [{k: to_np(v) for k, v in W.items()} for W in layers], n_q, n_kv, hd, tp,
                          trace=trace, block=block)
    blk = tpl.BLOCK_PARALLEL if block == "parallel" else tpl.BLOCK_SERIAL
    y = tpl.tp_decoder_stack(x, layers, n_q, n_kv, hd, tp, path=tpl.PATH_FUSED, block=blk)
    assert_within(y, ref, stack_allowance(trace, ref), what="fused stack, whole gate/up tiles")
    y2 = tpl.tp_decoder_stack(x, layers, n_q, n_kv, hd, tp, path=tpl.PATH_FUSED, block=blk)
    assert_equal(y2, to_np(y), what="second run")


# ------------------------------------------ parallel (PaLM) block, [L4] S5.5

@pytest.mark.parametrize("B", [1, 5, 17, 32, 40, 64, 128])
def test_decoder_stack_parallel_block(B):
    """y = x + Attn(RMSNorm(x)) + MLP(RMSNorm(x)) through the fused stack, against
    the oracle; one bf16 rounding of the residual stream per layer."""
    D, F, n_q, n_kv, hd, tp, L = 256, 512, 4, 2, 64, 2, 3
    x = si.activations(B, D, seed=9, device="cuda")
    layers = [si.layer_weights(D, F, n_q, n_kv, hd, seed=9, layer=l, sigma=0.05, device="cuda") for l in range(L)]
    trace = []
    ref = O.decoder_stack(to_np(x), [{k: to_np(v) for k, v in W.items()} for W in layers], n_q, n_kv, hd, tp,
                          trace=trace, block="parallel")
    y = tpl.tp_decoder_stack(x, layers, n_q, n_kv, hd, tp, block=tpl.BLOCK_PARALLEL)
    assert_within(y, ref, stack_allowance(trace, ref), what="parallel-block stack")
    y1 = tpl.tp_decoder_stack(x, layers[:1], n_q, n_kv, hd, tp, block=tpl.BLOCK_PARALLEL)
    assert_within(y1, trace[0], stack_allowance(trace[:1], trace[0]), what="first layer")
    y2 = tpl.tp_decoder_stack(x, layers, n_q, n_kv, hd, tp, block=tpl.BLOCK_PARALLEL)
    assert_equal(y2, to_np(y), what="second run")
