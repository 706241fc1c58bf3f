"""Parity at the full workload sizes, in the launch configurations the
benchmark times.  Rows of the token dimension are independent, so the oracle
computes a seeded sample of token rows exactly; layer stacks are also checked
against their layer-by-layer composition (bit-exact, any size)."""
import numpy as np
import pytest
import torch

import synthetic_inputs as si
from oracle import tp_layer as O
from tests.helpers import assert_close, assert_equal, assert_within, stack_allowance, to_np

pytestmark = pytest.mark.gpu
tpl = pytest.importorskip("mlp_megatron_tp_layer_b300")


@pytest.fixture(autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    torch.cuda.synchronize()
    assert tpl.device_status() == 0


def sample_rows(n, k, seed=0):
    """k distinct seeded rows of n, always including the first and last."""
    if n <= k:
        return np.arange(n)
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(1, n - 1), size=k - 2, replace=False)
    return np.sort(np.concatenate([[0, n - 1], mid]))


def np64(t):
    return t.detach().to("cpu", torch.float64).numpy()


# ------------------------------------------------------- Qwen decode layer

QW = si.QWEN_DECODE


@pytest.fixture(scope="module")
def qwen_layer():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    W = si.layer_weights(QW["D"], QW["F"], QW["n_q"], QW["n_kv"], QW["head_dim"], seed=0, layer=0, prefix="qwen",
                         device="cuda")
    return W, {k: np64(v) for k, v in W.items()}


@pytest.mark.parametrize("B", [1, 8, 32, 64])
def test_qwen_decode_layer_projections(qwen_layer, B):
    W, Wn = qwen_layer
    D, n_q, n_kv, hd, tp = QW["D"], QW["n_q"], QW["n_kv"], QW["head_dim"], QW["tp"]
    x = si.activations(B, D, seed=1, name=f"bench.x{B}", device="cuda")
    xn = np64(x)
    ya, qkv = tpl.tp_attn_proj(x, W["Wqkv"], W["Wo"], n_q, n_kv, hd, tp, out_dtype=torch.float32, qkv_out=True)
    _, QKV_ref, _, Pa = O.attn_proj_sharded(xn, Wn["Wqkv"], Wn["Wo"], n_q, n_kv, hd, tp)
    assert_close(ya, O.shard_reduce(Pa), what="attn Y")
    for s in range(tp):
        assert_close(qkv[s], QKV_ref[s], bf16_out=True, what=f"QKV_{s}")
    ym, P = tpl.tp_mlp_forward(x, W["Wg"], W["Wu"], W["Wd"], tp, out_dtype=torch.float32, partials=True)
    _, Pm, _ = O.mlp_sharded(xn, Wn["Wg"], Wn["Wu"], Wn["Wd"], tp)
    assert_close(ym, O.shard_reduce(Pm), what="MLP Y")
    for s in range(tp):
        assert_close(P[s], Pm[s], what=f"MLP P_{s}")


def check_layers_against_oracle(x, y, layers, n_q, n_kv, hd, tp, rows, what):
    """Stack output y of input x: (1) equals the layer-by-layer composition bit
    for bit; (2) every layer, fed the oracle's own residual stream on the
    sampled rows (the other rows keep x: rows are independent, and the batch
    size, hence the kernel path, stays the benchmarked one), matches the
    oracle's next residual value within the one-layer bound."""
    z = x
    for W in layers:
        z = tpl.tp_decoder_layer(z, W, n_q, n_kv, hd, tp)
    assert_equal(y, to_np(z), what=f"{what}: stack vs layer-by-layer")
    trace = []
    O.decoder_stack(np64(x)[rows], [{k: np64(v) for k, v in W.items()} for W in layers], n_q, n_kv, hd, tp,
                    trace=trace)
    idx = torch.as_tensor(rows, device=x.device)
    prev = O.bf16_round(np64(x)[rows])
    for l, W in enumerate(layers):
        inp = x.clone()
        inp[idx] = torch.from_numpy(prev).to(device=x.device, dtype=x.dtype)   # exact: bf16 values
        out = tpl.tp_decoder_layer(inp, W, n_q, n_kv, hd, tp)
        h_ref, y_ref = trace[2 * l], trace[2 * l + 1]
        assert_within(to_np(out)[rows], y_ref, stack_allowance([h_ref, y_ref], y_ref), what=f"{what}: layer {l}")
        prev = y_ref


@pytest.mark.parametrize("B", [1, 8, 32, 64])
def test_qwen_parallel_block_stack(B):
    """28 Qwen-shaped layers in the parallel arrangement ([L4] S5.5): every layer,
    fed the oracle's own residual stream on sampled rows, matches the oracle's
    next value; the stack equals its layer-by-layer composition."""
    D, F, n_q, n_kv, hd, tp, L = QW["D"], QW["F"], QW["n_q"], QW["n_kv"], QW["head_dim"], QW["tp"], QW["n_layers"]
    layers = [si.layer_weights(D, F, n_q, n_kv, hd, seed=0, layer=l, prefix="qwen", device="cuda")
              for l in range(L)]
    x = si.activations(B, D, seed=1, name=f"bench.x{B}", device="cuda")
    par = dict(block=tpl.BLOCK_PARALLEL)
    y = tpl.tp_decoder_stack(x, layers, n_q, n_kv, hd, tp, **par)
    z = x
    for W in layers:
        z = tpl.tp_decoder_stack(z, [W], n_q, n_kv, hd, tp, **par)
    assert_equal(y, to_np(z), what="parallel stack vs layer-by-layer")
    rows = sample_rows(B, 8, seed=B)
    trace = []
    O.decoder_stack(np64(x)[rows], [{k: np64(v) for k, v in W.items()} for W in layers], n_q, n_kv, hd, tp,
                    trace=trace, block="parallel")
    idx = torch.as_tensor(rows, device=x.device)
    prev = O.bf16_round(np64(x)[rows])
    for l, W in enumerate(layers):
        inp = x.clone()
        inp[idx] = torch.from_numpy(prev).to(device=x.device, dtype=x.dtype)
        out = tpl.tp_decoder_stack(inp, [W], n_q, n_kv, hd, tp, **par)
        assert_within(to_np(out)[rows], trace[l], stack_allowance([trace[l]], trace[l]), what=f"layer {l}")
        prev = trace[l]


@pytest.mark.parametrize("B", [1, 8, 32, 64])
def test_qwen_decode_stack_as_benchmarked(B):
    """The benchmark's decode step: 28 layers through tp_decoder_stack."""
    D, F, n_q, n_kv, hd, tp, L = QW["D"], QW["F"], QW["n_q"], QW["n_kv"], QW["head_dim"], QW["tp"], QW["n_layers"]
    layers = [si.layer_weights(D, F, n_q, n_kv, hd, seed=0, layer=l, prefix="qwen", device="cuda")
              for l in range(L)]
    x = si.activations(B, D, seed=1, name=f"bench.x{B}", device="cuda")
    y = tpl.tp_decoder_stack(x, layers, n_q, n_kv, hd, tp)
    check_layers_against_oracle(x, y, layers, n_q, n_kv, hd, tp, sample_rows(B, 8, seed=B), "Qwen 28-layer stack")


# ------------------------------------------------- Llama prefill MLP

LP = si.LLAMA_PREFILL


@pytest.fixture(scope="module")
def prefill():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return si.prefill_mlp(LP["B"], LP["D"], LP["F"], seed=0, device="cuda")


def test_llama_prefill_mlp_fused_and_partials(prefill):
    X, Wg, Wu, Wd, tp = prefill["X"], prefill["Wg"], prefill["Wu"], prefill["Wd"], LP["tp"]
    B, D = X.shape
    rows = sample_rows(B, 12, seed=4)
    Y32 = tpl.tp_mlp_forward(X, Wg, Wu, Wd, tp, out_dtype=torch.float32)          # fused (benchmarked)
    Yb = tpl.tp_mlp_forward(X, Wg, Wu, Wd, tp)
    Y2, P = tpl.tp_mlp_forward(X, Wg, Wu, Wd, tp, out_dtype=torch.float32, partials=True)
    torch.cuda.synchronize()
    Xs = np64(X[torch.as_tensor(rows, device="cuda")])
    Y_ref, P_ref, _ = O.mlp_sharded(Xs, np64(Wg), np64(Wu), np64(Wd), tp, bf16=True)
    y_ref = O.shard_reduce(P_ref)
    assert_close(to_np(Y32)[rows], y_ref, what="fused Y (fp32 out)")
    assert_close(to_np(Yb)[rows], y_ref, bf16_out=True, what="fused Y (bf16 out)")
    assert_close(to_np(Y2)[rows], y_ref, what="Y via partials")
    Pn = to_np(P)
    for s in range(tp):
        assert_close(Pn[s][rows], P_ref[s], what=f"P_{s}")


# ------------------------------------------------ four cases, full size

SC = si.SHARDED_CASES
CASES = [(1, 0, 0), (2, 0, 0), (3, 0, 0), (3, 1, 0), (4, 0, 0), (4, 0, 1)]


@pytest.fixture(scope="module")
def cases_operands():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = si.sharded_case_operands(SC["I"], SC["J"], SC["K"], seed=0, device="cuda")
    rows = sample_rows(SC["I"], 8, seed=2)
    C_ref = O.matmul(np64(d["A"])[rows], np64(d["Bt"]))
    return d, rows, C_ref


@pytest.mark.parametrize("case,mode,gather", CASES)
def test_sharded_cases_full_size(cases_operands, case, mode, gather):
    d, rows, C_ref = cases_operands
    X = SC["X"]
    C = tpl.sharded_matmul(case, d["A"], d["Bt"], X, mode, gather, out_dtype=torch.float32)
    Cn = to_np(C)
    k_sharded = (case == 3 and mode == 1) or (case == 4 and gather == 1)
    got = np.concatenate(list(Cn[:, rows, :]), axis=1) if k_sharded else Cn[rows]
    assert_close(got, C_ref, what=f"case {case}")
    if case == 3:
        _, P = tpl.sharded_matmul(case, d["A"], d["Bt"], X, mode, gather, out_dtype=torch.float32, partials=True)
        Pn = to_np(P)
        J = SC["J"]
        for s in (0, X - 1):
            js = O.shard_range(J, X, s)
            ref = O.matmul(np64(d["A"])[rows][:, js.start:js.stop], np64(d["Bt"])[:, js.start:js.stop])
            assert_close(Pn[s][rows], ref, what=f"case 3 partial {s}")


# ----------------------------------------------- Llama decode stack

LD = si.LLAMA_DECODE


@pytest.mark.parametrize("B", [1, 8, 32, 128])
def test_llama_decode_layers_full_width(B):
    D, F, n_q, n_kv, hd, tp = LD["D"], LD["F"], LD["n_q"], LD["n_kv"], LD["head_dim"], LD["tp"]
    L = 2
    layers = [si.layer_weights(D, F, n_q, n_kv, hd, seed=0, layer=l, prefix="llama", device="cuda")
              for l in range(L)]
    x = si.activations(B, D, seed=3, name=f"llama.x{B}", device="cuda")
    y = tpl.tp_decoder_stack(x, layers, n_q, n_kv, hd, tp)
    check_layers_against_oracle(x, y, layers, n_q, n_kv, hd, tp, sample_rows(B, 4, seed=B), "Llama 2-layer stack")
    del layers
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B", [1, 128])
def test_llama_decode_stack_8_layers_equals_composition(B):
    D, F, n_q, n_kv, hd, tp, L = LD["D"], LD["F"], LD["n_q"], LD["n_kv"], LD["head_dim"], LD["tp"], LD["n_layers"]
    layers = [si.layer_weights(D, F, n_q, n_kv, hd, seed=0, layer=l, prefix="llama", device="cuda")
              for l in range(L)]
    x = si.activations(B, D, seed=3, name=f"llama.x{B}", device="cuda")
    y = tpl.tp_decoder_stack(x, layers, n_q, n_kv, hd, tp)
    z = x
    for W in layers:
        z = tpl.tp_decoder_layer(z, W, n_q, n_kv, hd, tp)
    assert_equal(y, to_np(z), what="8-layer stack vs layer-by-layer")
    assert np.all(np.isfinite(to_np(y)))
    del layers
    torch.cuda.empty_cache()


def test_generator_is_device_independent():
    """GPU-generated inputs equal the CPU generator's values bit for bit."""
    idx = torch.tensor([0, 1, 12345, 28672 * 8192 - 1], dtype=torch.int64)
    g = si.normal((28672, 8192), 0.02, 0, "prefill.Wg", device="cuda").flatten()[idx.cuda()].cpu()
    c = si.normal((28672, 8192), 0.02, 0, "prefill.Wg", index=idx)
    assert torch.equal(g, c)
