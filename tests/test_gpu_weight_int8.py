"""Parity of the weight-only int8 path with the oracle, through the C ABI.

* The quantiser's codes and scales are integer / float32 decisions taken in
  float32 on both sides: they must match the oracle bit for bit.
* The int8 MLP computes what the bf16 MLP computes on the dequantised weights
  (every int8 code is a bf16 value, so only the fp32 accumulation order
  differs): the stated bar, max|err| <= 1e-2 * rms, against the oracle's
  sharded MLP on q * s, for the output and for every shard's partial sum --
  on both kernels (CUDA-core row-dot for one or two tokens, tensor cores
  above), at sizes that span several tiles, both token-tile widths, split K
  and ragged token counts, and at full Qwen2.5-1.5B / Llama-3.1-70B width on
  sampled rows.
"""
import numpy as np
import pytest
import torch

import synthetic_inputs as si
from oracle import weight_int8 as W8
from tests.helpers import assert_close, to_np

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


def quantized_mlp(B, D, F, tp, seed, sigma=0.02):
    W = si.layer_weights(D, F, 4, 2, 16, seed=seed, layer=0, prefix="w8", sigma=sigma, device="cuda")
    x = si.activations(B, D, seed=seed, name="w8.x", device="cuda")
    Qg, sg = tpl.quantize_w8(W["Wg"])
    Qu, su = tpl.quantize_w8(W["Wu"])
    Qd, sd = tpl.quantize_w8(W["Wd"], groups=tp)
    return x, W, (Qg, sg, Qu, su, Qd, sd)


@pytest.mark.parametrize("rows,cols,groups", [(300, 256, 1), (64, 1024, 4), (7, 96, 3), (128, 8960, 2)])
def test_quantiser_matches_oracle_bit_for_bit(rows, cols, groups):
    W = si.normal((rows, cols), 0.02, seed=rows, name="w8.q", device="cuda")
    W[0, : cols // groups] = 0                      # a group of zeros: scale 0, codes 0
    W[1, 5] = 1.0                                   # a large outlier sets its group's scale
    Q, s = tpl.quantize_w8(W, groups)
    q_ref, s_ref = W8.quantize_rows(W.float().cpu().numpy(), groups)
    assert np.array_equal(Q.cpu().numpy(), q_ref)
    assert np.array_equal(s.cpu().numpy(), s_ref)


def test_quantiser_ties_go_to_even():
    # amax 127 gives scale 1, so the codes are the rounded values themselves
    vals = torch.tensor([[127.0, 2.5, -3.5, 0.5, 1.5, -0.5, 126.5, -127.0]], dtype=torch.bfloat16, device="cuda")
    Q, s = tpl.quantize_w8(vals)
    assert s.item() == 1.0
    assert Q.cpu().tolist() == [[127, 2, -4, 0, 2, 0, 126, -127]]


@pytest.mark.parametrize("B,D,F,tp", [
    (1, 256, 1024, 2),       # CUDA-core row-dot (one token), split K on both projections
    (2, 512, 1536, 4),       # CUDA-core row-dot, two tokens
    (3, 256, 1024, 2),       # tensor cores, 16-token tile
    (5, 512, 1536, 4),
    (40, 256, 2048, 2),      # 64-token tile with 24 padded columns
    (17, 192, 768, 3),       # 32-token tile, three shards
    (130, 128, 1024, 2),     # two 128-token tiles
])
def test_w8_mlp_matches_oracle(B, D, F, tp):
    x, W, q = quantized_mlp(B, D, F, tp, seed=B)
    Qg, sg, Qu, su, Qd, sd = q
    Y, P = tpl.tp_mlp_forward_w8(x, *q, tp, out_dtype=torch.float32, partials=True)
    Yb = tpl.tp_mlp_forward_w8(x, *q, tp)
    n = lambda t: t.cpu().numpy()
    Y_ref, P_ref, _ = W8.mlp_sharded_w8(to_np(x), n(Qg), n(sg), n(Qu), n(su), n(Qd), n(sd), tp)
    y_ref = sum(P_ref[1:], P_ref[0].copy())
    assert_close(Y, y_ref, what="Y (fp32 out)")
    assert_close(Yb, y_ref, bf16_out=True, what="Y (bf16 out)")
    for s in range(tp):
        assert_close(P[s], P_ref[s], what=f"P_{s}")


def test_w8_mlp_tracks_bf16_mlp_and_is_deterministic():
    B, D, F, tp = 8, 512, 2048, 2
    x, W, q = quantized_mlp(B, D, F, tp, seed=11)
    Y1 = tpl.tp_mlp_forward_w8(x, *q, tp, out_dtype=torch.float32)
    Y2 = tpl.tp_mlp_forward_w8(x, *q, tp, out_dtype=torch.float32)
    assert torch.equal(Y1, Y2)
    Yf = tpl.tp_mlp_forward(x, W["Wg"], W["Wu"], W["Wd"], tp, out_dtype=torch.float32)
    err = (Y1 - Yf).abs().max().item()
    assert err < 0.05 * Yf.pow(2).mean().sqrt().item()     # quantisation error only, half a step per weight


@pytest.mark.parametrize("name,D,F,tp,B", [
    ("qwen2.5-1.5b", 1536, 8960, 2, 64),
    ("llama-3.1-70b", 8192, 28672, 8, 8),
    ("llama-3.1-70b", 8192, 28672, 8, 1),
])
def test_w8_mlp_full_width_sampled_rows(name, D, F, tp, B):
    """Full model width, in the launch configuration the benchmark times; the
    oracle checks sampled token rows (rows are independent)."""
    W = si.layer_weights(D, F, 8, 8, 128, seed=0, layer=0, prefix=name, device="cuda") if D == 8192 else \
        si.layer_weights(D, F, 12, 2, 128, seed=0, layer=0, prefix=name, device="cuda")
    x = si.activations(B, D, seed=1, name=f"{name}.w8x", device="cuda")
    Qg, sg = tpl.quantize_w8(W["Wg"])
    Qu, su = tpl.quantize_w8(W["Wu"])
    Qd, sd = tpl.quantize_w8(W["Wd"], groups=tp)
    Y, P = tpl.tp_mlp_forward_w8(x, Qg, sg, Qu, su, Qd, sd, tp, out_dtype=torch.float32, partials=True)
    del W
    torch.cuda.empty_cache()
    rows = [0, B // 3, B - 1]
    n = lambda t: t.cpu().numpy()
    Y_ref, P_ref, _ = W8.mlp_sharded_w8(to_np(x)[rows], n(Qg), n(sg), n(Qu), n(su), n(Qd), n(sd), tp)
    y_ref = sum(P_ref[1:], P_ref[0].copy())
    assert_close(to_np(Y)[rows], y_ref, what=f"{name} Y")
    Pn = to_np(P)
    for s in range(tp):
        assert_close(Pn[s][rows], P_ref[s], what=f"{name} P_{s}")
