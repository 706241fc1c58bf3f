"""Pins for the oracle: checks against what the pages and mathematics fix.

Nothing here retypes the oracle's formulas: each test compares the oracle with
an independent source -- a library routine (torch's bf16 cast, mpmath), exact
rational arithmetic, brute-force loops on tiny inputs, closed forms, identities
the pages state, or numbers the pages print (tests/golden/worked_examples.txt).
"""
import math
import os
from fractions import Fraction

import mpmath
import numpy as np
import pytest
import torch

from oracle import accounting as acc
from oracle import tp_layer as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.txt")


def golden():
    out = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, rest = line.split("=", 1)
        val = rest.split("|")[0].split()
        out[key.strip()] = (float(val[0]), val[1])
    return out


def rng(seed=0):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- bf16 rounding

def test_bf16_round_matches_torch_cast_on_fp32_values():
    r = rng(1)
    vals = np.concatenate([
        r.standard_normal(20000).astype(np.float32),
        (r.standard_normal(2000) * 1e-38).astype(np.float32),       # subnormal range
        (r.standard_normal(2000) * 1e30).astype(np.float32),
        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3.0e38, -3.0e38], np.float32),
    ])
    # exact ties: 1 + k/256 for odd k sits halfway between two bf16 neighbours
    ties = (1.0 + (2 * np.arange(64) + 1) / 256.0).astype(np.float32)
    vals = np.concatenate([vals, ties, -ties])
    ref = torch.from_numpy(vals).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.bf16_round(vals.astype(np.float64))
    assert np.array_equal(got, ref)


def _bf16_round_exact(x: float) -> float:
    """Round-to-nearest-even onto the bf16 grid using exact rationals."""
    if x == 0:
        return 0.0
    f = Fraction(x)
    e = math.frexp(x)[1]
    q = Fraction(2) ** (max(e, -125) - 8)
    n = f / q
    lo = math.floor(n)
    rem = n - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return float(lo * q)


def test_bf16_round_matches_exact_rational_rounding_on_fp64_values():
    r = rng(2)
    xs = list(r.standard_normal(3000) * np.exp(r.uniform(-20, 20, 3000)))
    xs += [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -9, -(1.0 + 2.0 ** -8 + 2.0 ** -40)]
    for x in xs:
        assert O.bf16_round(x) == _bf16_round_exact(float(x)), x


# ------------------------------------------------------------------------ SiLU

def test_silu_special_values_and_identity():
    assert O.silu(0.0) == 0.0
    z = np.linspace(-30, 30, 601)
    # silu(z) - silu(-z) = z  (z s(z) + z s(-z) = z)
    assert np.allclose(O.silu(z) - O.silu(-z), z, rtol=0, atol=1e-13)
    assert abs(O.silu(50.0) - 50.0) < 1e-12 and abs(O.silu(-50.0)) < 1e-18


def test_silu_matches_high_precision_library():
    mpmath.mp.dps = 40
    for z in [-7.25, -1.0, -0.3, 0.1, 0.5, 1.0, 2.75, 9.0]:
        ref = mpmath.mpf(z) / (1 + mpmath.exp(-mpmath.mpf(z)))
        assert abs(O.silu(z) - float(ref)) <= 4e-16 * max(1.0, abs(z))


# ------------------------------------------------------------------- products

def _brute_linear(x, w):
    """y[b][o] = sum_i x[b][i] * w[o][i] with Python loops."""
    B, Din = len(x), len(x[0])
    Dout = len(w)
    return [[sum(x[b][i] * w[o][i] for i in range(Din)) for o in range(Dout)] for b in range(B)]


def test_linear_brute_force_nonsquare():
    r = rng(3)
    x = r.standard_normal((3, 5))
    w = r.standard_normal((7, 5))
    assert np.allclose(O.linear(x, w), np.array(_brute_linear(x.tolist(), w.tolist())), rtol=1e-14, atol=1e-14)


def test_mlp_hand_worked_example():
    # X = [1, -1]; Wg = I (gate = X), Wu = diag(2, 3), Wd = [[0, 1], [1, 0]] (swap)
    X = np.array([[1.0, -1.0]])
    Wg = np.eye(2)
    Wu = np.diag([2.0, 3.0])
    Wd = np.array([[0.0, 1.0], [1.0, 0.0]])
    mpmath.mp.dps = 30
    s1 = float(1 / (1 + mpmath.exp(-1)))           # sigmoid(1)
    h0 = 1.0 * s1 * 2.0                              # silu(1) * 2
    h1 = -1.0 * (1 - s1) * -3.0                      # silu(-1) * (-3)
    Y = O.mlp_unsharded(X, Wg, Wu, Wd, bf16=False)
    assert np.allclose(Y, [[h1, h0]], rtol=1e-15, atol=0)
    Ys, P, H = O.mlp_sharded(X, Wg, Wu, Wd, tp=2, bf16=False)
    assert np.allclose(Ys, Y, rtol=1e-15, atol=0)
    # shard 0 owns hidden unit 0, which Wd sends to output 1; shard 1 the other way
    assert np.allclose(P[0], [[0.0, h0]]) and np.allclose(P[1], [[h1, 0.0]])


def test_mlp_brute_force_tiny():
    r = rng(4)
    B, D, F = 3, 4, 6
    X, Wg, Wu, Wd = r.standard_normal((B, D)), r.standard_normal((F, D)), r.standard_normal((F, D)), r.standard_normal((D, F))
    mpmath.mp.dps = 30
    H = [[0.0] * F for _ in range(B)]
    for b in range(B):
        for f in range(F):
            g = sum(X[b, i] * Wg[f, i] for i in range(D))
            u = sum(X[b, i] * Wu[f, i] for i in range(D))
            H[b][f] = float(mpmath.mpf(g) / (1 + mpmath.exp(-mpmath.mpf(g)))) * u
    Y = [[sum(H[b][f] * Wd[o, f] for f in range(F)) for o in range(D)] for b in range(B)]
    assert np.allclose(O.mlp_unsharded(X, Wg, Wu, Wd, bf16=False), Y, rtol=1e-12, atol=1e-12)
    for tp in (1, 2, 3, 6):
        Ys, _, _ = O.mlp_sharded(X, Wg, Wu, Wd, tp, bf16=False)
        assert np.allclose(Ys, Y, rtol=1e-12, atol=1e-12)


def test_mlp_zero_gate_gives_zero():
    r = rng(5)
    X, Wu, Wd = r.standard_normal((2, 8)), r.standard_normal((16, 8)), r.standard_normal((8, 16))
    Y = O.mlp_unsharded(X, np.zeros((16, 8)), Wu, Wd, bf16=True)
    assert np.array_equal(Y, np.zeros((2, 8)))


def test_column_parallel_concat_is_bit_exact():
    """[L4] S4.1: the column split needs no communication; concatenating the
    shards' hidden blocks is the single-device hidden, element for element."""
    r = rng(6)
    X, Wg, Wu = r.standard_normal((5, 32)), r.standard_normal((48, 32)), r.standard_normal((48, 32))
    full = O.bf16_round(O.silu(X @ Wg.T) * (X @ Wu.T))
    for tp in (1, 2, 3, 4, 6, 8):
        cat = np.concatenate([O.mlp_hidden_shard(X, Wg, Wu, tp, s) for s in range(tp)], axis=1)
        assert np.array_equal(cat, full)


def test_row_parallel_sum_is_exact_on_integers():
    """[L4] S3.2 case 3 / S4.1: the shards' partial sums add up to the product."""
    r = rng(7)
    H = r.integers(-2, 3, (6, 96)).astype(float)
    Wd = r.integers(-2, 3, (40, 96)).astype(float)
    ref = np.array(_brute_linear(H.tolist(), Wd.tolist()))
    for tp in (1, 2, 3, 4, 8, 12):
        P = [O.mlp_partial_shard(H[:, O.shard_range(96, tp, s).start:O.shard_range(96, tp, s).stop], Wd, tp, s)
             for s in range(tp)]
        assert np.array_equal(O.shard_reduce(P), ref)


def test_sharded_mlp_within_rounding_of_single_device():
    """[L4] S4.3: the sharded output equals the single-device output up to the
    order of the partial-sum additions."""
    r = rng(8)
    X = r.standard_normal((4, 64))
    Wg, Wu = r.standard_normal((128, 64)) / 8, r.standard_normal((128, 64)) / 8
    Wd = r.standard_normal((64, 128)) / 11
    Y = O.mlp_unsharded(X, Wg, Wu, Wd, bf16=False)
    for tp in (2, 4, 8):
        Ys, _, _ = O.mlp_sharded(X, Wg, Wu, Wd, tp, bf16=False)
        H = O.silu(X @ Wg.T) * (X @ Wu.T)
        bound = 128 * 2.3e-16 * (np.abs(H) @ np.abs(Wd).T)
        assert np.all(np.abs(Ys - Y) <= bound)


def test_shard_range_rejects_indivisible():
    with pytest.raises(ValueError):
        O.shard_range(10, 3, 0)
    assert list(O.shard_range(12, 3, 2)) == [8, 9, 10, 11]


def test_shard_reduce_order_and_rs_blocks():
    P = [np.full((2, 6), 1e16), np.full((2, 6), 1.0), np.full((2, 6), -1e16)]
    # left to right: (1e16 + 1) + -1e16 = 0 in fp64 (the 1 is absorbed)
    assert np.array_equal(O.shard_reduce(P), np.zeros((2, 6)))
    y = np.arange(12.0).reshape(2, 6)
    rs = O.reduce_scatter_blocks(y, 3)
    assert rs.shape == (3, 2, 2) and np.array_equal(rs[1], [[2, 3], [8, 9]])


# ----------------------------------------------------------------- heads/GQA

def _copies(n_q, n_kv, tp):
    m = O.head_shard_map(n_q, n_kv, tp)
    counts = {g: 0 for g in range(n_kv)}
    for _, kv in m:
        for g in kv:
            counts[g] += 1
    return set(counts.values())


def test_kv_copies_match_worked_numbers():
    g = golden()
    for tp in (1, 2, 4, 8):
        assert _copies(64, 8, tp) == {int(g["s44.llama70b_kv_copies_tp8"][0])}
    assert _copies(64, 8, 16) == {int(g["s44.llama70b_kv_copies_tp16"][0])}
    assert _copies(64, 1, 8) == {int(g["s44.mqa_kv_copies_tp8"][0])}
    assert _copies(8, 2, 4) == {2}          # the lecture's small model, 4 devices
    with pytest.raises(ValueError):
        O.head_shard_map(12, 2, 5)           # Q heads not divisible
    with pytest.raises(ValueError):
        O.head_shard_map(12, 4, 6)           # tp > n_kv but not a multiple


def test_head_map_tp1_is_unsharded_and_groups_follow_gqa():
    rows = O.qkv_rows_of_shard(12, 2, 4, 1, 0)
    assert np.array_equal(rows, np.arange((12 + 4) * 4))
    # GQA: consecutive blocks of n_q/n_kv query heads share one KV group
    assert [O.kv_group_of_head(h, 12, 2) for h in range(12)] == [0] * 6 + [1] * 6
    assert [O.kv_group_of_head(h, 64, 8) for h in range(0, 64, 8)] == list(range(8))
    # Qwen-shaped tp=2: shard 1 owns Q heads 6..11 and KV group 1
    q, kv = O.head_shard_map(12, 2, 2)[1]
    assert q == list(range(6, 12)) and kv == [1]
    rows = O.qkv_rows_of_shard(12, 2, 4, 2, 1)
    exp = list(range(24, 48)) + list(range(13 * 4, 14 * 4)) + list(range(15 * 4, 16 * 4))
    assert rows.tolist() == exp


def test_context1_attention_is_value_of_group():
    """Softmax over a single key is 1: each head returns its group's value vector."""
    r = rng(9)
    B, n_q, n_kv, hd = 3, 6, 2, 4
    Q, K, V = r.standard_normal((B, n_q * hd)), r.standard_normal((B, n_kv * hd)), r.standard_normal((B, n_kv * hd))
    Oa = O.context1_attention(Q, K, V, n_q, [0, 1], list(range(n_q)), n_q, n_kv, hd)
    for h in range(n_q):
        g = h // 3
        assert np.allclose(Oa[:, h * hd:(h + 1) * hd], V[:, g * hd:(g + 1) * hd], rtol=1e-15, atol=0)


def test_attention_sharded_equals_unsharded_on_integers():
    r = rng(10)
    B, D, n_q, n_kv, hd = 2, 16, 8, 2, 4
    X = r.integers(-2, 3, (B, D)).astype(float)
    Wqkv = r.integers(-1, 2, ((n_q + 2 * n_kv) * hd, D)).astype(float)
    Wo = r.integers(-1, 2, (D, n_q * hd)).astype(float)
    Y, QKV = O.attn_proj_unsharded(X, Wqkv, Wo, n_q, n_kv, hd, bf16=False)
    for tp in (1, 2, 4, 8):
        Ys, QKVs, Os, Ps = O.attn_proj_sharded(X, Wqkv, Wo, n_q, n_kv, hd, tp, bf16=False)
        assert np.array_equal(Ys, Y)
        for s in range(tp):
            assert np.array_equal(QKVs[s], QKV[:, O.qkv_rows_of_shard(n_q, n_kv, hd, tp, s)])
    # brute force of the whole projection path on the same data
    Vfull = QKV[:, (n_q + n_kv) * hd:]
    Ob = np.concatenate([Vfull[:, (h * n_kv // n_q) * hd:(h * n_kv // n_q + 1) * hd] for h in range(n_q)], axis=1)
    assert np.array_equal(Y, np.array(_brute_linear(Ob.tolist(), Wo.tolist())))


# -------------------------------------------------------------- four cases

def _ab(seed, I=16, J=24, K=32, integer=False):
    r = rng(seed)
    if integer:
        return r.integers(-2, 3, (I, J)).astype(float), r.integers(-2, 3, (K, J)).astype(float)
    return r.standard_normal((I, J)), r.standard_normal((K, J))


def test_case1_case2_case4B_are_the_product():
    A, Bt = _ab(11, integer=True)
    C = np.array(_brute_linear(A.tolist(), Bt.tolist()))
    for X in (1, 2, 4, 8):
        for case, kw in ((1, {}), (2, {}), (4, dict(gather="B"))):
            got, part = O.sharded_matmul(case, A, Bt, X, bf16=False, **kw)
            assert part is None and np.array_equal(got, C)


def test_case3_partials_sum_and_reduce_scatter_blocks():
    A, Bt = _ab(12, integer=True)
    C = np.array(_brute_linear(A.tolist(), Bt.tolist()))
    for X in (2, 4, 8):
        ar, P = O.sharded_matmul(3, A, Bt, X, mode="allreduce", bf16=False)
        assert np.array_equal(ar, C) and len(P) == X
        # each partial only sees its own slice of J
        js = O.shard_range(24, X, 1)
        assert np.array_equal(P[1], np.array(_brute_linear(A[:, js.start:js.stop].tolist(),
                                                           Bt[:, js.start:js.stop].tolist())))
        rs, _ = O.sharded_matmul(3, A, Bt, X, mode="reducescatter", bf16=False)
        for s in range(X):
            ks = O.shard_range(32, X, s)
            assert np.array_equal(rs[s], C[:, ks.start:ks.stop])


def test_case4_local_product_gives_only_diagonal_blocks_and_gather_A():
    A, Bt = _ab(13)
    C = A @ Bt.T
    X = 4
    blocks = O.case4_local_blocks(A, Bt, X)
    for d in range(X):
        i, k = O.shard_range(16, X, d), O.shard_range(32, X, d)
        assert np.allclose(blocks[d], C[i.start:i.stop, k.start:k.stop], rtol=1e-13, atol=1e-13)
    ga, _ = O.sharded_matmul(4, A, Bt, X, gather="A", bf16=False)
    for s in range(X):
        k = O.shard_range(32, X, s)
        assert np.allclose(ga[s], C[:, k.start:k.stop], rtol=1e-13, atol=1e-13)


def test_case_costs_match_worked_numbers():
    g = golden()
    I, J, K, n = 512, 8192, 28672, 8
    gB = acc.case_comm_bytes(4, I, J, K, n, gather="B")
    gA = acc.case_comm_bytes(4, I, J, K, n, gather="A")
    assert round(float(gB) / 1e6) == g["case4.gather_B"][0]
    assert round(float(gA) / 1e6) == g["case4.gather_A"][0]
    assert Fraction(I * K, I * J) == Fraction(g["case3.C_over_A"][0]).limit_denominator(10)
    ratio = acc.case_comm_bytes(3, I, J, K, n) / acc.case_comm_bytes(2, I, J, K, n)
    assert ratio == g["case3.comm_over_case2"][0]
    assert acc.case_comm_bytes(1, I, J, K, n) == 0


def test_shard_and_message_sizes_match_worked_numbers():
    g = golden()
    a = acc.shard_bytes((64, 8192), {1}, 8)
    w = acc.shard_bytes((8192, 28672), {0}, 8)
    assert round(a / 1e3) == g["ex1.A_shard"][0] and round(w / 1e6, 1) == g["ex1.W_shard"][0]
    msg = acc.allreduce_message_bytes(32, 4096)
    assert msg == g["ex3.message"][0]
    ring = acc.ring_allreduce_bytes_per_device(msg, 4)
    assert round(float(ring) / 1e3) == g["ex3.ring_per_allreduce"][0]
    per_step = ring * 32 * g["s42.allreduces_per_layer"][0]
    assert round(float(per_step) / 1e6, 1) == g["ex3.ring_per_step"][0]
    assert round(acc.allreduce_message_bytes(64, 8192) / 1e6, 2) == g["s45.allreduce_message"][0]
    assert round(acc.allreduce_message_bytes(256, 8192) / 1e6) == g["s61.message_B256"][0]


def test_layer_byte_counts():
    # Qwen2.5-1.5B-shaped: 93,585,408 B of projection weights per layer
    assert acc.layer_weight_bytes(1536, 8960, 12, 2, 128) == 93_585_408
    assert acc.layer_weight_bytes(8192, 28672, 64, 8, 128) == 1_711_276_032
    assert acc.mlp_flops(4096, 8192, 28672) == 5_772_436_045_824


# ------------------------------------------------------------------ layer

def test_rmsnorm_closed_forms():
    y = O.rmsnorm(np.array([[3.0, 4.0]]), eps=0.0)
    assert np.allclose(y, [[3 / math.sqrt(12.5), 4 / math.sqrt(12.5)]], rtol=1e-15)
    c = 0.01
    y = O.rmsnorm(np.full((1, 5), c))
    assert np.allclose(y, 1 / math.sqrt(1 + O.RMS_EPS / c ** 2), rtol=1e-15)


def test_decoder_layer_zero_output_projections_is_identity():
    r = rng(14)
    D, F, n_q, n_kv, hd = 16, 32, 4, 2, 4
    x = O.bf16_round(r.standard_normal((3, D)))
    W = dict(Wqkv=r.standard_normal(((n_q + 2 * n_kv) * hd, D)), Wo=np.zeros((D, n_q * hd)),
             Wg=r.standard_normal((F, D)), Wu=r.standard_normal((F, D)), Wd=np.zeros((D, F)))
    assert np.array_equal(O.decoder_layer(x, W, n_q, n_kv, hd, tp=2), x)
    # with only the MLP silenced the layer adds the attention sublayer once
    W["Wo"] = r.standard_normal((D, n_q * hd)) / 8
    y = O.decoder_layer(x, W, n_q, n_kv, hd, tp=2)
    a, _ = O.attn_proj_unsharded(O.rmsnorm(x), W["Wqkv"], W["Wo"], n_q, n_kv, hd, bf16=False)
    assert np.allclose(y, O.bf16_round(x + a), rtol=0, atol=2 ** -7 * np.abs(x + a).max())


def _serial_layer_with_silenced_attention():
    """[L4] S5.5 block formula, serial form, attention output projection zero:
    h = x exactly, so y = bf16(x + MLP(RMSNorm(x))), with the MLP written out
    here in plain loops (no shards; SiLU from math.exp; H rounded to bf16)."""
    r = rng(17)
    D, F, n_q, n_kv, hd = 12, 20, 4, 2, 3
    x = O.bf16_round(r.standard_normal((2, D)) * 1.5)
    W = dict(Wqkv=r.standard_normal(((n_q + 2 * n_kv) * hd, D)), Wo=np.zeros((D, n_q * hd)),
             Wg=r.standard_normal((F, D)) / 3, Wu=r.standard_normal((F, D)) / 3, Wd=r.standard_normal((D, F)) / 4)
    ref = np.zeros_like(x)
    for t in range(x.shape[0]):
        ms = sum(float(v) * float(v) for v in x[t]) / D
        inv = 1.0 / math.sqrt(ms + O.RMS_EPS)
        xn = [float(v) * inv for v in x[t]]
        H = []
        for f in range(F):
            g = sum(W["Wg"][f, d] * xn[d] for d in range(D))
            u = sum(W["Wu"][f, d] * xn[d] for d in range(D))
            H.append(float(O.bf16_round(np.array(g / (1.0 + math.exp(-g)) * u))))
        for d in range(D):
            ref[t, d] = x[t, d] + sum(W["Wd"][d, f] * H[f] for f in range(F))
    ref = O.bf16_round(ref)
    return x, W, ref, (n_q, n_kv, hd)


def _serial_mlp_pin_holds(x, W, ref, dims, tp):
    y = O.decoder_layer(x, W, *dims, tp=tp)
    # one bf16 rounding of nearby values (sum order only) may differ by an ulp
    return bool(np.all(np.abs(y - ref) <= 2 ** -7 * np.abs(ref) + 1e-12))


def test_serial_layer_mlp_branch_pin():
    x, W, ref, dims = _serial_layer_with_silenced_attention()
    for tp in (1, 2, 4):
        assert _serial_mlp_pin_holds(x, W, ref, dims, tp), tp


def test_serial_layer_mlp_branch_pin_catches_planted_mistakes(monkeypatch):
    x, W, ref, dims = _serial_layer_with_silenced_attention()
    real_norm, real_silu, real_hidden = O.rmsnorm, O.silu, O.mlp_hidden_shard
    monkeypatch.setattr(O, "rmsnorm", lambda v, eps=O.RMS_EPS: np.asarray(v, dtype=np.float64))  # norm dropped
    assert not _serial_mlp_pin_holds(x, W, ref, dims, 2)
    monkeypatch.setattr(O, "rmsnorm", real_norm)
    monkeypatch.setattr(O, "silu", lambda z: np.asarray(z, dtype=np.float64))                     # SiLU dropped
    assert not _serial_mlp_pin_holds(x, W, ref, dims, 2)
    monkeypatch.setattr(O, "silu", real_silu)

    def swapped(X, Wg, Wu, tp, s, bf16=True):                                                  # gate <-> up
        return real_hidden(X, Wu, Wg, tp, s, bf16)
    monkeypatch.setattr(O, "mlp_hidden_shard", swapped)
    assert not _serial_mlp_pin_holds(x, W, ref, dims, 2)
    monkeypatch.setattr(O, "mlp_hidden_shard", real_hidden)
    assert _serial_mlp_pin_holds(x, W, ref, dims, 2)


def test_parallel_block_reduces_to_its_sublayers():
    """[L4] S5.5 parallel block: silencing one sublayer's output projection leaves
    x plus the other sublayer on RMSNorm(x), each computed here without shards."""
    r = rng(16)
    D, F, n_q, n_kv, hd = 16, 32, 4, 2, 4
    x = O.bf16_round(r.standard_normal((3, D)))
    W = dict(Wqkv=r.standard_normal(((n_q + 2 * n_kv) * hd, D)) / 4, Wo=r.standard_normal((D, n_q * hd)) / 8,
             Wg=r.standard_normal((F, D)) / 4, Wu=r.standard_normal((F, D)) / 4, Wd=r.standard_normal((D, F)) / 8)
    xn = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + O.RMS_EPS)
    attn, _ = O.attn_proj_unsharded(xn, W["Wqkv"], W["Wo"], n_q, n_kv, hd, bf16=True)
    g, u = xn @ W["Wg"].T, xn @ W["Wu"].T
    mlp = O.bf16_round(g / (1 + np.exp(-g)) * u) @ W["Wd"].T
    tol = lambda ref: 2 ** -7 * np.abs(ref) + 1e-9   # noqa: E731  (one bf16 rounding, sum order)
    W0 = dict(W, Wo=np.zeros_like(W["Wo"]))
    ref = O.bf16_round(x + mlp)
    assert np.all(np.abs(O.decoder_layer_parallel(x, W0, n_q, n_kv, hd, tp=2) - ref) <= tol(ref))
    W1 = dict(W, Wd=np.zeros_like(W["Wd"]))
    ref = O.bf16_round(x + attn)
    assert np.all(np.abs(O.decoder_layer_parallel(x, W1, n_q, n_kv, hd, tp=2) - ref) <= tol(ref))
    ref = O.bf16_round(x + attn + mlp)
    assert np.all(np.abs(O.decoder_layer_parallel(x, W, n_q, n_kv, hd, tp=2) - ref) <= tol(ref))
    # and it is not the serial block: there the MLP sees RMSNorm(x + attn)
    assert np.abs(O.decoder_layer_parallel(x, W, n_q, n_kv, hd, tp=2)
                  - O.decoder_layer(x, W, n_q, n_kv, hd, tp=2)).max() > 1e-3


def test_decoder_stack_sharded_matches_unsharded():
    r = rng(15)
    D, F, n_q, n_kv, hd = 32, 64, 8, 2, 4
    x = r.standard_normal((2, D))
    layers = [dict(Wqkv=r.standard_normal(((n_q + 2 * n_kv) * hd, D)) * 0.1,
                   Wo=r.standard_normal((D, n_q * hd)) * 0.1, Wg=r.standard_normal((F, D)) * 0.1,
                   Wu=r.standard_normal((F, D)) * 0.1, Wd=r.standard_normal((D, F)) * 0.1) for _ in range(3)]
    ys = O.decoder_stack(x, layers, n_q, n_kv, hd, tp=4, sharded=True)
    yu = O.decoder_stack(x, layers, n_q, n_kv, hd, tp=4, sharded=False)
    rms = np.sqrt(np.mean(yu ** 2))
    assert np.max(np.abs(ys - yu)) <= 1e-2 * rms


# ---------------------------------------------- planted mistakes are caught

def test_planted_mistakes_fail_a_pin(monkeypatch):
    """Swap gate and up inside the oracle: the hand-worked example must fail."""
    real = O.mlp_unsharded

    def swapped(X, Wg, Wu, Wd, bf16=True):
        return real(X, Wu, Wg, Wd, bf16)
    monkeypatch.setattr(O, "mlp_unsharded", swapped)
    with pytest.raises(AssertionError):
        test_mlp_hand_worked_example()
    monkeypatch.setattr(O, "mlp_unsharded", real)

    # a partial sum that drops the last shard must fail the row-parallel identity
    real_reduce = O.shard_reduce
    monkeypatch.setattr(O, "shard_reduce", lambda P, bf16=False: real_reduce(P[:-1] if len(P) > 1 else P, bf16))
    with pytest.raises(AssertionError):
        test_row_parallel_sum_is_exact_on_integers()
    monkeypatch.setattr(O, "shard_reduce", real_reduce)

    # an off-by-one KV group map must fail the GQA pins
    real_g = O.kv_group_of_head
    monkeypatch.setattr(O, "kv_group_of_head", lambda h, n_q, n_kv: min(n_kv - 1, ((h + 1) * n_kv) // n_q))
    with pytest.raises((AssertionError, ValueError)):
        test_head_map_tp1_is_unsharded_and_groups_follow_gqa()
    monkeypatch.setattr(O, "kv_group_of_head", real_g)


@pytest.mark.parametrize("D", [16, 32, 48])
@pytest.mark.parametrize("F", [16, 32, 48])
@pytest.mark.parametrize("B", [1, 3, 8])
def test_sharded_and_unsharded_agree_over_tiny_shapes(D, F, B):
    """Every divisor of F as the shard count: the sharded MLP (per-shard H and
    partials, summed in shard order) equals the unsharded one to fp64
    rounding, and the partials sum to it exactly on integer data."""
    r = rng(100 + D + F + B)
    X = r.standard_normal((B, D))
    Wg, Wu = r.standard_normal((F, D)) * 0.2, r.standard_normal((F, D)) * 0.2
    Wd = r.standard_normal((D, F)) * 0.2
    Y = O.mlp_unsharded(X, Wg, Wu, Wd, bf16=False)
    Hi = r.integers(-2, 3, (B, F)).astype(float)
    Wdi = r.integers(-2, 3, (D, F)).astype(float)
    for tp in [t for t in range(1, F + 1) if F % t == 0]:
        Ys, P, _ = O.mlp_sharded(X, Wg, Wu, Wd, tp, bf16=False)
        assert np.allclose(Ys, Y, rtol=1e-12, atol=1e-12)
        Pi = [O.mlp_partial_shard(Hi[:, O.shard_range(F, tp, s).start:O.shard_range(F, tp, s).stop], Wdi, tp, s)
              for s in range(tp)]
        assert np.array_equal(O.shard_reduce(Pi), Hi @ Wdi.T)
