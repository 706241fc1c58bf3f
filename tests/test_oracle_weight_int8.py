"""Pins for the weight-only int8 oracle (no GPU): a hand-worked quantisation,
the rounding rule against Python's own round(), the error bound of rounding to
the nearest step, exact identities of the int8 layer with the (pinned) bf16
layer oracle, and the bytes-halved claim of the lecture."""
import numpy as np
import pytest

from oracle import tp_layer as O
from oracle import weight_int8 as W8


def test_hand_worked_row_with_unit_scale():
    # amax 127 gives s = 1 exactly, so q = round(w): ties go to the even integer
    w = np.array([[127.0, 2.5, -3.5, 0.5, 1.5, -127.0, 0.0, 99.25]])
    q, s = W8.quantize_rows(w)
    assert s.tolist() == [[1.0]]
    assert q.tolist() == [[127, 2, -4, 0, 2, -127, 0, 99]]


def test_rounding_matches_python_round_and_the_half_step_bound():
    r = np.random.default_rng(5)
    W = (r.standard_normal((40, 96)) * 0.02).astype(np.float32)
    W = np.asarray(W, dtype=np.float32)
    q, s = W8.quantize_rows(W, groups=3)
    for i in range(40):
        for g in range(3):
            cols = slice(32 * g, 32 * (g + 1))
            amax = max(abs(float(v)) for v in W[i, cols])
            sc = float(np.float32(amax) / np.float32(127))
            assert s[i, g] == np.float32(sc)
            for j in range(32 * g, 32 * (g + 1)):
                ratio = float(np.float32(W[i, j]) / np.float32(sc))
                assert q[i, j] == max(-127, min(127, round(ratio)))          # Python rounds half to even
                assert abs(q[i, j] * sc - W[i, j]) <= sc / 2 * (1 + 1e-6)    # nearest step
            # the largest magnitude lands on +-127
            jm = 32 * g + int(np.argmax(np.abs(W[i, cols])))
            assert abs(int(q[i, jm])) == 127


def test_zero_group_and_shape_rules():
    W = np.zeros((2, 8))
    W[1, 4:] = [0.5, -1.0, 0.25, 0.0]
    q, s = W8.quantize_rows(W, groups=2)
    assert s[0].tolist() == [0.0, 0.0] and s[1, 0] == 0.0 and np.all(q[0] == 0) and np.all(q[1, :4] == 0)
    assert q[1, 4:].tolist() == [64, -127, 32, 0]       # 0.5 / s is 63.5 in float32: a tie, to the even 64
    with pytest.raises(ValueError):
        W8.quantize_rows(np.ones((2, 9)), groups=2)


def test_int8_layer_with_unit_scales_is_the_bf16_layer_on_integer_weights():
    r = np.random.default_rng(2)
    B, D, F, tp = 3, 16, 24, 2
    X = O.bf16_round(r.standard_normal((B, D)))
    Qg, Qu = (r.integers(-127, 128, (F, D)).astype(np.int8) for _ in range(2))
    Qd = r.integers(-127, 128, (D, F)).astype(np.int8)
    ones_f, ones_d = np.ones((F, 1), np.float32), np.ones((D, tp), np.float32)
    Y, P, H = W8.mlp_sharded_w8(X, Qg, ones_f, Qu, ones_f, Qd, ones_d, tp)
    Y2, P2, H2 = O.mlp_sharded(X, Qg.astype(float), Qu.astype(float), Qd.astype(float), tp)
    assert np.array_equal(Y, Y2) and all(np.array_equal(a, b) for a, b in zip(P, P2))


def test_per_shard_scales_scale_only_their_own_shard():
    # a row-parallel weight quantised per shard: doubling shard 1's scale
    # doubles P_1 and leaves P_0 alone
    r = np.random.default_rng(4)
    B, D, F, tp = 2, 8, 16, 2
    X = O.bf16_round(r.standard_normal((B, D)))
    Qg, Qu = (r.integers(-127, 128, (F, D)).astype(np.int8) for _ in range(2))
    Qd = r.integers(-127, 128, (D, F)).astype(np.int8)
    sg = su = np.full((F, 1), 2.0 ** -7, np.float32)
    sd = np.full((D, tp), 2.0 ** -9, np.float32)
    _, P, _ = W8.mlp_sharded_w8(X, Qg, sg, Qu, su, Qd, sd, tp)
    sd2 = sd.copy()
    sd2[:, 1] *= 2
    _, P2, _ = W8.mlp_sharded_w8(X, Qg, sg, Qu, su, Qd, sd2, tp)
    assert np.array_equal(P2[0], P[0]) and np.array_equal(P2[1], 2 * P[1])


def test_quantised_layer_stays_close_to_the_bf16_layer():
    # the rounding error of each weight is at most half a step, so the int8 layer
    # tracks the bf16 one (a sanity bound, not a parity tolerance)
    r = np.random.default_rng(8)
    B, D, F, tp = 4, 64, 128, 2
    X = O.bf16_round(r.standard_normal((B, D)))
    Wg, Wu = (O.bf16_round(r.standard_normal((F, D)) * 0.02) for _ in range(2))
    Wd = O.bf16_round(r.standard_normal((D, F)) * 0.02)
    Qg, sg = W8.quantize_rows(Wg)
    Qu, su = W8.quantize_rows(Wu)
    Qd, sd = W8.quantize_rows(Wd, groups=tp)
    Y8 = W8.mlp_sharded_w8(X, Qg, sg, Qu, su, Qd, sd, tp, bf16=False)[0]
    Y = O.mlp_sharded(X, Wg, Wu, Wd, tp, bf16=False)[0]
    rms = np.sqrt(np.mean(Y ** 2))
    assert np.max(np.abs(Y8 - Y)) < 0.05 * rms


def test_int8_weights_take_half_the_bytes():
    for D, F, tp in ((1536, 8960, 2), (8192, 28672, 8)):
        bf16 = 3 * D * F * 2
        b8 = W8.weight_bytes_int8(D, F, tp)
        assert 0.5 < b8 / bf16 < 0.502
