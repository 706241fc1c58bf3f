"""Pins for the vocabulary-parallel lm_head oracle (no GPU).

Each check ties the oracle to something other than itself: the message size
the lecture prints (tests/golden/worked_examples.txt), brute force in plain
Python loops on tiny inputs, numpy's argmax and a full sort as independent
library routes, and exact ties constructed so the order is known in advance.
"""
import numpy as np
import pytest

from oracle import vocab_head as VH
from test_oracle_pins import golden


def _brute_topk(x, W, k):
    """Plain loops: every logit as an explicit sum, ranking by repeated
    selection of the best remaining (value, then lower index)."""
    out = []
    for b in range(len(x)):
        scores = []
        for v in range(len(W)):
            s = 0.0
            for d in range(len(x[b])):
                s += float(x[b][d]) * float(W[v][d])
            scores.append(s)
        chosen = []
        for _ in range(k):
            best = None
            for v, s in enumerate(scores):
                if v in chosen:
                    continue
                if best is None or s > scores[best]:
                    best = v
            chosen.append(best)
        out.append(chosen)
    return np.array(out)


def test_logit_message_size_matches_lecture():
    g = golden()
    gathered = VH.exchange_bytes(64, 128256, 8, 1, "gather")
    assert round(gathered / 1e6, 2) == g["s45.logits_B64"][0]
    # exchanging one (index, bf16 logit) candidate per shard and token instead
    cand = VH.exchange_bytes(64, 128256, 8, 1, "topk")
    assert cand == 8 * 64 * 6 and gathered / cand > 5000


@pytest.mark.parametrize("tp,k", [(1, 1), (2, 3), (3, 2), (4, 3)])
def test_candidate_exchange_equals_brute_force(tp, k):
    r = np.random.default_rng(10 + tp)
    B, D, V = 3, 5, 12
    x = r.integers(-3, 4, size=(B, D)).astype(float)
    W = r.integers(-3, 4, size=(V, D)).astype(float)
    idx, val, sidx, sval = VH.vocab_parallel_topk(x, W, tp, k)
    assert np.array_equal(idx, _brute_topk(x.tolist(), W.tolist(), k))
    for b in range(B):
        for j in range(k):
            assert val[b, j] == sum(x[b, d] * W[idx[b, j], d] for d in range(D))
    # each shard's list holds only its own rows, ranked the same way
    vs = V // tp
    for s in range(tp):
        Ws = W[s * vs:(s + 1) * vs]
        assert np.array_equal(sidx[s], _brute_topk(x.tolist(), Ws.tolist(), k) + s * vs)


def test_top1_is_numpy_argmax_and_topk_is_a_full_sort():
    r = np.random.default_rng(3)
    B, D, V, tp, k = 6, 64, 1000, 8, 5
    x = r.standard_normal((B, D))
    W = r.standard_normal((V, D)) * 0.02
    full = np.einsum("bd,vd->bv", x, W)
    idx1, val1, _, _ = VH.vocab_parallel_topk(x, W, tp, 1)
    assert np.array_equal(idx1[:, 0], np.argmax(full, axis=1))
    idx, val, _, _ = VH.vocab_parallel_topk(x, W, tp, k)
    ref = np.argsort(-full, axis=1, kind="stable")[:, :k]
    assert np.array_equal(idx, ref)
    assert np.allclose(val, np.take_along_axis(full, ref, 1), rtol=0, atol=1e-12)
    # the all-gather route reproduces the unsharded logits
    assert np.allclose(VH.gathered_logits(x, W, tp), full, rtol=0, atol=1e-12)


def test_maximum_in_a_late_shard_keeps_its_global_index():
    # a dropped shard offset would report the local row instead
    D, V, tp = 4, 16, 4
    W = np.zeros((V, D))
    W[13] = [1, 0, 0, 0]
    x = np.array([[2.0, 0, 0, 0]])
    idx, val, sidx, _ = VH.vocab_parallel_topk(x, W, tp, 1)
    assert idx[0, 0] == 13 and val[0, 0] == 2.0
    assert sidx[3, 0, 0] == 13 and sidx[0, 0, 0] == 0


def test_ties_go_to_the_lower_index_within_and_across_shards():
    D, V, tp, k = 3, 18, 3, 4
    W = np.zeros((V, D))
    W[[2, 5, 9, 14]] = [1.0, 1.0, 0.0]     # equal rows: two in shard 0, one each in 1 and 2
    W[7] = [0.5, 0.5, 0.0]
    x = np.array([[1.0, 1.0, 0.0]])
    idx, val, _, _ = VH.vocab_parallel_topk(x, W, tp, k)
    assert idx.tolist() == [[2, 5, 9, 14]] and val.tolist() == [[2.0] * 4]
    idx, _, _, _ = VH.vocab_parallel_topk(x, W, tp, 6)
    assert idx[0, 4] == 7 and idx[0, 5] == 0   # then 1.0, then the lowest zero


def test_zero_input_ranks_by_index_and_signed_zeros_are_equal():
    D, V, tp, k = 4, 8, 2, 3
    W = np.random.default_rng(0).standard_normal((V, D))
    idx, val, _, _ = VH.vocab_parallel_topk(np.zeros((2, D)), W, tp, k)
    assert idx.tolist() == [[0, 1, 2]] * 2 and np.all(val == 0)
    i, v = VH.ordered_topk(np.array([-0.0, 0.0, -0.0]), 3)
    assert i.tolist() == [0, 1, 2]


def test_shape_rules():
    with pytest.raises(ValueError):
        VH.vocab_shards(10, 3)
    with pytest.raises(ValueError):
        VH.vocab_parallel_topk(np.ones((1, 2)), np.ones((8, 2)), 4, 3)   # k > V/tp
    assert VH.vocab_shards(151936, 2) == [(0, 75968), (75968, 151936)]
