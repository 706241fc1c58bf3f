"""Parity of the vocabulary-parallel lm_head (per-shard top-k, then the
candidate exchange) with the oracle, through the C ABI.

The kernel ranks fp32 logits that it accumulates itself; the oracle ranks the
exact (fp64) logits.  Any fp32 summation of D exact products differs from the
exact sum by at most (D - 1) 2^-24 sum|x_d W_vd|; the tolerance below takes
twice that.  So the checks are:
  * each returned logit is the oracle's logit of the returned index within the
    tolerance;
  * the returned list is ordered (larger first, equal values by lower index);
  * no vocabulary entry left out is certainly larger than the k-th returned;
  * the j-th returned logit is within the largest allowance of the exact j-th
    largest (an order statistic moves no further than its inputs);
  * wherever the oracle's ranking is unambiguous at that resolution (gaps to
    both neighbours above the tolerance), the index is the oracle's exactly --
    at most positions for these inputs, and the test requires a share of them.
Constructed exact ties (identical rows) and the zero input fix the order
bit for bit.
"""
import numpy as np
import pytest
import torch

import synthetic_inputs as si
from oracle import vocab_head as VH

pytestmark = pytest.mark.gpu
tpl = pytest.importorskip("mlp_megatron_tp_layer_b300")

TOL_ULP = 2.0 ** -23


@pytest.fixture(autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.synchronize()
    yield
    torch.cuda.synchronize()
    assert tpl.device_status() == 0, "a device-side wait timed out"


def _np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def exact_logits(x64, W, rows=None, chunk=16384):
    """fp64 logits and the rounding allowance per element, for the tokens
    ``rows`` of x64 (all if None), streaming W from the device in chunks."""
    xs = x64 if rows is None else x64[rows]
    V, D = W.shape
    L = np.empty((xs.shape[0], V))
    A = np.empty((xs.shape[0], V))
    for a in range(0, V, chunk):
        Wc = _np(W[a:a + chunk])
        L[:, a:a + chunk] = xs @ Wc.T
        A[:, a:a + chunk] = np.abs(xs) @ np.abs(Wc).T
    return L, (D - 1) * TOL_ULP * A


def check_ranked(idx, val, L, tol, lo, hi, k, stats):
    """One token's returned top-k against exact logits L (vocabulary rows lo..hi)."""
    assert len(set(idx.tolist())) == k, idx
    assert np.all((idx >= lo) & (idx < hi)), idx
    assert np.all(np.abs(val - L[idx]) <= tol[idx]), (val, L[idx], tol[idx])
    for j in range(k - 1):
        assert val[j] > val[j + 1] or (val[j] == val[j + 1] and idx[j] < idx[j + 1]), (idx, val)
    # nothing excluded is certainly above the k-th returned
    excl = np.ones(hi - lo, bool)
    excl[idx - lo] = False
    last = idx[-1]
    if excl.any():
        assert np.max((L[lo:hi] - tol[lo:hi])[excl]) <= L[last] + tol[last]
    # positions the exact ranking fixes at this resolution must match exactly
    ref_i, ref_v = VH.ordered_topk(L[lo:hi], min(k + 1, hi - lo), offset=lo)
    margin = 2.0 * np.max(tol[lo:hi])
    # the j-th largest moves by at most the largest perturbation of any entry
    assert np.all(np.abs(val - ref_v[:k]) <= margin / 2), (val, ref_v)
    for j in range(k):
        above = j == 0 or ref_v[j - 1] - ref_v[j] > margin
        below = j + 1 >= len(ref_v) or ref_v[j] - ref_v[j + 1] > margin
        if above and below:
            stats["exact"] += 1
            assert idx[j] == ref_i[j], (j, idx, ref_i)
        stats["all"] += 1


def check_against_oracle(x, W, tp, k, got, rows=None, min_exact=0.9):
    idx, val, sidx, sval = (g.cpu().numpy() for g in got)
    x64 = _np(x)
    rows = np.arange(x.shape[0]) if rows is None else np.asarray(rows)
    L, tol = exact_logits(x64, W, rows)
    V = W.shape[0]
    stats = {"exact": 0, "all": 0}
    for r, b in enumerate(rows):
        check_ranked(idx[b], val[b].astype(np.float64), L[r], tol[r], 0, V, k, stats)
        for s, (lo, hi) in enumerate(VH.vocab_shards(V, tp)):
            check_ranked(sidx[s, b], sval[s, b].astype(np.float64), L[r], tol[r], lo, hi, k, stats)
        # the exchange: every final candidate comes from some shard's list
        assert set(idx[b].tolist()) <= set(sidx[:, b, :].reshape(-1).tolist())
    assert stats["exact"] >= min_exact * stats["all"], stats
    return stats


@pytest.mark.parametrize("B,D,V,tp,k", [
    (5, 256, 4000, 4, 1),      # 8 tiles per shard, last one 104 rows
    (5, 256, 4000, 4, 8),
    (1, 64, 96, 2, 3),         # shard smaller than one tile
    (40, 520, 3000, 3, 2),     # ragged K tail (520 = 8 x 64 + 8), 64-token tile
    (17, 136, 2048, 8, 5),     # 32-token tile with 15 padded columns
    (130, 128, 2048, 8, 4),    # two token tiles
    (128, 1536, 20000, 2, 1),
])
def test_vocab_topk_matches_oracle(B, D, V, tp, k):
    x, W = si.lm_head(B, D, V, seed=B + k, device="cuda")
    got = tpl.vocab_parallel_topk(x, W, tp, k, shard_outputs=True)
    check_against_oracle(x, W, tp, k, got)


def test_vocab_topk_is_deterministic_and_fills_given_outputs():
    x, W = si.lm_head(24, 512, 6000, seed=3, device="cuda")
    a = tpl.vocab_parallel_topk(x, W, 4, 6, shard_outputs=True)
    out = (torch.full((24, 6), -7, dtype=torch.int32, device="cuda"),
           torch.full((24, 6), float("nan"), device="cuda"))
    b = tpl.vocab_parallel_topk(x, W, 4, 6, shard_outputs=True, out=out)
    assert b[0] is out[0] and b[1] is out[1]
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    # without shard outputs the same final answer
    c = tpl.vocab_parallel_topk(x, W, 4, 6)
    assert torch.equal(c[0], a[0]) and torch.equal(c[1], a[1])


def test_vocab_topk_graph_replays_rank_each_replays_inputs():
    """Captured in a CUDA graph, where the merge kernel is a programmatic
    dependent of the GEMM: every replay ranks the inputs written before it,
    exactly as an eager call on them does (a merge that read the candidates
    before the GEMM completed would return the previous replay's answer)."""
    B, D, V, tp, k = 5, 512, 6000, 2, 3
    x, W = si.lm_head(B, D, V, seed=11, device="cuda")
    fresh = [si.lm_head(B, D, V, seed=20 + i, device="cuda")[0] for i in range(3)]
    idx = torch.empty(B, k, dtype=torch.int32, device="cuda")
    val = torch.empty(B, k, dtype=torch.float32, device="cuda")
    ws = tpl.workspace(tpl.vocab_topk_workspace_bytes(B, V, tp, k), torch.device("cuda"))
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        tpl.vocab_parallel_topk(x, W, tp, k, out=(idx, val), ws=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        tpl.vocab_parallel_topk(x, W, tp, k, out=(idx, val), ws=ws)
    for xn in fresh:
        x.copy_(xn)
        g.replay()
        torch.cuda.synchronize()
        want_idx, want_val = tpl.vocab_parallel_topk(xn, W, tp, k)
        assert torch.equal(idx, want_idx) and torch.equal(val, want_val)
    del g


def test_exact_ties_resolve_to_the_lower_index_across_tiles_and_shards():
    B, D, V, tp = 3, 256, 4096, 4
    x, W = si.lm_head(B, D, V, seed=7, device="cuda")
    # one row clearly above every random row, copied into several tiles and shards
    top = (x[0].float() * 0.05).to(torch.bfloat16)
    ties = [5, 300, 1023, 1024, 2999, 4095]
    W[ties] = top
    idx, val, sidx, sval = tpl.vocab_parallel_topk(x, W, tp, 4, shard_outputs=True)
    assert idx[0].tolist() == ties[:4]
    assert len(set(val[0].tolist())) == 1                 # identical rows, identical fp32 logits
    assert sidx[0, 0, :2].tolist() == [5, 300] and sidx[1, 0, 0].item() == 1024
    assert sidx[2, 0, 0].item() == 2999 and sidx[3, 0, 0].item() == 4095
    idx8, _ = tpl.vocab_parallel_topk(x, W, tp, 8)
    assert idx8[0, :6].tolist() == ties


def test_zero_input_ranks_by_index():
    B, D, V, tp, k = 4, 128, 1200, 3, 5
    x, W = si.lm_head(B, D, V, seed=1, device="cuda")
    x[1].zero_()
    x[3].zero_()
    idx, val, sidx, _ = tpl.vocab_parallel_topk(x, W, tp, k, shard_outputs=True)
    for b in (1, 3):
        assert idx[b].tolist() == list(range(k)) and torch.all(val[b] == 0)
        for s in range(tp):
            assert sidx[s, b].tolist() == list(range(s * 400, s * 400 + k))
    check_against_oracle(x[[0, 2]].contiguous(), W, tp, k,
                         tpl.vocab_parallel_topk(x[[0, 2]].contiguous(), W, tp, k, shard_outputs=True))


# At D = 8192 the rounding allowance (about 0.1 here) is a fair fraction of
# the typical gap between the largest logits (about 0.4 between the first two,
# less further down), so only part of the positions are fixed by the exact
# ranking; every other position is checked for validity.
@pytest.mark.parametrize("name,D,V,tp,B,k,rows,min_exact", [
    ("llama-3.1-70b", 8192, 128256, 8, 64, 1, [0, 21, 42, 63], 0.25),
    ("llama-3.1-70b", 8192, 128256, 8, 8, 8, [0, 7], 0.08),
    ("qwen2.5-1.5b", 1536, 151936, 2, 128, 1, [0, 1, 64, 127], 0.6),
])
def test_vocab_topk_full_vocabulary_sampled_tokens(name, D, V, tp, B, k, rows, min_exact):
    """Full vocabulary and hidden size, in the launch configuration the
    benchmark times; the oracle checks a sample of the tokens."""
    x, W = si.lm_head(B, D, V, seed=0, device="cuda")
    got = tpl.vocab_parallel_topk(x, W, tp, k, shard_outputs=True)
    check_against_oracle(x, W, tp, k, got, rows=rows, min_exact=min_exact)
