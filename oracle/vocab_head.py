"""Oracle for the vocabulary-parallel lm_head -- TEST INFRASTRUCTURE ONLY.

Plain CPU restatement of what the CUDA lm_head path computes.  Only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it; the product path never does, and it shares no code
with the CUDA library.  Inputs are numpy arrays (bf16 values already widened);
arithmetic is float64; the matrix product is the library matmul as one step.

Source: [L4] "Lecture 4 - Distributed Serving" (CS349E notes), S4.5 "lm_head
and sequence parallelism".  The lm_head is split by vocabulary: device s holds
the scores of V/n vocabulary entries, and the full logits are normally
all-gathered.  When only the next token is needed, each device can first take
its own maximum (or top-k) and only those candidates are exchanged.

Readings where the section is silent:
  * The lm_head weight is stored [V, D] (one row per vocabulary entry, the
    [out, in] layout of the other projections); shard s owns the contiguous
    rows [s V/tp, (s+1) V/tp), so V must divide by tp.
  * logits[b, v] = sum_d x[b, d] W[v, d]: the final hidden state as given (any
    final RMSNorm is applied by the caller; its positive per-token scale does
    not change the ranking).
  * "top-k" orders by logit, larger first, and breaks exact ties by the lower
    vocabulary index, so the result is unique.  Every logit compares equal to
    itself; +0 and -0 are equal.
  * The exchange is the union of the tp shard-local top-k lists, from which the
    global top-k is taken with the same order.
"""
from __future__ import annotations

import numpy as np

F64 = np.float64


def vocab_shards(V: int, tp: int) -> list[tuple[int, int]]:
    """Row range [start, stop) of each vocabulary shard ([L4] S4.5: V/n entries
    per device, contiguous as in the S3.1 sharding notation)."""
    if tp < 1 or V % tp:
        raise ValueError("V must be a positive multiple of tp")
    vs = V // tp
    return [(s * vs, (s + 1) * vs) for s in range(tp)]


def logits(x: np.ndarray, W: np.ndarray) -> np.ndarray:
    """The unsharded lm_head: logits[b, v] = x[b] . W[v]  (x [B, D], W [V, D])."""
    return np.asarray(x, F64) @ np.asarray(W, F64).T


def ordered_topk(values: np.ndarray, k: int, offset: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """Top-k of one row of scores: indices and values, larger value first, equal
    values by lower index.  ``offset`` is added to the returned indices (the
    first vocabulary row of a shard)."""
    v = np.asarray(values, F64) + 0.0          # -0 -> +0: the two compare equal
    idx = np.arange(v.shape[0])
    order = np.lexsort((idx, -v))[:k]          # primary key -v, secondary key index
    return order + offset, v[order]


def gathered_logits(x: np.ndarray, W: np.ndarray, tp: int) -> np.ndarray:
    """The all-gather route of [L4] S4.5: every shard computes its V/tp logits,
    and the full row is the concatenation of the shards' pieces."""
    return np.concatenate([logits(x, W[a:b]) for a, b in vocab_shards(W.shape[0], tp)], axis=1)


def vocab_parallel_topk(x: np.ndarray, W: np.ndarray, tp: int, k: int):
    """The candidate-exchange route of [L4] S4.5.

    Each shard ranks only its own V/tp logits and keeps its top-k (global
    vocabulary indices); the tp lists are exchanged and the top-k of their
    union is the result.  Returns (idx [B, k], val [B, k], shard_idx [tp, B, k],
    shard_val [tp, B, k])."""
    x = np.asarray(x, F64)
    B = x.shape[0]
    shards = vocab_shards(W.shape[0], tp)
    if not 1 <= k <= W.shape[0] // tp:
        raise ValueError("k must be in [1, V/tp]")
    sidx = np.zeros((tp, B, k), np.int64)
    sval = np.zeros((tp, B, k), F64)
    for s, (a, b) in enumerate(shards):
        local = logits(x, W[a:b])
        for t in range(B):
            sidx[s, t], sval[s, t] = ordered_topk(local[t], k, offset=a)
    idx = np.zeros((B, k), np.int64)
    val = np.zeros((B, k), F64)
    for t in range(B):
        cand_v = sval[:, t, :].reshape(-1)
        cand_i = sidx[:, t, :].reshape(-1)
        order = np.lexsort((cand_i, -cand_v))[:k]
        idx[t], val[t] = cand_i[order], cand_v[order]
    return idx, val, sidx, sval


def exchange_bytes(B: int, V: int, tp: int, k: int, mode: str, logit_bytes: int = 2,
                   index_bytes: int = 4) -> int:
    """Bytes of the lm_head's output exchange for one decode step.

    ``gather``: the full logits [B, V] in the logit dtype ([L4] S4.5 quotes this
    size for Llama-3.1-70B at B = 64).  ``topk``: tp shard lists of k (index,
    logit) pairs per token."""
    if mode == "gather":
        return B * V * logit_bytes
    if mode == "topk":
        return tp * B * k * (index_bytes + logit_bytes)
    raise ValueError(mode)
