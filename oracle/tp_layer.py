"""Oracle for the Megatron tensor-parallel layer forward -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct CPU implementation of what the CUDA path
computes.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import it; the product path never does.  It shares no
code with the CUDA library: inputs arrive as numpy arrays (bf16 values already
widened), all arithmetic is numpy float64, and matrix products use the library
matmul as a single step (no blocking or reordering of our own).

Sources (pages of the reference material, by title and section):
  [L4]  "Lecture 4 - Distributed Serving" (CS349E notes, semidirectx.com):
        S3.1 sharding notation, S3.2 the four cases, S4.1 MLP column-then-row,
        S4.2 attention split by head, S4.3 correctness, S4.4 KV groups vs TP,
        S5.5 block formula.
  [V4]  "vLLM model parallelism" article (intelliparadigm.com), S2.1 tensor
        parallelism: ColumnParallelLinear stores its weight as
        [output_size_per_partition, input_size] and applies F.linear.

Readings where the pages are silent:
  * SwiGLU is silu(gate) * up with silu(z) = z / (1 + exp(-z))  ([L4] S4.1 only
    says "element-wise").
  * Weights are stored [out, in] ([V4] S2.1); shard s of a split dimension of
    length n owns the contiguous block [s n/tp, (s+1) n/tp)  ([L4] S3.1).
  * Packed QKV weight rows are [Q heads | K heads | V heads], head-major.
  * When tp > n_kv, shard s holds a copy of KV group floor(s n_kv / tp)
    ([L4] S4.4: each device keeps its own copy).
  * Attention core is not on the path; with a context of one token the softmax
    weight is exactly 1, so the output of Q head h is the value of its KV group
    g(h) = floor(h n_kv / n_q).
  * Shard partials are summed in ascending shard order ([L4] S4.3: sharded and
    single-device results differ only by the order of that sum).
  * bf16 rounding (round-to-nearest-even) happens exactly where the CUDA path
    stores a bf16 tensor: the SwiGLU output H, the packed QKV output, the
    residual stream and every bf16 result.  Partials stay unrounded.  The
    RMSNorm output is not stored: its per-row scale 1/rms multiplies the
    consuming projection's products, RMSNorm(x) W^T = diag(1/rms(x)) (x W^T),
    so the normalised activations are never rounded to bf16.
  * A tensor sharded along its last dimension, e.g. C[I, K_X], is stored as the
    concatenation of the device-local shards: [X, I, K/X].  One sharded along
    its first dimension, C[I_X, K], is then simply [I, K] row-major.
"""
from __future__ import annotations

import numpy as np

F64 = np.float64
BF16_MAX = float.fromhex("0x1.fep127")


# ---------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------

def bf16_round(x) -> np.ndarray:
    """Round to the nearest bfloat16 value, ties to even; returned as float64.

    bfloat16 keeps 8 significant bits (1 implicit + 7 stored) and the fp32
    exponent range: the quantum of a normal number m*2**e (0.5 <= |m| < 1) is
    2**(e-8); below the smallest normal 2**-126 the quantum is fixed at 2**-133.
    Values past the largest finite bf16 after rounding become +-inf.
    """
    x = np.asarray(x, dtype=F64)
    _, e = np.frexp(x)
    k = np.maximum(e, -125) - 8
    r = np.ldexp(np.rint(np.ldexp(x, -k)), k)
    big = np.abs(r) > BF16_MAX
    if np.any(big):
        r = np.where(big, np.copysign(np.inf, x), r)
    return r


def silu(z) -> np.ndarray:
    """z * sigmoid(z) = z / (1 + exp(-z))  (the gate nonlinearity of SwiGLU)."""
    z = np.asarray(z, dtype=F64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=F64)


def _out(y: np.ndarray, bf16: bool) -> np.ndarray:
    return bf16_round(y) if bf16 else y


# ---------------------------------------------------------------------------
# Sharding notation ([L4] S3.1): A[I_X, J] -- dimension I split over mesh axis X,
# device d holds the d-th contiguous segment of I/|X| indices.
# ---------------------------------------------------------------------------

def shard_range(n: int, tp: int, s: int) -> range:
    """Indices of a length-n dimension held by shard s of tp (contiguous blocks)."""
    if tp <= 0 or n % tp != 0:
        raise ValueError(f"dimension {n} is not divisible by {tp} shards")
    if not 0 <= s < tp:
        raise ValueError(f"shard {s} out of range for {tp} shards")
    w = n // tp
    return range(s * w, (s + 1) * w)


def linear(x, w_out_in) -> np.ndarray:
    """y = x W with W stored [out, in]:  y[b, o] = sum_i x[b, i] w[o, i]."""
    return _f64(x) @ _f64(w_out_in).T


# ---------------------------------------------------------------------------
# Megatron MLP ([L4] S4.1): column-parallel gate/up, local SwiGLU, row-parallel down
# ---------------------------------------------------------------------------

def mlp_unsharded(X, Wg, Wu, Wd, bf16: bool = True) -> np.ndarray:
    """Single-device SwiGLU MLP: Y = (silu(X Wg^T) * (X Wu^T)) Wd^T.

    Wg, Wu stored [F, D]; Wd stored [D, F].  With ``bf16`` the hidden H is
    rounded to bf16 before the down projection and Y is rounded at the end.
    """
    G = linear(X, Wg)
    U = linear(X, Wu)
    H = silu(G) * U
    if bf16:
        H = bf16_round(H)
    return _out(linear(H, Wd), bf16)


def mlp_hidden_shard(X, Wg, Wu, tp: int, s: int, bf16: bool = True) -> np.ndarray:
    """Shard s's column-parallel hidden H_s[B, F/tp] (case 1 of [L4] S3.2: no comm).

    Wg/Wu [F, D] are split by output rows: shard s holds rows shard_range(F, tp, s).
    """
    F = np.shape(Wg)[0]
    rows = shard_range(F, tp, s)
    Wg_s = _f64(Wg)[rows.start:rows.stop]
    Wu_s = _f64(Wu)[rows.start:rows.stop]
    H_s = silu(linear(X, Wg_s)) * linear(X, Wu_s)
    return bf16_round(H_s) if bf16 else H_s


def mlp_partial_shard(H_s, Wd, tp: int, s: int) -> np.ndarray:
    """Row-parallel down partial P_s = H_s Wd_s^T (case 3: a partial sum, unreduced).

    Wd [D, F] is split along its input dimension F: shard s holds columns
    shard_range(F, tp, s).
    """
    F = np.shape(Wd)[1]
    cols = shard_range(F, tp, s)
    return linear(H_s, _f64(Wd)[:, cols.start:cols.stop])


def shard_reduce(partials, bf16: bool = False) -> np.ndarray:
    """All-reduce stand-in: Y = P_0 + P_1 + ... + P_{tp-1}, left to right."""
    partials = [_f64(p) for p in partials]
    y = partials[0].copy()
    for p in partials[1:]:
        y = y + p
    return _out(y, bf16)


def reduce_scatter_blocks(y_full, tp: int) -> np.ndarray:
    """Reduce-scatter ownership of a reduced [R, C] result: shard s keeps columns
    shard_range(C, tp, s); stored shard-blocked as [tp, R, C/tp]."""
    y_full = _f64(y_full)
    C = y_full.shape[1]
    return np.stack([y_full[:, shard_range(C, tp, s).start:shard_range(C, tp, s).stop]
                     for s in range(tp)])


def mlp_sharded(X, Wg, Wu, Wd, tp: int, bf16: bool = True):
    """Sharded MLP the Megatron way: per-shard H_s and P_s, then the partial sum.

    Returns (Y, [P_0..P_{tp-1}], [H_0..H_{tp-1}]).
    """
    H = [mlp_hidden_shard(X, Wg, Wu, tp, s, bf16) for s in range(tp)]
    P = [mlp_partial_shard(H[s], Wd, tp, s) for s in range(tp)]
    return shard_reduce(P, bf16), P, H


# ---------------------------------------------------------------------------
# Attention projections split by head ([L4] S4.2, S4.4)
# ---------------------------------------------------------------------------

def kv_group_of_head(h: int, n_q: int, n_kv: int) -> int:
    """KV group used by query head h under GQA: floor(h n_kv / n_q)."""
    return (h * n_kv) // n_q


def head_shard_map(n_q: int, n_kv: int, tp: int):
    """Per shard: (list of global Q heads, list of global KV groups it holds).

    Q heads are split in contiguous blocks of n_q/tp.  If tp <= n_kv the KV
    groups are split the same way (n_kv/tp each); if tp > n_kv every shard
    keeps a copy of the one group its Q heads use, floor(s n_kv / tp).
    """
    if n_q % tp != 0:
        raise ValueError("n_q must be divisible by tp")
    if n_q % n_kv != 0:
        raise ValueError("n_q must be a multiple of n_kv")
    out = []
    for s in range(tp):
        q = list(shard_range(n_q, tp, s))
        if tp <= n_kv:
            kv = list(shard_range(n_kv, tp, s))
        else:
            if tp % n_kv != 0:
                raise ValueError("tp > n_kv needs tp divisible by n_kv")
            kv = [(s * n_kv) // tp]
        if sorted({kv_group_of_head(h, n_q, n_kv) for h in q}) != kv:
            raise ValueError("head split does not keep each Q head with its KV group")
        out.append((q, kv))
    return out


def qkv_rows_of_shard(n_q: int, n_kv: int, head_dim: int, tp: int, s: int) -> np.ndarray:
    """Row indices into the packed Wqkv [(n_q + 2 n_kv) hd, D] that shard s uses,
    in the shard's [Q_s | K_s | V_s] output order."""
    q, kv = head_shard_map(n_q, n_kv, tp)[s]
    hd = head_dim
    rows = [np.arange(h * hd, (h + 1) * hd) for h in q]
    rows += [np.arange((n_q + g) * hd, (n_q + g + 1) * hd) for g in kv]
    rows += [np.arange((n_q + n_kv + g) * hd, (n_q + n_kv + g + 1) * hd) for g in kv]
    return np.concatenate(rows)


def context1_attention(Q, K, V, n_q_local: int, kv_local: list, heads_global: list,
                       n_q: int, n_kv: int, head_dim: int) -> np.ndarray:
    """Attention of each query head over a context of exactly one token (itself).

    softmax over a single score is 1, so each head's output is the value vector
    of its KV group.  Q[B, nq_local hd], K/V[B, len(kv_local) hd] -> O[B, nq_local hd].
    """
    B = Q.shape[0]
    O = np.zeros((B, n_q_local * head_dim))
    for j, h in enumerate(heads_global):
        g = kv_group_of_head(h, n_q, n_kv)
        c = kv_local.index(g)
        q = Q[:, j * head_dim:(j + 1) * head_dim]
        k = K[:, c * head_dim:(c + 1) * head_dim]
        v = V[:, c * head_dim:(c + 1) * head_dim]
        score = np.sum(q * k, axis=1, keepdims=True) / np.sqrt(head_dim)   # [B, 1]
        w = np.exp(score - score.max(axis=1, keepdims=True))
        w = w / w.sum(axis=1, keepdims=True)                                # == 1
        O[:, j * head_dim:(j + 1) * head_dim] = w * v
    return O


def attn_proj_unsharded(X, Wqkv, Wo, n_q: int, n_kv: int, head_dim: int, bf16: bool = True):
    """Single-device QKV projection, context-1 attention, o_proj.

    Returns (Y[B, D], QKV[B, (n_q + 2 n_kv) hd]).
    """
    QKV = linear(X, Wqkv)
    if bf16:
        QKV = bf16_round(QKV)
    hd = head_dim
    Q = QKV[:, :n_q * hd]
    K = QKV[:, n_q * hd:(n_q + n_kv) * hd]
    V = QKV[:, (n_q + n_kv) * hd:]
    O = context1_attention(Q, K, V, n_q, list(range(n_kv)), list(range(n_q)), n_q, n_kv, hd)
    return _out(linear(O, Wo), bf16), QKV


def attn_proj_sharded(X, Wqkv, Wo, n_q: int, n_kv: int, head_dim: int, tp: int, bf16: bool = True):
    """Head-partitioned attention projections ([L4] S4.2).

    Shard s: QKV_s = X Wqkv_s^T over its rows in [Q_s | K_s | V_s] order, its
    heads' attention O_s, and the row-parallel partial P_s = O_s Wo_s^T where
    Wo [D, n_q hd] is split by columns in Q-head blocks.  Returns
    (Y, [QKV_s], [O_s], [P_s]).
    """
    hd = head_dim
    smap = head_shard_map(n_q, n_kv, tp)
    QKVs, Os, Ps = [], [], []
    for s in range(tp):
        q, kv = smap[s]
        rows = qkv_rows_of_shard(n_q, n_kv, hd, tp, s)
        qkv = linear(X, _f64(Wqkv)[rows])
        if bf16:
            qkv = bf16_round(qkv)
        nq_l, nkv_l = len(q), len(kv)
        Q = qkv[:, :nq_l * hd]
        K = qkv[:, nq_l * hd:(nq_l + nkv_l) * hd]
        V = qkv[:, (nq_l + nkv_l) * hd:]
        O = context1_attention(Q, K, V, nq_l, kv, q, n_q, n_kv, hd)
        cols = shard_range(n_q * hd, tp, s)
        P = linear(O, _f64(Wo)[:, cols.start:cols.stop])
        QKVs.append(qkv)
        Os.append(O)
        Ps.append(P)
    return shard_reduce(Ps, bf16), QKVs, Os, Ps


# ---------------------------------------------------------------------------
# Sharded matrix multiply, the four cases ([L4] S3.2).  C = A B with A[I, J],
# B[J, K] stored transposed as Bt[K, J]; J is the contracting dimension.
# ---------------------------------------------------------------------------

def matmul(A, Bt) -> np.ndarray:
    """C[I, K] = A[I, J] B[J, K] with B stored as Bt[K, J]."""
    return linear(A, Bt)


def sharded_matmul(case: int, A, Bt, X: int, mode: str = "allreduce", gather: str = "B",
                   bf16: bool = True):
    """One of the four sharding cases on X logical devices.

    case 1  A[I_X, J] B[J, K]    -> C[I_X, K]: each device multiplies its rows, no comm.
    case 2  A[I, J_X] B[J, K]    -> all-gather A, then the full product C[I, K].
    case 3  A[I, J_X] B[J_X, K]  -> partial sums C[I, K]{U_X}; all-reduce gives C[I, K],
                                    reduce-scatter gives C[I, K_X] (stored [X, I, K/X]).
    case 4  A[I_X, J] B[J, K_X]  -> no legal local product; all-gather B (case 1,
                                    C[I_X, K]) or all-gather A (C[I, K_X], stored [X, I, K/X]).
    Returns (C, partials or None).  Row-sharded results are stored [I, K].
    """
    A = _f64(A)
    Bt = _f64(Bt)
    I, J = A.shape
    K = Bt.shape[0]
    if case == 1:
        blocks = [matmul(A[shard_range(I, X, s).start:shard_range(I, X, s).stop], Bt)
                  for s in range(X)]
        return _out(np.concatenate(blocks, axis=0), bf16), None
    if case == 2:
        shards = [A[:, shard_range(J, X, s).start:shard_range(J, X, s).stop] for s in range(X)]
        A_full = np.concatenate(shards, axis=1)            # the all-gather
        return _out(matmul(A_full, Bt), bf16), None
    if case == 3:
        P = []
        for s in range(X):
            js = shard_range(J, X, s)
            P.append(matmul(A[:, js.start:js.stop], Bt[:, js.start:js.stop]))
        C = shard_reduce(P, False)
        if mode == "allreduce":
            return _out(C, bf16), P
        if mode == "reducescatter":
            return _out(reduce_scatter_blocks(C, X), bf16), P
        raise ValueError("mode must be allreduce or reducescatter")
    if case == 4:
        if gather == "B":
            Bt_full = np.concatenate([Bt[shard_range(K, X, s).start:shard_range(K, X, s).stop]
                                      for s in range(X)], axis=0)
            return sharded_matmul(1, A, Bt_full, X, bf16=bf16)
        if gather == "A":
            A_full = np.concatenate([A[shard_range(I, X, s).start:shard_range(I, X, s).stop]
                                     for s in range(X)], axis=0)
            blocks = [matmul(A_full, Bt[shard_range(K, X, s).start:shard_range(K, X, s).stop])
                      for s in range(X)]
            return _out(np.stack(blocks), bf16), None
        raise ValueError("gather must be 'A' or 'B'")
    raise ValueError("case must be 1, 2, 3 or 4")


def case4_local_blocks(A, Bt, X: int) -> list:
    """What case 4 would compute without a gather: device d multiplies its row
    block of A by its column block of B, i.e. only the diagonal blocks C_dd."""
    A = _f64(A)
    Bt = _f64(Bt)
    I, K = A.shape[0], Bt.shape[0]
    return [matmul(A[shard_range(I, X, d).start:shard_range(I, X, d).stop],
                   Bt[shard_range(K, X, d).start:shard_range(K, X, d).stop]) for d in range(X)]


# ---------------------------------------------------------------------------
# Decoder layer composition (serial pre-norm block; [L4] S4.2 replicated RMSNorm,
# S5.5 block formula written for the serial arrangement)
# ---------------------------------------------------------------------------

RMS_EPS = 1e-6


def rmsnorm(x, eps: float = RMS_EPS) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) per row, unit gain."""
    x = _f64(x)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def decoder_layer(x, W: dict, n_q: int, n_kv: int, head_dim: int, tp: int, sharded: bool = True,
                  trace: list | None = None):
    """h = x + Attn(RMSNorm(x));  y = h + MLP(RMSNorm(h)); bf16 between steps.

    ``W`` holds Wqkv, Wo, Wg, Wu, Wd.  Returns y (bf16 values, float64 array).
    If ``trace`` is a list, the two rounded residual-stream values h and y are
    appended to it (read-only instrumentation; the arithmetic is unchanged).
    """
    xn = rmsnorm(x)          # not rounded: its scale is applied to the products
    if sharded:
        a, _, _, P = attn_proj_sharded(xn, W["Wqkv"], W["Wo"], n_q, n_kv, head_dim, tp)
        a_sum = shard_reduce(P, False)
    else:
        a_sum = linear_attn_sum(xn, W, n_q, n_kv, head_dim)
    h = bf16_round(_f64(x) + a_sum)
    hn = rmsnorm(h)
    if sharded:
        _, P, _ = mlp_sharded(hn, W["Wg"], W["Wu"], W["Wd"], tp, bf16=True)
        m_sum = shard_reduce(P, False)
    else:
        m_sum = linear(bf16_round(silu(linear(hn, W["Wg"])) * linear(hn, W["Wu"])), W["Wd"])
    y = bf16_round(h + m_sum)
    if trace is not None:
        trace.extend([h, y])
    return y


def decoder_layer_parallel(x, W: dict, n_q: int, n_kv: int, head_dim: int, tp: int, trace: list | None = None):
    """The parallel (PaLM) block of [L4] S5.5: y = x + Attn(RMSNorm(x)) + MLP(RMSNorm(x)).

    Both sublayers read the same normalised input, and their shard partials are
    summed together in one reduction (the shared all-reduce of S5.5); the
    residual stream is rounded to bf16 once per layer.  ``trace`` as in
    decoder_layer, with y only.
    """
    xn = rmsnorm(x)
    _, _, _, Pa = attn_proj_sharded(xn, W["Wqkv"], W["Wo"], n_q, n_kv, head_dim, tp)
    _, Pm, _ = mlp_sharded(xn, W["Wg"], W["Wu"], W["Wd"], tp, bf16=True)
    y = bf16_round(_f64(x) + shard_reduce(Pa, False) + shard_reduce(Pm, False))
    if trace is not None:
        trace.append(y)
    return y


def linear_attn_sum(xn, W, n_q, n_kv, head_dim):
    """Unsharded attention sublayer output before any rounding of the sum."""
    QKV = bf16_round(linear(xn, W["Wqkv"]))
    hd = head_dim
    V = QKV[:, (n_q + n_kv) * hd:]
    K = QKV[:, n_q * hd:(n_q + n_kv) * hd]
    Q = QKV[:, :n_q * hd]
    O = context1_attention(Q, K, V, n_q, list(range(n_kv)), list(range(n_q)), n_q, n_kv, hd)
    return linear(O, W["Wo"])


def decoder_stack(x, layers: list, n_q: int, n_kv: int, head_dim: int, tp: int, sharded: bool = True,
                  trace: list | None = None, block: str = "serial"):
    """Layers applied in order; returns the final residual stream (bf16 values).
    ``trace`` as in decoder_layer: every rounded residual-stream value, in order.
    ``block``: "serial" (pre-norm, attention then MLP) or "parallel" ([L4] S5.5)."""
    y = bf16_round(x)
    for W in layers:
        if block == "parallel":
            y = decoder_layer_parallel(y, W, n_q, n_kv, head_dim, tp, trace)
        else:
            y = decoder_layer(y, W, n_q, n_kv, head_dim, tp, sharded, trace)
    return y
