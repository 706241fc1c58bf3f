"""Byte accounting for the sharded layouts and the collectives that the
on-device partial-sum reduction replaces -- TEST INFRASTRUCTURE ONLY.

Written from "Lecture 4 - Distributed Serving" (CS349E notes): S3.1 (what one
device stores under the sharding notation), S3.2 (case costs), S3.3 (the
collective price list: all-gather ~ reduce-scatter ~ (n-1)/n V bytes per
device, all-reduce = reduce-scatter + all-gather), S4.5 (message sizes) and
the exercises.  Sizes are exact integers in bytes.
"""
from __future__ import annotations

from fractions import Fraction


def shard_bytes(shape, sharded_dims, n: int, elem_bytes: int = 2) -> int:
    """Bytes one device stores for a tensor whose dims listed in ``sharded_dims``
    are each split over the same n-device axis (S3.1)."""
    total = elem_bytes
    for i, d in enumerate(shape):
        if i in sharded_dims:
            if d % n:
                raise ValueError("dimension not divisible by the mesh axis")
            total *= d // n
        else:
            total *= d
    return total


def allgather_bytes_per_device(full_bytes: int, n: int) -> Fraction:
    """All-gather of a tensor of ``full_bytes``: each device receives the (n-1)/n it lacks."""
    return Fraction(n - 1, n) * full_bytes


def reducescatter_bytes_per_device(full_bytes: int, n: int) -> Fraction:
    """Reduce-scatter moves the same volume as all-gather (S3.3)."""
    return Fraction(n - 1, n) * full_bytes


def allreduce_bytes_per_device(full_bytes: int, n: int) -> Fraction:
    """All-reduce = reduce-scatter + all-gather: twice the all-gather volume (S3.3)."""
    return reducescatter_bytes_per_device(full_bytes, n) + allgather_bytes_per_device(full_bytes, n)


def case_comm_bytes(case: int, I: int, J: int, K: int, n: int, elem_bytes: int = 2,
                    mode: str = "allreduce", gather: str = "B") -> Fraction:
    """Per-device communication volume of the four cases (S3.2)."""
    A = I * J * elem_bytes
    B = J * K * elem_bytes
    C = I * K * elem_bytes
    if case == 1:
        return Fraction(0)
    if case == 2:
        return allgather_bytes_per_device(A, n)
    if case == 3:
        if mode == "allreduce":
            return allreduce_bytes_per_device(C, n)
        return reducescatter_bytes_per_device(C, n)
    if case == 4:
        return allgather_bytes_per_device(B if gather == "B" else A, n)
    raise ValueError("case must be 1..4")


def allreduce_message_bytes(B: int, D: int, elem_bytes: int = 2) -> int:
    """One Megatron all-reduce carries the [B, D] activation (S4.1, S4.2, S6.1)."""
    return B * D * elem_bytes


def ring_allreduce_bytes_per_device(message_bytes: int, n: int) -> Fraction:
    """A ring all-reduce sends 2 (n-1)/n of the message from each device."""
    return 2 * Fraction(n - 1, n) * message_bytes


def logits_bytes(B: int, vocab: int, elem_bytes: int = 2) -> int:
    """Gathered logits of a vocabulary-parallel lm_head (S4.5)."""
    return B * vocab * elem_bytes


def layer_weight_bytes(D: int, F: int, n_q: int, n_kv: int, head_dim: int, elem_bytes: int = 2) -> int:
    """Bytes of one layer's projection weights: QKV, o_proj, gate, up, down."""
    qkv = (n_q + 2 * n_kv) * head_dim * D
    o = D * n_q * head_dim
    mlp = 3 * D * F
    return (qkv + o + mlp) * elem_bytes


def layer_flops(B: int, D: int, F: int, n_q: int, n_kv: int, head_dim: int) -> int:
    """Multiply-add flops (2 per MAC) of one layer's projections for B tokens."""
    return 2 * B * layer_weight_bytes(D, F, n_q, n_kv, head_dim, 1)


def mlp_flops(B: int, D: int, F: int) -> int:
    """Gate + up + down: 2 B D 2F + 2 B F D."""
    return 2 * B * D * 2 * F + 2 * B * F * D
