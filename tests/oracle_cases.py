"""Small helpers shared by the oracle pin tests and the GPU parity tests.

Nothing here computes attention for the product: it converts values to bf16
bits, builds NaN-poisoned pools, and holds the brute-force contiguous
attention used to pin the oracle on tiny inputs.
"""
import numpy as np
import torch

from paged_kv_cache_110_gb300.workloads import BF16_NAN_BITS, bf16_bits, bf16_from_values


def bits(values) -> np.ndarray:
    """bf16 bits of exact small values (numpy uint16, same shape)."""
    return bf16_bits(bf16_from_values(values))


def values(b: np.ndarray) -> np.ndarray:
    """float64 values of bf16 bits."""
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).double().numpy()


def nan_pool(num_blocks, block_size, kv_heads, head_dim) -> np.ndarray:
    return np.full((num_blocks, block_size, kv_heads, head_dim), BF16_NAN_BITS, dtype=np.uint16)


def brute_force_attention(q, k, v, scale, causal=True):
    """Dense softmax attention of one sequence, written as matrices.

    q [Lq, Hq, d], k/v [Lk, Hkv, d] (float64 values, keys in logical order).
    The Lq queries are the last Lq positions of the Lk keys; with ``causal`` a
    query at position p may read keys 0..p.  Query head h reads kv head
    h // (Hq // Hkv).
    """
    lq, hq, d = q.shape
    lk, hkv, _ = k.shape
    group = hq // hkv
    kk = np.repeat(k, group, axis=1)  # [Lk, Hq, d]
    vv = np.repeat(v, group, axis=1)
    s = np.einsum("ihd,jhd->hij", q, kk) * scale
    if causal:
        qpos = np.arange(lq)[:, None] + (lk - lq)
        allowed = np.arange(lk)[None, :] <= qpos
        s = np.where(allowed[None], s, -np.inf)
    s = s - s.max(axis=-1, keepdims=True)
    w = np.exp(s)
    w /= w.sum(axis=-1, keepdims=True)
    return np.einsum("hij,jhd->ihd", w, vv), w


def bf16_round(x) -> np.ndarray:
    """Round doubles to the nearest bf16 value (ties to even), still as doubles:
    8 significant bits, without passing through float32."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
