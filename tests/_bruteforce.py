"""Dense numpy float64 attention on logically ordered K/V, for tiny shapes.

Written independently of the C oracle: logical K/V come from numpy fancy
indexing of the page pool, GQA from ``np.repeat`` over kv heads, the mask is an
additive -inf matrix and the softmax is ``exp(s - max) / sum``.  It is only used
to pin the oracle (and is deliberately unlike it: whole matrices, no per-key
loop, no split plan).
"""
from __future__ import annotations

import numpy as np


def widen(arr: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f64":
        return np.asarray(arr, dtype=np.float64)
    if dtype == "f32":
        return np.asarray(arr, dtype=np.float32).astype(np.float64)
    bits = np.asarray(arr).view(np.uint16)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def logical_kv(cache: np.ndarray, block_table: np.ndarray, L: int, page_size: int, dtype: str) -> np.ndarray:
    """[L, Hkv, D] float64 for one sequence via fancy indexing of [P, ps, Hkv, D]."""
    c = widen(cache, dtype)
    j = np.arange(L)
    pages = block_table[j // page_size].astype(np.int64)
    return c[pages, j % page_size]


def attention(wl, q=None, k_cache=None, v_cache=None, kv_dtype=None):
    """Returns (out [B, Sq, Hq, D], lse [B, Sq, Hq]) in float64.  ``kv_dtype`` ("f64" for
    already-dequantized pools) defaults to the query dtype."""
    q = wl.q if q is None else q
    kvd = wl.dtype if kv_dtype is None else kv_dtype
    k_cache = wl.k_cache if k_cache is None else k_cache
    v_cache = wl.v_cache if v_cache is None else v_cache
    qd = widen(q, wl.dtype)
    G = wl.Hq // wl.Hkv
    out = np.zeros((wl.B, wl.Sq, wl.Hq, wl.D))
    lse = np.full((wl.B, wl.Sq, wl.Hq), -np.inf)
    for b in range(wl.B):
        L = int(wl.seq_lens[b])
        if L <= 0:
            continue
        K = np.repeat(logical_kv(k_cache, wl.block_table[b], L, wl.page_size, kvd), G, axis=1)  # [L, Hq, D]
        V = np.repeat(logical_kv(v_cache, wl.block_table[b], L, wl.page_size, kvd), G, axis=1)
        s = np.einsum("ihd,jhd->hij", qd[b], K) * wl.scale                                 # [Hq, Sq, L]
        if wl.causal:
            qoff = (L - wl.Sq) if wl.q_offset is None else int(wl.q_offset[b])
            i = np.arange(wl.Sq)[:, None]
            j = np.arange(L)[None, :]
            mask = np.where(j <= qoff + i, 0.0, -np.inf)
            s = s + mask[None]
        m = s.max(axis=-1, keepdims=True)
        finite = np.isfinite(m)
        msafe = np.where(finite, m, 0.0)
        p = np.exp(s - msafe)
        l = p.sum(axis=-1, keepdims=True)
        o = np.einsum("hij,jhd->ihd", p, V) / np.where(l > 0, l, 1.0).transpose(1, 0, 2)
        o = np.where((l > 0).transpose(1, 0, 2), o, 0.0)
        out[b] = o
        with np.errstate(divide="ignore"):
            lse[b] = np.where(l[..., 0] > 0, msafe[..., 0] + np.log(l[..., 0]), -np.inf).T
    return out, lse
