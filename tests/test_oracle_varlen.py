"""The oracle on variable-length batches (CPU only), pinned to the batched oracle and to a numpy
brute force.

``oracle.rows_varlen`` evaluates each sequence as a batch of one.  Two facts pin it: a batch whose
sequences all have the same query count gives, row for row, exactly what the batched oracle gives
for the [B, Sq, Hq, D] layout (a different index path through the C code); and on mixed batches
(0, 1, a few and many query tokens, causal with and without explicit offsets) every sequence agrees
with a dense numpy fp64 softmax over its logically ordered keys.
"""
import types

import numpy as np
import pytest

import oracle
from paged_kv_cache_201_gb300 import workloads as W
from tests import _bruteforce


def _varlen_dims(wl):
    return oracle.make_dims(B=wl.B, Sq=wl.Sq, Hq=wl.Hq, Hkv=wl.Hkv, D=wl.D, page_size=wl.page_size,
                            bt_stride=int(wl.block_table.shape[1]), dtype=wl.dtype, num_pages=wl.num_pages)


def _varlen(wl, S):
    return oracle.rows_varlen(q=wl.q, k_cache=wl.k_cache, v_cache=wl.v_cache, block_table=wl.block_table,
                              seq_lens=wl.seq_lens, q_start=wl.q_start, q_offset=wl.q_offset, causal=wl.causal,
                              dims=_varlen_dims(wl), scale=wl.scale, split_kv=S)


@pytest.mark.parametrize("causal,offsets", [(True, None), (True, [3, 0, 40]), (False, None)])
def test_uniform_batch_matches_batched_oracle(causal, offsets):
    wl = W.make_custom(dtype="bf16", B=3, Sq=5, Hq=8, Hkv=2, D=64, page_size=16, seq_lens=[7, 33, 60],
                       causal=causal, q_offset=offsets, seed=21)
    ref = oracle.workload_rows(wl, split_kv=3)
    packed = W.Workload(**{**wl.__dict__, "Sq": wl.B * wl.Sq, "q": wl.q.reshape(wl.B * wl.Sq, wl.Hq, wl.D),
                           "q_start": np.arange(0, wl.B * wl.Sq + 1, wl.Sq, dtype=np.int32)})
    got = _varlen(packed, 3)
    n = wl.B * wl.Sq * wl.Hq
    assert np.array_equal(got["out"].reshape(n, wl.D), ref["out"])
    assert np.array_equal(got["lse"].reshape(n), ref["lse"])
    assert np.array_equal(np.moveaxis(got["part_out"], 0, 2).reshape(n, 3, wl.D), ref["part_out"])
    assert np.array_equal(got["comb_out"].reshape(n, wl.D), ref["comb_out"])


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_mixed_batch_matches_bruteforce(dtype):
    q_lens = [1, 0, 3, 12, 1, 7]
    seq_lens = [20, 9, 3, 50, 64, 31]
    offsets = [19, 4, 0, 30, 63, -2]
    for qo in (None, offsets):
        wl = W.make_varlen(dtype=dtype, q_lens=q_lens, seq_lens=seq_lens, Hq=6, Hkv=3, D=16, page_size=16,
                           causal=True, q_offset=qo, seed=5)
        got = _varlen(wl, 2)
        for b in range(wl.B):
            a, e = int(wl.q_start[b]), int(wl.q_start[b + 1])
            if e == a:
                continue
            one = types.SimpleNamespace(
                B=1, Sq=e - a, Hq=wl.Hq, Hkv=wl.Hkv, D=wl.D, page_size=wl.page_size, dtype=wl.dtype,
                seq_lens=wl.seq_lens[b:b + 1], block_table=wl.block_table[b:b + 1], causal=True,
                q_offset=None if qo is None else wl.q_offset[b:b + 1], scale=wl.scale, q=wl.q[a:e][None],
                k_cache=wl.k_cache, v_cache=wl.v_cache)
            out, lse = _bruteforce.attention(one)
            np.testing.assert_allclose(got["out"][a:e], out[0], rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(got["lse"][a:e], lse[0], rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(got["comb_out"][a:e], out[0], rtol=1e-10, atol=1e-10)
        # rows of no sequence do not exist; a sequence without query tokens contributes no row
        assert got["out"].shape[0] == sum(q_lens)
