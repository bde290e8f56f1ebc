"""GPU parity of the CUDA-core single-row decode kernel (one query row per (sequence, kv head): no
GQA sharing, one query token; bf16/f16, head_dim 64/128) against the fp64 oracle.

Bars: bf16/f16 atol=2e-3, rtol=2^-8, -inf patterns exact, no NaN.
"""
import numpy as np
import pytest

import oracle
from paged_kv_cache_201_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu

LENS = [0, 1, 15, 16, 17, 63, 64, 65, 200, 511, 1000, 2049]


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_201_gb300 as pa
    pa.load_library(build_if_missing=True)
    return pa


def _all(wl, S, variant=0):
    res = _gpu.run(_gpu.DeviceWorkload(wl), S, variant=variant)
    rows = oracle.all_rows(wl.B, wl.Sq, wl.Hq)
    ref = oracle.workload_rows(wl, split_kv=S, row_bih=rows)
    _gpu.compare_rows(res, ref, rows, wl, S, f"{wl.name} S={S}")
    return res


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("S", [1, 3])
def test_single_row_decode(pa, dtype, D, S):
    """MHA decode: ragged lengths (0 .. 2049, page and stage boundaries), shuffled pages."""
    wl = W.make_custom(name=f"mha_{dtype}_D{D}", dtype=dtype, B=len(LENS), Sq=1, Hq=4, Hkv=4, D=D,
                       page_size=16, seq_lens=LENS, seed=700 + D)
    res = _all(wl, S)
    assert np.isneginf(res["lse"][0]).all() and not res["out"][0].any()  # L = 0
    assert pa.paged_attn_last_error_word() == 0


@pytest.mark.parametrize("ps", [32, 64])
def test_single_row_page_sizes_and_offsets(pa, ps):
    """Pages of 32/64 tokens; causal with explicit offsets (a row that sees no key, one that sees a
    prefix of its sequence) against the automatic choice and the forced CUDA-core variant."""
    lens = [40, 300, 777, 5]
    wl = W.make_custom(name=f"mha_ps{ps}", dtype="bf16", B=4, Sq=1, Hq=2, Hkv=2, D=128, page_size=ps,
                       seq_lens=lens, causal=True, q_offset=[-1, 100, 776, 4], seed=710 + ps)
    res = _all(wl, 2)
    assert np.isneginf(res["lse"][0]).all()
    _all(wl, 1, variant=1)
    assert pa.paged_attn_last_error_word() == 0


def test_single_row_bad_page(pa):
    """An out-of-pool page id: zeros there and the error bit; the other sequence exact."""
    wl = W.make_custom(name="mha_bad", dtype="bf16", B=2, Sq=1, Hq=4, Hkv=4, D=128, page_size=16,
                       seq_lens=[100, 80], num_pages=20, seed=720)
    bt = wl.block_table.copy()
    bt[0, 1] = -7
    res = _gpu.run(_gpu.DeviceWorkload(W.Workload(**{**wl.__dict__, "block_table": bt})), 1)
    assert pa.paged_attn_last_error_word() & 1
    rows = oracle.all_rows(1, 1, wl.Hq)
    rows[:, 0] = 1
    ref = oracle.workload_rows(wl, split_kv=1, row_bih=rows)
    _gpu.assert_close(res["out"][1, 0], ref["out"], "bf16", "sequence 1")
    assert np.isfinite(res["out"][0]).all()


def test_mha_decode_full(pa):
    """The benchmarked single-head decode (B=64, L=4096, Hq=Hkv=32, 2 x 2 GiB pools drawn on the
    device) in its bench launch (split 1) on sampled sequences, every head."""
    wl = W.mha_decode()
    dw = _gpu.DeviceWorkload(wl)
    k, v = dw.host_pools()
    res = _gpu.run(dw, 1)
    assert not np.isnan(res["out"]).any() and np.isfinite(res["lse"]).all()
    seqs = [0, 1, 31, 32, 62, 63]
    b, h = np.meshgrid(np.asarray(seqs), np.arange(wl.Hq), indexing="ij")
    rows = np.stack([b.ravel(), np.zeros(b.size, dtype=np.int64), h.ravel()], axis=1).astype(np.int32)
    ref = oracle.workload_rows(wl, split_kv=1, row_bih=rows, k_cache=k, v_cache=v)
    _gpu.compare_rows(res, ref, rows, wl, 1, "mha full")
    assert pa.paged_attn_last_error_word() == 0
