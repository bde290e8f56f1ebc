"""GPU parity at head_dim 256 against the fp64 oracle: the transposed tensor-core kernel (bf16/f16,
8-row units), the CUDA-core kernel (f32 and single-head rows) and the combine at D = 256.

Bars as everywhere: bf16/f16 atol=2e-3, rtol=2^-8; f32 1e-5; -inf patterns exact; no NaN.
"""
import numpy as np
import pytest

import oracle
from paged_kv_cache_201_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_201_gb300 as pa
    pa.load_library(build_if_missing=True)
    return pa


def _all(pa, wl, S, variant=0):
    dw = _gpu.DeviceWorkload(wl)
    res = _gpu.run(dw, S, variant=variant)
    rows = oracle.all_rows(wl.B, wl.Sq, wl.Hq)
    ref = oracle.workload_rows(wl, split_kv=S, row_bih=rows)
    _gpu.compare_rows(res, ref, rows, wl, S, f"{wl.name} S={S} variant={variant}")
    return res


LENS = [1, 16, 17, 64, 65, 200, 511, 1000]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("G", [4, 8, 16])
@pytest.mark.parametrize("S", [1, 3])
def test_decode_d256(pa, dtype, G, S):
    """Ragged decode (one query token): 8-row units, G = 16 takes two units per kv head."""
    Hkv = 2
    wl = W.make_custom(name=f"d256_G{G}", dtype=dtype, B=len(LENS), Sq=1, Hq=G * Hkv, Hkv=Hkv, D=256,
                       page_size=16, seq_lens=LENS, seed=600 + G)
    _all(pa, wl, S)
    assert pa.paged_attn_last_error_word() == 0


@pytest.mark.parametrize("ps", [32, 64])
def test_causal_multi_token_d256(pa, ps):
    """Several query tokens per sequence (Sq=20, G=4: 80 rows, 10 units per kv head), causal with
    explicit offsets, one of which hides every key from the first rows; larger pages."""
    wl = W.make_custom(name=f"d256_prefill_ps{ps}", dtype="bf16", B=3, Sq=20, Hq=8, Hkv=2, D=256, page_size=ps,
                       seq_lens=[20, 300, 777], causal=True, q_offset=[-4, 280, 700], seed=620 + ps)
    res = _all(pa, wl, 2)
    assert np.isneginf(res["lse"][0, :4]).all()
    assert pa.paged_attn_last_error_word() == 0


def test_single_head_and_f32_d256(pa):
    """Single-head decode (CUDA-core kernel) and f32 pools at D = 256."""
    wl = W.make_custom(name="d256_mha", dtype="bf16", B=4, Sq=1, Hq=4, Hkv=4, D=256, page_size=16,
                       seq_lens=[5, 64, 300, 1000], seed=631)
    _all(pa, wl, 1)
    _all(pa, wl, 2)
    wl = W.make_custom(name="d256_f32", dtype="f32", B=3, Sq=2, Hq=8, Hkv=2, D=256, page_size=16,
                       seq_lens=[2, 100, 250], causal=True, seed=632)
    _all(pa, wl, 1)
    _all(pa, wl, 3)
    assert pa.paged_attn_last_error_word() == 0


def test_d256_bad_page_reads_zero(pa):
    """An out-of-pool page id at D = 256: the unit reads zeros there and reports it; other sequences exact."""
    wl = W.make_custom(name="d256_bad", dtype="bf16", B=2, Sq=1, Hq=8, Hkv=2, D=256, page_size=16,
                       seq_lens=[100, 80], num_pages=20, seed=640)
    bt = wl.block_table.copy()
    bt[0, 2] = wl.num_pages + 5
    bad = W.Workload(**{**wl.__dict__, "block_table": bt})
    res = _gpu.run(_gpu.DeviceWorkload(bad), 1)
    assert pa.paged_attn_last_error_word() & 1
    rows = oracle.all_rows(1, 1, wl.Hq)
    rows[:, 0] = 1
    ref = oracle.workload_rows(wl, split_kv=1, row_bih=rows)
    _gpu.assert_close(res["out"][1, 0], ref["out"], "bf16", "sequence 1")
    assert np.isfinite(res["out"][0]).all()


def test_d256_decode_full(pa):
    """The benchmarked head-dim-256 decode (B=128, L=4096, Hq=16, Hkv=8, 2 x 2 GiB pools drawn on the
    device) in its bench launch (split 1) on sampled sequences, every head."""
    wl = W.d256_decode()
    dw = _gpu.DeviceWorkload(wl)
    k, v = dw.host_pools()
    res = _gpu.run(dw, 1)
    assert not np.isnan(res["out"]).any() and np.isfinite(res["lse"]).all()
    seqs = [0, 1, 63, 64, 100, 127]
    b, h = np.meshgrid(np.asarray(seqs), np.arange(wl.Hq), indexing="ij")
    rows = np.stack([b.ravel(), np.zeros(b.size, dtype=np.int64), h.ravel()], axis=1).astype(np.int32)
    ref = oracle.workload_rows(wl, split_kv=1, row_bih=rows, k_cache=k, v_cache=v)
    _gpu.compare_rows(res, ref, rows, wl, 1, "d256 full")
    assert pa.paged_attn_last_error_word() == 0
