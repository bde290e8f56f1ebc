"""GPU parity: the CUDA path against the fp64 oracle on the five seeded workloads.

Every workload is compared on every output row (the full-size ones in the
launch configuration the benchmark times), partial outputs and partial lse of
every split included.  Bars: bf16/f16 atol=2e-3, rtol=2^-8; f32 1e-5; -inf
patterns and the absence of NaN exactly.
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


def _check_clean(pa):
    assert pa.paged_attn_last_error_word() == 0


# ----------------------------------------------------------------------------- tiny f32 decode
@pytest.mark.parametrize("split_kv", [1, 2])
def test_tiny_decode_f32(pa, split_kv):
    wl = W.tiny_decode_f32()
    dw = _gpu.DeviceWorkload(wl)
    res = _gpu.run(dw, split_kv)
    rows = oracle.all_rows(wl.B, wl.Sq, wl.Hq)
    ref = oracle.workload_rows(wl, split_kv=split_kv, row_bih=rows)
    _gpu.compare_rows(res, ref, rows, wl, split_kv, f"tiny S={split_kv}")
    _check_clean(pa)  # the -1 tail slots were never read


# ----------------------------------------------------------------------------- ragged decode
@pytest.fixture(scope="module")
def ragged():
    wl = W.ragged_decode()
    return wl, _gpu.DeviceWorkload(wl)


@pytest.mark.parametrize("split_kv", [8, 1])
def test_ragged_decode(pa, ragged, split_kv):
    wl, dw = ragged
    res = _gpu.run(dw, split_kv)
    rows = oracle.all_rows(wl.B, wl.Sq, wl.Hq)
    ref = oracle.workload_rows(wl, split_kv=split_kv, row_bih=rows)
    _gpu.compare_rows(res, ref, rows, wl, split_kv, f"ragged S={split_kv}")
    if split_kv == 8:
        # sequences shorter than 8 pages have empty trailing partitions: (0, -inf)
        plan = oracle.plan(wl.seq_lens, wl.page_size, 8)
        empty = plan[:, :, 0] == plan[:, :, 1]
        assert empty.any()
        for b, s in zip(*np.nonzero(empty)):
            assert np.all(res["part_lse"][s, b] == -np.inf)
            assert not res["part_out"][s, b].any()
    _check_clean(pa)  # the 0x7FFFFFFF tail was never dereferenced


@pytest.mark.parametrize("variant", [1, 3])
def test_ragged_decode_other_variants(pa, ragged, variant):
    """The CUDA-core kernel and the 64-row tensor-core kernel on the same bf16 decode."""
    wl, dw = ragged
    res = _gpu.run(dw, 8, variant=variant)
    rows = oracle.all_rows(wl.B, wl.Sq, wl.Hq)
    ref = oracle.workload_rows(wl, split_kv=8, row_bih=rows)
    _gpu.compare_rows(res, ref, rows, wl, 8, f"ragged variant={variant}")
    _check_clean(pa)


# ----------------------------------------------------------------------------- causal prefill
@pytest.fixture(scope="module")
def prefill():
    wl = W.causal_prefill()
    return wl, _gpu.DeviceWorkload(wl)


@pytest.mark.parametrize("split_kv", [8, 1])
def test_causal_prefill(pa, prefill, split_kv):
    """Every row of the causal prefill workload: 4 x 1024 tokens x 32 heads, and at split 8 all
    eight partial outputs and lse of each row (fully masked partitions included)."""
    wl, dw = prefill
    res = _gpu.run(dw, split_kv)
    assert not np.isnan(res["out"]).any()
    ref = _gpu.oracle_all_rows(wl, 8)   # its unsplit result is the split-1 reference
    _gpu.compare_all(res, ref, wl, split_kv, f"prefill S={split_kv}")
    if split_kv == 8:
        # fully masked partitions (keys all past a row's causal reach) have lse -inf; their partial
        # rows are 0 where written and never read by the combine (a tile whose split holds none of
        # its keys is not written at all); every other partial row is finite
        masked = np.isneginf(res["part_lse"])
        assert masked.any()
        assert np.isfinite(res["part_out"][~masked]).all()
    _check_clean(pa)


# ----------------------------------------------------------------------------- full-size decode (2-GiB pools)
@pytest.fixture(scope="module")
def llama8b():
    wl = W.llama8b_decode()
    dw = _gpu.DeviceWorkload(wl)
    k, v = dw.host_pools()
    return wl, dw, k, v


@pytest.mark.parametrize("split_kv", [1, 4])
def test_llama8b_decode(pa, llama8b, split_kv):
    """Every row of the Llama-3-8B decode (256 sequences x 32 heads over two 2-GiB pools)."""
    wl, dw, k, v = llama8b
    res = _gpu.run(dw, split_kv)
    assert not np.isnan(res["out"]).any() and np.isfinite(res["lse"]).all()
    ref = _gpu.oracle_all_rows(wl, 4, k, v)   # its unsplit result is the split-1 reference
    _gpu.compare_all(res, ref, wl, split_kv, f"llama8b S={split_kv}")
    _check_clean(pa)


@pytest.fixture(scope="module")
def over2g():
    wl = W.over2gib_decode()
    dw = _gpu.DeviceWorkload(wl)
    k, v = dw.host_pools()
    return wl, dw, k, v


def test_over2gib_decode(pa, over2g):
    """Every row of the decode over pools past 2^31 bytes (256 sequences x 64 heads, 8192 keys each),
    every sequence reading pages on both sides of byte 2^31."""
    wl, dw, k, v = over2g
    page_bytes = wl.page_size * wl.Hkv * wl.D * 2
    assert W.OVER2G_FIRST_HIGH * page_bytes == 2 ** 31
    hi = wl.block_table >= W.OVER2G_FIRST_HIGH
    assert hi.any(axis=1).all() and (~hi).any(axis=1).all()
    res = _gpu.run(dw, 4)
    assert not np.isnan(res["out"]).any()
    ref = _gpu.oracle_all_rows(wl, 4, k, v)
    _gpu.compare_all(res, ref, wl, 4, "over2gib S=4")
    _check_clean(pa)


def test_llama8b_decode_over2gib_same_shape(pa):
    """The Llama-3-8B decode shape over pools of 65536 + 2048 pages, every sequence reading pages on
    both sides of byte 2^31: every row at split 1 (the launch the benchmark's same-shape comparison
    times)."""
    wl = W.llama8b_decode_over2gib()
    page_bytes = wl.page_size * wl.Hkv * wl.D * 2
    assert W.LLAMA_OVER2G_FIRST_HIGH * page_bytes == 2 ** 31
    hi = wl.block_table >= W.LLAMA_OVER2G_FIRST_HIGH
    assert hi.any(axis=1).all() and (~hi).any(axis=1).all()
    dw = _gpu.DeviceWorkload(wl)
    k, v = dw.host_pools()
    res = _gpu.run(dw, 1)
    del dw
    ref = _gpu.oracle_all_rows(wl, 1, k, v)
    _gpu.compare_all(res, ref, wl, 1, "llama8b shape past 2^31 S=1")
    _check_clean(pa)
