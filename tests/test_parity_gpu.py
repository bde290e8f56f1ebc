"""GPU parity: the CUDA path against the fp64 oracle on the five seeded workloads.

Small workloads are compared on every output row; the full-size ones on sampled
rows the oracle computes one by one, with the launch configuration the
benchmark times.  Bars: bf16/f16 atol=2e-3, rtol=2^-8; f32 1e-5; -inf patterns
and the absence of NaN exactly.
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


def _prefill_rows(wl):
    toks = [0, 1, 2, 15, 16, 63, 64, 65, 127, 128, 511, 777, 1000, 1022, 1023]
    b, i, h = np.meshgrid(np.arange(wl.B), np.array(toks), np.arange(wl.Hq), indexing="ij")
    return np.stack([b.ravel(), i.ravel(), h.ravel()], axis=1).astype(np.int32)


@pytest.mark.parametrize("split_kv", [8, 1])
def test_causal_prefill(pa, prefill, split_kv):
    wl, dw = prefill
    res = _gpu.run(dw, split_kv)
    assert not np.isnan(res["out"]).any()
    rows = _prefill_rows(wl)
    ref = oracle.workload_rows(wl, split_kv=split_kv, row_bih=rows)
    _gpu.compare_rows(res, ref, rows, wl, split_kv, f"prefill S={split_kv}")
    if split_kv == 8:
        # fully masked partitions (keys all past a row's causal reach) hold exactly (0, -inf)
        assert np.isneginf(res["part_lse"]).any()
        masked = np.isneginf(res["part_lse"])
        assert not res["part_out"][masked].any()
        assert not np.isnan(res["part_out"]).any()
    _check_clean(pa)


# ----------------------------------------------------------------------------- full-size decode (2-GiB pools)
def _sample_rows(wl, seqs):
    b, h = np.meshgrid(np.asarray(seqs), np.arange(wl.Hq), indexing="ij")
    return np.stack([b.ravel(), np.zeros(b.size, dtype=np.int64), h.ravel()], axis=1).astype(np.int32)


@pytest.fixture(scope="module")
def llama8b():
    wl = W.llama8b_decode()
    dw = _gpu.DeviceWorkload(wl)
    k, v = dw.host_pools()
    return wl, dw, k, v


@pytest.mark.parametrize("split_kv", [1, 4])
def test_llama8b_decode(pa, llama8b, split_kv):
    wl, dw, k, v = llama8b
    res = _gpu.run(dw, split_kv)
    assert not np.isnan(res["out"]).any() and np.isfinite(res["lse"]).all()
    rows = _sample_rows(wl, [0, 1, 77, 128, 200, 255])
    ref = oracle.workload_rows(wl, split_kv=split_kv, row_bih=rows, k_cache=k, v_cache=v)
    _gpu.compare_rows(res, ref, rows, wl, split_kv, f"llama8b S={split_kv}")
    _check_clean(pa)


@pytest.fixture(scope="module")
def over2g():
    wl = W.over2gib_decode()
    dw = _gpu.DeviceWorkload(wl)
    k, v = dw.host_pools()
    return wl, dw, k, v


def test_over2gib_decode(pa, over2g):
    wl, dw, k, v = over2g
    page_bytes = wl.page_size * wl.Hkv * wl.D * 2
    assert W.OVER2G_FIRST_HIGH * page_bytes == 2 ** 31
    seqs = [0, 3, 100, 255]
    for b in seqs:  # every sampled sequence reads pages on both sides of byte 2^31
        row = wl.block_table[b]
        assert (row >= W.OVER2G_FIRST_HIGH).any() and (row < W.OVER2G_FIRST_HIGH).any()
    res = _gpu.run(dw, 4)
    assert not np.isnan(res["out"]).any()
    rows = _sample_rows(wl, seqs)
    ref = oracle.workload_rows(wl, split_kv=4, row_bih=rows, k_cache=k, v_cache=v)
    _gpu.compare_rows(res, ref, rows, wl, 4, "over2gib S=4")
    _check_clean(pa)
