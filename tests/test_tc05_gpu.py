"""GPU parity of the tcgen05 (tensor-memory) kernel against the oracle: prefill and long query
runs over paged K/V, causal with per-sequence offsets, GQA groups that divide 128, every page
size, split partitions (including empty and fully masked ones), bf16 and f16."""
import numpy as np
import pytest

import oracle
from paged_kv_cache_201_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu
TC05 = 4


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_201_gb300 as pa
    pa.load_library(build_if_missing=True)
    return pa


def _check(wl, S, what):
    dw = _gpu.DeviceWorkload(wl)
    res = _gpu.run(dw, S, TC05)
    rows = oracle.all_rows(wl.B, wl.Sq, wl.Hq)
    ref = oracle.workload_rows(wl, split_kv=S, row_bih=rows)
    _gpu.compare_rows(res, ref, rows, wl, S, what)
    return res


@pytest.mark.parametrize("S", [1, 4, 16])
def test_tc05_causal_prefill_small(pa, S):
    qo = [0, 5, 40, -3]
    Sq = 70
    lens = [o + Sq for o in qo[:3]] + [50]
    wl = W.make_custom(dtype="bf16", B=4, Sq=Sq, Hq=8, Hkv=2, D=128, page_size=16, seq_lens=lens, causal=True,
                       q_offset=qo, seed=205)
    _check(wl, S, f"tc05 prefill-small S={S}")
    assert pa.paged_attn_last_error_word() == 0


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
def test_tc05_gqa_groups(pa, G):
    Hkv = 2
    wl = W.make_custom(dtype="bf16", B=2, Sq=300 // G + 3, Hq=G * Hkv, Hkv=Hkv, D=128, page_size=16,
                       seq_lens=[400, 333], causal=True, seed=206 + G)
    _check(wl, 2, f"tc05 G={G}")


@pytest.mark.parametrize("page_size", [16, 32, 64])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_tc05_page_sizes_dtypes(pa, page_size, dtype):
    wl = W.make_custom(dtype=dtype, B=3, Sq=40, Hq=16, Hkv=4, D=128, page_size=page_size,
                       seq_lens=[40, 170, 260], causal=True, q_offset=[0, 100, 220], seed=207 + page_size)
    for S in (1, 3):
        _check(wl, S, f"tc05 ps={page_size} {dtype} S={S}")


def test_tc05_noncausal_and_decode_shapes(pa):
    wl = W.make_custom(dtype="bf16", B=2, Sq=33, Hq=8, Hkv=2, D=128, page_size=16, seq_lens=[33, 290],
                       causal=False, seed=208)
    _check(wl, 2, "tc05 noncausal")
    wl = W.make_custom(dtype="bf16", B=5, Sq=1, Hq=16, Hkv=4, D=128, page_size=16, seq_lens=[0, 1, 17, 128, 513],
                       seed=209)
    res = _check(wl, 4, "tc05 decode shape")
    assert np.all(res["lse"][0] == -np.inf)


def test_tc05_causal_prefill_full(pa):
    """The full causal prefill workload (B=4, Sq=1024, q_offset up to 3072) on the forced tcgen05
    variant: every row at split 8 (partials of every split included) and at split 1."""
    wl = W.causal_prefill()
    dw = _gpu.DeviceWorkload(wl)
    ref = _gpu.oracle_all_rows(wl, 8)   # its unsplit result is the split-1 reference
    for S in (8, 1):
        res = _gpu.run(dw, S, TC05)
        assert not np.isnan(res["out"]).any()
        _gpu.compare_all(res, ref, wl, S, f"tc05 full prefill S={S}")
    assert pa.paged_attn_last_error_word() == 0


def test_tc05_out_of_range_page(pa):
    wl = W.make_custom(dtype="bf16", B=2, Sq=64, Hq=8, Hkv=2, D=128, page_size=16, seq_lens=[100, 90], causal=True,
                       num_pages=16, W=8, seed=210)
    bt = wl.block_table.copy()
    bt[0, 2] = 1 << 29
    bad = W.Workload(**{**wl.__dict__, "block_table": bt})
    assert pa.paged_attn_last_error_word() == 0
    res = _gpu.run(_gpu.DeviceWorkload(bad), 1, TC05)
    assert pa.paged_attn_last_error_word() & pa.ERRBIT_PAGE_RANGE
    rows = oracle.all_rows(1, wl.Sq, wl.Hq)
    rows[:, 0] = 1
    ref = oracle.workload_rows(wl, split_kv=1, row_bih=rows)
    _gpu.assert_close(res["out"][1].reshape(-1, wl.D), ref["out"], "bf16", "unaffected sequence")


def test_tc05_many_units_per_cta(pa):
    """More work units than SMs: each persistent CTA walks several units (ragged causal lengths,
    empty and partial splits), so the cross-unit pipeline (Q and O double buffers) is exercised."""
    rng = np.random.default_rng(211)
    B, Sq = 8, 256
    qo = rng.integers(0, 300, size=B).tolist()
    lens = [o + Sq for o in qo]
    wl = W.make_custom(dtype="bf16", B=B, Sq=Sq, Hq=16, Hkv=2, D=128, page_size=16, seq_lens=lens, causal=True,
                       q_offset=qo, seed=212)
    for S in (4, 1):
        _check(wl, S, f"tc05 many units S={S}")
    assert pa.paged_attn_last_error_word() == 0


@pytest.mark.parametrize("scale_mult", [1.0, 8.0])
def test_tc05_f16_single_product(pa, scale_mult):
    """f16 runs P V as one product with P rounded to f16: causal prefill rows including peaky
    softmaxes (scores scaled up 8x, so a few keys carry the weight), every row against the oracle."""
    lens = [70, 333, 1000]
    wl = W.make_custom(dtype="f16", B=3, Sq=64, Hq=8, Hkv=2, D=128, page_size=16, seq_lens=lens, causal=True,
                       seed=880, scale=scale_mult / np.sqrt(128))
    for S in (1, 3):
        res = _gpu.run(_gpu.DeviceWorkload(wl), S, variant=4)
        rows = oracle.all_rows(wl.B, wl.Sq, wl.Hq)
        ref = oracle.workload_rows(wl, split_kv=S, row_bih=rows)
        _gpu.compare_rows(res, ref, rows, wl, S, f"f16 tc05 x{scale_mult} S={S}")
    assert pa.paged_attn_last_error_word() == 0


def test_tc05_split1_schedule_orders(pa):
    """split_kv = 1 hands units out longest sequence first (sequences ordered by key count in the
    CTA, ties by index) to CTAs that take the next one by cancelling a pending CTA's launch.  Equal
    lengths (ties), a zero-length and a fully masked sequence (units with no key tile), against the
    oracle; and the result does not depend on which CTA took which unit: a second run is bit-identical."""
    Sq = 128
    qo = [200, 200, 0, 37, -Sq, 200]
    lens = [328, 328, 0, 165, 40, 328]
    wl = W.make_custom(dtype="bf16", B=6, Sq=Sq, Hq=16, Hkv=2, D=128, page_size=16, seq_lens=lens, causal=True,
                       q_offset=qo, seed=213)
    dw = _gpu.DeviceWorkload(wl)
    first = _gpu.run(dw, 1, TC05)
    rows = oracle.all_rows(wl.B, wl.Sq, wl.Hq)
    _gpu.compare_rows(first, oracle.workload_rows(wl, split_kv=1, row_bih=rows), rows, wl, 1, "tc05 split-1 order")
    assert np.all(first["lse"][2] == -np.inf) and np.all(first["lse"][4] == -np.inf)
    again = _gpu.run(dw, 1, TC05)
    for key in first:
        assert np.array_equal(first[key], again[key], equal_nan=True), key
    assert pa.paged_attn_last_error_word() == 0


@pytest.mark.parametrize("empty", ["length0", "masked", "all0"])
def test_tc05_split1_runs_of_empty_units(pa, empty):
    """Units with no key tile in long runs.  length0: 60 sequences of length 0 come after the four
    real ones in the split-1 order, 3840 empty units for ~150 CTAs, so a CTA takes far more of them
    in a row than the unit ring holds while the last product of its last real unit is still held
    back.  masked: the 60 are fully masked instead (q_offset -Sq) and long, so they come first.
    all0: every sequence has length 0.  Every row against the oracle (rows with no key: output 0,
    lse -inf), and no wait gives up."""
    B, Sq = 64, 256
    lens, qo = ([0] * B, [0] * B) if empty != "masked" else ([600] * B, [-Sq] * B)
    real = (0, 17, 33, 50) if empty != "all0" else ()
    for b, (L, o) in zip(real, ((300, 44), (256, 0), (400, 144), (280, 24))):
        lens[b], qo[b] = L, o
    wl = W.make_custom(dtype="bf16", B=B, Sq=Sq, Hq=32, Hkv=8, D=128, page_size=16, seq_lens=lens, causal=True,
                       q_offset=qo, seed=216)
    res = _check(wl, 1, f"tc05 split-1 empty runs ({empty})")
    assert np.all(res["lse"][[b for b in range(B) if b not in real]] == -np.inf)
    assert pa.paged_attn_last_error_word() == 0


def test_tc05_split1_batch_past_the_sort(pa):
    """More sequences than the in-CTA ordering takes (256): the schedule falls back to the last
    sequence first.  300 sequences of 16 query tokens (G = 4: one 64-row tile each), ragged
    lengths, far more units than SMs, every row against the oracle."""
    rng = np.random.default_rng(214)
    B, Sq = 300, 16
    qo = rng.integers(0, 200, size=B).tolist()
    lens = [o + Sq for o in qo]
    wl = W.make_custom(dtype="bf16", B=B, Sq=Sq, Hq=8, Hkv=2, D=128, page_size=16, seq_lens=lens, causal=True,
                       q_offset=qo, seed=215)
    _check(wl, 1, "tc05 split-1 B=300")
    assert pa.paged_attn_last_error_word() == 0


def test_tc05_split1_in_cuda_graph(pa):
    """The split-1 schedule takes its units by cancelling its own grid's pending CTAs, so every launch
    carries its own schedule: replays of a captured call give the eager call's bits."""
    import torch
    wl = W.causal_prefill()
    dw = _gpu.DeviceWorkload(wl)
    eager = _gpu.run(dw, 1, TC05)
    out = torch.empty_like(dw.q)
    lse = torch.empty((wl.B, wl.Sq, wl.Hq), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):   # warm-up outside the capture
        pa.paged_attn_fwd_variant(dw.q, dw.k, dw.v, dw.bt, dw.sl, wl.causal, dw.qo, 1, wl.scale, out, lse, TC05)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pa.paged_attn_fwd_variant(dw.q, dw.k, dw.v, dw.bt, dw.sl, wl.causal, dw.qo, 1, wl.scale, out, lse, TC05)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(_gpu.to_f64(out, wl.dtype), eager["out"])
        assert np.array_equal(_gpu.to_f64(lse, "f32"), eager["lse"])
    assert pa.paged_attn_last_error_word() == 0
