"""GPU parity of the FP8 E4M3 pool path (one float scale per (page, kv head)) against the fp64
oracle's quantized reading: value = E4M3 element x its (page, kv head) scale.

Both sides read the same stored bits and scales; the kernel keeps the stored elements exact on the
tensor cores and adds only the float32 products scale x k_scale and p x v_scale, so the bars are those
of the 16-bit path: bf16/f16 atol=2e-3, rtol=2^-8, the -inf pattern exact, no NaN.
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


def _full(wl, split_kv, **kw):
    dw = _gpu.DeviceWorkload(wl)
    res = _gpu.run(dw, split_kv)
    rows = oracle.all_rows(wl.B, wl.Sq, wl.Hq)
    ref = oracle.workload_rows_kvq(wl, split_kv=split_kv, row_bih=rows)
    _gpu.compare_rows(res, ref, rows, wl, split_kv, f"{wl.name} S={split_kv}")
    return res


# ----------------------------------------------------------------------------- decode mode (<= 16 rows)
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("split_kv", [1, 3, 8])
def test_ragged_decode_fp8(pa, dtype, split_kv):
    """GQA 16, D=128, ps=16, lengths spanning 0..~1000 (several 64-key stages, ragged tails, empty
    trailing partitions), shuffled pages."""
    lens = [0, 1, 15, 16, 17, 63, 64, 65, 200, 511, 777, 1000]
    wl = W.make_custom_fp8(name="ragged_fp8", dtype=dtype, B=len(lens), Sq=1, Hq=64, Hkv=4, D=128, page_size=16,
                           seq_lens=lens, num_pages=200, seed=31)
    res = _full(wl, split_kv)
    assert np.all(res["lse"][0] == -np.inf) and not res["out"][0].any()   # L = 0: output 0, lse -inf
    _check_clean(pa)


@pytest.mark.parametrize("D,ps,G,Sq", [(64, 16, 8, 2), (64, 32, 4, 1), (128, 64, 2, 4), (128, 32, 1, 1)])
def test_decode_fp8_shapes(pa, D, ps, G, Sq):
    """Head dims 64/128, pages of 16/32/64 tokens, several query tokens per row tile, single-head rows."""
    lens = [5, 64, 129, 333, 700]
    Hkv = 2
    wl = W.make_custom_fp8(name=f"fp8_D{D}_ps{ps}", dtype="bf16", B=len(lens), Sq=Sq, Hq=G * Hkv, Hkv=Hkv, D=D,
                           page_size=ps, seq_lens=lens, seed=100 + D + ps, causal=Sq > 1)
    for S in (1, 2):
        _full(wl, S)
    _check_clean(pa)


# ----------------------------------------------------------------------------- prefill mode (> 16 rows)
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_causal_prefill_fp8(pa, dtype):
    """64-row tiles over all 64 keys of a stage: Sq=40 x G=4 = 160 rows (3 tiles, ragged), causal with
    explicit q_offset (including one that hides every key from the first rows)."""
    lens = [40, 300, 1000]
    wl = W.make_custom_fp8(name="prefill_fp8", dtype=dtype, B=3, Sq=40, Hq=16, Hkv=4, D=128, page_size=16,
                           seq_lens=lens, causal=True, q_offset=[-5, 260, 960], seed=77)
    for S in (1, 4):
        res = _full(wl, S)
        assert np.isneginf(res["lse"][0, :5]).all()   # rows whose causal reach is below key 0
    _check_clean(pa)


# ----------------------------------------------------------------------------- edge cases
def test_fp8_extreme_scales_and_subnormals(pa):
    """Scales from 1e-30 to 1e+30 across pages, and pools holding every E4M3 code except NaN
    (subnormals, +-0, +-448): the scores and weights stay in float32 range as the products say."""
    lens = [256, 130]
    wl = W.make_custom_fp8(name="fp8_scales", dtype="bf16", B=2, Sq=1, Hq=8, Hkv=2, D=128, page_size=16,
                           seq_lens=lens, seed=5)
    rng = np.random.default_rng(9)
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    k = rng.choice(codes, size=wl.k_cache.shape).astype(np.uint8)
    v = rng.choice(codes, size=wl.v_cache.shape).astype(np.uint8)
    ks = (10.0 ** rng.uniform(-30, -1, size=wl.k_scale.shape)).astype(np.float32)   # scores stay moderate
    vs = (10.0 ** rng.uniform(-30, 30, size=wl.v_scale.shape)).astype(np.float32)
    wl = W.Workload(**{**wl.__dict__, "k_cache": k, "v_cache": v, "k_scale": ks, "v_scale": vs})
    _full(wl, 1)
    _full(wl, 2)
    _check_clean(pa)


def test_fp8_bad_page_id_reads_zero(pa):
    """A page id past the pool is not dereferenced: its rows count as zeros (scale 0) and the error
    word reports it.  The oracle rejects such a table, so the reference is the same sequence with that
    slot pointing at an all-zero page."""
    lens = [100, 80]
    wl = W.make_custom_fp8(name="fp8_badpage", dtype="bf16", B=2, Sq=1, Hq=8, Hkv=2, D=128, page_size=16,
                           seq_lens=lens, num_pages=20, seed=12)
    bt = wl.block_table.copy()
    bt[0, 2] = wl.num_pages + 1000
    bad = W.Workload(**{**wl.__dict__, "block_table": bt})
    dw = _gpu.DeviceWorkload(bad)
    res = _gpu.run(dw, 1)
    assert pa.paged_attn_last_error_word() & 1
    # reference: an extra zero page with scale 0 at the bad slot
    k = np.concatenate([wl.k_cache, np.zeros_like(wl.k_cache[:1])])
    v = np.concatenate([wl.v_cache, np.zeros_like(wl.v_cache[:1])])
    ks = np.concatenate([wl.k_scale, np.zeros_like(wl.k_scale[:1])])
    vs = np.concatenate([wl.v_scale, np.zeros_like(wl.v_scale[:1])])
    bt_ref = wl.block_table.copy()
    bt_ref[0, 2] = wl.num_pages
    ref_wl = W.Workload(**{**wl.__dict__, "block_table": bt_ref, "num_pages": wl.num_pages + 1, "k_cache": k,
                           "v_cache": v, "k_scale": ks, "v_scale": vs})
    rows = oracle.all_rows(wl.B, wl.Sq, wl.Hq)
    ref = oracle.workload_rows_kvq(ref_wl, split_kv=1, row_bih=rows)
    _gpu.compare_rows(res, ref, rows, wl, 1, "fp8 bad page")


def test_fp8_singlecall_matches_two_calls(pa):
    """paged_attn_fwd_kvq_splitkv (forward + combine in one call, automatic split) equals the oracle."""
    import torch
    lens = [3000, 17, 1500, 64]
    wl = W.make_custom_fp8(name="fp8_single", dtype="bf16", B=4, Sq=1, Hq=32, Hkv=8, D=128, page_size=16,
                           seq_lens=lens, seed=3)
    dw = _gpu.DeviceWorkload(wl)
    S = pa.paged_attn_auto_split(dw.q, dw.k, dw.bt)
    assert S > 1
    ws = torch.empty(pa.paged_attn_workspace_bytes(dw.q, dw.k, dw.bt), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(dw.q)
    lse = torch.empty((wl.B, 1, wl.Hq), dtype=torch.float32, device="cuda")
    pa.paged_attn_fwd_kvq_splitkv(dw.q, dw.k, dw.v, dw.ks, dw.vs, dw.bt, dw.sl, False, None, 0, wl.scale, out, lse,
                                  ws)
    torch.cuda.synchronize()
    rows = oracle.all_rows(wl.B, wl.Sq, wl.Hq)
    ref = oracle.workload_rows_kvq(wl, split_kv=S, row_bih=rows)
    res = {"out": _gpu.to_f64(out, "bf16"), "lse": _gpu.to_f64(lse, "f32")}
    _gpu.assert_close(res["out"][rows[:, 0], rows[:, 1], rows[:, 2]], ref["comb_out"], "bf16", "single-call out")
    _gpu.assert_close(res["lse"][rows[:, 0], rows[:, 1], rows[:, 2]], ref["comb_lse"], "bf16", "single-call lse")
    _check_clean(pa)


# ----------------------------------------------------------------------------- full size (1-GiB pools)
@pytest.fixture(scope="module")
def llama8b_fp8():
    wl = W.llama8b_decode_fp8()
    dw = _gpu.DeviceWorkload(wl)
    k, v = dw.host_pools()
    ks, vs = dw.host_scales()
    return wl, dw, k, v, ks, vs


@pytest.mark.parametrize("split_kv", [1, 4])
def test_llama8b_decode_fp8(pa, llama8b_fp8, split_kv):
    """The benchmarked launch (B=256, L=4096, GQA 4, 65536 pages): every row, and at split 4 every
    partial."""
    wl, dw, k, v, ks, vs = llama8b_fp8
    res = _gpu.run(dw, split_kv)
    assert not np.isnan(res["out"]).any() and np.isfinite(res["lse"]).all()
    ref = _gpu.oracle_all_rows(wl, 4, k, v, ks, vs)   # its unsplit result is the split-1 reference
    _gpu.compare_all(res, ref, wl, split_kv, f"llama8b fp8 S={split_kv}")
    _check_clean(pa)
