"""GPU edge cases: empty and ragged sequences, shapes at the envelope, every variant,
bit-exact gather / plan / shuffle invariance, the combine kernel alone, and the
device error word on out-of-range page ids."""
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


def _full_check(wl, split_kv, variant=0, what=""):
    dw = _gpu.DeviceWorkload(wl)
    res = _gpu.run(dw, split_kv, variant)
    rows = oracle.all_rows(wl.B, wl.Sq, wl.Hq)
    ref = oracle.workload_rows(wl, split_kv=split_kv, row_bih=rows)
    _gpu.compare_rows(res, ref, rows, wl, split_kv, what or wl.name)
    return res, dw


LENS = [0, 1, 15, 16, 17, 63, 64, 65, 200, 129]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("split_kv", [1, 3, 64])
@pytest.mark.parametrize("variant", [0, 1, 3])
def test_ragged_lengths_gqa4(pa, dtype, split_kv, variant):
    wl = W.make_custom(dtype=dtype, B=len(LENS), Sq=1, Hq=8, Hkv=2, D=128, page_size=16, seq_lens=LENS,
                       num_pages=64, W=16, seed=101)
    res, _ = _full_check(wl, split_kv, variant, f"ragged {dtype} S={split_kv} v={variant}")
    b0 = LENS.index(0)
    assert np.all(res["out"][b0] == 0) and np.all(res["lse"][b0] == -np.inf)
    assert pa.paged_attn_last_error_word() == 0


@pytest.mark.parametrize("page_size", [16, 32, 64])
@pytest.mark.parametrize("D", [64, 128])
def test_page_sizes_and_head_dims(pa, page_size, D):
    lens = [1, 33, 130, 300, 64 * 3]
    wl = W.make_custom(dtype="bf16", B=len(lens), Sq=1, Hq=16, Hkv=2, D=D, page_size=page_size, seq_lens=lens,
                       seed=102 + page_size + D)
    for S in (1, 4):
        _full_check(wl, S, 0, f"ps={page_size} D={D} S={S}")
    assert pa.paged_attn_last_error_word() == 0


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_single_head_decode(pa, dtype):
    """G = 1 decode runs on CUDA cores."""
    wl = W.make_custom(dtype=dtype, B=3, Sq=1, Hq=4, Hkv=4, D=128, page_size=16, seq_lens=[5, 100, 513], seed=103)
    for S in (1, 2):
        _full_check(wl, S, 0, f"G=1 {dtype} S={S}")


@pytest.mark.parametrize("Sq,Hq,Hkv", [(2, 8, 1), (3, 8, 2), (4, 4, 4), (1, 32, 2)])
def test_multi_token_decode(pa, Sq, Hq, Hkv):
    """Several query tokens per sequence (speculative decode shapes), causal with default offsets."""
    lens = [Sq, 40, 257]
    wl = W.make_custom(dtype="bf16", B=3, Sq=Sq, Hq=Hq, Hkv=Hkv, D=128, page_size=16, seq_lens=lens, causal=True,
                       seed=104 + Sq)
    for variant in (0, 1, 3):
        _full_check(wl, 2, variant, f"Sq={Sq} G={Hq // Hkv} v={variant}")


@pytest.mark.parametrize("variant", [0, 1])
def test_causal_prefill_small(pa, variant):
    qo = [0, 5, 40, -3]
    Sq = 70
    lens = [o + Sq for o in qo[:3]] + [50]
    wl = W.make_custom(dtype="bf16", B=4, Sq=Sq, Hq=8, Hkv=2, D=128, page_size=16, seq_lens=lens, causal=True,
                       q_offset=qo, seed=105)
    for S in (1, 4, 16):
        _full_check(wl, S, variant, f"prefill-small S={S} v={variant}")


def test_noncausal_prefill_and_default_offset(pa):
    wl = W.make_custom(dtype="f16", B=2, Sq=33, Hq=4, Hkv=4, D=64, page_size=32, seq_lens=[33, 90], causal=False,
                       seed=106)
    _full_check(wl, 3, 0, "noncausal prefill")
    wl2 = W.make_custom(dtype="bf16", B=2, Sq=33, Hq=8, Hkv=2, D=128, page_size=16, seq_lens=[33, 90],
                        causal=True, seed=107)
    _full_check(wl2, 2, 0, "causal prefill, offsets from seq_lens")


def test_split_larger_than_pages(pa):
    wl = W.make_custom(dtype="bf16", B=2, Sq=1, Hq=16, Hkv=1, D=128, page_size=16, seq_lens=[17, 3], seed=108)
    res, _ = _full_check(wl, 64, 0, "S=64")
    assert np.isneginf(res["part_lse"][2:]).all()


def test_shuffle_invariance_bit_exact(pa):
    """Contiguous vs shuffled physical pages: identical output bits (rocMLIR PR #2222, Key Changes 2)."""
    import torch
    base = W.make_custom(dtype="bf16", B=4, Sq=1, Hq=16, Hkv=4, D=128, page_size=16, seq_lens=[100, 37, 512, 1],
                         num_pages=48, W=32, seed=109, shuffle=False)
    rng = np.random.default_rng(5)
    perm = rng.permutation(base.num_pages)
    k2, v2 = np.empty_like(base.k_cache), np.empty_like(base.v_cache)
    k2[perm] = base.k_cache
    v2[perm] = base.v_cache
    bt2 = base.block_table.copy()
    nb = base.nblk()
    for b in range(base.B):
        bt2[b, :nb[b]] = perm[base.block_table[b, :nb[b]]]
    shuf = W.Workload(**{**base.__dict__, "block_table": bt2, "k_cache": k2, "v_cache": v2})
    for S in (1, 3):
        r1 = _gpu.run(_gpu.DeviceWorkload(base), S)
        r2 = _gpu.run(_gpu.DeviceWorkload(shuf), S)
        for key in r1:
            assert np.array_equal(r1[key], r2[key]), key


def test_debug_gather_bit_exact(pa):
    import torch
    for dt in ("bf16", "f32", "f16"):
        wl = W.make_custom(dtype=dt, B=5, Sq=1, Hq=4, Hkv=2, D=64, page_size=16, seq_lens=[0, 1, 16, 17, 100],
                           W=8, seed=110)
        dw = _gpu.DeviceWorkload(wl)
        T = 112
        got = pa.paged_attn_debug_gather(dw.k, dw.bt, dw.sl, T)
        torch.cuda.synchronize()
        got64 = _gpu.to_f64(got, dt)
        d = oracle.dims_of(wl)
        for b in range(wl.B):
            L = int(wl.seq_lens[b])
            want = oracle.gather(wl.k_cache, wl.block_table, wl.seq_lens, d, b)
            assert np.array_equal(got64[b, :L], want), (dt, b)
            assert not got64[b, L:].any()
    assert pa.paged_attn_last_error_word() == 0


def test_plan_bit_exact(pa):
    import torch
    rng = np.random.default_rng(111)
    lens = np.concatenate([[0, 1, 16, 17, 4096, 1000], rng.integers(0, 5000, 50)]).astype(np.int32)
    sl = torch.from_numpy(lens).cuda()
    for ps in (16, 32, 64):
        for S in (1, 2, 3, 8, 64, 100):
            got = pa.paged_attn_plan(sl, ps, S).cpu().numpy()
            assert np.array_equal(got, oracle.plan(lens, ps, S)), (ps, S)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
def test_combine_kernel(pa, D, out_dtype):
    import torch
    rng = np.random.default_rng(112 + D)
    S, rows = 5, 300
    po = rng.standard_normal((S, rows, D)).astype(np.float32)
    pl = (rng.standard_normal((S, rows)) * 3).astype(np.float32)
    pl[rng.random((S, rows)) < 0.3] = -np.inf
    pl[:, :7] = -np.inf          # rows with every split empty
    po[np.isneginf(pl)] = 0.0
    ref_out, ref_lse = oracle.combine(np.moveaxis(po, 0, 1).astype(np.float64), pl.T.astype(np.float64))
    tdt = W.torch_dtype(out_dtype)
    out = torch.empty((rows, D), dtype=tdt, device="cuda")
    lse = torch.empty((rows,), dtype=torch.float32, device="cuda")
    pa.paged_attn_combine(torch.from_numpy(po).cuda(), torch.from_numpy(pl).cuda(), out, lse)
    torch.cuda.synchronize()
    _gpu.assert_close(_gpu.to_f64(out, out_dtype), ref_out, "bf16" if out_dtype == "bf16" else "f32", "combine out")
    _gpu.assert_close(_gpu.to_f64(lse, "f32"), ref_lse, "f32", "combine lse")
    assert not _gpu.to_f64(out, out_dtype)[:7].any()


def test_out_of_range_page_is_flagged_not_read(pa):
    """A page id outside the pool inside a sequence's pages: the kernel's own bounds check skips the
    read (zeros) and raises PA_ERRBIT_PAGE_RANGE; other sequences are unaffected."""
    wl = W.make_custom(dtype="bf16", B=2, Sq=1, Hq=8, Hkv=2, D=128, page_size=16, seq_lens=[40, 50], num_pages=8,
                       W=4, seed=113)
    bt = wl.block_table.copy()
    bt[0, 1] = 1 << 30
    bad = W.Workload(**{**wl.__dict__, "block_table": bt})
    for variant in (0, 1):
        assert pa.paged_attn_last_error_word() == 0
        res = _gpu.run(_gpu.DeviceWorkload(bad), 1, variant)
        status, bits = pa.paged_attn_last_error_status()
        assert bits & pa.ERRBIT_PAGE_RANGE and status == pa.PA_EBOUNDS
        assert pa.paged_attn_last_error_status() == (pa.PA_OK, 0)   # read and cleared
        rows = oracle.all_rows(1, 1, wl.Hq)
        rows[:, 0] = 1
        ref = oracle.workload_rows(wl, split_kv=1, row_bih=rows)
        _gpu.assert_close(res["out"][1, 0], ref["out"], "bf16", "unaffected sequence")
        assert np.isfinite(res["out"]).all()


def test_api_errors(pa):
    import torch
    wl = W.make_custom(dtype="bf16", B=1, Sq=1, Hq=4, Hkv=2, D=128, page_size=16, seq_lens=[5], seed=114)
    dw = _gpu.DeviceWorkload(wl)
    out = torch.empty_like(dw.q)
    with pytest.raises(pa.PagedAttnError) as e:     # split > 1 needs lse
        pa.paged_attn_fwd(dw.q, dw.k, dw.v, dw.bt, dw.sl, False, None, 2, 0.1, out, None)
    assert e.value.code == -1
    with pytest.raises(pa.PagedAttnError) as e:     # tensor-core decode cannot run f32
        q32 = dw.q.float()
        pa.paged_attn_fwd_variant(q32, dw.k.float(), dw.v.float(), dw.bt, dw.sl, False, None, 1, 0.1,
                                  torch.empty_like(q32), None, 2)
    assert e.value.code == -3


def test_bounded_wait_gives_up_and_context_survives(pa):
    """Failure path without a fault: a pipeline wait on a barrier nothing completes gives up after
    its limit (here 50 ms), sets the time-out bit, and the next attention call still runs exactly."""
    import time
    import torch
    assert pa.paged_attn_last_error_word() == 0
    t0 = time.perf_counter()
    pa.paged_attn_debug_wait_timeout(50_000)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert 0.04 < dt < 5.0
    assert pa.paged_attn_last_error_status() == (pa.PA_ETIMEOUT, pa.ERRBIT_TIMEOUT)
    assert pa.paged_attn_last_error_status() == (pa.PA_OK, 0)  # read and cleared
    wl = W.make_custom(dtype="bf16", B=2, Sq=1, Hq=8, Hkv=2, D=128, page_size=16, seq_lens=[33, 90], seed=77)
    res = _gpu.run(_gpu.DeviceWorkload(wl), 2)
    rows = oracle.all_rows(wl.B, wl.Sq, wl.Hq)
    _gpu.compare_rows(res, oracle.workload_rows(wl, split_kv=2, row_bih=rows), rows, wl, 2, "after time-out")
    assert pa.paged_attn_last_error_word() == 0


@pytest.mark.parametrize("S", [2, 3, 5, 8, 13])
@pytest.mark.parametrize("ps,D,dtype", [(16, 128, "bf16"), (32, 64, "f16"), (64, 128, "f16")])
def test_split_group_decode(pa, S, ps, D, dtype):
    """Decode with short splits (every split at most 8 pages), forced: one CTA per four consecutive
    splits, one warp per split (the planner takes it for the ragged decode's 1024 splits: B=32,
    Hkv=4, split 8).  Partial last groups, empty splits inside a group, sentinel tails, 1-3 query
    tokens with causal offsets, every row against the oracle."""
    lens = [0, 1, 15, ps, ps + 1, 3 * ps - 1, 5 * ps + 3, 8 * ps * S // 2 + 7]
    width = max(-(-max(lens) // ps), 1)
    assert -(-width // S) <= 8
    for Sq, Hq, Hkv in [(1, 16, 1), (3, 8, 2)]:
        qo = [max(L - Sq, 0) for L in lens] if Sq > 1 else None
        wl = W.make_custom(dtype=dtype, B=len(lens), Sq=Sq, Hq=Hq, Hkv=Hkv, D=D, page_size=ps, seq_lens=lens,
                           W=width, causal=Sq > 1, q_offset=qo, seed=140 + S + ps + Sq)
        _full_check(wl, S, pa.VARIANT_MMA_SPLIT_GROUP, f"split group S={S} ps={ps} D={D} Sq={Sq}")
    assert pa.paged_attn_last_error_word() == 0


CLIP_CASES = [
    # (name, variant, workload kwargs)
    ("gqa decode", 2, dict(dtype="bf16", Sq=1, Hq=8, Hkv=2, D=128, page_size=16)),
    ("single-head decode", 1, dict(dtype="bf16", Sq=1, Hq=4, Hkv=4, D=128, page_size=32)),
    ("f32 cuda cores", 1, dict(dtype="f32", Sq=2, Hq=4, Hkv=2, D=64, page_size=16, causal=True)),
    ("mma prefill", 3, dict(dtype="f16", Sq=20, Hq=8, Hkv=2, D=64, page_size=16, causal=True)),
    ("tcgen05 prefill", 4, dict(dtype="bf16", Sq=64, Hq=8, Hkv=2, D=128, page_size=16, causal=True)),
    ("head dim 256", 5, dict(dtype="bf16", Sq=3, Hq=8, Hkv=2, D=256, page_size=16, causal=True)),
]


@pytest.mark.parametrize("name,variant,kw", CLIP_CASES, ids=[c[0] for c in CLIP_CASES])
@pytest.mark.parametrize("S", [1, 3])
def test_overlong_sequence_is_clipped(pa, name, variant, kw, S):
    """seq_lens[b] beyond the block-table row (bt_stride x page_size tokens) is clipped to the row: the
    result is that of the clipped length (the default query offset follows it), the other sequences
    are exact, and PA_ERRBIT_SEQ_CLIPPED is set (a status of PA_OK: nothing outside the row is read)."""
    W_ = 6
    row = W_ * kw["page_size"]
    clipped = [row, 70, row]
    wl = W.make_custom(B=3, seq_lens=clipped, W=W_, seed=6161, **kw)
    over = W.Workload(**{**wl.__dict__, "seq_lens": np.array([row + 7, 70, row + 300], dtype=np.int32)})
    assert pa.paged_attn_last_error_word() == 0
    res = _gpu.run(_gpu.DeviceWorkload(over), S, variant)
    status, bits = pa.paged_attn_last_error_status()
    assert bits == pa.ERRBIT_SEQ_CLIPPED and status == pa.PA_OK
    rows = oracle.all_rows(wl.B, wl.Sq, wl.Hq)
    _gpu.compare_rows(res, oracle.workload_rows(wl, split_kv=S, row_bih=rows), rows, wl, S, f"{name} clipped S={S}")


def test_overlong_sequence_is_clipped_fp8(pa):
    """The same clipping on the 8-bit-pool decode kernel."""
    W_ = 5
    wl = W.make_custom_fp8(dtype="bf16", B=3, Sq=1, Hq=8, Hkv=2, D=128, page_size=16, seq_lens=[80, 33, 80], W=W_,
                           seed=6162)
    over = W.Workload(**{**wl.__dict__, "seq_lens": np.array([81, 33, 500], dtype=np.int32)})
    res = _gpu.run(_gpu.DeviceWorkload(over), 2)
    assert pa.paged_attn_last_error_word() == pa.ERRBIT_SEQ_CLIPPED
    rows = oracle.all_rows(wl.B, wl.Sq, wl.Hq)
    _gpu.compare_rows(res, oracle.workload_rows_kvq(wl, split_kv=2, row_bih=rows), rows, wl, 2, "fp8 clipped")
