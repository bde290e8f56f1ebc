"""q as a view: query tokens further apart than their heads, as when q is sliced out of a fused
QKV projection's output [tokens, (Hq + 2 Hkv) x D].  rocMLIR PR #2220 hands attention its operands
through address views; here q's token stride is pa_dims.q_stride.

Every kernel reads q through the same row offset, so a strided q must give bit for bit what the same
values in a dense q give, on every kernel the planner or a forced variant can pick; one case per
kernel family is also checked against the oracle."""
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


def _fused_view(q, extra_heads):
    """A fused buffer [..., Hq + extra_heads, D] holding q in its first Hq heads (the rest filled with
    values that must never be read), and the q view into it."""
    import torch
    shape = list(q.shape)
    shape[-2] += extra_heads
    fused = torch.full(shape, float("nan"), dtype=q.dtype, device=q.device)
    view = fused[..., :q.shape[-2], :]
    view.copy_(q)
    assert not view.is_contiguous()
    return fused, view


def _bits(t):
    import torch
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def _run_both(dw, split_kv, variant, extra_heads):
    """Run the workload with its dense q and with q as a view; return both results (numpy f64)."""
    import torch
    dense = _gpu.run(dw, split_kv, variant)
    dense_q = dw.q
    fused, dw.q = _fused_view(dense_q, extra_heads)
    try:
        strided = _gpu.run(dw, split_kv, variant)
    finally:
        dw.q = dense_q
    del fused
    torch.cuda.synchronize()
    return dense, strided


def _assert_identical(dense, strided, what):
    for key in dense:
        a, b = dense[key], strided[key]
        if key == "part_out":  # rows with lse -inf need not be written (the combine never reads them)
            keep = ~np.isneginf(dense["part_lse"])
            a, b = a[keep], b[keep]
        assert np.array_equal(a, b), f"{what}: {key} differs between dense and strided q"


CASES = [
    # (name, workload kwargs, split, variant)
    ("gqa decode", dict(dtype="bf16", B=5, Sq=1, Hq=16, Hkv=4, D=128, page_size=16, seq_lens=[1, 17, 100, 300, 64]),
     3, 0),
    ("gqa decode f16 d64", dict(dtype="f16", B=3, Sq=2, Hq=8, Hkv=2, D=64, page_size=32, seq_lens=[5, 90, 200],
                                causal=True), 1, 0),
    ("split groups", dict(dtype="bf16", B=40, Sq=1, Hq=8, Hkv=2, D=128, page_size=16,
                          seq_lens=list(range(17, 17 + 40 * 9, 9))), 8, 6),
    ("single-head decode", dict(dtype="bf16", B=4, Sq=1, Hq=8, Hkv=8, D=128, page_size=16,
                                seq_lens=[3, 100, 257, 64]), 2, 0),
    ("f32 cuda cores", dict(dtype="f32", B=3, Sq=2, Hq=4, Hkv=2, D=64, page_size=16, seq_lens=[2, 37, 50],
                            causal=True), 2, 0),
    ("tcgen05 prefill", dict(dtype="bf16", B=2, Sq=80, Hq=8, Hkv=2, D=128, page_size=16, seq_lens=[80, 250],
                             causal=True, q_offset=[0, 170]), 2, 0),
    ("mma prefill", dict(dtype="f16", B=2, Sq=40, Hq=8, Hkv=2, D=128, page_size=16, seq_lens=[40, 140],
                         causal=True), 1, 3),
    ("head dim 256", dict(dtype="bf16", B=3, Sq=3, Hq=8, Hkv=2, D=256, page_size=16, seq_lens=[3, 60, 150],
                          causal=True), 2, 0),
]


@pytest.mark.parametrize("name,kw,S,variant", CASES, ids=[c[0] for c in CASES])
def test_strided_q_bit_identical(pa, name, kw, S, variant):
    wl = W.make_custom(seed=5150, **kw)
    dw = _gpu.DeviceWorkload(wl)
    dense, strided = _run_both(dw, S, variant, extra_heads=2 * wl.Hkv)
    _assert_identical(dense, strided, name)
    rows = oracle.all_rows(wl.B, wl.Sq, wl.Hq)
    _gpu.compare_rows(strided, oracle.workload_rows(wl, split_kv=S, row_bih=rows), rows, wl, S, f"{name} strided")
    assert pa.paged_attn_last_error_word() == 0


@pytest.mark.parametrize("Sq,S", [(1, 3), (40, 1)])
def test_strided_q_fp8_pools(pa, Sq, S):
    wl = W.make_custom_fp8(dtype="bf16", B=3, Sq=Sq, Hq=16, Hkv=4, D=128, page_size=16, seq_lens=[40, 90, 300],
                           causal=True, seed=5151)
    dw = _gpu.DeviceWorkload(wl)
    dense, strided = _run_both(dw, S, 0, extra_heads=8)
    _assert_identical(dense, strided, f"fp8 Sq={Sq}")
    rows = oracle.all_rows(wl.B, wl.Sq, wl.Hq)
    ref = oracle.workload_rows_kvq(wl, split_kv=S, row_bih=rows)
    _gpu.compare_rows(strided, ref, rows, wl, S, f"fp8 Sq={Sq} strided")
    assert pa.paged_attn_last_error_word() == 0


def test_strided_q_varlen(pa):
    """A variable-length batch whose packed q [T, Hq, D] is a view of [T, Hq + 2 Hkv, D]: both of the
    call's kernels (tcgen05 for the long sequences, the one-grid kernel for the rest)."""
    import torch
    q_lens = [100, 1, 3, 1, 70]
    qo = [0, 40, 10, 300, 20]
    seq_lens = [o + n for o, n in zip(qo, q_lens)]
    wl = W.make_varlen(dtype="bf16", Hq=16, Hkv=4, D=128, page_size=16, q_offset=qo, seed=5152, q_lens=q_lens,
                       seq_lens=seq_lens)
    q = W.host_to_torch(wl.q, wl.dtype).cuda()
    k, v = W.host_to_torch(wl.k_cache, wl.dtype).cuda(), W.host_to_torch(wl.v_cache, wl.dtype).cuda()
    bt = torch.from_numpy(np.ascontiguousarray(wl.block_table)).cuda()
    sl = torch.from_numpy(np.ascontiguousarray(wl.seq_lens)).cuda()
    qs = torch.from_numpy(np.ascontiguousarray(wl.q_start)).cuda()
    qof = torch.from_numpy(np.ascontiguousarray(wl.q_offset)).cuda()
    fused, qv = _fused_view(q, 8)
    res = []
    for qq in (q, qv):
        out = torch.empty(q.shape, dtype=q.dtype, device="cuda")
        lse = torch.empty((wl.Sq, wl.Hq), dtype=torch.float32, device="cuda")
        pa.paged_attn_fwd_varlen(qq, k, v, bt, sl, qs, wl.causal, qof, 1, wl.scale, out, lse)
        res.append((out, lse))
    torch.cuda.synchronize()
    assert torch.equal(_bits(res[0][0]), _bits(res[1][0])) and torch.equal(_bits(res[0][1]), _bits(res[1][1]))
    ref = oracle.rows_varlen(q=wl.q, k_cache=wl.k_cache, v_cache=wl.v_cache, block_table=wl.block_table,
                             seq_lens=wl.seq_lens, q_start=wl.q_start, q_offset=wl.q_offset, causal=wl.causal,
                             dims=oracle.dims_of(wl), scale=wl.scale, split_kv=1, want_split=False)
    _gpu.assert_close(_gpu.to_f64(res[1][0], "bf16"), ref["out"], "bf16", "varlen strided out")
    assert pa.paged_attn_last_error_word() == 0
