"""The single-call split-KV forward (workspace + automatic split) against the two-call path and the oracle."""
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


def _single_call(pa, dw, split_kv):
    import torch
    wl = dw.wl
    out = torch.empty_like(dw.q)
    lse = torch.empty((wl.B, wl.Sq, wl.Hq), dtype=torch.float32, device="cuda")
    nbytes = pa.paged_attn_workspace_bytes(dw.q, dw.k, dw.bt, split_kv)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device="cuda")
    pa.paged_attn_fwd_splitkv(dw.q, dw.k, dw.v, dw.bt, dw.sl, wl.causal, dw.qo, split_kv, wl.scale, out, lse, ws)
    torch.cuda.synchronize()
    return out, lse, nbytes


@pytest.mark.parametrize("split_kv", [1, 3, 8])
def test_single_call_equals_two_calls(pa, split_kv):
    wl = W.ragged_decode()
    dw = _gpu.DeviceWorkload(wl)
    out, lse, _ = _single_call(pa, dw, split_kv)
    ref = _gpu.run(dw, split_kv)
    assert np.array_equal(_gpu.to_f64(out, wl.dtype), ref["out"])
    assert np.array_equal(_gpu.to_f64(lse, "f32"), ref["lse"])


def test_auto_split_parity(pa):
    wl = W.ragged_decode()
    dw = _gpu.DeviceWorkload(wl)
    S = pa.paged_attn_auto_split(dw.q, dw.k, dw.bt)
    assert S > 1   # 128 units at split 1 do not fill the GPU
    out, lse, nbytes = _single_call(pa, dw, 0)
    assert nbytes > 0
    rows = oracle.all_rows(wl.B, wl.Sq, wl.Hq)
    ref = oracle.workload_rows(wl, split_kv=S, row_bih=rows)
    _gpu.assert_close(_gpu.to_f64(out, wl.dtype).reshape(-1, wl.D), ref["comb_out"], wl.dtype, "auto split out")
    _gpu.assert_close(_gpu.to_f64(lse, "f32").ravel(), ref["comb_lse"], wl.dtype, "auto split lse")
    assert pa.paged_attn_last_error_word() == 0


def test_workspace_too_small_is_rejected(pa):
    import torch
    wl = W.ragged_decode()
    dw = _gpu.DeviceWorkload(wl)
    out = torch.empty_like(dw.q)
    need = pa.paged_attn_workspace_bytes(dw.q, dw.k, dw.bt, 4)
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PagedAttnError) as e:
        pa.paged_attn_fwd_splitkv(dw.q, dw.k, dw.v, dw.bt, dw.sl, False, None, 4, wl.scale, out, None, ws)
    assert e.value.code == -1


@pytest.mark.parametrize("S", [3, 8])
def test_single_call_equals_two_calls_prefill(pa, S):
    """The single call on the causal prefill (tcgen05 kernel, split partials in the workspace) gives
    the bits of paged_attn_fwd into caller partials followed by paged_attn_combine."""
    wl = W.causal_prefill()
    dw = _gpu.DeviceWorkload(wl)
    out, lse, _ = _single_call(pa, dw, S)
    ref = _gpu.run(dw, S)
    assert np.array_equal(_gpu.to_f64(out, wl.dtype), ref["out"])
    assert np.array_equal(_gpu.to_f64(lse, "f32"), ref["lse"])
    assert pa.paged_attn_last_error_word() == 0
