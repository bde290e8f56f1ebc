"""The entry point for callers that cannot allocate device memory at call time.

paged_attn_fwd_splitkv_noalloc keeps its split partials in a fixed array inside the library
instead of a caller workspace.  This file is collected last on purpose.  Its checks:
  - two calls in a row, with different inputs, both called through the C ABI;
  - each result matches the workspace entry point within the parity tolerance;
  - an oversized shape is rejected before anything is launched.
"""
import ctypes

import numpy as np
import pytest

from paged_kv_cache_201_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_201_gb300 as pa
    pa.load_library(build_if_missing=True)
    return pa


def _call_noalloc_cabi(pa, dw, split_kv):
    """Call the C entry point directly (ctypes), with the current stream."""
    import torch
    wl = dw.wl
    out = torch.empty_like(dw.q)
    lse = torch.empty((wl.B, wl.Sq, wl.Hq), dtype=torch.float32, device="cuda")
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    dims = pa.dims_of(dw.q, dw.k, dw.bt)
    qo = None if dw.qo is None else dw.qo.data_ptr()
    rc = pa.load_library().paged_attn_fwd_splitkv_noalloc(
        dw.q.data_ptr(), dw.k.data_ptr(), dw.v.data_ptr(), dw.bt.data_ptr(), dw.sl.data_ptr(), int(wl.causal), qo,
        split_kv, ctypes.c_float(wl.scale), out.data_ptr(), lse.data_ptr(), ctypes.byref(dims),
        props.multi_processor_count, props.total_memory, torch.cuda.current_stream().cuda_stream)
    return rc, out, lse


def _call_workspace(pa, dw, split_kv):
    import torch
    wl = dw.wl
    out = torch.empty_like(dw.q)
    lse = torch.empty((wl.B, wl.Sq, wl.Hq), dtype=torch.float32, device="cuda")
    nbytes = pa.paged_attn_workspace_bytes(dw.q, dw.k, dw.bt, split_kv)
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")
    pa.paged_attn_fwd_splitkv(dw.q, dw.k, dw.v, dw.bt, dw.sl, wl.causal, dw.qo, split_kv, wl.scale, out, lse, ws)
    return out, lse


def test_noalloc_matches_workspace_entry_two_calls(pa):
    import torch
    first = W.ragged_decode()
    second = W.make_custom(dtype="bf16", B=6, Sq=3, Hq=16, Hkv=4, D=128, page_size=16,
                           seq_lens=[3, 40, 129, 600, 17, 300], causal=True, seed=4242)
    for wl, S in ((first, 8), (second, 5)):
        dw = _gpu.DeviceWorkload(wl)
        rc, out, lse = _call_noalloc_cabi(pa, dw, S)
        assert rc == 0, pa.paged_attn_strerror(rc)
        ref_out, ref_lse = _call_workspace(pa, dw, S)
        torch.cuda.synchronize()
        _gpu.assert_close(_gpu.to_f64(out, wl.dtype), _gpu.to_f64(ref_out, wl.dtype), wl.dtype, f"{wl.name} out")
        _gpu.assert_close(_gpu.to_f64(lse, "f32"), _gpu.to_f64(ref_lse, "f32"), wl.dtype, f"{wl.name} lse")
    assert pa.paged_attn_last_error_word() == 0


def test_noalloc_rejects_partials_beyond_the_fixed_array(pa):
    wl = W.make_custom(dtype="bf16", B=64, Sq=1, Hq=64, Hkv=8, D=128, page_size=16, seq_lens=[40] * 64, seed=7)
    dw = _gpu.DeviceWorkload(wl)
    S = 40   # 40 splits x 4096 rows x 129 floats > 64 MiB
    assert pa.paged_attn_workspace_bytes(dw.q, dw.k, dw.bt, S) > pa.NOALLOC_SCRATCH_BYTES
    rc, _, _ = _call_noalloc_cabi(pa, dw, S)
    assert rc == -1
