"""The entry point for callers that cannot allocate device memory at call time.

paged_attn_fwd_splitkv_noalloc keeps its split partials in a fixed array inside the library
instead of a caller workspace.  This file is collected last on purpose, and its first test must
make the process's first call of the entry point.  Its checks, every call through the C ABI:
  - the array is claimed on the device by the first call (lazy module loading), not before;
  - two calls in a row, with different inputs, give bit for bit what the workspace entry point
    gives with the same split (both run the same kernels), and match the oracle on every row;
  - split_kv = 1 (no partials) and split_kv = 0 (the automatic split) work the same way;
  - an automatic split whose partials would overflow the array is lowered until they fit;
  - an explicit split that overflows it is rejected before anything is launched.
"""
import ctypes
import os

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


def _outputs(dw):
    import torch
    wl = dw.wl
    return torch.empty_like(dw.q), torch.empty((wl.B, wl.Sq, wl.Hq), dtype=torch.float32, device="cuda")


def _call_noalloc_cabi(pa, dw, split_kv, out, lse, num_sms=None):
    """Call the C entry point directly (ctypes), with the current stream."""
    import torch
    wl = dw.wl
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    dims = pa.dims_of(dw.q, dw.k, dw.bt)
    qo = None if dw.qo is None else dw.qo.data_ptr()
    return pa.load_library().paged_attn_fwd_splitkv_noalloc(
        dw.q.data_ptr(), dw.k.data_ptr(), dw.v.data_ptr(), dw.bt.data_ptr(), dw.sl.data_ptr(), int(wl.causal), qo,
        split_kv, ctypes.c_float(wl.scale), out.data_ptr(), lse.data_ptr(), ctypes.byref(dims),
        props.multi_processor_count if num_sms is None else num_sms, props.total_memory,
        torch.cuda.current_stream().cuda_stream)


def _call_workspace(pa, dw, split_kv):
    import torch
    wl = dw.wl
    out, lse = _outputs(dw)
    nbytes = pa.paged_attn_workspace_bytes(dw.q, dw.k, dw.bt, split_kv)
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")
    pa.paged_attn_fwd_splitkv(dw.q, dw.k, dw.v, dw.bt, dw.sl, wl.causal, dw.qo, split_kv, wl.scale, out, lse, ws)
    return out, lse


def _bits_equal(a, b):
    import torch
    return torch.equal(a.view(torch.int16) if a.element_size() == 2 else a.view(torch.int32),
                       b.view(torch.int16) if b.element_size() == 2 else b.view(torch.int32))


def _check_oracle(dw, out, lse, split_kv, what):
    wl = dw.wl
    rows = oracle.all_rows(wl.B, wl.Sq, wl.Hq)
    ref = oracle.workload_rows(wl, split_kv=split_kv, row_bih=rows)
    want_out, want_lse = (ref["out"], ref["lse"]) if split_kv == 1 else (ref["comb_out"], ref["comb_lse"])
    _gpu.assert_close(_gpu.to_f64(out, wl.dtype).reshape(-1, wl.D), want_out, wl.dtype, f"{what} out")
    _gpu.assert_close(_gpu.to_f64(lse, "f32").ravel(), want_lse, wl.dtype, f"{what} lse")


def test_noalloc_first_call_claims_the_array(pa):
    """Under lazy module loading (CUDA's default, and what torch sets when the variable is unset) the
    array's device memory is claimed by the first call on the device, as the header states."""
    import torch
    if os.environ.get("CUDA_MODULE_LOADING", "LAZY").upper() != "LAZY":
        pytest.skip("eager module loading claims the array when the library is first used")
    wl = W.ragged_decode()
    dw = _gpu.DeviceWorkload(wl)
    out, lse = _outputs(dw)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    assert _call_noalloc_cabi(pa, dw, 8, out, lse) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free0 - free1 >= pa.NOALLOC_SCRATCH_BYTES, (free0, free1)
    # later calls claim nothing more
    assert _call_noalloc_cabi(pa, dw, 8, out, lse) == 0
    torch.cuda.synchronize()
    free2, _ = torch.cuda.mem_get_info()
    assert free2 == free1
    _check_oracle(dw, out, lse, 8, "first call")


def test_noalloc_matches_workspace_entry_two_calls(pa):
    """Two calls in a row on different inputs: each bit-identical to the workspace entry point at the
    same split, and every row within tolerance of the oracle."""
    import torch
    first = W.ragged_decode()
    second = W.make_custom(dtype="bf16", B=6, Sq=3, Hq=16, Hkv=4, D=128, page_size=16,
                           seq_lens=[3, 40, 129, 600, 17, 300], causal=True, seed=4242)
    for wl, S in ((first, 8), (second, 5)):
        dw = _gpu.DeviceWorkload(wl)
        out, lse = _outputs(dw)
        rc = _call_noalloc_cabi(pa, dw, S, out, lse)
        assert rc == 0, pa.paged_attn_strerror(rc)
        ref_out, ref_lse = _call_workspace(pa, dw, S)
        torch.cuda.synchronize()
        assert _bits_equal(out, ref_out), f"{wl.name}: out differs from the workspace entry point"
        assert _bits_equal(lse, ref_lse), f"{wl.name}: lse differs from the workspace entry point"
        _check_oracle(dw, out, lse, S, f"{wl.name} S={S}")
    assert pa.paged_attn_last_error_word() == 0


@pytest.mark.parametrize("split_kv", [1, 0])
def test_noalloc_split_one_and_automatic(pa, split_kv):
    """split_kv = 1 writes the outputs directly (no partials); split_kv = 0 takes the automatic split,
    which fits the array on this shape unchanged.  Both bit-identical to the workspace entry point."""
    import torch
    wl = W.ragged_decode()
    dw = _gpu.DeviceWorkload(wl)
    S = split_kv or pa.paged_attn_auto_split(dw.q, dw.k, dw.bt)
    assert pa.paged_attn_workspace_bytes(dw.q, dw.k, dw.bt, S) <= pa.NOALLOC_SCRATCH_BYTES
    out, lse = _outputs(dw)
    assert _call_noalloc_cabi(pa, dw, split_kv, out, lse) == 0
    ref_out, ref_lse = _call_workspace(pa, dw, S)
    torch.cuda.synchronize()
    assert _bits_equal(out, ref_out) and _bits_equal(lse, ref_lse)
    _check_oracle(dw, out, lse, S, f"split_kv={split_kv} (S={S})")


def test_noalloc_automatic_split_is_lowered_to_fit(pa):
    """With split_kv = 0 and a GPU reported with 1024 SMs, the automatic split of this prefill shape
    (64 tiles of 128 rows) would be 32, whose partials (135 MB) overflow the array: the call lowers it
    to the largest split that fits (15) instead of failing."""
    import torch
    wl = W.make_custom(dtype="bf16", B=4, Sq=64, Hq=32, Hkv=2, D=128, page_size=16, seq_lens=[600, 500, 610, 90],
                       causal=True, W=40, seed=4343)
    dw = _gpu.DeviceWorkload(wl)
    big = 1024
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    S_auto = pa.paged_attn_auto_split(dw.q, dw.k, dw.bt, num_sms=big, device_bytes=props.total_memory)
    assert pa.paged_attn_workspace_bytes(dw.q, dw.k, dw.bt, S_auto) > pa.NOALLOC_SCRATCH_BYTES
    S = S_auto
    while S > 1 and pa.paged_attn_workspace_bytes(dw.q, dw.k, dw.bt, S) > pa.NOALLOC_SCRATCH_BYTES:
        S -= 1
    assert 1 < S < S_auto
    out, lse = _outputs(dw)
    rc = _call_noalloc_cabi(pa, dw, 0, out, lse, num_sms=big)
    assert rc == 0, pa.paged_attn_strerror(rc)
    ref_out, ref_lse = _call_workspace(pa, dw, S)
    torch.cuda.synchronize()
    assert _bits_equal(out, ref_out) and _bits_equal(lse, ref_lse)
    _check_oracle(dw, out, lse, S, f"lowered automatic split S={S}")
    assert pa.paged_attn_last_error_word() == 0


def test_noalloc_rejects_partials_beyond_the_fixed_array(pa):
    wl = W.make_custom(dtype="bf16", B=64, Sq=1, Hq=64, Hkv=8, D=128, page_size=16, seq_lens=[40] * 64, seed=7)
    dw = _gpu.DeviceWorkload(wl)
    S = 40   # 40 splits x 4096 rows x 129 floats > 64 MiB
    assert pa.paged_attn_workspace_bytes(dw.q, dw.k, dw.bt, S) > pa.NOALLOC_SCRATCH_BYTES
    out, lse = _outputs(dw)
    assert _call_noalloc_cabi(pa, dw, S, out, lse) == -1
