"""The C-ABI library loads, exports every symbol the header declares, and its host-side
argument validation returns the documented status codes (CPU only; no kernel is launched)."""
import ctypes
import math
import os
import re
import subprocess

import numpy as np
import pytest

import paged_kv_cache_201_gb300 as pa
from paged_kv_cache_201_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "paged_attn.h")
OK, EINVAL, EDTYPE, EUNSUP = 0, -1, -2, -3
FAKE = 0x10000  # never dereferenced: every call below fails validation (or has no work) first


@pytest.fixture(scope="module")
def lib():
    build.build()
    return pa.load_library()


def declared_functions():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return sorted(set(re.findall(r"\b(paged_attn_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"paged_attn_fwd", "paged_attn_combine", "paged_attn_plan", "paged_attn_debug_gather",
            "paged_attn_last_error_word", "paged_attn_strerror"} <= set(names)
    nm = subprocess.run(["nm", "-D", "--defined-only", build.LIB_PATH], capture_output=True, text=True,
                        check=True).stdout
    exported = {line.split()[-1] for line in nm.splitlines() if line.strip()}
    missing = [n for n in names if n not in exported]
    assert not missing, f"declared but not exported (C linkage): {missing}"
    for n in names:
        assert hasattr(lib, n)


def test_strerror_and_version(lib):
    assert pa.paged_attn_strerror(0) == "ok"
    assert pa.paged_attn_strerror(-3).startswith("unsupported")
    assert pa.paged_attn_strerror(12345) == "unknown status"
    assert "page id" in pa.paged_attn_strerror(pa.PA_EBOUNDS)
    assert "timed out" in pa.paged_attn_strerror(pa.PA_ETIMEOUT)
    assert pa.paged_attn_version() >= 100


def _dims(**kw):
    base = dict(batch=2, q_len=1, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16, num_pages=64,
                bt_stride=8, dtype=pa.PA_BF16)
    base.update(kw)
    return pa.PaDims(**base)


def _fwd(lib, dims, split=1, scale=0.1, lse=FAKE, q=FAKE, out=FAKE, variant=0):
    return lib.paged_attn_fwd_variant(q, FAKE, FAKE, FAKE, FAKE, 0, None, split, scale, out, lse,
                                      None if dims is None else ctypes.byref(dims), variant, None)


@pytest.mark.parametrize("kw,split,scale,extra,code", [
    (None, 1, 0.1, {}, EINVAL),
    (dict(dtype=7), 1, 0.1, {}, EDTYPE),
    (dict(head_dim=96), 1, 0.1, {}, EUNSUP),
    (dict(page_size=8), 1, 0.1, {}, EUNSUP),
    (dict(num_q_heads=6, num_kv_heads=4), 1, 0.1, {}, EINVAL),
    (dict(num_pages=0), 1, 0.1, {}, EINVAL),
    (dict(num_pages=1 << 27), 1, 0.1, {}, EUNSUP),
    ({}, 0, 0.1, {}, EINVAL),
    ({}, 1, math.nan, {}, EINVAL),
    ({}, 2, 0.1, dict(lse=None), EINVAL),
    ({}, 1, 0.1, dict(q=FAKE + 2), EINVAL),
    ({}, 1, 0.1, dict(q=None), EINVAL),
    (dict(dtype=pa.PA_F32), 1, 0.1, dict(variant=2), EUNSUP),
    (dict(head_dim=256), 1, 0.1, dict(variant=2), EUNSUP),
    (dict(head_dim=256), 1, 0.1, dict(variant=3), EUNSUP),
    (dict(head_dim=128), 1, 0.1, dict(variant=5), EUNSUP),
    (dict(head_dim=256, dtype=pa.PA_F32), 1, 0.1, dict(variant=5), EUNSUP),
    (dict(q_len=2, num_q_heads=32), 1, 0.1, dict(variant=2), EUNSUP),
    ({}, 1, 0.1, dict(variant=9), EINVAL),
    (dict(q_len=128), 1, 0.0, dict(variant=4), EUNSUP),   # tcgen05 prefill takes scale > 0 only
    (dict(bt_stride=17), 2, 0.1, dict(variant=6), EUNSUP),   # split group: a split past 8 pages
    (dict(q_len=5), 4, 0.1, dict(variant=6), EUNSUP),        # split group: 20 rows > 16
    (dict(head_dim=256), 4, 0.1, dict(variant=6), EUNSUP),
    (dict(dtype=pa.PA_F32), 4, 0.1, dict(variant=6), EUNSUP),
    (dict(q_len=128), 1, -0.1, dict(variant=4), EUNSUP),
    (dict(q_stride=8 * 128 - 8), 1, 0.1, {}, EINVAL),          # q tokens overlapping their heads
    (dict(q_stride=12 * 128 + 4), 1, 0.1, {}, EINVAL),         # bf16 rows not 16-byte aligned
    (dict(q_stride=12 * 128 + 2, dtype=pa.PA_F32), 1, 0.1, {}, EINVAL),
    (dict(q_stride=1 << 40), 1, 0.1, {}, EINVAL),
    (dict(batch=0, q_stride=12 * 128), 1, 0.1, {}, OK),       # a fused QKV view's stride is accepted
    (dict(batch=0), 1, 0.1, {}, OK),
    (dict(q_len=0), 4, 0.1, dict(lse=None), OK),
    (dict(q_len=0), 4, 0.1, {}, OK),
])
def test_fwd_validation(lib, kw, split, scale, extra, code):
    dims = None if kw is None else _dims(**kw)
    assert _fwd(lib, dims, split, scale, **extra) == code


def test_combine_plan_gather_validation(lib):
    f = lib.paged_attn_combine
    assert f(FAKE, FAKE, 2, 10, 128, 9, FAKE, None, None) == EDTYPE
    assert f(FAKE, FAKE, 2, 10, 96, 0, FAKE, None, None) == EUNSUP
    assert f(FAKE, FAKE, 0, 10, 128, 0, FAKE, None, None) == EINVAL
    assert f(FAKE, FAKE, 2, 0, 128, 0, FAKE, None, None) == OK
    assert f(FAKE + 4, FAKE, 2, 10, 128, 0, FAKE, None, None) == EINVAL
    assert f(None, FAKE, 2, 10, 128, 0, FAKE, None, None) == EINVAL
    p = lib.paged_attn_plan
    assert p(FAKE, -1, 16, 2, FAKE, None) == EINVAL
    assert p(FAKE, 4, 0, 2, FAKE, None) == EINVAL
    assert p(FAKE, 0, 16, 2, FAKE, None) == OK
    g = lib.paged_attn_debug_gather
    d = _dims()
    assert g(FAKE, FAKE, FAKE, ctypes.byref(d), -1, FAKE, None) == EINVAL
    assert g(FAKE, FAKE, FAKE, ctypes.byref(d), 0, FAKE, None) == OK
    assert g(FAKE, FAKE, FAKE, ctypes.byref(_dims(head_dim=32)), 4, FAKE, None) == EUNSUP


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """The binding never falls back: without the built library every call raises."""
    monkeypatch.setattr(pa, "_lib", None)
    monkeypatch.setattr(pa, "library_path", lambda: str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="not built"):
        pa.load_library()


def test_auto_split_and_workspace_host_logic(lib):
    """Split choice: two waves of units over the SMs, capped by bt_stride, 256 and the workspace budget
    (device memory / 8 clamped to [1 GiB, 8 GiB], rocMLIR PR #2371 split-KV prefilter)."""
    auto, wsb = lib.paged_attn_auto_split, lib.paged_attn_workspace_bytes
    d = _dims(batch=256, q_len=1, num_q_heads=32, num_kv_heads=8, bt_stride=256)   # 2048 units already
    assert auto(ctypes.byref(d), 152, 280 << 30) == 1
    assert wsb(ctypes.byref(d), 0, 152, 280 << 30) == 0
    d = _dims(batch=32, q_len=1, num_q_heads=64, num_kv_heads=4, bt_stride=63)     # 128 units -> ceil(304/128)
    assert auto(ctypes.byref(d), 152, 280 << 30) == 3
    # 3 splits x 2048 rows: out 3*2048*128*4 = 3145728 B, lse 3*2048*4 = 24576 B (256-B multiples)
    assert wsb(ctypes.byref(d), 0, 152, 280 << 30) == 3145728 + 24576
    d = _dims(batch=1, q_len=1, num_q_heads=32, num_kv_heads=8, bt_stride=20)      # capped by bt_stride
    assert auto(ctypes.byref(d), 152, 280 << 30) == 20
    d = _dims(batch=1024, q_len=1, num_q_heads=64, num_kv_heads=8, bt_stride=4096)
    # per split 1024*64*129*4 = 33816576 B; 1 GiB budget -> 31 splits; 8 GiB -> the 245 of two waves stands
    assert auto(ctypes.byref(d), 1000000, 8 << 30) == 31
    assert auto(ctypes.byref(d), 1000000, 80 << 30) == 245
    assert auto(ctypes.byref(d), 0, 8 << 30) == EINVAL
    assert wsb(ctypes.byref(d), -1, 152, 8 << 30) == EINVAL
    assert wsb(ctypes.byref(d), 1, 152, 8 << 30) == 0


def _kvq(lib, dims, kv_dtype=pa.PA_FP8_E4M3, split=1, k_scale=FAKE, v_scale=FAKE, lse=FAKE, k=FAKE):
    return lib.paged_attn_fwd_kvq(FAKE, k, FAKE, k_scale, v_scale, kv_dtype, FAKE, FAKE, 0, None, split, 0.1, FAKE,
                                  lse, None if dims is None else ctypes.byref(dims), None)


def test_fwd_kvq_validation(lib):
    """8-bit-pool entry points: element types, scales and the shared checks, all before any launch."""
    assert _kvq(lib, None) == EINVAL
    assert _kvq(lib, _dims(dtype=pa.PA_F32)) == EDTYPE              # f32 queries are not read against 8-bit pools
    assert _kvq(lib, _dims(), kv_dtype=pa.PA_BF16) == EDTYPE       # pools must be E4M3 or int8
    assert _kvq(lib, _dims(), kv_dtype=5) == EDTYPE
    assert _kvq(lib, _dims(), kv_dtype=-1) == EDTYPE
    for kvd in (pa.PA_FP8_E4M3, pa.PA_INT8):                       # both formats pass the type check
        assert _kvq(lib, _dims(), kv_dtype=kvd, k_scale=None) == EINVAL
        assert _kvq(lib, _dims(batch=0), kv_dtype=kvd, k_scale=None) == OK
    assert _kvq(lib, _dims(head_dim=96)) == EUNSUP
    assert _kvq(lib, _dims(head_dim=256)) == EUNSUP
    assert _kvq(lib, _dims(), split=0) == EINVAL
    assert _kvq(lib, _dims(), k_scale=None) == EINVAL
    assert _kvq(lib, _dims(), v_scale=FAKE + 2) == EINVAL
    assert _kvq(lib, _dims(), k=FAKE + 8) == EINVAL                # pools 16-byte aligned
    assert _kvq(lib, _dims(), split=2, lse=None) == EINVAL
    assert _kvq(lib, _dims(batch=0), k_scale=None) == OK            # no rows: nothing to check further
    f = lib.paged_attn_fwd_kvq_splitkv
    d = _dims()
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, pa.PA_F16, FAKE, FAKE, 0, None, 2, 0.1, FAKE, FAKE, ctypes.byref(d),
             FAKE, 1 << 20, 152, 280 << 30, None) == EDTYPE
    # split 2 needs 2 * 16 rows * (128 + 1) * 4 bytes rounded up: a 16-byte workspace is too small
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, pa.PA_FP8_E4M3, FAKE, FAKE, 0, None, 2, 0.1, FAKE, FAKE, ctypes.byref(d),
             FAKE, 16, 152, 280 << 30, None) == EINVAL


def test_fwd_varlen_validation(lib):
    """Variable-length entry point: element type, q_start and the shared checks before any launch."""
    f = lib.paged_attn_fwd_varlen

    def call(dims, q_start=FAKE, split=1, lse=FAKE):
        return f(FAKE, FAKE, FAKE, FAKE, FAKE, q_start, 1, None, split, 0.1, FAKE, lse,
                 None if dims is None else ctypes.byref(dims), None)
    assert call(None) == EINVAL
    assert call(_dims(q_len=40, dtype=pa.PA_F32)) == EDTYPE
    assert call(_dims(q_len=40), q_start=None) == EINVAL
    assert call(_dims(q_len=40), q_start=FAKE + 2) == EINVAL
    assert call(_dims(q_len=40), split=0) == EINVAL
    assert call(_dims(q_len=40), split=2, lse=None) == EINVAL
    assert call(_dims(q_len=40, head_dim=96)) == EUNSUP
    assert call(_dims(q_len=0), q_start=None) == OK   # no query token: nothing to do
    assert call(_dims(q_len=40, head_dim=256)) == EUNSUP


def test_debug_wait_timeout_validation(lib):
    assert lib.paged_attn_debug_wait_timeout(0, None) == EINVAL
    assert lib.paged_attn_debug_wait_timeout(2_000_001, None) == EINVAL


def test_varlen_hint_counts(lib):
    """paged_attn_varlen_hint against a direct count on the host: pairs of the sequences with at least
    64 query rows (causal reach with and without offsets), K/V tokens of the others; malformed
    q_start entries count as no tokens."""
    rng = np.random.default_rng(3)
    for causal in (True, False):
        for with_offset in (True, False):
            for G in (1, 4, 8):
                q_lens = rng.choice([0, 1, 1, 2, 7, 16, 40, 100, 300], size=23)
                B = q_lens.size
                q_start = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
                seq_lens = (q_lens + rng.integers(0, 500, size=B)).astype(np.int32)
                q_offset = (rng.integers(-20, 400, size=B).astype(np.int32) if with_offset else None)
                h = pa.paged_attn_varlen_hint(q_start, seq_lens, q_offset, causal, 8 * G, 8)
                want_long = want_short = 0
                for b in range(B):
                    n, L = int(q_lens[b]), int(seq_lens[b])
                    if n == 0:
                        continue
                    if n * G < 64:
                        want_short += L
                        continue
                    qoff = int(q_offset[b]) if q_offset is not None else L - n
                    for i in range(n):
                        want_long += min(L, max(0, qoff + i + 1)) if causal else L
                assert (h.long_pairs, h.short_kv_tokens) == (want_long, want_short)
    # T = q_start[B] = 300: a decreasing pair and entries past T count as no tokens
    qs = np.array([0, 100, 50, 20_000, 300], dtype=np.int32)
    h = pa.paged_attn_varlen_hint(qs, np.array([300, 300, 300, 300], dtype=np.int32), None, True, 32, 8)
    assert h.long_pairs == sum(range(201, 301)) and h.short_kv_tokens == 0


def test_varlen_overlap_share(lib):
    """The SM share of the overlapped call: 0 without work of both kinds or with fewer than 16 SMs,
    the balancing estimate x 1.3 otherwise (57 of 152 SMs for the benchmark's mixed batch, where a
    sweep measured 1.2-1.5 x the balancing share as fastest), clamped to [8, 3/4 of the SMs],
    non-decreasing in the long sequences' work, smaller for f16 (its higher tensor rate)."""
    share = pa.paged_attn_varlen_overlap_share
    H = pa.PaVarlenHint
    assert share(None, 152, 32, 8) == 0
    assert share(H(0, 0), 152, 32, 8) == 0
    assert share(H(10 ** 9, 0), 152, 32, 8) == 0 and share(H(0, 10 ** 9), 152, 32, 8) == 0
    assert share(H(7318528, 1048576), 15, 32, 8) == 0
    assert share(H(7318528, 1048576), 152, 32, 8) == 57
    flops, t_short = 4.0 * 128 * 32 * 7318528, 2.0 * 1048576 * 8 * 128 * 2 / 6.9e12
    assert share(H(7318528, 1048576), 152, 32, 8) == math.ceil(1.3 * flops / (4.4e12 * t_short))
    assert share(H(1, 10 ** 9), 152, 32, 8) == 8
    assert share(H(10 ** 12, 1), 152, 32, 8) == 114
    last = 0
    for lp in (10 ** 5, 10 ** 6, 3 * 10 ** 6, 10 ** 7, 3 * 10 ** 7, 10 ** 8):
        n = share(H(lp, 1048576), 152, 32, 8)
        assert 8 <= n <= 114 and n >= last
        last = n
    assert share(H(7318528, 1048576), 152, 32, 8, 128, pa.PA_F16) < 57
    with pytest.raises(pa.PagedAttnError):
        share(H(1, 1), 0, 32, 8)


def test_varlen_hint_binding_checks(lib):
    """The binding refuses arrays of the wrong lengths; an empty batch gives a zero hint."""
    with pytest.raises(ValueError):
        pa.paged_attn_varlen_hint(np.array([0, 3], dtype=np.int32), np.array([5, 6], dtype=np.int32), None, True,
                                  8, 2)
    with pytest.raises(ValueError):
        pa.paged_attn_varlen_hint(np.array([0, 3], dtype=np.int32), np.array([5], dtype=np.int32),
                                  np.array([1, 2], dtype=np.int32), True, 8, 2)
    h = pa.paged_attn_varlen_hint(np.array([0], dtype=np.int32), np.zeros(0, dtype=np.int32), None, True, 8, 2)
    assert (h.long_pairs, h.short_kv_tokens) == (0, 0)
    assert lib.paged_attn_varlen_hint(None, None, None, 1, None, None) == EINVAL


def test_q_token_stride_of_views():
    """The binding reads q's token stride from a view's strides (no GPU needed: strides only)."""
    import torch
    B, Sq, Hq, Hkv, D = 3, 5, 8, 2, 64
    fused = torch.empty(B, Sq, Hq + 2 * Hkv, D, dtype=torch.bfloat16)
    assert pa._q_token_stride(fused[:, :, :Hq]) == (Hq + 2 * Hkv) * D
    assert pa._q_token_stride(torch.empty(B, Sq, Hq, D)) == 0              # dense
    assert pa._q_token_stride(fused[:, :1, :Hq]) == Sq * (Hq + 2 * Hkv) * D  # one token per sequence
    packed = torch.empty(7, Hq + 2 * Hkv, D, dtype=torch.float16)
    assert pa._q_token_stride(packed[:, :Hq]) == (Hq + 2 * Hkv) * D
    with pytest.raises(ValueError):                                          # heads not dense
        pa._q_token_stride(fused[:, :, ::2])
    with pytest.raises(ValueError):                                          # tokens unevenly spaced
        pa._q_token_stride(fused[:, ::2, :Hq])
