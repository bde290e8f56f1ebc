"""Paged attention over a paged K/V cache on GB300 (sm_103a).

Thin Python binding of the C ABI in ``include/paged_attn.h``: it checks that the
tensors are CUDA, dense and of the right type, marshals their pointers and the
current stream, and calls the library.  Every step of the computation runs in
the library's CUDA kernels; there is no CPU or PyTorch fallback, and a missing
library is an error.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

from . import build as _build

__all__ = [
    "PagedAttnError", "load_library", "library_path", "paged_attn_fwd", "paged_attn_fwd_variant",
    "paged_attn_combine", "paged_attn_plan", "paged_attn_debug_gather", "paged_attn_last_error_word",
    "paged_attn_last_error_status",
    "paged_attn_strerror", "paged_attn_version", "attention", "paged_attn_auto_split",
    "paged_attn_workspace_bytes", "paged_attn_fwd_splitkv", "paged_attn_fwd_splitkv_noalloc", "paged_attn_fwd_kvq",
    "paged_attn_fwd_kvq_splitkv", "attention_kvq", "paged_attn_fwd_varlen", "attention_varlen",
    "paged_attn_fwd_varlen_overlap", "paged_attn_varlen_hint", "paged_attn_varlen_overlap_share", "PaVarlenHint", "PA_F32", "PA_F16", "PA_BF16", "PA_FP8_E4M3",
    "PA_INT8",
    "VARIANT_AUTO", "VARIANT_SIMT", "VARIANT_MMA_DECODE", "VARIANT_MMA_PREFILL", "VARIANT_TC05_PREFILL",
    "VARIANT_MMA_T", "VARIANT_MMA_SPLIT_GROUP",
]

PA_F32, PA_F16, PA_BF16, PA_FP8_E4M3, PA_INT8 = 0, 1, 2, 3, 4
VARIANT_AUTO, VARIANT_SIMT, VARIANT_MMA_DECODE, VARIANT_MMA_PREFILL, VARIANT_TC05_PREFILL, VARIANT_MMA_T = 0, 1, 2, 3, 4, 5
VARIANT_MMA_SPLIT_GROUP = 6
ERRBIT_PAGE_RANGE, ERRBIT_TIMEOUT, ERRBIT_SEQ_CLIPPED, ERRBIT_QSTART = 1, 2, 4, 8
PA_OK, PA_EINVAL, PA_EDTYPE, PA_EUNSUPPORTED, PA_ECUDA, PA_EBOUNDS, PA_ETIMEOUT = 0, -1, -2, -3, -4, -5, -6


class PaDims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("q_len", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_pages", ctypes.c_int64), ("bt_stride", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("q_stride", ctypes.c_int64)]


class PaVarlenHint(ctypes.Structure):
    """pa_varlen_hint: a variable-length batch's work split (``paged_attn_varlen_hint``)."""
    _fields_ = [("long_pairs", ctypes.c_int64), ("short_kv_tokens", ctypes.c_int64)]


class PagedAttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = f"{where}: status {code} ({paged_attn_strerror(code)})"
        if code == -4:
            msg += f": {load_library().paged_attn_cuda_error_string().decode()}"
        super().__init__(msg)


_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load_library(build_if_missing: bool = False):
    """Load the CUDA library (``_build/libpaged_attn_gb300.so``); raise if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"paged-attention CUDA library not built ({path}); run "
                               "paged_kv_cache_201_gb300.build.build()")
        _build.build()
    lib = ctypes.CDLL(path)
    P, I32, I64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    D = ctypes.POINTER(PaDims)
    lib.paged_attn_fwd.argtypes = [P, P, P, P, P, I32, P, I32, F, P, P, D, P]
    lib.paged_attn_fwd_variant.argtypes = [P, P, P, P, P, I32, P, I32, F, P, P, D, I32, P]
    lib.paged_attn_combine.argtypes = [P, P, I32, I64, I32, I32, P, P, P]
    lib.paged_attn_plan.argtypes = [P, I32, I32, I32, P, P]
    lib.paged_attn_auto_split.argtypes = [D, I32, I64]
    lib.paged_attn_auto_split.restype = ctypes.c_int
    lib.paged_attn_workspace_bytes.argtypes = [D, I32, I32, I64]
    lib.paged_attn_workspace_bytes.restype = ctypes.c_int64
    lib.paged_attn_fwd_splitkv.argtypes = [P, P, P, P, P, I32, P, I32, F, P, P, D, P, I64, I32, I64, P]
    lib.paged_attn_fwd_splitkv.restype = ctypes.c_int
    lib.paged_attn_fwd_splitkv_noalloc.argtypes = [P, P, P, P, P, I32, P, I32, F, P, P, D, I32, I64, P]
    lib.paged_attn_fwd_splitkv_noalloc.restype = ctypes.c_int
    lib.paged_attn_fwd_kvq.argtypes = [P, P, P, P, P, I32, P, P, I32, P, I32, F, P, P, D, P]
    lib.paged_attn_fwd_kvq.restype = ctypes.c_int
    lib.paged_attn_fwd_kvq_splitkv.argtypes = [P, P, P, P, P, I32, P, P, I32, P, I32, F, P, P, D, P, I64, I32, I64, P]
    lib.paged_attn_fwd_kvq_splitkv.restype = ctypes.c_int
    lib.paged_attn_fwd_varlen.argtypes = [P, P, P, P, P, P, I32, P, I32, F, P, P, D, P]
    lib.paged_attn_fwd_varlen.restype = ctypes.c_int
    lib.paged_attn_fwd_varlen_overlap.argtypes = [P, P, P, P, P, P, I32, P, I32, F, P, P, D,
                                                  ctypes.POINTER(PaVarlenHint), P]
    lib.paged_attn_fwd_varlen_overlap.restype = ctypes.c_int
    lib.paged_attn_varlen_hint.argtypes = [P, P, P, I32, D, ctypes.POINTER(PaVarlenHint)]
    lib.paged_attn_varlen_hint.restype = ctypes.c_int
    lib.paged_attn_varlen_overlap_share.argtypes = [D, ctypes.POINTER(PaVarlenHint), I32]
    lib.paged_attn_varlen_overlap_share.restype = ctypes.c_int
    lib.paged_attn_debug_gather.argtypes = [P, P, P, D, I32, P, P]
    lib.paged_attn_debug_wait_timeout.argtypes = [ctypes.c_uint32, P]
    lib.paged_attn_debug_wait_timeout.restype = ctypes.c_int
    lib.paged_attn_last_error_word.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    lib.paged_attn_strerror.argtypes = [I32]
    lib.paged_attn_strerror.restype = ctypes.c_char_p
    lib.paged_attn_version.argtypes = []
    lib.paged_attn_cuda_error_string.argtypes = []
    lib.paged_attn_cuda_error_string.restype = ctypes.c_char_p
    for name in ("paged_attn_fwd", "paged_attn_fwd_variant", "paged_attn_combine", "paged_attn_plan",
                 "paged_attn_debug_gather", "paged_attn_last_error_word", "paged_attn_version"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


# ----------------------------------------------------------------------------- marshalling helpers
def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    m = {torch.float32: PA_F32, torch.float16: PA_F16, torch.bfloat16: PA_BF16}
    if t.dtype not in m:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return m[t.dtype]


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check(t, name, dtype=None, ndim=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")


def _check_q(q, ndim):
    """q may be a view whose query tokens are further apart than its heads (for example sliced out of
    a fused QKV projection): its heads dense, tokens evenly spaced.  Other tensors must be
    contiguous."""
    if not q.is_cuda:
        raise ValueError("q must be a CUDA tensor")
    if q.dim() != ndim:
        raise ValueError(f"q must have {ndim} dims, got {q.dim()}")
    _q_token_stride(q)


def _q_token_stride(q) -> int:
    """Elements between consecutive query tokens of q ([B, Sq, Hq, D] or packed [T, Hq, D]); 0 when q
    is contiguous (the dense layout).  Raises if the tokens are not evenly spaced or the heads not dense."""
    if q.is_contiguous():
        return 0
    Hq, D = q.shape[-2], q.shape[-1]
    if (q.stride(-1) != 1 and D > 1) or (q.stride(-2) != D and Hq > 1):
        raise ValueError("q's heads must be dense ([..., Hq, D] contiguous)")
    if q.dim() == 3:
        return int(q.stride(0))
    B, Sq = q.shape[0], q.shape[1]
    tok = int(q.stride(1)) if Sq > 1 else int(q.stride(0))
    if B > 1 and Sq > 1 and q.stride(0) != Sq * q.stride(1):
        raise ValueError("q's tokens must be evenly spaced across sequences (stride(0) == Sq * stride(1))")
    return tok


def _stream(stream) -> int:
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def dims_of(q, k_cache, block_table) -> PaDims:
    B, Sq, Hq, D = q.shape
    P, ps, Hkv, D2 = k_cache.shape
    if D2 != D:
        raise ValueError("q and k_cache head dims differ")
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [B, W]")
    return PaDims(B, Sq, Hq, Hkv, D, ps, P, block_table.shape[1], _dtype_code(q), _q_token_stride(q))


def _raise(rc: int, where: str):
    if rc != 0:
        raise PagedAttnError(rc, where)


# ----------------------------------------------------------------------------- C ABI wrappers
def paged_attn_fwd_variant(q, k_cache, v_cache, block_table, seq_lens, causal, q_offset, split_kv, scale, out,
                           lse, variant: int = VARIANT_AUTO, stream=None) -> None:
    """Forward over the paged cache; see ``paged_attn_fwd`` in include/paged_attn.h."""
    torch = _torch()
    _check_q(q, 4)
    _check(k_cache, "k_cache", q.dtype, 4)
    _check(v_cache, "v_cache", q.dtype, 4)
    _check(block_table, "block_table", torch.int32, 2)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    _check(q_offset, "q_offset", torch.int32, 1)
    _check(out, "out")
    _check(lse, "lse", torch.float32)
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    dims = dims_of(q, k_cache, block_table)
    rc = load_library().paged_attn_fwd_variant(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens), int(bool(causal)),
        _ptr(q_offset), int(split_kv), float(scale), _ptr(out), _ptr(lse), ctypes.byref(dims), int(variant),
        _stream(stream))
    _raise(rc, "paged_attn_fwd")


def paged_attn_fwd(q, k_cache, v_cache, block_table, seq_lens, causal, q_offset, split_kv, scale, out, lse,
                   stream=None) -> None:
    paged_attn_fwd_variant(q, k_cache, v_cache, block_table, seq_lens, causal, q_offset, split_kv, scale, out, lse,
                           VARIANT_AUTO, stream)


def _device_info(device=None):
    torch = _torch()
    props = torch.cuda.get_device_properties(torch.cuda.current_device() if device is None else device)
    return int(props.multi_processor_count), int(props.total_memory)


def paged_attn_auto_split(q, k_cache, block_table, num_sms=None, device_bytes=None) -> int:
    """Split count the single-call forward picks for this shape (rocMLIR PR #2371 workspace budget)."""
    dims = dims_of(q, k_cache, block_table)
    if num_sms is None or device_bytes is None:
        n, m = _device_info(q.device)
        num_sms = n if num_sms is None else num_sms
        device_bytes = m if device_bytes is None else device_bytes
    rc = load_library().paged_attn_auto_split(ctypes.byref(dims), int(num_sms), int(device_bytes))
    if rc < 0:
        _raise(rc, "paged_attn_auto_split")
    return rc


def paged_attn_workspace_bytes(q, k_cache, block_table, split_kv: int = 0, num_sms=None, device_bytes=None) -> int:
    dims = dims_of(q, k_cache, block_table)
    if num_sms is None or device_bytes is None:
        n, m = _device_info(q.device)
        num_sms = n if num_sms is None else num_sms
        device_bytes = m if device_bytes is None else device_bytes
    v = load_library().paged_attn_workspace_bytes(ctypes.byref(dims), int(split_kv), int(num_sms), int(device_bytes))
    if v < 0:
        _raise(int(v), "paged_attn_workspace_bytes")
    return int(v)


def paged_attn_fwd_splitkv(q, k_cache, v_cache, block_table, seq_lens, causal, q_offset, split_kv, scale, out, lse,
                           workspace, num_sms=None, device_bytes=None, stream=None) -> None:
    """Split forward + combine in one call; ``workspace`` is a uint8 CUDA tensor (may be None when S == 1)."""
    torch = _torch()
    _check_q(q, 4)
    _check(k_cache, "k_cache", q.dtype, 4)
    _check(v_cache, "v_cache", q.dtype, 4)
    _check(block_table, "block_table", torch.int32, 2)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    _check(q_offset, "q_offset", torch.int32, 1)
    _check(out, "out", q.dtype)
    _check(lse, "lse", torch.float32)
    _check(workspace, "workspace")
    dims = dims_of(q, k_cache, block_table)
    if num_sms is None or device_bytes is None:
        n, m = _device_info(q.device)
        num_sms = n if num_sms is None else num_sms
        device_bytes = m if device_bytes is None else device_bytes
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load_library().paged_attn_fwd_splitkv(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens), int(bool(causal)), _ptr(q_offset),
        int(split_kv), float(scale), _ptr(out), _ptr(lse), ctypes.byref(dims), _ptr(workspace), int(ws_bytes),
        int(num_sms), int(device_bytes), _stream(stream))
    _raise(rc, "paged_attn_fwd_splitkv")


NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


def paged_attn_fwd_splitkv_noalloc(q, k_cache, v_cache, block_table, seq_lens, causal, q_offset, split_kv, scale,
                                   out, lse, num_sms=None, device_bytes=None, stream=None) -> None:
    """``paged_attn_fwd_splitkv`` without a workspace argument, for callers that cannot allocate device
    memory when they run attention: the split partials use a fixed NOALLOC_SCRATCH_BYTES array inside
    the library.  Calls that may overlap on the GPU share that array and must be serialised; the first
    call on a device should come before any stream capture there."""
    torch = _torch()
    _check_q(q, 4)
    _check(k_cache, "k_cache", q.dtype, 4)
    _check(v_cache, "v_cache", q.dtype, 4)
    _check(block_table, "block_table", torch.int32, 2)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    _check(q_offset, "q_offset", torch.int32, 1)
    _check(out, "out", q.dtype)
    _check(lse, "lse", torch.float32)
    dims = dims_of(q, k_cache, block_table)
    if num_sms is None or device_bytes is None:
        n, m = _device_info(q.device)
        num_sms = n if num_sms is None else num_sms
        device_bytes = m if device_bytes is None else device_bytes
    rc = load_library().paged_attn_fwd_splitkv_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens), int(bool(causal)), _ptr(q_offset),
        int(split_kv), float(scale), _ptr(out), _ptr(lse), ctypes.byref(dims), int(num_sms), int(device_bytes),
        _stream(stream))
    _raise(rc, "paged_attn_fwd_splitkv_noalloc")


def _check_q8_pool(t, name, kv_dtype):
    """An 8-bit pool [P, ps, Hkv, D]: uint8 bits of either format, torch.float8_e4m3fn for
    PA_FP8_E4M3 or torch.int8 for PA_INT8."""
    torch = _torch()
    _check(t, name, ndim=4)
    typed = {PA_FP8_E4M3: getattr(torch, "float8_e4m3fn", torch.uint8), PA_INT8: torch.int8}
    if kv_dtype not in typed:
        raise ValueError(f"kv_dtype must be PA_FP8_E4M3 or PA_INT8, got {kv_dtype}")
    if t.dtype not in (torch.uint8, typed[kv_dtype]):
        raise TypeError(f"{name} must be uint8 bits or {typed[kv_dtype]} for kv_dtype {kv_dtype}, got {t.dtype}")


def _kv_dtype_of(k_cache, kv_dtype):
    """kv_dtype as given, else PA_INT8 for an int8 pool and PA_FP8_E4M3 otherwise."""
    if kv_dtype is not None:
        return int(kv_dtype)
    return PA_INT8 if k_cache.dtype == _torch().int8 else PA_FP8_E4M3


def _kvq_args(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, q_offset, out, lse, kv_dtype):
    torch = _torch()
    _check_q(q, 4)
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError(f"q must be bf16 or f16 with 8-bit pools, got {q.dtype}")
    _check_q8_pool(k_cache, "k_cache", kv_dtype)
    _check_q8_pool(v_cache, "v_cache", kv_dtype)
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    P, _, Hkv, _ = k_cache.shape
    for t, name in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        _check(t, name, torch.float32, 2)
        if tuple(t.shape) != (P, Hkv):
            raise ValueError(f"{name} must be [num_pages, num_kv_heads] = {(P, Hkv)}, got {tuple(t.shape)}")
    _check(block_table, "block_table", torch.int32, 2)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    _check(q_offset, "q_offset", torch.int32, 1)
    _check(out, "out")
    _check(lse, "lse", torch.float32)
    return dims_of(q, k_cache, block_table)


def paged_attn_fwd_kvq(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, causal, q_offset, split_kv,
                       scale, out, lse, stream=None, kv_dtype=None) -> None:
    """Forward over 8-bit pools (``kv_dtype`` PA_FP8_E4M3 or PA_INT8; by default PA_INT8 for int8
    tensors, else PA_FP8_E4M3) with [num_pages, Hkv] float32 scales; see ``paged_attn_fwd_kvq`` in
    include/paged_attn.h.  Outputs as ``paged_attn_fwd``."""
    kv_dtype = _kv_dtype_of(k_cache, kv_dtype)
    dims = _kvq_args(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, q_offset, out, lse, kv_dtype)
    rc = load_library().paged_attn_fwd_kvq(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), kv_dtype, _ptr(block_table),
        _ptr(seq_lens), int(bool(causal)), _ptr(q_offset), int(split_kv), float(scale), _ptr(out), _ptr(lse),
        ctypes.byref(dims), _stream(stream))
    _raise(rc, "paged_attn_fwd_kvq")


def paged_attn_fwd_kvq_splitkv(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, causal, q_offset,
                               split_kv, scale, out, lse, workspace, num_sms=None, device_bytes=None,
                               stream=None, kv_dtype=None) -> None:
    """``paged_attn_fwd_splitkv`` over 8-bit pools (split forward + combine in one call); ``kv_dtype``
    as in ``paged_attn_fwd_kvq``."""
    kv_dtype = _kv_dtype_of(k_cache, kv_dtype)
    dims = _kvq_args(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, q_offset, out, lse, kv_dtype)
    _check(workspace, "workspace")
    if num_sms is None or device_bytes is None:
        n, m = _device_info(q.device)
        num_sms = n if num_sms is None else num_sms
        device_bytes = m if device_bytes is None else device_bytes
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load_library().paged_attn_fwd_kvq_splitkv(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), kv_dtype, _ptr(block_table),
        _ptr(seq_lens), int(bool(causal)), _ptr(q_offset), int(split_kv), float(scale), _ptr(out), _ptr(lse),
        ctypes.byref(dims), _ptr(workspace), int(ws_bytes), int(num_sms), int(device_bytes), _stream(stream))
    _raise(rc, "paged_attn_fwd_kvq_splitkv")


def paged_attn_varlen_hint(q_start, seq_lens, q_offset, causal, num_q_heads, num_kv_heads,
                           head_dim=128, dtype=PA_BF16) -> "PaVarlenHint":
    """The work split of a variable-length batch from HOST arrays (numpy or CPU tensors): q_start
    [B + 1], seq_lens [B], q_offset [B] or None; see ``paged_attn_varlen_hint`` in
    include/paged_attn.h."""
    qs = np.ascontiguousarray(np.asarray(q_start), dtype=np.int32)
    sl = np.ascontiguousarray(np.asarray(seq_lens), dtype=np.int32)
    qo = None if q_offset is None else np.ascontiguousarray(np.asarray(q_offset), dtype=np.int32)
    B = sl.shape[0]
    if qs.shape[0] != B + 1 or (qo is not None and qo.shape[0] != B):
        raise ValueError("q_start must hold B + 1 entries and q_offset B")
    T = int(qs[-1]) if B else 0
    dims = PaDims(B, max(T, 0), int(num_q_heads), int(num_kv_heads), int(head_dim), 16, 1, 1, int(dtype))
    hint = PaVarlenHint()
    rc = load_library().paged_attn_varlen_hint(qs.ctypes.data, sl.ctypes.data,
                                               None if qo is None else qo.ctypes.data, int(bool(causal)),
                                               ctypes.byref(dims), ctypes.byref(hint))
    _raise(rc, "paged_attn_varlen_hint")
    return hint


def paged_attn_varlen_overlap_share(hint, num_sms, num_q_heads, num_kv_heads, head_dim=128, dtype=PA_BF16) -> int:
    """SMs the overlapped call gives the tcgen05 kernel for ``hint`` (0: the kernels run one after
    the other); see ``paged_attn_varlen_overlap_share`` in include/paged_attn.h."""
    dims = PaDims(1, 1, int(num_q_heads), int(num_kv_heads), int(head_dim), 16, 1, 1, int(dtype))
    rc = load_library().paged_attn_varlen_overlap_share(ctypes.byref(dims),
                                                        None if hint is None else ctypes.byref(hint), int(num_sms))
    if rc < 0:
        _raise(rc, "paged_attn_varlen_overlap_share")
    return rc


def paged_attn_fwd_varlen(q, k_cache, v_cache, block_table, seq_lens, q_start, causal, q_offset, split_kv, scale,
                          out, lse, stream=None, hint=None) -> None:
    """Forward over a batch with a different query count per sequence; see ``paged_attn_fwd_varlen``
    in include/paged_attn.h.  q [T, Hq, D] packed, q_start int32 [B + 1]; out [T, Hq, D] (S = 1) or
    float32 [S, T, Hq, D]; lse [T, Hq] or [S, T, Hq].  With ``hint`` (a ``PaVarlenHint``, see
    ``paged_attn_varlen_hint``) the call is ``paged_attn_fwd_varlen_overlap``: the same results, its
    two kernels side by side."""
    torch = _torch()
    _check_q(q, 3)
    _check(k_cache, "k_cache", q.dtype, 4)
    _check(v_cache, "v_cache", q.dtype, 4)
    _check(block_table, "block_table", torch.int32, 2)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    _check(q_start, "q_start", torch.int32, 1)
    _check(q_offset, "q_offset", torch.int32, 1)
    _check(out, "out")
    _check(lse, "lse", torch.float32)
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    T, Hq, D = q.shape
    P, ps, Hkv, D2 = k_cache.shape
    B = block_table.shape[0]
    if D2 != D or q_start.shape[0] != B + 1 or seq_lens.shape[0] != B:
        raise ValueError("q / k_cache / block_table / q_start / seq_lens shapes disagree")
    dims = PaDims(B, T, Hq, Hkv, D, ps, P, block_table.shape[1], _dtype_code(q), _q_token_stride(q))
    args = (_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens), _ptr(q_start),
            int(bool(causal)), _ptr(q_offset), int(split_kv), float(scale), _ptr(out), _ptr(lse), ctypes.byref(dims))
    if hint is None:
        rc = load_library().paged_attn_fwd_varlen(*args, _stream(stream))
        _raise(rc, "paged_attn_fwd_varlen")
    else:
        rc = load_library().paged_attn_fwd_varlen_overlap(*args, ctypes.byref(hint), _stream(stream))
        _raise(rc, "paged_attn_fwd_varlen_overlap")


def paged_attn_fwd_varlen_overlap(q, k_cache, v_cache, block_table, seq_lens, q_start, causal, q_offset, split_kv,
                                  scale, out, lse, hint, stream=None) -> None:
    """``paged_attn_fwd_varlen`` with its two kernels side by side on disjoint SMs (``hint`` a
    ``PaVarlenHint``)."""
    paged_attn_fwd_varlen(q, k_cache, v_cache, block_table, seq_lens, q_start, causal, q_offset, split_kv, scale,
                          out, lse, stream, hint if hint is not None else PaVarlenHint())


def paged_attn_combine(part_out, part_lse, out, lse=None, stream=None) -> None:
    """Merge split partials: part_out [S, ..., D] f32, part_lse [S, ...] f32 -> out [..., D], lse [...]."""
    torch = _torch()
    _check(part_out, "part_out", torch.float32)
    _check(part_lse, "part_lse", torch.float32)
    _check(out, "out")
    _check(lse, "lse", torch.float32)
    S = part_out.shape[0]
    D = part_out.shape[-1]
    rows = part_out.numel() // (S * D) if S * D else 0
    if part_lse.numel() != S * rows or out.numel() != rows * D:
        raise ValueError("combine shapes disagree")
    rc = load_library().paged_attn_combine(_ptr(part_out), _ptr(part_lse), int(S), int(rows), int(D),
                                           _dtype_code(out), _ptr(out), _ptr(lse), _stream(stream))
    _raise(rc, "paged_attn_combine")


def paged_attn_plan(seq_lens, page_size: int, split_kv: int, plan=None, stream=None):
    torch = _torch()
    _check(seq_lens, "seq_lens", torch.int32, 1)
    B = seq_lens.shape[0]
    if plan is None:
        plan = torch.empty((B, split_kv, 2), dtype=torch.int32, device=seq_lens.device)
    _check(plan, "plan", torch.int32)
    rc = load_library().paged_attn_plan(_ptr(seq_lens), B, int(page_size), int(split_kv), _ptr(plan),
                                        _stream(stream))
    _raise(rc, "paged_attn_plan")
    return plan


def paged_attn_debug_gather(cache, block_table, seq_lens, out_tokens: int, out=None, stream=None):
    torch = _torch()
    _check(cache, "cache", ndim=4)
    _check(block_table, "block_table", torch.int32, 2)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    P, ps, Hkv, D = cache.shape
    B = block_table.shape[0]
    if out is None:
        out = torch.empty((B, out_tokens, Hkv, D), dtype=cache.dtype, device=cache.device)
    _check(out, "out", cache.dtype)
    dims = PaDims(B, 1, Hkv, Hkv, D, ps, P, block_table.shape[1], _dtype_code(cache))
    rc = load_library().paged_attn_debug_gather(_ptr(cache), _ptr(block_table), _ptr(seq_lens), ctypes.byref(dims),
                                                int(out_tokens), _ptr(out), _stream(stream))
    _raise(rc, "paged_attn_debug_gather")
    return out


def paged_attn_debug_wait_timeout(limit_us: int, stream=None) -> None:
    """Run the kernels' bounded pipeline wait on a barrier nothing completes; it gives up after
    ``limit_us`` and sets ERRBIT_TIMEOUT (see include/paged_attn.h)."""
    _raise(load_library().paged_attn_debug_wait_timeout(int(limit_us), _stream(stream)), "paged_attn_debug_wait_timeout")


def paged_attn_last_error_word() -> int:
    """Read and clear the device error word; returns its PA_ERRBIT_* bits.  The C call's statuses
    that describe the bits (PA_ETIMEOUT, PA_EBOUNDS, PA_EINVAL with bits set) are not raised here:
    the bits carry the same facts (see ``paged_attn_last_error_status``)."""
    return paged_attn_last_error_status()[1]


def paged_attn_last_error_status():
    """(status, bits) of paged_attn_last_error_word: status PA_OK, PA_ETIMEOUT, PA_EBOUNDS or
    PA_EINVAL (a bad q_start entry), as the header defines them.  A failed read raises."""
    v = ctypes.c_uint32(0)
    rc = load_library().paged_attn_last_error_word(ctypes.byref(v))
    if rc in (PA_ETIMEOUT, PA_EBOUNDS) or (rc == PA_EINVAL and v.value):
        return rc, int(v.value)
    _raise(rc, "paged_attn_last_error_word")
    return rc, int(v.value)


def paged_attn_strerror(code: int) -> str:
    return load_library().paged_attn_strerror(int(code)).decode()


def paged_attn_version() -> int:
    return int(load_library().paged_attn_version())


# ----------------------------------------------------------------------------- convenience
def attention(q, k_cache, v_cache, block_table, seq_lens, *, causal: bool = False, q_offset=None,
              split_kv: int = 1, scale: Optional[float] = None, want_lse: bool = False,
              variant: int = VARIANT_AUTO, partials=None, stream=None):
    """Full forward: allocate outputs, run the split forward and, when split_kv > 1, the combine.

    Returns ``out`` ([B, Sq, Hq, D], q's dtype) or ``(out, lse)`` with ``want_lse``.
    ``partials`` may pass preallocated (part_out [S,B,Sq,Hq,D] f32, part_lse [S,B,Sq,Hq] f32).
    """
    torch = _torch()
    B, Sq, Hq, D = q.shape
    if scale is None:
        scale = D ** -0.5
    out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    lse = torch.empty((B, Sq, Hq), dtype=torch.float32, device=q.device) if (want_lse or split_kv > 1) else None
    if split_kv == 1:
        paged_attn_fwd_variant(q, k_cache, v_cache, block_table, seq_lens, causal, q_offset, 1, scale, out, lse,
                               variant, stream)
    else:
        if partials is None:
            po = torch.empty((split_kv, B, Sq, Hq, D), dtype=torch.float32, device=q.device)
            pl = torch.empty((split_kv, B, Sq, Hq), dtype=torch.float32, device=q.device)
        else:
            po, pl = partials
        paged_attn_fwd_variant(q, k_cache, v_cache, block_table, seq_lens, causal, q_offset, split_kv, scale, po,
                               pl, variant, stream)
        paged_attn_combine(po, pl, out, lse, stream)
    return (out, lse) if want_lse else out


def attention_kvq(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, *, causal: bool = False,
                  q_offset=None, split_kv: int = 1, scale: Optional[float] = None, want_lse: bool = False,
                  stream=None, kv_dtype=None):
    """``attention`` over 8-bit pools with per-(page, kv head) scales; ``kv_dtype`` as in
    ``paged_attn_fwd_kvq``."""
    torch = _torch()
    B, Sq, Hq, D = q.shape
    if scale is None:
        scale = D ** -0.5
    out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    lse = torch.empty((B, Sq, Hq), dtype=torch.float32, device=q.device) if (want_lse or split_kv > 1) else None
    if split_kv == 1:
        paged_attn_fwd_kvq(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, causal, q_offset, 1, scale,
                           out, lse, stream, kv_dtype)
    else:
        po = torch.empty((split_kv, B, Sq, Hq, D), dtype=torch.float32, device=q.device)
        pl = torch.empty((split_kv, B, Sq, Hq), dtype=torch.float32, device=q.device)
        paged_attn_fwd_kvq(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, causal, q_offset, split_kv,
                           scale, po, pl, stream, kv_dtype)
        paged_attn_combine(po, pl, out, lse, stream)
    return (out, lse) if want_lse else out


def attention_varlen(q, k_cache, v_cache, block_table, seq_lens, q_start, *, causal: bool = False, q_offset=None,
                     split_kv: int = 1, scale: Optional[float] = None, want_lse: bool = False, stream=None,
                     hint=None):
    """``attention`` for a packed variable-length batch: q [T, Hq, D], q_start [B + 1].  With
    ``hint`` (``paged_attn_varlen_hint``) the forward runs its two kernels side by side."""
    torch = _torch()
    T, Hq, D = q.shape
    if scale is None:
        scale = D ** -0.5
    out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device) if (want_lse or split_kv > 1) else None
    if split_kv == 1:
        paged_attn_fwd_varlen(q, k_cache, v_cache, block_table, seq_lens, q_start, causal, q_offset, 1, scale, out,
                              lse, stream, hint)
    else:
        po = torch.empty((split_kv, T, Hq, D), dtype=torch.float32, device=q.device)
        pl = torch.empty((split_kv, T, Hq), dtype=torch.float32, device=q.device)
        paged_attn_fwd_varlen(q, k_cache, v_cache, block_table, seq_lens, q_start, causal, q_offset, split_kv,
                              scale, po, pl, stream, hint)
        paged_attn_combine(po, pl, out, lse, stream)
    return (out, lse) if want_lse else out
