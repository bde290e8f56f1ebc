"""fp64 CPU oracle for paged attention (ctypes wrapper around ``paged_attn_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline arm use it.  The library never imports it, and it imports nothing
from the library.

Arrays are numpy: q / k_cache / v_cache hold float32 values for ``f32`` and the
raw uint16 element bits for ``bf16`` / ``f16``; integer inputs are int32.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "paged_attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2}
KV_FP8E4M3 = 3
KV_INT8 = 4
KV_CODE = {"fp8e4m3": KV_FP8E4M3, "int8": KV_INT8}
OK, EINVAL, EBOUNDS, ENOMEM = 0, -1, -5, -6


class Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Sq", ctypes.c_int32), ("Hq", ctypes.c_int32),
                ("Hkv", ctypes.c_int32), ("D", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("bt_stride", ctypes.c_int32), ("dtype", ctypes.c_int32), ("num_pages", ctypes.c_int64)]


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle with gcc (fp64, OpenMP over query rows)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-Wall", "-Wextra",
           "-Wno-unused-parameter", *extra_flags, src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


_lib_cache = {}


def load(path: str = _LIB_PATH, rebuild_if_stale: bool = True):
    """Load (building first when missing or older than the source) the oracle library."""
    if path in _lib_cache:
        return _lib_cache[path]
    if path == _LIB_PATH and rebuild_if_stale:
        if not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_SRC):
            build()
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    lib.oracle_plan.argtypes = [P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, P]
    lib.oracle_plan.restype = ctypes.c_int
    lib.oracle_gather.argtypes = [P, P, P, ctypes.POINTER(Dims), ctypes.c_int32, P]
    lib.oracle_gather.restype = ctypes.c_int
    lib.oracle_key_limit.argtypes = [P, P, ctypes.c_int32, ctypes.POINTER(Dims), ctypes.c_int32, ctypes.c_int32]
    lib.oracle_key_limit.restype = ctypes.c_int64
    lib.oracle_combine.argtypes = [P, P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, P, P]
    lib.oracle_combine.restype = None
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_rows.argtypes = [P, P, P, P, P, P, ctypes.c_int32, ctypes.POINTER(Dims), ctypes.c_double,
                                ctypes.c_int32, P, P, P, ctypes.c_int64, ctypes.c_int32,
                                P, P, P, P, P, P]
    lib.oracle_rows.restype = ctypes.c_int
    lib.oracle_rows_kvq.argtypes = [P, P, P, ctypes.c_int32, P, P, P, P, P, ctypes.c_int32, ctypes.POINTER(Dims),
                                    ctypes.c_double, ctypes.c_int32, P, P, P, ctypes.c_int64, ctypes.c_int32,
                                    P, P, P, P, P, P]
    lib.oracle_rows_kvq.restype = ctypes.c_int
    lib.oracle_gather_kvq.argtypes = [P, ctypes.c_int32, P, P, P, ctypes.POINTER(Dims), ctypes.c_int32, P]
    lib.oracle_gather_kvq.restype = ctypes.c_int
    _lib_cache[path] = lib
    return lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _elems(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.ascontiguousarray(a, dtype=np.float32)
    return np.ascontiguousarray(a).view(np.uint16)


def make_dims(*, B, Sq, Hq, Hkv, D, page_size, bt_stride, dtype, num_pages) -> Dims:
    return Dims(B, Sq, Hq, Hkv, D, page_size, bt_stride, DTYPE_CODE[dtype], num_pages)


def dims_of(wl) -> Dims:
    """Dims from any object with the workload attributes (B, Sq, Hq, ... dtype)."""
    return make_dims(B=wl.B, Sq=wl.Sq, Hq=wl.Hq, Hkv=wl.Hkv, D=wl.D, page_size=wl.page_size,
                     bt_stride=int(wl.block_table.shape[1]), dtype=wl.dtype, num_pages=wl.num_pages)


def plan(seq_lens: np.ndarray, page_size: int, split_kv: int, lib=None) -> np.ndarray:
    """Split plan int32 [B, S, 2] = {first page, one past the last page} of each split."""
    lib = lib or load()
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    out = np.zeros((sl.shape[0], split_kv, 2), dtype=np.int32)
    rc = lib.oracle_plan(_ptr(sl), sl.shape[0], page_size, split_kv, _ptr(out))
    if rc != OK:
        raise ValueError(f"oracle_plan failed: {rc}")
    return out


def gather(cache: np.ndarray, block_table: np.ndarray, seq_lens: np.ndarray, dims: Dims, b: int,
           lib=None) -> np.ndarray:
    """Logically ordered cache rows of sequence b: float64 [L_b, Hkv, D]."""
    lib = lib or load()
    dt = {v: k for k, v in DTYPE_CODE.items()}[dims.dtype]
    c = _elems(cache, dt)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    L = max(int(sl[b]), 0)
    out = np.zeros((L, dims.Hkv, dims.D), dtype=np.float64)
    rc = lib.oracle_gather(_ptr(c), _ptr(bt), _ptr(sl), ctypes.byref(dims), b, _ptr(out))
    if rc != OK:
        raise ValueError(f"oracle_gather failed: {rc}")
    return out


def key_limit(seq_lens, q_offset, causal: bool, dims: Dims, b: int, i: int, lib=None) -> int:
    lib = lib or load()
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    qo = None if q_offset is None else np.ascontiguousarray(q_offset, dtype=np.int32)
    return int(lib.oracle_key_limit(_ptr(sl), _ptr(qo), int(causal), ctypes.byref(dims), b, i))


def combine(part_out: np.ndarray, part_lse: np.ndarray, lib=None):
    """Combine per-split results: part_out [n, S, D], part_lse [n, S] -> (out [n, D], lse [n])."""
    lib = lib or load()
    po = np.ascontiguousarray(part_out, dtype=np.float64)
    pl = np.ascontiguousarray(part_lse, dtype=np.float64)
    n, S, D = po.shape
    out = np.zeros((n, D), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    lib.oracle_combine(_ptr(po), _ptr(pl), n, S, D, _ptr(out), _ptr(lse))
    return out, lse


def num_threads(lib=None) -> int:
    lib = lib or load()
    return int(lib.oracle_num_threads())


def all_rows(B: int, Sq: int, Hq: int) -> np.ndarray:
    """Every (b, i, h) triple, b slowest: int32 [B*Sq*Hq, 3]."""
    b, i, h = np.meshgrid(np.arange(B), np.arange(Sq), np.arange(Hq), indexing="ij")
    return np.stack([b.ravel(), i.ravel(), h.ravel()], axis=1).astype(np.int32)


def rows(*, q, k_cache, v_cache, block_table, seq_lens, q_offset, causal: bool, dims: Dims, scale: float,
         split_kv: int = 1, row_bih: Optional[np.ndarray] = None, n_threads: int = 0, want_split: bool = True,
         lib=None) -> dict:
    """Attention for the chosen query rows (all rows when ``row_bih`` is None).

    Returns float64 arrays: ``out`` [n, D] / ``lse`` [n] (every valid key), and when
    ``want_split``: ``part_out`` [n, S, D] / ``part_lse`` [n, S] (the page plan's
    splits) and ``comb_out`` [n, D] / ``comb_lse`` [n] (those splits combined).
    """
    lib = lib or load()
    dt = {v: k for k, v in DTYPE_CODE.items()}[dims.dtype]
    qe = _elems(q, dt)
    ke = _elems(k_cache, dt)
    ve = _elems(v_cache, dt)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    qo = None if q_offset is None else np.ascontiguousarray(q_offset, dtype=np.int32)
    if row_bih is None:
        row_bih = all_rows(dims.B, dims.Sq, dims.Hq)
    row_bih = np.ascontiguousarray(row_bih, dtype=np.int32)
    rb = np.ascontiguousarray(row_bih[:, 0])
    ri = np.ascontiguousarray(row_bih[:, 1])
    rh = np.ascontiguousarray(row_bih[:, 2])
    n, D, S = row_bih.shape[0], dims.D, split_kv
    res = {"out": np.zeros((n, D)), "lse": np.zeros((n,))}
    if want_split:
        res.update(part_out=np.zeros((n, S, D)), part_lse=np.zeros((n, S)), comb_out=np.zeros((n, D)),
                   comb_lse=np.zeros((n,)))
    rc = lib.oracle_rows(_ptr(qe), _ptr(ke), _ptr(ve), _ptr(bt), _ptr(sl), _ptr(qo), int(causal),
                         ctypes.byref(dims), float(scale), S, _ptr(rb), _ptr(ri), _ptr(rh), n, n_threads,
                         _ptr(res["out"]), _ptr(res["lse"]), _ptr(res.get("part_out")),
                         _ptr(res.get("part_lse")), _ptr(res.get("comb_out")), _ptr(res.get("comb_lse")))
    if rc != OK:
        raise ValueError(f"oracle_rows failed: {rc}")
    return res


def workload_rows(wl, split_kv: int = 1, row_bih=None, n_threads: int = 0, want_split: bool = True,
                  k_cache=None, v_cache=None, lib=None) -> dict:
    """``rows`` on an object with the workload attributes; K/V pools may be passed explicitly."""
    return rows(q=wl.q, k_cache=wl.k_cache if k_cache is None else k_cache,
                v_cache=wl.v_cache if v_cache is None else v_cache, block_table=wl.block_table,
                seq_lens=wl.seq_lens, q_offset=wl.q_offset, causal=wl.causal, dims=dims_of(wl),
                scale=wl.scale, split_kv=split_kv, row_bih=row_bih, n_threads=n_threads,
                want_split=want_split, lib=lib)


# ----------------------------------------------------------------------------- quantized pools
def gather_kvq(cache_bits: np.ndarray, scales: np.ndarray, block_table, seq_lens, dims: Dims, b: int,
               lib=None, kv_dtype: str = "fp8e4m3") -> np.ndarray:
    """Dequantized logical rows of sequence b from a quantized pool (uint8 bits of FP8 E4M3 or
    int8 elements, ``kv_dtype``) with [num_pages, Hkv] float32 scales: float64 [L_b, Hkv, D]."""
    lib = lib or load()
    c = np.ascontiguousarray(cache_bits, dtype=np.uint8)
    sc = np.ascontiguousarray(scales, dtype=np.float32)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    L = max(int(sl[b]), 0)
    out = np.zeros((L, dims.Hkv, dims.D), dtype=np.float64)
    rc = lib.oracle_gather_kvq(_ptr(c), KV_CODE[kv_dtype], _ptr(sc), _ptr(bt), _ptr(sl), ctypes.byref(dims), b, _ptr(out))
    if rc != OK:
        raise ValueError(f"oracle_gather_kvq failed: {rc}")
    return out


def rows_kvq(*, q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, q_offset, causal: bool, dims: Dims,
             scale: float, split_kv: int = 1, row_bih: Optional[np.ndarray] = None, n_threads: int = 0,
             want_split: bool = True, lib=None, kv_dtype: str = "fp8e4m3") -> dict:
    """``rows`` with quantized K/V pools (uint8 bits of FP8 E4M3 or int8 elements, ``kv_dtype``) and
    [num_pages, Hkv] float32 scales per pool; q is float32 / uint16 bits of dims.dtype as in ``rows``."""
    lib = lib or load()
    dt = {v: k for k, v in DTYPE_CODE.items()}[dims.dtype]
    qe = _elems(q, dt)
    ke = np.ascontiguousarray(k_cache, dtype=np.uint8)
    ve = np.ascontiguousarray(v_cache, dtype=np.uint8)
    ks = np.ascontiguousarray(k_scale, dtype=np.float32)
    vs = np.ascontiguousarray(v_scale, dtype=np.float32)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    qo = None if q_offset is None else np.ascontiguousarray(q_offset, dtype=np.int32)
    if row_bih is None:
        row_bih = all_rows(dims.B, dims.Sq, dims.Hq)
    row_bih = np.ascontiguousarray(row_bih, dtype=np.int32)
    rb, ri, rh = (np.ascontiguousarray(row_bih[:, k]) for k in range(3))
    n, D, S = row_bih.shape[0], dims.D, split_kv
    res = {"out": np.zeros((n, D)), "lse": np.zeros((n,))}
    if want_split:
        res.update(part_out=np.zeros((n, S, D)), part_lse=np.zeros((n, S)), comb_out=np.zeros((n, D)),
                   comb_lse=np.zeros((n,)))
    rc = lib.oracle_rows_kvq(_ptr(qe), _ptr(ke), _ptr(ve), KV_CODE[kv_dtype], _ptr(ks), _ptr(vs), _ptr(bt), _ptr(sl),
                             _ptr(qo), int(causal), ctypes.byref(dims), float(scale), S, _ptr(rb), _ptr(ri),
                             _ptr(rh), n, n_threads, _ptr(res["out"]), _ptr(res["lse"]), _ptr(res.get("part_out")),
                             _ptr(res.get("part_lse")), _ptr(res.get("comb_out")), _ptr(res.get("comb_lse")))
    if rc != OK:
        raise ValueError(f"oracle_rows_kvq failed: {rc}")
    return res


def workload_rows_kvq(wl, split_kv: int = 1, row_bih=None, n_threads: int = 0, want_split: bool = True,
                      k_cache=None, v_cache=None, k_scale=None, v_scale=None, lib=None) -> dict:
    """``rows_kvq`` on an object with the workload attributes (pools as uint8 bits + scales; the
    element format is the workload's ``kv_dtype``)."""
    return rows_kvq(q=wl.q, k_cache=wl.k_cache if k_cache is None else k_cache,
                    v_cache=wl.v_cache if v_cache is None else v_cache,
                    k_scale=wl.k_scale if k_scale is None else k_scale,
                    v_scale=wl.v_scale if v_scale is None else v_scale, block_table=wl.block_table,
                    seq_lens=wl.seq_lens, q_offset=wl.q_offset, causal=wl.causal, dims=dims_of(wl), scale=wl.scale,
                    split_kv=split_kv, row_bih=row_bih, n_threads=n_threads, want_split=want_split, lib=lib,
                    kv_dtype=wl.kv_dtype)


# ----------------------------------------------------------------------------- variable-length batches
def rows_varlen(*, q, k_cache, v_cache, block_table, seq_lens, q_start, q_offset, causal: bool, dims: Dims,
                scale: float, split_kv: int = 1, n_threads: int = 0, want_split: bool = True, lib=None) -> dict:
    """A batch whose sequences have different query counts.  q holds every sequence's query tokens
    packed, [T, Hq, D] (dims.Sq = T); sequence b's tokens are rows q_start[b] .. q_start[b+1] - 1.
    Each sequence is the uniform case with a batch of one (its own query count, block-table row,
    length and offset; without an offset its queries are its last tokens), evaluated by ``rows``.

    Returns float64 arrays over the packed rows: ``out`` [T, Hq, D], ``lse`` [T, Hq] and, with
    ``want_split``, ``part_out`` [S, T, Hq, D], ``part_lse`` [S, T, Hq], ``comb_out`` / ``comb_lse``.
    """
    qs = np.asarray(q_start, dtype=np.int64)
    B = int(qs.shape[0]) - 1
    T, Hq, D, S = int(dims.Sq), int(dims.Hq), int(dims.D), split_kv
    assert B == dims.B and qs[0] == 0 and qs[-1] == T and np.all(np.diff(qs) >= 0)
    res = {"out": np.zeros((T, Hq, D)), "lse": np.full((T, Hq), -np.inf)}
    if want_split:
        res.update(part_out=np.zeros((S, T, Hq, D)), part_lse=np.full((S, T, Hq), -np.inf),
                   comb_out=np.zeros((T, Hq, D)), comb_lse=np.full((T, Hq), -np.inf))
    bt = np.ascontiguousarray(block_table)
    for b in range(B):
        a, e = int(qs[b]), int(qs[b + 1])
        if e == a:
            continue
        sub = Dims(1, e - a, Hq, dims.Hkv, D, dims.page_size, dims.bt_stride, dims.dtype, dims.num_pages)
        r = rows(q=np.ascontiguousarray(q[a:e])[None], k_cache=k_cache, v_cache=v_cache, block_table=bt[b:b + 1],
                 seq_lens=np.asarray(seq_lens)[b:b + 1], q_offset=None if q_offset is None else np.asarray(q_offset)[b:b + 1],
                 causal=causal, dims=sub, scale=scale, split_kv=split_kv, n_threads=n_threads, want_split=want_split,
                 lib=lib)
        res["out"][a:e] = r["out"].reshape(e - a, Hq, D)
        res["lse"][a:e] = r["lse"].reshape(e - a, Hq)
        if want_split:
            res["part_out"][:, a:e] = np.moveaxis(r["part_out"].reshape(e - a, Hq, S, D), 2, 0)
            res["part_lse"][:, a:e] = np.moveaxis(r["part_lse"].reshape(e - a, Hq, S), 2, 0)
            res["comb_out"][a:e] = r["comb_out"].reshape(e - a, Hq, D)
            res["comb_lse"][a:e] = r["comb_lse"].reshape(e - a, Hq)
    return res
