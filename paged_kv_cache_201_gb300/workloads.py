"""Seeded synthetic workloads for paged attention.

This module only draws inputs: queries, K/V page pools, block tables, sequence
lengths and query offsets.  It holds none of the attention arithmetic, so both
the CUDA path and the CPU oracle can consume exactly the same bytes.

Input structure follows the pages' workloads:

* K/V live in a pool of fixed-size pages ``[num_pages, page_size, Hkv, D]``
  whose physical order is a seeded random permutation ("shuffled page
  ordering", rocMLIR PR #2222, Key Changes 2; rocm-libraries PR #14349,
  Performance: "contiguous and random" page tables).
* A per-sequence block table ``int32 [B, W]`` maps logical page ``j // ps`` of
  sequence ``b`` to a physical page; slots past ``ceil(L_b / ps)`` hold a
  sentinel that must never be read (-1, or 0x7FFFFFFF as in PR #14349,
  Coverage: "the table's tail holds an unmapped page id").
* Values are N(0, 1) draws rounded to bf16/f16 with round-to-nearest-even.

Two generators are used for the page pools.  Small pools are drawn on the host
with ``numpy.random.default_rng``.  The two 2-GiB pools (Llama-3-8B decode and
the over-2^31 decode) are drawn on the device by ``torch.randn`` with a seeded
``torch.Generator`` and cast to bf16 by torch (round-to-nearest-even); tests
that check them copy the device bytes back to the host for the oracle.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np

SENTINEL_MAX = 0x7FFFFFFF  # unmapped page id used for table tails
SENTINEL_NEG = -1

DTYPES = ("f32", "f16", "bf16")
ESIZE = {"f32": 4, "f16": 2, "bf16": 2}


def bf16_bits_rne(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return the uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def f16_bits_rne(x: np.ndarray) -> np.ndarray:
    """Round float32 values to IEEE binary16 (numpy's cast is round-to-nearest-even)."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def _normal_elems(rng: np.random.Generator, n: int, dtype: str) -> np.ndarray:
    x = rng.standard_normal(n, dtype=np.float32)
    if dtype == "f32":
        return x
    if dtype == "bf16":
        return bf16_bits_rne(x)
    return f16_bits_rne(x)


@dataclasses.dataclass
class Workload:
    """One paged-attention problem instance (host arrays; K/V may live on the device)."""

    name: str
    dtype: str
    B: int
    Sq: int
    Hq: int
    Hkv: int
    D: int
    page_size: int
    num_pages: int
    causal: bool
    scale: float
    split_kv: tuple
    seq_lens: np.ndarray            # int32 [B]
    block_table: np.ndarray         # int32 [B, W]
    q: np.ndarray                   # [B, Sq, Hq, D]; float32 for f32, uint16 bits otherwise
    q_offset: Optional[np.ndarray] = None   # int32 [B] or None
    k_cache: Optional[np.ndarray] = None    # [P, ps, Hkv, D] (host) or None if device-drawn
    v_cache: Optional[np.ndarray] = None
    device_cache_seed: Optional[int] = None  # set when the pools are drawn on the device
    kv_dtype: Optional[str] = None           # "fp8e4m3" / "int8": pools hold 8-bit elements (uint8 bits)
                                             # with per-(page, kv head) scales
    k_scale: Optional[np.ndarray] = None     # float32 [num_pages, Hkv] (quantized pools only)
    v_scale: Optional[np.ndarray] = None
    # variable-length batches: q is [T, Hq, D] packed and Sq = T; sequence b's query tokens are
    # rows q_start[b] .. q_start[b+1] - 1
    q_start: Optional[np.ndarray] = None     # int32 [B + 1]

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def W(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def esize(self) -> int:
        return ESIZE[self.dtype]

    @property
    def cache_shape(self):
        return (self.num_pages, self.page_size, self.Hkv, self.D)

    def nblk(self) -> np.ndarray:
        """Pages each sequence occupies (ceil(L_b / page_size))."""
        ps = self.page_size
        return (self.seq_lens.astype(np.int64) + ps - 1) // ps

    def host_cache_available(self) -> bool:
        return self.k_cache is not None

    @property
    def kv_esize(self) -> int:
        return 1 if self.kv_dtype in QUANT_KV else ESIZE[self.dtype]


def _pack_tables(B: int, W: int, nblk: Sequence[int], pages: np.ndarray, tail: int) -> np.ndarray:
    bt = np.full((B, W), tail, dtype=np.int64)
    pos = 0
    for b in range(B):
        n = int(nblk[b])
        bt[b, :n] = pages[pos:pos + n]
        pos += n
    return bt.astype(np.int32)


def make_custom(*, name: str = "custom", dtype: str = "bf16", B: int, Sq: int, Hq: int, Hkv: int,
                D: int, page_size: int, seq_lens: Sequence[int], num_pages: Optional[int] = None,
                W: Optional[int] = None, causal: bool = False, q_offset: Optional[Sequence[int]] = None,
                split_kv: Sequence[int] = (1,), seed: int = 0, shuffle: bool = True,
                tail: int = SENTINEL_MAX, scale: Optional[float] = None,
                zero_q: bool = False) -> Workload:
    """Draw a small host-resident workload with the given shape.

    Pages are assigned to sequences in order from a seeded permutation of the
    pool (or in identity order when ``shuffle`` is False).
    """
    assert dtype in DTYPES
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    assert seq_lens.shape == (B,)
    nblk = (seq_lens.astype(np.int64) + page_size - 1) // page_size
    need = int(nblk.sum())
    if num_pages is None:
        num_pages = max(need, 1)
    assert num_pages >= need, "page pool smaller than the sequences need"
    if W is None:
        W = max(int(nblk.max()) if B else 1, 1)
    assert W >= (int(nblk.max()) if B else 0)
    q = _normal_elems(rng, B * Sq * Hq * D, dtype).reshape(B, Sq, Hq, D)
    if zero_q:
        q = np.zeros_like(q)
    n_cache = num_pages * page_size * Hkv * D
    k = _normal_elems(rng, n_cache, dtype).reshape(num_pages, page_size, Hkv, D)
    v = _normal_elems(rng, n_cache, dtype).reshape(num_pages, page_size, Hkv, D)
    perm = rng.permutation(num_pages) if shuffle else np.arange(num_pages)
    bt = _pack_tables(B, W, nblk, perm, tail)
    qo = None if q_offset is None else np.asarray(q_offset, dtype=np.int32)
    return Workload(name=name, dtype=dtype, B=B, Sq=Sq, Hq=Hq, Hkv=Hkv, D=D, page_size=page_size,
                    num_pages=num_pages, causal=causal,
                    scale=(1.0 / math.sqrt(D)) if scale is None else float(scale),
                    split_kv=tuple(split_kv), seq_lens=seq_lens, block_table=bt, q=q, q_offset=qo,
                    k_cache=k, v_cache=v)


def tiny_decode_f32(seed: int = 1001) -> Workload:
    """Tiny f32 decode: B=2, L={37,50}, Hq=4, Hkv=2, D=64, 16 shuffled pages, table 4 wide, tail -1."""
    return make_custom(name="tiny_decode_f32", dtype="f32", B=2, Sq=1, Hq=4, Hkv=2, D=64,
                       page_size=16, seq_lens=[37, 50], num_pages=16, W=4, split_kv=(1, 2),
                       seed=seed, tail=SENTINEL_NEG)


def ragged_decode(seed: int = 1003) -> Workload:
    """Ragged bf16 decode: B=32, Hq=64, Hkv=4, D=128, L~U[17,1000], table 63 wide, 2048 pages."""
    rng = np.random.default_rng(seed)
    B, Hq, Hkv, D, ps, P, W = 32, 64, 4, 128, 16, 2048, 63
    seq_lens = rng.integers(17, 1001, size=B).astype(np.int32)
    q = _normal_elems(rng, B * Hq * D, "bf16").reshape(B, 1, Hq, D)
    n_cache = P * ps * Hkv * D
    k = _normal_elems(rng, n_cache, "bf16").reshape(P, ps, Hkv, D)
    v = _normal_elems(rng, n_cache, "bf16").reshape(P, ps, Hkv, D)
    nblk = (seq_lens.astype(np.int64) + ps - 1) // ps
    perm = rng.permutation(P)
    bt = _pack_tables(B, W, nblk, perm, SENTINEL_MAX)
    return Workload(name="ragged_decode", dtype="bf16", B=B, Sq=1, Hq=Hq, Hkv=Hkv, D=D, page_size=ps,
                    num_pages=P, causal=False, scale=1.0 / math.sqrt(D), split_kv=(8,),
                    seq_lens=seq_lens, block_table=bt, q=q, k_cache=k, v_cache=v)


def causal_prefill(seed: int = 1005, B: int = 4, Sq: int = 1024, max_q_offset: int = 3072,
                   num_pages: int = 1024, W: int = 256) -> Workload:
    """Causal bf16 prefill: B=4, Sq=1024, Hq=32, Hkv=8, D=128, q_offset~U[0,3072], L=q_offset+Sq."""
    rng = np.random.default_rng(seed)
    Hq, Hkv, D, ps = 32, 8, 128, 16
    q_offset = rng.integers(0, max_q_offset + 1, size=B).astype(np.int32)
    seq_lens = (q_offset + Sq).astype(np.int32)
    q = _normal_elems(rng, B * Sq * Hq * D, "bf16").reshape(B, Sq, Hq, D)
    n_cache = num_pages * ps * Hkv * D
    k = _normal_elems(rng, n_cache, "bf16").reshape(num_pages, ps, Hkv, D)
    v = _normal_elems(rng, n_cache, "bf16").reshape(num_pages, ps, Hkv, D)
    nblk = (seq_lens.astype(np.int64) + ps - 1) // ps
    assert int(nblk.sum()) <= num_pages and int(nblk.max()) <= W
    perm = rng.permutation(num_pages)
    bt = _pack_tables(B, W, nblk, perm, SENTINEL_MAX)
    return Workload(name="causal_prefill", dtype="bf16", B=B, Sq=Sq, Hq=Hq, Hkv=Hkv, D=D, page_size=ps,
                    num_pages=num_pages, causal=True, scale=1.0 / math.sqrt(D), split_kv=(8,),
                    seq_lens=seq_lens, block_table=bt, q=q, q_offset=q_offset, k_cache=k, v_cache=v)


def llama8b_decode(seed: int = 1002, B: int = 256) -> Workload:
    """Llama-3-8B-shaped bf16 decode: Hq=32, Hkv=8, D=128, L=4096, 65536 pages (2 GiB per pool).

    The page pools are drawn on the device (see ``fill_device_cache``).
    """
    rng = np.random.default_rng(seed)
    Hq, Hkv, D, ps, L = 32, 8, 128, 16, 4096
    per_seq = L // ps
    P = 65536 if B == 256 else B * per_seq
    q = _normal_elems(rng, B * Hq * D, "bf16").reshape(B, 1, Hq, D)
    perm = rng.permutation(P).astype(np.int64)
    bt = perm[:B * per_seq].reshape(B, per_seq).astype(np.int32)
    seq_lens = np.full(B, L, dtype=np.int32)
    return Workload(name="llama8b_decode", dtype="bf16", B=B, Sq=1, Hq=Hq, Hkv=Hkv, D=D, page_size=ps,
                    num_pages=P, causal=False, scale=1.0 / math.sqrt(D), split_kv=(1, 4),
                    seq_lens=seq_lens, block_table=bt, q=q, device_cache_seed=seed)


OVER2G_PAGES = 135168          # 2 GiB + 64 MiB per pool at 16 KiB pages
OVER2G_FIRST_HIGH = 131072     # page whose first byte sits at byte 2^31


def over2gib_decode(seed: int = 1004, B: int = 256) -> Workload:
    """bf16 decode past 2^31 bytes: Hq=64, Hkv=4, D=128, L=8192, 135168 pages per pool.

    Every sequence gets 16 pages from the top 4096 (which start at or past byte
    2^31 of the pool) and 496 from below, shuffled within its table row.
    """
    rng = np.random.default_rng(seed)
    Hq, Hkv, D, ps, L = 64, 4, 128, 16, 8192
    per_seq = L // ps                     # 512
    n_high = 16
    n_low = per_seq - n_high
    assert B * n_high <= OVER2G_PAGES - OVER2G_FIRST_HIGH
    q = _normal_elems(rng, B * Hq * D, "bf16").reshape(B, 1, Hq, D)
    high = OVER2G_FIRST_HIGH + rng.permutation(OVER2G_PAGES - OVER2G_FIRST_HIGH).astype(np.int64)
    low = rng.permutation(OVER2G_FIRST_HIGH).astype(np.int64)
    rows = np.concatenate([high[:B * n_high].reshape(B, n_high),
                           low[:B * n_low].reshape(B, n_low)], axis=1)
    rows = rng.permuted(rows, axis=1)
    bt = rows.astype(np.int32)
    seq_lens = np.full(B, L, dtype=np.int32)
    return Workload(name="over2gib_decode", dtype="bf16", B=B, Sq=1, Hq=Hq, Hkv=Hkv, D=D, page_size=ps,
                    num_pages=OVER2G_PAGES, causal=False, scale=1.0 / math.sqrt(D), split_kv=(4,),
                    seq_lens=seq_lens, block_table=bt, q=q, device_cache_seed=seed)


LLAMA_OVER2G_PAGES = 65536 + 2048   # 2 GiB + 64 MiB per pool at 32 KiB pages (Hkv=8, D=128)
LLAMA_OVER2G_FIRST_HIGH = 65536     # page whose first byte sits at byte 2^31


def llama8b_decode_over2gib(seed: int = 1012, B: int = 256) -> Workload:
    """The Llama-3-8B decode shape (Hq=32, Hkv=8, D=128, L=4096, bf16) over pools just past 2^31
    bytes: 65536 + 2048 pages per pool.  Every sequence gets 8 of the 2048 pages that start at or
    past byte 2^31 and 248 from below, shuffled within its table row, so every row reads on both
    sides of byte 2^31.  The same work as ``llama8b_decode``; only where the pages lie differs."""
    rng = np.random.default_rng(seed)
    Hq, Hkv, D, ps, L = 32, 8, 128, 16, 4096
    per_seq = L // ps                     # 256
    n_high = (LLAMA_OVER2G_PAGES - LLAMA_OVER2G_FIRST_HIGH) // 256   # 8
    n_low = per_seq - n_high
    assert B * n_high <= LLAMA_OVER2G_PAGES - LLAMA_OVER2G_FIRST_HIGH
    q = _normal_elems(rng, B * Hq * D, "bf16").reshape(B, 1, Hq, D)
    high = LLAMA_OVER2G_FIRST_HIGH + rng.permutation(LLAMA_OVER2G_PAGES - LLAMA_OVER2G_FIRST_HIGH).astype(np.int64)
    low = rng.permutation(LLAMA_OVER2G_FIRST_HIGH).astype(np.int64)
    rows = np.concatenate([high[:B * n_high].reshape(B, n_high), low[:B * n_low].reshape(B, n_low)], axis=1)
    bt = rng.permuted(rows, axis=1).astype(np.int32)
    seq_lens = np.full(B, L, dtype=np.int32)
    return Workload(name="llama8b_decode_over2gib", dtype="bf16", B=B, Sq=1, Hq=Hq, Hkv=Hkv, D=D, page_size=ps,
                    num_pages=LLAMA_OVER2G_PAGES, causal=False, scale=1.0 / math.sqrt(D), split_kv=(1, 4),
                    seq_lens=seq_lens, block_table=bt, q=q, device_cache_seed=seed)


CONFIGS = {
    "tiny_decode_f32": tiny_decode_f32,
    "llama8b_decode": llama8b_decode,
    "ragged_decode": ragged_decode,
    "over2gib_decode": over2gib_decode,
    "causal_prefill": causal_prefill,
    "llama8b_decode_over2gib": llama8b_decode_over2gib,
}


def make(name: str, **kw) -> Workload:
    return CONFIGS[name](**kw)


# ----------------------------------------------------------------------------- device helpers
def torch_dtype(dtype: str):
    import torch
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]


def host_to_torch(arr: np.ndarray, dtype: str):
    """Wrap host element bits as a CPU torch tensor of the workload dtype (no copy of values)."""
    import torch
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32))
    t = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16))
    return t.view(torch_dtype(dtype))


def fill_device_cache(wl: Workload, device="cuda", chunk: int = 1 << 27):
    """Draw the K and V pools on the device from the workload's seed.

    ``torch.randn`` (float32, seeded ``torch.Generator`` on the device) rounded to
    the workload dtype by torch's cast (round-to-nearest-even).
    """
    import torch
    assert wl.device_cache_seed is not None
    tdt = torch_dtype(wl.dtype)
    out = []
    for which in (0, 1):
        g = torch.Generator(device=device)
        g.manual_seed(int(wl.device_cache_seed) * 2 + which)
        t = torch.empty(wl.cache_shape, dtype=tdt, device=device)
        flat = t.view(-1)
        n = flat.numel()
        for s in range(0, n, chunk):
            e = min(n, s + chunk)
            flat[s:e].copy_(torch.randn(e - s, generator=g, device=device, dtype=torch.float32))
        out.append(t)
    return out[0], out[1]


# ----------------------------------------------------------------------------- quantized pools
QUANT_KV = ("fp8e4m3", "int8")  # 8-bit pool element formats
E4M3_MAX = 448.0
INT8_MAX = 127.0


def quantize_pool_e4m3(x: np.ndarray):
    """Quantize a float32 pool [P, ps, Hkv, D] to FP8 E4M3 with one scale per (page, kv head):
    scale = max |x| / 448 over the page's rows of that head (1 where the block is all zero), and
    the stored element is x / scale rounded to E4M3 (round to nearest even, torch's cast).
    Returns (uint8 bits [P, ps, Hkv, D], float32 scales [P, Hkv])."""
    import torch
    amax = np.abs(x).max(axis=(1, 3))                            # [P, Hkv]
    scale = np.where(amax > 0, amax / E4M3_MAX, 1.0).astype(np.float32)
    y = x / scale[:, None, :, None]
    bits = torch.from_numpy(np.ascontiguousarray(y, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8)
    return bits.numpy().copy(), scale


def quantize_pool_int8(x: np.ndarray):
    """Quantize a float32 pool [P, ps, Hkv, D] to int8 with one scale per (page, kv head):
    scale = max |x| / 127 over the page's rows of that head (1 where the block is all zero), and
    the stored element is x / scale rounded to the nearest integer (ties to even), within
    [-127, 127].  Returns (uint8 bits [P, ps, Hkv, D], float32 scales [P, Hkv])."""
    amax = np.abs(x).max(axis=(1, 3))                            # [P, Hkv]
    scale = np.where(amax > 0, amax / INT8_MAX, 1.0).astype(np.float32)
    y = np.rint(x.astype(np.float32) / scale[:, None, :, None])
    q = np.clip(y, -INT8_MAX, INT8_MAX).astype(np.int8)
    return q.view(np.uint8).copy(), scale


def int8_bits_to_float(bits: np.ndarray) -> np.ndarray:
    """int8 bits (uint8 storage) -> float64 values by numpy's reinterpretation (a library routine)."""
    return np.ascontiguousarray(bits, dtype=np.uint8).view(np.int8).astype(np.float64)


def q8_bits_to_float(bits: np.ndarray, kv_dtype: str) -> np.ndarray:
    """Element values of a quantized pool's bits (without the scales)."""
    return e4m3_bits_to_float(bits) if kv_dtype == "fp8e4m3" else int8_bits_to_float(bits)


def e4m3_bits_to_float(bits: np.ndarray) -> np.ndarray:
    """E4M3 bits -> float64 values by torch's conversion (a library routine)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def make_custom_q8(kv_dtype: str = "fp8e4m3", **kw) -> Workload:
    """``make_custom`` (bf16 or f16 queries) whose K/V pools are then quantized to ``kv_dtype``
    (FP8 E4M3 or int8) with per-(page, kv head) scales (``quantize_pool_e4m3`` /
    ``quantize_pool_int8``) from the same N(0,1) draws, in float32."""
    assert kv_dtype in QUANT_KV
    dtype = kw.pop("dtype", "bf16")
    assert dtype in ("bf16", "f16")
    wl = make_custom(dtype="f32", **kw)
    rng = np.random.default_rng(kw.get("seed", 0) + 7919)
    q = _normal_elems(rng, wl.q.size, dtype).reshape(wl.q.shape)
    quant = quantize_pool_e4m3 if kv_dtype == "fp8e4m3" else quantize_pool_int8
    kb, ks = quant(wl.k_cache)
    vb, vs = quant(wl.v_cache)
    return Workload(**{**wl.__dict__, "name": kw.get("name", f"custom_{kv_dtype}"), "dtype": dtype, "q": q,
                       "k_cache": kb, "v_cache": vb, "kv_dtype": kv_dtype, "k_scale": ks, "v_scale": vs})


def make_custom_fp8(**kw) -> Workload:
    """``make_custom_q8`` with FP8 E4M3 pools."""
    return make_custom_q8("fp8e4m3", **kw)


def make_custom_int8(**kw) -> Workload:
    """``make_custom_q8`` with int8 pools."""
    return make_custom_q8("int8", **kw)


def llama8b_decode_fp8(seed: int = 1006, B: int = 256) -> Workload:
    """The Llama-3-8B-shaped decode with FP8 E4M3 pools (1 GiB each) and per-(page, kv head) scales;
    pools and scales are drawn on the device (``fill_device_cache_fp8``)."""
    wl = llama8b_decode(seed=seed, B=B)
    return Workload(**{**wl.__dict__, "name": "llama8b_decode_fp8", "kv_dtype": "fp8e4m3"})


CONFIGS["llama8b_decode_fp8"] = llama8b_decode_fp8


def llama8b_decode_int8(seed: int = 1011, B: int = 256) -> Workload:
    """The Llama-3-8B-shaped decode with int8 pools (1 GiB each) and per-(page, kv head) scales;
    pools and scales are drawn on the device (``fill_device_cache_q8``)."""
    wl = llama8b_decode(seed=seed, B=B)
    return Workload(**{**wl.__dict__, "name": "llama8b_decode_int8", "kv_dtype": "int8"})


CONFIGS["llama8b_decode_int8"] = llama8b_decode_int8


def fill_device_cache_q8(wl: Workload, device="cuda", pages_per_chunk: int = 4096):
    """Draw the K and V pools on the device (seeded torch.randn, float32) and quantize them to the
    workload's 8-bit format with per-(page, kv head) scales: max|x| / 448 and torch's E4M3 cast, or
    max|x| / 127 and rounding to the nearest integer (ties to even).  Returns (k_bits, v_bits,
    k_scale, v_scale)."""
    import torch
    assert wl.device_cache_seed is not None and wl.kv_dtype in QUANT_KV
    fp8 = wl.kv_dtype == "fp8e4m3"
    out = []
    for which in (0, 1):
        g = torch.Generator(device=device)
        g.manual_seed(int(wl.device_cache_seed) * 2 + which)
        bits = torch.empty(wl.cache_shape, dtype=torch.uint8, device=device)
        scales = torch.empty((wl.num_pages, wl.Hkv), dtype=torch.float32, device=device)
        for p0 in range(0, wl.num_pages, pages_per_chunk):
            p1 = min(wl.num_pages, p0 + pages_per_chunk)
            x = torch.randn((p1 - p0,) + wl.cache_shape[1:], generator=g, device=device, dtype=torch.float32)
            amax = x.abs().amax(dim=(1, 3))
            sc = torch.where(amax > 0, amax / (E4M3_MAX if fp8 else INT8_MAX), torch.ones_like(amax))
            y = x / sc[:, None, :, None]
            if fp8:
                bits[p0:p1] = y.to(torch.float8_e4m3fn).view(torch.uint8)
            else:
                bits[p0:p1] = torch.round(y).clamp_(-INT8_MAX, INT8_MAX).to(torch.int8).view(torch.uint8)
            scales[p0:p1] = sc
        out += [bits, scales]
    return out[0], out[2], out[1], out[3]


# ----------------------------------------------------------------------------- variable-length batches
def make_varlen(*, name: str = "varlen", dtype: str = "bf16", q_lens: Sequence[int], seq_lens: Sequence[int],
                Hq: int, Hkv: int, D: int, page_size: int, causal: bool = True,
                q_offset: Optional[Sequence[int]] = None, num_pages: Optional[int] = None, W: Optional[int] = None,
                split_kv: Sequence[int] = (1,), seed: int = 0, tail: int = SENTINEL_MAX) -> Workload:
    """A host-resident batch whose sequences have their own query counts ``q_lens`` (0 allowed),
    packed into q [T, Hq, D].  Values and pages are drawn as in ``make_custom``."""
    q_lens = np.asarray(q_lens, dtype=np.int64)
    B = int(q_lens.shape[0])
    T = int(q_lens.sum())
    wl = make_custom(name=name, dtype=dtype, B=B, Sq=1, Hq=Hq, Hkv=Hkv, D=D, page_size=page_size,
                     seq_lens=seq_lens, num_pages=num_pages, W=W, causal=causal, q_offset=q_offset,
                     split_kv=split_kv, seed=seed, tail=tail)
    rng = np.random.default_rng(seed + 104729)
    q = _normal_elems(rng, T * Hq * D, dtype).reshape(T, Hq, D)
    q_start = np.zeros(B + 1, dtype=np.int32)
    q_start[1:] = np.cumsum(q_lens)
    return Workload(**{**wl.__dict__, "Sq": T, "q": q, "q_start": q_start})


def mixed_decode_prefill(seed: int = 1007, n_decode: int = 256, n_prefill: int = 4) -> Workload:
    """One batch mixing the Llama-3-8B decode (n_decode sequences, one query token, L=4096) and the
    causal prefill (n_prefill sequences, 1024 query tokens, q_offset~U[0,3072], L = q_offset + 1024):
    Hq=32, Hkv=8, D=128, bf16, page_size 16, prefill sequences first in the packed order.  Pools are
    drawn on the device (``fill_device_cache``): 65536 pages for the decode sequences plus the
    prefill sequences' pages, shuffled together."""
    rng = np.random.default_rng(seed)
    Hq, Hkv, D, ps, L = 32, 8, 128, 16, 4096
    pre_off = rng.integers(0, 3072 + 1, size=n_prefill).astype(np.int64)
    q_lens = np.array([1024] * n_prefill + [1] * n_decode, dtype=np.int64)
    seq_lens = np.concatenate([pre_off + 1024, np.full(n_decode, L)]).astype(np.int32)
    q_offset = (seq_lens.astype(np.int64) - q_lens).astype(np.int32)
    q_offset[:n_prefill] = pre_off
    B = n_prefill + n_decode
    nblk = (seq_lens.astype(np.int64) + ps - 1) // ps
    P = int(nblk.sum())
    W = int(nblk.max())
    T = int(q_lens.sum())
    q = _normal_elems(rng, T * Hq * D, "bf16").reshape(T, Hq, D)
    perm = rng.permutation(P)
    bt = _pack_tables(B, W, nblk, perm, SENTINEL_MAX)
    q_start = np.zeros(B + 1, dtype=np.int32)
    q_start[1:] = np.cumsum(q_lens)
    return Workload(name="mixed_decode_prefill", dtype="bf16", B=B, Sq=T, Hq=Hq, Hkv=Hkv, D=D, page_size=ps,
                    num_pages=P, causal=True, scale=1.0 / math.sqrt(D), split_kv=(1,), seq_lens=seq_lens,
                    block_table=bt, q=q, q_offset=q_offset, device_cache_seed=seed, q_start=q_start)


CONFIGS["mixed_decode_prefill"] = mixed_decode_prefill


def d256_decode(seed: int = 1008, B: int = 128) -> Workload:
    """Head-dim-256 decode shaped like Gemma-2-9B attention: Hq=16, Hkv=8, D=256, L=4096, bf16,
    page_size 16, B * 256 pages per pool (2 GiB each at B=128) in a seeded permutation; pools drawn
    on the device."""
    rng = np.random.default_rng(seed)
    Hq, Hkv, D, ps, L = 16, 8, 256, 16, 4096
    per_seq = L // ps
    P = B * per_seq
    q = _normal_elems(rng, B * Hq * D, "bf16").reshape(B, 1, Hq, D)
    perm = rng.permutation(P).astype(np.int64)
    bt = perm[:B * per_seq].reshape(B, per_seq).astype(np.int32)
    return Workload(name="d256_decode", dtype="bf16", B=B, Sq=1, Hq=Hq, Hkv=Hkv, D=D, page_size=ps,
                    num_pages=P, causal=False, scale=1.0 / math.sqrt(D), split_kv=(1,),
                    seq_lens=np.full(B, L, dtype=np.int32), block_table=bt, q=q, device_cache_seed=seed)


CONFIGS["d256_decode"] = d256_decode


def mha_decode(seed: int = 1009, B: int = 64) -> Workload:
    """Single-head-group decode (no GQA): Hq=Hkv=32, D=128, L=4096, bf16, page_size 16, B * 256 pages
    per pool (2 GiB each at B=64) in a seeded permutation; pools drawn on the device."""
    rng = np.random.default_rng(seed)
    Hq, Hkv, D, ps, L = 32, 32, 128, 16, 4096
    per_seq = L // ps
    P = B * per_seq
    q = _normal_elems(rng, B * Hq * D, "bf16").reshape(B, 1, Hq, D)
    perm = rng.permutation(P).astype(np.int64)
    bt = perm[:B * per_seq].reshape(B, per_seq).astype(np.int32)
    return Workload(name="mha_decode", dtype="bf16", B=B, Sq=1, Hq=Hq, Hkv=Hkv, D=D, page_size=ps,
                    num_pages=P, causal=False, scale=1.0 / math.sqrt(D), split_kv=(1,),
                    seq_lens=np.full(B, L, dtype=np.int32), block_table=bt, q=q, device_cache_seed=seed)


CONFIGS["mha_decode"] = mha_decode


def causal_prefill_f16(seed: int = 1010) -> Workload:
    """The causal prefill shape (B=4, Sq=1024, Hq=32, Hkv=8, D=128, q_offset~U[0,3072]) in f16."""
    wl = causal_prefill(seed=seed)
    def to16(bits):  # bf16 bits -> the same values as f16 bits (exact for these N(0,1) draws)
        f32 = (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
        return f32.astype(np.float16).view(np.uint16)
    return Workload(**{**wl.__dict__, "name": "causal_prefill_f16", "dtype": "f16", "q": to16(wl.q),
                       "k_cache": to16(wl.k_cache), "v_cache": to16(wl.v_cache)})


CONFIGS["causal_prefill_f16"] = causal_prefill_f16
