"""Helpers for the GPU tests: place a workload on the device, run the library, compare with the oracle."""
from __future__ import annotations

import numpy as np

from paged_kv_cache_201_gb300 import workloads as W

# Tolerances: bf16/f16 atol=2e-3, rtol=2^-8 (rocm-libraries PR #14349 numeric tests); f32 1e-5.
TOL = {"bf16": (2e-3, 2.0 ** -8), "f16": (2e-3, 2.0 ** -8), "f32": (1e-5, 1e-5)}


class DeviceWorkload:
    """Device tensors of a workload (K/V drawn on the device when the workload says so)."""

    def __init__(self, wl: W.Workload, device="cuda"):
        import torch
        self.wl = wl
        self.q = W.host_to_torch(wl.q, wl.dtype).to(device)
        self.kvq = getattr(wl, "kv_dtype", None) in W.QUANT_KV
        self.kv_code = {"fp8e4m3": 3, "int8": 4}.get(getattr(wl, "kv_dtype", None))  # PA_FP8_E4M3 / PA_INT8
        self.ks = self.vs = None
        if self.kvq:
            if wl.k_cache is not None:
                self.k = torch.from_numpy(np.ascontiguousarray(wl.k_cache, dtype=np.uint8)).to(device)
                self.v = torch.from_numpy(np.ascontiguousarray(wl.v_cache, dtype=np.uint8)).to(device)
                self.ks = torch.from_numpy(np.ascontiguousarray(wl.k_scale, dtype=np.float32)).to(device)
                self.vs = torch.from_numpy(np.ascontiguousarray(wl.v_scale, dtype=np.float32)).to(device)
            else:
                self.k, self.v, self.ks, self.vs = W.fill_device_cache_q8(wl, device)
        elif wl.k_cache is not None:
            self.k = W.host_to_torch(wl.k_cache, wl.dtype).to(device)
            self.v = W.host_to_torch(wl.v_cache, wl.dtype).to(device)
        else:
            self.k, self.v = W.fill_device_cache(wl, device)
        self.bt = torch.from_numpy(np.ascontiguousarray(wl.block_table)).to(device)
        self.sl = torch.from_numpy(np.ascontiguousarray(wl.seq_lens)).to(device)
        self.qo = None if wl.q_offset is None else torch.from_numpy(np.ascontiguousarray(wl.q_offset)).to(device)

    def host_pools(self):
        """The device pools as host element arrays (uint16 bits or float32; uint8 bits for
        quantized pools), for the oracle."""
        if self.kvq:
            return self.k.cpu().numpy(), self.v.cpu().numpy()
        return to_host_elems(self.k, self.wl.dtype), to_host_elems(self.v, self.wl.dtype)

    def host_scales(self):
        return self.ks.cpu().numpy(), self.vs.cpu().numpy()


def to_host_elems(t, dtype):
    import torch
    if dtype == "f32":
        return t.detach().cpu().numpy()
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def to_f64(t, dtype):
    """Device tensor of the workload dtype (or float32) -> float64 numpy."""
    import torch
    if t.dtype == torch.float32:
        # partial rows with lse -inf may hold any bits (they need not be written), signalling NaNs
        # included
        with np.errstate(invalid="ignore"):
            return t.detach().cpu().numpy().astype(np.float64)
    return t.detach().float().cpu().numpy().astype(np.float64)


def run(dw: DeviceWorkload, split_kv: int, variant: int = 0):
    """Forward (+ combine for split_kv > 1).  Returns dict of float64 numpy arrays:
    out [B,Sq,Hq,D], lse [B,Sq,Hq] and, for split_kv > 1, part_out [S,B,Sq,Hq,D], part_lse [S,B,Sq,Hq]."""
    import torch
    import paged_kv_cache_201_gb300 as pa
    wl = dw.wl
    B, Sq, Hq, D = wl.B, wl.Sq, wl.Hq, wl.D
    res = {}

    def fwd(S, o, l):
        if dw.kvq:
            assert variant == 0
            pa.paged_attn_fwd_kvq(dw.q, dw.k, dw.v, dw.ks, dw.vs, dw.bt, dw.sl, wl.causal, dw.qo, S, wl.scale, o, l,
                                  kv_dtype=dw.kv_code)
        else:
            pa.paged_attn_fwd_variant(dw.q, dw.k, dw.v, dw.bt, dw.sl, wl.causal, dw.qo, S, wl.scale, o, l, variant)

    if split_kv == 1:
        out = torch.empty(dw.q.shape, dtype=dw.q.dtype, device=dw.q.device)
        lse = torch.empty((B, Sq, Hq), dtype=torch.float32, device=dw.q.device)
        fwd(1, out, lse)
    else:
        po = torch.empty((split_kv, B, Sq, Hq, D), dtype=torch.float32, device=dw.q.device)
        pl = torch.empty((split_kv, B, Sq, Hq), dtype=torch.float32, device=dw.q.device)
        fwd(split_kv, po, pl)
        out = torch.empty(dw.q.shape, dtype=dw.q.dtype, device=dw.q.device)
        lse = torch.empty((B, Sq, Hq), dtype=torch.float32, device=dw.q.device)
        pa.paged_attn_combine(po, pl, out, lse)
        res["part_out"] = to_f64(po, "f32")
        res["part_lse"] = to_f64(pl, "f32")
    torch.cuda.synchronize()
    res["out"] = to_f64(out, wl.dtype)
    res["lse"] = to_f64(lse, "f32")
    return res


def assert_close(got, want, dtype, what):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert not np.isnan(got).any(), f"{what}: NaN in GPU result"
    ninf_w, ninf_g = np.isneginf(want), np.isneginf(got)
    assert np.array_equal(ninf_w, ninf_g), f"{what}: -inf pattern differs ({ninf_w.sum()} vs {ninf_g.sum()})"
    fin = ~ninf_w
    assert np.isfinite(got[fin]).all(), f"{what}: non-finite GPU values"
    atol, rtol = TOL[dtype]
    err = np.abs(got[fin] - want[fin])
    bound = atol + rtol * np.abs(want[fin])
    bad = err > bound
    if bad.any():
        k = int(np.argmax(err - bound))
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements beyond atol={atol} rtol={rtol}; "
                             f"worst |d|={err[k]:.3g} at want={want[fin][k]:.6g} got={got[fin][k]:.6g}")
    return float(err.max()) if err.size else 0.0


def _written(part_out, ref_part_lse):
    """The GPU partial outputs [n, S, D] with the rows of partitions that hold no valid key (lse -inf,
    checked separately) set to the oracle's 0: those rows need not be written, and the combine never
    reads them."""
    po = np.array(part_out, dtype=np.float64, copy=True)
    po[np.isneginf(ref_part_lse)] = 0.0
    return po


def compare_rows(res, ref, rows_bih, wl, split_kv, what):
    """Compare GPU results at the sampled rows with oracle row results."""
    b, i, h = rows_bih[:, 0], rows_bih[:, 1], rows_bih[:, 2]
    dt = wl.dtype
    if split_kv == 1:
        e = assert_close(res["out"][b, i, h], ref["out"], dt, f"{what} out")
        assert_close(res["lse"][b, i, h], ref["lse"], dt, f"{what} lse")
    else:
        e = assert_close(res["out"][b, i, h], ref["comb_out"], dt, f"{what} combined out")
        assert_close(res["lse"][b, i, h], ref["comb_lse"], dt, f"{what} combined lse")
        po = np.moveaxis(res["part_out"][:, b, i, h], 0, 1)  # [n, S, D]
        pl = np.moveaxis(res["part_lse"][:, b, i, h], 0, 1)  # [n, S]
        assert_close(pl, ref["part_lse"], dt, f"{what} partial lse")
        assert_close(_written(po, ref["part_lse"]), ref["part_out"], dt, f"{what} partial out")
    return e


def compare_all(res, ref, wl, split_kv, what, chunk=1 << 14):
    """Compare every output row of a GPU result with an oracle result computed on
    ``oracle.all_rows`` (b slowest, then i, then h), in chunks of rows so that the
    full-size workloads' partials (up to 1 GiB of float64) need no indexed copies.

    ``ref`` may come from an oracle call with a larger split count than ``split_kv``
    only when split_kv == 1: then its unsplit ``out`` / ``lse`` are the reference."""
    D, dt = wl.D, wl.dtype
    n = wl.B * wl.Sq * wl.Hq
    out = res["out"].reshape(n, D)
    lse = res["lse"].reshape(n)
    if split_kv > 1:
        po = res["part_out"].reshape(split_kv, n, D)
        pl = res["part_lse"].reshape(split_kv, n)
    worst = 0.0
    for a in range(0, n, chunk):
        e = min(n, a + chunk)
        tag = f"{what} rows {a}..{e - 1}"
        if split_kv == 1:
            worst = max(worst, assert_close(out[a:e], ref["out"][a:e], dt, f"{tag} out"))
            assert_close(lse[a:e], ref["lse"][a:e], dt, f"{tag} lse")
        else:
            worst = max(worst, assert_close(out[a:e], ref["comb_out"][a:e], dt, f"{tag} combined out"))
            assert_close(lse[a:e], ref["comb_lse"][a:e], dt, f"{tag} combined lse")
            assert_close(np.moveaxis(pl[:, a:e], 0, 1), ref["part_lse"][a:e], dt, f"{tag} partial lse")
            assert_close(_written(np.moveaxis(po[:, a:e], 0, 1), ref["part_lse"][a:e]), ref["part_out"][a:e], dt,
                         f"{tag} partial out")
    return worst


_ORACLE_CACHE = {}


def oracle_all_rows(wl, split_kv, k_cache=None, v_cache=None, k_scale=None, v_scale=None):
    """The oracle on every row of a named workload (unsplit result plus the split_kv partials and
    their combination), computed once per (workload, split_kv) in this process: several test files
    check the same full-size workloads, and one fp64 pass over them takes seconds to tens of seconds.
    Quantized pools (8-bit elements) take their scales."""
    import oracle
    key = (wl.name, wl.B, wl.Sq, split_kv)
    if key not in _ORACLE_CACHE:
        rows = oracle.all_rows(wl.B, wl.Sq, wl.Hq)
        if getattr(wl, "kv_dtype", None) in W.QUANT_KV:
            _ORACLE_CACHE[key] = oracle.workload_rows_kvq(wl, split_kv=split_kv, row_bih=rows, k_cache=k_cache,
                                                          v_cache=v_cache, k_scale=k_scale, v_scale=v_scale)
        else:
            _ORACLE_CACHE[key] = oracle.workload_rows(wl, split_kv=split_kv, row_bih=rows, k_cache=k_cache,
                                                      v_cache=v_cache)
    return _ORACLE_CACHE[key]
