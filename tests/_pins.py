"""Pins for the fp64 oracle: checks against facts the pages and the mathematics fix.

Each ``pin_*`` takes a loaded oracle library (so the mutation test can run the
same pins against deliberately broken builds) and raises ``AssertionError`` when
the oracle disagrees with the fact it pins.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle
from paged_kv_cache_201_gb300 import workloads as W
from tests import _bruteforce as bf

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _num(x):
    return -math.inf if x == "-inf" else float(x)


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _wl_from_pool(pool, case, scale, Sq=1, q=None, causal=False, q_offset=None):
    k = np.asarray(pool["k"], dtype=np.float32).reshape(-1, pool["page_size"], 1, 1)
    v = np.asarray(pool["v"], dtype=np.float32).reshape(-1, pool["page_size"], 1, 1)
    qq = np.asarray(q if q is not None else [1.0] * Sq, dtype=np.float32).reshape(1, Sq, 1, 1)
    bt = np.asarray([case["block_table"]], dtype=np.int32)
    return W.Workload(name=case["name"], dtype="f32", B=1, Sq=Sq, Hq=1, Hkv=1, D=1,
                      page_size=pool["page_size"], num_pages=k.shape[0], causal=causal, scale=scale,
                      split_kv=(1,), seq_lens=np.asarray([case["L"]], dtype=np.int32), block_table=bt,
                      q=qq, q_offset=None if q_offset is None else np.asarray([q_offset], dtype=np.int32),
                      k_cache=k, v_cache=v)


# ----------------------------------------------------------------------------- golden fixtures
def pin_golden_plan(lib):
    """Split plan equals the hand-worked ceil-div + clamp values (PR #2371)."""
    g = _golden("split_plan.json")
    for c in g["cases"]:
        got = oracle.plan(np.asarray([c["L"]], dtype=np.int32), c["page_size"], c["split_kv"], lib=lib)[0]
        assert got.tolist() == c["plan"], (c, got.tolist())


def pin_golden_attention(lib):
    """D=1 worked examples (unsplit, causal with and without prefix offset, single key)."""
    g = _golden("worked_attention.json")
    for c in g["cases"]:
        wl = _wl_from_pool(g["pool"], c, g["scale"], Sq=c["Sq"], q=c["q"], causal=c["causal"],
                           q_offset=c["q_offset"])
        r = oracle.workload_rows(wl, split_kv=1, lib=lib)
        np.testing.assert_allclose(r["out"][:, 0], c["out"], rtol=0, atol=1e-12, err_msg=c["name"])
        np.testing.assert_allclose(r["lse"], c["lse"], rtol=0, atol=1e-12, err_msg=c["name"])


def pin_golden_split(lib):
    """Per-split partials and their combination on the worked 3-key example."""
    g = _golden("worked_attention.json")
    for c in g["split_cases"]:
        wl = _wl_from_pool(g["pool"], c, g["scale"])
        r = oracle.workload_rows(wl, split_kv=c["split_kv"], lib=lib)
        np.testing.assert_allclose(r["part_out"][0, :, 0], c["part_out"], rtol=0, atol=1e-12, err_msg=c["name"])
        want_lse = np.array([_num(x) for x in c["part_lse"]])
        got_lse = r["part_lse"][0]
        assert np.array_equal(np.isinf(got_lse), np.isinf(want_lse)), (c["name"], got_lse)
        fin = np.isfinite(want_lse)
        np.testing.assert_allclose(got_lse[fin], want_lse[fin], rtol=0, atol=1e-12, err_msg=c["name"])
        np.testing.assert_allclose(r["comb_out"][0, 0], c["out"], rtol=0, atol=1e-12, err_msg=c["name"])
        np.testing.assert_allclose(r["comb_lse"][0], c["lse"], rtol=0, atol=1e-12, err_msg=c["name"])


def pin_golden_combine(lib):
    g = _golden("worked_attention.json")
    for c in g["combine_cases"]:
        po = np.asarray(c["part_out"], dtype=np.float64).reshape(1, -1, 1)
        pl = np.asarray([_num(x) for x in c["part_lse"]]).reshape(1, -1)
        out, lse = oracle.combine(po, pl, lib=lib)
        assert np.isfinite(out).all(), c["name"]
        np.testing.assert_allclose(out[0, 0], _num(c["out"]), rtol=0, atol=1e-12, err_msg=c["name"])
        want = _num(c["lse"])
        if math.isinf(want):
            assert lse[0] == want, (c["name"], lse[0])
        else:
            np.testing.assert_allclose(lse[0], want, rtol=0, atol=1e-12, err_msg=c["name"])


# ----------------------------------------------------------------------------- brute force
def _small_prefill():
    return W.make_custom(name="small_prefill", dtype="bf16", B=2, Sq=8, Hq=8, Hkv=2, D=16, page_size=4,
                         seq_lens=[23, 40], causal=True, q_offset=[15, 27], num_pages=24, W=12, seed=77)


def _small_gqa_f16():
    return W.make_custom(name="small_gqa_f16", dtype="f16", B=3, Sq=2, Hq=6, Hkv=3, D=8, page_size=4,
                         seq_lens=[9, 1, 16], causal=False, num_pages=10, W=5, seed=78)


def pin_bruteforce(lib):
    """Oracle agrees with dense numpy float64 attention on logically ordered K/V (1e-12)."""
    for wl in (W.tiny_decode_f32(), _small_prefill(), _small_gqa_f16()):
        ref_out, ref_lse = bf.attention(wl)
        r = oracle.workload_rows(wl, split_kv=1, lib=lib, want_split=False)
        got = r["out"].reshape(wl.B, wl.Sq, wl.Hq, wl.D)
        np.testing.assert_allclose(got, ref_out, rtol=1e-12, atol=1e-12, err_msg=wl.name)
        np.testing.assert_allclose(r["lse"].reshape(wl.B, wl.Sq, wl.Hq), ref_lse, rtol=1e-12, atol=1e-12,
                                   err_msg=wl.name)


# ----------------------------------------------------------------------------- invariants
def pin_shuffle_invariance(lib):
    """Shuffling the physical page order leaves the result bit-identical (PR #2222 Key Changes 2)."""
    base = W.make_custom(name="contig", dtype="bf16", B=3, Sq=2, Hq=4, Hkv=2, D=16, page_size=4,
                         seq_lens=[13, 4, 21], num_pages=16, W=6, seed=5, shuffle=False, causal=True)
    rng = np.random.default_rng(9)
    perm = rng.permutation(base.num_pages)          # physical slot of logical page p is perm[p]
    k2 = np.empty_like(base.k_cache)
    v2 = np.empty_like(base.v_cache)
    k2[perm] = base.k_cache
    v2[perm] = base.v_cache
    bt2 = base.block_table.copy()
    nb = base.nblk()
    for b in range(base.B):
        bt2[b, :nb[b]] = perm[base.block_table[b, :nb[b]]]
    assert not np.array_equal(bt2, base.block_table)
    r1 = oracle.workload_rows(base, split_kv=3, lib=lib)
    shuf = W.Workload(**{**base.__dict__, "block_table": bt2, "k_cache": k2, "v_cache": v2})
    r2 = oracle.workload_rows(shuf, split_kv=3, lib=lib)
    for key in r1:
        assert np.array_equal(r1[key], r2[key]), key


def pin_gather_matches_fancy_index(lib):
    """Logical gather equals numpy fancy indexing of the pool, bit for bit, all dtypes."""
    for dt in ("f32", "bf16", "f16"):
        wl = W.make_custom(dtype=dt, B=3, Sq=1, Hq=4, Hkv=2, D=8, page_size=4, seq_lens=[7, 12, 1],
                           num_pages=9, W=4, seed=11)
        d = oracle.dims_of(wl)
        for b in range(wl.B):
            L = int(wl.seq_lens[b])
            got = oracle.gather(wl.k_cache, wl.block_table, wl.seq_lens, d, b, lib=lib)
            want = bf.logical_kv(wl.k_cache, wl.block_table[b], L, wl.page_size, dt)
            assert np.array_equal(got, want), (dt, b)


def pin_widening_special_values(lib):
    """bf16/f16 widening is exact on subnormals, signed zeros, extremes (format definitions)."""
    bits_f16 = np.array([0x0001, 0x03FF, 0x0400, 0x3C00, 0x7BFF, 0x8001, 0x8000, 0xC000, 0x3555, 0x0200],
                        dtype=np.uint16)
    bits_bf16 = np.array([0x0001, 0x007F, 0x0080, 0x3F80, 0x7F7F, 0x8001, 0x8000, 0xC000, 0x3EAB, 0x4049],
                         dtype=np.uint16)
    for dt, bits, want in (("f16", bits_f16, bits_f16.view(np.float16).astype(np.float64)),
                           ("bf16", bits_bf16,
                            (bits_bf16.astype(np.uint32) << 16).view(np.float32).astype(np.float64))):
        cache = bits.reshape(len(bits), 1, 1, 1)
        bt = np.arange(len(bits), dtype=np.int32).reshape(1, -1)
        d = oracle.make_dims(B=1, Sq=1, Hq=1, Hkv=1, D=1, page_size=1, bt_stride=len(bits), dtype=dt,
                             num_pages=len(bits))
        got = oracle.gather(cache, bt, np.array([len(bits)], dtype=np.int32), d, 0, lib=lib)[:, 0, 0]
        assert np.array_equal(got, want), (dt, got, want)
        assert np.array_equal(np.signbit(got), np.signbit(want)), dt


def pin_single_key_exact(lib):
    """One valid key returns exactly its V row (L=1, and causal row 0 with q_offset 0)."""
    wl = W.make_custom(dtype="bf16", B=2, Sq=3, Hq=4, Hkv=2, D=16, page_size=4, seq_lens=[1, 9],
                       causal=True, q_offset=[-2, 0], num_pages=4, W=3, seed=21)
    r = oracle.workload_rows(wl, split_kv=2, lib=lib)
    G = wl.G
    rows = oracle.all_rows(wl.B, wl.Sq, wl.Hq)
    out = r["out"]
    for n, (b, i, h) in enumerate(rows):
        lim = min(int(wl.seq_lens[b]), max(int(wl.q_offset[b]) + i + 1, 0))
        if lim == 1:
            page = wl.block_table[b, 0]
            v0 = bf.widen(wl.v_cache[page, 0, h // G], "bf16")
            assert np.array_equal(out[n], v0), (b, i, h)
            assert np.array_equal(r["comb_out"][n], v0), (b, i, h)
    # b=0 (L=1): every row sees key 0 only when its reach is >= 1 (row 2: reach 1)
    assert np.array_equal(out[(0 * 3 + 2) * 4 + 1], bf.widen(wl.v_cache[wl.block_table[0, 0], 0, 0], "bf16"))


def pin_equal_scores_mean(lib):
    """q = 0 makes every score equal: out is the mean of the valid V rows and lse = ln(count)."""
    wl = W.make_custom(dtype="f32", B=2, Sq=2, Hq=2, Hkv=1, D=8, page_size=4, seq_lens=[10, 3],
                       causal=True, q_offset=[5, 0], num_pages=4, W=3, seed=31, zero_q=True)
    r = oracle.workload_rows(wl, split_kv=1, lib=lib, want_split=False)
    rows = oracle.all_rows(wl.B, wl.Sq, wl.Hq)
    for n, (b, i, h) in enumerate(rows):
        lim = min(int(wl.seq_lens[b]), int(wl.q_offset[b]) + i + 1)
        V = bf.logical_kv(wl.v_cache, wl.block_table[b], lim, wl.page_size, "f32")[:, 0]
        np.testing.assert_allclose(r["out"][n], V.mean(axis=0), rtol=1e-14, atol=1e-15)
        np.testing.assert_allclose(r["lse"][n], math.log(lim), rtol=0, atol=1e-14)


def pin_two_key_closed_form(lib):
    """D=1, two keys: out = v2 + (v1 - v2) * sigmoid(s1 - s2); lse = log(e^s1 + e^s2)."""
    rng = np.random.default_rng(41)
    for _ in range(5):
        kq = rng.standard_normal(3).astype(np.float32)
        v = rng.standard_normal(2).astype(np.float32)
        k = np.array([kq[0], kq[1]], dtype=np.float32).reshape(2, 1, 1, 1)
        wl = W.Workload(name="two", dtype="f32", B=1, Sq=1, Hq=1, Hkv=1, D=1, page_size=1, num_pages=2,
                        causal=False, scale=0.7, split_kv=(1,), seq_lens=np.array([2], dtype=np.int32),
                        block_table=np.array([[1, 0]], dtype=np.int32), q=np.array(kq[2]).reshape(1, 1, 1, 1),
                        k_cache=k, v_cache=v.reshape(2, 1, 1, 1))
        s1 = 0.7 * float(kq[2]) * float(kq[1])      # logical key 0 is physical page 1
        s2 = 0.7 * float(kq[2]) * float(kq[0])
        v1, v2 = float(v[1]), float(v[0])
        want = v2 + (v1 - v2) / (1.0 + math.exp(-(s1 - s2)))
        r = oracle.workload_rows(wl, split_kv=2, lib=lib)
        np.testing.assert_allclose(r["out"][0, 0], want, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(r["lse"][0], max(s1, s2) + math.log1p(math.exp(-abs(s1 - s2))), rtol=1e-13,
                                   atol=1e-15)
        np.testing.assert_allclose(r["comb_out"][0, 0], want, rtol=1e-13, atol=1e-15)


def pin_split_equals_unsplit(lib):
    """Every split count, including S > nblk, combines back to the unsplit softmax (1e-12)."""
    wl = _small_prefill()
    for S in (1, 2, 4, 8, 64):
        r = oracle.workload_rows(wl, split_kv=S, lib=lib)
        np.testing.assert_allclose(r["comb_out"], r["out"], rtol=1e-12, atol=1e-12, err_msg=f"S={S}")
        fin = np.isfinite(r["lse"])
        assert np.array_equal(fin, np.isfinite(r["comb_lse"])), S
        np.testing.assert_allclose(r["comb_lse"][fin], r["lse"][fin], rtol=1e-12, atol=1e-12, err_msg=f"S={S}")


def pin_empty_partitions(lib):
    """Empty or fully masked splits give (0, -inf); rows with no key give (0, -inf), never NaN."""
    wl = W.make_custom(dtype="bf16", B=3, Sq=4, Hq=2, Hkv=1, D=8, page_size=4, seq_lens=[17, 0, 6],
                       causal=True, q_offset=[-3, 0, 0], num_pages=7, W=5, seed=51)
    S = 8
    r = oracle.workload_rows(wl, split_kv=S, lib=lib)
    for key in r:
        assert not np.isnan(r[key]).any(), key
    plan = oracle.plan(wl.seq_lens, wl.page_size, S, lib=lib)
    rows = oracle.all_rows(wl.B, wl.Sq, wl.Hq)
    for n, (b, i, h) in enumerate(rows):
        L = int(wl.seq_lens[b])
        lim = min(L, max(int(wl.q_offset[b]) + i + 1, 0))
        for s in range(S):
            lo = plan[b, s, 0] * wl.page_size
            hi = min(plan[b, s, 1] * wl.page_size, L, lim)
            if hi <= lo:
                assert r["part_lse"][n, s] == -np.inf, (b, i, h, s)
                assert np.array_equal(r["part_out"][n, s], np.zeros(wl.D)), (b, i, h, s)
        if lim == 0:
            assert r["lse"][n] == -np.inf and r["comb_lse"][n] == -np.inf
            assert not r["out"][n].any() and not r["comb_out"][n].any()
    # sequence 0 has nblk 5: splits 5..7 are empty under the clamp
    assert (plan[0, 5:] == 5).all()


def pin_mask_counts(lib):
    """Valid keys per row = min(L_b, q_offset_b + i + 1) by brute-force counting (causal), L_b otherwise."""
    wl = W.make_custom(dtype="f32", B=3, Sq=5, Hq=1, Hkv=1, D=1, page_size=4, seq_lens=[12, 5, 9],
                       causal=True, q_offset=[7, -2, 4], num_pages=8, W=3, seed=61)
    d = oracle.dims_of(wl)
    for causal in (True, False):
        for b in range(wl.B):
            for i in range(wl.Sq):
                L = int(wl.seq_lens[b])
                count = sum(1 for j in range(L) if (not causal) or j <= int(wl.q_offset[b]) + i)
                assert oracle.key_limit(wl.seq_lens, wl.q_offset, causal, d, b, i, lib=lib) == count
        # default offset: q_offset = L - Sq
        for b in range(wl.B):
            for i in range(wl.Sq):
                L = int(wl.seq_lens[b])
                count = sum(1 for j in range(L) if (not causal) or j <= L - wl.Sq + i)
                assert oracle.key_limit(wl.seq_lens, None, causal, d, b, i, lib=lib) == count


def pin_gqa_head_sharing(lib):
    """Query heads of one group (h // G equal) with equal q give identical rows; other groups differ."""
    wl = W.make_custom(dtype="f32", B=1, Sq=1, Hq=6, Hkv=3, D=4, page_size=2, seq_lens=[5], num_pages=3,
                       W=3, seed=71)
    q = wl.q.copy()
    q[0, 0, :] = q[0, 0, 0]
    wl2 = W.Workload(**{**wl.__dict__, "q": q})
    r = oracle.workload_rows(wl2, split_kv=1, lib=lib, want_split=False)["out"]
    for h in range(0, 6, 2):
        assert np.array_equal(r[h], r[h + 1]), h
    assert not np.allclose(r[0], r[2]) and not np.allclose(r[2], r[4])


def pin_rejects_bad_page(lib):
    """A page id inside the sequence's pages that is not a pool page is an error, not a read."""
    wl = W.make_custom(dtype="f32", B=1, Sq=1, Hq=1, Hkv=1, D=2, page_size=2, seq_lens=[3], num_pages=2,
                       W=3, seed=81)
    bt = wl.block_table.copy()
    bt[0, 1] = 2
    # the pool is a view of a larger buffer, so a build that skips the check reads owned memory
    kbig = np.concatenate([wl.k_cache, wl.k_cache])
    vbig = np.concatenate([wl.v_cache, wl.v_cache])
    bad = W.Workload(**{**wl.__dict__, "block_table": bt, "k_cache": kbig[:2], "v_cache": vbig[:2]})
    try:
        oracle.workload_rows(bad, lib=lib)
    except ValueError:
        return
    raise AssertionError("out-of-pool page id was accepted")


# ----------------------------------------------------------------------------- quantized pools
def pin_e4m3_all_codes(lib):
    """Every FP8 E4M3 code decodes as the format defines (library cast for reference; hand-checked
    anchors: 0x38 = 1, 0x7E = 448, 0x08 = 2^-6, 0x01 = 2^-9, 0xB8 = -1, 0x80 = -0, 0x7F = NaN)."""
    codes = np.arange(256, dtype=np.uint8)
    d = oracle.make_dims(B=1, Sq=1, Hq=1, Hkv=1, D=1, page_size=1, bt_stride=256, dtype="bf16", num_pages=256)
    got = oracle.gather_kvq(codes.reshape(256, 1, 1, 1), np.ones((256, 1), np.float32),
                            np.arange(256, dtype=np.int32).reshape(1, -1), np.array([256], dtype=np.int32), d, 0,
                            lib=lib)[:, 0, 0]
    want = W.e4m3_bits_to_float(codes)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan]) and np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))
    for code, val in ((0x38, 1.0), (0x7E, 448.0), (0x08, 2.0 ** -6), (0x01, 2.0 ** -9), (0xB8, -1.0)):
        assert got[code] == val, (hex(code), got[code])
    assert got[0x80] == 0.0 and np.signbit(got[0x80]) and np.isnan(got[0x7F]) and np.isnan(got[0xFF])


def _fp8_small(seed=91, **kw):
    base = dict(B=3, Sq=2, Hq=8, Hkv=2, D=16, page_size=4, seq_lens=[13, 4, 21], num_pages=16, W=6,
                causal=True, seed=seed)
    base.update(kw)
    return W.make_custom_fp8(**base)


def pin_kvq_unit_scale_equals_unquantized(lib):
    """With every scale 1, quantized pools give bit-identical results to bf16 pools holding the same
    (exactly representable) values."""
    wl = _fp8_small()
    ones = np.ones_like(wl.k_scale)
    rq = oracle.workload_rows_kvq(wl, split_kv=3, k_scale=ones, v_scale=ones, lib=lib)
    kb = W.bf16_bits_rne(W.e4m3_bits_to_float(wl.k_cache).astype(np.float32))
    vb = W.bf16_bits_rne(W.e4m3_bits_to_float(wl.v_cache).astype(np.float32))
    plain = W.Workload(**{**wl.__dict__, "k_cache": kb, "v_cache": vb, "kv_dtype": None})
    rp = oracle.workload_rows(plain, split_kv=3, lib=lib)
    for key in rq:
        assert np.array_equal(rq[key], rp[key]), key


def pin_kvq_bruteforce(lib):
    """Quantized pools with per-(page, kv head) scales on shuffled pages agree with dense fp64
    attention on the dequantized pools (1e-12)."""
    for wl in (_fp8_small(), _fp8_small(seed=92, B=2, Sq=1, Hq=6, Hkv=3, D=8, seq_lens=[9, 16], causal=False,
                                         num_pages=7, W=4)):
        kd = W.e4m3_bits_to_float(wl.k_cache) * wl.k_scale[:, None, :, None].astype(np.float64)
        vd = W.e4m3_bits_to_float(wl.v_cache) * wl.v_scale[:, None, :, None].astype(np.float64)
        ref_out, ref_lse = bf.attention(wl, k_cache=kd, v_cache=vd, kv_dtype="f64")
        r = oracle.workload_rows_kvq(wl, split_kv=1, want_split=False, lib=lib)
        np.testing.assert_allclose(r["out"].reshape(ref_out.shape), ref_out, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(r["lse"].reshape(ref_lse.shape), ref_lse, rtol=1e-12, atol=1e-12)
        assert len(np.unique(wl.k_scale)) > 4


def pin_kvq_power_of_two_scales(lib):
    """Power-of-two scales are exact: quantized results equal those of f32 pools holding value x scale."""
    wl = _fp8_small(seed=93)
    rng = np.random.default_rng(94)
    ks = (2.0 ** rng.integers(-6, 7, size=wl.k_scale.shape)).astype(np.float32)
    vs = (2.0 ** rng.integers(-6, 7, size=wl.v_scale.shape)).astype(np.float32)
    rq = oracle.workload_rows_kvq(wl, split_kv=2, k_scale=ks, v_scale=vs, lib=lib)
    kf = (W.e4m3_bits_to_float(wl.k_cache) * ks[:, None, :, None]).astype(np.float32)
    vf = (W.e4m3_bits_to_float(wl.v_cache) * vs[:, None, :, None]).astype(np.float32)
    qf = bf.widen(wl.q, wl.dtype).astype(np.float32)
    plain = W.Workload(**{**wl.__dict__, "dtype": "f32", "q": qf, "k_cache": kf, "v_cache": vf, "kv_dtype": None})
    rp = oracle.workload_rows(plain, split_kv=2, lib=lib)
    for key in rq:
        assert np.array_equal(rq[key], rp[key]), key


def pin_int8_all_codes(lib):
    """Every int8 code decodes as two's complement (numpy's reinterpretation for reference;
    hand-checked anchors: 0x00 = 0, 0x01 = 1, 0x7F = 127, 0x80 = -128, 0x81 = -127, 0xFF = -1)."""
    codes = np.arange(256, dtype=np.uint8)
    d = oracle.make_dims(B=1, Sq=1, Hq=1, Hkv=1, D=1, page_size=1, bt_stride=256, dtype="bf16", num_pages=256)
    got = oracle.gather_kvq(codes.reshape(256, 1, 1, 1), np.ones((256, 1), np.float32),
                            np.arange(256, dtype=np.int32).reshape(1, -1), np.array([256], dtype=np.int32), d, 0,
                            lib=lib, kv_dtype="int8")[:, 0, 0]
    assert np.array_equal(got, W.int8_bits_to_float(codes))
    for code, val in ((0x00, 0.0), (0x01, 1.0), (0x7F, 127.0), (0x80, -128.0), (0x81, -127.0), (0xFF, -1.0)):
        assert got[code] == val, (hex(code), got[code])


def _int8_small(seed=95, **kw):
    base = dict(B=3, Sq=2, Hq=8, Hkv=2, D=16, page_size=4, seq_lens=[13, 4, 21], num_pages=16, W=6,
                causal=True, seed=seed)
    base.update(kw)
    return W.make_custom_int8(**base)


def pin_int8_power_of_two_scales_equal_unquantized(lib):
    """int8 pools with power-of-two scales give bit-identical results to bf16 pools holding
    element x scale (every such value is a bf16 number: at most 8 significant bits)."""
    wl = _int8_small()
    rng = np.random.default_rng(96)
    ks = (2.0 ** rng.integers(-6, 7, size=wl.k_scale.shape)).astype(np.float32)
    vs = (2.0 ** rng.integers(-6, 7, size=wl.v_scale.shape)).astype(np.float32)
    rq = oracle.workload_rows_kvq(wl, split_kv=3, k_scale=ks, v_scale=vs, lib=lib)
    kb = W.bf16_bits_rne((W.int8_bits_to_float(wl.k_cache) * ks[:, None, :, None]).astype(np.float32))
    vb = W.bf16_bits_rne((W.int8_bits_to_float(wl.v_cache) * vs[:, None, :, None]).astype(np.float32))
    assert np.array_equal(bf.widen(kb, "bf16"), W.int8_bits_to_float(wl.k_cache) * ks[:, None, :, None])
    assert (W.int8_bits_to_float(wl.k_cache) < 0).any() and (W.int8_bits_to_float(wl.v_cache) < 0).any()
    plain = W.Workload(**{**wl.__dict__, "k_cache": kb, "v_cache": vb, "kv_dtype": None})
    rp = oracle.workload_rows(plain, split_kv=3, lib=lib)
    for key in rq:
        assert np.array_equal(rq[key], rp[key]), key


def pin_int8_bruteforce(lib):
    """int8 pools with per-(page, kv head) scales on shuffled pages agree with dense fp64 attention
    on the dequantized pools (1e-12)."""
    for wl in (_int8_small(), _int8_small(seed=97, B=2, Sq=1, Hq=6, Hkv=3, D=8, seq_lens=[9, 16], causal=False,
                                          num_pages=7, W=4)):
        kd = W.int8_bits_to_float(wl.k_cache) * wl.k_scale[:, None, :, None].astype(np.float64)
        vd = W.int8_bits_to_float(wl.v_cache) * wl.v_scale[:, None, :, None].astype(np.float64)
        ref_out, ref_lse = bf.attention(wl, k_cache=kd, v_cache=vd, kv_dtype="f64")
        r = oracle.workload_rows_kvq(wl, split_kv=1, want_split=False, lib=lib)
        np.testing.assert_allclose(r["out"].reshape(ref_out.shape), ref_out, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(r["lse"].reshape(ref_lse.shape), ref_lse, rtol=1e-12, atol=1e-12)
        assert len(np.unique(wl.k_scale)) > 4


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
