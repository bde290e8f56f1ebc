"""GPU parity of the variable-length entry point (decode and prefill sequences in one call) against
the oracle's variable-length evaluation (each sequence as a batch of one).

Bars as everywhere: bf16/f16 atol=2e-3, rtol=2^-8, -inf patterns exact, no NaN.  On a batch whose
sequences all have the same query count, the variable-length call runs the same per-unit code as
the uniform entry point's kernel for that shape (the tcgen05 kernel for 64 rows or more, the
tensor-core decode units below), so the two agree bit for bit.
"""
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


def _device(wl, k=None, v=None):
    import torch
    dw = _gpu.DeviceWorkload(wl) if k is None else None
    d = {"q": W.host_to_torch(wl.q, wl.dtype).cuda(),
         "k": dw.k if dw else k, "v": dw.v if dw else v,
         "bt": torch.from_numpy(np.ascontiguousarray(wl.block_table)).cuda(),
         "sl": torch.from_numpy(np.ascontiguousarray(wl.seq_lens)).cuda(),
         "qs": torch.from_numpy(np.ascontiguousarray(wl.q_start)).cuda(),
         "qo": None if wl.q_offset is None else torch.from_numpy(np.ascontiguousarray(wl.q_offset)).cuda()}
    return d


def _run(pa, wl, d, S, hint=None):
    """Returns float64 numpy out [T, Hq, D], lse [T, Hq] (+ part_out / part_lse for S > 1).  With
    ``hint`` the call is the overlapped one."""
    import torch
    T, Hq, D = wl.Sq, wl.Hq, wl.D
    res = {}
    if S == 1:
        out = torch.empty_like(d["q"])
        lse = torch.empty((T, Hq), dtype=torch.float32, device="cuda")
        pa.paged_attn_fwd_varlen(d["q"], d["k"], d["v"], d["bt"], d["sl"], d["qs"], wl.causal, d["qo"], 1, wl.scale,
                                 out, lse, hint=hint)
    else:
        po = torch.empty((S, T, Hq, D), dtype=torch.float32, device="cuda")
        pl = torch.empty((S, T, Hq), dtype=torch.float32, device="cuda")
        pa.paged_attn_fwd_varlen(d["q"], d["k"], d["v"], d["bt"], d["sl"], d["qs"], wl.causal, d["qo"], S, wl.scale,
                                 po, pl, hint=hint)
        out = torch.empty_like(d["q"])
        lse = torch.empty((T, Hq), dtype=torch.float32, device="cuda")
        pa.paged_attn_combine(po, pl, out, lse)
        res["part_out"], res["part_lse"] = _gpu.to_f64(po, "f32"), _gpu.to_f64(pl, "f32")
    torch.cuda.synchronize()
    res["out"], res["lse"] = _gpu.to_f64(out, wl.dtype), _gpu.to_f64(lse, "f32")
    return res


def _oracle(wl, S, k=None, v=None):
    dims = oracle.make_dims(B=wl.B, Sq=wl.Sq, Hq=wl.Hq, Hkv=wl.Hkv, D=wl.D, page_size=wl.page_size,
                            bt_stride=int(wl.block_table.shape[1]), dtype=wl.dtype, num_pages=wl.num_pages)
    return oracle.rows_varlen(q=wl.q, k_cache=wl.k_cache if k is None else k, v_cache=wl.v_cache if v is None else v,
                              block_table=wl.block_table, seq_lens=wl.seq_lens, q_start=wl.q_start,
                              q_offset=wl.q_offset, causal=wl.causal, dims=dims, scale=wl.scale, split_kv=S)


def _compare(res, ref, wl, S, what, rows=None):
    sel = slice(None) if rows is None else rows
    dt = wl.dtype
    if S == 1:
        _gpu.assert_close(res["out"][sel], ref["out"][sel], dt, f"{what} out")
        _gpu.assert_close(res["lse"][sel], ref["lse"][sel], dt, f"{what} lse")
    else:
        _gpu.assert_close(res["out"][sel], ref["comb_out"][sel], dt, f"{what} combined out")
        _gpu.assert_close(res["lse"][sel], ref["comb_lse"][sel], dt, f"{what} combined lse")
        _gpu.assert_close(res["part_out"][:, sel], ref["part_out"][:, sel], dt, f"{what} partial out")
        _gpu.assert_close(res["part_lse"][:, sel], ref["part_lse"][:, sel], dt, f"{what} partial lse")


# ----------------------------------------------------------------------------- mixed small batches
MIXED = dict(q_lens=[1, 0, 4, 1, 40, 3, 17, 1, 100], seq_lens=[300, 50, 4, 1000, 600, 70, 17, 1, 333])


@pytest.mark.parametrize("dtype,D,Hq,Hkv", [("bf16", 128, 32, 8), ("f16", 64, 16, 2), ("bf16", 128, 16, 16)])
@pytest.mark.parametrize("S", [1, 3])
def test_mixed_batch(pa, dtype, D, Hq, Hkv, S):
    """Decode sequences (1-4 tokens), empty ones and prefill chunks (17-100 tokens) in one call,
    causal with the default offsets (queries are each sequence's newest tokens)."""
    wl = W.make_varlen(dtype=dtype, Hq=Hq, Hkv=Hkv, D=D, page_size=16, seed=40 + D + Hq, **MIXED)
    res = _run(pa, wl, _device(wl), S)
    ref = _oracle(wl, S)
    _compare(res, ref, wl, S, f"mixed {dtype} D={D} G={Hq // Hkv} S={S}")
    assert pa.paged_attn_last_error_word() == 0


def test_mixed_batch_offsets_and_noncausal(pa):
    """Explicit offsets (one hides every key from the first rows) and a non-causal batch."""
    qo = [299, 10, 0, 999, -3, 67, 0, 0, 200]
    wl = W.make_varlen(dtype="bf16", Hq=32, Hkv=8, D=128, page_size=32, q_offset=qo, seed=77, **MIXED)
    res = _run(pa, wl, _device(wl), 2)
    ref = _oracle(wl, 2)
    _compare(res, ref, wl, 2, "offsets")
    a = int(wl.q_start[4])
    assert np.isneginf(res["lse"][a:a + 3]).all()  # reach <= 0 for the first 3 rows of sequence 4
    wl2 = W.Workload(**{**wl.__dict__, "causal": False, "q_offset": None})
    res = _run(pa, wl2, _device(wl2), 1)
    _compare(res, _oracle(wl2, 1), wl2, 1, "non-causal")
    assert pa.paged_attn_last_error_word() == 0


@pytest.mark.parametrize("q_len,variant", [(1, 2), (3, 2), (37, 4)])
def test_uniform_batch_bit_identical(pa, q_len, variant):
    """Every sequence with the same query count: the variable-length launch equals the uniform
    kernel bit for bit (16-row decode units for 4-12 rows; the tcgen05 kernel's 128-row tiles for
    148 rows, whose last tile runs past each sequence)."""
    import torch
    wl = W.make_custom(dtype="bf16", B=5, Sq=q_len, Hq=32, Hkv=8, D=128, page_size=16,
                       seq_lens=[64, 200, 500, 37, 1000], causal=True, seed=9)
    dw = _gpu.DeviceWorkload(wl)
    want = _gpu.run(dw, 2, variant=variant)
    T = wl.B * q_len
    packed = W.Workload(**{**wl.__dict__, "Sq": T, "q": wl.q.reshape(T, wl.Hq, wl.D),
                           "q_start": np.arange(0, T + 1, q_len, dtype=np.int32)})
    got = _run(pa, packed, _device(packed, dw.k, dw.v), 2)
    assert np.array_equal(got["out"], want["out"].reshape(T, wl.Hq, wl.D))
    assert np.array_equal(got["lse"], want["lse"].reshape(T, wl.Hq))
    # partial rows with lse -inf need not be written (the combine never reads them)
    keep = ~np.isneginf(want["part_lse"].reshape(2, T, wl.Hq))
    assert np.array_equal(got["part_lse"], want["part_lse"].reshape(2, T, wl.Hq))
    assert np.array_equal(got["part_out"][keep], want["part_out"].reshape(2, T, wl.Hq, wl.D)[keep])
    del torch


@pytest.mark.parametrize("D,q_lens", [(64, [2, 3, 4]), (128, [20, 30, 40])])
def test_bad_q_start_is_reported(pa, D, q_lens):
    """A q_start entry past the packed tokens: that sequence is skipped (its rows untouched), the
    others are exact, and the error word says so (short sequences: one-grid kernel; 80-160 rows at
    head dim 128: tcgen05 kernel)."""
    import torch
    wl = W.make_varlen(dtype="bf16", Hq=8, Hkv=2, D=D, page_size=16, seed=3, q_lens=q_lens,
                       seq_lens=[q + 40 for q in q_lens])
    d = _device(wl)
    bad = d["qs"].clone()
    bad[2] = 1000  # sequence 1 ends, and sequence 2 starts, past T
    out = torch.full_like(d["q"], 7.0)
    lse = torch.empty((wl.Sq, wl.Hq), dtype=torch.float32, device="cuda")
    pa.paged_attn_fwd_varlen(d["q"], d["k"], d["v"], d["bt"], d["sl"], bad, True, None, 1, wl.scale, out, lse)
    torch.cuda.synchronize()
    assert pa.paged_attn_last_error_word() & pa.ERRBIT_QSTART
    ref = _oracle(wl, 1)
    got = _gpu.to_f64(out, "bf16")
    q0 = q_lens[0]
    _gpu.assert_close(got[0:q0], ref["out"][0:q0], "bf16", "sequence 0")
    assert np.all(got[q0:] == 7.0)


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (16, 16), (64, 4)])
@pytest.mark.parametrize("S", [1, 3])
def test_long_sequences_on_tcgen05(pa, Hq, Hkv, S):
    """Head dim 128, bf16: sequences of at least 64 query rows run on the tcgen05 kernel, the rest on
    the one-grid kernel.  Row counts on both sides of 64, last tiles that end inside an epilogue
    warp's rows (those rows are stored one per lane), sequences spanning several tiles, an empty
    sequence, explicit offsets that hide every key from the first rows of one sequence."""
    G = Hq // Hkv
    q_lens = [64 // G, 64 // G - 1, 1, 0, 333 // G + 5, 129, 5, 2 * (128 // G) + 1]
    qo = [40, 7, 300, 0, -3, 500, 12, 64]
    seq_lens = [max(o, 0) + q for o, q in zip(qo, q_lens)]
    wl = W.make_varlen(dtype="bf16", Hq=Hq, Hkv=Hkv, D=128, page_size=16, q_offset=qo, seed=90 + G + S,
                       q_lens=q_lens, seq_lens=seq_lens)
    res = _run(pa, wl, _device(wl), S)
    ref = _oracle(wl, S)
    _compare(res, ref, wl, S, f"tcgen05 varlen G={G} S={S}")
    assert pa.paged_attn_last_error_word() == 0


# ----------------------------------------------------------------------------- overlapped call
def _hint(pa, wl, kind):
    h = pa.paged_attn_varlen_hint(wl.q_start, wl.seq_lens, wl.q_offset, wl.causal, wl.Hq, wl.Hkv, wl.D,
                                  pa.PA_BF16 if wl.dtype == "bf16" else pa.PA_F16)
    if kind == "long_heavy":    # the tcgen05 kernel gets its largest share of the SMs
        h.long_pairs *= 1000
    elif kind == "short_heavy":  # and its smallest
        h.short_kv_tokens *= 1000
    return h


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("S", [1, 3])
@pytest.mark.parametrize("kind", ["computed", "long_heavy", "short_heavy"])
def test_overlap_bit_identical(pa, dtype, S, kind):
    """paged_attn_fwd_varlen_overlap runs the tcgen05 kernel (long sequences) beside the one-grid
    kernel on a share of the SMs that the hint sets; a unit's work does not depend on the CTA or SM
    that takes it, so every output is bit-identical to paged_attn_fwd_varlen's, whatever the share."""
    rng = np.random.default_rng(7 + S)
    q_lens = [300, 1, 1, 200, 17, 0, 64, 3] + [1] * 40 + [130, 2]
    qo = [int(x) for x in rng.integers(0, 600, size=len(q_lens))]
    seq_lens = [o + q for o, q in zip(qo, q_lens)]
    wl = W.make_varlen(dtype=dtype, Hq=32, Hkv=8, D=128, page_size=16, q_offset=qo, seed=123 + S,
                       q_lens=q_lens, seq_lens=seq_lens)
    d = _device(wl)
    h = _hint(pa, wl, kind)
    assert h.long_pairs > 0 and h.short_kv_tokens > 0
    plain = _run(pa, wl, d, S)
    over = _run(pa, wl, d, S, hint=h)
    for key in plain:
        assert np.array_equal(plain[key], over[key], equal_nan=True), key
    if kind == "computed":
        _compare(over, _oracle(wl, S), wl, S, f"overlap {dtype} S={S}")
    assert pa.paged_attn_last_error_word() == 0


def test_overlap_falls_back_without_both_kinds(pa):
    """A hint with no short work (or a batch the tcgen05 kernel does not take) gives the plain call."""
    q_lens = [100, 90, 1]
    wl = W.make_varlen(dtype="bf16", Hq=32, Hkv=8, D=128, page_size=16, q_offset=[10, 0, 200], seed=5,
                       q_lens=q_lens, seq_lens=[110, 90, 201])
    d = _device(wl)
    plain = _run(pa, wl, d, 1)
    for h in (pa.PaVarlenHint(0, 0), pa.PaVarlenHint(10 ** 9, 0), pa.PaVarlenHint(0, 10 ** 9)):
        over = _run(pa, wl, d, 1, hint=h)
        for key in plain:
            assert np.array_equal(plain[key], over[key], equal_nan=True), key


# ----------------------------------------------------------------------------- full size
@pytest.fixture(scope="module")
def mixed_full():
    wl = W.mixed_decode_prefill()
    dw = _gpu.DeviceWorkload(W.Workload(**{**wl.__dict__, "q": wl.q[:1].reshape(1, 1, wl.Hq, wl.D)}))
    k, v = dw.host_pools()
    return wl, dw.k, dw.v, k, v


def test_mixed_decode_prefill_full(pa, mixed_full):
    """The benchmarked mixed batch (4 causal prefill chunks of 1024 tokens + 256 decode sequences of
    4096 keys, 2 x 2 GiB pools): every token and head against the oracle."""
    wl, kd, vd, k, v = mixed_full
    res = _run(pa, wl, _device(wl, kd, vd), 1)
    assert not np.isnan(res["out"]).any() and np.isfinite(res["lse"]).all()
    ref = oracle.rows_varlen(q=wl.q, k_cache=k, v_cache=v, block_table=wl.block_table, seq_lens=wl.seq_lens,
                             q_start=wl.q_start, q_offset=wl.q_offset, causal=wl.causal, dims=oracle.dims_of(wl),
                             scale=wl.scale, split_kv=1, want_split=False)
    _gpu.assert_close(res["out"], ref["out"], "bf16", "mixed full out")
    _gpu.assert_close(res["lse"], ref["lse"], "bf16", "mixed full lse")
    assert pa.paged_attn_last_error_word() == 0


def test_mixed_decode_prefill_full_overlap(pa, mixed_full):
    """The benchmarked mixed batch through the overlapped call: every output element equals the
    plain call's."""
    import torch
    wl, kd, vd, k, v = mixed_full
    d = _device(wl, kd, vd)
    h = _hint(pa, wl, "computed")
    outs = []
    for hint in (None, h):
        out = torch.empty_like(d["q"])
        lse = torch.empty((wl.Sq, wl.Hq), dtype=torch.float32, device="cuda")
        pa.paged_attn_fwd_varlen(d["q"], d["k"], d["v"], d["bt"], d["sl"], d["qs"], wl.causal, d["qo"], 1, wl.scale,
                                 out, lse, hint=hint)
        outs.append((out, lse))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    assert torch.equal(outs[0][1].view(torch.int32), outs[1][1].view(torch.int32))
    assert pa.paged_attn_last_error_word() == 0


def test_overlap_under_graph_capture(pa):
    """The overlapped call forks onto the library's stream and joins back, so it can be captured in a
    CUDA graph; replays give the plain call's outputs bit for bit."""
    import torch
    q_lens = [300, 1, 1, 200, 3] + [1] * 20
    qo = [50 * i for i in range(len(q_lens))]
    seq_lens = [o + q for o, q in zip(qo, q_lens)]
    wl = W.make_varlen(dtype="bf16", Hq=32, Hkv=8, D=128, page_size=16, q_offset=qo, seed=77, q_lens=q_lens,
                       seq_lens=seq_lens)
    d = _device(wl)
    h = _hint(pa, wl, "computed")
    T, Hq = wl.Sq, wl.Hq
    ref_out, ref_lse = torch.empty_like(d["q"]), torch.empty((T, Hq), dtype=torch.float32, device="cuda")
    pa.paged_attn_fwd_varlen(d["q"], d["k"], d["v"], d["bt"], d["sl"], d["qs"], wl.causal, d["qo"], 1, wl.scale,
                             ref_out, ref_lse)
    out, lse = torch.zeros_like(ref_out), torch.zeros_like(ref_lse)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up outside the capture (creates the library's stream)
        pa.paged_attn_fwd_varlen(d["q"], d["k"], d["v"], d["bt"], d["sl"], d["qs"], wl.causal, d["qo"], 1,
                                 wl.scale, out, lse, stream=s, hint=h)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    out.zero_()
    lse.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pa.paged_attn_fwd_varlen(d["q"], d["k"], d["v"], d["bt"], d["sl"], d["qs"], wl.causal, d["qo"], 1,
                                 wl.scale, out, lse, stream=torch.cuda.current_stream(), hint=h)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))
    assert pa.paged_attn_last_error_word() == 0


def test_batch_past_the_tcgen05_sequence_limit(pa):
    """More sequences than the tcgen05 variable-length kernel stages (1030 > 1024): every sequence,
    the long ones included, runs on the one-grid kernel, plain and with a hint (which then falls
    back), and matches the oracle on every row."""
    import torch
    rng = np.random.default_rng(7171)
    B = 1030
    q_lens = np.where(rng.random(B) < 0.01, 70, rng.integers(0, 3, size=B))
    seq_lens = q_lens + rng.integers(0, 120, size=B)
    wl = W.make_varlen(dtype="bf16", Hq=8, Hkv=2, D=128, page_size=16, seed=7172, q_lens=q_lens.tolist(),
                       seq_lens=seq_lens.tolist())
    assert (np.diff(wl.q_start) * wl.G >= 64).any()   # sequences the tcgen05 kernel would take below the limit
    d = _device(wl)
    ref = oracle.rows_varlen(q=wl.q, k_cache=wl.k_cache, v_cache=wl.v_cache, block_table=wl.block_table,
                             seq_lens=wl.seq_lens, q_start=wl.q_start, q_offset=wl.q_offset, causal=wl.causal,
                             dims=oracle.dims_of(wl), scale=wl.scale, split_kv=1, want_split=False)
    for kind in ("plain", "computed"):
        res = _run(pa, wl, d, 1, hint=None if kind == "plain" else _hint(pa, wl, "computed"))
        _gpu.assert_close(res["out"], ref["out"], "bf16", f"B=1030 {kind} out")
        _gpu.assert_close(res["lse"], ref["lse"], "bf16", f"B=1030 {kind} lse")
    assert pa.paged_attn_last_error_word() == 0
