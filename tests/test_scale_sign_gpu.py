"""scale multiplies q.k whatever its sign, and may be 0 (every weight equal): every kernel, chosen
by the planner or forced, against the oracle.  The tcgen05 prefill kernel takes its row maximum
over unscaled scores, which holds only for scale > 0, so the planner sends scale <= 0 to the
mma.sync prefill kernel and a forced tcgen05 call with it is refused."""
import pytest

import oracle
from paged_kv_cache_201_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu

SCALES = [0.0, -0.0884, -0.5]


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_201_gb300 as pa
    pa.load_library(build_if_missing=True)
    return pa


def _check(wl, split_kv, variant, what):
    dw = _gpu.DeviceWorkload(wl)
    res = _gpu.run(dw, split_kv, variant)
    rows = oracle.all_rows(wl.B, wl.Sq, wl.Hq)
    rows_fn = oracle.workload_rows_kvq if dw.kvq else oracle.workload_rows
    ref = rows_fn(wl, split_kv=split_kv, row_bih=rows)
    _gpu.compare_rows(res, ref, rows, wl, split_kv, what)


@pytest.mark.parametrize("scale", SCALES)
def test_prefill_scale_sign(pa, scale):
    qo = [3, 40]
    Sq = 80  # 320 rows per kv head: the planner's tcgen05 shape for scale > 0
    wl = W.make_custom(dtype="bf16", B=2, Sq=Sq, Hq=8, Hkv=2, D=128, page_size=16,
                       seq_lens=[o + Sq for o in qo], causal=True, q_offset=qo, scale=scale, seed=131)
    for S in (1, 3):
        for variant in (0, 1, 3):
            _check(wl, S, variant, f"prefill scale={scale} S={S} v={variant}")
    dw = _gpu.DeviceWorkload(wl)
    with pytest.raises(pa.PagedAttnError):
        _gpu.run(dw, 1, pa.VARIANT_TC05_PREFILL)
    assert pa.paged_attn_last_error_word() == 0


@pytest.mark.parametrize("scale", SCALES)
def test_decode_scale_sign(pa, scale):
    lens = [1, 37, 300]
    for name, kw, variants in [
        ("gqa4 D128", dict(Hq=8, Hkv=2, D=128), (0, 1, 2)),
        ("single head", dict(Hq=4, Hkv=4, D=128), (0, 1)),
        ("D256", dict(Hq=8, Hkv=2, D=256), (0, 1, 5)),
    ]:
        wl = W.make_custom(dtype="f16", B=len(lens), Sq=1, page_size=16, seq_lens=lens, scale=scale, seed=132, **kw)
        for S in (1, 2):
            for variant in variants:
                _check(wl, S, variant, f"{name} scale={scale} S={S} v={variant}")
    wl = W.make_custom_fp8(name="fp8 scale sign", dtype="bf16", B=len(lens), Sq=1, Hq=8, Hkv=2, D=128,
                           page_size=16, seq_lens=lens, scale=scale, seed=133)
    for S in (1, 2):
        _check(wl, S, 0, f"fp8 scale={scale} S={S}")
    assert pa.paged_attn_last_error_word() == 0
