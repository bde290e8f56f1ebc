"""Planted mistakes in the oracle must each fail at least one pin (CPU only).

Each mutation rewrites one line of a copy of the oracle source, builds it into a
temporary library and runs every pin against it.  A mutation that no pin catches
means the pins leave that part of the oracle unchecked.
"""
import os
import tempfile

import pytest

import oracle
from tests import _pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "paged_attn_oracle.c")

MUTATIONS = {
    # in-page offset loses the kv-head term (rocm-libraries PR #14349, Coverage)
    "drop_kv_head_term": ("return (tok * d->Hkv + kvh) * d->D + e;", "return (tok * d->Hkv + 0) * d->D + e;"),
    # wrong in-page row
    "wrong_in_page_row": ("int64_t tok = (int64_t)page * d->page_size + j % d->page_size;",
                          "int64_t tok = (int64_t)page * d->page_size + (j + 1) % d->page_size;"),
    # wrong table slot
    "wrong_table_slot": ("block_table[(int64_t)b * d->bt_stride + j / d->page_size]",
                         "block_table[(int64_t)b * d->bt_stride + (j / d->page_size) % 2]"),
    # GQA mapping interleaved instead of grouped
    "gqa_modulo": ("const int32_t kvh = h / G;", "const int32_t kvh = h % d->Hkv;"),
    # causal reach off by one
    "causal_off_by_one": ("int64_t reach = qoff + i + 1;", "int64_t reach = qoff + i;"),
    # default query offset off by one
    "default_offset": (": L - d->Sq;", ": L - d->Sq + 1;"),
    # truncating split division (rocMLIR PR #2371, the bug it fixes)
    "truncating_split": ("int64_t per = (nblk + split_kv - 1) / split_kv;", "int64_t per = nblk / split_kv;"),
    # end of a split not clamped
    "no_end_clamp": ("if (end > nblk) end = nblk;", "(void)0;"),
    # scale dropped
    "no_scale": ("s *= scale;", "s *= 1.0;"),
    # lse in the wrong base
    "lse_log2": ("*lse = m + log(l);", "*lse = m + log2(l);"),
    # max not subtracted in exp (output unchanged, lse wrong)
    "exp_without_max": ("double p = exp(scratch[j - lo] - m);", "double p = exp(scratch[j - lo]);"),
    # combine forgets to normalise
    "combine_no_normalise": ("        out[e] /= wsum;", "        out[e] /= 1.0;"),
    # combine -inf guard removed: all-empty rows become NaN
    "combine_no_guard": ("if (M == -INFINITY) {", "if (0) {"),
    # combine weights in the wrong sign
    "combine_weight_sign": ("double w = exp(part_lse[s] - M);", "double w = exp(M - part_lse[s]);"),
    # query read from the wrong head
    "q_wrong_head": ("* d->Hq + h) * D;", "* d->Hq + (d->Hq - 1 - h)) * D;"),
    # bf16 widening shifted by one bit
    "bf16_shift": ("uint32_t bits = (uint32_t)h << 16;", "uint32_t bits = (uint32_t)h << 15;"),
    # f16 subnormal exponent off by one
    "f16_subnormal": ("v = ldexp((double)m, -24);", "v = ldexp((double)m, -25);"),
    # split partial range starts at the split's end page
    "split_range_start": ("int64_t lo = (int64_t)plan[((int64_t)b * S + s) * 2 + 0] * d->page_size;",
                          "int64_t lo = (int64_t)plan[((int64_t)b * S + s) * 2 + 0] * d->page_size + 1;"),
    # quantized pools: scale looked up by logical page instead of the physical page
    "kvq_scale_logical_page": ("x *= (double)sc[(int64_t)table_page(d, block_table, b, j) * d->Hkv + kvh];",
                               "x *= (double)sc[(int64_t)(j / d->page_size) * d->Hkv + kvh];"),
    # quantized pools: K and V scales swapped
    "kvq_scales_swapped": ("const float *sc = which ? kv->v_scale : kv->k_scale;",
                           "const float *sc = which ? kv->k_scale : kv->v_scale;"),
    # E4M3 exponent bias off by one
    "e4m3_bias": ("v = ldexp((double)(8 + m), e - 10);", "v = ldexp((double)(8 + m), e - 11);"),
    # E4M3 subnormals scaled wrong
    "e4m3_subnormal": ("v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);"),
    # int8 read as unsigned
    "int8_unsigned": ("return (double)(h & 0x7F) - ((h & 0x80) ? 128.0 : 0.0);",
                      "return (double)(h & 0x7F) + ((h & 0x80) ? 128.0 : 0.0);"),
    # int8 read as sign-magnitude
    "int8_sign_magnitude": ("return (double)(h & 0x7F) - ((h & 0x80) ? 128.0 : 0.0);",
                            "return (h & 0x80) ? -(double)(h & 0x7F) : (double)(h & 0x7F);"),
    # int8 pools decoded as E4M3
    "int8_as_e4m3": ("return int8_bits_to_double(((const uint8_t *)base)[idx]);",
                     "return e4m3_bits_to_double(((const uint8_t *)base)[idx]);"),
    # page ids not range checked
    "no_page_range_check": ("if (page < 0 || (int64_t)page >= d->num_pages)", "if (page < 0)"),
}


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, source, tmp_path):
    old, new = MUTATIONS[name]
    assert source.count(old) == 1, f"mutation anchor not unique or missing: {old!r}"
    mutated = source.replace(old, new)
    src = tmp_path / "mutant.c"
    src.write_text(mutated)
    lib_path = str(tmp_path / "libmutant.so")
    oracle.build(src=str(src), out=lib_path)
    lib = oracle.load(lib_path, rebuild_if_stale=False)
    failures = []
    for pin in _pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError) as e:  # a pin failing, or the oracle rejecting input
            failures.append(pin.__name__)
    assert failures, f"mutation {name} passed every pin"
