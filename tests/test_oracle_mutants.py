"""Pin sensitivity: plant plausible mistakes in copies of the oracle (CPU only)
and check that the pins reject every one of them."""
import os
import subprocess

import numpy as np
import pytest

import oracle
from synth import F32, BF16
from tests._helpers import PagedCase, dense_causal_last_row, to_f64

SRC = os.path.join(os.path.dirname(oracle.__file__), "attention.c")

MUTANTS = {
    "scale_dropped": ("const double scale = 1.0 / sqrt((double)D);", "const double scale = 1.0;"),
    "scale_squared": ("const double scale = 1.0 / sqrt((double)D);", "const double scale = 1.0 / D;"),
    "new_key_excluded": ("seq_lens[b], qh / group,", "seq_lens[b] - 1 + (seq_lens[b] == 1), qh / group,"),
    "group_head_map": ("seq_lens[b], qh / group,", "seq_lens[b], qh % H,"),
    "window_start": ("const int64_t j0 = (window > 0 && t > window) ? t - window : 0;",
                     "const int64_t j0 = (window > 0 && t > window) ? t - window + 1 : 0;"),
    "slot_index": ("int64_t off = pool_offset(page, h, j % P, H, P, D);",
                   "int64_t off = pool_offset(page, h, (j + 1) % P, H, P, D);"),
    "page_index": ("int64_t page = table[j / P];\n        if", "int64_t page = table[j / (P + 1)];\n        if"),
    "k_for_v": ("mix += scores[j] * load_elem(v_pool,", "mix += scores[j] * load_elem(k_pool,"),
    "no_normalise": ("scores[j] /= sum;", "scores[j] /= 1.0;"),
    "no_max_shift_sign": ("scores[j] = exp(scores[j] - m);", "scores[j] = exp(m - scores[j]);"),
    "append_slot": ("pool_offset(page, h, pos % P, H, P, D);", "pool_offset(page, h, (pos + 1) % P, H, P, D);"),
    "first_table_row": ("tables + (int64_t)b * max_pages, seq_lens[b]", "tables, seq_lens[b]"),
    "layout_transposed": ("return ((page * H + head) * P + slot) * (int64_t)D;",
                          "return ((page * P + slot) * H + head) * (int64_t)D;"),
    "bf16_shift": ("<< 16;   /* bf16", "<< 15;   /* bf16"),
    "head_of_query": ("q + lane * D,", "q + (int64_t)b * H * D,"),
    "prefill_position": ("const int32_t t = (int32_t)(L0 + i + 1);",
                         "const int32_t t = (int32_t)(L0 + n);"),
    "prefill_row": ("const int64_t x = cu_new[b] + i;", "const int64_t x = cu_new[b] + (i > 0 ? i - 1 : 0);"),
}


def _pins_pass(lib) -> bool:
    """The pins of test_oracle_pins, run against one library."""
    try:
        if not _gqa_pin_passes(lib) or not _window_pin_passes(lib):
            return False
        if not _prefill_pins_pass(lib):
            return False
        for lens, H, D, P, dtype in [([5, 17, 33], 2, 2, 16, F32), ([31, 48, 2], 2, 8, 16, BF16),
                                     ([1], 2, 4, 16, F32)]:
            case = PagedCase(lens, H, D, P, dtype, seed=11)
            kp, vp = case.k_pool.copy(), case.v_pool.copy()
            out = oracle.paged_decode_attention(kp, vp, case.q, case.k_new, case.v_new,
                                                case.tables, case.seq_lens, dtype, library=lib)
            for b in range(case.B):
                pg, slot = case.tables[b, (lens[b] - 1) // P], (lens[b] - 1) % P
                if not np.array_equal(kp[pg, :, slot], case.k_new[b]):
                    return False
                for h in range(H):
                    lane = b * H + h
                    ref, _ = dense_causal_last_row(case.query_rows(b, h), to_f64(case.K[lane], dtype),
                                                   to_f64(case.V[lane], dtype))
                    if not np.allclose(out[b, h], ref, rtol=0, atol=1e-12):
                        return False
    except (ValueError, FloatingPointError):
        return False
    return True


def _gqa_pin_passes(lib) -> bool:
    """Grouped-query attention equals multi-head attention on KV heads repeated."""
    from tests.test_oracle_pins import gqa_case
    case, q, group, kp_rep, vp_rep, knew_rep, vnew_rep = gqa_case(group=2)
    kp, vp = case.k_pool.copy(), case.v_pool.copy()
    a = oracle.paged_decode_attention(kp, vp, q, case.k_new, case.v_new, case.tables,
                                      case.seq_lens, case.dtype, library=lib, group=group)
    b = oracle.paged_decode_attention(kp_rep, vp_rep, q, knew_rep, vnew_rep, case.tables,
                                      case.seq_lens, case.dtype, library=lib)
    return np.allclose(a, b, rtol=0, atol=1e-12)


def _window_pin_passes(lib) -> bool:
    from tests.test_oracle_pins import banded_last_row
    case = PagedCase([3, 17, 50], 2, 8, 16, F32, seed=21)
    out = oracle.paged_decode_attention(case.k_pool.copy(), case.v_pool.copy(), case.q, case.k_new,
                                        case.v_new, case.tables, case.seq_lens, F32, library=lib,
                                        window=17)
    for b in range(case.B):
        for h in range(2):
            lane = b * 2 + h
            ref = banded_last_row(case.query_rows(b, h), to_f64(case.K[lane], F32),
                                  to_f64(case.V[lane], F32), 17)
            if not np.allclose(out[b, h], ref, rtol=0, atol=1e-12):
                return False
    return True


def _prefill_pins_pass(lib) -> bool:
    from tests.test_oracle_pins import PREFILL_PINS, check_prefill_pin
    try:
        for args in PREFILL_PINS:
            check_prefill_pin(*args, library=lib)
    except AssertionError:
        return False
    return True


def _compile(tmp_path, name, text):
    src = tmp_path / f"{name}.c"
    src.write_text(text)
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", str(src), "-o", str(so), "-lm"],
                   check=True, capture_output=True)
    return oracle.load(str(so))


def test_unmutated_copy_passes(tmp_path):
    assert _pins_pass(_compile(tmp_path, "clean", open(SRC).read()))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site for {name} not found exactly once"
    lib = _compile(tmp_path, name, text.replace(old, new))
    with np.errstate(all="ignore"):
        assert not _pins_pass(lib), f"pins accepted mutant {name}"
