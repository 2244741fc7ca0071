"""Planted mistakes in copies of the oracle must fail at least one pin.

Each mutant is a one-line textual change to a temporary copy of the oracle
source (a dropped term, a wrong sign, index or bias, a transposed operand),
compiled on the CPU.  The committed oracle is never modified.
"""
import os
import tempfile

import pytest

import oracle
from tests import pins

MUTANTS = {
    "head_map_mod": ("int j = h / G;\n        const int32_t* bt_row",
                     "int j = h % Hkv;\n        const int32_t* bt_row"),
    "prefill_head_map": ("int j = h / G;\n        int64_t cap",
                         "int j = h % Hkv;\n        int64_t cap"),
    "page_index_mod": ("int64_t page = bt_row[t / page_size];",
                       "int64_t page = bt_row[t % page_size];"),
    "slot_uses_head_stride": ("slot * p->token_stride", "slot * p->head_stride"),
    "e4m3_bias8": ("mag = ldexp(1.0 + (double)f / 8.0, e - 7);",
                   "mag = ldexp(1.0 + (double)f / 8.0, e - 8);"),
    "e4m3_subnormal": ("mag = ldexp((double)f, -9);", "mag = ldexp((double)f, -10);"),
    "e4m3_no_sign": ("return sign ? -mag : mag;\n}\n\n/* ---",
                     "return mag;\n}\n\n/* ---"),
    "f16_subnormal": ("mag = ldexp((double)f, -24);", "mag = ldexp((double)f, -25);"),
    "f16_truncate": ("double q = nearbyint(ldexp(m, 11));", "double q = floor(ldexp(m, 11));"),
    "no_softmax_scale": ("x[i] = softmax_scale * dot;", "x[i] = dot;"),
    "pv_uses_k": ("o[d] += w * pool_value(V,", "o[d] += w * pool_value(K,"),
    "tail_drops_p": ("for (int64_t t = 4 * own; t <= p; ++t) {   /* causal tail",
                     "for (int64_t t = 4 * own; t < p; ++t) {   /* causal tail"),
    "sel_allows_own": ("if (b >= own) {\n                    or_flag",
                       "if (b > own) {\n                    or_flag"),
    "no_seq_clamp": ("if (L > max_seq_len) {\n            or_flag(flags, ORC_FLAG_SEQ_CLAMPED);\n"
                     "            L = max_seq_len;",
                     "if (L > max_seq_len) {\n            or_flag(flags, ORC_FLAG_SEQ_CLAMPED);\n"
                     "            L = L;"),
    "kv_scale_dropped": ("return orc_e4m3_to_f64(((const uint8_t*)p->base)[off]) * p->scale;",
                         "return orc_e4m3_to_f64(((const uint8_t*)p->base)[off]);"),
    "normaliser_off_by_one": ("double w = x[i] / l;", "double w = x[i] / (l + 1e-3);"),
    "select_ties_to_higher_index": ("return -c;\n    return (a->idx > b->idx) - (a->idx < b->idx);",
                                    "return -c;\n    return (a->idx < b->idx) - (a->idx > b->idx);"),
    "select_negatives_not_reversed": ("return a > b ? -1 : 1;\n}", "return a < b ? -1 : 1;\n}"),
    "select_sign_flipped": ("return neg_a ? -1 : 1;", "return neg_a ? 1 : -1;"),
    "select_includes_own_block": ("int64_t n = p / 4;", "int64_t n = p / 4 + 1;"),
    "select_keeps_k_minus_1": ("const int64_t m = n < k ? n : k;",
                               "const int64_t m = n < k ? n : k - 1;"),
    "select_unsorted_output": ("qsort(pick, (size_t)m, sizeof(int32_t), orc_int32_ascending);",
                               ";"),
    "select_no_qpos_clamp": ("fl |= ORC_FLAG_QPOS_CLAMPED;\n            p = kv_len - 1;",
                             "fl |= ORC_FLAG_QPOS_CLAMPED;\n            p = p;"),
    "mask_ties_to_higher_index": ("return (a->idx > b->idx) - (a->idx < b->idx);\n}\n\n/* Returns 0, -1",
                                  "return (a->idx < b->idx) - (a->idx > b->idx);\n}\n\n/* Returns 0, -1"),
    "mask_keeps_at_threshold": ("if (S[j] > cut)", "if (S[j] >= cut)"),
    "mask_cut_uses_p": ("cut = (1.0 - p) * Z;", "cut = p * Z;"),
    "mask_ignores_topk": ("const int K = k < V ? k : V;", "const int K = V;"),
    "mask_no_max_shift": ("const double x0 = (double)l[0].x;", "const double x0 = 0.0;"),
    "mask_count_off_by_one": ("m = j + 1;", "m = j;"),
    "bad_page_kept": ("if (page < 0 || page >= num_pages)\n        return -1;",
                      "if (page < 0 || page > num_pages)\n        return -1;"),
}


def _run_pins(o):
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(o) if pin is not pins.pin_f16_encode else pin(o, sample=4000)
        except AssertionError:
            failed.append(pin.__name__)
        except Exception:  # a crash of the broken oracle also counts as caught
            failed.append(pin.__name__ + "(error)")
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, f"mut_{name}.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        lib = oracle.compile_source(path, os.path.join(d, f"libmut_{name}.so"))
        failed = _run_pins(oracle.Oracle(lib))
    assert failed, f"mutant {name} passed every pin"
