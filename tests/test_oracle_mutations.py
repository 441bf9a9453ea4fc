"""Planted mistakes in the oracle must fail its pins.

Each case copies the oracle's C source, plants one plausible mistake (a dropped
term, a wrong sign or index, a wrong bias, a transposed order), compiles the
copy on the CPU and runs the pin battery of `test_oracle_pins.py` against it.
At least one pin must fail for every mutant.  The real oracle is untouched.
"""
import inspect
import os

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "mqa_oracle.c")

MUTANTS = {
    "relu_dropped": ("double relu = dot > 0.0 ? dot : 0.0;", "double relu = dot;"),
    "relu_sign": ("double relu = dot > 0.0 ? dot : 0.0;", "double relu = dot < 0.0 ? -dot : 0.0;"),
    "weight_dropped": ("s += (double)w_row[h] * relu;", "s += relu;"),
    "weight_index": ("s += (double)w_row[h] * relu;", "s += (double)w_row[heads - 1 - h] * relu;"),
    "scale_dropped": ("return scale * s;", "return s;"),
    "head_index": ("const double *qh = qd + (int64_t)h * dim;", "const double *qh = qd;"),
    "dim_transposed": ("dot += qh[d] * kd[d];", "dot += qh[d] * kd[dim - 1 - d];"),
    "absolute_index": ("o[t] = (int32_t)(buf[t].key - s);", "o[t] = (int32_t)(buf[t].key);"),
    "order_reversed": ("if (x->score > y->score) return -1;\n    if (x->score < y->score) return 1;",
                       "if (x->score > y->score) return 1;\n    if (x->score < y->score) return -1;"),
    "pad_value": ("for (int64_t t = c; t < J->topk; ++t) o[t] = -1;",
                  "for (int64_t t = c; t < J->topk; ++t) o[t] = 0;"),
    "range_off_by_one": ("int64_t n = e > s ? e - s : 0;", "int64_t n = e > s + 1 ? e - s - 1 : 0;"),
    "e4m3_bias": ("else mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);",
                  "else mag = ldexp(1.0 + (double)m / 8.0, (int)e - 8);"),
    "e4m3_subnormal": ("if (e == 0u) mag = ldexp((double)m, -9);", "if (e == 0u) mag = ldexp((double)m, -10);"),
    "e4m3_sign": ("return s ? -mag : mag;", "return mag;"),
    "block_absolute_index": ("o[t] = (int32_t)(blk[t].block - b0);", "o[t] = (int32_t)(blk[t].block);"),
    "block_last_not_max": ("if (buf[t].score > blk[b].score) blk[b].score = buf[t].score;",
                           "blk[b].score = buf[t].score;"),
    "block_order": ("if (x->score > y->score) return -1;\n    if (x->score < y->score) return 1;\n    return (x->block",
                    "if (x->score > y->score) return 1;\n    if (x->score < y->score) return -1;\n    return (x->block"),
    "mask_bit_index": ("if (!((word >> ((j >> 3) & 31)) & 1u)) continue;", "if (!((word >> ((j >> 4) & 31)) & 1u)) continue;"),
    "mask_ignored": ("            if (J->mask) {", "            if (0) {"),
    "fold_exponent_low": ("    return ex - 9 + (f > 0.875 ? 1 : 0);", "    return ex - 10 + (f > 0.875 ? 1 : 0);"),
    "fold_ties_odd": ("if (d < bd || (d == bd && (c & 1u) == 0u)) {", "if (d < bd || (d == bd && (c & 1u) == 1u)) {"),
    "fold_weight_index": ("acc = fmaf(w[row * heads + h], (float)g_e4m3[q[(row * heads + h) * (int64_t)dim + d]], acc);",
                          "acc = fmaf(w[row * heads + (heads - 1 - h)], (float)g_e4m3[q[(row * heads + h) * (int64_t)dim + d]], acc);"),
    "fold_residual_sign": ("r[d] = r[d] - (float)ldexp(g_e4m3[u[d]], e);", "r[d] = r[d] + (float)ldexp(g_e4m3[u[d]], e);"),
    "ue8m0_shift": ("uint32_t bits = ((uint32_t)J->scale_groups[4 * j]) << 23;",
                    "uint32_t bits = ((uint32_t)J->scale_groups[4 * j + 1] + 1) << 23;"),
}


def battery():
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        params = inspect.signature(fn).parameters
        if "lib" not in params:
            continue
        marks = getattr(fn, "pytestmark", [])
        arglists = [{}]
        for m in marks:
            if m.name == "parametrize":
                argname, values = m.args[0], m.args[1]
                arglists = [dict(a, **{argname: v}) for a in arglists for v in values]
        for a in arglists:
            yield name, fn, a


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(mutant, tmp_path):
    old, new = MUTANTS[mutant]
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation site for {mutant} not found"
    src = tmp_path / f"{mutant}.c"
    src.write_text(text.replace(old, new))
    lib = oracle.load_library(oracle.build(force=True, src=str(src), out=str(tmp_path / f"{mutant}.so")))
    failed = []
    for name, fn, args in battery():
        try:
            fn(lib=lib, **args)
        except Exception:  # any failure of a pin counts
            failed.append(name)
    assert failed, f"no pin caught mutant {mutant}"
