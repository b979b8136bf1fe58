"""The oracle's pins catch plausible mistakes.

Each case below plants one mistake in a temporary copy of ``oracle/qknr_oracle.c``
(a dropped term, a flipped sign, a wrong index, a misread type, ...), builds that
copy with gcc on the CPU and runs every pin against it: at least one pin must
fail. All planted mistakes keep memory accesses in bounds for the pins' inputs.
"""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import oracle  # noqa: E402
from oracle_pins import ALL_PINS  # noqa: E402

# (name, original text, replacement, which occurrence)
MUTANTS = [
    ("mean_over_rope_dim", "r = 1.0 / sqrt(ss / (double)D + eps);",
     "r = 1.0 / sqrt(ss / (double)R + eps);", 0),
    ("eps_outside_root", "r = 1.0 / sqrt(ss / (double)D + eps);",
     "r = 1.0 / (sqrt(ss / (double)D) + eps);", 0),
    ("eps_dropped", "r = 1.0 / sqrt(ss / (double)D + eps);",
     "r = 1.0 / sqrt(ss / (double)D);", 0),
    ("root_dropped", "r = 1.0 / sqrt(ss / (double)D + eps);",
     "r = 1.0 / (ss / (double)D + eps);", 0),
    ("abs_not_square", "ss += xi * xi;", "ss += fabs(xi);", 0),
    ("weight_dropped", "n[i] = n[i] * r * qknr_oracle_decode(dtype, w[i]);",
     "n[i] = n[i] * r;", 0),
    ("weight_offset_one", "n[i] = n[i] * r * qknr_oracle_decode(dtype, w[i]);",
     "n[i] = n[i] * r * (1.0 + qknr_oracle_decode(dtype, w[i]));", 0),
    ("interleaved_even_sign", "out[2 * i] = a * c - b * s;", "out[2 * i] = a * c + b * s;", 0),
    ("interleaved_odd_sign", "out[2 * i + 1] = b * c + a * s;",
     "out[2 * i + 1] = b * c - a * s;", 0),
    ("neox_low_sign", "out[i] = a * c - b * s;", "out[i] = a * c + b * s;", 0),
    ("neox_high_sign", "out[i + half] = b * c + a * s;", "out[i + half] = b * c - a * s;", 0),
    ("neox_partner_adjacent", "double a = n[i], b = n[i + half];",
     "double a = n[i], b = n[i ^ 1];", 0),
    ("neox_as_interleaved", "if (!is_neox) {", "if (1) {", 0),
    ("interleaved_one_frequency", "double c = (double)cos_row[i], s = (double)sin_row[i];",
     "double c = (double)cos_row[0], s = (double)sin_row[0];", 0),
    ("neox_half_frequency", "double c = (double)cos_row[i], s = (double)sin_row[i];",
     "double c = (double)cos_row[i / 2], s = (double)sin_row[i / 2];", 1),
    ("tail_zeroed", "out[i] = n[i];", "out[i] = 0.0;", 0),
    ("sin_from_cos_half", "sin_row = cos_row + R / 2;", "sin_row = cos_row;", 0),
    ("cache_row_stride", "cos_row = cache + pos * R;", "cos_row = cache + pos * (R / 2);", 0),
    ("int64_read_as_int32", "((const int64_t *)positions)[t]",
     "(int64_t)((const int32_t *)positions)[t]", 0),
    ("k_heads_use_q_weight",
     "rc = qknr_oracle_head(k + t * k_stride + (int64_t)h * head_stride, k_w,",
     "rc = qknr_oracle_head(k + t * k_stride + (int64_t)h * head_stride, q_w,", 0),
    ("fp16_exponent_bias", "ldexp((double)(frac + 1024), expo - 25)",
     "ldexp((double)(frac + 1024), expo - 24)", 0),
    ("fp16_subnormal_scale", "ldexp((double)frac, -24)", "ldexp((double)frac, -25)", 0),
    ("bf16_shift", "(uint32_t)bits << 16", "(uint32_t)bits << 15", 0),
]


def _mutate(src: str, old: str, new: str, nth: int) -> str:
    idx = -1
    for _ in range(nth + 1):
        idx = src.find(old, idx + 1)
        assert idx >= 0, f"mutation anchor not found: {old!r}"
    return src[:idx] + new + src[idx + len(old):]


@pytest.mark.parametrize("name,old,new,nth", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_kill_mutant(name, old, new, nth, tmp_path):
    with open(oracle.SOURCE) as f:
        src = f.read()
    mutated = _mutate(src, old, new, nth)
    assert mutated != src
    c_path = tmp_path / f"{name}.c"
    so_path = tmp_path / f"lib{name}.so"
    c_path.write_text(mutated)
    oracle.build(force=True, source=str(c_path), output=str(so_path))
    lib = oracle.load(str(so_path))
    killed_by = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError):
            killed_by.append(pin.__name__)
    assert killed_by, f"mutant {name} survived every pin"
