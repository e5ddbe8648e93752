"""Planted mistakes in copies of the oracle must each trip at least one pin.

Each mutant is the oracle source with one plausible slip (a dropped term, a wrong
sign, index or operand), compiled on the CPU into a temporary library and run
through every pin in tests/oracle_pins.py.  The real oracle is never modified.
"""

import os
import subprocess

import pytest

import oracle
from oracle_pins import PINS

MUTANTS = {
    "causal_off_by_one": ("long long n = (long long)i + (Tk - Tq) + 1;",
                          "long long n = (long long)i + (Tk - Tq);"),
    "causal_top_left_when_rectangular": ("long long n = (long long)i + (Tk - Tq) + 1;",
                                         "long long n = (long long)i + 1;"),
    "gqa_head_modulo": ("const int kvh = h / group;\n                const uint16_t *qrow",
                        "const int kvh = h % Hkv;\n                const uint16_t *qrow"),
    "scale_dropped": ("p[j] = scale * acc;", "p[j] = acc;"),
    "lse_without_max": ("*lse = m + log(l);", "*lse = log(l);"),
    "lse_log2": ("*lse = m + log(l);", "*lse = m + log2(l);"),
    "scores_use_v": ("bf16_to_double(kr[j][d]);", "bf16_to_double(vr[j][d]);"),
    "not_normalised": ("for (int j = 0; j < n_vis; ++j) p[j] /= l;",
                       "for (int j = 0; j < n_vis; ++j) p[j] /= 1.0;"),
    "exp_sign_flipped": ("p[j] = exp(p[j] - m);", "p[j] = exp(m - p[j]);"),
    "paged_slot_index": ("* bs + (t % bs)) * (long long)D;", "* bs + (t / bs)) * (long long)D;"),
    "paged_block_index": ("block_table[(long long)r * max_blocks + t / bs];",
                          "block_table[(long long)r * max_blocks + t % bs];"),
    "paged_head_stride": ("(((long long)phys * Hkv + kvh) * bs", "(((long long)phys + kvh) * bs"),
    "decode_drops_last_key": ("attend_row(q + rh * D, kr, vr, L, D,",
                              "attend_row(q + rh * D, kr, vr, L - 1, D,"),
    "q_row_stride": ("const uint16_t *qrow = q + r * D;", "const uint16_t *qrow = q + (r / Tq) * D;"),
}


def _run_pins(lib):
    caught = []
    for pin in PINS:
        try:
            pin(lib)
        except Exception as exc:  # AssertionError or a numeric blow-up both count
            caught.append(f"{pin.__name__}: {type(exc).__name__}")
    return caught


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    pytest.importorskip("mpmath")
    pytest.importorskip("scipy")
    old, new = MUTANTS[name]
    with open(oracle._SRC) as fh:
        src = fh.read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutated = src.replace(old, new)
    c_path = os.path.join(tmp_path, "mutant.c")
    so_path = os.path.join(tmp_path, "libmutant.so")
    with open(c_path, "w") as fh:
        fh.write(mutated)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", so_path,
                    c_path, "-lm"], check=True)
    caught = _run_pins(oracle.load(so_path))
    assert caught, f"mutant {name} passed every pin"
