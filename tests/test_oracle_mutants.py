"""Plant plausible mistakes in a copy of the C oracle; every one must trip a pin.

Each mutant is a textual edit of oracle/kda_oracle.c compiled into a temporary
directory. The real oracle source is never modified.
"""
import os

import pytest

import oracle
import pins

MUTANTS = {
    "error_sign": ("scratch[j] = vrow[j] - p;", "scratch[j] = vrow[j] + p;"),
    "no_decay": ("S[(size_t)i * ncol + j] *= alpha[i];", "S[(size_t)i * ncol + j] *= 1.0;"),
    "decay_on_columns": ("S[(size_t)i * ncol + j] *= alpha[i];",
                         "S[(size_t)i * ncol + j] *= alpha[j % dk];"),
    "drop_beta": ("+= beta * k[i] * scratch[j];", "+= k[i] * scratch[j];"),
    "read_with_key": ("acc += q[i] * S[(size_t)i * ncol + j];",
                      "acc += k[i] * S[(size_t)i * ncol + j];"),
    "no_prediction": ("p += k[i] * S[(size_t)i * ncol + j];", "p += 0.0 * S[(size_t)i * ncol + j];"),
    "drop_gate": ("(gate ? gate[j] : 1.0)", "1.0"),
    "drop_scale": ("o[j] = scale * acc", "o[j] = acc"),
    "no_l2norm": ("      if (l2norm) {\n        l2_normalise(qq, dk);",
                  "      if (0) {\n        l2_normalise(qq, dk);"),
    "decay_exp_sign": ("al[i] = exp((double)log_alpha[rk + i]);\n      load_vec(vv",
                       "al[i] = exp(-(double)log_alpha[rk + i]);\n      load_vec(vv"),
    "summary_zero_init": ("Y[(size_t)i * ncol + i] = 1.0;", "Y[(size_t)i * ncol + i] = 0.0;"),
    "scan_transposed_X": ("acc += Xs[(size_t)i * dk + l] * E[(size_t)l * dv + j];",
                          "acc += Xs[(size_t)l * dk + i] * E[(size_t)l * dv + j];"),
    "scan_drop_Z": ("double acc = Zs[(size_t)i * dv + j];", "double acc = 0.0;"),
    "decode_ignores_slot": ("int64_t row = slot ? slot[n] : n;", "int64_t row = n;"),
    "ignores_initial_state": ("    if (S0)\n      memcpy(S, S0", "    if (0)\n      memcpy(S, S0"),
    "prefix_stop_off_by_one": ("t1 = t0 + t_stop[s];", "t1 = t0 + t_stop[s] + 1;"),
}


def _run_all_pins(orc):
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, RuntimeError, ValueError, FloatingPointError):
            failed.append(pin.__name__)
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    path = os.path.join(tmp_path, "mutant.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.compile_source(path, os.path.join(tmp_path, "libmutant.so"))
    failed = _run_all_pins(oracle.Oracle(lib))
    assert failed, f"mutant {name} passed every pin"
