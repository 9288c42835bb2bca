"""Plant plausible mistakes in copies of the oracle (on the CPU) and check a pin catches each.

Each mutant is the oracle's C source with one textual change, compiled into a
temporary directory.  A mutant that passes every pin would mean the pins do
not fix that part of the definition.
"""
import os

import pytest

from oracle import oracle as orc_mod
from tests.pins import PINS

SRC = os.path.join(os.path.dirname(orc_mod.__file__), "kda_oracle.c")

MUTANTS = {
    "delta_sign": ("S[(int64_t)i * nj + j] += b * kk[i]", "S[(int64_t)i * nj + j] -= b * kk[i]"),
    "beta_dropped": ("+= b * kk[i] * (", "+= kk[i] * ("),
    "decay_dropped": ("S[(int64_t)i * nj + j] *= alpha[i];", "S[(int64_t)i * nj + j] *= 1.0;"),
    "decay_on_columns": ("S[(int64_t)i * nj + j] *= alpha[i];",
                         "S[(int64_t)i * nj + j] *= alpha[(j0 + j) % dk];"),
    "alpha_not_exp": ("alpha[i] = exp(gate(", "alpha[i] = 1.0 + (gate("),
    "gate_sign": ("return g_min / (1.0 + exp(-x));", "return g_min / (1.0 + exp(x));"),
    "gate_no_exp_A": ("double x = exp(A) * z;", "double x = A * z;"),
    "a_uses_q": ("s += kk[i] * S[(int64_t)i * nj + j];", "s += qq[i] * S[(int64_t)i * nj + j];"),
    "o_uses_k": ("s += S[(int64_t)i * nj + j] * qq[i];", "s += S[(int64_t)i * nj + j] * kk[i];"),
    "v_index": ("ld(v, dt, vb + j0 + j)", "ld(v, dt, vb + j0)"),
    "h0_ignored": ("h0 ? h0[sbase + (int64_t)i * dv + j0 + j] : 0.0", "0.0"),
    "tile_no_restart": ("if ((t - cu_seqlens[n]) % tile == 0) run = 0.0;",
                        "if (t == cu_seqlens[n]) run = 0.0;"),
    "range_open_low": ("run >= -80.0", "run > -80.0"),
    "bf16_shift": ("<< 16;", "<< 15;"),
}


@pytest.fixture(scope="module")
def source():
    return open(SRC).read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source, tmp_path):
    old, new = MUTANTS[name]
    assert source.count(old) >= 1, f"mutation anchor for {name} not found"
    src = tmp_path / "mutant.c"
    src.write_text(source.replace(old, new))
    lib = orc_mod.build(force=True, src=str(src), out=str(tmp_path / "libmutant.so"))
    mutant = orc_mod.Oracle(lib)
    caught = []
    for pin in PINS:
        try:
            pin(mutant)
        except Exception:  # an assertion or a numerical blow-up both count as caught
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passes every pin"
