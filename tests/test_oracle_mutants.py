"""The oracle's pins catch plausible mistakes: each case plants one mistake in a copy of the
oracle source (a dropped term, a wrong sign, a swapped operand or index, an off-by-one in a
scan or window), compiles it on the CPU with the oracle's own flags, and runs the named pins
against it; at least one of them must fail. The real oracle is untouched and restored after
each case. Every mutation keeps all indices in bounds."""
import ctypes
import os

import pytest

import oracle
from oracle import build as obuild
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(obuild.__file__), "kda_oracle.cpp")

MUTANTS = [
    ("decay dropped",
     [("S[(int64_t)c * nc + j] *= a[c];", "S[(int64_t)c * nc + j] *= 1.0;")],
     ["test_p1_beta_zero_closed_form", "test_p3_single_token_matrix_form"]),
    ("write subtracts",
     [("S[(int64_t)c * nc + j] += b * kk[c] * u[j];", "S[(int64_t)c * nc + j] -= b * kk[c] * u[j];")],
     ["test_p4_write_invariant", "test_p3_single_token_matrix_form"]),
    ("prediction error sign",
     [("u[j] = vcol(t, j0 + j) - acc;", "u[j] = vcol(t, j0 + j) + acc;")],
     ["test_p4_write_invariant", "test_p3_single_token_matrix_form"]),
    ("read with the key instead of the query",
     [("acc += qq[c] * S[(int64_t)c * nc + j];", "acc += kk[c] * S[(int64_t)c * nc + j];")],
     ["test_p3_single_token_matrix_form", "test_p1_beta_zero_closed_form"]),
    ("composition order swapped",
     [("acc += M2[(int64_t)r * dk + x] * M1[(int64_t)x * dk + c];",
       "acc += M1[(int64_t)r * dk + x] * M2[(int64_t)x * dk + c];")],
     ["test_p5b_package_is_affine_map", "test_p5_package_composition_all_cuts"]),
    ("inclusive instead of exclusive scan",
     [("      std::memcpy(seg_init + (p * H + h) * sd, cur.data(), sd * 8);\n", ""),
      ("      cur.swap(nxt);\n",
       "      cur.swap(nxt);\n      std::memcpy(seg_init + (p * H + h) * sd, cur.data(), sd * 8);\n")],
     ["test_p5_package_composition_all_cuts"]),
    ("logit sign",
     [("1.0 / (1.0 + std::exp(-beta[i]))", "1.0 / (1.0 + std::exp(beta[i]))")],
     ["test_window_logit_extremes_closed_forms"]),
    ("window ignores its read slot",
     [("std::vector<double> S(pool + (r * H + h) * sd, pool + (r * H + h) * sd + sd);",
       "std::vector<double> S(sd, 0.0);")],
     ["test_window_snapshots_exact_rational"]),
    ("snapshot stored into the neighbouring slot",
     [("std::memcpy(pool + (w * H + h) * sd, S.data(), sd * sizeof(double));",
       "std::memcpy(pool + (((w + 1) % n_slots) * H + h) * sd, S.data(), sd * sizeof(double));")],
     ["test_window_snapshots_exact_rational", "test_window_fork_rollback_and_slots"]),
    ("conv taps reversed",
     [("y += w[(int64_t)c * W + i] * z[u - hw + i];",
       "y += w[(int64_t)c * W + (W - 1 - i)] * z[u - hw + i];")],
     ["test_short_conv_matches_library_convolution"]),
    ("conv window keeps the oldest inputs",
     [("pool[(wr * hw + j) * C + c] = z[n - hw + j];", "pool[(wr * hw + j) * C + c] = z[j];")],
     ["test_short_conv_split_packing_and_slots"]),
]


@pytest.mark.parametrize("name,edits,pin_names", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, edits, pin_names, tmp_path):
    with open(SRC) as f:
        src = f.read()
    for old, new in edits:
        assert src.count(old) == 1, (name, old)
        src = src.replace(old, new)
    path = tmp_path / "mutant.cpp"
    path.write_text(src)
    lib = oracle._bind(ctypes.CDLL(obuild.compile_source(str(path), str(tmp_path / "mut.so"))))
    saved = oracle._load()
    oracle._lib = lib
    caught = []
    try:
        for pin in pin_names:
            try:
                getattr(pins, pin)(oracle)
            except AssertionError:
                caught.append(pin)
    finally:
        oracle._lib = saved
    assert caught, f"no pin caught the mutant '{name}'"


def test_unmutated_copy_passes_every_pin(tmp_path):
    """Control: the same harness on an unchanged copy of the source fails no pin."""
    path = tmp_path / "copy.cpp"
    with open(SRC) as f:
        path.write_text(f.read())
    lib = oracle._bind(ctypes.CDLL(obuild.compile_source(str(path), str(tmp_path / "copy.so"))))
    saved = oracle._load()
    oracle._lib = lib
    try:
        for pin in sorted({p for m in MUTANTS for p in m[2]}):
            getattr(pins, pin)(oracle)
    finally:
        oracle._lib = saved
