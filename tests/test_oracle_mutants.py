"""Plants plausible mistakes in a copy of the oracle and checks the pins catch
each one (CPU only). The planted copies are built in a temporary directory;
the committed oracle is never modified."""
from __future__ import annotations

import os
import tempfile

import pytest

import oracle
from tests import test_oracle as pins

# (name, text in gemm_ref.cpp, replacement)
MUTANTS = [
    ("b_read_row_major", "p.B[(l * p.N + j) * p.K + k]", "p.B[(l * p.K + k) * p.N + j]"),
    ("dropped_last_k", "k < p.K; ++k", "k + 1 < p.K; ++k"),
    ("beta_sign", "v += p.beta *", "v -= p.beta *"),
    ("a_batch_ignored", "p.A[(l * p.M + i) * p.K + k]", "p.A[(i) * p.K + k]"),
    ("alpha_scales_c", "v += p.beta *", "v += p.alpha * p.beta *"),
    ("fp32_accumulator", "double s = 0.0;", "float s = 0.0f;"),
    ("c_transposed", "p.C[(l * p.M + i) * p.N + j]", "p.C[(l * p.N + j) * p.M + i]"),
    ("b_batch_ignored", "p.B[(l * p.N + j) * p.K + k]", "p.B[(j) * p.K + k]"),
    ("bf16_decode_shift", "bits) << 16", "bits) << 15"),
    ("alpha_dropped", "double v = p.alpha * s;", "double v = s;"),
    ("k_starts_at_one", "int64_t k = 0; k < p.K", "int64_t k = 1; k < p.K"),
    ("batch_row_split", "const int64_t l = g / p.M;\n  const int64_t i = g % p.M;",
     "const int64_t l = g % p.L;\n  const int64_t i = g / p.L;"),
]

PINS = [
    lambda: pins.test_identity_b_returns_a(64),
    lambda: pins.test_all_ones_gives_k(7),
    pins.test_alpha_zero_is_beta_c,
    pins.test_k_zero_gives_beta_c,
    *[(lambda s=s: pins.test_bruteforce_rational(s)) for s in range(12)],
    pins.test_integer_inputs_exact_vs_integer_matmul,
    pins.test_linearity_in_alpha_beta,
    pins.test_handworked_fixture,
]


def _build_mutant(tmp, name, old, new):
    with open(oracle.SRC) as f:
        src = f.read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    path = os.path.join(tmp, f"{name}.cpp")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    return oracle.compile_oracle(path, os.path.join(tmp, f"lib{name}.so"))


def _pins_fail_with(lib) -> bool:
    saved = oracle._lib
    oracle._lib = lib
    try:
        for pin in PINS:
            try:
                pin()
            except (AssertionError, ValueError):
                return True
        return False
    finally:
        oracle._lib = saved


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, old, new):
    with tempfile.TemporaryDirectory() as tmp:
        lib = oracle.load(_build_mutant(tmp, name, old, new))
        assert _pins_fail_with(lib), f"no pin caught the planted mistake {name}"


def test_unmutated_copy_passes_every_pin():
    with tempfile.TemporaryDirectory() as tmp:
        lib = oracle.load(_build_mutant(tmp, "none", "double s = 0.0;", "double s = 0.0;"))
        assert not _pins_fail_with(lib)
