"""The multi-core build of the oracle (CPU only).

The same C source compiled with OpenMP splits every loop over rows or vector entries across
threads and sums each dot product in fixed 4096-entry chunks (chunk sums added in chunk order).
Pinned here:
  * every pin of the plain build holds for it too (tests/oracle_pins.py);
  * its results are bit-identical on 1, 2, 5 and all host threads (the chunking, not the
    thread count, fixes the summation order);
  * it agrees with the plain build to rounding, with the same iteration counts;
  * planted mistakes in its chunked dot product each fail a pin.
"""
import os

import numpy as np
import pytest

import oracle
from oracle_pins import ALL_PINS
from workloads import diffusion_dirichlet, poisson_5pt

SRC = os.path.join(os.path.dirname(oracle.__file__), "sla_oracle.c")


@pytest.fixture(scope="module")
def plib():
    return oracle.load_parallel()


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_pin_parallel_build(pin, plib):
    pin(plib)


def _run_all(lib, A, b, g, precond):
    f = oracle.cg(A.row_ptr, A.col_idx, A.values, b, rtol=1e-10, maxit=4000, precond=precond, history=True, lib=lib)
    a = oracle.cg_adjoint(A.row_ptr, A.col_idx, A.values, f["x"], g, rtol=1e-10, maxit=4000, precond=precond, lib=lib)
    return f, a


@pytest.mark.parametrize("precond", [0, 1])
def test_parallel_build_independent_of_thread_count(precond):
    m = 90  # n = 8100: two chunks and a ragged third
    A = diffusion_dirichlet(m, np.random.default_rng(71).lognormal(0, 1.0, 2 * m * (m + 1)))
    rng = np.random.default_rng(72)
    b, g = rng.standard_normal(A.n), rng.standard_normal(A.n)
    outs = []
    for th in sorted({1, 2, 5, oracle.host_cores()}):
        lib = oracle.load_parallel(th)
        assert lib.orc_threads(0) == th
        outs.append(_run_all(lib, A, b, g, precond))
    oracle.load_parallel()
    f0, a0 = outs[0]
    for f, a in outs[1:]:
        assert f["iters"] == f0["iters"] and a["iters"] == a0["iters"]
        for key in ("x", "history"):
            assert np.array_equal(f[key], f0[key])
        for key in ("grad_b", "grad_values"):
            assert np.array_equal(a[key], a0[key])


def test_parallel_build_agrees_with_plain_build():
    A = poisson_5pt(100)
    rng = np.random.default_rng(73)
    b, g = rng.standard_normal(A.n), rng.standard_normal(A.n)
    fp, ap = _run_all(oracle.load_parallel(), A, b, g, 0)
    fs, as_ = _run_all(oracle.load(), A, b, g, 0)
    assert abs(fp["iters"] - fs["iters"]) <= 1 and abs(ap["iters"] - as_["iters"]) <= 1
    assert np.linalg.norm(fp["x"] - fs["x"]) <= 1e-12 * np.linalg.norm(fs["x"])
    assert np.linalg.norm(ap["grad_b"] - as_["grad_b"]) <= 1e-12 * np.linalg.norm(as_["grad_b"])
    assert np.linalg.norm(ap["grad_values"] - as_["grad_values"]) <= 1e-12 * np.linalg.norm(as_["grad_values"])
    k = min(50, len(fs["history"]) - 1)
    assert np.all(np.abs(fp["history"][:k] - fs["history"][:k]) <= 1e-12 * fs["history"][:k])


CHUNK_MUTANTS = [
    ("chunk_count_drops_tail", "const int64_t nc = (n + ORC_CHUNK - 1) / ORC_CHUNK;",
     "const int64_t nc = n / ORC_CHUNK;"),
    ("chunk_sums_skip_first", "for (int64_t c = 0; c < nc; ++c) s += cs[c];",
     "for (int64_t c = 1; c < nc; ++c) s += cs[c];"),
    ("chunk_start_off_by_one", "for (int64_t i = c * ORC_CHUNK; i < i1; ++i) s += a[i] * b[i];",
     "for (int64_t i = c * ORC_CHUNK + 1; i < i1; ++i) s += a[i] * b[i];"),
    ("chunk_wrong_operand", "for (int64_t i = c * ORC_CHUNK; i < i1; ++i) s += a[i] * b[i];",
     "for (int64_t i = c * ORC_CHUNK; i < i1; ++i) s += a[i] * a[i];"),
]


@pytest.mark.parametrize("name,orig,mut", CHUNK_MUTANTS, ids=[m[0] for m in CHUNK_MUTANTS])
def test_chunk_mutant_is_caught(name, orig, mut, tmp_path):
    text = open(SRC).read()
    assert text.count(orig) == 1, f"mutation site for {name} not unique"
    src = tmp_path / f"{name}.c"
    src.write_text(text.replace(orig, mut))
    so = str(tmp_path / f"lib{name}.so")
    oracle.build(force=True, src=str(src), out=so, openmp=True)
    lib = oracle.load(so)
    lib.orc_threads(2)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except Exception as e:  # noqa: BLE001 - any failure counts as caught
            caught.append((pin.__name__, type(e).__name__))
    assert caught, f"mutant {name} passed every pin"
