"""The fp64 oracle against its pins (CPU only), and a check that the pins are
sharp: copies of the oracle with one planted mistake each must fail at least
one pin."""
import os
import shutil

import numpy as np
import pytest

import oracle
import oracle_pins as pins


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", pins.FAST_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_naive_sum_wrong_under_decay(orc):
    errs = pins.naive_wrong(orc)
    # context only: every head is far from the true state (the pages quote 22%
    # at 256 tokens for a slow-decay head with an unstated gamma and split)
    assert all(e >= 0.10 for e in errs)


def _mutants(src):
    """(name, mutated source) pairs; each plants one plausible mistake."""
    gate_block = (
        "  if (kind == 2) {\n"
        "    for (int i = 0; i < dk; i++) {\n"
        "      double a = exp(gv[i]);\n"
        "      for (int j = 0; j < m; j++) X[i * ld + j] *= a;\n"
        "    }\n"
        "  }\n")
    assert gate_block in src
    moved = src.replace(gate_block, "").replace("  if (kind == 1) {\n", gate_block + "  if (kind == 1) {\n", 1)
    muts = [
        ("beta dropped from the write", "double c = has_beta(var) ? b : 1.0;", "double c = 1.0;"),
        ("erase sign flipped", "X[i * ld + j] -= b * kv[i] * tmp[j];", "X[i * ld + j] += b * kv[i] * tmp[j];"),
        ("GQA head map wrong", "int kh = (int)(((int64_t)h * hk) / hv);\n  const double *kv",
         "int kh = h % hk;\n  const double *kv"),
        ("compose uses T^T", "acc += Tc[r * dk + c] * S[c * dv + j];", "acc += Tc[c * dk + r] * S[c * dv + j];"),
        ("compose drops S(C|0)", "S2[r * dv + j] = acc + Sc[r * dv + j];", "S2[r * dv + j] = acc;"),
        ("seam not excluded", "int64_t s = seg_offsets[i] + seam_w, e", "int64_t s = seg_offsets[i], e"),
        ("vector gate dropped", "  if (kind == 2) {\n", "  if (kind == 3) {\n"),
        ("scalar gate on wrong head", "case OR_GDN: *gs = exp(g[t * hv + h]);", "case OR_GDN: *gs = exp(g[t * hv]);"),
        ("merge order swapped", "acc += a[r * dk + x] * b[x * dk + c];", "acc += b[r * dk + x] * a[x * dk + c];"),
    ]
    out = []
    for name, a, b in muts:
        assert a in src, name
        out.append((name, src.replace(a, b, 1)))
    out.append(("channel gate after the erase", moved))
    return out


def test_pins_catch_planted_mistakes(tmp_path):
    src = open(oracle._SRC).read()
    for i, (name, msrc) in enumerate(_mutants(src)):
        c = tmp_path / f"m{i}.c"
        c.write_text(msrc)
        so = oracle.compile_oracle(str(c), str(tmp_path / f"m{i}.so"))
        orc = oracle.OracleLib(so)
        caught = []
        for pin in pins.FAST_PINS:
            try:
                pin(orc)
            except AssertionError:
                caught.append(pin.__name__)
        assert caught, f"planted mistake '{name}' passed every pin"


def _rerotate_mutant(form):
    """oracle.rerotate with one planted mistake in the transformation."""
    def rr(variant, T, S, deltas, rot_dim, layout="interleaved", base=10000.0):
        T, S = np.array(T, dtype=np.float64), np.array(S, dtype=np.float64)
        To, So = T.copy(), np.empty_like(S)
        for m, dl in enumerate(np.asarray(deltas).reshape(-1)):
            R = oracle.rerotation_matrix(S.shape[-2], dl, rot_dim, layout, base)
            So[m] = (R.T if form == "S by R^T" else R) @ S[m]
            if variant in ("gdn", "deltanet"):
                To[m] = {"T by R only": R @ T[m], "T by R^T T R": R.T @ T[m] @ R}.get(form, R @ T[m] @ R.T)
        return To, So
    return rr


@pytest.mark.parametrize("form", ["T by R only", "T by R^T T R", "S by R^T"])
def test_rerotation_pins_catch_planted_mistakes(orc, form):
    with pytest.raises(AssertionError):
        pins.rerotation_keys(orc, rerotate=_rerotate_mutant(form))
