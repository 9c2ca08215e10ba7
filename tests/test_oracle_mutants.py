"""Planted mistakes in the oracle must be caught by the pins.

Each case copies ssd_oracle.c, plants one plausible mistake by text
substitution (a dropped term, a wrong sign, a wrong index or mask, a swapped
operand), builds the copy with gcc into a temporary directory, swaps it in as
the oracle library and runs the pin suites of test_oracle_pins.py,
test_oracle_bwd_pins.py and test_oracle_s6_pins.py.  At least
one pin must fail for every mutant.  All of this runs on the CPU.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_bwd_pins as bwd_pins
from tests import test_oracle_pins as pins
from tests import test_oracle_s6_pins as s6_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "ssd_oracle.c")

MUTANTS = {
    "output-uses-previous-state": (
        "acc += j->Cm[IX_BC(j, b, t, g, s)] * v;",
        "acc += j->Cm[IX_BC(j, b, t, g, s)] * ((v - dtv * j->Bm[IX_BC(j, b, t, g, s)] * xp) / alpha);"),
    "wrong-group-mapping": (
        "static void seq_unit(const job_t *j, int64_t b, int64_t h, double *st)\n{\n    const int64_t H = j->H, S = j->S;\n    const int64_t g = h / (j->nheads / j->ngroups);",
        "static void seq_unit(const job_t *j, int64_t b, int64_t h, double *st)\n{\n    const int64_t H = j->H, S = j->S;\n    const int64_t g = h % j->ngroups;"),
    "decay-sign-flipped": (
        "const double alpha = exp(j->A[h] * dtv);          /* exp(A dt_t) */",
        "const double alpha = exp(-j->A[h] * dtv);"),
    "b-and-c-swapped": (
        "double v = alpha * st[p * S + s] + dtv * j->Bm[IX_BC(j, b, t, g, s)] * xp;",
        "double v = alpha * st[p * S + s] + dtv * j->Cm[IX_BC(j, b, t, g, s)] * xp;"),
    "missing-dt-on-input": (
        "double v = alpha * st[p * S + s] + dtv * j->Bm[IX_BC(j, b, t, g, s)] * xp;",
        "double v = alpha * st[p * S + s] + j->Bm[IX_BC(j, b, t, g, s)] * xp;"),
    "chunk-cumsum-exclusive": (
        "run += j->A[h] * j->dt[IX_DT(j, b, t0 + i, h)];\n            G[i] = run;",
        "G[i] = run;\n            run += j->A[h] * j->dt[IX_DT(j, b, t0 + i, h)];"),
    "chunk-mask-drops-diagonal": (
        "for (int64_t jj = 0; jj <= i; ++jj) intra += P[jj]",
        "for (int64_t jj = 0; jj < i; ++jj) intra += P[jj]"),
    "chunk-skip-term-dropped": (
        "j->y[IX_X(j, b, ti, h, p)] = carried + intra + j->D[h] * j->x[IX_X(j, b, ti, h, p)];",
        "j->y[IX_X(j, b, ti, h, p)] = carried + intra;"),
    "chunk-carried-state-undecayed": (
        "carried *= exp(G[i]);",
        "carried *= 1.0;"),
    "chunk-jump-missing-decay": (
        "for (int64_t e = 0; e < H * S; ++e) st[e] = decay * st[e] + snew[e];",
        "for (int64_t e = 0; e < H * S; ++e) st[e] = st[e] + snew[e];"),
    "chunk-state-transposed": (
        "j->Bm[IX_BC(j, b, ti, g, s)] * j->x[IX_X(j, b, ti, h, p)];",
        "j->Bm[IX_BC(j, b, ti, g, p % j->S)] * j->x[IX_X(j, b, ti, h, s % j->H)];"),
    "step-decay-missing": (
        "row[s] = alpha * row[s] + dtv * Bv[s] * xp;",
        "row[s] = row[s] + dtv * Bv[s] * xp;"),
    # gradients (oracle_ssd_bwd_seq)
    "bwd-adjoint-undecayed": (
        "for (int64_t e = 0; e < HS; ++e) lam[e] *= alpha;",
        "for (int64_t e = 0; e < HS; ++e) lam[e] *= 1.0;"),
    "bwd-dx-missing-dt": (
        "j->dx[BIX_X(j, b, t, h, p)] = dtv * acc + j->D[h] * dyp;",
        "j->dx[BIX_X(j, b, t, h, p)] = acc + j->D[h] * dyp;"),
    "bwd-dC-uses-previous-state": (
        "for (int64_t p = 0; p < H; ++p) acc += hcur[p * S + s] * j->dy[BIX_X(j, b, t, h, p)];",
        "for (int64_t p = 0; p < H; ++p) acc += hprev[p * S + s] * j->dy[BIX_X(j, b, t, h, p)];"),
    "bwd-ddt-drops-decay-path": (
        "j->ddt[BIX_DT(j, b, t, h)] = via_b + Ah * da;",
        "j->ddt[BIX_DT(j, b, t, h)] = via_b;"),
    "bwd-dA-missing-dt": (
        "dA += dtv * da;",
        "dA += da;"),
    "bwd-decay-path-uses-current-state": (
        "lam_hprev += lam[p * S + s] * hprev[p * S + s];",
        "lam_hprev += lam[p * S + s] * hcur[p * S + s];"),
    "bwd-dB-wrong-group": (
        "const int64_t g = h / hpg;\n                    for (int64_t s = 0; s < S; ++s) {",
        "const int64_t g = h % ngroups;\n                    for (int64_t s = 0; s < S; ++s) {"),
    "bwd-dB-transposed-operand": (
        "for (int64_t p = 0; p < H; ++p) acc += lam[p * S + s] * j->x[BIX_X(j, b, t, h, p)];",
        "for (int64_t p = 0; p < H; ++p) acc += lam[p * S + s] * j->dy[BIX_X(j, b, t, h, p)];"),
    "bwd-dD-drops-x": (
        "dD += dyp * j->x[BIX_X(j, b, t, h, p)];",
        "dD += dyp;"),
    # Mamba-1 selective scan (oracle_s6_fwd_seq)
    "s6-A-transposed": (
        "const double abar = exp(dl * A[d * N + n]);",
        "const double abar = exp(dl * A[(n * dim + d) % (dim * N)]);"),
    "s6-bbar-missing-delta": (
        "const double bbar = dl * Bm[((b * ngroups + g) * N + n) * seqlen + t];",
        "const double bbar = Bm[((b * ngroups + g) * N + n) * seqlen + t];"),
    "s6-output-uses-previous-state": (
        "h[n] = abar * h[n] + bbar * xt;\n                    acc += Cm[((b * ngroups + g) * N + n) * seqlen + t] * h[n];",
        "acc += Cm[((b * ngroups + g) * N + n) * seqlen + t] * h[n];\n                    h[n] = abar * h[n] + bbar * xt;"),
    "s6-wrong-group": (
        "const int64_t g = d / cpg;\n            for (int64_t n = 0; n < N; ++n) h[n] = h0",
        "const int64_t g = d % ngroups;\n            for (int64_t n = 0; n < N; ++n) h[n] = h0"),
    "s6-skip-dropped": (
        "y[(b * dim + d) * seqlen + t] = acc + (D ? D[d] * xt : 0.0);",
        "y[(b * dim + d) * seqlen + t] = acc;"),
    "bwd-dh-final-ignored": (
        "lam[p * S + s] = j->dhf ? j->dhf[BIX_H(j, b, h, p, s)] : 0.0;",
        "lam[p * S + s] = 0.0;"),
}


def _pin_functions():
    out = []
    for mod, name in [(m, n) for m in (pins, bwd_pins, s6_pins) for n in dir(m)]:
        if not name.startswith("test_"):
            continue
        fn = getattr(mod, name)
        marks = getattr(fn, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        if params:
            argname, values = params[0].args
            for v in values:
                out.append((f"{name}[{v}]", lambda fn=fn, v=v: fn(v)))
        else:
            out.append((name, fn))
    return out


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_is_caught(mutant, tmp_path, monkeypatch):
    old, new = MUTANTS[mutant]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {mutant} not unique"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", str(so), str(path),
                    "-lpthread", "-lm"], check=True)
    real = oracle._load()
    lib = ctypes.CDLL(str(so))
    for fname in ("oracle_ssd_fwd_seq", "oracle_ssd_fwd_chunked", "oracle_ssd_step", "oracle_ssd_bwd_seq",
                  "oracle_s6_fwd_seq"):
        getattr(lib, fname).argtypes = getattr(real, fname).argtypes
        getattr(lib, fname).restype = getattr(real, fname).restype
    monkeypatch.setattr(oracle, "_lib", lib)
    failed = []
    for name, fn in _pin_functions():
        try:
            fn()
        except AssertionError:
            failed.append(name)
    assert failed, f"no pin caught the planted mistake {mutant}"
