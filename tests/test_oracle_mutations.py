"""The oracle's pins must be strong enough to catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (a dropped
term, a wrong sign, a wrong index, a transposed operand, a reversed product),
compiles it on the CPU, and runs the whole pin battery of
``test_oracle_pins`` against it: at least one pin must fail.
"""
import inspect
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")

MUTATIONS = {
    "gate_dropped_on_correction": ("- alpha * b * sk[i] * kt[j]", "- b * sk[i] * kt[j]"),
    "correction_sign_flipped": ("- alpha * b * sk[i] * kt[j]", "+ alpha * b * sk[i] * kt[j]"),
    "beta_dropped_on_write": ("+ b * vt[i] * kt[j]", "+ vt[i] * kt[j]"),
    "gate_not_exponentiated": ("const double alpha = exp(g[t * d->h_v + hv]);",
                               "const double alpha = 1.0 + g[t * d->h_v + hv];"),
    "readout_uses_key": ("(d->scale * qt[j])", "(d->scale * kt[j])"),
    "readout_scale_dropped": ("(d->scale * qt[j])", "(qt[j])"),
    "gqa_heads_interleaved": ("const int64_t hk = hv / group;", "const int64_t hk = hv % d->h_k;"),
    "transition_operand_transposed": ("- b * kt[i] * ktT[j]);", "- b * ktT[i] * kt[j]);"),
    "compose_product_reversed": ("matmul(prod, Tm, tmp, dk, dk, dk);", "matmul(Tm, prod, tmp, dk, dk, dk);"),
    "compose_drops_entering_state": ("(c->S_in ? 0 : 1)", "1"),
    "norm_skipped_on_query": ("l2_normalise(qin, dk, qt);", "memcpy(qt, qin, sizeof(double) * (size_t)dk);"),
    "scalar_family_keeps_projection": ("d->scalar_decay ? alpha * S[i * dk + j] + b * vt[i] * kt[j]",
                                       "d->scalar_decay ? alpha * S[i * dk + j] - alpha * b * sk[i] * kt[j] + b * vt[i] * kt[j]"),
    "scalar_family_transition_undecayed": ("d->scalar_decay ? alpha * Tc[i * dk + j]", "d->scalar_decay ? Tc[i * dk + j]"),
}


def _pin_calls():
    calls = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        marks = getattr(fn, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        if params:
            argnames, values = params[0].args
            argnames = [a.strip() for a in argnames.split(",")] if isinstance(argnames, str) else list(argnames)
            for val in values:
                val = val if isinstance(val, tuple) else (val,)
                calls.append((f"{name}{val}", fn, dict(zip(argnames, val))))
        else:
            calls.append((name, fn, {}))
    return calls


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(mutation, tmp_path, monkeypatch):
    old, new = MUTATIONS[mutation]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mutated = tmp_path / "mut.c"
    mutated.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", "-pthread", str(mutated), "-o", str(so), "-lm"],
                   check=True)
    monkeypatch.setattr(oracle, "_lib", oracle._open(str(so)))
    failed = []
    for label, fn, kwargs in _pin_calls():
        try:
            fn(**kwargs)
        except AssertionError:
            failed.append(label)
    assert failed, f"no pin caught mutation {mutation}"
