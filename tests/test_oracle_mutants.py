"""Planted mistakes in the oracle must be caught by the pins.

Each mutant is a one-line change to a copy of the oracle's C source
(compiled to a temporary library); the pins of tests/test_oracle.py are run
against it and at least one must fail.  This shows the pins constrain the
oracle rather than restate it.
"""
import ctypes
import inspect

import pytest

import oracle
from tests import test_oracle as pins

MUTANTS = {
    "nibble order": ("(r / 2 + 4 * (r % 2))", "(r)"),
    "byte order": ("(rr / 2 + 2 * (rr % 2))", "(rr)"),
    "unpack offset": ("int u = (int)((packed[w] >> sh) & mask);\n      q_out[k * N + n] = (int8_t)(u - off);",
                      "int u = (int)((packed[w] >> sh) & mask);\n      q_out[k * N + n] = (int8_t)(u - off + 1);"),
    "round half away": ("rintf(W[k * N + n] / sc)", "roundf(W[k * N + n] / sc)"),
    "no upper clamp": ("if (r > hi) r = hi;", ""),
    "int4 qpos 8": ("static int qpos_of(int bits) { return bits == 4 ? 7 : 127; }",
                    "static int qpos_of(int bits) { return bits == 4 ? 8 : 127; }"),
    "dequant drops scale": ("bf16_to_f32(s[(k / group) * N + n]) * (float)q[k * N + n]",
                            "(float)q[k * N + n]"),
    "dequant wrong group": ("bf16_to_f32(s[(k / group) * N + n]) * (float)q[k * N + n]",
                            "bf16_to_f32(s[(k % group) % (K / group) * N + n]) * (float)q[k * N + n]"),
    "fp32 accumulation": ("y[n] += x * (double)wrow[n];", "y[n] = (float)(y[n] + x * (double)wrow[n]);"),
    "X row stride": ("j->X[m * j->K + k]", "j->X[m * j->N + k]"),
    "group stride": ("(nt * (K / 128) + g) * 8 + j8", "(nt + g) * 8 + j8"),
    "int8 half split": ("((slab * 2 + word / 4) * 32 + lane) * 4 + word % 4",
                        "((slab * 2 + word % 2) * 32 + lane) * 4 + word / 2"),
    "bf16 round half up": ("u += 0x7FFFu + lsb;", "u += 0x8000u;"),
}


def _pin_functions():
    out = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        marks = getattr(fn, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        combos = [{}]
        for m in params:
            argnames = [a.strip() for a in m.args[0].split(",")] \
                if isinstance(m.args[0], str) else list(m.args[0])
            new = []
            for c in combos:
                for v in m.args[1]:
                    vals = v if len(argnames) > 1 else (v,)
                    d = dict(c)
                    d.update(zip(argnames, vals))
                    new.append(d)
            combos = new
        for c in combos:
            out.append((name, fn, c))
    return out


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_planted_mistake(mutant, tmp_path, monkeypatch):
    old, new = MUTANTS[mutant]
    src = oracle.source_text()
    assert src.count(old) >= 1, f"mutation site for {mutant!r} not found"
    lib_path = oracle.compile_variant(src.replace(old, new),
                                      str(tmp_path / "mutant.so"))
    lib = oracle._bind(ctypes.CDLL(lib_path))
    monkeypatch.setattr(oracle, "_lib", lib)
    failures = []
    for name, fn, kwargs in _pin_functions():
        try:
            fn(**kwargs)
        except Exception as e:  # noqa: BLE001 - any failure counts
            failures.append((name, type(e).__name__))
    assert failures, f"no pin caught the mutant {mutant!r}"
