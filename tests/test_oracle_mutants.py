"""The pins have teeth: each plausible mistake, planted in a copy of the
oracle's C source and compiled on the CPU, must fail at least one pin."""
import os

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text in oracle.c, replacement)
MUTANTS = [
    ("truncate-instead-of-rne", "float r = nearbyintf(t);", "float r = truncf(t);"),
    ("int8-scale-over-128", "a / 127.0f", "a / 128.0f"),
    ("int4-scale-over-16", "(hi - lo) / 15.0f", "(hi - lo) / 16.0f"),
    ("int4-sign-flip", "(xg[k] - lo) / sc", "(lo - xg[k]) / sc"),
    ("int4-dropped-zero-point", "return m + z[e / G];", "return m;"),
    ("int4-nibbles-swapped", "code << ((e & 1) ? 4 : 0)", "code << ((e & 1) ? 0 : 4)"),
    ("reduce-reversed", "for (int p = 0; p < P; ++p) acc = acc + d[p][i];",
     "for (int p = P - 1; p >= 0; --p) acc = acc + d[p][i];"),
    ("reduce-starts-at-minus-zero", "float acc = 0.0f;\n    for (int p = 0; p < P; ++p) acc",
     "float acc = -0.0f;\n    for (int p = 0; p < P; ++p) acc"),
    ("two-step-skips-last-slab", "for (int p = 0; p < P; ++p)\n        acc = acc + deq_one",
     "for (int p = 0; p < P - 1; ++p)\n        acc = acc + deq_one"),
    ("eps-outside-sqrt", "sqrt(ss / (double)H + (double)eps)", "(sqrt(ss / (double)H) + (double)eps)"),
    ("mean-over-h-minus-1", "ss / (double)H", "ss / (double)(H - 1)"),
    ("gamma-dropped", "or_f64_to_bf16((v * inv) * g)", "or_f64_to_bf16(v * inv)"),
    ("bf16-round-half-up", "u += 0x7FFFu + lsb;", "u += 0x8000u;"),
    ("double-rounding-f64", "if ((double)f != d) {", "if (0) {"),
    ("residual-not-added", "float hf = ot[k] + or_bf16_to_f32(rt[k]);", "float hf = ot[k];"),
    ("tag-in-word-0", "w[3] = epoch;", "w[0] = epoch;"),
    ("tag-check-inverted", "if (blocks[4 * b + 3] != epoch) return b;",
     "if (blocks[4 * b + 3] == epoch) return b;"),
    ("qtagged-scale-before-codes", "memcpy(payload + cb, &scales[g], 4);",
     "memcpy(payload, &scales[g], 4);"),
    ("gather-forgets-shard-offset", "out[g0 * G + e] = deq_one(", "out[e] = deq_one("),
    ("gather-shard-size-floor", "int64_t per = (ng + P - 1) / P;\n  for (int j = 0; j < P; ++j) {\n    int64_t g0 = (int64_t)j * per, g1 = g0 + per;\n    if (g1 > ng) g1 = ng;\n    if (g0 >= g1) continue; /* an empty shard */",
     "int64_t per = ng / P ? ng / P : 1;\n  for (int j = 0; j < P; ++j) {\n    int64_t g0 = (int64_t)j * per, g1 = g0 + per;\n    if (g1 > ng) g1 = ng;\n    if (g0 >= g1) continue; /* an empty shard */"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    lib = oracle.build(force=True, src=str(mpath), out=str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            check(orc)
        except (AssertionError, ValueError):
            failed.append(check.__name__)
    assert failed, f"mutant {name} passed every pin"
