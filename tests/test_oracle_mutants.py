"""Mutation check of the oracle's pins (CPU only).

Each case below plants one plausible mistake in a private copy of
oracle/oracle.c (a swapped matrix index, a dropped compensation term, a
wrong rounding, an init dropped / applied per element / applied on the
wrong side, a wrong stride...), rebuilds that copy and runs the pins of
tests/test_oracle.py against it in a separate process. Every mutant must
fail at least one pin; the unmutated copy must pass. The real oracle is
never modified.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, [(old, new), ...]): every `old` must occur exactly once in oracle.c.
MUTANTS = [
    ("mat2 entry c11 uses a transposed operand",
     [("c[0] = (uint32_t)((a11 * b11 + a12 * b21) % p);", "c[0] = (uint32_t)((a11 * b11 + a21 * b12) % p);")]),
    ("mat2 entry c12 uses the wrong row",
     [("c[2] = (uint32_t)((a11 * b12 + a12 * b22) % p);", "c[2] = (uint32_t)((a12 * b11 + a22 * b12) % p);")]),
    ("compensation term dropped",
     [("if (fabs(a->s) >= fabs(v)) a->c += (a->s - t) + v;", "if (fabs(a->s) >= fabs(v)) a->c += 0;")]),
    ("bf16 rounding ties away from zero",
     [("double r = nearbyint(ldexp(v, -lsb));", "double r = round(ldexp(v, -lsb));")]),
    ("bf16 keeps one bit too many", [("int lsb = e - 8; ", "int lsb = e - 9; ")]),
    ("max(-0, +0) keeps the left operand",
     [("return signbit(a) ? b : a; /* equal: only", "return a; /* equal: only")]),
    ("abs2 computes abs", [("case ORC_MAP_ABS2: return v * v;", "case ORC_MAP_ABS2: return fabs(v);")]),
    ("no wrap to 32 bits", [("if (bits == 64) {", "if (bits == 64 || bits == 32) {")]),
    ("scan: mat2 init on the right",
     [("if (init) orc_mat2_mul(init, x + 4 * e, a);", "if (init) orc_mat2_mul(x + 4 * e, init, a);")]),
    ("scan: mat2 operands swapped",
     [("orc_mat2_mul(a, x + 4 * k, t);\n            memcpy(a, t, sizeof a);\n            memcpy(y + 4 * k",
       "orc_mat2_mul(x + 4 * k, a, t);\n            memcpy(a, t, sizeof a);\n            memcpy(y + 4 * k")]),
    ("dims: wrong stride of a kept / reduced dimension",
     [("off += (o % p->shape[d]) * p->stride[d];", "off += (o % p->shape[d]) * p->stride[d ? d - 1 : 0];")]),
    ("scan: line stride off by one", [("if (d == dim) st_dim = st;", "if (d == dim) st_dim = st * 1 + (d > 0);")]),
    ("bf16 double rounding through f32", [("float f = (float)q; ", "float f = (float)(float)v; ")]),
    ("reduce: float init dropped",
     [("    if (has_init) ffold_start(&a, init);\n    else if (n > 0) ffold_start(&a, fmap(",
       "    if (0) ffold_start(&a, init);\n    else if (n > 0) ffold_start(&a, fmap(")]),
    ("dims: float init dropped",
     [("        if (has_init) ffold_start(&a, init);\n        else ffold_start(&a, fmap(",
       "        if (0) ffold_start(&a, init);\n        else ffold_start(&a, fmap(")]),
    ("dims: float init applied to every element",
     [("ffold_step(&a, fmap(load_float(x, in_type, base + offset_of(&p, p.red, p.nred, r)), map), op);",
       "ffold_step(&a, fmap(load_float(x, in_type, base + offset_of(&p, p.red, p.nred, r)), map)"
       " + (has_init ? init : 0.0), op);")]),
    ("dims: int init dropped",
     [("        if (has_init) a = wrap((uint64_t)init, acc_bits);\n        else a = imap(",
       "        if (0) a = wrap((uint64_t)init, acc_bits);\n        else a = imap(")]),
    ("dims: int init applied twice",
     [("                      op, acc_bits);\n        out[o] = a;",
       "                      op, acc_bits);\n        out[o] = has_init ? istep(a, wrap((uint64_t)init, acc_bits), op, acc_bits) : a;")]),
    ("dims: mat2 init on the right",
     [("        if (init) memcpy(a, init, sizeof a);\n        else memcpy(a, x + 4 * (base",
       "        if (0) memcpy(a, init, sizeof a);\n        else memcpy(a, x + 4 * (base"),
      ("        memcpy(out + 4 * o, a, sizeof a);",
       "        if (init) { orc_mat2_mul(a, init, t); memcpy(a, t, sizeof a); }\n"
       "        memcpy(out + 4 * o, a, sizeof a);")]),
    ("scan: float init dropped",
     [("        if (has_init) {\n            ffold_start(&a, init);", "        if (0) {\n            ffold_start(&a, init);")]),
    ("scan: float init applied to every element",
     [("ffold_step(&a, load_float(x, in_type, k), op);\n            y[k] = ffold_value(&a);",
       "ffold_step(&a, load_float(x, in_type, k) + (has_init ? init : 0.0), op);\n            y[k] = ffold_value(&a);")]),
    ("scan: float line stride off by one",
     [("            int64_t k = e + j * s.step;\n            ffold_step(&a, load_float(x, in_type, k), op);\n            y[k]",
       "            int64_t k = e + j * (s.step > 1 ? s.step - 1 : 1);\n"
       "            ffold_step(&a, load_float(x, in_type, k), op);\n            y[k]")]),
    ("exclusive int scan stores after the combine",
     [("            y[k] = a;\n            a = istep(a, wrap((uint64_t)load_int(x, in_type, k), acc_bits), op, acc_bits);",
       "            a = istep(a, wrap((uint64_t)load_int(x, in_type, k), acc_bits), op, acc_bits);\n            y[k] = a;")]),
    ("exclusive float scan stores after the combine",
     [("            y[k] = ffold_value(&a);\n            ffold_step(&a, load_float(x, in_type, k), op);",
       "            ffold_step(&a, load_float(x, in_type, k), op);\n            y[k] = ffold_value(&a);")]),
    ("exclusive mat2 scan: operands swapped",
     [("            memcpy(y + 4 * k, a, sizeof a);\n            orc_mat2_mul(a, x + 4 * k, t);",
       "            memcpy(y + 4 * k, a, sizeof a);\n            orc_mat2_mul(x + 4 * k, a, t);")]),
    ("findall: floats selected by sign", [("set = ((const float*)x)[i] != 0.0f;", "set = ((const float*)x)[i] > 0.0f;")]),
    ("findall: only the byte 1 selected", [("set = ((const uint8_t*)x)[i] != 0;", "set = ((const uint8_t*)x)[i] == 1;")]),
    ("reduce2: square of the difference dropped",
     [("case ORC_MAP2_SQDIFF: return (a - b) * (a - b);", "case ORC_MAP2_SQDIFF: return (a - b);")]),
    ("reduce2: integer product uses one source twice",
     [("case ORC_MAP2_MUL: return wrap((uint64_t)a * (uint64_t)b, bits);",
       "case ORC_MAP2_MUL: return wrap((uint64_t)a * (uint64_t)a, bits);")]),
    ("strided view read as dense", [("p->stride[d] = strides ? strides[d] : st;", "p->stride[d] = st;")]),
    ("affine maps composed in the wrong order",
     [("uint64_t b = ((uint64_t)g[0] * f[1] + g[1]) % p;", "uint64_t b = ((uint64_t)f[0] * g[1] + f[1]) % p;")]),
    ("affine exclusive scan stores the inclusive value",
     [("if (exclusive) memcpy(y + 2 * i, a, sizeof a);", "if (0) memcpy(y + 2 * i, a, sizeof a);"),
      ("if (!exclusive) memcpy(y + 2 * i, a, sizeof a);", "memcpy(y + 2 * i, a, sizeof a);")]),
]


def _copy_tree(dst: str) -> None:
    shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(dst, "oracle"),
                    ignore=shutil.ignore_patterns("_build", "__pycache__"))
    os.makedirs(os.path.join(dst, "tests"))
    for f in ("test_oracle.py", "conftest.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), os.path.join(dst, "tests", f))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(dst, "tests", "golden"))
    for f in ("synth.py", "pytest.ini"):
        shutil.copy(os.path.join(ROOT, f), os.path.join(dst, f))


def _run_pins(edits) -> int:
    with tempfile.TemporaryDirectory(prefix="orc_mut_") as d:
        _copy_tree(d)
        path = os.path.join(d, "oracle", "oracle.c")
        src = open(path).read()
        for old, new in edits:
            assert src.count(old) == 1, f"mutation site not unique or missing: {old!r}"
            src = src.replace(old, new)
        with open(path, "w") as f:
            f.write(src)
        r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                            "tests/test_oracle.py"], cwd=d, capture_output=True, text=True, timeout=600)
        return r.returncode


def test_every_planted_mistake_fails_a_pin():
    cases = [("unmutated", [])] + MUTANTS
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        rcs = dict(zip([c[0] for c in cases], ex.map(lambda c: _run_pins(c[1]), cases)))
    assert rcs["unmutated"] == 0, "the pins fail on an unmodified copy of the oracle"
    survivors = [name for name, rc in rcs.items() if name != "unmutated" and rc == 0]
    assert not survivors, f"mutants that no pin catches: {survivors}"


if __name__ == "__main__":
    pytest.main([__file__, "-q"])
