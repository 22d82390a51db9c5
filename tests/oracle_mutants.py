"""Planted mistakes for the oracle's pin tests.

The oracle's sources hold the plain definition and no test hook.  A mutant is
a copy of one of those sources with one mistake planted by textual edits
(each edit's text must occur exactly once in the source, so an edit that no
longer applies fails loudly); the C mutants are compiled on their own, the
Python mutants imported on their own, and the pins run against them
unchanged.  Every mutant here must fail at least one pin.
"""
from __future__ import annotations

import contextlib
import hashlib
import importlib.util
import os
import tempfile

import oracle

_ORACLE_DIR = os.path.dirname(os.path.abspath(oracle.__file__))
C_SOURCE = os.path.join(_ORACLE_DIR, "cfa_oracle.c")
PY_INIT = os.path.join(_ORACLE_DIR, "__init__.py")
PY_ROWSPARSE = os.path.join(_ORACLE_DIR, "rowsparse.py")

# id: (what the mistake is, [(text in cfa_oracle.c, replacement), ...])
C_MUTANTS = {
    1: ("chunk mask lets a row see one future key",
        [("const int nc = t + 1;", "const int nc = t + 2 <= lc ? t + 2 : lc;")]),
    2: ("softmax scale dropped from dQ",
        [("const double f = scale * dsj;", "const double f = dsj;")]),
    3: ("wrong sign of delta in dS",
        [("const double dsj = P[j] * (dpj - dl);", "const double dsj = P[j] * (dpj + dl);"),
         ("const double ds = p * (dp - delta[(size_t)hh * lc + t]);",
          "const double ds = p * (dp + delta[(size_t)hh * lc + t]);")]),
    4: ("dV accumulates dS instead of P",
        [("if (dv) for (int c = 0; c < d; ++c) dv[c] += p * dot_[c];",
          "if (dv) for (int c = 0; c < d; ++c) dv[c] += ds * dot_[c];")]),
    5: ("softmax scale dropped from dK",
        [("const double fk = scale * ds;", "const double fk = ds;")]),
    6: ("dQ multiplies dS by V instead of K",
        [("dqt[c] += f * kj[c];", "dqt[c] += f * vj[c];")]),
    7: ("LSE taken in log2",
        [("const double L = m + log(sum);", "const double L = m + log2(sum);")]),
    8: ("O sums K rows instead of V rows",
        [("ot[c] += P[j] * vj[c];",
          "ot[c] += P[j] * (j < lp ? kp + (size_t)j * d : kc + (size_t)(j - lp) * d)[c];")]),
    9: ("prefix dropped from the softmax denominator",
        [("for (int j = 0; j < n; ++j) sum += exp(S[j] - m);",
          "for (int j = lp; j < n; ++j) sum += exp(S[j] - m);")]),
    10: ("dK/dV sum only the first head of the group",
         [("for (int hh = 0; hh < g; ++hh) {      /* the group's query heads */",
           "for (int hh = 0; hh < 1; ++hh) {")]),
    11: ("q8_0 scale read as bf16 bits",
          [("static double half_bits_to_double(uint16_t h)\n{\n",
            "static double half_bits_to_double(uint16_t h)\n{\n"
            "    { uint32_t u = (uint32_t)h << 16; float f; memcpy(&f, &u, 4); return (double)f; }\n")]),
    12: ("q8_0 codes read unsigned",
         [("int qi = (int)(int8_t)blk[2 + i];", "int qi = (int)blk[2 + i];")]),
    13: ("softmax scale dropped from the prefix dK",
         [("const double fkp = scale * ds;", "const double fkp = ds;")]),
    14: ("prefix dK/dV sum only the first head of the group",
         [("for (int hh = 0; hh < g; ++hh) {      /* every query head of the group */",
           "for (int hh = 0; hh < 1; ++hh) {")]),
    15: ("q8_0 encoder rounds halves to even",
         [("q = (int)roundf(r);", "q = (int)rintf(r);")]),
    16: ("q8_0 encoder divides by the fp16-rounded scale",
         [("const float r = v[i] / d;", "const float r = v[i] / (float)half_bits_to_double(dh);")]),
}

# Python mutants: (what the mistake is, source file, [(text, replacement), ...])
PY_MUTANTS = {
    "head_map": ("query head h read from KV head h % hkv instead of h // g", PY_INIT,
                 [("heads = list(range(hk * g, (hk + 1) * g))",
                   "heads = [h for h in range(hq) if h % hkv == hk]")]),
    "dw_rows": ("dW reads the first n_keep rows of X instead of the kept ones", PY_ROWSPARSE,
                [("rows = xs[idx]", "rows = xs[: len(idx)]")]),
    "dw_transposed": ("dW returned transposed (X[keep]^T dY_keep)", PY_ROWSPARSE,
                      [("dw = dy.T @ rows", "dw = rows.T @ dy")]),
    "dx_rows": ("dX writes row i instead of row keep[i]", PY_ROWSPARSE,
                [("out[idx] = vals", "out[: len(idx)] = vals")]),
    "dx_transposed": ("dX multiplies by W^T instead of W", PY_ROWSPARSE,
                      [("vals = dy @ ws", "vals = dy @ ws.T")]),
}

_DIR = None


def _edited(path: str, edits) -> str:
    with open(path) as f:
        src = f.read()
    for old, new in edits:
        n = src.count(old)
        assert n == 1, f"edit text found {n} times in {os.path.basename(path)}: {old!r}"
        src = src.replace(old, new)
    return src


def _workdir() -> str:
    global _DIR
    if _DIR is None:
        _DIR = tempfile.mkdtemp(prefix="cfa_oracle_mutants_")
    return _DIR


def c_mutant_library(n: int) -> str:
    """Compile C mutant `n`; returns the shared library's path."""
    src = _edited(C_SOURCE, C_MUTANTS[n][1])
    tag = hashlib.sha1(src.encode()).hexdigest()[:12]
    out = os.path.join(_workdir(), f"libcfa_oracle_m{n}_{tag}.so")
    if not os.path.exists(out):
        c_path = os.path.join(_workdir(), f"cfa_oracle_m{n}_{tag}.c")
        with open(c_path, "w") as f:
            f.write(src)
        oracle.compile_library(c_path, out)
    return out


@contextlib.contextmanager
def c_mutant(n: int):
    """Within the block, every oracle function runs on C mutant `n`."""
    lb = oracle.load(c_mutant_library(n))
    oracle.lib()  # the plain library, so that it is the one restored afterwards
    saved = oracle._lib
    oracle._lib = lb
    try:
        yield
    finally:
        oracle._lib = saved


def py_mutant(name: str):
    """Python mutant `name`, imported as a module of its own (the original
    module's file name is kept, so its paths resolve as before)."""
    _, path, edits = PY_MUTANTS[name]
    src = _edited(path, edits)
    spec = importlib.util.spec_from_loader(f"oracle_mutant_{name}", loader=None, origin=path)
    mod = importlib.util.module_from_spec(spec)
    mod.__file__ = path
    exec(compile(src, path, "exec"), mod.__dict__)
    return mod
