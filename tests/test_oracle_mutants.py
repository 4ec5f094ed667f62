"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a scratch copy of oracle.c (a transposed
ratio, a flipped residual sign, T multiplied instead of divided, a wrong row
or slot index, ...), rebuilds it there and runs the pin suite against the
copy: at least one pin has to fail.  Nothing here touches the real oracle or
any GPU code.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = [
    ("return u < fmin(1.0, px / qx);", "return u < fmin(1.0, qx / px);"),
    ("r[j] = fmax(p[j] - q[j], 0.0);", "r[j] = fmax(q[j] - p[j], 0.0);"),
    ("- m) / T);", "- m) * T);"),
    ("fallbacks += residual(p, q, V, r);", "memcpy(r, p, (size_t)V * sizeof *r);"),
    ("        r[j] /= S;", "        r[j] /= 1.0;"),
    ("if (x > m)", "if (x < m)"),
    ("if (u < C) {", "if (u < Cprev) {"),
    ("return px > 0.0;", "return 1;"),
    ("orow[j] = tokens[(size_t)b * Kmax + j];", "orow[j] = tokens[(size_t)b * Kmax + 0];"),
    ("const float u = uniforms[(size_t)b * (Kmax + 1) + Kb];",
     "const float u = uniforms[(size_t)b * (Kmax + 1) + nacc];"),
    ("const size_t doff = ((size_t)b * Kmax + i) * (size_t)V;\n            if (x < 0",
     "const size_t doff = ((size_t)b * (Kmax + 1) + i) * (size_t)V;\n            if (x < 0"),
    ("if (x != g) { rejected = 1; break; }", "if (x == g) { rejected = 1; break; }"),
    ("if (logit_at(base, dtype, off + (size_t)j) == m) {",
     "if (logit_at(base, dtype, off + (size_t)j) == m && j > 0) {"),
    # the tie flag (parity exempts the sequences it marks)
    ("if (fabs(u - Cprev) < ORC_TIE_BAND || fabs(u - C) < ORC_TIE_BAND)", "if (1)"),   # every draw flagged
    ("#define ORC_TIE_BAND 1e-6", "#define ORC_TIE_BAND 1e-3"),                        # a band 1000x wider
    ("if (q[x] > 0.0 && fabs((double)u - p[x] / q[x]) < ORC_TIE_BAND)", "if (0)"),     # accept ties dropped
    ("if (q[x] > 0.0 && fabs((double)u - p[x] / q[x]) < ORC_TIE_BAND)", "if (q[x] > 0.0)"),  # every test flagged
    ("fabs(u - Cprev) < ORC_TIE_BAND || fabs(u - C)", "fabs(u - Cprev) < ORC_TIE_BAND && fabs(u - C)"),
    ("if (fabs(u - Cprev) < ORC_TIE_BAND || ", "if ("),                                 # lower boundary dropped
    ("|| fabs(u - C) < ORC_TIE_BAND)", ")"),                                            # upper boundary dropped
]


# token-tree verification (oracle_tree_verify), against tests/test_oracle_tree.py
TREE_MUTANTS = [
    ("                if (S > 0.0)", "                if (S < 0.0)"),          # no residual after a rejection
    ("if (keep((double)u, r[x], q[x])) {", "if (keep((double)u, p[x], q[x])) {"),   # siblings tested against p
    ("const float u0 = uniforms[row0];", "const float u0 = uniforms[row0 + 1];"),  # wrong final uniform
    ("                    if (x == g) {", "                    if (x != g) {"),     # greedy test flipped
    ("out_tokens[row0 + j] = tokens[row0 + path[j]];", "out_tokens[row0 + j] = tokens[row0 + j + 1];"),
    ("if (q[x] > 0.0 && fabs((double)u - r[x] / q[x]) < ORC_TIE_BAND)", "if (0)"),    # child ties dropped
    ("if (q[x] > 0.0 && fabs((double)u - r[x] / q[x]) < ORC_TIE_BAND)",
     "if (q[x] > 0.0 && fabs((double)u - p[x] / q[x]) < ORC_TIE_BAND)"),              # band around p/q, not R/q
]


def _run_pins(tmp_path, before, after, pins):
    src = open(os.path.join(ROOT, "oracle", "oracle.c")).read()
    assert before in src, "mutation site no longer present in oracle.c"
    for sub in ("oracle", "workloads"):
        shutil.copytree(os.path.join(ROOT, sub), tmp_path / sub,
                        ignore=shutil.ignore_patterns("*.so", "__pycache__"))
    os.makedirs(tmp_path / "tests")
    for f in ("conftest.py", pins):
        shutil.copy(os.path.join(ROOT, "tests", f), tmp_path / "tests" / f)
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), tmp_path / "tests" / "golden")
    (tmp_path / "oracle" / "oracle.c").write_text(src.replace(before, after, 1))
    return subprocess.run([sys.executable, "-m", "pytest", f"tests/{pins}", "-q",
                           "-x", "-p", "no:cacheprovider"], cwd=tmp_path, capture_output=True,
                          text=True, timeout=600)


@pytest.mark.parametrize("before,after", TREE_MUTANTS, ids=[f"t{i}" for i in range(len(TREE_MUTANTS))])
def test_tree_pins_detect_planted_mistake(tmp_path, before, after):
    r = _run_pins(tmp_path, before, after, "test_oracle_tree.py")
    assert r.returncode != 0, "no tree pin failed for mutant:\n" + after + "\n" + r.stdout[-2000:]


@pytest.mark.parametrize("before,after", MUTANTS, ids=[f"m{i}" for i in range(len(MUTANTS))])
def test_pins_detect_planted_mistake(tmp_path, before, after):
    src = open(os.path.join(ROOT, "oracle", "oracle.c")).read()
    assert before in src, "mutation site no longer present in oracle.c"
    for sub in ("oracle", "workloads"):
        shutil.copytree(os.path.join(ROOT, sub), tmp_path / sub,
                        ignore=shutil.ignore_patterns("*.so", "__pycache__"))
    os.makedirs(tmp_path / "tests")
    for f in ("conftest.py", "test_oracle_pins.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), tmp_path / "tests" / f)
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), tmp_path / "tests" / "golden")
    (tmp_path / "oracle" / "oracle.c").write_text(src.replace(before, after, 1))
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle_pins.py", "-q",
                        "-x", "-p", "no:cacheprovider"], cwd=tmp_path, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode != 0, "no pin failed for mutant:\n" + after + "\n" + r.stdout[-2000:]
