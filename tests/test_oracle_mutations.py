"""The oracle's pins must catch plausible mistakes.

Each case below plants one mistake in a copy of oracle/oracle.c (in a
temporary directory, on the CPU), rebuilds that copy and runs the pin suite
against it.  The pin suite has to fail for every planted mistake.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = [
    ("accept test with p and q swapped", "(double)u[i] * qx < px) {", "(double)u[i] * px < qx) {"),
    ("residual q - p instead of p - q", "double d = p[t] - q[t];", "double d = q[t] - p[t];"),
    ("residual without the clamp at zero", "w[t] = d > 0.0 ? d : 0.0;", "w[t] = d;"),
    ("bonus draw uses the resample uniform", "o->drawn = inverse_cdf(p, V, (double)u[k], &mg);",
     "o->drawn = inverse_cdf(p, V, (double)u[k + 1], &mg);"),
    ("bonus drawn from the last draft position's row", "const double* p = ROW(k);", "const double* p = ROW(k - 1);"),
    ("temperature multiplies instead of divides", "r[t].z = l / temperature;", "r[t].z = l * temperature;"),
    ("top-p counts the token's own mass", "if (!(before < top_p)) break;",
     "if (!(before + exp(r[t].z - m) / zk < top_p) && t > 0) break;"),
    ("top-k keeps one extra token", "n_topk = (top_k > 0 && top_k < V) ? top_k : V;",
     "n_topk = (top_k > 0 && top_k < V) ? top_k + 1 : V;"),
    ("ties ranked by higher index first", "return (x->idx < y->idx) ? -1 : (x->idx > y->idx);",
     "return (x->idx > y->idx) ? -1 : (x->idx < y->idx);"),
    ("inverse CDF picks the index before the crossing", "return t;\n    }\n  }\n  if (margin) *margin = 0.0;",
     "return t > 0 ? t - 1 : t;\n    }\n  }\n  if (margin) *margin = 0.0;"),
    ("greedy argmax keeps the last of equal maxima", "    if (v > bv) {", "    if (v >= bv) {"),
    ("tree compares a node with its own row", "agreed[j] = agreed[pj] && tok[j] == am[pj];",
     "agreed[j] = agreed[pj] && tok[j] == am[j];"),
    ("tree prefers the highest index among equally deep nodes",
     "if (agreed[j] && depth[j] > depth[best]) best = j;", "if (agreed[j] && depth[j] >= depth[best]) best = j;"),
    ("expected tokens drops the last power", "for (i = 0; i <= gamma; ++i) {", "for (i = 0; i < gamma; ++i) {"),
    ("tree sibling tested against p, not the residual", "if ((double)u[j] * q[x] < r[x]) {",
     "if ((double)u[j] * q[x] < p[x]) {"),
    ("tree accept test takes the draw uniform", "if ((double)u[j] * q[x] < r[x]) {",
     "if ((double)u[0] * q[x] < r[x]) {"),
    ("tree residual subtracts p", "double d = r[t] - q[t];", "double d = r[t] - p[t];"),
    ("tree residual left unnormalised", "for (t = 0; t < V; ++t) r[t] /= s;", "s = s;"),
    ("tree final draw from p", "drawn = inverse_cdf(r, V, (double)u[0], &mg);",
     "drawn = inverse_cdf(p, V, (double)u[0], &mg);"),
    ("tree walk keeps the parent's rows after an acceptance", "        v = accepted;\n        continue;",
     "        (void)accepted;\n        continue;"),
    ("tree siblings tried from the last", "for (j = v + 1; j < N && n_test > 0; ++j) {",
     "for (j = N - 1; j > v && n_test > 0; --j) {"),
    ("boundary flags 10x wider", "#define BOUNDARY_EPS 1e-6", "#define BOUNDARY_EPS 1e-5"),
    ("boundary flags 10x narrower", "#define BOUNDARY_EPS 1e-6", "#define BOUNDARY_EPS 1e-7"),
    ("top-p cut re-scan skipped", "if (differs) o.flags |= OFLAG_CUT_BOUNDARY;", "(void)differs;"),
    ("top-p cut flagged whether or not it matters", "if (differs) o.flags |= OFLAG_CUT_BOUNDARY;",
     "o.flags |= OFLAG_CUT_BOUNDARY;"),
    ("accept flag tested on q/p", "double mg = fabs((double)u[i] - px / qx);", "double mg = fabs((double)u[i] - qx / px);"),
    ("draw flag measured against the far edge only", "if (margin) *margin = (a < b ? a : b) / s;",
     "if (margin) *margin = b / s;"),
    ("tree degenerate residual not put back to p",
     "flags |= OFLAG_DEGENERATE;\n          for (t = 0; t < V; ++t) r[t] = p[t];",
     "flags |= OFLAG_DEGENERATE;"),
]

PIN_FILES = ("test_oracle_pins.py", "test_oracle_tree_sample.py", "test_oracle_boundary_pins.py")


def _run_mutated(tmp_root, src, idx, name, old, new):
    assert src.count(old) == 1, f"mutation site not unique: {name}"
    d = os.path.join(tmp_root, f"m{idx}")
    shutil.copytree(os.path.join(ROOT, "workloads"), os.path.join(d, "workloads"))
    os.makedirs(os.path.join(d, "oracle"))
    for f in ("__init__.py", "exact.py"):
        shutil.copy(os.path.join(ROOT, "oracle", f), os.path.join(d, "oracle", f))
    with open(os.path.join(d, "oracle", "oracle.c"), "w") as fh:
        fh.write(src.replace(old, new))
    os.makedirs(os.path.join(d, "tests"))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(d, "tests", "golden"))
    for f in ("conftest.py",) + PIN_FILES:
        shutil.copy(os.path.join(ROOT, "tests", f), os.path.join(d, "tests", f))
    env = dict(os.environ, PYTHONPATH=d, PYTHONDONTWRITEBYTECODE="1", OMP_NUM_THREADS="1")
    r = subprocess.run(
        [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "--rootdir", d,
         *[os.path.join(d, "tests", f) for f in PIN_FILES]],
        cwd=d, env=env, capture_output=True, text=True, timeout=900,
    )
    return name, r.returncode, r.stdout[-1500:] + r.stderr[-1500:]


def test_pins_catch_every_planted_mistake(tmp_path):
    with open(os.path.join(ROOT, "oracle", "oracle.c")) as f:
        src = f.read()
    workers = max(1, min(len(MUTATIONS), os.cpu_count() or 1))
    with ThreadPoolExecutor(workers) as pool:
        results = list(pool.map(lambda a: _run_mutated(str(tmp_path), src, *a),
                                [(i, *m) for i, m in enumerate(MUTATIONS)]))
    survivors = [(name, log) for name, rc, log in results if rc != 1]
    assert not survivors, "planted mistakes not caught:\n" + "\n\n".join(f"{n}:\n{l}" for n, l in survivors)
