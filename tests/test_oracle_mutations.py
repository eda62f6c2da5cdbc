"""The pins catch plausible mistakes in the oracle (CPU).

Each case plants one mistake in a copy of oracle/fathom_oracle.c (an offset, a
wrong sign or index, a dropped term, a transposed operand, a wrong rounding or
tie rule), builds the copy, and runs the pins of test_oracle_pins.py against
it in a child process: the pins must fail.  The real oracle is never
modified; a mistake the pins let through would mean an unpinned part.

Two plausible edits are left out because they change nothing: dropping the
exact-floor corrections in oracle_code (an fp32 key and an fp16-derived step
put the fp64 quotient at least 2^-25 away, relatively, from any integer it
is not equal to, far beyond its 2^-53 rounding), and centring the second
factor of a covariance term on the wrong channel's mean (the other factor
sums to zero over the rows)."""
import concurrent.futures as cf
import os
import subprocess
import sys

import pytest

from oracle import oracle as O

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
ORACLE_C = os.path.join(ROOT, "oracle", "fathom_oracle.c")
PINS = os.path.join(HERE, "test_oracle_pins.py")

# (what the mistake is, original text, mistaken text): the first occurrence is replaced
MUTANTS = [
    ("code offset by one", "return (int)f + 8;", "return (int)f + 7;"),
    ("quantiser step a/16", "double s = a16 / 8.0;                           /* exact */",
     "double s = a16 / 16.0;"),
    ("scale not rounded to fp16", "double a16 = oracle_round_fp16(a);", "double a16 = a;"),
    ("fp16 rounding truncates", "double r = rint(a / quantum);", "double r = floor(a / quantum);"),
    ("plane 0 is the LSB", "uint64_t bit = (uint64_t)((c >> (3 - p)) & 1);", "uint64_t bit = (uint64_t)((c >> p) & 1);"),
    ("token i at bit 63 - i", "P[p] |= bit << (i - i0);", "P[p] |= bit << (63 - (i - i0));"),
    ("mid-rise offset dropped", "return ((double)c_t + 0.5 - half) * a16 / half;",
     "return ((double)c_t - half) * a16 / half;"),
    ("mid-rise scale halved", "return ((double)c_t + 0.5 - half) * a16 / half;",
     "return ((double)c_t + 0.5 - half) * a16 / (2.0 * half);"),
    ("prefix read LSB first", "c_t = (c_t << 1) | (int)((w >> bit) & 1u);",
     "c_t = c_t | ((int)((w >> bit) & 1u) << p);"),
    ("importance |q| not q^2", "s = s + x * x;", "s = s + fabs(x);"),
    ("importance without Var", "g[j] = s * (double)var[j];", "g[j] = s;"),
    ("depth breakpoints at 2^(2m)", "if (g >= theta * ldexp(1.0, 2 * m + 1)) ++t;",
     "if (g >= theta * ldexp(1.0, 2 * m)) ++t;"),
    ("arithmetic instead of geometric bisection", "double mid = sqrt(lo * hi);", "double mid = 0.5 * (lo + hi);"),
    ("plan from the infeasible end", "for (int j = 0; j < D; ++j) depth[j] = (uint8_t)oracle_depth_of(g[j], hi);\n    *theta = hi;",
     "for (int j = 0; j < D; ++j) depth[j] = (uint8_t)oracle_depth_of(g[j], lo);\n    *theta = lo;"),
    ("bisection step inverted", "if (s <= B) hi = mid; else lo = mid;", "if (s < B) hi = mid; else lo = mid;"),
    ("fixed plan keeps the smallest g", "if (g[i] > g[j] || (g[i] == g[j] && i < j)) ++better;",
     "if (g[i] < g[j] || (g[i] == g[j] && i < j)) ++better;"),
    ("run length of one plane", "r[1] = t * nb;", "r[1] = nb;"),
    ("scores skip channel 0", "int t = depth[(size_t)u * D + j];", "int t = j == 0 ? 0 : depth[(size_t)u * D + j];"),
    ("scores with head 0's query", "s += (double)q[((size_t)u * G + h) * D + j] * oracle_dequant(c_t, t, a16);",
     "s += (double)q[((size_t)u * G + 0) * D + j] * oracle_dequant(c_t, t, a16);"),
    ("ties to the higher index", "return (a->i < b->i) ? -1 : (a->i > b->i);   /* R9 */",
     "return (a->i > b->i) ? -1 : (a->i < b->i);"),
    ("recent tokens not forced", "if (i < n_sink || i >= n - n_recent) { forced[i] = 1; ++nf; }",
     "if (i < n_sink) { forced[i] = 1; ++nf; }"),
    ("attention without 1/sqrt(D)", "double scale = 1.0 / sqrt((double)D);", "double scale = 1.0;"),
    ("variance with ddof 0", "var[j] = s / (double)(m - 1);", "var[j] = s / (double)m;"),
    ("greedy adds to the smallest drop", "if (best == -1 || drop > best_drop) { best = l; best_drop = drop; }",
     "if (best == -1 || drop < best_drop) { best = l; best_drop = drop; }"),
    ("exact scores transposed", "d += (double)q[(size_t)h * D + j] * (double)keys[(size_t)i * D + j];",
     "d += (double)q[(size_t)h * D + j] * (double)keys[(size_t)j * D + (i % D)];"),
    ("code clipped at 14", "if (f > 7.0) f = 7.0;", "if (f > 6.0) f = 6.0;"),
    ("subnormal fp16 scale encoded as normal", "if (v < ldexp(1.0, -14)) return (uint16_t)(v / ldexp(1.0, -24));", ""),
    ("fp16 exponent bias off by one", "return sgn * ldexp(1024.0 + mant, exp - 25);",
     "return sgn * ldexp(1024.0 + mant, exp - 24);"),
    ("bf16 widened from the low half", "uint32_t u = ((uint32_t)b) << 16;", "uint32_t u = ((uint32_t)b);"),
    ("gather reads the next word", "stage_planes[r[2] + w] = store_planes[r[0] + w];",
     "stage_planes[r[2] + w] = store_planes[r[0] + w + 1];"),
    ("staged scores take the wrong block's scale",
     "double a16 = oracle_fp16_value(stage_scales[r[5] + (uint32_t)(i / 64)]);",
     "double a16 = oracle_fp16_value(stage_scales[r[5]]);"),
    ("keys rebuilt from three planes", "keys[(size_t)i * D + j] = oracle_dequant(c, 4, oracle_fp16_value(scales[(size_t)j * cb + beta]));",
     "keys[(size_t)i * D + j] = oracle_dequant(c >> 1, 3, oracle_fp16_value(scales[(size_t)j * cb + beta]));"),
    ("attention over the rebuilt keys without 1/sqrt(D)",
     "double scale = 1.0 / sqrt((double)D);\n    for (int h = 0; h < G; ++h) {\n        double mx = -INFINITY;\n"
     "        for (int r = 0; r < k; ++r) {\n            int i = idx[(size_t)h * k + r];\n            double d = 0.0;\n"
     "            for (int j = 0; j < D; ++j)\n                d += (double)q[(size_t)h * D + j] * keys[",
     "double scale = 1.0;\n    for (int h = 0; h < G; ++h) {\n        double mx = -INFINITY;\n"
     "        for (int r = 0; r < k; ++r) {\n            int i = idx[(size_t)h * k + r];\n            double d = 0.0;\n"
     "            for (int j = 0; j < D; ++j)\n                d += (double)q[(size_t)h * D + j] * keys["),
    ("calibration mean over m - 1", "mean[j] = s / (double)m;", "mean[j] = s / (double)(m - 1);"),
    ("covariance with ddof 0", "cov[(size_t)a * D + b] = s / (double)(m - 1);", "cov[(size_t)a * D + b] = s / (double)m;"),
    ("Jacobi rotation sign flipped", "A[(size_t)x * D + p] = c * axp - s * axr;", "A[(size_t)x * D + p] = c * axp + s * axr;"),
    ("eigenvalues ascending", "for (int b = a + 1; b < D; ++b) if (lam[b] > lam[best]) best = b;",
     "for (int b = a + 1; b < D; ++b) if (lam[b] < lam[best]) best = b;"),
    ("keys rotated without centring", "s += ((double)keys[(size_t)i * D + j] - mu[j]) * V[(size_t)j * D + c];",
     "s += (double)keys[(size_t)i * D + j] * V[(size_t)j * D + c];"),
    ("queries rotated by V transposed", "for (int j = 0; j < D; ++j) s += (double)q[(size_t)h * D + j] * V[(size_t)j * D + c];",
     "for (int j = 0; j < D; ++j) s += (double)q[(size_t)h * D + j] * V[(size_t)c * D + j];"),
    ("auto bracket too narrow", "lo = gmin / 512.0;", "lo = gmin / 8.0;"),
    ("staging offsets skip a word", "dst_w += r[1];", "dst_w += r[1] + (r[1] > 0);"),
    ("scales staged for inactive channels", "r[4] = t > 0 ? nb : 0;", "r[4] = nb;"),
    ("one winner too few", "for (int r = 0; r < k - nf; ++r) out[o++] = c[r].i;",
     "for (int r = 0; r + 1 < k - nf; ++r) out[o++] = c[r].i;\n        if (k - nf > 0) out[o++] = c[m - 1].i;"),
    ("softmax not normalised", "for (int j = 0; j < D; ++j) out[(size_t)h * D + j] /= den;", ""),
    ("fixed plan ignores its depth", "depth[j] = (uint8_t)(better < n_sel ? t_fixed : 0);",
     "depth[j] = (uint8_t)(better < n_sel ? 4 : 0);"),
    ("depth ties round down", "if (g >= theta * ldexp(1.0, 2 * m + 1)) ++t;", "if (g > theta * ldexp(1.0, 2 * m + 1)) ++t;"),
    ("eigenvector sign rule inverted", "if (V[(size_t)arg * D + c] < 0.0)", "if (V[(size_t)arg * D + c] > 0.0)"),
    ("sink tokens not forced", "if (i < n_sink || i >= n - n_recent) { forced[i] = 1; ++nf; }",
     "if (i >= n - n_recent) { forced[i] = 1; ++nf; }"),
    ("budget-not-binding case ignored", "if (total_depth(D, g, lo) <= B) {  /* budget not binding */", "if (0) {"),
    ("exact scores miss the last channel",
     "for (int j = 0; j < D; ++j)\n                d += (double)q[(size_t)h * D + j] * (double)keys[(size_t)i * D + j];",
     "for (int j = 0; j + 1 < D; ++j)\n                d += (double)q[(size_t)h * D + j] * (double)keys[(size_t)i * D + j];"),
    ("importance over one head", "for (int h = 0; h < G; ++h) {\n            double x",
     "for (int h = 0; h < 1; ++h) {\n            double x"),
    ("channels with g = 0 read", "if (g >= theta * ldexp(1.0, 2 * m + 1)) ++t;",
     "if (g >= theta * ldexp(1.0, 2 * m + 1) || g == 0.0) ++t;"),
    ("selection keeps the lowest scores", "if (a->s > b->s) return -1;          /* score descending */",
     "if (a->s < b->s) return -1;"),
    ("attention with head 0's query", "d += (double)q[(size_t)h * D + j] * oracle_bf16_value(krows[(size_t)i * D + j]);",
     "d += (double)q[j] * oracle_bf16_value(krows[(size_t)i * D + j]);"),
    ("rotated keys scaled", "out[(size_t)i * D + c] = (float)s;", "out[(size_t)i * D + c] = (float)(s * (1.0 + 1e-6));"),
    ("greedy starts one level up", "int *lev = (int *)calloc((size_t)layers, sizeof(int));",
     "int *lev = (int *)calloc((size_t)layers, sizeof(int));\n    for (int l = 0; l < layers && levels > 1; ++l) lev[l] = 1;"),
    ("greedy ties to the higher layer", "if (best == -1 || drop > best_drop) { best = l; best_drop = drop; }",
     "if (best == -1 || drop >= best_drop) { best = l; best_drop = drop; }"),
]

CHILD = r"""
import ctypes, importlib.util, itertools, sys
sys.path.insert(0, {root!r})
from oracle import oracle as O
L = ctypes.CDLL(sys.argv[1])
for name, (res, args) in O._SIGS.items():
    fn = getattr(L, name)
    fn.restype = res
    fn.argtypes = args
O._lib = L
spec = importlib.util.spec_from_file_location("pins", {pins!r})
pins = importlib.util.module_from_spec(spec)
spec.loader.exec_module(pins)
tests = [getattr(pins, n) for n in dir(pins) if n.startswith("test_")]
tests.sort(key=lambda f: f.__code__.co_firstlineno)
for f in tests:
    calls = [()]
    for m in getattr(f, "pytestmark", []):
        if m.name == "parametrize":
            names, values = m.args[0], m.args[1]
            single = "," not in names
            calls = [tuple([v]) if single else tuple(v) for v in values]
    for args in calls:
        try:
            f(*args)
        except BaseException as e:
            print("KILLED by", f.__name__, type(e).__name__)
            sys.exit(0)
print("SURVIVED")
"""


def _run_mutant(tmp_dir, idx, old, new):
    src = open(ORACLE_C, encoding="utf-8").read()
    assert old in src, f"mutant {idx}: text not found"
    path_c = os.path.join(tmp_dir, f"mutant{idx}.c")
    path_so = os.path.join(tmp_dir, f"mutant{idx}.so")
    open(path_c, "w", encoding="utf-8").write(src.replace(old, new, 1))
    subprocess.run(["gcc", *O.CFLAGS, "-o", path_so, path_c, "-lm"], check=True, capture_output=True)
    code = CHILD.format(root=ROOT, pins=PINS)
    r = subprocess.run([sys.executable, "-c", code, path_so], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    if r.returncode != 0:      # a crash is a failing pin too
        return f"KILLED by a crash (exit {r.returncode})"
    return r.stdout.strip().splitlines()[-1] if r.stdout.strip() else "no output"


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    O.build()
    tmp = str(tmp_path_factory.mktemp("mutants"))
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
        futs = [ex.submit(_run_mutant, tmp, i, old, new) for i, (_, old, new) in enumerate(MUTANTS)]
        return [f.result() for f in futs]


def test_the_real_oracle_passes_the_pins(tmp_path):
    so = O.build()
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, pins=PINS), so], cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("SURVIVED"), r.stdout[-2000:] + r.stderr[-2000:]


@pytest.mark.parametrize("i", range(len(MUTANTS)), ids=[m[0] for m in MUTANTS])
def test_a_planted_mistake_fails_a_pin(outcomes, i):
    assert outcomes[i].startswith("KILLED"), f"{MUTANTS[i][0]}: {outcomes[i]}"
