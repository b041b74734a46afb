"""Planted mistakes in the oracle must fail its pins.

Each case copies oracle/oracle.c, plants one plausible mistake in the copy (a
dropped term, a wrong sign or index, a transposed operand, a format constant
off by one, a missing step of the selection), builds it with gcc and runs the
pin suite (tests/test_oracle.py) against it in a child process through
IDX_ORACLE_LIB.  An unchanged copy must pass; every mutant must fail a pin
(pytest exit status 1, not a crash).  The mistakes live only in temporary
copies: the oracle itself is never modified.

Not among them: swapping the two nibbles of an MXFP4 byte.  Elements 2i and
2i+1 share a scale block, so the swap permutes q and k alike within every
block and leaves every dot product, hence every score and index, unchanged;
no output can tell the two packings apart.
"""
import os
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")
PINS = os.path.join(ROOT, "tests", "test_oracle.py")

# (what the mistake is, text of oracle.c, the text with the mistake)
MUTANTS = [
    ("dropped ReLU",
     "const double relu = dot[h] > 0.0 ? dot[h] : 0.0;", "const double relu = dot[h];"),
    ("reversed tie rule",
     "return (x->j > y->j) - (x->j < y->j);", "return (x->j < y->j) - (x->j > y->j);"),
    ("e4m3 exponent bias off by one",
     "ldexp(1.0 + (double)mant / 8.0, expo - 7)", "ldexp(1.0 + (double)mant / 8.0, expo - 8)"),
    ("e4m3 subnormal exponent",
     "ldexp((double)mant / 8.0, 1 - 7)", "ldexp((double)mant / 8.0, -7)"),
    ("bf16 mantissa width",
     "ldexp(1.0 + (double)mant / 128.0, expo - 127)",
     "ldexp(1.0 + (double)mant / 256.0, expo - 127)"),
    ("key scale indexed row-relative",
     "out[j - ks] = (double)k_scale[j] * s;", "out[j - ks] = (double)k_scale[j - ks] * s;"),
    ("q heads and dimensions transposed",
     "decode(q, q_sf, (r * (long long)H + h) * D + d, dtype)",
     "decode(q, q_sf, (r * (long long)D + d) * H + h, dtype)"),
    ("row 0's head weights used for every row",
     "s += (double)w[r * H + h] * relu;", "s += (double)w[h] * relu;"),
    ("head sum kept in fp32",
     "        double s = 0.0;\n        for (int h = 0; h < H; ++h) {",
     "        float s = 0.0f;\n        for (int h = 0; h < H; ++h) {"),
    ("bottom-k instead of top-k",
     "out[i] = (int32_t)it[i].j;", "out[i] = (int32_t)it[n - 1 - i].j;"),
    ("selected indices left in score order",
     "    qsort(out, (size_t)take, sizeof(int32_t), by_index);\n", ""),
    ("padding 0 instead of -1",
     "for (long long i = take; i < topk; ++i) out[i] = -1;",
     "for (long long i = take; i < topk; ++i) out[i] = 0;"),
    ("page-table row ignored",
     "v = (long long)table[t * table_stride + page] * page_size + p % page_size;",
     "v = (long long)table[page] * page_size + p % page_size;"),
    ("table-row bound ignored",
     "const int row_ok = t >= 0 && t < table_rows;", "const int row_ok = t >= 0;"),
    ("offset within the page dropped",
     "v = (long long)table[t * table_stride + page] * page_size + p % page_size;",
     "v = (long long)table[t * table_stride + page] * page_size;"),
    ("e2m1 exponent bias",
     "ldexp(1.0 + (double)mant / 2.0, expo - 1)", "ldexp(1.0 + (double)mant / 2.0, expo)"),
    ("e8m0 bias",
     "ldexp(1.0, (int)(code & 0xFF) - 127)", "ldexp(1.0, (int)(code & 0xFF) - 128)"),
    ("q decoded with k's MXFP4 block scales",
     "decode(q, q_sf, (r * (long long)H + h) * D + d, dtype)",
     "decode(q, k_sf, (r * (long long)H + h) * D + d, dtype)"),
    ("MXFP4 scale block found from the byte index",
     "tab_e8m0[sf[i / 32]]", "tab_e8m0[sf[(i >> 1) / 32]]"),
]

CFLAGS = ["-O1", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-pthread"]


def _build(src_text: str, where: str) -> str:
    c = os.path.join(where, "oracle.c")
    so = os.path.join(where, "liboracle.so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", *CFLAGS, "-o", so, c, "-lm"], check=True)
    return so


def _run_pins(lib: str) -> subprocess.CompletedProcess:
    env = dict(os.environ, IDX_ORACLE_LIB=lib, OMP_NUM_THREADS="1")
    return subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q", "-p",
                           "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True,
                          text=True, timeout=600)


def _case(args):
    name, old, new, text, tmp = args
    where = tempfile.mkdtemp(dir=tmp)
    mutated = text if old is None else text.replace(old, new)
    proc = _run_pins(_build(mutated, where))
    return name, proc.returncode, proc.stdout[-400:]


def test_pins_fail_on_every_planted_mistake():
    text = open(SRC).read()
    for name, old, _ in MUTANTS:
        assert text.count(old) == 1, f"mutation '{name}' no longer matches oracle.c"
    cases = [("unchanged copy", None, None)] + MUTANTS
    with tempfile.TemporaryDirectory() as tmp:
        jobs = [(n, o, w, text, tmp) for n, o, w in cases]
        workers = max(1, min(8, (os.cpu_count() or 2)))
        with ThreadPoolExecutor(workers) as ex:
            results = list(ex.map(_case, jobs))
    control = results[0]
    assert control[1] == 0, "the pins fail on an unchanged copy:\n" + control[2]
    survivors = [n for n, rc, _ in results[1:] if rc == 0]
    crashed = [(n, rc) for n, rc, _ in results[1:] if rc not in (0, 1)]
    assert not survivors, f"planted mistakes that no pin catches: {survivors}"
    assert not crashed, f"mutants that crashed instead of failing a pin: {crashed}"
