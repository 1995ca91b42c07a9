"""The oracle's pins are strong enough to catch plausible mistakes (CPU only).

Each case copies the oracle package into a temporary directory, plants one
mistake in the copy (a dropped term, a wrong sign, index, bias or order), and
runs the pin suite against the copy in a child process: at least one pin must
fail.  The unmodified copy must pass, so a failure is the planted mistake's.
Nothing here touches the oracle in the repository.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE = os.path.join(ROOT, "oracle")
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

C, PY = "sa_oracle.c", "__init__.py"

# (name, file, text in the oracle, planted replacement)
MUTATIONS = [
    # attention
    ("sink left out of the denominator", C, "den = exp(sink - M);", "den = 0.0;"),
    ("sink multiplied by the scale", C, "den = exp(sink - M);", "den = exp(scale * sink - M);"),
    ("scale left out of the scores", C, "s[j] = scale * acc;", "s[j] = acc;"),
    ("value row one index off", C, "kr = kvb + (size_t)idx[j] * D;",
     "kr = kvb + (size_t)(idx[j] > 0 ? idx[j] - 1 : 0) * D;"),
    ("last list entry left out of the weighted sum", C,
     "    for (j = 0; j < K; ++j) {\n        double p;", "    for (j = 0; j < K - 1; ++j) {\n        double p;"),
    ("list read only up to its first -1", C,
     "        if (r == -1) {\n            s[j] = -INFINITY;\n            continue;",
     "        if (r == -1) {\n            for (; j < K; ++j)\n                s[j] = -INFINITY;\n            break;"),
    ("every query reads batch row 0", C, "const uint16_t *kvb = kv + (size_t)b * N * D;",
     "const uint16_t *kvb = kv;"),
    # inverse rotary embedding
    ("forward rotation instead of the inverse (one component)", C, "x[2 * i + 1] = -a * sn + b * c;",
     "x[2 * i + 1] = a * sn + b * c;"),
    ("frequency index off by one", C, "double w = pow(theta, -2.0 * i / rope_dim);",
     "double w = pow(theta, -2.0 * (i + 1) / rope_dim);"),
    ("rotation applied to the first features", C, "+ (D - rope_dim);", "+ 0;"),
    ("pairs (i, i + half) instead of (2i, 2i + 1)", C,
     "double a = x[2 * i], b = x[2 * i + 1];\n                x[2 * i] = a * c + b * sn;\n"
     "                x[2 * i + 1] = -a * sn + b * c;",
     "double a = x[i], b = x[i + rope_dim / 2];\n                x[i] = a * c + b * sn;\n"
     "                x[i + rope_dim / 2] = -a * sn + b * c;"),
    # grouped projection
    ("wo_a block of the wrong group", C, "const uint16_t *w = W + ((size_t)g * R + r) * Din;",
     "const uint16_t *w = W + ((size_t)(G - 1 - g) * R + r) * Din;"),
    # fp8 / fp4 decoding and bf16 rounding
    ("E4M3 exponent bias 8", PY, "np.exp2(e - 7.0)", "np.exp2(e - 8.0)"),
    ("E4M3 subnormal step 2^-10", PY, "m * 2.0 ** -9", "m * 2.0 ** -10"),
    ("e2m1 nibbles in the other order", PY, "np.stack([c & 15, c >> 4]", "np.stack([c >> 4, c & 15]"),
    ("e2m1 largest magnitude 5", PY, "(0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)",
     "(0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 5.0)"),
    ("bf16 ties rounded away from zero", PY, "r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16", "r = (u + 0x8000) >> 16"),
    ("fp8 block scales transposed", PY, "s = np.repeat(np.repeat(sc, FP8_BLOCK",
     "s = np.repeat(np.repeat(sc.T if sc.shape[0] == sc.shape[1] else sc, FP8_BLOCK"),
    # fp4 quantization
    ("e2m1 halfway values rounded up", PY,
     "pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(np.asarray(even)[lo], lo, hi)))",
     "pick = np.where(dlo < dhi, lo, hi)"),
    ("fp4 scale over 4 instead of 6", PY, "sb = e4m3_encode(amax / np.float32(6.0))",
     "sb = e4m3_encode(amax / np.float32(4.0))"),
    ("fp4 codes without their sign", PY, "return (idx | np.where(np.signbit(x), 8, 0)).astype(np.uint8)",
     "return idx.astype(np.uint8)"),
    ("fp4 codes packed with the odd feature low", PY, "codes = (c[..., 0::2] | (c[..., 1::2] << 4))",
     "codes = (c[..., 1::2] | (c[..., 0::2] << 4))"),
    ("E4M3 values past 448 to NaN instead of 448", PY, "return np.where(a >= g[-1], len(g) - 1, pick)",
     "return np.where(a > g[-1], 0x7F, np.where(a == g[-1], len(g) - 1, pick))"),
    # top-k selection
    ("top-k ties to the larger position", PY, "pos[np.lexsort((pos, -row[pos]))]", "pos[np.lexsort((-pos, -row[pos]))]"),
    ("top-k may choose -inf", PY, "~(np.isnan(row) | (row == -np.inf))", "~np.isnan(row)"),
    ("top-k output in score order", PY, "chosen = np.sort(order)", "chosen = order"),
    # two latent sources
    ("compressed rows before the window rows", PY,
     "kv = np.concatenate(parts, axis=1) if parts", "kv = np.concatenate(parts[::-1], axis=1) if parts"),
    ("compressed rows of the wrong batch element", PY, "_as_bf16_bits(compressed_kv)[:B, :C]",
     "_as_bf16_bits(compressed_kv)[-B:, :C]"),
]

RUN = ("import sys; sys.path.insert(0, sys.argv[1]); import oracle; "
       "assert oracle.__file__.startswith(sys.argv[1]), oracle.__file__; "
       "import pytest; sys.exit(pytest.main([sys.argv[2], '-x', '-q', '-p', 'no:cacheprovider']))")


def _run_pins(tmp, mutation):
    pkg = os.path.join(tmp, "oracle")
    shutil.copytree(ORACLE, pkg, ignore=shutil.ignore_patterns("*.so", "*.tmp*", "__pycache__"))
    if mutation is not None:
        _, fname, old, new = mutation
        path = os.path.join(pkg, fname)
        text = open(path).read()
        assert text.count(old) == 1, (mutation[0], "text to replace not found exactly once")
        open(path, "w").write(text.replace(old, new))
    env = dict(os.environ, OMP_NUM_THREADS="2")
    p = subprocess.run([sys.executable, "-c", RUN, tmp, PINS], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    return p.returncode, p.stdout[-2000:] + p.stderr[-2000:]


def test_unmodified_copy_passes_the_pins(tmp_path):
    code, out = _run_pins(str(tmp_path), None)
    assert code == 0, out


def test_every_planted_mistake_fails_a_pin(tmp_path):
    dirs = []
    for i in range(len(MUTATIONS)):
        d = tmp_path / f"m{i}"
        d.mkdir()
        dirs.append(str(d))
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(_run_pins, dirs, MUTATIONS))
    missed = []
    for m, (code, out) in zip(MUTATIONS, results):
        # pytest exits 1 when a test failed; anything else (2..5) is a harness problem
        assert code in (0, 1), (m[0], code, out)
        if code == 0:
            missed.append(m[0])
    assert not missed, f"planted mistakes no pin caught: {missed}"
