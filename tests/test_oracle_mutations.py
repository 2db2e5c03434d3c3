"""The oracle's pins must catch plausible mistakes.

Each case below plants one mistake in a copy of the oracle's C source on the
CPU, compiles it, and runs the pins of tests/test_oracle_pins.py against the
broken library: at least one pin must fail.  The unmodified copy must pass.
"""
import os
import subprocess
import sys

import pytest

from oracle import build as obuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = open(obuild.SRC).read()

# (name, text in the oracle, replacement)
MUTANTS = [
    ("reduction starts from +0", "s[h] = (r == 0) ? v : s[h] + v;",
     "s[h] = (r == 0) ? 0.0f + v : s[h] + v;"),
    ("reversed rank order", "const uint16_t *p = partials + ((size_t)r * T + t) * H;",
     "const uint16_t *p = partials + ((size_t)(R - 1 - r) * T + t) * H;"),
    ("transposed [T,R,H] layout", "const uint16_t *p = partials + ((size_t)r * T + t) * H;",
     "const uint16_t *p = partials + ((size_t)t * R + r) * H;"),
    ("FP32 sum of squares",
     "double acc = 0.0;\n    for (int h = 0; h < H; ++h)\n        acc += (double)x[h] * (double)x[h];",
     "float acc = 0.0f;\n    for (int h = 0; h < H; ++h)\n        acc += x[h] * x[h];"),
    ("eps outside the square root", "return 1.0f / sqrtf(mean + eps);",
     "return 1.0f / (sqrtf(mean) + eps);"),
    ("mean over H-1", "float mean = ss / (float)H;", "float mean = ss / (float)(H - 1);"),
    ("1 + gamma", "float y = (s[h] * r1) * gamma_post[h];",
     "float y = (s[h] * r1) * (1.0f + gamma_post[h]);"),
    ("residual not added", "hbuf[h] = bf16_to_f32(res_in[h]) + y;", "hbuf[h] = y + 0.0f * res_in[h];"),
    ("residual subtracted", "hbuf[h] = bf16_to_f32(res_in[h]) + y;",
     "hbuf[h] = bf16_to_f32(res_in[h]) - y;"),
    ("gamma_post used by the pre-norm",
     "out[h] = f32_to_bf16_rn((hbuf[h] * r2) * gamma_pre[h]);",
     "{ out[h] = f32_to_bf16_rn((hbuf[h] * r2) * gamma_post[h]); (void)gamma_pre; }"),
    ("rounding by truncation",
     "if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))",
     "if (dropped > 0xffffffu)"),
    ("finalize not rounded locally", "float v = bf16_to_f32(z[h]);", "float v = zf_last[h];"),
    ("perm read as a scatter", "const int32_t *pr = perm + ((size_t)r * T + t) * k;",
     "static int32_t inv[64]; for (int j = 0; j < k; ++j) for (int q = 0; q < T * k; ++q) "
     "if (perm[(size_t)r * T * k + q] == t * k + j) inv[j] = q; const int32_t *pr = inv;"),
    ("weights of the wrong slot",
     "acc = acc + w[j] * bf16_to_f32(xr[(size_t)perm[j] * H + h]);",
     "acc = acc + w[k - 1 - j] * bf16_to_f32(xr[(size_t)perm[j] * H + h]);"),
    ("shared expert dropped", "if (shared_row) acc = acc + bf16_to_f32(shared_row[h]);",
     "(void)shared_row;"),
    ("shard 0's perm for every shard", "const int32_t *pr = perm + ((size_t)r * T + t) * k;",
     "const int32_t *pr = perm + ((size_t)0 * T + t) * k;"),
    ("shard 0's weights for every shard", "const float *wr = w + ((size_t)r * T + t) * k;",
     "const float *wr = w + ((size_t)0 * T + t) * k;"),
]


def _compile(src: str, d) -> str:
    c = d / "beamnorm_oracle.c"
    c.write_text(src)
    (d / "beamnorm_oracle.h").write_text(open(obuild.HDR).read())
    lib = d / "liboracle.so"
    flags = [f for f in obuild.CFLAGS if f != "-Werror"]
    subprocess.run(["gcc", *flags, "-shared", "-o", str(lib), str(c), "-lm"], check=True)
    return str(lib)


def _pins_pass(lib: str) -> bool:
    env = dict(os.environ, BEAMNORM_ORACLE_LIB=lib)
    p = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return p.returncode == 0


def test_unmodified_copy_passes(tmp_path):
    assert _pins_pass(_compile(SRC, tmp_path))


@pytest.mark.parametrize("name,find,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, find, repl):
    assert SRC.count(find) >= 1, f"mutation site not found: {name}"
    src = SRC.replace(find, repl)
    if name == "finalize not rounded locally":
        src = src.replace("static int token_of", "static float zf_last[65536];\nstatic int token_of")
        src = src.replace("z[h] = f32_to_bf16_rn(acc);", "z[h] = f32_to_bf16_rn(acc); zf_last[h] = acc;")
    assert not _pins_pass(_compile(src, tmp_path)), f"no pin caught: {name}"
