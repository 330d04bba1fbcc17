"""Mutation check of the oracle's pins.

Each mutation below is a plausible mistake in the oracle's C source (a wrong tie-break, swapped
nibbles, a sign, an index, a rounding mode, a reduction order).  The test compiles a copy of the
oracle with one mutation applied, runs the pin suite (tests/test_oracle_pins.py) against that copy in
a child process, and requires the suite to FAIL: a mutation that every pin lets through would mean
the pins do not fix that part of the oracle.  The unmutated copy must pass.  CPU only.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "kq_oracle.c")

# (name, text in kq_oracle.c, replacement): each text occurs exactly once
MUTATIONS = [
    ("q8k amax tie-break", "if (ax > amax) { amax = ax; mx = x[i]; }", "if (ax >= amax) { amax = ax; mx = x[i]; }"),
    ("q8k iscale sign", "float iscale = -127.0f / mx;", "float iscale = 127.0f / mx;"),
    ("q8k rounding mode", "return (int)rintf(p);", "return (int)roundf(p);"),
    ("q8k bsum length", "for (int i = 0; i < 16; ++i) s += q[16 * j + i];",
     "for (int i = 0; i < 15; ++i) s += q[16 * j + i];"),
    ("q4k nibble order", "return r < 32 ? (b & 0x0f) : (b >> 4);", "return r < 32 ? (b >> 4) : (b & 0x0f);"),
    ("q4k min high bits", "*mn = (s12[j + 4] >> 4) | ((s12[j] >> 6) << 4);",
     "*mn = (s12[j + 4] >> 4) | ((s12[j - 4] >> 6) << 4);"),
    ("q5k high bit", "int hb = (blk[16 + l] >> (2 * c + (r >= 32))) & 1;", "int hb = (blk[16 + l] >> (2 * c)) & 1;"),
    ("q6k qh bit order", "int hi = (qh[l] >> (2 * quarter)) & 3;", "int hi = (qh[l] >> (6 - 2 * quarter)) & 3;"),
    ("q6k code offset", "acc += (q6k_code(wb, i) - 32) * q[i];", "acc += (q6k_code(wb, i) - 31) * q[i];"),
    ("q4k min term sign", "float t5 = t2 - t4;", "float t5 = t2 + t4;"),
    ("q4k bsum pairing", "*summ += (int64_t)mn * (rd_i16(xb + 260 + 4 * j) + rd_i16(xb + 262 + 4 * j));",
     "*summ += (int64_t)mn * (rd_i16(xb + 260 + 2 * j) + rd_i16(xb + 262 + 2 * j));"),
    ("q8_1 butterfly order", "for (int stride = 16; stride >= 1; stride /= 2) {",
     "for (int stride = 1; stride <= 16; stride *= 2) {"),
    ("q8_1 rounding", "float r = amax == 0.0f ? 0.0f : roundf(x[i] / d);",
     "float r = amax == 0.0f ? 0.0f : rintf(x[i] / d);"),
    ("rmsnorm order", "for (int64_t i = 0; i < K; ++i) {\n            float sq = xr[i] * xr[i];",
     "for (int64_t i = K - 1; i >= 0; --i) {\n            float sq = xr[i] * xr[i];"),
    ("rmsnorm mean", "float mean = total / (float)K;", "float mean = total / (float)(K - 1);"),
    ("grouped per-row index", "int64_t r = xq_rows_per_token == 1 ? t : p;",
     "int64_t r = xq_rows_per_token == 1 ? p : t;"),
    ("weighted sum slot", "float prod = wts[t * top_k + k] * y_slots[(t * top_k + k) * N + n];",
     "float prod = wts[t * top_k] * y_slots[(t * top_k + k) * N + n];"),
    ("half rounding", "double r = nearbyint(q);", "double r = floor(q + 0.5);"),
]


def _compile(src_text: str, out_dir: str) -> str:
    c = os.path.join(out_dir, "kq_oracle.c")
    so = os.path.join(out_dir, "libkq_oracle.so")
    with open(c, "w") as fh:
        fh.write(src_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
                    "-fvisibility=hidden", c, "-o", so, "-lm"], check=True, capture_output=True)
    return so


def _pins_pass(so: str) -> bool:
    env = dict(os.environ, KQ_ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"), "-x",
                        "-q", "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True)
    return r.returncode == 0


@pytest.fixture(scope="module")
def source():
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    with open(SRC) as fh:
        return fh.read()


def test_every_mutation_applies_once(source):
    for name, old, new in MUTATIONS:
        assert source.count(old) == 1, f"mutation '{name}': its text must occur exactly once in the oracle"
        assert old != new


def test_every_mutation_fails_a_pin(source):
    with tempfile.TemporaryDirectory() as tmp:
        dirs = []
        for i in range(len(MUTATIONS) + 1):
            d = os.path.join(tmp, f"m{i}")
            os.makedirs(d)
            dirs.append(d)
        texts = [source] + [source.replace(old, new, 1) for (_, old, new) in MUTATIONS]

        def run(i):
            return _pins_pass(_compile(texts[i], dirs[i]))

        with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
            passed = list(ex.map(run, range(len(texts))))
    assert passed[0], "the unmutated oracle must pass its pins"
    survivors = [MUTATIONS[i - 1][0] for i in range(1, len(texts)) if passed[i]]
    assert not survivors, f"mutations no pin detects: {survivors}"
