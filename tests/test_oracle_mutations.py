"""Plant plausible mistakes in a copy of the oracle (CPU only) and check that the pins catch each.

Each mutant is compiled from an edited copy of ``oracle/pkv_oracle.c`` into a temporary
library; the pin suite then runs against it in a subprocess and must fail.
"""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pkv_oracle.c")

MUTANTS = [
    ("rope sign", "    y[i] = a * c - b * s;", "    y[i] = a * c + b * s;"),
    ("rope frequency exponent", "pow(theta, -2.0 * (double)i / (double)d)", "pow(theta, -1.0 * (double)i / (double)d)"),
    ("rope pairing", "double a = x[i], b = x[i + half];", "double a = x[i], b = x[d - 1 - i];"),
    ("gqa head mapping", "s, h / G, window_start(len, window), len,", "s, h % Hkv, window_start(len, window), len,"),
    ("window off by one", "return (window > 0 && len > window) ? len - window : 0;",
     "return (window > 0 && len > window) ? len - window + 1 : 0;"),
    ("sink weight sign", "ws = exp(sink - M);", "ws = exp(M - sink);"),
    ("sink dropped by the combine", "    if (sinks != NULL) apply_sink(o, lse + sh, d, sinks[sh % Hq]);\n", "\n"),
    ("windowed chunk start", "      if (t0 < ws) t0 = ws;\n      if (t1 > len) t1 = len;\n      if (t0 > len) t0 = len;\n      r = attend(g, pool, q, s, h / G,",
     "      if (t1 > len) t1 = len;\n      if (t0 > len) t0 = len;\n      r = attend(g, pool, q, s, h / G,"),
    ("windowed balanced start", "    const int64_t f = vfirst[s], ws = window_start(len, window);", "    const int64_t f = 0, ws = window_start(len, window);"),
    ("int4 nibble order", "const int nibble = (int)((packed >> (4 * (k % 8))) & 0xFu);",
     "const int nibble = (int)((packed >> (4 * (7 - k % 8))) & 0xFu);"),
    ("int4 centering", "wrow[k] = dec(orc_f64_to_f16((double)(nibble - 7) * scale));",
     "wrow[k] = dec(orc_f64_to_f16((double)(nibble - 8) * scale));"),
    ("int4 product not rounded to fp16", "wrow[k] = dec(orc_f64_to_f16((double)(nibble - 7) * scale));",
     "wrow[k] = (double)(nibble - 7) * scale;"),
    ("int4 scale group", "const double scale = dec(scales[(int64_t)n * groups + k / 32]);",
     "const double scale = dec(scales[(int64_t)n * groups + k / 64]);"),
    ("prefill not causal", "window_start(p + 1, window), p + 1, page_indptr,", "window_start(p + 1, window), p + 2, page_indptr,"),
    ("int8 rounding truncates", "float q = nearbyintf((float)dec(x[i]) / s);", "float q = truncf((float)dec(x[i]) / s);"),
    ("int8 scale divisor", "const float s = amax / 127.0f;", "const float s = amax / 128.0f;"),
    ("int8 scale offset", "out[pool_row(g, page, kv, h, slot) + i] = (double)((int)blk[code8(d, kv, slot, i)] - 128) * (double)sc;",
     "out[pool_row(g, page, kv, h, slot) + i] = (double)((int)blk[code8(d, kv, slot, i)] - 128);"),
    ("int8 byte bias on read", "out[pool_row(g, page, kv, h, slot) + i] = (double)((int)blk[code8(d, kv, slot, i)] - 128) * (double)sc;",
     "out[pool_row(g, page, kv, h, slot) + i] = (double)((int)blk[code8(d, kv, slot, i)] - 127) * (double)sc;"),
    ("int8 byte stored without its bias", "blk[code8(d, kv, slot, i)] = (uint8_t)(codes[i] + 128);",
     "blk[code8(d, kv, slot, i)] = (uint8_t)codes[i];"),
    ("int8 V block read slot-major",
     "static int64_t code8(int d, int kv, int slot, int i) { return kv == 0 ? (int64_t)slot * d + i : (int64_t)i * 16 + slot; }",
     "static int64_t code8(int d, int kv, int slot, int i) { return (int64_t)slot * d + i; }"),
    ("last page length ignored", "*len = (n - 1) * ORC_PAGE + last;", "*len = n * ORC_PAGE;"),
    ("slot index", "const int64_t krow = pool_row(g, page, 0, kv_head, t % ORC_PAGE);",
     "const int64_t krow = pool_row(g, page, 0, kv_head, (t + 1) % ORC_PAGE);"),
    ("softmax scale dropped", "score[t - t0] = sm_scale * dot;", "score[t - t0] = dot;"),
    ("combine lse", "lse[sh] = M + log(W);", "lse[sh] = log(W);"),
    ("fp16 rounding truncates", "double n = nearbyint(a / quantum);", "double n = floor(a / quantum);"),
    ("append page lookup", "      int64_t page = page_indices[page_indptr[s] + p / ORC_PAGE];",
     "      int64_t page = page_indices[page_indptr[s] + p % ORC_PAGE];"),
    ("empty chunk lse", "    *lse = -INFINITY;\n    return ORC_OK;\n  }\n  double* score",
     "    *lse = 0.0;\n    return ORC_OK;\n  }\n  double* score"),
    ("split partition floors", "int c = chunk_pages > 0 ? chunk_pages : (n + num_splits - 1) / num_splits;\n    double* q",
     "int c = chunk_pages > 0 ? chunk_pages : n / num_splits + (n % num_splits > 1);\n    double* q"),
    ("v not copied", "memcpy(vd, vs, sizeof(uint16_t) * (size_t)d);", "memcpy(vd, ks, sizeof(uint16_t) * (size_t)d);"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for '{name}' must be unique"
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(oracle.build_command(str(mutant), str(lib)), check=True)
    env = dict(os.environ, PKV_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_window_sinks.py"),
                        os.path.join(ROOT, "tests", "test_oracle_qkv.py"),
                        os.path.join(ROOT, "tests", "test_oracle_prefill.py"),
                        os.path.join(ROOT, "tests", "test_oracle_int8.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"the pins did not catch the planted mistake '{name}'"
