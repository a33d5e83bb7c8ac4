"""Plant plausible mistakes in copies of oracle.c and check that the pins
catch every one of them.  Runs on the CPU only; the real oracle is untouched.
"""
import os
import subprocess
import sys
from pathlib import Path

import pytest

import oracle

ROOT = Path(__file__).resolve().parent.parent
SRC = (ROOT / "oracle" / "oracle.c").read_text()

# (name, original text, mutated text): each original must occur exactly once
MUTANTS = [
    ("eps dropped", "ss / (double)n + eps", "ss / (double)n"),
    ("sum instead of mean", "ss / (double)n + eps", "ss + eps"),
    ("norm gain dropped", "y[i] = orc_bf16(g[i]) * (x[i] * inv);", "y[i] = (x[i] * inv);"),
    ("rope sin sign", "v[i] = a * c - b * s;", "v[i] = a * c + b * s;"),
    ("rope frequency exponent", "pow(theta, -2.0 * (double)i / (double)d)", "pow(theta, -1.0 * (double)i / (double)d)"),
    ("rope pairs adjacent", "double a = v[i], b = v[i + half];\n        v[i] = a * c - b * s;\n        v[i + half] = a * s + b * c;",
     "double a = v[2 * i], b = v[2 * i + 1];\n        v[2 * i] = a * c - b * s;\n        v[2 * i + 1] = a * s + b * c;"),
    ("query rotated at pos + 1", "orc_rope(d, q + (size_t)h * d, pos, cfg->rope_theta);",
     "orc_rope(d, q + (size_t)h * d, pos + 1, cfg->rope_theta);"),
    ("attention scale 1/d", "double scale = 1.0 / sqrt((double)d);\n    double m = -INFINITY;",
     "double scale = 1.0 / (double)d;\n    double m = -INFINITY;"),
    ("softmax without max shift", "s[j] = exp(s[j] - m);", "s[j] = exp(s[j]);"),
    ("values read from keys", "out[e] += (s[j] / den) * V[(size_t)j * stride + e];",
     "out[e] += (s[j] / den) * K[(size_t)j * stride + e];"),
    ("current token excluded", "orc_attention_head(pos + 1, d,", "orc_attention_head(pos > 0 ? pos : 1, d,"),
    ("gqa head mapping modulo", "int hk = h / group; /* consecutive", "int hk = h % nkv; /* consecutive"),
    ("attention residual dropped", "orc_matvec(H, nq * d, w->wo, att, o);\n    for (int i = 0; i < H; ++i) x[i] += o[i];",
     "orc_matvec(H, nq * d, w->wo, att, o);\n    for (int i = 0; i < H; ++i) x[i] = o[i];"),
    ("gate and up swapped", "hm[j] = orc_silu(g[j]) * u[j];", "hm[j] = orc_silu(u[j]) * g[j];"),
    ("silu sign", "return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    ("matvec operand reversed", "acc += orc_bf16(w[c]) * x[c];", "acc += orc_bf16(w[c]) * x[cols - 1 - c];"),
    ("kv written one slot late", "memcpy(kc + (size_t)pos * nkv * d, k,", "memcpy(kc + (size_t)(pos + 1 < max_seq ? pos + 1 : pos) * nkv * d, k,"),
    ("head uses embedding", "if (rc == 0) orc_head(cfg, w->final_norm, w->lm_head, x, logits);",
     "if (rc == 0) orc_head(cfg, w->final_norm, w->embed, x, logits);"),
    ("mask leaks next token", "if (j > i) {", "if (j > i + 1) {"),
    ("mlp norm uses attention gain", "orc_rmsnorm(H, x, w->mlp_norm, cfg->rms_eps, xn);",
     "orc_rmsnorm(H, x, w->attn_norm, cfg->rms_eps, xn);"),
    ("bf16 rounding keeps 9 bits", "ldexp(1.0, ilogb(x) - 7)", "ldexp(1.0, ilogb(x) - 8)"),
    ("bf16 cache leaves values unrounded", "            v[i] = orc_round_bf16(v[i]);", "            v[i] = v[i];"),
    ("full forward rounds keys only",
     "Vx[(size_t)t * nkv * d + i] = orc_round_bf16(Vx[(size_t)t * nkv * d + i]);",
     "Vx[(size_t)t * nkv * d + i] = Vx[(size_t)t * nkv * d + i];"),
]


@pytest.mark.parametrize("name,orig,mut", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, orig, mut):
    assert SRC.count(orig) == 1, f"mutation anchor for '{name}' not unique"
    src = tmp_path / "oracle_mut.c"
    src.write_text(SRC.replace(orig, mut))
    lib = oracle.compile_source(src, tmp_path / "liboracle_mut.so")
    env = dict(os.environ, MK_ORACLE_LIB=str(lib), OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        str(ROOT / "tests" / "test_oracle_pins.py")], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"no pin caught the planted mistake '{name}'"
