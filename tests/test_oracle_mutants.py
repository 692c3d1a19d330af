"""Plants plausible mistakes in a copy of the oracle's source and checks the pins catch each.

Every mutant is compiled from a text edit of oracle/moe_oracle.c into a temporary library and the
pin suite (tests/test_oracle_pins.py) is run against it in a child process; the suite must fail.
The oracle's own source is never modified.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moe_oracle.c")

MUTANTS = {
    "bias dropped": ("return scale * q + bias;", "return scale * q;"),
    "scale read from the next group": ("p->scales[r * groups + c / 64]",
                                       "p->scales[r * groups + (c / 64 + 1) % groups]"),
    "bias read from the wrong row": ("p->biases[r * groups + c / 64]",
                                     "p->biases[((r + 1) % p->rows) * groups + c / 64]"),
    "bit stream read MSB first": ("<< t;", "<< (bits - 1 - t);"),
    "fp16 exponent off by one": ("e - 25)", "e - 24)"),
    "silu sign flipped": ("double oracle_silu(double z) { return z / (1.0 + exp(-z)); }",
                          "double oracle_silu(double z) { return z / (1.0 + exp(z)); }"),
    "sigmoid sign flipped": ("double oracle_sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }",
                             "double oracle_sigmoid(double z) { return 1.0 / (1.0 + exp(z)); }"),
    "gate and up swapped": ("act[j] = oracle_silu(g[j]) * u[j];", "act[j] = oracle_silu(u[j]) * g[j];"),
    "transposed weight": ("acc += oracle_weight(p, r, c) * v[c];",
                          "acc += oracle_weight(p, c % p->rows, r % p->cols) * v[c];"),
    "score ignored": ("routed[t] += (double)scores[k] * y[t];", "routed[t] += y[t];"),
    "scores reversed": ("routed[t] += (double)scores[k] * y[t];",
                        "routed[t] += (double)scores[top_k - 1 - k] * y[t];"),
    "resid dropped": ("out[t] = r + (routed[t] + scalar * shared[t]);",
                      "out[t] = (routed[t] + scalar * shared[t]);"),
    "shared scalar dropped": ("out[t] = r + (routed[t] + scalar * shared[t]);",
                              "out[t] = r + (routed[t] + shared[t]);"),
    "shared term dropped": ("shared[t] += y[t];", "shared[t] += 0.0 * y[t];"),
    "bf16 read as fp16 bits": ("uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 13;"),
    "inversion keeps the last expert id": ("    if (found) {\n      uniq[u++] = e;",
                                           "    if (found) {\n      uniq[u++] = n_experts - 1 - e;"),
    "inversion drops the last pair": ("for (int32_t p = 0; p < m * k; ++p) {",
                                      "for (int32_t p = 0; p < m * k - 1; ++p) {"),
    "router ties keep the higher id": ("if (best < 0 || logits[e] > logits[best]) best = e;",
                                       "if (best < 0 || logits[e] >= logits[best]) best = e;"),
    "router softmax without the max shift": ("sum += exp((double)logits[ids[t]] - mx);",
                                             "sum += exp((double)logits[ids[t]]);"),
    "rmsnorm without eps": ("sqrt(ss / n + (double)eps)", "sqrt(ss / n)"),
    "rmsnorm sums instead of averaging": ("sqrt(ss / n + (double)eps)", "sqrt(ss + (double)eps)"),
    "rmsnorm weight dropped": ("oracle_round_bf16(oracle_bf16(gamma[c]) * ((double)v[c] * r))",
                               "oracle_round_bf16((double)v[c] * r)"),
    "bf16 rounding truncates": ("ldexp(nearbyint(ldexp(y, -s)), s)", "ldexp(trunc(ldexp(y, -s)), s)"),
    "bf16 ties away from zero": ("ldexp(nearbyint(ldexp(y, -s)), s)", "ldexp(round(ldexp(y, -s)), s)"),
    "gemv drops the last column": ("for (int32_t i = 0; i < n_in; ++i)\n        acc +=",
                                   "for (int32_t i = 0; i < n_in - 1; ++i)\n        acc +="),
    "gemv reads W transposed": ("oracle_bf16(W[(int64_t)o * n_in + i])",
                                "oracle_bf16(W[((int64_t)i * n_out + o) % ((int64_t)n_out * n_in)])"),
    "gemv reads the first token for all": ("oracle_bf16(x[(int64_t)t * n_in + i])",
                                           "oracle_bf16(x[i])"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name!r} not found exactly once"
    mut_c = tmp_path / "mutant.c"
    mut_c.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                           "-o", str(so), str(mut_c), "-lm"])
    env = dict(os.environ, MOE_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutant {name!r}:\n{r.stdout[-2000:]}"
