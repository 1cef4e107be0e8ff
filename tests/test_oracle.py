"""The CPU oracle against its pins (no GPU), and planted mistakes in it.

Every pin lives in tests/oracle_pins.py.  The planted-mistake test compiles
altered copies of oracle/dsa_oracle.c (a dropped term, a wrong sign or index,
a transposed operand, ...) into a temporary directory and checks that at
least one pin rejects each of them.
"""
import os
import shutil
import subprocess
import tempfile

import pytest

import oracle
from tests import oracle_pins as P


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("name", sorted(P.ALL_PINS))
def test_pin(lib, name):
    P.ALL_PINS[name](lib)


# (what the mistake is, text in dsa_oracle.c, its replacement)
MUTATIONS = [
    ("e4m3 exponent bias 8", "ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    ("e4m3 subnormal scale", "ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)"),
    ("e2m1 exponent bias", "ldexp(1.0 + 0.5 * m, e - 1)", "ldexp(1.0 + 0.5 * m, e)"),
    ("e8m0 bias", "ldexp(1.0, (int)b - 127)", "ldexp(1.0, (int)b - 128)"),
    ("nibble order swapped", "uint8_t nib = (i & 1) ? (byte >> 4) : (byte & 15);\n            k[i]",
     "uint8_t nib = (i & 1) ? (byte & 15) : (byte >> 4);\n            k[i]"),
    ("MX scale block of 16", "oracle_e8m0_decode(sc[i / 32])", "oracle_e8m0_decode(sc[i / 16])"),
    ("per-token scale dropped", "double a = s * dot;", "double a = dot;"),
    ("relu dropped", "(a > 0.0 ? a : 0.0)", "a"),
    ("head weight index", "w[(int64_t)r * OR_IDX_HEADS + h]", "w[(int64_t)r * OR_IDX_HEADS + (h ^ 1)]"),
    ("query head transposed", "q[h][i] * k[i]", "q[i % OR_IDX_HEADS][(i + h) % OR_IDX_DIM] * k[i]"),
    ("causal extent off by one", "t1 = row_ctx[r] < t0 + OR_CHUNK ? row_ctx[r] : t0 + OR_CHUNK;",
     "t1 = row_ctx[r] - 1 < t0 + OR_CHUNK ? row_ctx[r] - 1 : t0 + OR_CHUNK;"),
    ("tie break to higher index", "return (x->t > y->t) - (x->t < y->t);", "return (x->t < y->t) - (x->t > y->t);"),
    ("top-k ascending", "if (x->v > y->v) return -1;", "if (x->v < y->v) return -1;"),
    ("slot offset", "bt[t / OR_PAGE] * OR_PAGE + t % OR_PAGE", "bt[t / OR_PAGE] * OR_PAGE + t / OR_PAGE"),
    ("softmax scale dropped", "sc[t] = sm_scale * s;", "sc[t] = s;"),
    ("rope dims dropped from scores", "for (int i = 0; i < OR_LAT_DIM; ++i) s += qh[i]",
     "for (int i = 0; i < OR_V_DIM; ++i) s += qh[i]"),
    ("latent tensor scale dropped", "kv[i] = oracle_e4m3_decode(codes[i]) * tensor_scale;",
     "kv[i] = oracle_e4m3_decode(codes[i]);"),
    ("nvfp4 scale block of 32", "oracle_e4m3_decode(sc[i / 16])", "oracle_e4m3_decode(sc[i / 32])"),
    ("lse without max", "lse[(int64_t)r * num_heads + h] = m + log(l);", "lse[(int64_t)r * num_heads + h] = log(l);"),
    ("output not normalised", "o[d] /= l;", "o[d] /= 1.0;"),
    ("value uses rope dims", "o[d] += p * kv[(int64_t)t * OR_LAT_DIM + d];",
     "o[d] += p * kv[(int64_t)t * OR_LAT_DIM + d + 64];"),
    ("e4m3 rounds half away from zero", "double r = nearbyint(a / q) * q;\n    if (r == 0.0)",
     "double r = floor(a / q + 0.5) * q;\n    if (r == 0.0)"),
    ("e4m3 saturates to 480", "if (a >= 448.0) return (uint8_t)((s << 7) | 0x7E);",
     "if (a >= 480.0) return (uint8_t)((s << 7) | 0x7F);"),
    ("e4m3 subnormal quantum", "if (ue < -6) ue = -6;   /* below", "if (ue < -7) ue = -7;   /* below"),
    ("e2m1 binade boundary", "double q = a < 2.0 ? 0.5 : (a < 4.0 ? 1.0 : 2.0);",
     "double q = a < 1.0 ? 0.5 : (a < 4.0 ? 1.0 : 2.0);"),
    ("FP8 key scale over 240", "float sc = amax > 0.0f ? amax / 448.0f : 1.0f;", "float sc = amax > 0.0f ? amax / 240.0f : 1.0f;"),
    ("MX exponent offset", "E = (e - 1) - 2 + 127;", "E = (e - 1) - 1 + 127;"),
    ("NVFP4 scale over 4", "uint8_t scode = oracle_e4m3_encode(amax / 6.0f);", "uint8_t scode = oracle_e4m3_encode(amax / 4.0f);"),
    ("MSA block score keeps the last key", "if (dot > best[g]) best[g] = dot;", "best[g] = dot;"),
    ("MSA block score past the causal edge", "for (int t = b * OR_MSA_PAGE; t < L && t < (b + 1) * OR_MSA_PAGE; ++t) {\n                    const uint8_t *key",
     "for (int t = b * OR_MSA_PAGE; t <= L && t < (b + 1) * OR_MSA_PAGE; ++t) {\n                    const uint8_t *key"),
    ("MSA index key row of a 64-token page", "(int64_t)(t % OR_MSA_PAGE) * OR_MSA_DIM;", "(int64_t)(t % 64) * OR_MSA_DIM;"),
    ("MSA recent block not forced", "out[m++] = nb - 1;", "out[m++] = buf[OR_MSA_BLOCKS - 1].t;"),
    ("MSA 16 best others, recent dropped", "for (int i = 0; i < OR_MSA_BLOCKS - 1; ++i) out[m++] = buf[i].t;\n        out[m++] = nb - 1;",
     "for (int i = 0; i < OR_MSA_BLOCKS; ++i) out[m++] = buf[i].t;"),
    ("MSA head groups interleaved", "const int h = g * heads_per_group + hh;", "const int h = hh * OR_MSA_GROUPS + g;"),
    ("MSA value read from K", "V[(int64_t)n * OR_MSA_DIM + d] = oracle_e4m3_decode(vp[j * OR_MSA_DIM + d]) * v_scale;",
     "V[(int64_t)n * OR_MSA_DIM + d] = oracle_e4m3_decode(kp[j * OR_MSA_DIM + d]) * v_scale;"),
    ("MSA query scale dropped", "oracle_e4m3_decode(q[((int64_t)r * H + h) * OR_MSA_DIM + d]) * q_scale;",
     "oracle_e4m3_decode(q[((int64_t)r * H + h) * OR_MSA_DIM + d]);"),
    ("MSA key scale dropped", "K[(int64_t)n * OR_MSA_DIM + d] = oracle_e4m3_decode(kp[j * OR_MSA_DIM + d]) * k_scale;",
     "K[(int64_t)n * OR_MSA_DIM + d] = oracle_e4m3_decode(kp[j * OR_MSA_DIM + d]);"),
    ("MSA V of the next head", "const uint8_t *vp = kp + OR_MSA_PAGE * OR_MSA_DIM;", "const uint8_t *vp = kp + 2 * OR_MSA_PAGE * OR_MSA_DIM;"),
    ("MSA attention past the causal edge", "for (int t = b * OR_MSA_PAGE; t < L && t < (b + 1) * OR_MSA_PAGE; ++t, ++n) {",
     "for (int t = b * OR_MSA_PAGE; t < (b + 1) * OR_MSA_PAGE; ++t, ++n) {"),
    ("MSA softmax scale dropped", "sc[t] = s * sm_scale;", "sc[t] = s;"),
    ("MSA output not normalised", "o[d] = o[d] / l;", "o[d] = o[d] / 1.0;"),
    ("insert nibble order", "codes[(16 * b + d) / 2] = (uint8_t)(lo | (hi << 4));", "codes[(16 * b + d) / 2] = (uint8_t)(hi | (lo << 4));"),
]


def _build_mutant(src_text, tmpdir, i):
    path = os.path.join(tmpdir, f"m{i}.c")
    with open(path, "w") as f:
        f.write(src_text)
    so = os.path.join(tmpdir, f"m{i}.so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-fopenmp", path, "-o", so,
                    "-lm"], check=True)
    return so


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_planted_mistakes_are_caught():
    src = open(oracle._SRC).read()
    missed = []
    with tempfile.TemporaryDirectory() as td:
        for i, (what, old, new) in enumerate(MUTATIONS):
            assert src.count(old) == 1, f"mutation anchor not unique: {what}"
            lib = oracle.load(_build_mutant(src.replace(old, new), td, i))
            caught = False
            for pin in P.ALL_PINS.values():
                try:
                    pin(lib)
                except AssertionError:
                    caught = True
                    break
                except Exception:
                    caught = True
                    break
            if not caught:
                missed.append(what)
    assert not missed, f"pins missed planted mistakes: {missed}"
