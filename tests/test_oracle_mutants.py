"""Planted mistakes: each mutant is a copy of the oracle's C source with one plausible slip
(a dropped term, a wrong sign, index or shift, a transposed output).  Every mutant must
fail at least one of the pins, which shows the pins constrain the oracle beyond agreeing
with itself.  The mutants are built from the oracle's source into a temporary directory on
the CPU; the oracle itself is never modified.  CPU only."""
import os
import subprocess
import tempfile

import pytest

import oracle
import test_oracle_pins as pins

MUTANTS = [
    ("q4_0 high nibble pairs with element j", "si += v1 * (int8_t)ab[2 + j + 16];", "si += v1 * (int8_t)ab[2 + j];"),
    ("q4_0 decode reads the low nibble twice", "(qs[i - 16] >> 4)) - 8", "(qs[i - 16] & 0x0F)) - 8"),
    ("q4_0 dot drops the -8", "int v0 = (wb[2 + j] & 0x0F) - 8;", "int v0 = (wb[2 + j] & 0x0F);"),
    ("q4_K min term sign", "s -= dmin * (float)minterm;\n            s += d * (float)value;\n        } else if (wtype == ORC_Q2_K)",
     "s += dmin * (float)minterm;\n            s += d * (float)value;\n        } else if (wtype == ORC_Q2_K)"),
    ("q4_K bsum pair index", "for (int s = 0; s < 8; s++) m += mn[s] * (bs[2 * s] + bs[2 * s + 1]);",
     "for (int s = 0; s < 8; s++) m += mn[s] * (bs[2 * s] + bs[2 * s]);"),
    ("q8_0 scale 128/amax", "float id = (amax != 0.0f) ? 127.0f / amax : 0.0f;\n        for (int i = 0; i < 32; i++) {",
     "float id = (amax != 0.0f) ? 128.0f / amax : 0.0f;\n        for (int i = 0; i < 32; i++) {"),
    ("f16 ties round up", "if (rest > 0x1000u || (rest == 0x1000u && (h & 1u))) h += 1u;", "if (rest >= 0x1000u) h += 1u;"),
    ("q2_K pack shift", "(uint8_t)(q[128 * h + 32 * s + l] << (2 * s));", "(uint8_t)(q[128 * h + 32 * s + l] << s);"),
    ("q6_K high bits slot", "((c1 >> 4) << 2)", "((c1 >> 4) << 4)"),
    ("transposed output", "j->out[t * j->N + o] =", "j->out[o * j->M + t] ="),
    ("q4_0 scale +8", "float d = m / -8.0f;", "float d = m / 8.0f;"),
    ("q4_0 rounding offset", "float t = xb[i] * id + 8.5f;", "float t = xb[i] * id + 8.0f;"),
    ("q6_K fold -31", "s += d * (float)(value - 32 * minterm);", "s += d * (float)(value - 31 * minterm);"),
    ("q4_K high scale bits", "sc[s] = (b[s + 4] & 15) | ((b[s - 4] >> 6) << 4);", "sc[s] = (b[s + 4] & 15) | ((b[s - 4] >> 6) << 3);"),
    ("q8_K bsums skip a code", "for (int i = 0; i < 16; i++) {\n                float v = xb[g * 16 + i] * id;\n                int q = clampi(rne(v), -128, 127);\n                ob[4 + g * 16 + i] = (uint8_t)(int8_t)q;\n                sum += q;",
     "for (int i = 0; i < 16; i++) {\n                float v = xb[g * 16 + i] * id;\n                int q = clampi(rne(v), -128, 127);\n                ob[4 + g * 16 + i] = (uint8_t)(int8_t)q;\n                if (i) sum += q;"),
    ("q8_0 rounds half away from zero", "float r = nearbyintf(v);", "float r = roundf(v);"),
    ("fifth bit read transposed", "return (qh[i / 8] >> (i % 8)) & 1;", "return (qh[i % 4] >> (i / 4)) & 1;"),
    ("q4_1 drops the min term", "s += (float)act_block_sum(a) * mx * dy;", "s += 0.0f * mx * dy;"),
    ("q5_K fifth bit shift", "int high = (blk[16 + l] >> (2 * j + (r >= 32))) & 1;",
     "int high = (blk[16 + l] >> (j + (r >= 32))) & 1;"),
    ("q5_1 high bits at the q5_0 offset", "nibble_code(blk + 8, i) | (fifth_bit(blk + 4, i) << 4)",
     "nibble_code(blk + 8, i) | (fifth_bit(blk + 2, i) << 4)"),
    ("q5_0 rounding offset", "float t = xb[i] * id + 16.5f;", "float t = xb[i] * id + 16.0f;"),
    ("q5_K quantizer 15 levels", "scl[s] = (hi + mns[s]) / 31.0f;", "scl[s] = (hi + mns[s]) / 15.0f;"),
    ("kv heads interleaved", "const int kvh = h / G;\n        for (int64_t p = 0; p < P; p++) {\n            const uint8_t* kr",
     "const int kvh = h % Hkv;\n        for (int64_t p = 0; p < P; p++) {\n            const uint8_t* kr"),
    ("rmsnorm drops eps", "const float sc = 1.0f / sqrtf(mean + eps);", "const float sc = 1.0f / sqrtf(mean);"),
    ("rmsnorm ignores w", "h[t * K + i] = (xr[i] * sc) * w[i];", "h[t * K + i] = xr[i] * sc;"),
    ("rmsnorm mean over K-1", "const float mean = (float)ss / (float)K;",
     "const float mean = (float)ss / (float)(K - 1);"),
    ("rmsnorm sums |x|, not x^2", "ss += (double)xr[i] * (double)xr[i];", "ss += fabs((double)xr[i]);"),
    ("rmsnorm skips the last value", "for (int64_t i = 0; i < K; i++) ss +=", "for (int64_t i = 1; i < K; i++) ss +="),
    ("kv cache head-major", "const uint8_t* vr = vc + (p * Hkv + kvh) * rb;", "const uint8_t* vr = vc + (kvh * P + p) * rb;"),
    ("kv scale 128/amax", "float id = (amax != 0.0f) ? 127.0f / amax : 0.0f;\n        for (int i = 0; i < hd; i++)",
     "float id = (amax != 0.0f) ? 128.0f / amax : 0.0f;\n        for (int i = 0; i < hd; i++)"),
]

PINS = [name for name in dir(pins) if name.startswith("test_")]


def _run_pins():
    failed = []
    for name in PINS:
        fn = getattr(pins, name)
        params = getattr(fn, "pytestmark", [])
        args = [None]
        for mark in params:
            if mark.name == "parametrize":
                args = mark.args[1]
        for a in args:
            try:
                if a is None:
                    fn(oracle)
                else:
                    fn(oracle, a)
            except AssertionError:
                failed.append(name if a is None else "%s[%s]" % (name, a))
            except Exception as e:  # a crash counts as caught too
                failed.append("%s: %s" % (name, type(e).__name__))
    return failed


@pytest.mark.parametrize("label,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(label, old, new, tmp_path):
    src = open(oracle.SRC).read()
    assert src.count(old) == 1, "mutation anchor not unique: " + label
    mutated = src.replace(old, new)
    c = tmp_path / "mutant.c"
    so = tmp_path / "libmutant.so"
    c.write_text(mutated)
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-std=c11", "-fPIC", "-shared", "-o", str(so), str(c),
                    "-lm", "-lpthread"], check=True)
    saved = oracle._lib
    oracle.lib()  # make sure the real one is built first
    saved = oracle._lib
    try:
        oracle._lib = oracle.load(str(so))
        failed = _run_pins()
    finally:
        oracle._lib = saved
    assert failed, "no pin caught the mutant: " + label
