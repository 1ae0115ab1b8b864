"""The oracle's pins are sharp: a plausible mistake planted in a copy of
``oracle/oracle.c`` (a dropped term, a wrong sign, index or operand, a
rounding rule or a precision changed) makes at least one pin fail.

Each case edits one line of the oracle's source, compiles the copy with the
oracle's own flags into a temporary directory, points the ``oracle`` module
at it, runs the named pins and expects one of them to fail.  The real
library is restored afterwards.  CPU only.
"""

import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "oracle.c")


def _micro(k):
    return lambda o: pins.test_bruteforce_matches_oracle(o, pins.MICRO[k])


def _all_micro(o):
    for k in range(len(pins.MICRO)):
        _micro(k)(o)


MUTATIONS = {
    # causal mask off by one: a query no longer sees its own key
    "mask": ("visible[j] = (char)(j <= pos);", "visible[j] = (char)(j < pos);", [_all_micro]),
    # sign of the rotation's second term (float64 route)
    "rope-sign": ("        y[i] = ac - bs;\n        y[i + h] = bc + as;\n    }\n}\n\n/* The stored",
                  "        y[i] = ac + bs;\n        y[i + h] = bc + as;\n    }\n}\n\n/* The stored", [_all_micro]),
    # frequency index shifted by one pair
    "frequency": ("pow(theta, -2.0 * (double)i / (double)d)", "pow(theta, -2.0 * (double)(i + 1) / (double)d)",
                  [_all_micro]),
    # scale dropped from the scores
    "scale": ("w[j] = J->scale * acc;", "w[j] = acc;", [_all_micro]),
    # softmax not normalised
    "normalise": ("double pj = w[j] / sum;", "double pj = w[j];", [_all_micro]),
    # query head h mapped to kv head h % Hkv instead of h / G
    "gqa-map": ("for (int hh = g * G; hh < (g + 1) * G; ++hh) {", "for (int hh = g; hh < Hq; hh += Hkv) {",
                [_all_micro]),
    # gather through the arena at the wrong slot
    "gather-slot": ("(size_t)(j % J->bs)) * d;", "(size_t)((j + 1) % J->bs)) * d;",
                    [lambda o: [pins.test_arena_route_equals_logical_route(o, m) for m in pins.MICRO]]),
    # arena image written to the wrong slot
    "image-slot": ("int slot = (int)(p % bs);", "int slot = (int)((p + 1) % bs);",
                   [lambda o: [pins.test_arena_image_placement(o, m) for m in pins.MICRO]]),
    # stored rotation with a fused multiply-add
    "stored-fma": ("        y[i] = ac - bs;\n        y[i + h] = bc + as;\n    }\n}\n\n/* Expected bits",
                   "        y[i] = fmaf(a, cf, -bs);\n        y[i + h] = bc + as;\n    }\n}\n\n/* Expected bits",
                   [lambda o: pins.test_stored_rotation_bit_for_bit(o, "f16", 64, 1.0e4)]),
    # stored rotation from a float32 angle and float32 cos/sin
    "stored-cos32": ("float cf = (float)c, sf = (float)s;",
                     "float ang32 = (float)pos * powf((float)theta, -2.0f * (float)i / (float)d); "
                     "float cf = cosf(ang32), sf = sinf(ang32); (void)c; (void)s;",
                     [lambda o: pins.test_stored_rotation_bit_for_bit(o, "bf16", 128, 5.0e5)]),
    # round half away from zero instead of half to even
    "rounding-ties": ("if (rem > half || (rem == half && (kept & 1)))", "if (rem >= half)",
                      [pins.test_round_to_f16_matches_numpy, pins.test_round_to_bf16_bruteforce]),
    # subnormal decoding exponent off by one
    "subnormal": ("v = ldexp((double)f, 1 - bias - mbits);", "v = ldexp((double)f, -bias - mbits);",
                  [pins.test_decode_f16_exhaustive, pins.test_decode_bf16_exhaustive]),
}


@pytest.fixture(scope="module")
def source():
    oracle.build()
    return open(SRC).read()


def _failures(text, tmp_path, checks):
    """Compiles ``text`` as the oracle, runs the checks against it, and
    returns how many failed."""
    path = tmp_path / "oracle_copy.c"
    path.write_text(text)
    so = str(tmp_path / "liboracle_copy.so")
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared", "-ffp-contract=off", "-o",
                           so, str(path), "-lm", "-lpthread"])
    saved = oracle._lib
    oracle._lib = oracle.open_library(so)
    try:
        failed = 0
        for check in checks:
            try:
                check(oracle)
            except (AssertionError, ValueError):
                failed += 1
        return failed
    finally:
        oracle._lib = saved


def test_unmodified_copy_passes_every_pin(source, tmp_path):
    # the control: the same harness on the source as it stands fails nothing
    checks = [c for _, _, cs in MUTATIONS.values() for c in cs]
    assert _failures(source, tmp_path, checks) == 0


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_fails_a_pin(source, tmp_path, name):
    old, new, checks = MUTATIONS[name]
    assert source.count(old) == 1, "mutation site of %s not unique" % name
    assert _failures(source.replace(old, new), tmp_path, checks) > 0, "no pin caught the planted mistake %r" % name
