"""The pins catch plausible mistakes in the oracle.

Each case below plants one plausible mistake in a copy of the oracle's C
source: a wrong destination member, an interleaved token split, a transposed
index order, a misplaced group.  It compiles that copy and runs the pin
suite of test_oracle_pins.py / test_oracle_variants.py against it.  Every
planted mistake must make at least one pin fail; the unmodified source must
pass them all.  The mistakes are planted on the CPU only.
"""
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins
import test_oracle_variants as variants

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "oracle", "basp_oracle.c")

MUTATIONS = [
    ("destination member from an interleaved head split",
     "const int64_t jp = h / Hk;", "const int64_t jp = h % K;"),
    ("interleaved token split across the group",
     "const int64_t s = j * Sk + sl;", "const int64_t s = sl * K + j;"),
    ("head within the block taken from the wrong modulus",
     "const int64_t hl = h % Hk;", "const int64_t hl = h / K;"),
    ("destination rank with group and member swapped",
     "const int64_t r_out = g * K + jp;", "const int64_t r_out = jp * (N / K) + g;"),
    ("source group taken modulo instead of divided",
     "const int64_t g = r_in / K;      /* group of the source rank   */",
     "const int64_t g = r_in % (N / K);"),
    ("batch-first destination token order transposed",
     "const int64_t t_out = order ? s * Bg + bl  : bl * S + s;",
     "const int64_t t_out = order ? s * Bg + bl  : s * Bg + bl;"),
    ("sequence-first source token order transposed",
     "const int64_t t_in  = order ? sl * Bg + bl : bl * Sk + sl;",
     "const int64_t t_in  = order ? bl * Sk + sl : bl * Sk + sl;"),
    ("head and element index transposed in the source",
     "const int64_t src = r_in * P + (t_in * H + h) * d + e;",
     "const int64_t src = r_in * P + (t_in * d + e) * H + h;"),
]


def _pin_failures():
    """Run the pin tests against whatever library oracle._lib holds; return
    how many of them fail."""
    fails = 0

    def attempt(fn, *args):
        nonlocal fails
        try:
            fn(*args)
        except (AssertionError, ValueError):
            fails += 1

    for c in pins.GOLDEN_CASES:
        attempt(pins.test_hand_worked_values if c["kind"] == "case"
                else pins.test_hand_worked_packed_qkv, c)
    for shape in pins.LIB_SHAPES:
        attempt(pins.test_library_permute_form, shape)
        attempt(pins.test_index_values_decode_to_their_place, shape)
        attempt(variants.test_seq_first_library_form, shape)
    attempt(pins.test_brute_force_two_forms_agree)
    attempt(variants.test_seq_first_brute_force)
    return fails


def _compile(text, tmp_path, name):
    src = tmp_path / (name + ".c")
    src.write_text(text)
    so = tmp_path / (name + ".so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(so),
                    str(src)], check=True)
    return oracle.load_from(str(so))


@pytest.fixture
def swap_oracle():
    saved = oracle._load()
    yield
    oracle._lib = saved


def test_unmodified_source_passes_every_pin(tmp_path, swap_oracle):
    oracle._lib = _compile(open(SRC).read(), tmp_path, "clean")
    assert _pin_failures() == 0


@pytest.mark.parametrize("what,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(what, old, new, tmp_path, swap_oracle):
    text = open(SRC).read()
    # the mistakes go into the plain element loop the pins check; the
    # all-core form after it is pinned against that loop separately
    cut = text.index("/*\n * All-core form")
    plain, rest = text[:cut], text[cut:]
    assert plain.count(old) == 1, "mutation anchor not found: " + old
    oracle._lib = _compile(plain.replace(old, new) + rest, tmp_path, "mutant")
    assert _pin_failures() > 0, "no pin caught: " + what
