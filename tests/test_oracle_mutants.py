"""Plant one plausible mistake at a time in a copy of the oracle's source and
check that at least one pin (tests/pins.py) fails on it.

This is how the pins are shown to be strong enough: a dropped term, a wrong
sign, index, constant or operand anywhere in the oracle must be caught.  The
mistakes are planted in a temporary copy of ``oracle/fs_oracle.c`` on the CPU;
the committed oracle is never modified.
"""
import os
import tempfile

import pytest

import oracle
from oracle import build as obuild
from pins import ALL_PINS

SRC = open(obuild.SOURCE).read()

# (name, text in fs_oracle.c, replacement, which occurrence (0 = first))
MUTANTS = [
    ("philox-multiplier", "0xCD9E8D57u", "0xCD9E8D59u", 0),
    ("philox-weyl-swapped", "k1 += PHILOX_WEYL_1;", "k1 += PHILOX_WEYL_0;", 0),
    ("philox-nine-rounds", "round < 10", "round < 9", 0),
    ("philox-bump-first-round", "if (round > 0) {", "if (round >= 0) {", 0),
    ("philox-output-order", "uint32_t n1 = lo1;", "uint32_t n1 = lo0;", 0),
    ("uniform-no-centre", "+ 0.5) * (1.0 / 8388608.0)", "+ 0.0) * (1.0 / 8388608.0)", 0),
    ("uniform-wrong-bits", "(word & 0x7fffffu)", "(word & 0xffffffu)", 0),
    ("uniform-top-bits", "(word & 0x7fffffu)", "(word >> 9)", 0),
    ("gumbel-sign", "return -log(-log(u));", "return log(-log(u));", 0),
    ("gumbel-single-log", "return -log(-log(u));", "return -log(u);", 0),
    ("counter-drops-row", "counter[1] = (uint32_t)b;", "counter[1] = 0;", 0),
    ("counter-word-fixed", "return out[(uint64_t)v & 3u];", "return out[0];", 0),
    ("counter-vocab-unshifted", "(uint32_t)((uint64_t)v >> 2)", "(uint32_t)((uint64_t)v >> 3)", 0),
    ("key-drops-high-word", "key[1] = (uint32_t)(seed >> 32);", "key[1] = 0;", 0),
    ("counter-drops-offset-high", "counter[3] = (uint32_t)(offset >> 32);", "counter[3] = 0;", 0),
    ("temperature-multiplies", "lp[v] = l[v] / T;", "lp[v] = l[v] * T;", 0),
    ("logit-drops-first-term", "for (int64_t k = 0; k < d; ++k) acc +=",
     "for (int64_t k = 1; k < d; ++k) acc +=", 0),
    ("logit-reversed-operand", "bf16_to_double(w[k]);", "bf16_to_double(w[d - 1 - k]);", 0),
    ("tile-ties-to-highest", "if (arg < 0 || s[v] > best) {", "if (arg < 0 || s[v] >= best) {", 0),
    ("row-ties-to-highest", "if (arg < 0 || s[v] > best) {", "if (arg < 0 || s[v] >= best) {", 1),
    ("tile-gap-not-tracked", "second = best;\n          best = s[v];\n          arg = v;\n        } else if",
     "best = s[v];\n          arg = v;\n        } else if", 0),
    ("lse-over-noisy-scores", "acc += exp(lp[v] - lmax);", "acc += exp(s[v] - lmax);", 0),
    ("lse-without-shift", "acc += exp(lp[v] - lmax);\n        lse = lmax + log(acc);",
     "acc += exp(lp[v]);\n        lse = log(acc);", 0),
    ("lse-includes-masked", "if (ok[v]) acc += exp(lp[v] - lmax);", "acc += exp(lp[v] - lmax);", 0),
    ("mask-polarity", "return (int)((mask[b * mask_ld + v / 32] >> (v % 32)) & 1u);",
     "return (int)(((mask[b * mask_ld + v / 32] >> (v % 32)) & 1u) ^ 1u);", 0),
    ("mask-wrong-word", "mask[b * mask_ld + v / 32]", "mask[b * mask_ld + v / 31]", 0),
    ("greedy-threshold", "return !(T > 0.0) || isinf(T);", "return !(T >= 0.0) || isinf(T);", 0),
    ("greedy-adds-noise", "lp[v] = l[v];\n        s[v] = l[v];",
     "lp[v] = l[v];\n        s[v] = l[v] + fso_noise(sd, offset, b, v);", 0),
    ("tile-boundary-short", "hi = (lo + tile < V) ? lo + tile : V;", "hi = (lo + tile < V) ? lo + tile - 1 : V;", 0),
    ("merge-domain-not-separated", "counter[1] = (uint32_t)b | 0x80000000u;",
     "counter[1] = (uint32_t)b;", 0),
    ("per-row-seed-ignored", "uint64_t sd = seeds ? seeds[b] : seed;\n    for", "uint64_t sd = seed;\n    for", 0),
]


def mutate(name, old, new, which):
    start = -1
    for _ in range(which + 1):
        start = SRC.find(old, start + 1)
        assert start >= 0, f"mutant {name}: text not found in fs_oracle.c"
    return SRC[:start] + new + SRC[start + len(old):]


@pytest.fixture(scope="module")
def workdir():
    with tempfile.TemporaryDirectory(prefix="fs_oracle_mutants_") as d:
        yield d


@pytest.mark.parametrize("name,old,new,which", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(workdir, name, old, new, which):
    text = mutate(name, old, new, which)
    lib = obuild.build_variant(text, name.replace("-", "_"), workdir)
    o = oracle.Oracle(lib)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            caught.append(pin.__name__)
            break
        except (ValueError, FloatingPointError, ZeroDivisionError, IndexError):
            caught.append(pin.__name__)
            break
    assert caught, f"no pin catches the planted mistake {name!r}"
