"""Plant one plausible mistake at a time in a copy of the oracle's source and
check that at least one pin (tests/pins.py) fails on it.

This is how the pins are shown to be strong enough: a dropped term, a wrong
sign, index, constant or operand anywhere in the oracle must be caught.  The
mistakes are planted in a temporary copy of ``oracle/fs_oracle.c`` (compiled
to its own library) or of ``oracle/merge.py`` (loaded as a separate module and
handed to the pins in place of the real merges), on the CPU; the committed
oracle is never modified.
"""
import os
import tempfile
import types

import pytest

import oracle
import oracle.merge
import pins
from oracle import build as obuild
from pins import ALL_PINS

SRC = open(obuild.SOURCE).read()
MERGE_SRC = open(oracle.merge.__file__).read()
MERGE_NAMES = ("chi_square_gof", "group_gumbel_max", "lse_merge", "online_merge",
               "partition_argmax")

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


# The same for oracle/merge.py: the group merges and the goodness-of-fit
# instrument behind every distributional pin.
MERGE_MUTANTS = [
    ("ggm-noise-sign", "keys = L - np.log(-np.log(u))", "keys = L + np.log(-np.log(u))", 0),
    ("ggm-single-log", "keys = L - np.log(-np.log(u))", "keys = L - np.log(u)", 0),
    ("ggm-ignores-mass", "keys = L - np.log(-np.log(u))", "keys = -np.log(-np.log(u))", 0),
    ("online-switch-reversed", "if u[k] < np.exp(Lk - new_L):", "if u[k] > np.exp(Lk - new_L):", 0),
    ("online-max-not-logaddexp", "new_L = np.logaddexp(cur_L, Lk)", "new_L = max(cur_L, Lk)", 0),
    ("online-old-mass", "if u[k] < np.exp(Lk - new_L):", "if u[k] < np.exp(Lk - cur_L):", 0),
    ("partition-tie-in-partition", "tile_max[t] > m_p", "tile_max[t] >= m_p", 0),
    ("partition-tie-across", "m_p > best_m", "m_p >= best_m", 0),
    ("lse-merge-no-shift", "return float(m + np.log(np.sum(np.exp(a - m))))",
     "return float(np.log(np.sum(np.exp(a))))", 0),
    ("chi-square-over-n", "stat = float(np.sum((obs_b[keep] - exp_b[keep]) ** 2 / exp_b[keep]))",
     "stat = float(np.sum((obs_b[keep] - exp_b[keep]) ** 2 / exp_b[keep])) / n", 0),
    ("chi-square-observed-denominator", "** 2 / exp_b[keep]))", "** 2 / np.maximum(obs_b[keep], 1.0)))", 0),
    ("chi-square-dof-not-minus-one", "dof = int(keep.sum() - 1)", "dof = int(keep.sum())", 0),
    ("chi-square-pool-dropped", "obs_b.append(counts[~big].sum())\n        exp_b.append(exp[~big].sum())",
     "pass", 0),
    ("chi-square-impossible-ignored", "if np.any(obs_b[~keep] > 0):", "if False:", 0),
    ("chi-square-sf-of-half", "float(chi2.sf(stat, dof))", "float(chi2.sf(stat / 2, dof))", 0),
]


def replace_nth(text, name, old, new, which, what):
    start = -1
    for _ in range(which + 1):
        start = text.find(old, start + 1)
        assert start >= 0, f"mutant {name}: text not found in {what}"
    return text[:start] + new + text[start + len(old):]


def mutate(name, old, new, which):
    return replace_nth(SRC, name, old, new, which, "fs_oracle.c")


def first_failing_pin(o):
    for pin in ALL_PINS:
        try:
            pin(o)
        except (AssertionError, ValueError, FloatingPointError, ZeroDivisionError, IndexError):
            return pin.__name__
    return None


@pytest.fixture(scope="module")
def workdir():
    with tempfile.TemporaryDirectory(prefix="fs_oracle_mutants_") as d:
        yield d


@pytest.mark.parametrize("name,old,new,which", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(workdir, name, old, new, which):
    text = mutate(name, old, new, which)
    lib = obuild.build_variant(text, name.replace("-", "_"), workdir)
    o = oracle.Oracle(lib)
    assert first_failing_pin(o), f"no pin catches the planted mistake {name!r}"


@pytest.mark.parametrize("name,old,new,which", MERGE_MUTANTS, ids=[m[0] for m in MERGE_MUTANTS])
def test_merge_mutant_is_caught(monkeypatch, name, old, new, which):
    text = replace_nth(MERGE_SRC, name, old, new, which, "merge.py")
    mod = types.ModuleType(f"merge_mutant_{name.replace('-', '_')}")
    exec(compile(text, f"<merge.py: {name}>", "exec"), mod.__dict__)
    for fn in MERGE_NAMES:
        monkeypatch.setattr(pins, fn, getattr(mod, fn))
    assert first_failing_pin(oracle.default()), f"no pin catches the planted mistake {name!r}"


def test_merge_mutants_reach_the_pins(monkeypatch):
    """Control for the test above: the real merge module, loaded the same way,
    passes every pin (so a caught mutant is caught for its mistake)."""
    mod = types.ModuleType("merge_unmodified")
    exec(compile(MERGE_SRC, "<merge.py>", "exec"), mod.__dict__)
    for fn in MERGE_NAMES:
        monkeypatch.setattr(pins, fn, getattr(mod, fn))
    assert first_failing_pin(oracle.default()) is None
