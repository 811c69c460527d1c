"""Plant plausible mistakes in copies of the oracle source and require the
pins to catch every one.  This shows the pins constrain each part of the
oracle: dequantisation, alignment, both projections, the activation, the
combine and the router."""
import os

import pytest

import oracle
from tests import oracle_pins

MUTANTS = [
    ("zero point 7", "(double)(code - 8)", "(double)(code - 7)"),
    ("nibble order swapped", "(kk & 1) ? (byte >> 4) : (byte & 0x0F)",
     "(kk & 1) ? (byte & 0x0F) : (byte >> 4)"),
    ("first group scale only", "s[n * (K / group) + kk / group]", "s[n * (K / group)]"),
    ("group size fixed at 32", "s[n * (K / group) + kk / group]", "s[n * (K / group) + kk / 32]"),
    ("silu sign", "exp(-v)", "exp(v)"),
    ("gate and up swapped", "a[n] = silu(g) * u;", "a[n] = silu(u) * g;"),
    ("up rows interleaved", "weight_at(q13, sc13, H, group, I + n, h)",
     "weight_at(q13, sc13, H, group, 2 * n + 1 < 2 * I ? 2 * n + 1 : n, h)"),
    ("down projection transposed", "weight_at(q2, sc2, I, group, hh, n)",
     "weight_at(q2, sc2, I, group, n, hh % I)"),
    ("first hidden element dropped", "for (int64_t h = 0; h < H; ++h)",
     "for (int64_t h = 1; h < H; ++h)"),
    ("combine ignores topk_w", "acc += (double)topk_w[t * k + j] * yrow",
     "acc += 1.0 * yrow"),
    ("combine reads slot 0 only", "int32_t pos = inv_perm[t * k + j];",
     "int32_t pos = inv_perm[t * k];"),
    ("unstable placement", "int32_t pos = offsets[e] + counts[e];",
     "int32_t pos = offsets[e + 1] - 1 - counts[e];"),
    ("token index from slot modulo", "int64_t t = f / k;", "int64_t t = f % k;"),
    ("router ties to the higher index", "return ea < eb;", "return ea > eb;"),
    ("router NaN ranked first", "if (an != bn) return bn;", "if (an != bn) return an;"),
    ("router ascending order", "return a > b;", "return a < b;"),
    ("router weights not renormalised", "/ z) / sel);", "/ z));"),
    ("router softmax without shift", "z += exp((double)l[e] - mx);", "z += exp((double)l[e]);"),
    ("router bad rows kept", "if (bad || mx == -INFINITY)", "if (mx == -INFINITY)"),
    ("router weight of the top slot everywhere", "(float)((exp((double)l[id[j]] - mx)",
     "(float)((exp((double)l[id[0]] - mx)"),
    ("sigmoid instead of SiLU", "return v / (1.0 + exp(-v));", "return 1.0 / (1.0 + exp(-v));"),
    ("scale row stride dropped", "s[n * (K / group) + kk / group]", "s[kk / group]"),
    ("code row stride halved", "q[n * (K / 2) + kk / 2]", "q[n * (K / 4) + kk / 2]"),
    ("down projection drops the last intermediate element",
     "for (int64_t n = 0; n < I; ++n)\n                acc += a[n]",
     "for (int64_t n = 0; n + 1 < I; ++n)\n                acc += a[n]"),
    ("combine weight of slot 0 for every slot", "acc += (double)topk_w[t * k + j]",
     "acc += (double)topk_w[t * k]"),
    ("bf16 bits not shifted", "((uint32_t)bits) << 16", "((uint32_t)bits)"),
]


def _run_pins(orc):
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except AssertionError as exc:
            failed.append((pin.__name__, str(exc)[:80]))
    return failed


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(oracle.SOURCE).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mutated = src.replace(old, new)
    path = tmp_path / "mutant.c"
    path.write_text(mutated)
    so = oracle.compile_source(str(path), str(tmp_path / "libmutant.so"))
    failed = _run_pins(oracle.Oracle(so))
    assert failed, f"mutant '{name}' passed every pin"
