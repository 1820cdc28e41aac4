"""Epilogue inputs that tell the step orderings apart.

The int8 epilogue of "conv_ops_fused_int8.cc" rounds three times (scale,
side-input fma, bias add).  A different arrangement of the same arithmetic
(the older fma(acc, scale, bias) order, an unfused side term, or a compiler
contracting steps (1) and (3)) changes the int8 result only when a value
lands within a rounding error of a half-integer.  This module searches for
such inputs with exact rational arithmetic (oracle.exact), grouped by the
per-run scalars (conv_scale, side_scale, bias, relu) so that each group can
be fed to one convolution launch.
"""
from __future__ import annotations

import functools

import numpy as np

from oracle import exact

VARIANTS = ("fma_scale_bias", "no_side_fma", "contract_13")

# (conv_scale, side_scale, bias, relu): scales are binary32 values.
GROUPS = (
    (float(np.float32(0.001)), 0.0, -100.0, False),
    (float(np.float32(0.002)), 0.5, -100.0, True),
    (0.015625, float(np.float32(0.3)), 0.0, False),
    (float(np.float32(0.05)), float(np.float32(0.1)), -300.0, True),
    (float(np.float32(0.004)), float(np.float32(0.7)), -64.0, False),
    (float(np.float32(0.1)), 0.0, -3000.0, False),
)

ACC_LIMIT = 400_000   # the GPU tests build each sum from 32 int8 channels


def _differs(acc, cs, side, ss, bias, relu):
    base = exact.epilogue_i8(acc, cs, side, ss, bias, relu)
    return [v for v in VARIANTS
            if exact.epilogue_i8_other_order(acc, cs, side, ss, bias, relu, v) != base]


@functools.lru_cache(maxsize=None)
def _search(group, per_group=16):
    cs, ss, bias, relu = group
    rng = np.random.default_rng(GROUPS.index(group) + 100)
    found = []
    # candidates: y = acc*cs + side*ss + bias near odd half-integers t
    sides = [0] if ss == 0.0 else list(range(-128, 128))
    for _ in range(4000):
        if len(found) >= per_group:
            break
        side = int(rng.choice(sides))
        t = int(rng.integers(-80, 80)) + 0.5
        if relu and t < 0:
            t = -t
        a0 = (t - bias - side * ss) / cs
        for acc in range(int(a0) - 2, int(a0) + 3):
            if abs(acc) > ACC_LIMIT:
                continue
            v = _differs(acc, cs, None if ss == 0.0 else side, ss, bias, relu)
            if v:
                found.append((acc, None if ss == 0.0 else side, tuple(v)))
                break
    return tuple(found)


def discriminating_cases():
    """{(cs, ss, relu): [(acc, side, bias, variants)]} -- bias folded in."""
    out = {}
    for g in GROUPS:
        cs, ss, bias, relu = g
        rows = [(acc, side, bias, v) for acc, side, v in _search(g)]
        if rows:
            out.setdefault((cs, ss, relu), []).extend(rows)
    return out


def discriminating_groups():
    """[((cs, ss, bias, relu), [(acc, side, expected_int8)])] for GPU launches."""
    res = []
    for g in GROUPS:
        cs, ss, bias, relu = g
        rows = []
        for acc, side, _ in _search(g):
            rows.append((acc, side, exact.epilogue_i8(acc, cs, side, ss, bias, relu)))
        if rows:
            res.append((g, rows))
    return res


def random_tuples(n, seed):
    """(acc, conv_scale, side, side_scale, bias) with scales from a small set."""
    rng = np.random.default_rng(seed)
    scales = [float(np.float32(s)) for s in (0.05, 0.002, 0.004, 0.001, 0.5, 0.1, 1.0)]
    sscales = [float(np.float32(s)) for s in (0.0, 0.5, 0.25, 0.1, 0.3)]
    out = []
    for _ in range(n):
        mag = 10 ** rng.uniform(0, 7.5)
        acc = int(np.clip(rng.choice([-1, 1]) * mag, -2 ** 31, 2 ** 31 - 1))
        out.append((acc, scales[rng.integers(len(scales))], int(rng.integers(-128, 128)),
                    sscales[rng.integers(len(sscales))],
                    float(np.float32(rng.standard_normal() * 4))))
    return out
