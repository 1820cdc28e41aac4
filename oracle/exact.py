"""Exact-rational restatement of the int8 epilogue, for pinning the C oracle.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The epilogue of BiasActivationOutputKernel ("conv_ops_fused_int8.cc") is
three fp32 operations, each rounded once to nearest-even: a multiply by the
conv input scale, a fused multiply-add of the side input, and a bias add,
followed by round-half-to-even and a clip to [lower, 127].  Here each step is
done in exact rational arithmetic and then rounded to binary32 by an explicit
round-to-nearest-even, so the result does not depend on the host's float
unit, its fma or the compiler's contraction settings.
"""
from __future__ import annotations

from fractions import Fraction

F32_MANT = 24          # significant bits of binary32
F32_EMIN = -126        # smallest normal exponent
F32_MAX = Fraction((2 ** 24 - 1) * 2 ** (127 - 23))


def _floor_log2(a: Fraction) -> int:
    """Largest e with 2**e <= a, for a > 0."""
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    return e


def round_half_even_int(a: Fraction) -> int:
    """Nearest integer, ties to the even one."""
    n = a.numerator // a.denominator          # floor
    rem = a - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return n


def to_f32(a: Fraction) -> Fraction:
    """Round a rational to the nearest binary32 value (ties to even).

    Values beyond the largest finite binary32 are not needed by the tests and
    raise OverflowError.
    """
    if a == 0:
        return Fraction(0)
    sign = -1 if a < 0 else 1
    m = abs(a)
    e = max(_floor_log2(m), F32_EMIN)
    ulp = Fraction(2) ** (e - (F32_MANT - 1))
    n = round_half_even_int(m / ulp)
    r = n * ulp
    if r > F32_MAX:
        raise OverflowError("beyond binary32 range")
    return sign * r


def f(x: float) -> Fraction:
    """Exact value of a Python float (binary64, so any binary32 too)."""
    return Fraction(x)


def epilogue_i8(acc: int, conv_scale: float, side: int | None, side_scale: float,
                bias: float, relu, alpha: float = 0.0, beta: float = 0.0) -> int:
    """int8 result of the three-step epilogue for one element, exactly.

    relu: a bool (BiasAdd / BiasAdd+Relu) or an activation code: 2 leaky
    (y < 0: alpha*y, rounded once), 3 clipped (min(max(y, 0), alpha)),
    4 clamp (min(max(y, alpha), beta)), applied after the bias add."""
    v = to_f32(Fraction(acc))                       # int32 -> fp32
    v = to_f32(v * f(conv_scale))                   # (1) scale
    if side is not None and side_scale != 0.0:      # (2) side input, fused
        v = to_f32(Fraction(side) * f(side_scale) + v)
    v = to_f32(v + f(bias))                         # (3) bias
    act = (1 if relu else 0) if isinstance(relu, bool) else int(relu)
    a, b = f(alpha), f(beta)
    if act == 2 and v < 0:
        v = to_f32(v * a)
    elif act == 3:
        v = min(max(v, Fraction(0)), a)
    elif act == 4:
        v = min(max(v, a), b)
    r = round_half_even_int(v)
    lower = 0 if act == 1 else -128
    return max(lower, min(127, r))


def epilogue_i8_other_order(acc: int, conv_scale: float, side: int | None,
                            side_scale: float, bias: float, relu: bool,
                            variant: str) -> int:
    """The same epilogue with the operations arranged differently.

    Used only to show that a test set tells the orders apart:
      "fma_scale_bias":  v = fma(acc, scale, bias); v = fma(side, sscale, v)
                         (the older cuDNN order the page's comment describes)
      "no_side_fma":     step (2) as a rounded multiply then a rounded add
      "contract_13":     steps (1) and (3) fused into one rounding when there
                         is no side input, else (1) rounded then a rounding-free
                         side term added together with the bias
    """
    a = to_f32(Fraction(acc))
    cs, ss, b = f(conv_scale), f(side_scale), f(bias)
    use_side = side is not None and side_scale != 0.0
    if variant == "fma_scale_bias":
        v = to_f32(a * cs + b)
        if use_side:
            v = to_f32(Fraction(side) * ss + v)
    elif variant == "no_side_fma":
        v = to_f32(a * cs)
        if use_side:
            v = to_f32(to_f32(Fraction(side) * ss) + v)
        v = to_f32(v + b)
    elif variant == "contract_13":
        if use_side:
            v = to_f32(a * cs)
            v = to_f32(Fraction(side) * ss + v + b)
        else:
            v = to_f32(a * cs + b)
    else:
        raise ValueError(variant)
    r = round_half_even_int(v)
    lower = 0 if relu else -128
    return max(lower, min(127, r))
