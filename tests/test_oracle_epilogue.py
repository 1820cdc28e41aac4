"""Pins for the oracle's int8 epilogue (BiasActivationOutputKernel of
"conv_ops_fused_int8.cc"): hand-worked ties, saturation and ReLU cases, and
agreement with an exact-rational evaluation of the three rounded steps.
Also builds the set of inputs on which other orderings of the steps give a
different int8 result, which the GPU parity tests reuse.  No GPU needed."""
import numpy as np
import pytest

import oracle
from oracle import exact

from epilogue_cases import discriminating_cases, random_tuples


def _run(acc, cs, side, ss, bias, relu):
    acc = np.array([[acc]], np.int32)
    side_a = None if side is None else np.array([[side]], np.int8)
    return int(oracle.epilogue_i8(acc, np.array([bias], np.float32), side_a, cs, ss, relu)[0, 0])


@pytest.mark.parametrize("acc,cs,side,ss,bias,relu,expect", [
    # ties go to the even integer: 5*0.5 = 2.5 -> 2, 7*0.5 = 3.5 -> 4, -2.5 -> -2
    (5, 0.5, None, 0.0, 0.0, False, 2),
    (7, 0.5, None, 0.0, 0.0, False, 4),
    (-5, 0.5, None, 0.0, 0.0, False, -2),
    (-7, 0.5, None, 0.0, 0.0, False, -4),
    (1, 0.5, None, 0.0, 0.0, False, 0),
    # ReLU floors at 0, BiasAdd at -128
    (-5, 0.5, None, 0.0, 0.0, True, 0),
    (-1000, 1.0, None, 0.0, 0.0, False, -128),
    (-1000, 1.0, None, 0.0, 0.0, True, 0),
    # saturation at 127
    (1000, 1.0, None, 0.0, 0.0, False, 127),
    (127, 1.0, None, 0.0, 0.4, False, 127),
    (126, 1.0, None, 0.0, 0.6, False, 127),
    # side input: 0 + 3*0.5 = 1.5 -> 2; 0 + 5*0.5 = 2.5 -> 2
    (0, 1.0, 3, 0.5, 0.0, False, 2),
    (0, 1.0, 5, 0.5, 0.0, False, 2),
    # side scale 0 means no side term at all
    (4, 1.0, 100, 0.0, 0.0, False, 4),
    # bias: -0.5 -> -0 -> 0; 1.5 -> 2; 0.5 -> 0
    (0, 1.0, None, 0.0, -0.5, False, 0),
    (0, 1.0, None, 0.0, 1.5, False, 2),
    (0, 1.0, None, 0.0, 0.5, False, 0),
    # int32 -> fp32 rounds to nearest even: 2^24+1 -> 2^24, scaled by 2^-20 -> 16
    (2 ** 24 + 1, 2.0 ** -20, None, 0.0, 0.0, False, 16),
    # 2^24 + 3 -> 2^24 + 4 (tie to even), times 2^-2 -> 4194305 -> saturates
    (2 ** 24 + 3, 0.25, None, 0.0, 0.0, False, 127),
])
def test_epilogue_hand_cases(acc, cs, side, ss, bias, relu, expect):
    assert _run(acc, cs, side, ss, bias, relu) == expect
    assert exact.epilogue_i8(acc, cs, side, ss, bias, relu) == expect


def test_epilogue_matches_exact_rational_random():
    tuples = random_tuples(4000, seed=11)
    acc = np.array([t[0] for t in tuples], np.int32)
    for relu in (False, True):
        for (cs, ss) in {(t[1], t[3]) for t in tuples}:
            sel = [i for i, t in enumerate(tuples) if (t[1], t[3]) == (cs, ss)]
            a = acc[sel].reshape(-1, 1)
            side = np.array([tuples[i][2] for i in sel], np.int8).reshape(-1, 1)
            for i_row, i in enumerate(sel):
                bias = np.array([tuples[i][4]], np.float32)
                got = int(oracle.epilogue_i8(a[i_row:i_row + 1], bias, side[i_row:i_row + 1],
                                             cs, ss, relu)[0, 0])
                want = exact.epilogue_i8(int(a[i_row, 0]), cs, int(side[i_row, 0]), ss,
                                         float(bias[0]), relu)
                assert got == want, (tuples[i], relu)


def test_discriminating_set_tells_orders_apart():
    cases = discriminating_cases()
    assert len(cases) >= 3
    seen = set()
    for (cs, ss, relu), rows in cases.items():
        for acc, side, bias, variants in rows:
            got = _run(acc, cs, side, ss, bias, relu)
            assert got == exact.epilogue_i8(acc, cs, side, ss, bias, relu)
            for v in variants:
                assert exact.epilogue_i8_other_order(acc, cs, side, ss, bias, relu, v) != got
                seen.add(v)
    # every alternative ordering is caught by at least one case
    assert seen == {"fma_scale_bias", "no_side_fma", "contract_13"}


def test_exact_rounding_helper_pins():
    from fractions import Fraction
    # values every reader can check: 1/3 in binary32 is 11184811 * 2^-25
    assert exact.to_f32(Fraction(1, 3)) == Fraction(11184811, 2 ** 25)
    # 2^24 + 1 is a tie between 2^24 and 2^24 + 2: even mantissa wins
    assert exact.to_f32(Fraction(2 ** 24 + 1)) == 2 ** 24
    assert exact.to_f32(Fraction(2 ** 24 + 3)) == 2 ** 24 + 4
    assert exact.to_f32(Fraction(-(2 ** 24 + 3))) == -(2 ** 24 + 4)
    # numpy's float32 conversion is a library RNE rounding of a double
    rng = np.random.default_rng(12)
    for v in rng.standard_normal(200) * 1e3:
        assert exact.to_f32(Fraction(float(v))) == Fraction(float(np.float32(v)))
    assert exact.round_half_even_int(Fraction(5, 2)) == 2
    assert exact.round_half_even_int(Fraction(-5, 2)) == -2
    assert exact.round_half_even_int(Fraction(7, 2)) == 4


# ---------------------------------------------------------------- per-channel scale
# BiasActivationOutputKernel, step (1) Scale: a conv_input_scale tensor of more
# than one element is read at the output channel's offset, one value per k.

def test_per_channel_scale_matches_exact_rational():
    rng = np.random.default_rng(21)
    rows, K = 40, 24
    acc = rng.integers(-3_000_000, 3_000_000, size=(rows, K)).astype(np.int32)
    side = rng.integers(-128, 128, size=(rows, K)).astype(np.int8)
    bias = rng.normal(0.0, 3.0, size=K).astype(np.float32)
    # scales spread over many binades so a wrong channel index changes results
    sk = (2.0 ** rng.integers(-24, -12, size=K) * rng.uniform(1, 2, size=K)).astype(np.float32)
    for relu in (False, True):
        got = oracle.epilogue_i8(acc, bias, side, sk, 0.75, relu)
        for i in range(rows):
            for k in range(K):
                want = exact.epilogue_i8(int(acc[i, k]), float(sk[k]), int(side[i, k]), 0.75,
                                         float(bias[k]), relu)
                assert got[i, k] == want, (i, k, relu)


def test_per_channel_scale_with_equal_values_is_the_scalar_epilogue():
    rng = np.random.default_rng(22)
    acc = rng.integers(-2 ** 22, 2 ** 22, size=(300, 32)).astype(np.int32)
    bias = rng.normal(0.0, 1.0, size=32).astype(np.float32)
    side = rng.integers(-128, 128, size=acc.shape).astype(np.int8)
    for cs in (0.002, 1.0 / 3.0, 2.0 ** -17):
        vec = np.full(32, cs, np.float32)
        for relu in (False, True):
            assert np.array_equal(oracle.epilogue_i8(acc, bias, side, vec, 0.5, relu),
                                  oracle.epilogue_i8(acc, bias, side, cs, 0.5, relu))


def test_per_channel_scale_f64_reference():
    rng = np.random.default_rng(23)
    acc = rng.normal(0.0, 50.0, size=(64, 16))
    bias = rng.normal(0.0, 0.1, size=16).astype(np.float32)
    sk = rng.uniform(0.25, 4.0, size=16).astype(np.float32)
    side_bits = (np.arange(64 * 16, dtype=np.uint32).reshape(64, 16) % 7 + 0x3F80).astype(np.uint16)
    got = oracle.epilogue_f64(acc, bias, side_bits, sk, 0.5, False)
    side = oracle.bf16_bits_to_f64(side_bits)
    # written out per element in fp64: acc*s[k] + side*0.5 + bias[k]
    for i in range(64):
        for k in range(16):
            want = acc[i, k] * float(sk[k]) + side[i, k] * 0.5 + float(bias[k])
            assert got[i, k] == want


# ---------------------------------------------------------------- activations
# MIOpen's fusion tables list leaky Relu, clipped Relu and CLAMP as fusable
# activations; the readings are y < 0 ? alpha*y : y, min(max(y, 0), alpha)
# and min(max(y, alpha), beta), applied after the bias add.
A = oracle

def _run_act(acc, cs, bias, act, alpha, beta):
    return int(oracle.epilogue_i8(np.array([[acc]], np.int32), np.array([bias], np.float32), None,
                                  cs, 0.0, act, alpha, beta)[0, 0])


@pytest.mark.parametrize("acc,cs,bias,act,alpha,beta,expect", [
    # leaky, alpha 0.5: -5 -> -2.5 -> -2 (ties to even), -7 -> -3.5 -> -4, positives pass
    (-5, 1.0, 0.0, A.ACT_LEAKY_RELU, 0.5, 0.0, -2),
    (-7, 1.0, 0.0, A.ACT_LEAKY_RELU, 0.5, 0.0, -4),
    (6, 1.0, 0.0, A.ACT_LEAKY_RELU, 0.5, 0.0, 6),
    (-1000, 1.0, 0.0, A.ACT_LEAKY_RELU, 0.5, 0.0, -128),
    # clipped at 6: 5.5 -> 6 (tie to even), 6.5 -> 6 -> 6, negatives -> 0
    (11, 0.5, 0.0, A.ACT_CLIPPED_RELU, 6.0, 0.0, 6),
    (13, 0.5, 0.0, A.ACT_CLIPPED_RELU, 6.0, 0.0, 6),
    (9, 0.5, 0.0, A.ACT_CLIPPED_RELU, 6.0, 0.0, 4),
    (-3, 1.0, 0.0, A.ACT_CLIPPED_RELU, 6.0, 0.0, 0),
    # clipped at 2.5: 3.5 -> 2.5 -> 2
    (7, 0.5, 0.0, A.ACT_CLIPPED_RELU, 2.5, 0.0, 2),
    # clamp to [-3.5, 2.5]: -100 -> -3.5 -> -4, 100 -> 2.5 -> 2, 1 stays
    (-100, 1.0, 0.0, A.ACT_CLAMP, -3.5, 2.5, -4),
    (100, 1.0, 0.0, A.ACT_CLAMP, -3.5, 2.5, 2),
    (1, 1.0, 0.0, A.ACT_CLAMP, -3.5, 2.5, 1),
    # a clamp wider than int8: the int8 clip still applies
    (1000, 1.0, 0.0, A.ACT_CLAMP, -200.0, 300.0, 127),
    (-1000, 1.0, 0.0, A.ACT_CLAMP, -200.0, 300.0, -128),
])
def test_activation_hand_cases(acc, cs, bias, act, alpha, beta, expect):
    assert _run_act(acc, cs, bias, act, alpha, beta) == expect
    assert exact.epilogue_i8(acc, cs, None, 0.0, bias, act, alpha, beta) == expect


@pytest.mark.parametrize("act", [A.ACT_LEAKY_RELU, A.ACT_CLIPPED_RELU, A.ACT_CLAMP])
def test_activations_match_exact_rational(act):
    rng = np.random.default_rng(31 + act)
    rows, K = 60, 16
    acc = rng.integers(-4_000_000, 4_000_000, size=(rows, K)).astype(np.int32)
    side = rng.integers(-128, 128, size=(rows, K)).astype(np.int8)
    bias = rng.normal(0.0, 2.0, size=K).astype(np.float32)
    for alpha, beta in [(0.1, 0.0), (0.37, 0.0), (6.0, 0.0), (-20.5, 33.25), (2.75, 90.0)]:
        got = oracle.epilogue_i8(acc, bias, side, 2.0 ** -15, 0.5, act, alpha, beta)
        for i in range(rows):
            for k in range(K):
                want = exact.epilogue_i8(int(acc[i, k]), 2.0 ** -15, int(side[i, k]), 0.5,
                                         float(bias[k]), act,
                                         float(np.float32(alpha)), float(np.float32(beta)))
                assert got[i, k] == want, (act, alpha, beta, i, k)


def test_activations_reduce_to_relu_and_none():
    rng = np.random.default_rng(40)
    acc = rng.integers(-2 ** 22, 2 ** 22, size=(200, 32)).astype(np.int32)
    bias = rng.normal(0.0, 3.0, size=32).astype(np.float32)
    side = rng.integers(-128, 128, size=acc.shape).astype(np.int8)
    args = (acc, bias, side, 2.0 ** -14, 0.25)
    relu = oracle.epilogue_i8(*args, True)
    none = oracle.epilogue_i8(*args, False)
    assert np.array_equal(oracle.epilogue_i8(*args, A.ACT_LEAKY_RELU, 0.0), relu)
    assert np.array_equal(oracle.epilogue_i8(*args, A.ACT_CLIPPED_RELU, 127.0), relu)
    assert np.array_equal(oracle.epilogue_i8(*args, A.ACT_CLAMP, 0.0, 1e6), relu)
    assert np.array_equal(oracle.epilogue_i8(*args, A.ACT_CLAMP, -128.0, 127.0), none)
    assert np.array_equal(oracle.epilogue_i8(*args, A.ACT_LEAKY_RELU, 1.0), none)


def test_activations_f64_reference():
    rng = np.random.default_rng(41)
    acc = rng.normal(0.0, 3.0, size=(50, 8))
    bias = rng.normal(0.0, 0.5, size=8).astype(np.float32)
    for act, alpha, beta in [(A.ACT_LEAKY_RELU, 0.2, 0.0), (A.ACT_CLIPPED_RELU, 1.5, 0.0),
                             (A.ACT_CLAMP, -1.25, 2.0)]:
        got = oracle.epilogue_f64(acc, bias, None, 1.0, 0.0, act, alpha, beta)
        a, b = float(np.float32(alpha)), float(np.float32(beta))
        for i in range(50):
            for k in range(8):
                v = acc[i, k] + float(bias[k])
                if act == A.ACT_LEAKY_RELU:
                    want = v * a if v < 0 else v
                elif act == A.ACT_CLIPPED_RELU:
                    want = min(max(v, 0.0), a)
                else:
                    want = min(max(v, a), b)
                assert got[i, k] == want
