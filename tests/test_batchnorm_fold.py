"""Batch-norm inference folded into the per-channel conv scale and bias
(fconv_fold_batchnorm), checked on the host against the normalisation it
replaces.  MIOpen's "use-fusion-api" page lists BatchNorm inference among the
fusable operators (the CBNA combination) without a formula; the reading is
the per-channel inference form gamma * (y - mean) / sqrt(var + eps) + beta on
the biased conv output y = acc * conv_scale + bias."""
import math

import numpy as np
import pytest

import quantized_conv2d_gb300 as fc


def _params(seed, K):
    rng = np.random.default_rng(seed)
    return dict(
        gamma=rng.uniform(0.2, 3.0, K).astype(np.float32) * rng.choice([-1, 1], K).astype(np.float32),
        beta=rng.normal(0, 2, K).astype(np.float32),
        mean=rng.normal(0, 5, K).astype(np.float32),
        var=rng.uniform(0.01, 9.0, K).astype(np.float32),
        bias=rng.normal(0, 1, K).astype(np.float32),
    )


@pytest.mark.parametrize("seed,cs,eps", [(0, 0.002, 1e-5), (1, 1.0, 1e-3), (2, 3.0e-4, 0.0)])
def test_folded_affine_equals_the_normalisation(seed, cs, eps):
    K = 97
    p = _params(seed, K)
    scale_k, bias_k = fc.fconv_fold_batchnorm(cs, p["gamma"], p["beta"], p["mean"], p["var"], eps,
                                              bias=p["bias"])
    rng = np.random.default_rng(100 + seed)
    acc = rng.integers(-(1 << 26), 1 << 26, size=(64, K)).astype(np.float64)
    f64 = lambda a: a.astype(np.float64)
    # the normalisation applied to the biased conv output, in double, with
    # the float32 scale and eps the call receives
    cs32, eps32 = float(np.float32(cs)), float(np.float32(eps))
    y = acc * cs32 + f64(p["bias"])
    want = f64(p["gamma"]) * (y - f64(p["mean"])) / np.sqrt(f64(p["var"]) + eps32) + f64(p["beta"])
    got = acc * f64(scale_k) + f64(bias_k)
    # scale_k and bias_k are each one float rounding of their exact values
    tol = 2.0 ** -24 * (np.abs(acc * f64(scale_k)) + np.abs(f64(bias_k))) * 1.0001 + 1e-9
    assert np.all(np.abs(got - want) <= tol)


def test_unit_normalisation_leaves_scale_and_bias():
    """var + eps = 4 and gamma = 2 give g = 1 exactly; beta = mean cancels."""
    K = 8
    mean = np.linspace(-3, 3, K).astype(np.float32)
    bias = np.linspace(-1, 1, K).astype(np.float32)
    scale_k, bias_k = fc.fconv_fold_batchnorm(0.125, np.full(K, 2.0, np.float32), mean, mean,
                                              np.full(K, 3.75, np.float32), 0.25, bias=bias)
    assert np.array_equal(scale_k, np.full(K, 0.125, np.float32))
    assert np.array_equal(bias_k, bias)


def test_missing_bias_is_zero():
    p = _params(5, 16)
    a = fc.fconv_fold_batchnorm(0.5, p["gamma"], p["beta"], p["mean"], p["var"], 1e-5)
    b = fc.fconv_fold_batchnorm(0.5, p["gamma"], p["beta"], p["mean"], p["var"], 1e-5,
                                bias=np.zeros(16, np.float32))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_single_rounding_from_double():
    """Each output is the double-precision value rounded once to float."""
    p = _params(7, 33)
    cs, eps = 0.003, 1e-5
    scale_k, bias_k = fc.fconv_fold_batchnorm(cs, p["gamma"], p["beta"], p["mean"], p["var"], eps,
                                              bias=p["bias"])
    for k in range(33):
        g = float(p["gamma"][k]) / math.sqrt(float(p["var"][k]) + float(np.float32(eps)))
        assert scale_k[k] == np.float32(float(np.float32(cs)) * g)
        assert bias_k[k] == np.float32((float(p["bias"][k]) - float(p["mean"][k])) * g
                                       + float(p["beta"][k]))


def _err(fn, *args, **kw):
    with pytest.raises(fc.FconvError) as ei:
        fn(*args, **kw)
    return ei.value.status


def test_invalid_arguments():
    p = _params(9, 4)
    args = (1.0, p["gamma"], p["beta"], p["mean"])
    assert _err(fc.fconv_fold_batchnorm, *args, p["var"], -1e-3) == fc.FCONV_ERR_INVALID_VALUE
    assert _err(fc.fconv_fold_batchnorm, *args, p["var"], float("nan")) == fc.FCONV_ERR_INVALID_VALUE
    assert _err(fc.fconv_fold_batchnorm, *args, np.array([1, 0, 1, 1], np.float32), 0.0) == \
        fc.FCONV_ERR_INVALID_VALUE
    assert _err(fc.fconv_fold_batchnorm, *args, np.array([1, -2, 1, 1], np.float32), 1.0) == \
        fc.FCONV_ERR_INVALID_VALUE
    with pytest.raises(ValueError):
        fc.fconv_fold_batchnorm(1.0, p["gamma"], p["beta"][:3], p["mean"], p["var"], 1e-5)
    lib = fc._load()
    out = np.zeros(4, np.float32)
    assert lib.fconv_fold_batchnorm(0, 1.0, None, p["gamma"].ctypes.data, p["beta"].ctypes.data,
                                    p["mean"].ctypes.data, p["var"].ctypes.data, 1e-5,
                                    out.ctypes.data, out.ctypes.data) == fc.FCONV_ERR_INVALID_VALUE
    assert lib.fconv_fold_batchnorm(4, 1.0, None, None, p["beta"].ctypes.data,
                                    p["mean"].ctypes.data, p["var"].ctypes.data, 1e-5,
                                    out.ctypes.data, out.ctypes.data) == fc.FCONV_ERR_INVALID_VALUE
