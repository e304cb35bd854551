"""Pins for the fp64 backward oracle: things other than the backward itself.

- central finite differences of the FORWARD oracle (a separate function) for
  every gradient, on small cases with non-square weights (so a transposed
  operand fails), soft masks, two batch elements and both directions;
- the incoming/outgoing transpose identity, applied to the gradients (with
  the a/b weight swap of the forward identity);
- the LayerNorm invariant: the gradient of z sums to zero over D for every
  pair (LN_in subtracts the mean);
- linearity in dout, and zero gradients for zero dout.
"""

import math

import numpy as np
import pytest

from oracle import trimul_backward as OB
from oracle import trimul_oracle as O


def rand_case(rng, B, N, D, C):
    p = {
        "W_a": rng.standard_normal((C, D)) / math.sqrt(D),
        "W_ga": rng.standard_normal((C, D)) / math.sqrt(D),
        "W_b": rng.standard_normal((C, D)) / math.sqrt(D),
        "W_gb": rng.standard_normal((C, D)) / math.sqrt(D),
        "W_o": rng.standard_normal((D, C)) / math.sqrt(C),
        "W_g": rng.standard_normal((D, D)) / math.sqrt(D),
        "ln_in_gamma": 1 + 0.3 * rng.standard_normal(D),
        "ln_in_beta": 0.3 * rng.standard_normal(D),
        "ln_out_gamma": 1 + 0.3 * rng.standard_normal(C),
        "ln_out_beta": 0.3 * rng.standard_normal(C),
    }
    z = rng.standard_normal((B, N, N, D))
    m = rng.random((B, N, N))
    m[:, 0, :] = 1.0
    m[:, :, 1] = 0.0        # some exactly masked pairs
    dout = rng.standard_normal((B, N, N, D))
    return z, m, p, dout


def loss(z, m, p, direction, dout, eps):
    return float((O.trimul_forward(z, m, p, direction, eps=eps) * dout).sum())


def central_difference(f, arr, h=1e-5):
    """d f / d arr by central differences, one element at a time (arr is
    perturbed in place and restored)."""
    g = np.zeros_like(arr)
    it = np.nditer(arr, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = arr[i]
        arr[i] = old + h
        fp = f()
        arr[i] = old - h
        fm = f()
        arr[i] = old
        g[i] = (fp - fm) / (2 * h)
    return g


@pytest.mark.parametrize("direction", ["outgoing", "incoming"])
def test_every_gradient_matches_finite_differences(direction):
    rng = np.random.default_rng(11 if direction == "outgoing" else 12)
    B, N, D, C, eps = 2, 4, 5, 3, 1e-5
    z, m, p, dout = rand_case(rng, B, N, D, C)
    got = OB.trimul_backward(z, m, p, direction, dout, eps=eps)
    f = lambda: loss(z, m, p, direction, dout, eps)  # noqa: E731
    fd = {"dz": central_difference(f, z)}
    for k in OB.GRAD_KEYS:
        fd[k] = central_difference(f, p[k])
    for k, ref in fd.items():
        assert got[k].shape == ref.shape, k
        scale = np.abs(ref).max()
        assert scale > 1e-3, f"{k}: finite difference is ~0, the case does not exercise it"
        np.testing.assert_allclose(got[k], ref, rtol=1e-6, atol=1e-7 * scale, err_msg=k)


def test_gradients_with_eps_dominated_layer_norm():
    """A pair row that is nearly constant (variance << eps) keeps eps in the
    LayerNorm derivative; finite differences still agree."""
    rng = np.random.default_rng(13)
    z, m, p, dout = rand_case(rng, 1, 3, 4, 2)
    z[0, 1, 2] = 0.7 + 1e-4 * rng.standard_normal(4)
    eps = 1e-3
    got = OB.trimul_backward(z, m, p, "outgoing", dout, eps=eps)
    f = lambda: loss(z, m, p, "outgoing", dout, eps)  # noqa: E731
    np.testing.assert_allclose(got["dz"], central_difference(f, z, h=1e-6), rtol=1e-5, atol=1e-8)


def test_transpose_identity_on_gradients():
    """incoming(z; a, b) = T(outgoing(z^T; b, a)) for the forward, hence the
    incoming gradients equal the transposed outgoing gradients of the
    transposed problem, with the a and b weight gradients swapped."""
    rng = np.random.default_rng(14)
    z, m, p, dout = rand_case(rng, 2, 5, 6, 4)
    t = lambda u: np.swapaxes(u, 1, 2)  # noqa: E731
    gi = OB.trimul_backward(z, m, p, "incoming", dout)
    ps = dict(p, W_a=p["W_b"], W_ga=p["W_gb"], W_b=p["W_a"], W_gb=p["W_ga"])
    go = OB.trimul_backward(t(z), t(m), ps, "outgoing", t(dout))
    np.testing.assert_allclose(gi["dz"], t(go["dz"]), rtol=1e-10, atol=1e-12)
    swap = {"W_a": "W_b", "W_ga": "W_gb", "W_b": "W_a", "W_gb": "W_ga"}
    for k in OB.GRAD_KEYS:
        np.testing.assert_allclose(gi[k], go[swap.get(k, k)], rtol=1e-10, atol=1e-12, err_msg=k)


@pytest.mark.parametrize("direction", ["outgoing", "incoming"])
def test_dz_sums_to_zero_over_features(direction):
    rng = np.random.default_rng(15)
    z, m, p, dout = rand_case(rng, 1, 6, 8, 4)
    dz = OB.trimul_backward(z, m, p, direction, dout)["dz"]
    assert np.abs(dz.sum(-1)).max() <= 1e-12 * np.abs(dz).max() * 8


def test_linear_in_dout_and_zero_for_zero_dout():
    rng = np.random.default_rng(16)
    z, m, p, d1 = rand_case(rng, 1, 4, 6, 3)
    d2 = rng.standard_normal(d1.shape)
    g1 = OB.trimul_backward(z, m, p, "outgoing", d1)
    g2 = OB.trimul_backward(z, m, p, "outgoing", d2)
    g12 = OB.trimul_backward(z, m, p, "outgoing", 2.0 * d1 - 3.0 * d2)
    g0 = OB.trimul_backward(z, m, p, "outgoing", np.zeros_like(d1))
    for k in ("dz",) + OB.GRAD_KEYS:
        np.testing.assert_allclose(g12[k], 2.0 * g1[k] - 3.0 * g2[k], rtol=1e-9, atol=1e-11, err_msg=k)
        assert np.all(g0[k] == 0), k


def test_backward_flop_count():
    B, N, D, C = 2, 16, 8, 4
    P = B * N * N
    fwd = O.gemm_flops(B, N, D, C)
    bwd = (2 * P * (D * C + D * D) + 4 * B * C * N ** 3 + 2 * P * 4 * C * D
           + 2 * P * (D * C + D * D) + 2 * P * 4 * C * D)
    assert OB.backward_flops(B, N, D, C) == fwd + bwd
