"""Pins for the fp64 oracle: things other than the oracle itself that fix its values.

- an independent pure-Python brute force (scalar loops, math module only);
- a hand-derived closed-form example stored under tests/golden/;
- closed forms: two-element LayerNorm, N = 1, zero gate weights, fully masked pairs;
- invariants: token-permutation equivariance, the incoming/outgoing transpose
  identity (with the a/b weight swap), masked-position insensitivity,
  LayerNorm shift/scale behaviour, sampled evaluation == full evaluation.
"""

import json
import math
import os

import numpy as np
import pytest

from oracle import trimul_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers

def rand_case(rng, B, N, D, C, mask_kind="tokens"):
    p = {
        "W_a": rng.standard_normal((C, D)) / math.sqrt(D),
        "W_ga": rng.standard_normal((C, D)) / math.sqrt(D),
        "W_b": rng.standard_normal((C, D)) / math.sqrt(D),
        "W_gb": rng.standard_normal((C, D)) / math.sqrt(D),
        "W_o": rng.standard_normal((D, C)) / math.sqrt(C),
        "W_g": rng.standard_normal((D, D)) / math.sqrt(D),
        "ln_in_gamma": 1 + 0.1 * rng.standard_normal(D),
        "ln_in_beta": 0.1 * rng.standard_normal(D),
        "ln_out_gamma": 1 + 0.1 * rng.standard_normal(C),
        "ln_out_beta": 0.1 * rng.standard_normal(C),
    }
    z = rng.standard_normal((B, N, N, D))
    if mask_kind == "ones":
        m = np.ones((B, N, N))
    elif mask_kind == "tokens":
        t = (rng.random((B, N)) > 0.3).astype(np.float64)
        t[:, 0] = 1.0
        m = t[:, :, None] * t[:, None, :]
    else:  # arbitrary weights in [0, 1]
        m = rng.random((B, N, N))
    return z, m, p


def brute_force(z, m, p, direction, eps):
    """Scalar-loop TriMul written independently of the oracle (lists + math only)."""
    B, N, D = len(z), len(z[0]), len(z[0][0][0])
    C = len(p["W_a"])

    def ln(vec, g, b):
        n = len(vec)
        mu = sum(vec) / n
        var = sum((v - mu) * (v - mu) for v in vec) / n
        r = 1.0 / math.sqrt(var + eps)
        return [(vec[d] - mu) * r * g[d] + b[d] for d in range(n)]

    def dot(u, w):
        s = 0.0
        for ui, wi in zip(u, w):
            s += ui * wi
        return s

    def sig(t):
        return 1.0 / (1.0 + math.exp(-t))

    zn = [[[ln(list(z[b][i][j]), p["ln_in_gamma"], p["ln_in_beta"]) for j in range(N)]
           for i in range(N)] for b in range(B)]
    A = [[[[sig(dot(zn[b][i][j], p["W_ga"][c])) * dot(zn[b][i][j], p["W_a"][c]) * m[b][i][j]
            for c in range(C)] for j in range(N)] for i in range(N)] for b in range(B)]
    Bv = [[[[sig(dot(zn[b][i][j], p["W_gb"][c])) * dot(zn[b][i][j], p["W_b"][c]) * m[b][i][j]
             for c in range(C)] for j in range(N)] for i in range(N)] for b in range(B)]
    out = []
    for b in range(B):
        ob = []
        for i in range(N):
            oi = []
            for j in range(N):
                x = []
                for c in range(C):
                    s = 0.0
                    for k in range(N):
                        if direction == "outgoing":
                            s += A[b][i][k][c] * Bv[b][j][k][c]
                        else:
                            s += A[b][k][i][c] * Bv[b][k][j][c]
                    x.append(s)
                y = ln(x, p["ln_out_gamma"], p["ln_out_beta"])
                oi.append([sig(dot(zn[b][i][j], p["W_g"][d])) * dot(y, p["W_o"][d]) for d in range(D)])
            ob.append(oi)
        out.append(ob)
    return np.array(out)


def listify(p):
    return {k: np.asarray(v).tolist() for k, v in p.items()}


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("direction", ["outgoing", "incoming"])
@pytest.mark.parametrize("mask_kind", ["ones", "tokens", "weights"])
def test_oracle_matches_brute_force(direction, mask_kind):
    rng = np.random.default_rng(11 if direction == "outgoing" else 12)
    z, m, p = rand_case(rng, B=2, N=5, D=6, C=3, mask_kind=mask_kind)
    eps = 1e-5
    ref = brute_force(z.tolist(), m.tolist(), listify(p), direction, eps)
    got = O.trimul_forward(z, m, p, direction, eps=eps)
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)


def test_brute_force_distinguishes_directions_and_weight_swap():
    """The pins above would fail on a transposed operand or an a/b swap."""
    rng = np.random.default_rng(5)
    z, m, p = rand_case(rng, B=1, N=4, D=4, C=2, mask_kind="ones")
    out_o = O.trimul_forward(z, m, p, "outgoing")
    out_i = O.trimul_forward(z, m, p, "incoming")
    q = dict(p)
    q["W_a"], q["W_b"], q["W_ga"], q["W_gb"] = p["W_b"], p["W_a"], p["W_gb"], p["W_ga"]
    out_swapped = O.trimul_forward(z, m, q, "outgoing")
    assert np.abs(out_o - out_i).max() > 1e-3
    assert np.abs(out_o - out_swapped).max() > 1e-3


# ---------------------------------------------------------------- golden closed form

@pytest.mark.parametrize("direction", ["outgoing", "incoming"])
def test_hand_derived_golden(direction):
    with open(os.path.join(GOLDEN, "trimul_2x2_closed_form.json")) as f:
        g = json.load(f)
    p = {k: np.array(g[k], dtype=np.float64) for k in O.PARAM_KEYS}
    z = np.array(g["z"], dtype=np.float64)
    got = O.trimul_forward(z, None, p, direction, eps=g["eps"])
    np.testing.assert_allclose(got, np.array(g["expected"][direction]), rtol=0, atol=1e-14)


# ---------------------------------------------------------------- closed forms

def test_layer_norm_two_elements_closed_form():
    """LN([u, v]) = sign(u-v) * h / sqrt(h^2 + eps) * [1, -1] * gamma + beta with h = |u-v|/2."""
    rng = np.random.default_rng(3)
    for _ in range(20):
        u, v = rng.standard_normal(2) * 3
        g = rng.standard_normal(2)
        b = rng.standard_normal(2)
        eps = 10 ** rng.uniform(-6, 0)
        h = (u - v) / 2
        want = np.array([h, -h]) / math.sqrt(h * h + eps) * g + b
        np.testing.assert_allclose(O.layer_norm(np.array([u, v]), g, b, eps), want, rtol=1e-13, atol=1e-14)


def test_layer_norm_constant_vector_gives_beta():
    g = np.array([2.0, -1.0, 0.5])
    b = np.array([0.1, 0.2, 0.3])
    np.testing.assert_array_equal(O.layer_norm(np.full(3, 7.25), g, b, 1e-5), b)


def test_layer_norm_shift_scale_moves_eps():
    """LN_eps(alpha z + c) == LN_{eps/alpha^2}(z) for alpha > 0 (exact identity)."""
    rng = np.random.default_rng(4)
    z = rng.standard_normal((7, 16))
    g, b = rng.standard_normal(16), rng.standard_normal(16)
    for alpha, c in [(3.0, 5.0), (0.01, -2.0), (250.0, 1e3)]:
        np.testing.assert_allclose(O.layer_norm(alpha * z + c, g, b, 1e-5),
                                   O.layer_norm(z, g, b, 1e-5 / alpha ** 2), rtol=1e-9, atol=1e-9)


@pytest.mark.parametrize("direction", ["outgoing", "incoming"])
def test_n1_closed_form(direction):
    """N = 1: the contraction has one term, x[c] = a[c] b[c]."""
    rng = np.random.default_rng(6)
    z, m, p = rand_case(rng, B=3, N=1, D=8, C=5, mask_kind="ones")
    out, inter = O.trimul_forward(z, m, p, direction, return_intermediates=True)
    np.testing.assert_allclose(inter["x"], inter["a"] * inter["b"], rtol=1e-14, atol=0)


def test_zero_gate_weights_give_half():
    """sigmoid(0) = 1/2: with W_ga = 0 the gate of a is exactly one half."""
    rng = np.random.default_rng(7)
    z, m, p = rand_case(rng, B=1, N=3, D=4, C=2, mask_kind="weights")
    p["W_ga"] = np.zeros_like(p["W_ga"])
    _, inter = O.trimul_forward(z, m, p, "outgoing", return_intermediates=True)
    want = 0.5 * (inter["zn"] @ p["W_a"].T) * m[..., None]
    np.testing.assert_allclose(inter["a"], want, rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("direction", ["outgoing", "incoming"])
def test_fully_masked_gives_beta_projection(direction):
    """m = 0 everywhere: x = 0, LN_out(0) = beta_out, out = sigmoid(z' W_g^T) * (beta_out W_o^T)."""
    rng = np.random.default_rng(8)
    z, m, p = rand_case(rng, B=1, N=4, D=6, C=3)
    m = np.zeros_like(m)
    out, inter = O.trimul_forward(z, m, p, direction, return_intermediates=True)
    assert np.all(inter["x"] == 0)
    gate = 1 / (1 + np.exp(-(inter["zn"] @ p["W_g"].T)))
    np.testing.assert_allclose(out, gate * (p["ln_out_beta"] @ p["W_o"].T), rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("direction", ["outgoing", "incoming"])
def test_permutation_equivariance(direction):
    """Permuting the tokens of z and the mask permutes out identically on both token axes."""
    rng = np.random.default_rng(9)
    z, m, p = rand_case(rng, B=2, N=7, D=8, C=4)
    perm = rng.permutation(7)
    out = O.trimul_forward(z, m, p, direction)
    out_p = O.trimul_forward(z[:, perm][:, :, perm], m[:, perm][:, :, perm], p, direction)
    np.testing.assert_allclose(out_p, out[:, perm][:, :, perm], rtol=1e-12, atol=1e-13)


def test_incoming_equals_transposed_outgoing_with_swapped_weights():
    """incoming(z, m; a, b) = transpose_ij(outgoing(z^T, m^T; b, a)).

    Outgoing on z^T with the a/b weights swapped gives x'[i,j] = sum_k b[k,i] a[k,j]
    = x_in[j,i], and the output gate is read at (i, j) of z^T = (j, i) of z.
    """
    rng = np.random.default_rng(10)
    z, m, p = rand_case(rng, B=2, N=6, D=8, C=4)
    q = dict(p)
    q["W_a"], q["W_ga"], q["W_b"], q["W_gb"] = p["W_b"], p["W_gb"], p["W_a"], p["W_ga"]
    zt = np.swapaxes(z, 1, 2)
    mt = np.swapaxes(m, 1, 2)
    out_in = O.trimul_forward(z, m, p, "incoming")
    out_t = O.trimul_forward(zt, mt, q, "outgoing")
    np.testing.assert_allclose(out_in, np.swapaxes(out_t, 1, 2), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("direction", ["outgoing", "incoming"])
def test_masked_positions_do_not_matter(direction):
    """Changing z where m = 0 leaves out unchanged wherever m = 1 (a = b = 0 exactly there)."""
    rng = np.random.default_rng(13)
    z, m, p = rand_case(rng, B=2, N=8, D=6, C=3, mask_kind="tokens")
    z2 = z.copy()
    z2[m == 0] = rng.standard_normal(z2[m == 0].shape) * 10
    out = O.trimul_forward(z, m, p, direction)
    out2 = O.trimul_forward(z2, m, p, direction)
    keep = m == 1
    assert keep.sum() > 0 and (~keep).sum() > 0
    np.testing.assert_array_equal(out[keep], out2[keep])


def test_mask_scale_scales_x_quadratically():
    """A constant mask value s scales a and b by s and x by s^2."""
    rng = np.random.default_rng(14)
    z, _, p = rand_case(rng, B=1, N=5, D=4, C=3, mask_kind="ones")
    s = 0.37
    _, i1 = O.trimul_forward(z, np.ones((1, 5, 5)), p, "outgoing", return_intermediates=True)
    _, i2 = O.trimul_forward(z, np.full((1, 5, 5), s), p, "outgoing", return_intermediates=True)
    np.testing.assert_allclose(i2["x"], s * s * i1["x"], rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("direction", ["outgoing", "incoming"])
def test_sampled_equals_full(direction):
    rng = np.random.default_rng(15)
    z, m, p = rand_case(rng, B=2, N=9, D=8, C=4)
    full = O.trimul_forward(z, m, p, direction)
    rows = [np.array([0, 3, 8]), np.array([2, 5])]
    cols = [np.array([1, 3, 4, 7]), np.array([0, 8])]
    got = O.trimul_forward_sampled(z, m, p, direction, rows, cols)
    for b in range(2):
        np.testing.assert_allclose(got[b], full[b][np.ix_(rows[b], cols[b])], rtol=1e-12, atol=1e-13)


def test_gemm_flop_count_matches_definition():
    """Four D->C projections, one N^3 contraction per channel, two output projections."""
    B, N, D, C = 2, 8, 16, 4
    assert O.gemm_flops(B, N, D, C) == B * (4 * (2 * N * N * D * C) + C * (2 * N ** 3)
                                              + 2 * N * N * C * D + 2 * N * N * D * D)
