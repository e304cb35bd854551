"""fp64 CPU oracle for the forward pass of the triangular multiplicative update (TriMul).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
links this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may use it.  It shares no code, table or helper
with the CUDA path under ``co_folding_pair_gb300/``.

What it computes
----------------
The fold-cp-ops README ("Use" section) builds the layer from six sub-modules:
``norm_in`` and ``norm_out`` (``nn.LayerNorm(D)``), ``p_in`` and ``g_in``
(``nn.Linear(D, 2D, bias=False)``), ``p_out`` and ``g_out``
(``nn.Linear(D, D, bias=False)``), and takes a ``direction`` ("outgoing" or
"incoming") and a pair mask of shape (B, N, N).  The pages never write the
update's equation; this oracle takes the standard triangular multiplicative
update that those parts assemble into, with the width of ``a`` and ``b``
called C (the README's layer has C = D):

    z'        = LN_in(z)                                   per pair, over D
    a[..., c] = sigmoid(z' . W_ga[c]) * (z' . W_a[c]) * m  per pair
    b[..., c] = sigmoid(z' . W_gb[c]) * (z' . W_b[c]) * m  per pair
    outgoing: x[b,i,j,c] = sum_k a[b,i,k,c] * b[b,j,k,c]
    incoming: x[b,i,j,c] = sum_k a[b,k,i,c] * b[b,k,j,c]
    out       = sigmoid(z' W_g^T) * (LN_out(x) W_o^T)

Weights use the ``nn.Linear`` layout (out_features, in_features):
W_a, W_ga, W_b, W_gb are [C, D], W_o is [D, C], W_g is [D, D].  LayerNorm is
``nn.LayerNorm``'s: biased variance, ``eps`` inside the square root, then the
affine gamma/beta.  The mask multiplies ``a`` and ``b`` only; ``out`` is not
masked.

Everything is evaluated in float64 from the exact values passed in (bf16
inputs are widened exactly).  Matrix products use ``numpy.matmul`` as a
library primitive; nothing is blocked, fused or reordered beyond the
definition above.

Pins
----
Every function here is pinned in ``tests/test_oracle_pins.py`` against
things other than itself: an independent pure-Python brute force on tiny
inputs, closed forms (a two-element LayerNorm, N = 1, zero gate weights, a
fully masked row), and invariants (token permutation equivariance, the
incoming/outgoing transpose identity, masked-position insensitivity, LayerNorm
shift/scale invariance, sampled == full).
"""

from __future__ import annotations

import numpy as np

OUTGOING = "outgoing"
INCOMING = "incoming"

# Names of the weight arrays, in nn.Linear (out, in) layout.
PARAM_KEYS = ("W_a", "W_ga", "W_b", "W_gb", "W_o", "W_g",
              "ln_in_gamma", "ln_in_beta", "ln_out_gamma", "ln_out_beta")


def _f64(v):
    return np.asarray(v, dtype=np.float64)


def layer_norm(v, gamma, beta, eps):
    """LayerNorm over the last axis, as ``torch.nn.LayerNorm``.

    fold-cp-ops README, "Use": ``norm_in`` / ``norm_out`` are ``nn.LayerNorm``;
    that module normalises with the biased variance and adds ``eps`` under
    the square root before the affine step.
    """
    v = _f64(v)
    mu = v.mean(axis=-1, keepdims=True)
    var = ((v - mu) ** 2).mean(axis=-1, keepdims=True)
    return (v - mu) / np.sqrt(var + eps) * _f64(gamma) + _f64(beta)


def sigmoid(t):
    """Logistic function 1 / (1 + exp(-t)) in float64."""
    t = _f64(t)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-t))


def gated_projection(zn, W_value, W_gate, mask):
    """One gated input projection: sigmoid(zn W_gate^T) * (zn W_value^T) * mask.

    fold-cp-ops README, "Use": ``p_in`` and ``g_in`` are the value and gate
    projections (bias-free ``nn.Linear``); the pair mask of shape (B, N, N)
    multiplies the projected pair features.  ``zn`` is [..., D], ``mask`` is
    [...] and the result is [..., C].
    """
    zn = _f64(zn)
    value = zn @ _f64(W_value).T
    gate = sigmoid(zn @ _f64(W_gate).T)
    return gate * value * _f64(mask)[..., None]


def triangle(a, b, direction):
    """The triangle contraction over the third token k, per batch and channel.

    fold-cp-ops README, "Use": ``direction="outgoing"`` or ``"incoming"``.
    ``a`` and ``b`` are [B, N, N, C]; the result is [B, N, N, C].

    outgoing: x[b,i,j,c] = sum_k a[b,i,k,c] b[b,j,k,c]   (X_c = A_c B_c^T)
    incoming: x[b,i,j,c] = sum_k a[b,k,i,c] b[b,k,j,c]   (X_c = A_c^T B_c)
    """
    a = _f64(a)
    b = _f64(b)
    A = np.moveaxis(a, -1, 1)  # [B, C, N, N]: A[b, c, i, k] = a[b, i, k, c]
    Bm = np.moveaxis(b, -1, 1)
    if direction == OUTGOING:
        X = A @ np.swapaxes(Bm, -1, -2)
    elif direction == INCOMING:
        X = np.swapaxes(A, -1, -2) @ Bm
    else:
        raise ValueError(f"direction must be 'outgoing' or 'incoming', got {direction!r}")
    return np.moveaxis(X, 1, -1)


def output_projection(x, zn, params, eps):
    """out = sigmoid(zn W_g^T) * (LN_out(x) W_o^T), per pair.

    fold-cp-ops README, "Use": ``norm_out`` then ``p_out``, gated by ``g_out``
    applied to the normalised input pair features.
    """
    y = layer_norm(x, params["ln_out_gamma"], params["ln_out_beta"], eps)
    return sigmoid(_f64(zn) @ _f64(params["W_g"]).T) * (y @ _f64(params["W_o"]).T)


def trimul_forward(z, mask, params, direction, eps=1e-5, return_intermediates=False):
    """Full TriMul forward on a [B, N, N, D] pair representation.

    ``mask`` is [B, N, N] or None (all ones).  Returns ``out`` [B, N, N, D]
    and, when asked, a dict with z', a, b and x (all float64).
    """
    z = _f64(z)
    if z.ndim != 4 or z.shape[1] != z.shape[2]:
        raise ValueError(f"z must be [B, N, N, D], got {z.shape}")
    m = np.ones(z.shape[:3]) if mask is None else _f64(mask)
    zn = layer_norm(z, params["ln_in_gamma"], params["ln_in_beta"], eps)
    a = gated_projection(zn, params["W_a"], params["W_ga"], m)
    b = gated_projection(zn, params["W_b"], params["W_gb"], m)
    x = triangle(a, b, direction)
    out = output_projection(x, zn, params, eps)
    if return_intermediates:
        return out, {"zn": zn, "a": a, "b": b, "x": x}
    return out


def trimul_forward_sampled(z, mask, params, direction, rows, cols, eps=1e-5):
    """TriMul forward evaluated exactly at the grid of pairs rows x cols, per batch.

    ``rows`` and ``cols`` are lists (one entry per batch) of 1-D integer
    arrays of token indices.  The result is a list of [len(rows[b]),
    len(cols[b]), D] arrays with out[b, rows[b][r], cols[b][s], :].

    This is the definition restricted to what those outputs depend on:
    outgoing needs the token rows a[b, i, :, :] (i in rows) and b[b, j, :, :]
    (j in cols); incoming needs the token columns a[b, :, i, :] and
    b[b, :, j, :].  Each needed line is computed once with the same functions
    as the full evaluation.
    """
    if not hasattr(z, "shape"):
        z = np.asarray(z)
    # z may be any array-like with .shape and numpy-style indexing; each slice
    # is widened to float64 on its own, so a full copy of z is never made.
    B, N = z.shape[0], z.shape[1]
    m = np.ones((B, N, N)) if mask is None else mask
    results = []
    for bb in range(B):
        ri = np.asarray(rows[bb], dtype=np.int64)
        cj = np.asarray(cols[bb], dtype=np.int64)
        g_in, be_in = params["ln_in_gamma"], params["ln_in_beta"]
        zb = z[bb]                       # [N, N, D]
        mb = np.asarray(m[bb])            # [N, N]
        if direction == OUTGOING:
            # a[b, i, k, :] for i in rows, b[b, j, k, :] for j in cols
            z_a, m_a = _f64(zb[ri, :, :]), _f64(mb[ri, :])       # [R, K, D], [R, K]
            z_b, m_b = _f64(zb[cj, :, :]), _f64(mb[cj, :])       # [S, K, D], [S, K]
        elif direction == INCOMING:
            # a[b, k, i, :] for i in rows, b[b, k, j, :] for j in cols
            z_a, m_a = _f64(np.swapaxes(zb[:, ri, :], 0, 1)), _f64(mb[:, ri].T)
            z_b, m_b = _f64(np.swapaxes(zb[:, cj, :], 0, 1)), _f64(mb[:, cj].T)
        else:
            raise ValueError(f"direction must be 'outgoing' or 'incoming', got {direction!r}")
        a_lines = gated_projection(layer_norm(z_a, g_in, be_in, eps), params["W_a"], params["W_ga"], m_a)
        b_lines = gated_projection(layer_norm(z_b, g_in, be_in, eps), params["W_b"], params["W_gb"], m_b)
        # x[r, s, c] = sum_k a_lines[r, k, c] * b_lines[s, k, c]; both directions
        # reduce to this once the lines are indexed by the contracted token k.
        A = np.moveaxis(a_lines, -1, 0)  # [C, R, K]
        Bm = np.moveaxis(b_lines, -1, 0)  # [C, S, K]
        x = np.moveaxis(A @ np.swapaxes(Bm, -1, -2), 0, -1)  # [R, S, C]
        zn = layer_norm(_f64(zb[np.ix_(ri, cj)]), g_in, be_in, eps)  # [R, S, D]
        results.append(output_projection(x, zn, params, eps))
    return results


def gemm_flops(B, N, D, C):
    """Algorithmic GEMM FLOPs of one forward: in-projections, triangle, out-projection."""
    return B * (2 * N * N * D * 4 * C + 2 * C * N ** 3 + 2 * N * N * (D * D + C * D))
