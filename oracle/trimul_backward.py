"""fp64 CPU oracle for the backward pass (gradients) of the TriMul forward.

TEST INFRASTRUCTURE ONLY, like the forward oracle beside it: nothing on the
product path imports, calls or links this module.

What it computes
----------------
The fold-cp-ops README ("Use" section) ships the layer for inference only;
its backward is not on the pages.  This is the plain reverse-mode derivative
of the forward that ``trimul_oracle`` defines, for a scalar loss L whose
gradient with respect to ``out`` is ``dout``:

    z'  = LN_in(z);  pa = z' W_a^T, ga = z' W_ga^T, pb = z' W_b^T, gb = z' W_gb^T
    a   = sigmoid(ga) pa m;   b = sigmoid(gb) pb m
    x   = triangle(a, b);  y = LN_out(x);  g = z' W_g^T;  v = y W_o^T
    out = sigmoid(g) v

taken backward step by step in the reverse order:

    dv = dout sigmoid(g),  dg = dout v sigmoid(g) (1 - sigmoid(g))
    dW_o = sum_p dv_p^T y_p,  dW_g = sum_p dg_p^T z'_p
    dy = dv W_o,  dz' (gate part) = dg W_g
    dx, d gamma_out, d beta_out = LayerNorm backward of dy
    da, db = triangle backward of dx
      outgoing (x[i,j] = sum_k a[i,k] b[j,k]):
          da[i,k] = sum_j dx[i,j] b[j,k],   db[j,k] = sum_i dx[i,j] a[i,k]
      incoming (x[i,j] = sum_k a[k,i] b[k,j]):
          da[k,i] = sum_j dx[i,j] b[k,j],   db[k,j] = sum_i dx[i,j] a[k,i]
    dpa = da sigmoid(ga) m,  dga = da pa m sigmoid(ga) (1 - sigmoid(ga));  the same for b
    dW_a = sum_p dpa_p^T z'_p  (and W_ga, W_b, W_gb alike)
    dz' += dpa W_a + dga W_ga + dpb W_b + dgb W_gb
    dz, d gamma_in, d beta_in = LayerNorm backward of dz'

(channel indices are implicit: each triangle product is per batch and channel).

Readings where the pages are silent: the pair mask is data (a padding mask),
so it gets no gradient; the weight gradients are the sums over all B N^2
pairs.  The LayerNorm backward is ``nn.LayerNorm``'s: with v^ = (v - mu) r,
dv = r (dv^ - mean(dv^) - v^ mean(dv^ v^)), dv^ = dy gamma.

Pins
----
``tests/test_oracle_backward_pins.py``: central finite differences of the
forward oracle for every gradient on small cases (both directions, soft
masks, two batch elements), the incoming/outgoing transpose identity applied
to the gradients, the LayerNorm invariant sum_d dz[p, d] = 0, linearity in
dout, and zero gradients for zero dout.
"""

from __future__ import annotations

import numpy as np

from .trimul_oracle import INCOMING, OUTGOING, _f64, sigmoid, triangle

GRAD_KEYS = ("W_a", "W_ga", "W_b", "W_gb", "W_o", "W_g",
             "ln_in_gamma", "ln_in_beta", "ln_out_gamma", "ln_out_beta")


def layer_norm_backward(v, gamma, eps, dy):
    """Gradients of y = LayerNorm(v) (affine gamma, beta) over the last axis.

    Returns (dv, d_gamma, d_beta) with d_gamma, d_beta summed over all
    leading axes.  ``nn.LayerNorm``'s normalisation: biased variance, eps
    under the square root.
    """
    v = _f64(v)
    dy = _f64(dy)
    mu = v.mean(axis=-1, keepdims=True)
    var = ((v - mu) ** 2).mean(axis=-1, keepdims=True)
    r = 1.0 / np.sqrt(var + eps)
    vh = (v - mu) * r
    dvh = dy * _f64(gamma)
    dv = r * (dvh - dvh.mean(axis=-1, keepdims=True) - vh * (dvh * vh).mean(axis=-1, keepdims=True))
    lead = tuple(range(v.ndim - 1))
    return dv, (dy * vh).sum(axis=lead), dy.sum(axis=lead)


def triangle_backward(a, b, dx, direction):
    """Gradients of the triangle contraction with respect to a and b.

    ``a``, ``b``, ``dx`` are [B, N, N, C]; index letters are (batch, token,
    token, channel).  outgoing: x[i,j] = sum_k a[i,k] b[j,k]; incoming:
    x[i,j] = sum_k a[k,i] b[k,j].
    """
    # per (batch, channel) matrices A[i, k] = a[b, i, k, c], and so on
    A = np.moveaxis(_f64(a), -1, 1)
    Bm = np.moveaxis(_f64(b), -1, 1)
    dX = np.moveaxis(_f64(dx), -1, 1)
    T = lambda M: np.swapaxes(M, -1, -2)  # noqa: E731
    if direction == OUTGOING:      # X = A B^T
        dA, dB = dX @ Bm, T(dX) @ A
    elif direction == INCOMING:    # X = A^T B
        dA, dB = Bm @ T(dX), A @ dX
    else:
        raise ValueError(f"direction must be 'outgoing' or 'incoming', got {direction!r}")
    return np.moveaxis(dA, 1, -1), np.moveaxis(dB, 1, -1)


def _pair_sum(u, w):
    """sum over all pairs of u_p^T w_p: u [..., F], w [..., G] -> [F, G]."""
    return u.reshape(-1, u.shape[-1]).T @ w.reshape(-1, w.shape[-1])


def trimul_backward(z, mask, params, direction, dout, eps=1e-5):
    """Gradients of sum(out * dout) for the TriMul forward of ``trimul_oracle``.

    ``z`` is [B, N, N, D], ``mask`` [B, N, N] or None (all ones), ``dout``
    [B, N, N, D].  Returns a dict with ``dz`` [B, N, N, D] and the gradient of
    every entry of GRAD_KEYS (same shape as the parameter).
    """
    z = _f64(z)
    dout = _f64(dout)
    m = np.ones(z.shape[:3]) if mask is None else _f64(mask)
    mm = m[..., None]
    P = {k: _f64(params[k]) for k in GRAD_KEYS}

    # forward, keeping what the backward needs
    mu = z.mean(axis=-1, keepdims=True)
    var = ((z - mu) ** 2).mean(axis=-1, keepdims=True)
    zn = (z - mu) / np.sqrt(var + eps) * P["ln_in_gamma"] + P["ln_in_beta"]
    pa, ga = zn @ P["W_a"].T, zn @ P["W_ga"].T
    pb, gb = zn @ P["W_b"].T, zn @ P["W_gb"].T
    sa, sb = sigmoid(ga), sigmoid(gb)
    a, b = sa * pa * mm, sb * pb * mm
    x = triangle(a, b, direction)
    xmu = x.mean(axis=-1, keepdims=True)
    xvar = ((x - xmu) ** 2).mean(axis=-1, keepdims=True)
    y = (x - xmu) / np.sqrt(xvar + eps) * P["ln_out_gamma"] + P["ln_out_beta"]
    sg = sigmoid(zn @ P["W_g"].T)
    v = y @ P["W_o"].T

    # output gate and output projection
    dv = dout * sg
    dg = dout * v * sg * (1.0 - sg)
    grads = {"W_o": _pair_sum(dv, y), "W_g": _pair_sum(dg, zn)}
    dy = dv @ P["W_o"]
    dzn = dg @ P["W_g"]

    # LN_out
    dx, grads["ln_out_gamma"], grads["ln_out_beta"] = layer_norm_backward(x, P["ln_out_gamma"], eps, dy)

    # triangle
    da, db = triangle_backward(a, b, dx, direction)

    # gated input projections
    dpa, dga = da * sa * mm, da * pa * mm * sa * (1.0 - sa)
    dpb, dgb = db * sb * mm, db * pb * mm * sb * (1.0 - sb)
    grads["W_a"], grads["W_ga"] = _pair_sum(dpa, zn), _pair_sum(dga, zn)
    grads["W_b"], grads["W_gb"] = _pair_sum(dpb, zn), _pair_sum(dgb, zn)
    dzn = dzn + dpa @ P["W_a"] + dga @ P["W_ga"] + dpb @ P["W_b"] + dgb @ P["W_gb"]

    # LN_in
    dz, grads["ln_in_gamma"], grads["ln_in_beta"] = layer_norm_backward(z, P["ln_in_gamma"], eps, dzn)
    grads["dz"] = dz
    return grads


def backward_flops(B, N, D, C):
    """Algorithmic GEMM FLOPs of one backward that recomputes the forward.

    Forward recompute: the four input projections, the triangle, the two
    output projections.  Backward: dy = dv W_o and the gate path dg W_g,
    the two triangle gradients, dz' from the four input projections, and the
    six weight gradients (each a sum over B N^2 pairs of outer products).
    """
    P = B * N * N
    fwd = P * 2 * D * 4 * C + B * 2 * C * N ** 3 + P * 2 * (D * D + C * D)
    bwd = (P * 2 * (D * C + D * D)          # dy, dz' (gate)
           + B * 2 * 2 * C * N ** 3          # da, db
           + P * 2 * 4 * C * D               # dz' (input projections)
           + P * 2 * (D * C + D * D)         # dW_o, dW_g
           + P * 2 * 4 * C * D)              # dW_a, dW_ga, dW_b, dW_gb
    return fwd + bwd
