"""The backward at full size, checked against the forward: directional derivatives.

The fp64 backward oracle needs every pair's a and b, which is out of reach
at N = 4096.  What holds at any size is the definition of the gradient: for
a direction dz_dir,

    < dout, out(z + e dz_dir) - out(z - e dz_dir) >  =  < dz, (z + e dz_dir) - (z - e dz_dir) > + O(e^3)

with dz = trimul_backward(z, dout), and the same for the parameters (both
sides summed over all ten parameter tensors).  Both forwards are the
library's own; every perturbed input is rounded to its storage type first
and the right-hand side uses the rounded difference, so the only gaps are
the O(e^2) relative curvature term and the two paths' roundings.

dout is the centred difference at a second step e1, (out(+e1) - out(-e1)) / e1,
so the signal is coherent (dout points where the output moves) while the
forward's rounding noise at the checked step e2 is independent of dout and
averages out over the 4.3e9 outputs.

Both sides are taken at two steps, e2 and e2 / 2.  For a correct backward
the signed relative gap d(e) = (rhs - lhs) / lhs is c e^2 + r: a curvature
term that falls fourfold when e halves, plus a floor r from the two paths'
roundings.  Richardson extrapolation, r = (4 d(e2 / 2) - d(e2)) / 3, removes
the curvature term.  A wrong gradient instead leaves a gap that does not
shrink with e.

Bounds:
- r: the fp64 oracle with the same scheme and bf16 roundings gives |r| of
  at most 8.3e-4 on four small shapes (few terms there to average the
  roundings of z, dout and out); the GPU paths add roundings that are
  random from one weight or pair to the next.  |r| <= 3e-3, about thirty
  times below the share of one of the nine triangle launch groups at
  N = 4096;
- d(e2) at e2 = 0.01: the oracle's curvature at small shapes was at most
  1.4e-3 (z on the per-token-scaled workload); |d| <= 1e-2 leaves room for
  the larger curvature of the full sizes.

What it catches: a gradient missing or wrong for one launch group, batch
slice or tile range removes that part's coherent share of the sum (each of
the nine triangle launches at N = 4096 carries about a ninth of it); with
one ninth of da's channels zeroed in the oracle's backward, the gaps were
5.8e-2 (z) and 2.7e-2 (parameters) at every step.

Also at full size: sum_d dz[p, d] = 0 on sampled pairs (the LayerNorm
invariant), and finite gradients.
"""

import pytest
import torch

from co_folding_pair_gb300 import synthetic as S

pytestmark = pytest.mark.gpu

E1, E2 = 0.05, 0.01
TOL_D, TOL_R = 1e-2, 3e-3
ROWS = 256  # rows i per elementwise block


@pytest.fixture(scope="module")
def T():
    from co_folding_pair_gb300 import trimul
    return trimul


def _dir_block(shape, seed, i0, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed * 100003 + i0)
    return torch.randn(shape, generator=g, device=device)


def perturbed(z, e, seed):
    """bf16(z + e * d), d ~ N(0, 1) drawn block by block from seeded generators."""
    out = torch.empty_like(z)
    for b in range(z.shape[0]):
        for i0 in range(0, z.shape[1], ROWS):
            blk = z[b, i0:i0 + ROWS]
            d = _dir_block(blk.shape, seed + b, i0, z.device)
            out[b, i0:i0 + ROWS] = (blk.float() + e * d).to(torch.bfloat16)
    return out


def blockwise(fn, *ts):
    """sum over row blocks of fn(blocks...) in float64."""
    acc = torch.zeros((), dtype=torch.float64, device=ts[0].device)
    for b in range(ts[0].shape[0]):
        for i0 in range(0, ts[0].shape[1], ROWS):
            acc += fn(*(t[b, i0:i0 + ROWS] for t in ts))
    return float(acc)


def centred_dout(outp, outm, e):
    d = torch.empty_like(outp)
    for b in range(outp.shape[0]):
        for i0 in range(0, outp.shape[1], ROWS):
            d[b, i0:i0 + ROWS] = ((outp[b, i0:i0 + ROWS].float() - outm[b, i0:i0 + ROWS].float()) / e).to(torch.bfloat16)
    return d


def dot(u, v):
    return (u.double() * v.double()).sum()


def perturbed_params(params, e, seed):
    """The weights (bf16) and LayerNorm affines (float32) moved by e times a seeded
    direction; weight directions are scaled by each matrix's rms."""
    g = torch.Generator()
    g.manual_seed(seed)
    out = {}
    for k in sorted(params):
        v = params[k]
        d = torch.randn(v.shape, generator=g)
        if k.startswith("W"):
            d = d * v.float().pow(2).mean().sqrt()
        out[k] = (v.float() + e * d).to(v.dtype)
    return out


def forward(T, params, z, mask, direction):
    h = T.trimul_create(params)
    try:
        out = T.trimul_forward(h, z, mask, direction, flags=T.FLAG_CHECK)
    finally:
        T.trimul_destroy(h)
    return out


@pytest.mark.parametrize("name,direction", [("n4096_d256_c256", "outgoing"),
                                            ("n3072_d256_c128_scaled", "incoming")])
def test_backward_directional_derivatives_full_size(T, name, direction):
    gaps = directional_gaps(T, S.WORKLOADS[name], direction)
    for what, (d1, d2) in gaps.items():
        r = (4 * d2 - d1) / 3
        assert abs(d1) <= TOL_D and abs(r) <= TOL_R, (what, d1, d2, r)


def directional_gaps(T, w, direction, device="cuda"):
    """Signed relative gaps (rhs - lhs) / lhs of the two directional-derivative
    identities (z, parameters) at the steps E2 and E2 / 2."""
    z, mask, params = S.make_case(w, device=device)
    seed = w.seed + 500
    steps = (E2, E2 / 2)
    gaps = {}

    # z: dout from the step E1, the checks at the steps E2 and E2 / 2
    def fz(e):
        return forward(T, params, perturbed(z, e, seed), mask, direction)

    op, om = fz(E1), fz(-E1)
    dout = centred_dout(op, om, E1)
    del op, om
    lhs = []
    for e in steps:
        op, om = fz(e), fz(-e)
        lhs.append(blockwise(lambda d, a, b: dot(d, a.float() - b.float()), dout, op, om))
        del op, om
    h = T.trimul_create(params)
    try:
        dz, _ = T.trimul_backward(h, z, mask, dout, direction, flags=T.FLAG_CHECK)
    finally:
        T.trimul_destroy(h)
    assert bool(torch.isfinite(dz.float()[0, ::64]).all())
    rhs = []
    for e in steps:
        zp, zm = perturbed(z, e, seed), perturbed(z, -e, seed)
        rhs.append(blockwise(lambda g, a, b: dot(g, a.float() - b.float()), dz, zp, zm))
        del zp, zm
    gaps["z"] = tuple((r - l) / l for l, r in zip(lhs, rhs))
    # the LayerNorm invariant on sampled pairs: each dz row sums to ~0 over D
    rows = dz[:, ::37, ::41].float()
    assert bool((rows.sum(-1).abs() <= 2e-2 * rows.abs().sum(-1) + 1e-30).all())
    del dz, dout

    # parameters, all ten tensors at once
    def fp(e):
        return forward(T, perturbed_params(params, e, seed), z, mask, direction)

    op, om = fp(E1), fp(-E1)
    dout = centred_dout(op, om, E1)
    del op, om
    lhs = []
    for e in steps:
        op, om = fp(e), fp(-e)
        lhs.append(blockwise(lambda d, a, b: dot(d, a.float() - b.float()), dout, op, om))
        del op, om
    h = T.trimul_create(params)
    try:
        _, grads = T.trimul_backward(h, z, mask, dout, direction, flags=T.FLAG_CHECK)
    finally:
        T.trimul_destroy(h)
    rhs = []
    for e in steps:
        pp, pm = perturbed_params(params, e, seed), perturbed_params(params, -e, seed)
        acc = 0.0
        for k, g in grads.items():
            assert bool(torch.isfinite(g).all()), k
            acc += float(dot(g.cpu(), pp[k].float() - pm[k].float()))
        rhs.append(acc)
    gaps["parameters"] = tuple((r - l) / l for l, r in zip(lhs, rhs))
    print(f"\n{w.name} {direction}: " + "; ".join(
        f"{k} gaps {d1:+.2e} (e2), {d2:+.2e} (e2/2), extrapolated {(4 * d2 - d1) / 3:+.2e}" for k, (d1, d2) in gaps.items()))
    return gaps
