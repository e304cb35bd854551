"""Stress parity of trimul_forward against the fp64 oracle: inputs that strain
the binary16 operand path.

a, b and x are binary16 on the GPU, and x is stored as x * 2^-s with a power of
two s chosen per call from the call's own max |a|, |b|.  These cases would
break a weaker choice of s, or a LayerNorm whose statistics cancel:

  - a "loose" layer (a few gamma_in features at 4, a few W_a / W_b rows at 4x
    the norm of the rest), whose worst-case bound on |a|, |b| is far above the
    values that occur, combined with
      * tokens that keep only 1-3 unmasked partners (x of those rows is a sum
        of a few products), and
      * soft masks with pair weights down to 1e-4 (x of those pairs is tiny);
    with s taken from the bound, such x fall into the binary16 subnormals and
    LayerNorm over C magnifies their rounding;
  - z with a large common offset (50 + N(0, 1)), which cancels in one-pass
    LayerNorm statistics and in the folded output projection;
  - a per-token LogNormal(0, 0.5) scale at N = 1024 in both directions.

Tolerance as everywhere: |gpu - ref| <= 1e-2 + 1e-2 |ref| per element and
relative Frobenius <= 5e-3 over the evaluated set.  Also here: mask values
outside [0, 1] are reported with TRIMUL_FLAG_CHECK.
"""

import numpy as np
import pytest
import torch

from co_folding_pair_gb300 import synthetic as S
from oracle import trimul_oracle as O
from tests._util import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def T():
    from co_folding_pair_gb300 import trimul
    return trimul


def _np(t):
    return t.detach().double().cpu().numpy()


def _params_np(params):
    return {k: v.double().numpy() for k, v in params.items()}


def _full(T, w, direction):
    z, mask, params = S.make_case(w, device="cuda")
    h = T.trimul_create(params)
    try:
        out = T.trimul_forward(h, z, mask, direction, flags=T.FLAG_CHECK)
        torch.cuda.synchronize()
    finally:
        T.trimul_destroy(h)
    ref = O.trimul_forward(_np(z), _np(mask), _params_np(params), direction)
    return _np(out), ref


@pytest.mark.parametrize("direction", ["outgoing", "incoming"])
@pytest.mark.parametrize("mask_kind", ["few_partners", "soft"])
def test_loose_layer(T, direction, mask_kind):
    w = S.custom(1, 256, 256, 128, seed=51, mask_kind=mask_kind, layer_kind="loose")
    got, ref = _full(T, w, direction)
    assert_close(got, ref, f"loose layer, {mask_kind}, {direction}")


@pytest.mark.parametrize("direction", ["outgoing", "incoming"])
def test_loose_layer_soft_mask_two_batches(T, direction):
    w = S.custom(2, 136, 192, 64, seed=52, mask_kind="soft", layer_kind="loose")
    got, ref = _full(T, w, direction)
    assert_close(got, ref, f"loose layer, soft mask, B=2, {direction}")


@pytest.mark.parametrize("direction", ["outgoing", "incoming"])
def test_large_common_offset(T, direction):
    w = S.custom(1, 128, 256, 128, seed=53, z_kind="offset", z_offset=50.0,
                 mask_kind="random_frac", mask_frac=0.2)
    got, ref = _full(T, w, direction)
    assert_close(got, ref, f"z = 50 + N(0,1), {direction}")


@pytest.mark.parametrize("direction", ["outgoing", "incoming"])
def test_token_scale_n1024_sampled(T, direction):
    """Per-token LogNormal(0, 0.5) scale with a random 20% token mask at
    N = 1024, D = 256, C = 128; the oracle evaluates a seeded 48 x 48 grid."""
    w = S.custom(1, 1024, 256, 128, seed=54, z_kind="token_scale", mask_kind="random_frac",
                 mask_frac=0.2)
    z, mask, params = S.make_case(w, device="cuda")
    h = T.trimul_create(params)
    try:
        out = T.trimul_forward(h, z, mask, direction, flags=T.FLAG_CHECK)
        torch.cuda.synchronize()
    finally:
        T.trimul_destroy(h)
    rows, cols = S.sample_grid(w, 48, 48)
    got = out[0][np.ix_(rows[0], cols[0])].double().cpu().numpy()
    ref = O.trimul_forward_sampled(S.Bf16HostView.of(z.cpu()), mask.float().cpu().numpy(),
                                   _params_np(params), direction, rows, cols)[0]
    assert_close(got, ref, f"token scale N=1024 {direction}")


# ---------------------------------------------------------------- mask values outside [0, 1]

@pytest.mark.parametrize("bad", [1.5, -0.25, float("nan")])
def test_mask_outside_unit_interval_is_reported(T, bad):
    w = S.custom(1, 64, 32, 32, seed=55)
    z, mask, params = S.make_case(w, device="cuda")
    mask[0, 5, 7] = bad
    h = T.trimul_create(params)
    try:
        for call in ("forward", "inproj", "host"):
            with pytest.raises(T.TrimulError) as ei:
                if call == "forward":
                    T.trimul_forward(h, z, mask, "outgoing", flags=T.FLAG_CHECK)
                elif call == "inproj":
                    T.trimul_inproj(h, z, mask, flags=T.FLAG_CHECK)
                else:
                    T.trimul_forward_host(h, z.cpu().pin_memory(), mask.cpu().pin_memory(), "outgoing",
                                          flags=T.FLAG_CHECK)
            assert ei.value.status == 1 and "mask" in str(ei.value), call
        # the flag does not outlive the call: a valid mask passes again
        mask[0, 5, 7] = 1.0
        T.trimul_forward(h, z, mask, "outgoing", flags=T.FLAG_CHECK)
        torch.cuda.synchronize()
    finally:
        T.trimul_destroy(h)


def test_mask_bounds_are_inclusive(T):
    """0 and 1 themselves, and soft values between, are valid."""
    w = S.custom(1, 64, 32, 32, seed=56, mask_kind="soft")
    z, mask, params = S.make_case(w, device="cuda")
    mask[0, 0, :] = 0.0
    mask[0, 1, :] = 1.0
    h = T.trimul_create(params)
    try:
        out = T.trimul_forward(h, z, mask, "incoming", flags=T.FLAG_CHECK)
        torch.cuda.synchronize()
    finally:
        T.trimul_destroy(h)
    ref = O.trimul_forward(_np(z), _np(mask), _params_np(params), "incoming")
    assert_close(_np(out), ref, "soft mask with 0 and 1 rows")
