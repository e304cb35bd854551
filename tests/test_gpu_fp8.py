"""The opt-in 8-bit triangle path (TRIMUL_FLAG_FP8) against the fp64 oracle.

With the flag, a and b are rounded to e4m3 after a power-of-two scale s8 (the
largest one that keeps the layer's bound on |a|, |b| within 448), and the
triangle contraction runs on the 8-bit tensor cores.  e4m3 keeps 3 mantissa
bits, so a and b carry a relative rounding error of up to 2^-4 each; over the
contraction the errors are independent and partly cancel, and LN_out divides
by the row's own spread.  An fp64 emulation of exactly this rounding
(e4m3 of a * s8 and b * s8, the fp16 x and the rest of the layer as in the
default path) over five layers and masks gave a relative Frobenius error of at
most 3.9e-2 and a worst element of at most 0.42 (rms(ref) + |ref| / 4).  The
bounds below take twice that:

    ||gpu - ref||_F / ||ref||_F <= 8e-2,
    |gpu - ref| <= 0.8 rms(ref) + 0.2 |ref|   per element.

The flag is outgoing-only, needs N % 16 == 0 (a plane row of N bytes must be a
multiple of 16 bytes for the tensor maps), and every other entry point rejects
it.
"""

import ctypes

import numpy as np
import pytest
import torch

from co_folding_pair_gb300 import synthetic as S
from oracle import trimul_oracle as O
from tests._util import RECORD

pytestmark = pytest.mark.gpu

FRO8 = 8e-2
ELEM_RMS8 = 0.8
ELEM_REL8 = 0.2


@pytest.fixture(scope="module")
def T():
    from co_folding_pair_gb300 import trimul
    return trimul


def _np(t):
    return t.detach().double().cpu().numpy()


def _params_np(params):
    return {k: v.double().numpy() for k, v in params.items()}


def assert_close_fp8(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    rms = float(np.sqrt((ref ** 2).mean()))
    worst = float((err / (ELEM_RMS8 * rms + ELEM_REL8 * np.abs(ref))).max())
    fro = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    RECORD.append((what + " [e4m3 bound]", worst, fro))
    assert worst <= 1.0 and fro <= FRO8, (
        f"{what}: worst element at {worst:.3f} of the e4m3 bound, rel Frobenius {fro:.3e} (bound {FRO8:.0e})")
    return worst, fro


def _full_fp8(T, w):
    z, mask, params = S.make_case(w, device="cuda")
    h = T.trimul_create(params)
    try:
        out = T.trimul_forward(h, z, mask, "outgoing", flags=T.FLAG_CHECK | T.FLAG_FP8)
        torch.cuda.synchronize()
    finally:
        T.trimul_destroy(h)
    ref = O.trimul_forward(_np(z), _np(mask), _params_np(params), "outgoing")
    return _np(out), ref


def test_fp8_n64_d32(T):
    got, ref = _full_fp8(T, S.WORKLOADS["n64_d32_c32"])
    assert_close_fp8(got, ref, "e4m3 n64")


def test_fp8_n256_tailmask(T):
    got, ref = _full_fp8(T, S.WORKLOADS["n256_d128_c128_tailmask"])
    assert_close_fp8(got, ref, "e4m3 n256 tail mask")


@pytest.mark.parametrize("B,N,D,C,mask_kind", [
    # K tail: 144 = 128 + 16 (a second, mostly out-of-range K block)
    (2, 144, 64, 32, "padding"),
    (1, 208, 256, 256, "random_frac"),
    (3, 32, 32, 64, "ones"),
    (1, 16, 8, 8, "ones"),
    # three 128-channel weight groups (the a/b straddle inside one staged box)
    (1, 64, 192, 192, "random_frac"),
    (1, 272, 128, 128, "random_frac"),
])
def test_fp8_ragged(T, B, N, D, C, mask_kind):
    w = S.custom(B, N, D, C, seed=N + D + 7, mask_kind=mask_kind, mask_frac=0.2)
    got, ref = _full_fp8(T, w)
    assert_close_fp8(got, ref, f"e4m3 B{B} N{N} D{D} C{C}")


def test_fp8_loose_layer(T):
    """A layer whose weight-derived bound on |a|, |b| is loose (a few large
    gamma_in features and W_a / W_b rows): the static power-of-two scale then
    keeps a and b at most near 45 of e4m3's 448, nearer its subnormals.  The
    fp64 emulation of this case: relative Frobenius 3.6e-2, worst element 0.63
    of the bound."""
    w = S.custom(1, 256, 256, 128, seed=61, mask_kind="few_partners", layer_kind="loose")
    got, ref = _full_fp8(T, w)
    assert_close_fp8(got, ref, "e4m3 loose layer, few partners")


def test_fp8_structured(T):
    w = S.custom(2, 128, 128, 128, seed=2, z_kind="outer", mask_kind="padding", mask_frac=0.15)
    got, ref = _full_fp8(T, w)
    assert_close_fp8(got, ref, "e4m3 outer-product structure")


def test_fp8_n4096_sampled(T):
    """The full 4096-token, 256-channel workload; the oracle evaluates a 64 x 64
    grid of pairs exactly."""
    w = S.WORKLOADS["n4096_d256_c256"]
    z, mask, params = S.make_case(w, device="cuda")
    h = T.trimul_create(params)
    try:
        out = T.trimul_forward(h, z, mask, "outgoing", flags=T.FLAG_CHECK | T.FLAG_FP8)
        torch.cuda.synchronize()
    finally:
        T.trimul_destroy(h)
    rows, cols = S.sample_grid(w, 64, 64)
    got = out[0][np.ix_(rows[0], cols[0])].double().cpu().numpy()
    del out
    zh = S.Bf16HostView.of(z.cpu())
    del z
    ref = O.trimul_forward_sampled(zh, mask.float().cpu().numpy(), _params_np(params), "outgoing", rows, cols)
    assert_close_fp8(got.ravel(), ref[0].ravel(), "e4m3 n4096")


def test_fp8_deterministic_and_distinct(T):
    """Repeated calls give the same bits; the 8-bit result is not the 16-bit one
    (the flag really switches the path) but stays within the e4m3 bound of it."""
    w = S.custom(1, 160, 128, 64, seed=22, mask_kind="random_frac", mask_frac=0.3)
    z, mask, params = S.make_case(w, device="cuda")
    h = T.trimul_create(params)
    try:
        o1 = T.trimul_forward(h, z, mask, "outgoing", flags=T.FLAG_FP8).clone()
        o2 = T.trimul_forward(h, z, mask, "outgoing", flags=T.FLAG_FP8).clone()
        o16 = T.trimul_forward(h, z, mask, "outgoing")
        torch.cuda.synchronize()
        assert torch.equal(o1, o2)
        assert not torch.equal(o1, o16)
        assert_close_fp8(_np(o1), _np(o16), "e4m3 vs fp16 path")
    finally:
        T.trimul_destroy(h)


def test_fp8_masked_positions_do_not_matter_bitwise(T):
    w = S.custom(1, 128, 64, 64, seed=23, mask_kind="random_frac", mask_frac=0.3)
    z, mask, params = S.make_case(w, device="cuda")
    z2 = z.clone()
    sel = mask == 0
    z2[sel] = (torch.randn_like(z2[sel].float()) * 50).to(torch.bfloat16)
    h = T.trimul_create(params)
    try:
        o1 = T.trimul_forward(h, z, mask, "outgoing", flags=T.FLAG_FP8).clone()
        o2 = T.trimul_forward(h, z2, mask, "outgoing", flags=T.FLAG_FP8)
        torch.cuda.synchronize()
        keep = mask == 1
        assert torch.equal(o1[keep], o2[keep])
    finally:
        T.trimul_destroy(h)


def test_fp8_flag_rejections(T):
    """Incoming, N % 16 != 0 and every entry point but trimul_forward refuse the
    flag before launching anything."""
    w = S.custom(1, 64, 32, 32, seed=27)
    z, mask, params = S.make_case(w, device="cuda")
    h = T.trimul_create(params)
    try:
        lib = T._lib.load()
        s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        F = T.FLAG_FP8
        o = torch.empty_like(z)
        zp, op, mp = ctypes.c_void_p(z.data_ptr()), ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(mask.data_ptr())
        assert lib.trimul_forward(h.ptr, zp, mp, 1, 64, 1, op, s, F) == 1     # incoming
        assert "outgoing" in T.trimul_last_error()
        z8 = torch.zeros(1, 72, 72, 32, dtype=torch.bfloat16, device="cuda")
        o8 = torch.empty_like(z8)
        assert lib.trimul_forward(h.ptr, ctypes.c_void_p(z8.data_ptr()), None, 1, 72, 0,
                                  ctypes.c_void_p(o8.data_ptr()), s, F) == 2  # N % 16
        ab = torch.empty(1, 32, 64, 64, dtype=torch.float16, device="cuda")
        abp = ctypes.c_void_p(ab.data_ptr())
        assert lib.trimul_inproj(h.ptr, zp, mp, 1, 64, abp, abp, s, F) == 1
        assert lib.trimul_triangle(h.ptr, abp, abp, 1, 64, 0, abp, s, F) == 1
        assert lib.trimul_outproj(h.ptr, abp, zp, 1, 64, op, s, F) == 1
        assert lib.trimul_forward_noalloc(h.ptr, zp, mp, 1, 64, 0, op, s, F) == 1
        assert lib.trimul_forward_host(h.ptr, zp, mp, 1, 64, 0, op, s, F) == 1  # rejected before any copy
        assert "trimul_forward only" in T.trimul_last_error()
        # the handle is still usable
        out = T.trimul_forward(h, z, mask, "outgoing", flags=T.FLAG_CHECK | F)
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
    finally:
        T.trimul_destroy(h)
