"""Per-kernel parity through the C ABI: each stage against the fp64 oracle.

Each stage is fed exact inputs (the same values the oracle sees) so its own
error is measured alone:
  stage 1 (LN_in + gated in-projection): a, b vs oracle.gated_projection;
  stage 2 (triangle GEMM): x vs the fp64 contraction of the same fp16 a, b;
  stage 3 (LN_out + out-projection + gate): out vs oracle.output_projection of
  the same x, given in stage 2's format (fp16 x * 2^-s, s from the handle's
  static bound).
"""

import numpy as np
import pytest
import torch

from co_folding_pair_gb300 import synthetic as S
from oracle import trimul_oracle as O
from tests._util import assert_close

pytestmark = pytest.mark.gpu

SIZES = [  # (B, N, D, C): several tiles, ragged tails, small widths
    (1, 64, 32, 32),
    (2, 136, 128, 128),
    (1, 200, 256, 256),
    (1, 256, 256, 128),
    (2, 24, 64, 96),
]


@pytest.fixture(scope="module")
def T():
    from co_folding_pair_gb300 import trimul
    return trimul


def _np(t):
    return t.detach().double().cpu().numpy()


def _params_np(params):
    return {k: v.double().numpy() for k, v in params.items()}


@pytest.mark.parametrize("B,N,D,C", SIZES)
def test_stage1_inproj(T, B, N, D, C):
    w = S.custom(B, N, D, C, seed=100 + N, mask_kind="random_frac", mask_frac=0.25)
    z, mask, params = S.make_case(w, device="cuda")
    h = T.trimul_create(params)
    try:
        a, b = T.trimul_inproj(h, z, mask, flags=T.FLAG_CHECK)
        torch.cuda.synchronize()
        pn = _params_np(params)
        zn = O.layer_norm(_np(z), pn["ln_in_gamma"], pn["ln_in_beta"], 1e-5)
        m = _np(mask)
        ref_a = np.moveaxis(O.gated_projection(zn, pn["W_a"], pn["W_ga"], m), -1, 1)  # [B, C, N, N]
        ref_b = np.moveaxis(O.gated_projection(zn, pn["W_b"], pn["W_gb"], m), -1, 1)
        assert_close(_np(a), ref_a, "a")
        assert_close(_np(b), ref_b, "b")
        # masked pairs are exactly zero
        mz = (m == 0)[:, None, :, :].repeat(C, axis=1)
        assert np.all(_np(a)[mz] == 0) and np.all(_np(b)[mz] == 0)
    finally:
        T.trimul_destroy(h)


@pytest.mark.parametrize("direction", ["outgoing", "incoming"])
@pytest.mark.parametrize("B,N,C", [(1, 64, 8), (1, 200, 8), (2, 136, 8), (1, 384, 16), (1, 8, 8)])
def test_stage2_triangle(T, direction, B, N, C):
    g = torch.Generator().manual_seed(7 * N + C)
    a = torch.randn(B, C, N, N, generator=g).to(torch.float16)
    b = torch.randn(B, C, N, N, generator=g).to(torch.float16)
    params = S.make_params(S.custom(B, N, 32, C, seed=1), torch.Generator().manual_seed(1))
    h = T.trimul_create(params)
    try:
        x = T.trimul_triangle(h, a.cuda(), b.cuda(), direction, flags=T.FLAG_CHECK)
        torch.cuda.synchronize()
        A, Bm = a.double().numpy(), b.double().numpy()
        ref = A @ np.swapaxes(Bm, -1, -2) if direction == "outgoing" else np.swapaxes(A, -1, -2) @ Bm
        # x is stored as fp16 x * 2^-s (an exact power-of-two scale)
        got = _np(x) * 2.0 ** T.trimul_x_scale_log2(h, N)
        # fp32 accumulation, one fp16 rounding of the (scaled) result
        scale = np.sqrt(N)
        err = np.abs(got - ref)
        assert np.all(err <= 2 ** -8 * np.abs(ref) + 1e-3 * scale), f"max err {err.max()}"
        assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < 3e-3
    finally:
        T.trimul_destroy(h)


@pytest.mark.parametrize("B,N,D,C", SIZES)
def test_stage3_outproj(T, B, N, D, C):
    w = S.custom(B, N, D, C, seed=300 + N)
    z, _, params = S.make_case(w, device="cuda")
    g = torch.Generator().manual_seed(N)
    # x with a per-pair offset and scale, so LayerNorm over C has work to do
    x = torch.randn(B, C, N, N, generator=g) * 3 + torch.randn(B, 1, N, N, generator=g) * 2
    x[:, :, 0, :] = 0  # LN of a zero vector gives beta_out
    h = T.trimul_create(params)
    try:
        # stage 3 takes x in stage 2's format: fp16 x * 2^-s
        sc = 2.0 ** T.trimul_x_scale_log2(h, N)
        xs = (x / sc).to(torch.float16)
        out = T.trimul_outproj(h, xs.cuda(), z, flags=T.FLAG_CHECK)
        torch.cuda.synchronize()
        pn = _params_np(params)
        zn = O.layer_norm(_np(z), pn["ln_in_gamma"], pn["ln_in_beta"], 1e-5)
        ref = O.output_projection(np.moveaxis(xs.double().numpy() * sc, 1, -1), zn, pn, 1e-5)
        assert_close(_np(out), ref, "out")
    finally:
        T.trimul_destroy(h)
