"""Guard bands around every caller buffer: no entry point writes outside its outputs.

A parity test reads only the elements it compares, so it cannot see a store
that lands past the end of an output or in bytes between its rows.  Here
every buffer the library is given (inputs and outputs) sits inside a larger
allocation with 4 KB guard bands on both sides, filled with a fixed byte
pattern; after each call the bands must be bitwise intact, and the inputs
bitwise unchanged.  Shapes are the ragged ones of the parity tests (token
counts that are not multiples of the 128- and 256-wide tiles, feature widths
that are not multiples of 64, several batch elements), through the three
stage entry points, the three forward entry points and the backward.
"""

import numpy as np
import pytest
import torch

from co_folding_pair_gb300 import synthetic as S

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


@pytest.fixture(scope="module")
def T():
    from co_folding_pair_gb300 import trimul
    return trimul


class Guarded:
    """A tensor of `shape` and `dtype` at byte offset GUARD of a buffer with
    GUARD pattern bytes on both sides."""

    def __init__(self, shape, dtype, device="cuda", fill=None):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((GUARD + n + GUARD,), PATTERN, dtype=torch.uint8, device=device)
        self.n = n
        self.t = self.raw[GUARD:GUARD + n].view(dtype).view(shape)
        if fill is not None:
            self.t.copy_(fill)

    def bands_intact(self):
        torch.cuda.synchronize()
        lo = self.raw[:GUARD]
        hi = self.raw[GUARD + self.n:]
        return bool((lo == PATTERN).all()) and bool((hi == PATTERN).all())


CASES = [  # (B, N, D, C)
    (3, 8, 136, 64),
    (3, 24, 136, 192),
    (1, 136, 136, 64),
    (2, 200, 136, 192),
]


@pytest.mark.parametrize("B,N,D,C", CASES)
def test_stage_calls_write_only_their_outputs(T, B, N, D, C):
    w = S.custom(B, N, D, C, seed=60 + N, mask_kind="random_frac", mask_frac=0.25)
    z0, m0, params = S.make_case(w, device="cuda")
    h = T.trimul_create(params)
    try:
        z = Guarded(z0.shape, torch.bfloat16, fill=z0)
        m = Guarded(m0.shape, torch.bfloat16, fill=m0)
        a = Guarded((B, C, N, N), torch.float16)
        b = Guarded((B, C, N, N), torch.float16)
        T.trimul_inproj(h, z.t, m.t, a_out=a.t, b_out=b.t, flags=T.FLAG_CHECK)
        for g, what in ((z, "z"), (m, "mask"), (a, "a"), (b, "b")):
            assert g.bands_intact(), f"stage 1 wrote outside {what}"
        assert torch.equal(z.t, z0) and torch.equal(m.t, m0), "stage 1 changed an input"
        a0, b0 = a.t.clone(), b.t.clone()
        for direction in ("outgoing", "incoming"):
            x = Guarded((B, C, N, N), torch.float16)
            T.trimul_triangle(h, a.t, b.t, direction, x_out=x.t, flags=T.FLAG_CHECK)
            for g, what in ((a, "a"), (b, "b"), (x, "x")):
                assert g.bands_intact(), f"stage 2 ({direction}) wrote outside {what}"
            assert torch.equal(a.t, a0) and torch.equal(b.t, b0), "stage 2 changed an input"
            x0 = x.t.clone()
            out = Guarded(z0.shape, torch.bfloat16)
            T.trimul_outproj(h, x.t, z.t, out=out.t, flags=T.FLAG_CHECK)
            for g, what in ((x, "x"), (z, "z"), (out, "out")):
                assert g.bands_intact(), f"stage 3 wrote outside {what}"
            assert torch.equal(x.t, x0) and torch.equal(z.t, z0), "stage 3 changed an input"
    finally:
        T.trimul_destroy(h)


@pytest.mark.parametrize("B,N,D,C", CASES)
def test_forward_calls_write_only_out(T, B, N, D, C):
    w = S.custom(B, N, D, C, seed=70 + N, mask_kind="padding", mask_frac=0.15)
    z0, m0, params = S.make_case(w, device="cuda")
    h = T.trimul_create(params)
    try:
        z = Guarded(z0.shape, torch.bfloat16, fill=z0)
        m = Guarded(m0.shape, torch.bfloat16, fill=m0)
        for direction in ("outgoing", "incoming"):
            out = Guarded(z0.shape, torch.bfloat16)
            T.trimul_forward(h, z.t, m.t, direction, out=out.t, flags=T.FLAG_CHECK)
            assert out.bands_intact() and z.bands_intact() and m.bands_intact(), f"forward {direction}"
            ref = out.t.clone()
            if (6 * C + 8) * B * N * N <= T.trimul_noalloc_scratch_bytes():
                out2 = Guarded(z0.shape, torch.bfloat16)
                T.trimul_forward_noalloc(h, z.t, m.t, direction, out2.t, flags=T.FLAG_CHECK)
                assert out2.bands_intact() and z.bands_intact(), f"noalloc {direction}"
                assert torch.equal(out2.t, ref), "noalloc differs from forward"
            zh = Guarded(z0.shape, torch.bfloat16, device="cpu", fill=z0.cpu())
            mh = Guarded(m0.shape, torch.bfloat16, device="cpu", fill=m0.cpu())
            oh = Guarded(z0.shape, torch.bfloat16, device="cpu")
            T.trimul_forward_host(h, zh.t, mh.t, direction, out_host=oh.t, flags=T.FLAG_CHECK)
            torch.cuda.synchronize()
            for g, what in ((zh, "z_host"), (mh, "mask_host"), (oh, "out_host")):
                lo, hi = g.raw[:GUARD], g.raw[GUARD + g.n:]
                assert bool((lo == PATTERN).all()) and bool((hi == PATTERN).all()), f"host call wrote outside {what}"
            assert torch.equal(oh.t, ref.cpu()), "host-buffer call differs from forward"
        assert torch.equal(z.t, z0) and torch.equal(m.t, m0), "forward changed an input"
    finally:
        T.trimul_destroy(h)


BACKWARD_CASES = [  # (B, N, D, C)
    (3, 8, 136, 64),
    (2, 136, 136, 192),
    (1, 200, 136, 64),
]


@pytest.mark.parametrize("B,N,D,C", BACKWARD_CASES)
def test_backward_writes_only_its_outputs(T, B, N, D, C):
    """trimul_backward writes dz and the ten parameter gradients, nothing
    around them, and leaves z, mask and dout unchanged (both directions)."""
    w = S.custom(B, N, D, C, seed=80 + N, mask_kind="random_frac", mask_frac=0.25)
    z0, m0, params = S.make_case(w, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(81 + N)
    d0 = torch.randn(z0.shape, generator=g, device="cuda").to(torch.bfloat16)
    shapes = {"W_a": (C, D), "W_ga": (C, D), "W_b": (C, D), "W_gb": (C, D), "W_o": (D, C), "W_g": (D, D),
              "ln_in_gamma": (D,), "ln_in_beta": (D,), "ln_out_gamma": (C,), "ln_out_beta": (C,)}
    h = T.trimul_create(params)
    try:
        z = Guarded(z0.shape, torch.bfloat16, fill=z0)
        m = Guarded(m0.shape, torch.bfloat16, fill=m0)
        d = Guarded(d0.shape, torch.bfloat16, fill=d0)
        for direction in ("outgoing", "incoming"):
            dz = Guarded(z0.shape, torch.bfloat16)
            grads = {k: Guarded(s, torch.float32) for k, s in shapes.items()}
            T.trimul_backward(h, z.t, m.t, d.t, direction, dz=dz.t, grads={k: v.t for k, v in grads.items()},
                              flags=T.FLAG_CHECK)
            for gd, what in [(z, "z"), (m, "mask"), (d, "dout"), (dz, "dz")] + [(v, k) for k, v in grads.items()]:
                assert gd.bands_intact(), f"backward ({direction}) wrote outside {what}"
            assert bool(torch.isfinite(dz.t.float()).all())
        assert torch.equal(z.t, z0) and torch.equal(m.t, m0) and torch.equal(d.t, d0), "backward changed an input"
    finally:
        T.trimul_destroy(h)
