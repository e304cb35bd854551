"""trimul_forward_noalloc: the forward for callers that must not allocate.

Some callers of this library cannot call cudaMalloc while they run: a
framework whose caching allocator already owns the GPU's memory, or a serving
loop that forbids device allocation after start-up.  trimul_forward_noalloc
keeps its a, b and x planes in a fixed scratch array that is part of the
library's device image instead of a workspace it allocates.  These tests call
it through the C ABI and check it against trimul_forward, twice in a row with
different inputs and directions (the second call must not see the first
one's scratch contents), and check that a size beyond the fixed scratch is
refused with a clear error.

This file is named so that pytest collects it last.
"""

import ctypes

import pytest
import torch

from co_folding_pair_gb300 import _lib
from co_folding_pair_gb300 import synthetic as S
from tests._util import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def T():
    from co_folding_pair_gb300 import trimul
    return trimul


def _noalloc(lib, h, z, mask, direction, out, flags):
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.trimul_forward_noalloc(h.ptr, ctypes.c_void_p(z.data_ptr()),
                                      ctypes.c_void_p(mask.data_ptr()) if mask is not None else None,
                                      z.shape[0], z.shape[1], 0 if direction == "outgoing" else 1,
                                      ctypes.c_void_p(out.data_ptr()), s, flags)


def test_noalloc_matches_forward_on_two_calls(T):
    lib = _lib.load()
    w1 = S.custom(2, 136, 64, 64, seed=41, mask_kind="random_frac", mask_frac=0.25)
    w2 = S.custom(2, 136, 64, 64, seed=42, mask_kind="padding", mask_frac=0.15)
    z1, m1, params = S.make_case(w1, device="cuda")
    z2, m2, _ = S.make_case(w2, device="cuda")
    assert (6 * 64 + 8) * 2 * 136 * 136 <= lib.trimul_noalloc_scratch_bytes()
    h = T.trimul_create(params)
    try:
        for z, m, direction in ((z1, m1, "outgoing"), (z2, m2, "incoming")):
            ref = T.trimul_forward(h, z, m, direction, flags=T.FLAG_CHECK)
            out = torch.full_like(z, float("nan"))
            assert _noalloc(lib, h, z, m, direction, out, T.FLAG_CHECK) == 0, T.trimul_last_error()
            torch.cuda.synchronize()
            assert_close(out.double().cpu().numpy(), ref.double().cpu().numpy(), f"noalloc {direction}")
    finally:
        T.trimul_destroy(h)


def test_noalloc_on_a_fresh_handle_allocates_nothing(T):
    """On a handle that has never run trimul_forward (so it owns no workspace),
    trimul_forward_noalloc leaves the device's free memory unchanged and
    matches trimul_forward, which runs only afterwards.

    The library's device image, which holds the fixed scratch, is loaded by
    the CUDA driver when the library is first used on the device; one call
    on another handle comes first so that this load is not counted."""
    lib = _lib.load()
    w = S.custom(1, 128, 64, 64, seed=44, mask_kind="random_frac", mask_frac=0.2)
    z, m, params = S.make_case(w, device="cuda")
    out = torch.empty_like(z)
    warm = T.trimul_create(params)
    try:
        assert _noalloc(lib, warm, z, m, "incoming", out, T.FLAG_CHECK) == 0, T.trimul_last_error()
    finally:
        T.trimul_destroy(warm)
    h = T.trimul_create(params)
    try:
        out.fill_(float("nan"))
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        assert _noalloc(lib, h, z, m, "outgoing", out, T.FLAG_CHECK) == 0, T.trimul_last_error()
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info()
        assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
        ref = T.trimul_forward(h, z, m, "outgoing", flags=T.FLAG_CHECK)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    finally:
        T.trimul_destroy(h)


def test_noalloc_rejects_sizes_beyond_its_scratch(T):
    lib = _lib.load()
    w = S.custom(1, 1024, 64, 64, seed=43)
    z, mask, params = S.make_case(w, device="cuda")
    out = torch.empty_like(z)
    h = T.trimul_create(params)
    try:
        assert (6 * 64 + 8) * 1024 * 1024 > lib.trimul_noalloc_scratch_bytes()
        assert _noalloc(lib, h, z, mask, "outgoing", out, 0) == 2  # TRIMUL_ERR_SHAPE
        assert "fixed scratch" in T.trimul_last_error()
    finally:
        T.trimul_destroy(h)
