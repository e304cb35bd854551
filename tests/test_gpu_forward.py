"""End-to-end parity of trimul_forward (C ABI) against the fp64 oracle, plus edge
cases and error paths.

Tolerance (per element and over the evaluated set):
    |gpu - ref| <= 1e-2 + 1e-2 |ref|,   ||gpu - ref||_F / ||ref||_F <= 5e-3.
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


def _full_case(T, w, direction, mask_none=False):
    z, mask, params = S.make_case(w, device="cuda")
    h = T.trimul_create(params)
    try:
        out = T.trimul_forward(h, z, None if mask_none else mask, direction, flags=T.FLAG_CHECK)
        torch.cuda.synchronize()
    finally:
        T.trimul_destroy(h)
    ref = O.trimul_forward(_np(z), None if mask_none else _np(mask), _params_np(params), direction)
    return _np(out), ref


# ---------------------------------------------------------------- full oracle

@pytest.mark.parametrize("direction", ["outgoing", "incoming"])
def test_forward_n64_d32(T, direction):
    got, ref = _full_case(T, S.WORKLOADS["n64_d32_c32"], direction)
    assert_close(got, ref, f"n64 {direction}")


@pytest.mark.parametrize("direction", ["outgoing", "incoming"])
def test_forward_n256_tailmask(T, direction):
    got, ref = _full_case(T, S.WORKLOADS["n256_d128_c128_tailmask"], direction)
    assert_close(got, ref, f"n256 {direction}")


@pytest.mark.parametrize("direction", ["outgoing", "incoming"])
@pytest.mark.parametrize("B,N,D,C,mask_kind", [
    (2, 136, 64, 32, "padding"),
    (1, 200, 256, 256, "random_frac"),
    (3, 24, 32, 64, "ones"),
    (1, 8, 8, 8, "ones"),
    (1, 72, 256, 128, "random_frac"),
    # input projection with three resident weight slabs and a ring of four z buffers
    (1, 80, 136, 64, "padding"),
    # three 128-channel weight groups (the pair's last group lies past the weights)
    (1, 64, 192, 192, "random_frac"),
])
def test_forward_ragged(T, direction, B, N, D, C, mask_kind):
    w = S.custom(B, N, D, C, seed=N + D, mask_kind=mask_kind, mask_frac=0.2)
    got, ref = _full_case(T, w, direction)
    assert_close(got, ref, f"B{B} N{N} D{D} C{C} {direction}")


def test_forward_token_scale(T):
    w = S.custom(1, 128, 256, 128, seed=4, z_kind="token_scale", mask_kind="random_frac", mask_frac=0.2)
    got, ref = _full_case(T, w, "incoming")
    assert_close(got, ref, "token scale incoming")


def test_forward_structured(T):
    w = S.custom(2, 128, 128, 128, seed=2, z_kind="outer", mask_kind="padding", mask_frac=0.15)
    got, ref = _full_case(T, w, "outgoing")
    assert_close(got, ref, "outer-product structure")


# ---------------------------------------------------------------- sampled oracle at the workload sizes

def _sampled(T, w, direction, n_rows=64, n_cols=64):
    """Forward at the workload's full size; the oracle evaluates a seeded
    rows x cols grid of pairs per batch element exactly."""
    z, mask, params = S.make_case(w, device="cuda")
    h = T.trimul_create(params)
    try:
        out = T.trimul_forward(h, z, mask, direction, flags=T.FLAG_CHECK)
        torch.cuda.synchronize()
    finally:
        T.trimul_destroy(h)
    rows, cols = S.sample_grid(w, n_rows, n_cols)
    got = [out[b][np.ix_(rows[b], cols[b])].double().cpu().numpy() for b in range(w.B)]
    del out
    zh = S.Bf16HostView.of(z.cpu())  # the oracle widens only the slices it reads
    del z
    ref = O.trimul_forward_sampled(zh, mask.float().cpu().numpy(), _params_np(params), direction, rows, cols)
    return np.concatenate([g.ravel() for g in got]), np.concatenate([r.ravel() for r in ref])


@pytest.mark.parametrize("direction", ["outgoing", "incoming"])
def test_forward_b2_n1024_sampled(T, direction):
    got, ref = _sampled(T, S.WORKLOADS["b2_n1024_d128_c128_outer"], direction, 48, 48)
    assert_close(got, ref, f"b2 n1024 {direction}")


def test_forward_n4096_sampled(T):
    got, ref = _sampled(T, S.WORKLOADS["n4096_d256_c256"], "outgoing", 64, 64)
    assert_close(got, ref, "n4096 outgoing")


def test_forward_n3072_sampled(T):
    got, ref = _sampled(T, S.WORKLOADS["n3072_d256_c128_scaled"], "incoming", 64, 64)
    assert_close(got, ref, "n3072 incoming")


# ---------------------------------------------------------------- semantics / edge cases

def test_null_mask_equals_ones_mask_bitwise(T):
    w = S.custom(1, 96, 64, 64, seed=21)
    z, mask, params = S.make_case(w, device="cuda")
    h = T.trimul_create(params)
    try:
        o1 = T.trimul_forward(h, z, None, "outgoing")
        o2 = T.trimul_forward(h, z, torch.ones_like(mask), "outgoing")
        torch.cuda.synchronize()
        assert torch.equal(o1, o2)
    finally:
        T.trimul_destroy(h)


def test_deterministic(T):
    w = S.custom(1, 160, 128, 64, seed=22, mask_kind="random_frac", mask_frac=0.3)
    z, mask, params = S.make_case(w, device="cuda")
    h = T.trimul_create(params)
    try:
        o1 = T.trimul_forward(h, z, mask, "incoming").clone()
        o2 = T.trimul_forward(h, z, mask, "incoming")
        torch.cuda.synchronize()
        assert torch.equal(o1, o2)
    finally:
        T.trimul_destroy(h)


def test_two_handles_on_two_streams_concurrently(T):
    """Handles own separate workspaces: two handles running at the same time on
    two streams give the same bits as each run alone."""
    w1 = S.custom(1, 128, 128, 64, seed=31, mask_kind="random_frac", mask_frac=0.2)
    w2 = S.custom(2, 96, 64, 128, seed=32)
    z1, m1, p1 = S.make_case(w1, device="cuda")
    z2, m2, p2 = S.make_case(w2, device="cuda")
    h1, h2 = T.trimul_create(p1), T.trimul_create(p2)
    try:
        ref1 = T.trimul_forward(h1, z1, m1, "outgoing").clone()
        ref2 = T.trimul_forward(h2, z2, m2, "incoming").clone()
        torch.cuda.synchronize()
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        outs = []
        for _ in range(3):
            with torch.cuda.stream(s1):
                a = T.trimul_forward(h1, z1, m1, "outgoing", stream=s1)
            with torch.cuda.stream(s2):
                b = T.trimul_forward(h2, z2, m2, "incoming", stream=s2)
            outs.append((a, b))
        torch.cuda.synchronize()
        for a, b in outs:
            assert torch.equal(a, ref1) and torch.equal(b, ref2)
    finally:
        T.trimul_destroy(h1)
        T.trimul_destroy(h2)


@pytest.mark.parametrize("direction", ["outgoing", "incoming"])
def test_masked_positions_do_not_matter_bitwise(T, direction):
    """Changing z where m = 0 leaves out bitwise unchanged where m = 1 (a = b = 0 exactly)."""
    w = S.custom(1, 128, 64, 64, seed=23, mask_kind="random_frac", mask_frac=0.3)
    z, mask, params = S.make_case(w, device="cuda")
    z2 = z.clone()
    sel = mask == 0
    z2[sel] = (torch.randn_like(z2[sel].float()) * 50).to(torch.bfloat16)
    h = T.trimul_create(params)
    try:
        o1 = T.trimul_forward(h, z, mask, direction).clone()
        o2 = T.trimul_forward(h, z2, mask, direction)
        torch.cuda.synchronize()
        keep = mask == 1
        assert torch.equal(o1[keep], o2[keep])
    finally:
        T.trimul_destroy(h)


def test_fully_masked_closed_form(T):
    """m = 0: x = 0, LN_out(0) = beta_out, out = sigmoid(z' W_g^T) * (beta_out W_o^T)."""
    w = S.custom(1, 64, 64, 32, seed=24)
    z, mask, params = S.make_case(w, device="cuda")
    mask.zero_()
    h = T.trimul_create(params)
    try:
        out = T.trimul_forward(h, z, mask, "outgoing", flags=T.FLAG_CHECK)
        torch.cuda.synchronize()
    finally:
        T.trimul_destroy(h)
    pn = _params_np(params)
    zn = O.layer_norm(_np(z), pn["ln_in_gamma"], pn["ln_in_beta"], 1e-5)
    ref = 1 / (1 + np.exp(-(zn @ pn["W_g"].T))) * (pn["ln_out_beta"] @ pn["W_o"].T)
    assert_close(_np(out), ref, "fully masked")


def test_forward_host_matches_device(T):
    w = S.custom(2, 88, 64, 64, seed=25, mask_kind="padding", mask_frac=0.15)
    z, mask, params = S.make_case(w, device="cuda")
    h = T.trimul_create(params)
    try:
        od = T.trimul_forward(h, z, mask, "outgoing")
        zh, mh = z.cpu().pin_memory(), mask.cpu().pin_memory()
        oh = T.trimul_forward_host(h, zh, mh, "outgoing", flags=T.FLAG_CHECK)
        torch.cuda.synchronize()
        assert torch.equal(od.cpu(), oh)
    finally:
        T.trimul_destroy(h)


def test_forward_host_chunked_matches_device(T):
    """z above the chunking threshold (256 MB): the host-buffer path copies and
    computes in tile ranges on three streams; the result is bitwise the device path's."""
    w = S.custom(1, 1024, 128, 64, seed=29, mask_kind="random_frac", mask_frac=0.1)
    z, mask, params = S.make_case(w, device="cuda")
    assert z.numel() * 2 >= 256 << 20
    h = T.trimul_create(params)
    try:
        od = T.trimul_forward(h, z, mask, "incoming")
        zh, mh = z.cpu().pin_memory(), mask.cpu().pin_memory()
        oh = T.trimul_forward_host(h, zh, mh, "incoming", flags=T.FLAG_CHECK)
        torch.cuda.synchronize()
        assert torch.equal(od.cpu(), oh)
    finally:
        T.trimul_destroy(h)


@pytest.mark.parametrize("defer", [False, True])
def test_forward_host_back_to_back_calls(T, defer):
    """Three host-buffer calls enqueued without a sync in between (alternate
    staging slots, copies overlapping the previous call; with FLAG_DEFER_OUTPUT
    the output copies also overlap the next call's kernels, joined by
    trimul_host_join) each match the device path."""
    w = S.custom(2, 512, 128, 64, seed=30, mask_kind="padding", mask_frac=0.1)
    zs = []
    for k in range(3):
        z, mask, params = S.make_case(S.custom(2, 512, 128, 64, seed=30 + k, mask_kind="padding", mask_frac=0.1),
                                      device="cuda")
        zs.append((z, mask))
    _, _, params = S.make_case(w, device="cpu")
    h = T.trimul_create(params)
    try:
        ref = [T.trimul_forward(h, z, m, "outgoing").cpu() for z, m in zs]
        host = [(z.cpu().pin_memory(), m.cpu().pin_memory()) for z, m in zs]
        outs = [torch.empty_like(hz).pin_memory() for hz, _ in host]
        for (hz, hm), o in zip(host, outs):
            T.trimul_forward_host(h, hz, hm, "outgoing", out_host=o, flags=T.FLAG_DEFER_OUTPUT if defer else 0)
        if defer:
            T.trimul_host_join(h)
        torch.cuda.synchronize()
        for k in range(3):
            assert torch.equal(outs[k], ref[k]), f"call {k}"
    finally:
        T.trimul_destroy(h)


def test_prepare_then_larger_call_grows_workspace(T):
    w = S.custom(1, 64, 32, 32, seed=26)
    z, mask, params = S.make_case(w, device="cuda")
    h = T.trimul_create(params)
    try:
        T.trimul_prepare(h, 1, 16)
        out = T.trimul_forward(h, z, mask, "outgoing", flags=T.FLAG_CHECK)
        torch.cuda.synchronize()
        ref = O.trimul_forward(_np(z), _np(mask), _params_np(params), "outgoing")
        assert_close(_np(out), ref, "grown workspace")
    finally:
        T.trimul_destroy(h)


# ---------------------------------------------------------------- errors

def test_argument_errors(T):
    w = S.custom(1, 64, 32, 32, seed=27)
    z, mask, params = S.make_case(w, device="cuda")
    h = T.trimul_create(params)
    try:
        lib = T._lib.load()
        import ctypes
        s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        zp, op = ctypes.c_void_p(z.data_ptr()), ctypes.c_void_p(torch.empty_like(z).data_ptr())
        assert lib.trimul_forward(h.ptr, zp, None, 1, 60, 0, op, s, 0) == 2     # N % 8
        assert lib.trimul_forward(h.ptr, None, None, 1, 64, 0, op, s, 0) == 1   # null z
        assert lib.trimul_forward(h.ptr, zp, None, 1, 64, 5, op, s, 0) == 1     # bad direction
        assert lib.trimul_forward(h.ptr, zp, None, 0, 64, 0, op, s, 0) == 2     # B = 0
        assert lib.trimul_forward(h.ptr, zp, None, 1, 0, 0, op, s, 0) == 2      # N = 0 (empty)
        assert lib.trimul_forward(h.ptr, zp, None, 1, 46344, 0, op, s, 0) == 2  # N*N beyond 2^31 pairs
        assert lib.trimul_inproj(h.ptr, zp, None, 1, 0, op, op, s, 0) == 2      # stage calls check too
        assert lib.trimul_forward(h.ptr, zp, None, 1, 64, 0, zp, s, 0) == 1     # out aliases z
        assert lib.trimul_forward(None, zp, None, 1, 64, 0, op, s, 0) == 1      # null handle
        assert "handle" in T.trimul_last_error()
    finally:
        T.trimul_destroy(h)


def test_weights_outside_fp16_range_rejected(T):
    params = S.make_params(S.custom(1, 8, 32, 32, seed=1), torch.Generator().manual_seed(1))
    params["W_g"] = params["W_g"].clone()
    params["W_g"][0, 0] = 1e6
    with pytest.raises(T.TrimulError) as ei:
        T.trimul_create(params)
    assert ei.value.status == 1


def test_injected_stall_times_out_and_context_survives(T):
    """The producer issues no loads; the consumers' bounded waits expire, the
    call reports TRIMUL_ERR_TIMEOUT, and the next normal call is correct."""
    w = S.custom(1, 64, 32, 32, seed=28)
    z, mask, params = S.make_case(w, device="cuda")
    h = T.trimul_create(params)
    try:
        with pytest.raises(T.TrimulError) as ei:
            T.trimul_forward(h, z, mask, "outgoing", flags=T.FLAG_CHECK | T.FLAG_INJECT_STALL)
        assert ei.value.status == 6
        out = T.trimul_forward(h, z, mask, "outgoing", flags=T.FLAG_CHECK)
        torch.cuda.synchronize()
        ref = O.trimul_forward(_np(z), _np(mask), _params_np(params), "outgoing")
        assert_close(_np(out), ref, "after stall")
    finally:
        T.trimul_destroy(h)
