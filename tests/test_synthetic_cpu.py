"""The seeded input recipe on CPU: shapes, dtypes, mask structures, value
structure and determinism of the synthetic workloads (no GPU, no method
arithmetic)."""

import math

import numpy as np
import pytest
import torch

from co_folding_pair_gb300 import synthetic as S


def _token_mask_from_pairs(mask):
    """The token mask t with mask = t_i t_j (0/1 values): the diagonal."""
    m = mask.float()
    return torch.stack([torch.diagonal(m[b]) for b in range(m.shape[0])])


def test_shapes_dtypes_and_weight_layout():
    w = S.custom(2, 16, 24, 40, seed=5)
    z, mask, p = S.make_case(w)
    assert z.shape == (2, 16, 16, 24) and z.dtype == torch.bfloat16
    assert mask.shape == (2, 16, 16) and mask.dtype == torch.bfloat16
    for k in ("W_a", "W_ga", "W_b", "W_gb"):
        assert p[k].shape == (40, 24) and p[k].dtype == torch.bfloat16
    assert p["W_o"].shape == (24, 40) and p["W_g"].shape == (24, 24)
    assert p["ln_in_gamma"].shape == (24,) and p["ln_out_beta"].shape == (40,)
    assert p["ln_in_gamma"].dtype == torch.float32


def test_deterministic_per_seed_and_different_across_seeds():
    w = S.custom(1, 16, 32, 32, seed=9)
    z1, m1, p1 = S.make_case(w)
    z2, m2, p2 = S.make_case(w)
    assert torch.equal(z1, z2) and torch.equal(m1, m2)
    assert all(torch.equal(p1[k], p2[k]) for k in p1)
    z3, _, p3 = S.make_case(S.custom(1, 16, 32, 32, seed=10))
    assert not torch.equal(z1, z3) and not torch.equal(p1["W_a"], p3["W_a"])


def test_weight_scale_is_one_over_fan_in():
    w = S.custom(1, 8, 256, 128, seed=3)
    _, _, p = S.make_case(w)
    # N(0, 1/fan_in): the sample variance over 32k draws is within a few percent
    assert abs(p["W_a"].float().var().item() * 256 - 1.0) < 0.05
    assert abs(p["W_o"].float().var().item() * 128 - 1.0) < 0.05
    g = p["ln_in_gamma"]
    assert abs(g.mean().item() - 1.0) < 0.05 and 0.05 < g.std().item() < 0.15


def test_last_frac_mask_masks_the_tail_tokens():
    w = S.WORKLOADS["n256_d128_c128_tailmask"]
    _, mask, _ = S.make_case(w)
    t = _token_mask_from_pairs(mask)[0]
    cut = math.floor(0.9 * w.N)
    assert t[:cut].eq(1).all() and t[cut:].eq(0).all()
    # the pair mask is the outer product of the token mask
    assert torch.equal(mask[0].float(), t[:, None] * t[None, :])


def test_padding_mask_is_a_tail_of_at_most_15_percent_per_sample():
    w = S.custom(4, 64, 32, 32, seed=2, mask_kind="padding", mask_frac=0.15)
    _, mask, _ = S.make_case(w)
    t = _token_mask_from_pairs(mask)
    for b in range(4):
        n_pad = int((t[b] == 0).sum())
        assert n_pad <= math.floor(0.15 * 64)
        assert t[b, :64 - n_pad].eq(1).all() and t[b, 64 - n_pad:].eq(0).all()


def test_random_frac_mask_masks_exactly_the_rounded_fraction():
    w = S.custom(2, 50, 32, 32, seed=4, mask_kind="random_frac", mask_frac=0.2)
    _, mask, _ = S.make_case(w)
    t = _token_mask_from_pairs(mask)
    for b in range(2):
        assert int((t[b] == 0).sum()) == round(0.2 * 50)
    assert set(torch.unique(mask.float()).tolist()) <= {0.0, 1.0}


def test_token_scale_structure():
    """z[b,i,j,:] = n * s_i s_j: rows scale with s_i (log-normal spread)."""
    w = S.custom(1, 64, 128, 32, seed=4, z_kind="token_scale")
    z, _, _ = S.make_case(w)
    rms = z.float().pow(2).mean(-1).sqrt()[0]  # [N, N] ~ s_i s_j
    row = rms.mean(1)
    # a LogNormal(0, 0.5) scale spreads the per-token rms over well more than 2x
    assert row.max() / row.min() > 2.0
    # separable in i and j: log rms ~ log s_i + log s_j
    lr = rms.log()
    resid = lr - lr.mean(1, keepdim=True) - lr.mean(0, keepdim=True) + lr.mean()
    assert resid.abs().mean() < 0.1


def test_outer_structure_is_per_channel():
    """z = noise + 0.5 u_i v_j per channel: every channel's N x N slice carries a
    rank-one component (top singular value ~ N/2) well above the noise edge
    (~ 2 sqrt(N)); plain N(0,1) inputs have no such gap."""
    def gaps(z):
        sv = torch.linalg.svdvals(z.float()[0].permute(2, 0, 1))  # [D, N] per channel
        return (sv[:, 0] / sv[:, 1])
    outer = gaps(S.make_case(S.custom(1, 128, 16, 16, seed=2, z_kind="outer"))[0])
    plain = gaps(S.make_case(S.custom(1, 128, 16, 16, seed=2))[0])
    assert outer.median() > 2.0 and plain.max() < 1.3


def test_sample_grid_is_sorted_distinct_and_seeded():
    w = S.WORKLOADS["n4096_d256_c256"]
    r1, c1 = S.sample_grid(w, 64, 64)
    r2, c2 = S.sample_grid(w, 64, 64)
    assert np.array_equal(r1[0], r2[0]) and np.array_equal(c1[0], c2[0])
    for a in (r1[0], c1[0]):
        assert len(a) == 64 and len(np.unique(a)) == 64 and np.all(np.diff(a) > 0)
        assert a.min() >= 0 and a.max() < w.N


def test_bf16_host_view_widens_exactly():
    t = torch.randn(3, 5).to(torch.bfloat16)
    v = S.Bf16HostView.of(t)
    assert np.array_equal(np.asarray(v), t.float().numpy())
    assert np.array_equal(np.asarray(v[1, 2:4]), t[1, 2:4].float().numpy())
    with pytest.raises(TypeError):
        S.Bf16HostView.of(t.float())


# ---------------------------------------------------------------- stress inputs

def test_few_partner_mask():
    w = S.custom(2, 40, 16, 8, seed=9, mask_kind="few_partners")
    _, m, _ = S.make_case(w)
    m = m.float()
    assert torch.equal(m, m.transpose(1, 2))                     # both axes see it
    assert set(torch.unique(m).tolist()) <= {0.0, 1.0}
    assert int(m[:, 20:].sum(-1).max()) <= 3                     # tokens >= N/2: at most 3 partners
    assert bool((m[:, :20, :20] == 1).all())                     # the first half is unmasked among itself


def test_soft_mask_values():
    w = S.custom(1, 256, 16, 8, seed=9, mask_kind="soft")
    _, m, _ = S.make_case(w)
    m = m.float()
    assert float(m.min()) > 0.0 and float(m.max()) <= 1.0
    assert float(m.min()) < 1e-3                                  # pair weights down to ~1e-4
    assert 0.3 < float((m.diagonal(dim1=1, dim2=2) == 1).float().mean()) < 0.7  # about half the tokens keep 1


def test_loose_layer():
    w = S.custom(1, 8, 64, 32, seed=9, layer_kind="loose")
    p = S.make_params(w, torch.Generator().manual_seed(9))
    q = S.make_params(S.custom(1, 8, 64, 32, seed=9), torch.Generator().manual_seed(9))
    assert int((p["ln_in_gamma"] == 4.0).sum()) == 4
    for k in ("W_a", "W_b"):
        changed = (p[k] != q[k]).any(dim=1)
        assert int(changed.sum()) == 4
        ratio = p[k][changed].float().norm(dim=1) / q[k][changed].float().norm(dim=1)
        assert torch.allclose(ratio, torch.full_like(ratio, 4.0), rtol=1e-2)
    for k in ("W_ga", "W_gb", "W_o", "W_g", "ln_in_beta", "ln_out_gamma", "ln_out_beta"):
        assert torch.equal(p[k], q[k])


def test_common_offset():
    w = S.custom(1, 32, 64, 8, seed=9, z_kind="offset", z_offset=50.0)
    z, _, _ = S.make_case(w)
    z = z.float()
    assert abs(float(z.mean()) - 50.0) < 0.05 and 0.9 < float(z.std()) < 1.1
