"""Seeded synthetic inputs for TriMul: pair features, weights, LayerNorm affine, pair masks.

This module only draws random numbers and builds masks; it holds none of the
update's arithmetic.  Both the CUDA path's tests/benchmark and the CPU oracle
take their inputs from here.

Shapes follow the fold-cp-ops README ("Use" section): z is [B, N, N, D] bf16,
the pair mask is [B, N, N] bf16, and the layer's weights use the ``nn.Linear``
(out, in) layout.  The value distributions and mask structures are the five
workloads listed in ``WORKLOADS``.

Draw order for one case (both generators seeded with the case's seed):
  CPU generator: W_a, W_ga, W_b, W_gb, W_g ~ N(0, 1/D) and W_o ~ N(0, 1/C);
    then gamma = 1 + 0.1 N(0,1), beta = 0.1 N(0,1) for ln_in and ln_out;
    then the token-mask draws; then the structure draws (u, v or s).
  generator on ``device``: z ~ N(0, 1) float32 in blocks of rows i, each block
    given its structure and rounded to bf16 at once.
Weights and the mask are bf16; LayerNorm affine parameters stay float32.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    N: int
    D: int
    C: int
    directions: tuple
    seed: int
    z_kind: str = "normal"        # "normal" | "outer" | "token_scale" | "offset"
    mask_kind: str = "ones"       # "ones" | "last_frac" | "padding" | "random_frac" | "few_partners" | "soft"
    mask_frac: float = 0.0
    layer_kind: str = "default"   # "default" | "loose" (see make_params)
    z_offset: float = 0.0         # z_kind "offset": a common offset added to every z value


WORKLOADS = {
    # tiny correctness case
    "n64_d32_c32": Workload("n64_d32_c32", 1, 64, 32, 32, ("outgoing",), 0),
    # last 10% of tokens masked
    "n256_d128_c128_tailmask": Workload("n256_d128_c128_tailmask", 1, 256, 128, 128,
                                        ("outgoing", "incoming"), 1,
                                        mask_kind="last_frac", mask_frac=0.10),
    # structured pairs (per-channel outer product of two token vectors),
    # per-sample padding of 0-15% of tokens
    "b2_n1024_d128_c128_outer": Workload("b2_n1024_d128_c128_outer", 2, 1024, 128, 128,
                                         ("outgoing", "incoming"), 2, z_kind="outer",
                                         mask_kind="padding", mask_frac=0.15),
    # the fold-cp-ops README's shape: B=1, N=4096, D=256
    "n4096_d256_c256": Workload("n4096_d256_c256", 1, 4096, 256, 256, ("outgoing",), 3),
    # the README's feature width at a quarter of its token count (profiling case)
    "n1024_d256_c256": Workload("n1024_d256_c256", 1, 1024, 256, 256, ("outgoing",), 3),
    # half the feature width at a quarter of the token count (profiling case for
    # the backward, whose workspace is about 15 planes of B N^2 max(C, D) bf16)
    "n1024_d128_c128": Workload("n1024_d128_c128", 1, 1024, 128, 128, ("outgoing",), 3),
    # the token count of the README's shape with narrow features (profiling
    # case for the triangle GEMM's DRAM traffic at N = 4096)
    "n4096_d32_c32": Workload("n4096_d32_c32", 1, 4096, 32, 32, ("outgoing",), 3),
    # the same with 56 channels: two triangle launches of 28 planes, close to
    # the 29-plane launches of the README's shape (profiling case for the
    # triangle GEMM's DRAM traffic per plane)
    "n4096_d32_c56": Workload("n4096_d32_c56", 1, 4096, 32, 56, ("outgoing",), 3),
    # per-token LogNormal(0, 0.5) scale, random 20% of tokens masked
    "n3072_d256_c128_scaled": Workload("n3072_d256_c128_scaled", 1, 3072, 256, 128,
                                       ("incoming",), 4, z_kind="token_scale",
                                       mask_kind="random_frac", mask_frac=0.20),
}


def custom(B, N, D, C, seed, z_kind="normal", mask_kind="ones", mask_frac=0.0,
           directions=("outgoing", "incoming"), layer_kind="default", z_offset=0.0):
    """A workload outside the named list (odd sizes, stress layers and masks)."""
    return Workload(f"b{B}_n{N}_d{D}_c{C}_s{seed}", B, N, D, C, tuple(directions), seed,
                    z_kind, mask_kind, mask_frac, layer_kind, z_offset)


def _token_mask(w: Workload, g: torch.Generator) -> torch.Tensor:
    """[B, N] float32 token mask t (1 = kept, 0 = masked)."""
    t = torch.ones(w.B, w.N)
    if w.mask_kind == "ones":
        return t
    if w.mask_kind == "last_frac":
        t[:, int(math.floor((1.0 - w.mask_frac) * w.N)):] = 0.0
        return t
    if w.mask_kind == "padding":
        f = torch.rand(w.B, generator=g) * w.mask_frac
        for b in range(w.B):
            n_pad = int(math.floor(float(f[b]) * w.N))
            if n_pad:
                t[b, w.N - n_pad:] = 0.0
        return t
    if w.mask_kind == "random_frac":
        n_mask = int(round(w.mask_frac * w.N))
        for b in range(w.B):
            idx = torch.randperm(w.N, generator=g)[:n_mask]
            t[b, idx] = 0.0
        return t
    if w.mask_kind == "soft":
        # half of the tokens get a weight 10^U(-2, 0); pair weights go down to 1e-4
        for b in range(w.B):
            sel = torch.rand(w.N, generator=g) < 0.5
            wt = 10.0 ** (-2.0 * torch.rand(w.N, generator=g))
            t[b, sel] = wt[sel]
        return t
    raise ValueError(f"unknown mask kind {w.mask_kind!r}")


def _few_partner_mask(w: Workload, g: torch.Generator) -> torch.Tensor:
    """[B, N, N] pair mask: tokens i >= N/2 keep only 1 to 3 partners.

    A row pattern R has, for i >= N/2, ones at 1-3 random columns (all ones
    for i < N/2); the mask is R[i, k] R[k, i], so those tokens have only a
    few unmasked pairs along both axes (both contraction directions see it).
    """
    R = torch.ones(w.B, w.N, w.N)
    for b in range(w.B):
        for i in range(w.N // 2, w.N):
            k = int(torch.randint(1, 4, (1,), generator=g))
            cols = torch.randperm(w.N, generator=g)[:k]
            R[b, i] = 0.0
            R[b, i, cols] = 1.0
    return R * R.transpose(1, 2)


def make_params(w: Workload, g: torch.Generator) -> dict:
    """Weights (bf16, nn.Linear layout) and LayerNorm affine parameters (float32).

    layer_kind "loose": after the default draws, four features of gamma_in are
    set to 4 and four rows each of W_a and W_b are multiplied by 4.  The
    layer stays ordinary, but the worst-case bound on |a|, |b| that the
    weights allow grows about 16-fold over the values that actually occur.
    """
    D, C = w.D, w.C

    def lin(out_f, in_f):
        return (torch.randn(out_f, in_f, generator=g) / math.sqrt(in_f)).to(torch.bfloat16)

    p = {}
    p["W_a"] = lin(C, D)
    p["W_ga"] = lin(C, D)
    p["W_b"] = lin(C, D)
    p["W_gb"] = lin(C, D)
    p["W_g"] = lin(D, D)
    p["W_o"] = lin(D, C)
    p["ln_in_gamma"] = 1.0 + 0.1 * torch.randn(D, generator=g)
    p["ln_in_beta"] = 0.1 * torch.randn(D, generator=g)
    p["ln_out_gamma"] = 1.0 + 0.1 * torch.randn(C, generator=g)
    p["ln_out_beta"] = 0.1 * torch.randn(C, generator=g)
    if w.layer_kind == "loose":
        idx = torch.randperm(D, generator=g)[:4]
        p["ln_in_gamma"][idx] = 4.0
        for k in ("W_a", "W_b"):
            rows = torch.randperm(C, generator=g)[:4]
            p[k] = p[k].clone()
            p[k][rows] = (p[k][rows].float() * 4.0).to(torch.bfloat16)
    elif w.layer_kind != "default":
        raise ValueError(f"unknown layer kind {w.layer_kind!r}")
    return p


def make_case(w: Workload, device="cpu", row_block: int = 256):
    """Build (z, mask, params) for workload ``w``.

    z [B, N, N, D] bf16 and mask [B, N, N] bf16 live on ``device``; params stay
    on the CPU (bf16 weights, float32 LayerNorm affine).  z comes from its own
    generator on ``device`` (values drawn on a CUDA device differ from those
    drawn on the CPU for the same seed; each is deterministic for its device);
    everything else comes from one CPU generator.
    """
    device = torch.device(device)
    g = torch.Generator()
    g.manual_seed(w.seed)
    params = make_params(w, g)
    pair_mask = None
    if w.mask_kind == "few_partners":
        pair_mask = _few_partner_mask(w, g)
        t = torch.ones(w.B, w.N)
    else:
        t = _token_mask(w, g)
    u = v = s = None
    if w.z_kind == "outer":
        u = torch.randn(w.B, w.N, w.D, generator=g).to(device)
        v = torch.randn(w.B, w.N, w.D, generator=g).to(device)
    elif w.z_kind == "token_scale":
        s = torch.exp(0.5 * torch.randn(w.B, w.N, generator=g)).to(device)
    elif w.z_kind not in ("normal", "offset"):
        raise ValueError(f"unknown z kind {w.z_kind!r}")

    gz = torch.Generator(device=device)
    gz.manual_seed(w.seed)
    z = torch.empty(w.B, w.N, w.N, w.D, dtype=torch.bfloat16, device=device)
    for b in range(w.B):
        for i0 in range(0, w.N, row_block):
            i1 = min(w.N, i0 + row_block)
            blk = torch.randn(i1 - i0, w.N, w.D, generator=gz, device=device)
            if u is not None:
                # z[b, i, j, d] += 0.5 u[b, i, d] v[b, j, d]
                blk += 0.5 * u[b, i0:i1, None, :] * v[b, None, :, :]
            if s is not None:
                # z[b, i, j, :] *= s[b, i] s[b, j]
                blk *= (s[b, i0:i1, None] * s[b, None, :])[..., None]
            if w.z_kind == "offset":
                blk += w.z_offset
            z[b, i0:i1] = blk.to(torch.bfloat16)
    if pair_mask is None:
        pair_mask = t[:, :, None] * t[:, None, :]
    mask = pair_mask.to(torch.bfloat16).to(device)
    return z, mask, params


def sample_grid(w: Workload, n_rows: int, n_cols: int, seed_offset: int = 1000):
    """Seeded rows x cols token grid per batch (a sample of n_rows*n_cols pairs each)."""
    g = torch.Generator()
    g.manual_seed(w.seed + seed_offset)
    rows, cols = [], []
    for _ in range(w.B):
        r = torch.randperm(w.N, generator=g)[:min(n_rows, w.N)]
        c = torch.randperm(w.N, generator=g)[:min(n_cols, w.N)]
        rows.append(torch.sort(r).values.numpy())
        cols.append(torch.sort(c).values.numpy())
    return rows, cols


class Bf16HostView:
    """Lazy read-only view of a host (CPU) bf16 tensor for array consumers.

    Indexing returns another view; converting with ``numpy.asarray`` widens
    only the selected elements, exactly, to float32 (a bf16 value is the high
    half of the float32 with the same bits).  This lets a CPU consumer slice a
    multi-gigabyte bf16 tensor without a full float copy.
    """

    def __init__(self, u16: np.ndarray):
        self._u16 = u16
        self.shape = u16.shape
        self.ndim = u16.ndim

    @classmethod
    def of(cls, t: torch.Tensor) -> "Bf16HostView":
        if t.dtype != torch.bfloat16 or t.device.type != "cpu":
            raise TypeError("expects a CPU bf16 tensor")
        return cls(t.contiguous().view(torch.int16).numpy().view(np.uint16))

    def __getitem__(self, idx):
        return Bf16HostView(np.asarray(self._u16[idx]))

    def __array__(self, dtype=None, copy=None):
        f = (self._u16.astype(np.uint32) << 16).view(np.float32)
        return f if dtype is None else f.astype(dtype)
