"""Seeded synthetic inputs shaped like the pages' attention workloads.

This module holds shapes and random draws only -- none of the attention
arithmetic -- so that the CUDA path and the CPU oracle can be fed the same
tensors without sharing any code of the method.

Recipe (identical for every workload): a CPU ``torch.Generator`` seeded with
the workload's seed draws fp32 normals in the order q, k, v, then the bias
tables; q/k/v are N(0, 1) and cast with round-to-nearest-even to the
workload dtype; the Swin table is N(0, 0.02) kept in fp32; the SAM tables
R_h, R_w are N(0, 0.02) cast to the workload dtype.  Layout is
[B, H, N, d] contiguous with d innermost.  For Swin, B counts windows:
b' = image * nW + w with w row-major over the window grid.  A variable-length
batch (``seqlens_q`` set) draws q as one [H * sum(Lq), d] buffer -- the
concatenation over sequences of [H][Lq_s][d] -- and k, v likewise.

The workloads stand in for real images through the models the pages
profile (SAM image encoder, Swin-T stage 1, Stable Diffusion UNet): those
need datasets and trained weights, so the shapes alone are reproduced.
"""
from __future__ import annotations

import dataclasses
import itertools
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int            # slices along batch (windows for the windowed cases)
    H: int
    Nq: int
    Nk: int
    d: int
    dtype: str        # "bf16" | "fp16"
    bias: str         # "none" | "swin" | "sam"
    seed: int
    # Swin window geometry
    win: int = 0
    grid_h: int = 0
    grid_w: int = 0
    shift: int = 0
    # SAM grid (query grid == key grid) and table rows (0: 2*side-1)
    s_h: int = 0
    s_w: int = 0
    rel_len: int = 0
    # variable-length batch: per-sequence query / key token counts (B of each)
    seqlens_q: tuple = ()
    seqlens_k: tuple = ()
    note: str = ""

    @property
    def varlen(self) -> bool:
        return len(self.seqlens_q) > 0

    @property
    def cu_seqlens_q(self) -> list:
        return [0] + list(itertools.accumulate(self.seqlens_q))

    @property
    def cu_seqlens_k(self) -> list:
        return [0] + list(itertools.accumulate(self.seqlens_k))

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float16

    @property
    def flops(self) -> int:
        """4*B*H*Nq*Nk*d with the true head dim (two GEMMs, 2 flops/MAC);
        summed over the sequences of a variable-length batch."""
        if self.varlen:
            return sum(4 * self.H * a * b * self.d for a, b in zip(self.seqlens_q, self.seqlens_k))
        return 4 * self.B * self.H * self.Nq * self.Nk * self.d

    @property
    def io_bytes(self) -> int:
        """Algorithmic HBM bytes: Q, K, V read once, O written once, plus
        the bias tables."""
        e = 2
        if self.varlen:
            return 2 * self.H * (sum(self.seqlens_q) + sum(self.seqlens_k)) * self.d * e
        qo = 2 * self.B * self.H * self.Nq * self.d * e
        kv = 2 * self.B * self.H * self.Nk * self.d * e
        tab = 0
        if self.bias == "swin":
            tab = (2 * self.win - 1) ** 2 * self.H * 4
        elif self.bias == "sam":
            lh = self.rel_len or 2 * self.s_h - 1
            lw = self.rel_len or 2 * self.s_w - 1
            tab = (lh + lw) * self.d * e
        return qo + kv + tab

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# latent tokens of images of 512, 384, 256 and 448 pixels per side
_SD_RAGGED = tuple([64 * 64, 48 * 48, 32 * 32, 56 * 56] * 4)

WORKLOADS = {
    "toy": Workload("toy", B=1, H=2, Nq=64, Nk=64, d=32, dtype="bf16", bias="none", seed=0,
                    note="toy SDPA"),
    "swin_t_stage1": Workload(
        "swin_t_stage1", B=32 * 64, H=3, Nq=49, Nk=49, d=32, dtype="fp16", bias="swin", seed=1,
        win=7, grid_h=56, grid_w=56, shift=3,
        note="Swin-T stage-1 shifted-window attention: 32 images x 64 windows of 7x7"),
    "sam_vith_window": Workload(
        "sam_vith_window", B=8 * 25, H=16, Nq=196, Nk=196, d=80, dtype="bf16", bias="sam", seed=2,
        s_h=14, s_w=14,
        note="SAM ViT-H windowed encoder attention: 8 images x 25 windows of 14x14"),
    "sam_vith_global": Workload(
        "sam_vith_global", B=8, H=16, Nq=4096, Nk=4096, d=80, dtype="bf16", bias="sam", seed=3,
        s_h=64, s_w=64, note="SAM ViT-H global encoder attention on the 64x64 grid"),
    "sam_vith_global_768": Workload(
        "sam_vith_global_768", B=8, H=16, Nq=48 * 48, Nk=48 * 48, d=80, dtype="bf16", bias="sam", seed=7,
        s_h=48, s_w=48, rel_len=127,
        note="SAM ViT-H global attention on a 768-pixel input (48x48 grid) with the 1024-pixel "
             "model's 127-row tables, resampled to 95 rows"),
    "sd_unet_self": Workload(
        "sd_unet_self", B=16, H=8, Nq=4096, Nk=4096, d=40, dtype="fp16", bias="none", seed=4,
        note="Stable Diffusion UNet 64x64-latent self-attention"),
    "sd_unet_cross": Workload(
        "sd_unet_cross", B=16, H=8, Nq=4096, Nk=77, d=40, dtype="fp16", bias="none", seed=5,
        note="Stable Diffusion UNet cross-attention over 77 text tokens"),
    "sd_unet_self_varlen": Workload(
        "sd_unet_self_varlen", B=16, H=8, Nq=4096, Nk=4096, d=40, dtype="fp16", bias="none", seed=6,
        seqlens_q=_SD_RAGGED, seqlens_k=_SD_RAGGED,
        note="Stable Diffusion UNet self-attention over a nested batch of 16 images of "
             "different sizes (latent grids 64x64, 48x48, 32x32, 56x56, four of each)"),
}


@dataclasses.dataclass
class Inputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    table: torch.Tensor | None = None   # Swin [(2M-1)^2, H] fp32
    rel_h: torch.Tensor | None = None   # SAM [2*s_h-1, d] in the workload dtype
    rel_w: torch.Tensor | None = None   # SAM [2*s_w-1, d]


def make_inputs(w: Workload, seed: int | None = None) -> Inputs:
    """Draw the seeded CPU tensors of a workload (see the module recipe)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    dt = w.torch_dtype

    def normal(shape, std=1.0):
        return torch.randn(shape, generator=g, dtype=torch.float32) * std

    if w.varlen:
        tq, tk = sum(w.seqlens_q), sum(w.seqlens_k)
        q = normal((w.H * tq, w.d)).to(dt)
        k = normal((w.H * tk, w.d)).to(dt)
        v = normal((w.H * tk, w.d)).to(dt)
        return Inputs(q, k, v)
    q = normal((w.B, w.H, w.Nq, w.d)).to(dt)
    k = normal((w.B, w.H, w.Nk, w.d)).to(dt)
    v = normal((w.B, w.H, w.Nk, w.d)).to(dt)
    out = Inputs(q, k, v)
    if w.bias == "swin":
        out.table = normal(((2 * w.win - 1) ** 2, w.H), 0.02).contiguous()
    elif w.bias == "sam":
        out.rel_h = normal((w.rel_len or 2 * w.s_h - 1, w.d), 0.02).to(dt)
        out.rel_w = normal((w.rel_len or 2 * w.s_w - 1, w.d), 0.02).to(dt)
    return out
