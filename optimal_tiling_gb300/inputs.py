"""Seeded synthetic inputs: the one module both the CUDA path's callers and the
oracle's callers draw from.  It holds no attention arithmetic at all: only
random draws, casts and the block-mask pattern.

Recipe (same for every workload):
  * one CPU ``torch.Generator`` seeded with ``seed`` (0 by default) draws fp32
    ``randn`` tensors of shape [B, H, N, d] in the order Q, K, V, dO;
  * bf16 workloads cast each draw to bf16 (round to nearest even);
  * the score scale is 1/sqrt(d) unless the workload fixes it (the fp32 case
    uses s = 1).

The block mask for the block-sparse workload is a uint8 [nb, nb] array,
nb = ceil(N / 128), shared by every (batch, head): key block bj is kept for
query block bi when bj - bi is in {-2, -1, 0, +1} (a band four blocks wide
around the diagonal, clipped at the edges), and every other block is kept
independently with probability 0.1 from its own CPU generator seeded with 0.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

MASK_BLOCK = 128


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shape, dtype, scale and mask kind."""
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str            # "f32" or "bf16"
    scale: float
    mask: str = "none"    # "none" | "band_random"
    passes: tuple = ("fwd",)
    extra: dict = field(default_factory=dict)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def shape(self):
        return (self.B, self.H, self.N, self.d)


def _s(d: int) -> float:
    return 1.0 / math.sqrt(d)


# The five workloads the target names, plus the dense shape of the fifth one
# (the throughput target is stated at N=16384, d=128 without a mask).
WORKLOADS = {
    "fp32_small": Workload("fp32_small", 1, 1, 256, 64, "f32", 1.0, passes=("fwd", "bwd")),
    "teaching": Workload("teaching", 4, 16, 4096, 64, "bf16", _s(64), passes=("fwd", "bwd")),
    "dsweep_d64": Workload("dsweep_d64", 2, 16, 8192, 64, "bf16", _s(64), passes=("fwd", "mat")),
    "dsweep_d128": Workload("dsweep_d128", 2, 16, 8192, 128, "bf16", _s(128), passes=("fwd", "mat")),
    "dsweep_d256": Workload("dsweep_d256", 2, 16, 8192, 256, "bf16", _s(256), passes=("fwd", "mat", "bwd")),
    "bwd_d128": Workload("bwd_d128", 4, 16, 4096, 128, "bf16", _s(128), passes=("fwd", "bwd", "matbwd")),
    "sparse_16k": Workload("sparse_16k", 1, 16, 16384, 128, "bf16", _s(128), mask="band_random",
                           passes=("fwd", "bwd")),
    "dense_16k": Workload("dense_16k", 1, 16, 16384, 128, "bf16", _s(128), passes=("fwd", "bwd")),
}


def make_inputs(B: int, H: int, N: int, d: int, dtype=torch.bfloat16, seed: int = 0,
                with_do: bool = True):
    """Draw Q, K, V (and dO) on the CPU in that order from one seeded generator."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    names = ("q", "k", "v", "do") if with_do else ("q", "k", "v")
    out = {}
    for nm in names:
        x = torch.randn((B, H, N, d), generator=g, dtype=torch.float32)
        out[nm] = x.to(dtype) if dtype != torch.float32 else x
    return out


def make_decode_inputs(B: int, H: int, Nq: int, Nk: int, d: int, dtype=torch.bfloat16, seed: int = 0):
    """Rectangular (decode-shaped) inputs: Q [B, H, Nq, d], then K and V [B, H, Nk, d],
    drawn in that order from one seeded CPU generator."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    out = {"q": torch.randn((B, H, Nq, d), generator=g, dtype=torch.float32)}
    for nm in ("k", "v"):
        out[nm] = torch.randn((B, H, Nk, d), generator=g, dtype=torch.float32)
    return {k: (v.to(dtype) if dtype != torch.float32 else v) for k, v in out.items()}


# Decode workload: one new query per head against a 32k-token K/V cache held in HBM.
DECODE_WORKLOAD = {"name": "decode_32k", "B": 8, "H": 32, "Nq": 1, "Nk": 32768, "d": 128}


def num_mask_blocks(N: int) -> int:
    return (N + MASK_BLOCK - 1) // MASK_BLOCK


def band_random_mask(N: int, seed: int = 0, p: float = 0.1) -> torch.Tensor:
    """Band {-2,-1,0,+1} around the diagonal plus independent off-band blocks with probability p."""
    nb = num_mask_blocks(N)
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    r = torch.rand((nb, nb), generator=g)
    bi = torch.arange(nb).view(nb, 1)
    bj = torch.arange(nb).view(1, nb)
    off = bj - bi
    band = (off >= -2) & (off <= 1)
    return (band | (r < p)).to(torch.uint8)


def band_random_mask_fine(N: int, heads: int, seed: int = 0, p: float = 0.1) -> torch.Tensor:
    """One mask per head over 64-row blocks, [heads, nb, nb] with nb = ceil(N / 64): the same band
    {-2,-1,0,+1} around the diagonal (now of 64-blocks) plus independent off-band blocks with
    probability p, head h drawn from a generator seeded seed + h."""
    nb = (N + 63) // 64
    bi = torch.arange(nb).view(nb, 1)
    bj = torch.arange(nb).view(1, nb)
    off = bj - bi
    band = (off >= -2) & (off <= 1)
    out = torch.empty((heads, nb, nb), dtype=torch.uint8)
    for h in range(heads):
        g = torch.Generator(device="cpu")
        g.manual_seed(seed + h)
        out[h] = (band | (torch.rand((nb, nb), generator=g) < p)).to(torch.uint8)
    return out


def block_diagonal_mask(N: int) -> torch.Tensor:
    nb = num_mask_blocks(N)
    return torch.eye(nb, dtype=torch.uint8)


def random_block_mask(N: int, seed: int, p: float, keep_diagonal: bool = True) -> torch.Tensor:
    nb = num_mask_blocks(N)
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    m = torch.rand((nb, nb), generator=g) < p
    if keep_diagonal:
        m |= torch.eye(nb, dtype=torch.bool)
    return m.to(torch.uint8)


def workload_inputs(w: Workload, seed: int = 0, with_do: bool = True):
    """Inputs plus mask (or None) for a named workload."""
    x = make_inputs(w.B, w.H, w.N, w.d, w.torch_dtype, seed=seed, with_do=with_do)
    mask = band_random_mask(w.N, seed=seed) if w.mask == "band_random" else None
    return x, mask
