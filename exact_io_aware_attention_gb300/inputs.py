"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module holds no attention arithmetic: it only draws random numbers. Both
the CUDA path and the fp64 oracle are fed from here, so they see bit-identical
inputs (bf16 values widen exactly to float64).

Recipe:
  * Q, K, V, dO: iid N(0, 1) fp32 from ``torch.Generator('cpu').manual_seed``,
    rounded to bf16 with round-to-nearest-even (``.to(torch.bfloat16)``), or
    to fp16 the same way where a test asks for fp16 inputs.
  * seed = 1000 * case + tensor index, with Q = 0, K = 1, V = 2, dO = 3,
    mask = 4 (``case`` numbers the workloads listed in ``WORKLOADS``).
  * block mask: ``T x T`` uint8 with T = N / 128, every diagonal tile kept and
    each off-diagonal tile kept independently with probability ``density``
    (``Tq x Tk`` for queries and keys of different lengths).
  * queries and keys of different lengths: Q and dO have Nq rows, K and V Nk
    rows, drawn with the same seeds.
"""
from __future__ import annotations

import dataclasses
import math

import torch

TILE = 128
SEED_STRIDE = 1000
TENSOR_INDEX = {"q": 0, "k": 1, "v": 2, "do": 3, "mask": 4}


@dataclasses.dataclass(frozen=True)
class Workload:
    case: int
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    sparse_density: float | None = None  # None = dense

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# The five attention workloads the method is checked and measured on.
WORKLOADS = {
    "single_head_n256_d64": Workload(1, "single_head_n256_d64", 1, 1, 256, 64, False),
    "gpt2_small_causal": Workload(2, "gpt2_small_causal", 8, 12, 1024, 64, True),
    "gpt2_medium_causal": Workload(3, "gpt2_medium_causal", 4, 16, 4096, 128, True),
    "gpt2_medium_dense": Workload(3, "gpt2_medium_dense", 4, 16, 4096, 128, False),
    "long_context_n65536": Workload(4, "long_context_n65536", 1, 16, 65536, 128, True),
    "block_sparse_n8192": Workload(5, "block_sparse_n8192", 4, 16, 8192, 64, False, 0.25),
}


def seed_for(case: int, tensor: str) -> int:
    return SEED_STRIDE * case + TENSOR_INDEX[tensor]


def normal_bf16(shape, seed: int, dtype=torch.bfloat16) -> torch.Tensor:
    """iid N(0,1) drawn in fp32 on the CPU from ``seed``, rounded to bf16 (RNE),
    or to ``dtype`` (fp16)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return torch.randn(tuple(shape), generator=g, dtype=torch.float32).to(dtype)


def block_mask(n_tiles: int, density: float, seed: int, n_key_tiles: int | None = None):
    """uint8 [n_tiles, n_key_tiles] (square by default): diagonal kept,
    off-diagonal kept iid with p=density."""
    tk = n_tiles if n_key_tiles is None else n_key_tiles
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    keep = torch.rand((n_tiles, tk), generator=g, dtype=torch.float64) < density
    keep |= torch.eye(n_tiles, tk, dtype=torch.bool)
    return keep.to(torch.uint8)


def make_inputs(B, H, N, d, case: int, with_do: bool = True, Nk: int | None = None,
                dtype=torch.bfloat16):
    """CPU tensors q (and do) of shape [B, H, N, d], k and v of shape
    [B, H, Nk, d] (Nk = N by default), bf16 or ``dtype``."""
    nk = N if Nk is None else Nk
    out = {t: normal_bf16((B, H, N if t in ("q", "do") else nk, d), seed_for(case, t), dtype)
           for t in ("q", "k", "v")}
    if with_do:
        out["do"] = normal_bf16((B, H, N, d), seed_for(case, "do"), dtype)
    return out


def make_workload_inputs(w: Workload, with_do: bool = True):
    out = make_inputs(w.B, w.H, w.N, w.d, w.case, with_do)
    out["mask"] = None
    if w.sparse_density is not None:
        out["mask"] = block_mask(w.N // TILE, w.sparse_density, seed_for(w.case, "mask"))
    return out
