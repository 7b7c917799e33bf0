"""Seeded synthetic inputs for the 2:4 SpMM workloads.

This module only draws random numbers and casts them to the element types;
it holds none of the method's arithmetic (no pruning, no compression, no
product).  Both the CPU oracle's tests and the CUDA path's tests and
benchmark draw their inputs from here, so that both sides see the same bytes.

Every draw uses a ``torch.Generator`` seeded explicitly, in a fixed order:
A (weights), then B (activations), then C_in, then the per-row scale.

Workloads (weights are M x K and pruned along K; activations are stored as
X[N, K], i.e. B is K-major; outputs are Y[N, M]):

* ``small_f16``: A 256x256 fp16 N(0,1), B 256x128 fp16 N(0,1), fp32 out.
* ``decode_bf16``: A 4096x4096 bf16 N(0,0.02), B N(0,1) with N in {1,8,16,32}, bf16 out.
* ``prefill_bf16``: A 11008x4096 and 4096x11008 bf16 N(0,0.02), N = 4096,
  B N(0,1), bf16 out, beta = 1 with C_in N(0,1).
* ``int8``: A 8192x8192 int8 uniform in [-127, 127], B int8 the same, N in
  {16, 2048}, int32 accumulation, per-row fp32 scale (1/127 * U(0.5, 1.5)), bf16 out.
* ``fp8``: A 28672x8192 N(0,0.02) cast to e4m3, B N(0,1) cast to e4m3, N in
  {1, 64, 512, 4096, 8192}, bf16 out; prune/compress on the same weight in bf16.
"""
from __future__ import annotations

import dataclasses

import torch

TORCH_DTYPE = {
    "f16": torch.float16,
    "bf16": torch.bfloat16,
    "e4m3": torch.float8_e4m3fn,
    "s8": torch.int8,
    "f32": torch.float32,
    "s32": torch.int32,
}

ELEM_SIZE = {"f16": 2, "bf16": 2, "e4m3": 1, "s8": 1, "f32": 4, "s32": 4}


def generator(seed: int) -> torch.Generator:
    return torch.Generator().manual_seed(int(seed))


def draw(dtype: str, shape, std: float, gen: torch.Generator) -> torch.Tensor:
    """A CPU tensor of ``dtype``: N(0, std) cast to the type, or for int8 uniform in [-127, 127]."""
    if dtype == "s8":
        return torch.randint(-127, 128, tuple(shape), generator=gen, dtype=torch.int64).to(torch.int8)
    x = torch.randn(tuple(shape), generator=gen, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(TORCH_DTYPE[dtype])


def row_scale(M: int, gen: torch.Generator) -> torch.Tensor:
    """Per-output-channel fp32 scale, 1/127 * U(0.5, 1.5)."""
    return ((0.5 + torch.rand(M, generator=gen, dtype=torch.float32)) / 127.0).contiguous()


def raw(t: torch.Tensor) -> torch.Tensor:
    """The raw storage of a tensor as an unsigned/signed integer view (for byte-exact work)."""
    view = {1: torch.uint8, 2: torch.int16, 4: torch.int32}[t.element_size()]
    if t.dtype == torch.int8:
        return t
    return t.view(view)


@dataclasses.dataclass
class SpmmCase:
    """One sparse product C = alpha * scale[m] * (prune(A) @ B) + beta * C_in."""

    name: str
    ab: str            # element type of A and B
    c: str             # element type of C
    M: int
    N: int
    K: int
    alpha: float
    beta: float
    A: torch.Tensor    # [M, K] dense weights (pruned by the path under test)
    X: torch.Tensor    # [N, K] activations (B K-major)
    C_in: torch.Tensor | None   # [N, M] or None
    scale: torch.Tensor | None  # [M] fp32 or None


def spmm_case(ab: str, c: str, M: int, N: int, K: int, *, a_std: float = 1.0, b_std: float = 1.0,
              alpha: float = 1.0, beta: float = 0.0, with_scale: bool = False, seed: int = 0,
              name: str = "") -> SpmmCase:
    g = generator(seed)
    A = draw(ab, (M, K), a_std, g)
    X = draw(ab, (N, K), b_std, g)
    C_in = draw(c if c != "s32" else "f32", (N, M), 1.0, g) if beta != 0.0 else None
    scale = row_scale(M, g) if with_scale else None
    return SpmmCase(name or f"{ab}->{c} {M}x{N}x{K}", ab, c, M, N, K, alpha, beta, A, X, C_in, scale)


# The five workload families, as (constructor arguments) per instance.
def small_f16(seed: int = 0) -> SpmmCase:
    return spmm_case("f16", "f32", 256, 128, 256, a_std=1.0, seed=seed, name="small_f16 256x128x256")


def decode_bf16(N: int, seed: int = 0) -> SpmmCase:
    return spmm_case("bf16", "bf16", 4096, N, 4096, a_std=0.02, seed=seed, name=f"decode_bf16 N={N}")


def prefill_bf16(M: int, K: int, N: int = 4096, seed: int = 0) -> SpmmCase:
    return spmm_case("bf16", "bf16", M, N, K, a_std=0.02, beta=1.0, seed=seed,
                     name=f"prefill_bf16 {M}x{N}x{K}")


def int8(N: int, out: str = "bf16", seed: int = 0) -> SpmmCase:
    return spmm_case("s8", out, 8192, N, 8192, with_scale=(out != "s32"), seed=seed,
                     name=f"int8 N={N} -> {out}")


def fp8(N: int, seed: int = 0, M: int = 28672, K: int = 8192) -> SpmmCase:
    return spmm_case("e4m3", "bf16", M, N, K, a_std=0.02, seed=seed, name=f"fp8 {M}x{N}x{K}")


def prune_weight_bf16(M: int = 28672, K: int = 8192, seed: int = 0) -> torch.Tensor:
    """The bf16 N(0, 0.02) weight that the prune/compress timing runs on."""
    return draw("bf16", (M, K), 0.02, generator(seed))


DECODE_NS = (1, 8, 16, 32)
INT8_NS = (16, 2048)
FP8_NS = (1, 64, 512, 4096, 8192)
PREFILL_SHAPES = ((11008, 4096), (4096, 11008))
