"""Seeded synthetic workloads shared by the CPU oracle and the CUDA path.

This module only describes *inputs*: parameter shape lists in registration
order and seeded gradient values.  It holds none of the synchronisation
arithmetic (no chunking, no reduction order, no rounding, no bucketing), so
both sides of every parity test can draw their inputs from it without sharing
any of the method.

Recipe (rank r, micro-batch m, world size N):
  * host inputs: ``torch.Generator('cpu').manual_seed(seed)`` then
    ``torch.randn`` / ``torch.rand`` in float32; seed = r for a single bucket,
    seed = r + N*m for the m-th accumulation micro-batch.
  * device inputs at full size: the same recipe on a CUDA generator, so the
    values live only in HBM; tests snapshot the inputs they need to the host
    before any kernel runs.
  * bf16 payloads are the float32 draw converted by torch's own
    float32 -> bfloat16 cast (round to nearest even); the cast is input
    preparation, not part of the method.

The two parameter lists stand in for the models the pages measured
(a GPT-2-medium-like decoder and ResNet-50): shapes only, no weights.
"""
from __future__ import annotations

import math
from typing import List, Sequence, Tuple

import torch

Shape = Tuple[int, ...]


def numel_of(shape: Shape) -> int:
    return int(math.prod(shape)) if len(shape) else 1


def decoder_param_shapes(n_layer: int = 24, d_model: int = 1024, d_ff: int = 4096,
                         vocab: int = 50257, n_pos: int = 1024) -> List[Tuple[str, Shape]]:
    """Registration-order parameter list of a 24-layer decoder with tied LM head.

    The default sizes give 292 tensors and 354,823,168 parameters
    (1,419,292,672 bytes of fp32 gradients), the "~355M params, ~1.4 GB"
    decoder of the DDP step workload.
    """
    out: List[Tuple[str, Shape]] = [("wte", (vocab, d_model)), ("wpe", (n_pos, d_model))]
    for i in range(n_layer):
        p = f"h.{i}."
        out += [
            (p + "ln1.w", (d_model,)), (p + "ln1.b", (d_model,)),
            (p + "attn.qkv.W", (d_model, 3 * d_model)), (p + "attn.qkv.b", (3 * d_model,)),
            (p + "attn.proj.W", (d_model, d_model)), (p + "attn.proj.b", (d_model,)),
            (p + "ln2.w", (d_model,)), (p + "ln2.b", (d_model,)),
            (p + "mlp.fc.W", (d_model, d_ff)), (p + "mlp.fc.b", (d_ff,)),
            (p + "mlp.proj.W", (d_ff, d_model)), (p + "mlp.proj.b", (d_model,)),
        ]
    out += [("lnf.w", (d_model,)), ("lnf.b", (d_model,))]
    return out


def resnet50_param_shapes() -> List[Tuple[str, Shape]]:
    """Registration-order parameter list of ResNet-50 (bottleneck [3,4,6,3]).

    Convolution weights are [Cout, Cin, k, k]; every BatchNorm contributes a
    weight and a bias (running statistics are buffers, not parameters); the
    first block of each stage carries a 1x1 downsample conv + BN.  161 tensors,
    25,557,032 parameters.
    """
    out: List[Tuple[str, Shape]] = [("conv1.w", (64, 3, 7, 7)), ("bn1.w", (64,)), ("bn1.b", (64,))]
    in_ch = 64
    for li, (planes, blocks) in enumerate(zip((64, 128, 256, 512), (3, 4, 6, 3)), start=1):
        for b in range(blocks):
            p = f"layer{li}.{b}."
            out += [
                (p + "conv1.w", (planes, in_ch, 1, 1)), (p + "bn1.w", (planes,)), (p + "bn1.b", (planes,)),
                (p + "conv2.w", (planes, planes, 3, 3)), (p + "bn2.w", (planes,)), (p + "bn2.b", (planes,)),
                (p + "conv3.w", (planes * 4, planes, 1, 1)), (p + "bn3.w", (planes * 4,)), (p + "bn3.b", (planes * 4,)),
            ]
            if b == 0:
                out += [(p + "downsample.conv.w", (planes * 4, in_ch, 1, 1)),
                        (p + "downsample.bn.w", (planes * 4,)), (p + "downsample.bn.b", (planes * 4,))]
            in_ch = planes * 4
    out += [("fc.w", (1000, 2048)), ("fc.b", (1000,))]
    return out


def param_numels(shapes: Sequence[Tuple[str, Shape]]) -> List[int]:
    return [numel_of(s) for _, s in shapes]


# --------------------------------------------------------------------------
# Seeded values
# --------------------------------------------------------------------------

def _gen(seed: int, device: str = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn_f32(n: int, seed: int, std: float = 1.0, device: str = "cpu") -> torch.Tensor:
    """float32 N(0, std^2) vector of n values from generator seed ``seed``."""
    x = torch.randn(int(n), generator=_gen(seed, device), dtype=torch.float32, device=device)
    if std != 1.0:
        x.mul_(std)
    return x


def uniform_pm1_f32(n: int, seed: int, device: str = "cpu") -> torch.Tensor:
    """float32 uniform [-1, 1) vector of n values (rand * 2 - 1)."""
    x = torch.rand(int(n), generator=_gen(seed, device), dtype=torch.float32, device=device)
    return x.mul_(2.0).sub_(1.0)


def small_int_f32(n: int, seed: int, lo: int = -8, hi: int = 8, device: str = "cpu") -> torch.Tensor:
    """float32 vector of small integers in [lo, hi]: every summation order is exact."""
    return torch.randint(lo, hi + 1, (int(n),), generator=_gen(seed, device), device=device).to(torch.float32)


def to_bf16(x: torch.Tensor) -> torch.Tensor:
    """Input preparation: torch's float32 -> bfloat16 cast (round to nearest even)."""
    return x.to(torch.bfloat16)


def rank_vectors(world: int, n: int, kind: str = "randn", std: float = 1.0, dtype: str = "f32",
                 seed0: int = 0, device: str = "cpu") -> torch.Tensor:
    """[world, n] tensor; row r is drawn from seed ``seed0 + r``.

    kind: "randn" (N(0, std^2)), "uniform" (U[-1,1)), "int" (small integers).
    dtype: "f32" or "bf16" (bf16 rows are the float32 draw cast by torch).
    """
    rows = []
    for r in range(world):
        s = seed0 + r
        if kind == "randn":
            v = randn_f32(n, s, std, device)
        elif kind == "uniform":
            v = uniform_pm1_f32(n, s, device)
        elif kind == "int":
            v = small_int_f32(n, s, device=device)
        else:
            raise ValueError(kind)
        rows.append(v)
    out = torch.stack(rows) if rows else torch.empty((0, n), dtype=torch.float32, device=device)
    if dtype == "bf16":
        out = to_bf16(out)
    elif dtype != "f32":
        raise ValueError(dtype)
    return out


def microbatch_seed(rank: int, world: int, m: int) -> int:
    """Seed of rank ``rank``'s m-th accumulation micro-batch: r + N*m."""
    return rank + world * m
