"""Seeded synthetic workloads for the deterministic attention backward.

This module holds shapes and random-number recipes only: no attention
arithmetic.  Both the CUDA path (through the Python binding) and the CPU
oracle consume the tensors it draws, so the two sides see identical inputs.

Recipe (the pages use "random BF16 inputs" with no stated distribution, DASH
paper write-up, experimental setup paragraph): Q, K, V and dO are drawn
i.i.d. N(0, 1) in fp32 by a CPU ``torch.Generator`` seeded with
``seed + i`` for the i-th tensor (Q, K, V, dO), multiplied by ``gain`` and
rounded to bf16.  scale = 1/sqrt(D).  O and LSE come from the forward pass.

The four large named workloads keep the pages' hidden size of 2048
(H * D = 2048); the small one is sized so that the fp64 oracle finishes it in
well under a second.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

SEED = 1234

ALL_SCHEDULES = ("atomic", "serial", "descending_q", "shift", "symmetric_shift")


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    S: int
    D: int
    causal: bool
    tile: int
    gain: float = 1.0
    schedules: tuple = field(default_factory=tuple)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def n_blocks(self) -> int:
        return (self.S + self.tile - 1) // self.tile

    def flops(self) -> float:
        """Conventional attention-backward FLOP count (five matmuls):
        10*B*H*S^2*D for a full mask, half of it for a causal mask."""
        f = 10.0 * self.B * self.H * self.S * self.S * self.D
        return f / 2 if self.causal else f

    def describe(self) -> str:
        return (f"B={self.B} H={self.H} S={self.S} D={self.D} "
                f"{'causal' if self.causal else 'full'} tile={self.tile}")


def _valid(causal: bool, schedules):
    out = []
    for s in schedules:
        if s == "shift" and causal:
            continue
        if s == "symmetric_shift" and not causal:
            continue
        out.append(s)
    return tuple(out)


WORKLOADS = {
    # small case: the fp64 oracle finishes it in well under a second
    "small_full_s256_d64": Workload("small_full_s256_d64", 1, 2, 256, 64, False, 64, 1.0,
                                    _valid(False, ALL_SCHEDULES)),
    "causal_s2048_d128": Workload("causal_s2048_d128", 4, 16, 2048, 128, True, 128, 1.0,
                                  _valid(True, ALL_SCHEDULES)),
    "full_s4096_d128": Workload("full_s4096_d128", 2, 16, 4096, 128, False, 128, 1.0,
                                _valid(False, ALL_SCHEDULES)),
    "causal_s8192_d64": Workload("causal_s8192_d64", 1, 32, 8192, 64, True, 128, 0.5,
                                 _valid(True, ALL_SCHEDULES)),
    "causal_s16384_d128": Workload("causal_s16384_d128", 1, 16, 16384, 128, True, 128, 1.0,
                                   _valid(True, ALL_SCHEDULES)),
}

WORKLOAD_ORDER = list(WORKLOADS)


def draw(shape, seed: int, gain: float = 1.0) -> torch.Tensor:
    """One bf16 tensor of i.i.d. N(0, gain^2) values, drawn on the CPU."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if gain != 1.0:
        x = x * gain
    return x.to(torch.bfloat16)


def make_inputs(B: int, H: int, S: int, D: int, gain: float = 1.0, seed: int = SEED):
    """Q, K, V, dO as contiguous bf16 CPU tensors of shape [B, H, S, D]."""
    shape = (B, H, S, D)
    return tuple(draw(shape, seed + i, gain) for i in range(4))


def make_workload_inputs(w: Workload, seed: int = SEED):
    return make_inputs(w.B, w.H, w.S, w.D, w.gain, seed)


# The pages' sweep (DASH paper write-up, experimental setup paragraph): the total
# token count fixed at 16384, sequence lengths 512 to 16384 (batch = 16384 / S),
# hidden size 2048 with head dimension 64 or 128 (so 32 or 16 heads), both masks.
PAGES_SWEEP_TOKENS = 16384
PAGES_SWEEP_HIDDEN = 2048
PAGES_SWEEP_S = (512, 1024, 2048, 4096, 8192, 16384)


def pages_sweep():
    """The pages' sweep as workloads named ``sweep_{full|causal}_s{S}_d{D}``, tile 128."""
    out = []
    for causal in (False, True):
        for D in (64, 128):
            for S in PAGES_SWEEP_S:
                B, H = PAGES_SWEEP_TOKENS // S, PAGES_SWEEP_HIDDEN // D
                name = f"sweep_{'causal' if causal else 'full'}_s{S}_d{D}"
                out.append(Workload(name, B, H, S, D, causal, 128, 1.0, _valid(causal, ALL_SCHEDULES)))
    return out
