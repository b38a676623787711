"""The synthetic workloads: layer shapes, replica counts, step counts, seeds and
gradient distributions of the five benchmark configurations, as input recipes
(no optimizer arithmetic here).

Layer shapes are the decoder layers of the Qwen3 family that the SlideDP page
fine-tunes (its Results section), flattened and concatenated per unit in the
order q, k, v, o, gate, up, down, norm1, norm2.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import numpy as np

from . import GRAD_NORMAL, GRAD_STUDENT3, TAG_SCALE, uniform


def decoder_layer(h: int, kv: int, ffn: int, norms: bool = True) -> List[Tuple[str, int]]:
    t = [("q", h * h), ("k", h * kv), ("v", h * kv), ("o", h * h),
         ("gate", h * ffn), ("up", h * ffn), ("down", ffn * h)]
    if norms:
        t += [("norm1", h), ("norm2", h)]
    return t


def h2560_layer():
    # q 2560x4096 and o 4096x2560 (32 heads x 128), k/v 2560x1024, SwiGLU 9728
    return [("q", 2560 * 4096), ("k", 2560 * 1024), ("v", 2560 * 1024), ("o", 4096 * 2560),
            ("gate", 2560 * 9728), ("up", 2560 * 9728), ("down", 9728 * 2560),
            ("norm1", 2560), ("norm2", 2560)]


def h5120_layer():
    return decoder_layer(5120, 1024, 17408)


def h8192_layer():
    return decoder_layer(8192, 1024, 29568)


@dataclass
class Unit:
    name: str
    tensors: List[Tuple[str, int]]

    @property
    def numel(self) -> int:
        return sum(n for _, n in self.tensors)

    def segments(self):
        """(offset, length) of each tensor inside the unit's flat vector."""
        out, off = [], 0
        for _, n in self.tensors:
            out.append((off, n))
            off += n
        return out


@dataclass
class Workload:
    name: str
    units: List[Unit]
    R: int
    steps: int
    seed: int
    max_grad_norm: float = 0.0
    prewarm_steps: int = 0
    grad_kind: int = GRAD_NORMAL
    grad_scale: float = 1e-3
    per_tensor_scale: bool = False       # log-uniform sigma per tensor in [1e-5, 1e-2]
    zero_prob: float = 0.0
    streamed: bool = False
    master_scale: float = 0.02
    fp32_grads: bool = False             # FP32 gradient replicas instead of BF16
    lr: float = 1e-5
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    description: str = ""

    @property
    def numel(self) -> int:
        return sum(u.numel for u in self.units)

    def tensor_scales(self, unit_index: int) -> List[float]:
        """FP32 gradient scale of each tensor of a unit."""
        u = self.units[unit_index]
        if not self.per_tensor_scale:
            return [float(np.float32(self.grad_scale))] * len(u.tensors)
        out = []
        for k in range(len(u.tensors)):
            x = uniform(self.seed, TAG_SCALE, unit_index, 0, 0, k)   # (0, 1]
            out.append(float(np.float32(10.0 ** (-5.0 + 3.0 * float(x)))))
        return out

    def hparams_tuple(self):
        return (self.lr, self.beta1, self.beta2, self.eps, self.weight_decay, self.max_grad_norm)


def h2560_r1() -> Workload:
    return Workload("h2560_R1", [Unit("layer", h2560_layer())], R=1, steps=3, seed=0,
                    description="one h=2560 decoder layer (100,930,560 params), R=1, 3 AdamW steps")


def h2560_r4_clip() -> Workload:
    return Workload("h2560_R4_clip", [Unit("layer", h2560_layer())], R=4, steps=10, seed=1,
                    max_grad_norm=1.0, prewarm_steps=5,
                    description="one h=2560 decoder layer, R=4 replicas averaged in-kernel, "
                                "global grad-norm clip 1.0, m/v pre-warmed by 5 oracle steps, "
                                "then 10 steps")


def h5120_r8_logscale() -> Workload:
    return Workload("h5120_R8_logscale", [Unit("layer", h5120_layer())], R=8, steps=20, seed=2,
                    per_tensor_scale=True,
                    description="one h=5120 decoder layer (330,311,680 params), R=8, per-tensor "
                                "gradient scale log-uniform in [1e-5, 1e-2], 20 steps")


def h5120x40_streamed() -> Workload:
    units = ([Unit("embed", [("embed", 152064 * 5120)])]
             + [Unit(f"layer{i}", h5120_layer()) for i in range(40)]
             + [Unit("head", [("head", 152064 * 5120)])])
    return Workload("h5120x40_streamed", units, R=4, steps=2, seed=3, streamed=True,
                    description="40 h=5120 layers + 152064x5120 embedding and head "
                                "(14,769,602,560 params), host-resident, 2-unit HBM window, R=4")


def h8192x8_streamed() -> Workload:
    units = [Unit(f"layer{i}", h8192_layer()) for i in range(8)]
    return Workload("h8192x8_streamed", units, R=8, steps=2, seed=4, streamed=True,
                    grad_kind=GRAD_STUDENT3, zero_prob=0.001,
                    description="8 h=8192 layers (7,021,395,968 params), host-resident, "
                                "2-unit HBM window, R=8, Student-t(3) gradients x 1e-3 with "
                                "0.1% exact zeros")


def h2560_r4_clip_fp32grads() -> Workload:
    w = h2560_r4_clip()
    w.name = "h2560_R4_clip_fp32grads"
    w.fp32_grads = True
    w.description = ("the h=2560 R=4 clipped layer with FP32 gradient replicas (FP32 gradient accumulation): "
                     "26 + 4R bytes per parameter")
    return w


ALL = {f().name: f for f in (h2560_r1, h2560_r4_clip, h5120_r8_logscale, h5120x40_streamed, h8192x8_streamed,
                             h2560_r4_clip_fp32grads)}
HBM_RESIDENT = ("h2560_R1", "h2560_R4_clip", "h5120_R8_logscale")
STREAMED = ("h8192x8_streamed", "h5120x40_streamed")
