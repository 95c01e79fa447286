"""The synthetic workloads: parameter shape lists and optimizer settings.

Shape lists only -- no weights or data.  Each workload is a model's list of
parameter tensors in module order, the number of emulated data-parallel ranks,
the ZeRO stage, the 16-bit gradient format, the gradient distribution and the
optimizer settings.  Where a workload leaves a setting open the tiny flat
model's settings carry over: lr 1e-3, betas (0.9, 0.999), eps 1e-8, master
weights N(0, 0.02), seed 0, no weight decay.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence, Tuple

FP16, BF16 = 0, 1


@dataclasses.dataclass
class Workload:
    name: str
    shapes: List[Tuple[int, ...]]
    nd: int
    stage: int
    dtype: int
    grad_sigma: float
    loss_scale: float = 1.0
    dynamic_scale: int = 0
    clip: float = 0.0
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    decoupled_wd: int = 1
    steps: int = 1
    inf_steps: Tuple[int, ...] = ()
    units: Optional[List[int]] = None      # stage 3: unit index of each tensor
    master_sigma: float = 0.02
    seed: int = 0

    @property
    def psi(self) -> int:
        return sum(math.prod(s) for s in self.shapes)

    def hparams(self) -> dict:
        return dict(lr=self.lr, beta1=self.beta1, beta2=self.beta2, eps=self.eps,
                    weight_decay=self.weight_decay, decoupled_wd=self.decoupled_wd,
                    clip_norm=self.clip, loss_scale=self.loss_scale,
                    dynamic_scale=self.dynamic_scale, backoff=0.5, growth_interval=1000)

    def unit_lengths(self) -> List[int]:
        assert self.units is not None
        lens = [0] * (max(self.units) + 1)
        for s, u in zip(self.shapes, self.units):
            lens[u] += math.prod(s)
        return lens


def gpt2_shapes(layers: int, h: int, ffn: int, vocab: int, ctx: int) -> List[Tuple[int, ...]]:
    """GPT-2 parameter list in module order (tied output head)."""
    shapes: List[Tuple[int, ...]] = [(vocab, h), (ctx, h)]
    for _ in range(layers):
        shapes += [(h,), (h,),                  # ln_1 weight, bias
                   (h, 3 * h), (3 * h,),        # attn.c_attn
                   (h, h), (h,),                # attn.c_proj
                   (h,), (h,),                  # ln_2
                   (h, ffn), (ffn,),            # mlp.c_fc
                   (ffn, h), (h,)]              # mlp.c_proj
    shapes += [(h,), (h,)]                      # ln_f
    return shapes


def llama_shapes(layers: int, h: int, ffn: int, q_heads: int, kv_heads: int,
                 vocab: int) -> Tuple[List[Tuple[int, ...]], List[int]]:
    """LLaMA parameter list (untied head) and its ZeRO-3 units: the embedding,
    one unit per transformer layer, and the final norm with the head."""
    hd = h // q_heads
    kv = kv_heads * hd
    shapes: List[Tuple[int, ...]] = [(vocab, h)]
    units = [0]
    for layer in range(layers):
        shapes += [(h, h), (kv, h), (kv, h), (h, h),          # q, k, v, o
                   (ffn, h), (ffn, h), (h, ffn),              # gate, up, down
                   (h,), (h,)]                                # the two RMSNorms
        units += [layer + 1] * 9
    shapes += [(h,), (vocab, h)]
    units += [layers + 1] * 2
    return shapes, units


def tiny() -> Workload:
    return Workload("tiny-flat-4t", [(512, 1024), (1024,), (1024, 512), (512,)], nd=4, stage=2,
                    dtype=FP16, grad_sigma=1e-3, loss_scale=1024.0, dynamic_scale=1, steps=3)


def gpt2_small() -> Workload:
    return Workload("gpt2-small", gpt2_shapes(12, 768, 3072, 50257, 1024), nd=8, stage=1,
                    dtype=BF16, grad_sigma=1e-2, clip=1.0, weight_decay=0.01, decoupled_wd=1,
                    steps=10)


def gpt2_xl() -> Workload:
    return Workload("gpt2-1.5b", gpt2_shapes(48, 1600, 6400, 50257, 1024), nd=16, stage=2,
                    dtype=FP16, grad_sigma=1e-3, loss_scale=65536.0, dynamic_scale=1, clip=1.0,
                    steps=10, inf_steps=(3, 7))


def llama3_8b() -> Workload:
    shapes, units = llama_shapes(32, 4096, 14336, 32, 8, 128256)
    return Workload("llama3-8b", shapes, nd=64, stage=3, dtype=BF16, grad_sigma=1e-2,
                    steps=1, units=units)


SWEEP_PSI = (1 << 20, 1 << 24, 1 << 28, 1 << 30, 1 << 31)
SWEEP_ND = (1, 2, 8, 32)


def sweep(psi: int, nd: int) -> Workload:
    return Workload(f"flat-{psi}-nd{nd}", [(psi,)], nd=nd, stage=2, dtype=BF16, grad_sigma=1e-2,
                    steps=6)


def scaled_gpt2(layers: int, h: int, ffn: int, vocab: int, ctx: int, nd: int,
                base: Workload) -> Workload:
    """A smaller model of the same family and settings, for parity at sizes the
    oracle finishes in seconds."""
    return dataclasses.replace(base, name=f"{base.name}-L{layers}h{h}",
                               shapes=gpt2_shapes(layers, h, ffn, vocab, ctx), nd=nd)


def scaled_llama(layers: int, h: int, ffn: int, q: int, kv: int, vocab: int, nd: int,
                 base: Workload) -> Workload:
    shapes, units = llama_shapes(layers, h, ffn, q, kv, vocab)
    return dataclasses.replace(base, name=f"{base.name}-L{layers}h{h}", shapes=shapes,
                               units=units, nd=nd)


def flatten_dims(shapes: Sequence[Tuple[int, ...]]):
    dims, ndims = [], []
    for s in shapes:
        dims += list(s)
        ndims.append(len(s))
    return dims, ndims
