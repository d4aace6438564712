"""Seeded synthetic MoE-layer inputs shaped like the pages' models.

This module holds NO arithmetic of the reader itself: it draws weights,
activations, routing and the rotation signs, and converts fp32 draws to BF16
bit patterns.  Both the CUDA path and the fp64 oracle consume what it makes.

Value recipe (the same for every workload):
  * weights G, V (as [E][I][H]) and D (as [E][H][I]): BF16 of N(0, 1/H), each
    entry independently multiplied by 10 with probability 0.001;
  * x: fp32 N(0, 1) with 4 fixed outlier coordinates (drawn from the seed)
    multiplied by 20;
  * router logits N(0, 1) per token; the topk largest are routed and the
    routing weights are the softmax renormalised over the chosen experts;
  * rotation signs sigma: independent +-1 per padded hidden coordinate.

Layer shapes follow the model table of the expert-prefetching page
("Speculating Experts Accelerates Inference for Mixture-of-Experts", model
configuration table): Qwen3-30B-A3B (E 128, H 2048, I 768, top-8),
Qwen3-235B-A22B (E 128, H 4096, I 1536, top-8), GPT-OSS-120B (E 32, H 2880,
I 2880, top-4).  Trained weights are not used anywhere.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

OUTLIER_P = 0.001
OUTLIER_W = 10.0
X_OUTLIERS = 4
X_OUTLIER_SCALE = 20.0

# Read shares of the two overhead parts at the 17.8% budget (sketch 4.9% +
# recovery 0.6% of the dense routed reads); the rest of a budget buys exact
# channels, each costing 1/N of the dense reads.
OVERHEAD_SHARE = 0.049 + 0.006


@dataclass(frozen=True)
class Workload:
    name: str
    H: int
    E: int
    topk: int
    I: int
    c: int
    r: int
    k: int
    batches: tuple
    seed: int = 0

    @property
    def Hp(self) -> int:
        return 128 * math.ceil(self.H / 128)

    @property
    def N(self) -> int:
        return self.topk * self.I


def budget_to_k(budget: float, N: int) -> int:
    """Exact-channel count for a read budget (fraction of dense routed reads)."""
    return int(round((budget - OVERHEAD_SHARE) * N))


TINY = Workload("tiny", H=256, E=16, topk=2, I=128, c=80, r=8, k=32, batches=(1,))
QWEN3_30B = Workload("qwen3_30b_a3b_layer", H=2048, E=128, topk=8, I=768, c=80, r=32,
                     k=budget_to_k(0.178, 8 * 768), batches=(1, 4, 8, 16))
QWEN3_30B_LOW = Workload("qwen3_30b_a3b_layer_12.8", H=2048, E=128, topk=8, I=768, c=80, r=32,
                         k=budget_to_k(0.128, 8 * 768), batches=(1, 8))
QWEN3_235B = Workload("qwen3_235b_a22b_layer", H=4096, E=128, topk=8, I=1536, c=80, r=32,
                      k=budget_to_k(0.128, 8 * 1536), batches=(1, 4, 8, 16))
GPT_OSS_120B = Workload("gpt_oss_120b_layer", H=2880, E=32, topk=4, I=2880, c=80, r=32,
                        k=budget_to_k(0.178, 4 * 2880), batches=(1, 16, 64, 128))
WORKLOADS = {w.name: w for w in (TINY, QWEN3_30B, QWEN3_30B_LOW, QWEN3_235B, GPT_OSS_120B)}


# --------------------------------------------------------------------------
# numpy (host) generators: PCG64, platform independent
# --------------------------------------------------------------------------
def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> BF16, returned as uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounding = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + rounding) >> 16).astype(np.uint16)


def _weight_draw(rng, shape, H):
    w = rng.standard_normal(shape, dtype=np.float32) / np.float32(math.sqrt(H))
    out = rng.random(shape, dtype=np.float32) < OUTLIER_P
    w[out] *= np.float32(OUTLIER_W)
    return f32_to_bf16_bits(w)


def weights(seed: int, E: int, I: int, H: int):
    """(G, V, D) as BF16 bit patterns: G, V uint16 [E][I][H]; D uint16 [E][H][I]."""
    rng = np.random.Generator(np.random.PCG64([seed, 1]))
    G = _weight_draw(rng, (E, I, H), H)
    V = _weight_draw(rng, (E, I, H), H)
    D = _weight_draw(rng, (E, H, I), H)
    return G, V, D


def activations(seed: int, B: int, H: int) -> np.ndarray:
    """x float32 [B][H]: N(0,1) with 4 seeded outlier coordinates x20."""
    rng = np.random.Generator(np.random.PCG64([seed, 2]))
    x = rng.standard_normal((B, H), dtype=np.float32)
    cols = rng.choice(H, size=min(X_OUTLIERS, H), replace=False)
    x[:, cols] *= np.float32(X_OUTLIER_SCALE)
    return x


def routing(seed: int, B: int, E: int, topk: int):
    """(ids int32 [B][topk], w float32 [B][topk]) from N(0,1) router logits.

    Experts are ordered by decreasing logit (ties to the lower id); weights are
    the softmax over the chosen logits only."""
    rng = np.random.Generator(np.random.PCG64([seed, 3]))
    logits = rng.standard_normal((B, E))
    ids = np.zeros((B, topk), np.int32)
    w = np.zeros((B, topk), np.float32)
    for t in range(B):
        order = np.lexsort((np.arange(E), -logits[t]))[:topk]
        ids[t] = order
        z = logits[t, order] - logits[t, order].max()
        ez = np.exp(z)
        w[t] = (ez / ez.sum()).astype(np.float32)
    return ids, w


def signs(seed: int, Hp: int) -> np.ndarray:
    """Rotation signs sigma int8 [Hp], each +1 or -1."""
    rng = np.random.Generator(np.random.PCG64([seed, 4]))
    return np.where(rng.random(Hp) < 0.5, -1, 1).astype(np.int8)


# --------------------------------------------------------------------------
# torch (device) weight generator for layers too large to draw on the host
# --------------------------------------------------------------------------
def weights_device(seed: int, E: int, I: int, H: int, device):
    """(G, V, D) as torch.bfloat16 tensors drawn on `device` (same recipe;
    different random stream from `weights`)."""
    import torch

    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed) * 7919 + 17)

    def draw(shape):
        w = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        w.mul_(1.0 / math.sqrt(H))
        out = torch.rand(shape, generator=gen, device=device) < OUTLIER_P
        w[out] *= OUTLIER_W
        return w.to(torch.bfloat16)

    return draw((E, I, H)), draw((E, I, H)), draw((E, H, I))


def bf16_tensor_to_bits(t) -> np.ndarray:
    """Host uint16 bit patterns of a torch.bfloat16 tensor."""
    import torch

    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
