"""Seeded synthetic inputs for the W4A16 routed-expert MoE layer.

This module only draws random numbers and lays them out in the canonical
"qpacked" byte format; it holds none of the layer's arithmetic (no
unpacking, no dequantisation, no routing).  Both the CPU oracle (in tests)
and the CUDA path consume what it returns.

Canonical per-expert arrays (row-major, K contiguous):
  gate_q, up_q : uint8  [I, H/2]      two signed int4 values per byte
  gate_s, up_s : uint16 [I, ceil(H/256)]  IEEE fp16 bit patterns
  down_q       : uint8  [H, I/2]
  down_s       : uint16 [H, ceil(I/256)]
Drawing every packed byte uniformly from [0, 255] makes each nibble
independently uniform over its 16 codes, i.e. every int4 value is uniform
over [-8, 7] whatever nibble order or sign convention a reader uses.

Distributions (the workloads of the Horizon RunMap campaign, re-shaped to
one layer): activations x ~ N(0, 1) rounded to fp16; router weight
~ N(0, 0.02) rounded to fp16; scales ~ U[0.002, 0.02] rounded to fp16.

Seeds: a weight stream PCG64(seed) draws, in this order, the router weight,
then for each expert e = 0..E-1 gate_q, gate_s, up_q, up_s, down_q, down_s,
then the logit bias (when the workload has one), then the resident subset
and its slot permutation (partial residency only).  Activations come from a
separate stream PCG64(SeedSequence([seed, T])) so that the same weights serve
every token count.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

BLOCK = 256


@dataclasses.dataclass(frozen=True)
class LayerShape:
    hidden: int
    inter: int
    num_experts: int
    top_k: int

    @property
    def nb_h(self) -> int:
        return math.ceil(self.hidden / BLOCK)

    @property
    def nb_i(self) -> int:
        return math.ceil(self.inter / BLOCK)

    def packed_bytes_per_expert(self) -> int:
        """int4 bytes + fp16 scale bytes of one expert (gate + up + down)."""
        H, I = self.hidden, self.inter
        q = 3 * I * H // 2
        s = 2 * (2 * I * self.nb_h + H * self.nb_i)
        return q + s


TINY = LayerShape(hidden=256, inter=128, num_experts=8, top_k=2)
OLMOE = LayerShape(hidden=2048, inter=1024, num_experts=64, top_k=8)
QWEN = LayerShape(hidden=2048, inter=1408, num_experts=60, top_k=4)

# Seeds of the named workloads: 1000 + workload id + 100 * variant.
SEED_TINY = 1000
SEED_OLMOE_DECODE = 1001
SEED_QWEN_PARTIAL = 1002
SEED_OLMOE_PREFILL = 1003          # variant 1: no bias
SEED_OLMOE_PREFILL_SKEW = 1103     # variant 2: bias ~ N(0, 1)
SEED_OLMOE_STACK = 1004
QWEN_RESIDENT = 39


@dataclasses.dataclass
class Experts:
    """Canonical qpacked arrays of n experts (leading axis = expert)."""
    gate_q: np.ndarray
    gate_s: np.ndarray
    up_q: np.ndarray
    up_s: np.ndarray
    down_q: np.ndarray
    down_s: np.ndarray

    def select(self, idx) -> "Experts":
        idx = np.asarray(idx)
        return Experts(*(np.ascontiguousarray(a[idx]) for a in dataclasses.astuple(self)))

    def arrays(self):
        return dataclasses.astuple(self)


@dataclasses.dataclass
class Layer:
    shape: LayerShape
    router_w: np.ndarray            # fp16 [E, H]
    experts: Experts                 # all E experts, canonical layout
    bias: Optional[np.ndarray]       # fp32 [E] or None
    expert_to_slot: np.ndarray       # int32 [E], -1 = not resident
    num_slots: int

    def slot_experts(self) -> Experts:
        """Experts in slot order: slot s holds expert slot_to_expert[s]."""
        s2e = np.full(self.num_slots, -1, np.int64)
        for e, s in enumerate(self.expert_to_slot):
            if s >= 0:
                s2e[s] = e
        assert (s2e >= 0).all()
        return self.experts.select(s2e)


def _scales(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.uniform(0.002, 0.02, size=shape).astype(np.float16).view(np.uint16)


def _bytes(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.integers(0, 256, size=shape, dtype=np.uint8)


def draw_experts(rng: np.random.Generator, shape: LayerShape, n: int) -> Experts:
    H, I = shape.hidden, shape.inter
    gq = np.empty((n, I, H // 2), np.uint8)
    gs = np.empty((n, I, shape.nb_h), np.uint16)
    uq = np.empty_like(gq)
    us = np.empty_like(gs)
    dq = np.empty((n, H, I // 2), np.uint8)
    ds = np.empty((n, H, shape.nb_i), np.uint16)
    for e in range(n):
        gq[e] = _bytes(rng, gq.shape[1:])
        gs[e] = _scales(rng, gs.shape[1:])
        uq[e] = _bytes(rng, uq.shape[1:])
        us[e] = _scales(rng, us.shape[1:])
        dq[e] = _bytes(rng, dq.shape[1:])
        ds[e] = _scales(rng, ds.shape[1:])
    return Experts(gq, gs, uq, us, dq, ds)


def draw_x(seed: int, T: int, hidden: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, T])))
    return rng.standard_normal((T, hidden)).astype(np.float16)


def make_layer(shape: LayerShape, seed: int, *, bias_sigma: Optional[float] = None,
               num_resident: Optional[int] = None, rng: Optional[np.random.Generator] = None) -> Layer:
    """One layer's weights.  bias_sigma draws a per-expert N(0, sigma) logit
    bias; num_resident < E draws a resident subset at permuted slot indices
    and sets the logit bias of every absent expert to -inf."""
    if rng is None:
        rng = np.random.Generator(np.random.PCG64(seed))
    E = shape.num_experts
    router_w = (rng.standard_normal((E, shape.hidden)) * 0.02).astype(np.float16)
    experts = draw_experts(rng, shape, E)
    bias = None
    if bias_sigma is not None:
        bias = (rng.standard_normal(E) * bias_sigma).astype(np.float32)
    if num_resident is None or num_resident >= E:
        e2s = np.arange(E, dtype=np.int32)
        nslots = E
    else:
        resident = np.sort(rng.choice(E, size=num_resident, replace=False))
        slots = rng.permutation(num_resident)
        e2s = np.full(E, -1, np.int32)
        e2s[resident] = slots.astype(np.int32)
        nslots = num_resident
        if bias is None:
            bias = np.zeros(E, np.float32)
        bias[e2s < 0] = -np.inf
    return Layer(shape, router_w, experts, bias, e2s, nslots)


# ---------------------------------------------------------------- workloads

def tiny_layer() -> Layer:
    return make_layer(TINY, SEED_TINY)


def olmoe_decode_layer() -> Layer:
    return make_layer(OLMOE, SEED_OLMOE_DECODE)


def qwen_partial_layer() -> Layer:
    return make_layer(QWEN, SEED_QWEN_PARTIAL, num_resident=QWEN_RESIDENT)


def olmoe_prefill_layer(variant: int = 1) -> Layer:
    if variant == 1:
        return make_layer(OLMOE, SEED_OLMOE_PREFILL)
    return make_layer(OLMOE, SEED_OLMOE_PREFILL_SKEW, bias_sigma=1.0)


def olmoe_stack(num_layers: int = 16):
    """Independent OLMoE-shaped layers drawn one after another from one stream."""
    rng = np.random.Generator(np.random.PCG64(SEED_OLMOE_STACK))
    return [make_layer(OLMOE, SEED_OLMOE_STACK, rng=rng) for _ in range(num_layers)]


def device_random_experts(shape: LayerShape, n: int, seed: int, device):
    """Same distributions as draw_experts, drawn on a CUDA device with a seeded
    torch generator (for throughput runs whose weight sets are too large to
    draw on the host in reasonable time).  Returns canonical torch tensors."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    H, I = shape.hidden, shape.inter

    def qb(*s):
        return torch.randint(0, 256, s, dtype=torch.uint8, device=device, generator=g)

    def sc(*s):
        v = torch.rand(s, device=device, generator=g, dtype=torch.float32) * 0.018 + 0.002
        return v.to(torch.float16).view(torch.int16)

    return (qb(n, I, H // 2), sc(n, I, shape.nb_h), qb(n, I, H // 2), sc(n, I, shape.nb_h),
            qb(n, H, I // 2), sc(n, H, shape.nb_i))
