"""CPU oracle of the W4A16 routed-expert MoE layer -- TEST INFRASTRUCTURE ONLY.

Plain, slow, float64 numpy restatement of what the layer computes.  Only the
test suite, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference
leg of ``bench.py`` may import it; the library never does, and it shares no
code, tables or helpers with the CUDA path.

Sources (Horizon RunMap pages):
  * "Horizon RunMap - architecture", section "Representation and computation":
    routed experts are INT4 "qpacked" with 256-value blocks and FP16 scales;
    activations are FP16; no persistent expanded expert.
  * Landing page (/en), section "08 / Precision & quality": kernels convert
    compact weights during computation, with FP32 accumulation stages and
    explicit rounding; routing stays outside INT4.
  * Landing page (/en), section "06 / Follow a token": routing selects the
    experts of each routed layer.
The pages fix no nibble order, sign convention, activation function, router
rule or rounding point.  The readings taken here (and listed in the design
notes) are: signed two's-complement int4, low nibble first, w = q * s with
no zero-point, one scale per 256 consecutive K values of one output row
(the last block of a row may be short), expert FFN = down(SiLU(gate x) *
(up x)), router = softmax over all E logits (+ optional bias), top-k by the
largest logit with ties to the lower expert index, listed in descending
order, weights = the softmax entries (no renormalisation), combine summed in
rank order.

Everything here is float64 and unrounded: the oracle is the exact definition
(up to float64 rounding).  The GPU rounds at its own points; the parity
tolerances absorb that.

Parity status: every function below is pinned by tests that do not re-use its
own formula (exhaustive byte tables, hand-derived closed forms, a dense
brute-force formulation, invariants and planted-mistake checks).
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional

import numpy as np

BLOCK = 256          # K values per FP16 scale
NEAR_TIE_GAP = 1e-4  # logit gap below which a routing decision is flagged
FP16_MAX = 65504.0   # largest finite IEEE binary16 value


# ------------------------------------------------------------------ format

def unpack_int4(packed: np.ndarray) -> np.ndarray:
    """uint8 [..., K/2] -> int64 [..., K]: low nibble is the even K index,
    high nibble the odd one; each nibble is a signed two's-complement int4."""
    packed = np.asarray(packed, dtype=np.uint8)
    lo = (packed & 0x0F).astype(np.int64)
    hi = (packed >> 4).astype(np.int64)
    nib = np.stack([lo, hi], axis=-1).reshape(*packed.shape[:-1], 2 * packed.shape[-1])
    return np.where(nib >= 8, nib - 16, nib)


def pack_int4(q: np.ndarray) -> np.ndarray:
    """Inverse of unpack_int4: int values in [-8, 7], K even -> uint8 [..., K/2]."""
    q = np.asarray(q, dtype=np.int64)
    if q.shape[-1] % 2:
        raise ValueError("K must be even")
    if q.min(initial=0) < -8 or q.max(initial=0) > 7:
        raise ValueError("int4 values must lie in [-8, 7]")
    nib = (q & 0xF).astype(np.uint8)
    return (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)


def fp16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def dequantize(q_packed: np.ndarray, scale_bits: np.ndarray) -> np.ndarray:
    """Dense float64 weight [R, K] of one matrix: w[r, k] = q[r, k] * s[r, k // 256]."""
    q = unpack_int4(q_packed)
    K = q.shape[-1]
    s = fp16_bits_to_f64(scale_bits)
    if s.shape[-1] != math.ceil(K / BLOCK):
        raise ValueError("need ceil(K/256) scales per row")
    block_of_k = np.arange(K) // BLOCK
    return q.astype(np.float64) * s[..., block_of_k]


# ----------------------------------------------------------------- routing

def rms_prenorm(x: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """x / sqrt(mean_h x^2 + eps), per token, unweighted (stacked-layer reading)."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def router_logits(x: np.ndarray, router_w: np.ndarray, bias: Optional[np.ndarray]) -> np.ndarray:
    """l[t, e] = sum_h x[t, h] * W_r[e, h] (+ bias[e])."""
    l = np.asarray(x, np.float64) @ np.asarray(router_w, np.float64).T
    if bias is not None:
        l = l + np.asarray(bias, np.float64)[None, :]
    return l


def softmax(logits: np.ndarray) -> np.ndarray:
    """Softmax over the expert axis; a -inf logit gets probability 0."""
    m = np.max(logits, axis=-1, keepdims=True)
    z = np.exp(logits - m)
    return z / np.sum(z, axis=-1, keepdims=True)


def topk_ids(logits: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest logits per token, largest first, equal logits
    ordered by lower expert index (a stable sort of the negated logits)."""
    order = np.argsort(-logits, axis=-1, kind="stable")
    return order[:, :k].astype(np.int64)


def route(x: np.ndarray, router_w: np.ndarray, bias: Optional[np.ndarray], k: int):
    """Returns (logits, probs, ids [T,k], weights [T,k]); weights = probs[ids]."""
    logits = router_logits(x, router_w, bias)
    probs = softmax(logits)
    ids = topk_ids(logits, k)
    w = np.take_along_axis(probs, ids, axis=-1)
    return logits, probs, ids, w


def near_tie_flags(logits: np.ndarray, k: int, gap: float = NEAR_TIE_GAP) -> np.ndarray:
    """True for tokens whose routing may legitimately differ between float
    orders: some adjacent gap among the k+1 largest logits is below `gap`."""
    s = -np.sort(-logits, axis=-1)[:, : k + 1]
    d = s[:, :-1] - s[:, 1:]
    with np.errstate(invalid="ignore"):
        return np.any(d < gap, axis=-1)


# ------------------------------------------------------------- permutation

@dataclass
class Permutation:
    counts: np.ndarray          # [E] pairs per expert
    offsets: np.ndarray         # [E+1] exclusive prefix sum of counts
    sorted_pairs: np.ndarray    # [P] flat pair index p = t*k + j at sorted row r
    pair_to_row: np.ndarray     # [P] inverse of sorted_pairs


def permutation(ids: np.ndarray, num_experts: int) -> Permutation:
    """Pairs grouped by expert (ascending), and inside a group by flat pair
    index p = t*k + j (ascending)."""
    flat = np.asarray(ids, np.int64).reshape(-1)
    P = flat.size
    counts = np.bincount(flat, minlength=num_experts).astype(np.int64)
    offsets = np.zeros(num_experts + 1, np.int64)
    offsets[1:] = np.cumsum(counts)
    sorted_pairs = np.empty(P, np.int64)
    fill = offsets[:-1].copy()
    for p in range(P):
        e = flat[p]
        sorted_pairs[fill[e]] = p
        fill[e] += 1
    pair_to_row = np.empty(P, np.int64)
    pair_to_row[sorted_pairs] = np.arange(P)
    return Permutation(counts, offsets, sorted_pairs, pair_to_row)


# ------------------------------------------------------------------ expert

def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def expert_ffn(x_rows: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray, w_down: np.ndarray) -> np.ndarray:
    """y = W_d (SiLU(W_g x) * (W_u x)) for each row x of x_rows [M, H]."""
    g = x_rows @ w_gate.T
    u = x_rows @ w_up.T
    h = silu(g) * u
    return h @ w_down.T


# ------------------------------------------------------------------- layer

FLAG_RESIDUAL = 1
FLAG_PRENORM = 2


@dataclass
class LayerResult:
    out: np.ndarray             # [T, H] float64
    logits: np.ndarray          # [T, E]
    ids: np.ndarray             # [T, k]
    weights: np.ndarray         # [T, k]
    perm: Permutation
    near_tie: np.ndarray        # [T] bool
    overflow: np.ndarray        # [T, H] bool: |out| > FP16_MAX (an FP16 output is +-inf there)
    y: Optional[np.ndarray] = None   # [P, H] per-pair expert outputs (pair order)


def moe_layer(x, router_w, bias, experts, k: int, flags: int = 0,
              expert_to_slot=None, keep_y: bool = False) -> LayerResult:
    """The routed-expert FFN layer for x [T, H] (fp16 values, taken exactly).

    experts: six canonical arrays (gate_q, gate_s, up_q, up_s, down_q, down_s)
    indexed by *slot*; expert_to_slot [E] maps an expert id to its slot (None
    = identity).  A routed expert without a slot contributes 0.
    out[t] = (x[t] if RESIDUAL) + sum_j w[t, j] * y[t*k + j] summed in j order.
    With PRENORM the router and experts see x / rms(x); the residual stays x.
    overflow flags the outputs whose magnitude is beyond the largest finite
    FP16 value, where an FP16 result rounds to +-inf.
    """
    gq, gs, uq, us, dq, ds = experts
    x0 = np.asarray(x, np.float64)
    T, H = x0.shape
    E = router_w.shape[0]
    xin = rms_prenorm(x0) if flags & FLAG_PRENORM else x0
    logits, probs, ids, w = route(xin, router_w, bias, k)
    perm = permutation(ids, E)
    y = np.zeros((T * k, H), np.float64)
    for e in range(E):
        rows = perm.sorted_pairs[perm.offsets[e]:perm.offsets[e + 1]]
        if rows.size == 0:
            continue
        slot = e if expert_to_slot is None else int(expert_to_slot[e])
        if slot < 0:
            continue
        Wg = dequantize(gq[slot], gs[slot])
        Wu = dequantize(uq[slot], us[slot])
        Wd = dequantize(dq[slot], ds[slot])
        y[rows] = expert_ffn(xin[rows // k], Wg, Wu, Wd)
    out = x0.copy() if flags & FLAG_RESIDUAL else np.zeros_like(x0)
    for j in range(k):
        out += w[:, j:j + 1] * y[np.arange(T) * k + j]
    return LayerResult(out, logits, ids, w, perm, near_tie_flags(logits, k),
                       np.abs(out) > FP16_MAX, y if keep_y else None)

