"""Seeded synthetic inputs shaped like the pages' MoE-layer workloads.

This module is the only code that the CUDA library's tests and the fp64
oracle share: it draws random numbers and lays them out, and it holds none of
the layer's arithmetic (no routing, no products, no activation).

Recipe (every draw seeded, nothing read from disk):
  * Normal draws are made in fp32 and cast round-to-nearest-even to bf16 where
    the workload is bf16.
  * Weights ~ N(0, 1/fan_in): fan_in = m for the router W_r and for W1/W3,
    fan_in = p for W2.  Activations ~ N(0, 1).  With these scales the router
    logits x.W_r are ~N(0, 1): a uniform router.
  * Skewed (Zipf) routing adds a per-expert router bias b_e = ln P(e) with
    P(e) proportional to (e + 1)^-s, expert 0 hottest, so that a few hot experts
    take most tokens (HARMOEny write-up, part 2: hot and cold experts).
  * Temporal locality: for t >= 1, with probability 0.5 the token row x_t is a
    copy of x_{t-1} (chained), so the token keeps its predecessor's expert set
    (expert-cache article, section 2.1: consecutive tokens reuse experts).
  * Paged decode trace: per (step s, layer l, sequence b) the expert pair is
    copied from (s, l-1, b) with p = 0.44 when l > 0, else copied from
    (s-1, l, b) with p = 0.5 when s > 0, else two distinct experts are drawn
    uniformly (expert-cache article, section 2.1: 44% consecutive-layer reuse,
    40-60% consecutive-token reuse).  The k weights come from two N(0,1) logits.

Two back ends draw the same distributions: ``numpy`` (PCG64, identical on
every platform; used on CPU and for small layers) and ``torch`` on a CUDA
device (Philox; used for the multi-GB layers, whose host copies are then what
both the library and the oracle read).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

try:
    import torch
except ImportError:  # the oracle-only tests do not need torch
    torch = None

RELU2, SWIGLU = "relu2", "swiglu"


@dataclasses.dataclass(frozen=True)
class LayerShape:
    """Shape and numeric types of one MoE FFN layer."""
    name: str
    m: int            # hidden size
    p: int            # expert FFN size
    E: int            # experts
    k: int            # experts per token
    expert: str       # RELU2 (x.W1 -> ReLU -> .W2) or SWIGLU (W1 gate, W3 up, W2 down)
    act: str          # "f32" | "bf16": activations and router weights
    weight: str       # "f32" | "bf16" | "i8": expert weights ("i8" is quantised from bf16)
    zipf_s: Optional[float] = None   # router bias making popularity Zipf(s)

    @property
    def has_w3(self) -> bool:
        return self.expert == SWIGLU

    def with_weight(self, weight: str) -> "LayerShape":
        return dataclasses.replace(self, weight=weight, name=f"{self.name}-{weight}")

    def with_zipf(self, s: float) -> "LayerShape":
        return dataclasses.replace(self, zipf_s=s, name=f"{self.name}-zipf{s}")


# The workloads the pages speak of (model shapes of the expert-cache article:
# Mixtral 8x7B with 8 experts, Phi-3.5-MoE with 16 smaller experts).
TINY_FP32 = LayerShape("tiny-fp32", m=128, p=256, E=8, k=2, expert=RELU2, act="f32", weight="f32")
MIXTRAL = LayerShape("mixtral-8x7b", m=4096, p=14336, E=8, k=2, expert=SWIGLU, act="bf16",
                     weight="bf16")
PHI35 = LayerShape("phi-3.5-moe", m=4096, p=6400, E=16, k=2, expert=SWIGLU, act="bf16",
                   weight="bf16")

DECODE_TOKENS = (1, 4, 16, 64)
BATCH_TOKENS = (512, 2048, 8192)
PHI_TOKENS = (1, 8, 64, 512, 4096)


def zipf_bias(E: int, s: float) -> np.ndarray:
    """b_e = ln P(e), P(e) proportional to (e+1)^-s (expert 0 hottest), as the
    fp32 values both the library and the oracle receive."""
    w = np.array([(e + 1.0) ** (-s) for e in range(E)], dtype=np.float64)
    return np.log(w / w.sum()).astype(np.float32)


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream])))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even) and return the 16-bit patterns."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    rounding = ((u >> 16) & 1) + 0x7FFF
    return ((u + rounding) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class Layer:
    """Host copies of one layer's parameters, exactly as both sides receive them.

    Arrays are row-major numpy arrays: float32, or uint16 bf16 bit patterns.
    w1/w3 are lists of E (m x p) matrices, w2 a list of E (p x m) matrices.
    For int8 layers these are the bf16 originals; the library and the oracle
    each quantise them with their own code.
    """
    shape: LayerShape
    w_router: np.ndarray
    b_router: Optional[np.ndarray]
    w1: list
    w2: list
    w3: Optional[list]


def _normal_np(rng, shape, std, dtype):
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a if dtype == "f32" else f32_to_bf16_bits(a)


def _normal_torch(gen, shape, std, dtype, device):
    t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if dtype == "f32":
        return t.cpu().numpy()
    return t.to(torch.bfloat16).view(torch.int16).cpu().numpy().view(np.uint16)


def make_layer(shape: LayerShape, seed: int = 0, device: str = "cpu") -> Layer:
    """Draw one layer's router and expert weights.

    device="cpu" draws with numpy PCG64; a CUDA device draws with torch's
    Philox generator on that device (fast for multi-GB layers) and copies the
    result to the host.
    """
    wdt = "bf16" if shape.weight == "i8" else shape.weight
    m, p, E = shape.m, shape.p, shape.E
    if device == "cpu":
        draw = lambda stream, shp, std, dt: _normal_np(_rng(seed, stream), shp, std, dt)
    else:
        def draw(stream, shp, std, dt):
            g = torch.Generator(device=device)
            g.manual_seed(seed * 1000003 + stream)
            return _normal_torch(g, shp, std, dt, device)
    w_router = draw(1, (m, E), 1.0 / math.sqrt(m), shape.act)
    b_router = zipf_bias(E, shape.zipf_s) if shape.zipf_s is not None else None
    w1, w2, w3 = [], [], []
    for e in range(E):
        w1.append(draw(100 + 3 * e, (m, p), 1.0 / math.sqrt(m), wdt))
        if shape.has_w3:
            w3.append(draw(101 + 3 * e, (m, p), 1.0 / math.sqrt(m), wdt))
        w2.append(draw(102 + 3 * e, (p, m), 1.0 / math.sqrt(p), wdt))
    return Layer(shape, w_router, b_router, w1, w2, w3 if shape.has_w3 else None)


def make_tokens(shape: LayerShape, T: int, seed: int = 0, locality: float = 0.0,
                device: str = "cpu") -> np.ndarray:
    """Token activations x [T, m] ~ N(0, 1) in the layer's activation type.

    locality > 0: for t >= 1, with that probability row t copies row t-1."""
    if device == "cpu":
        x = _normal_np(_rng(seed, 7 + T), (T, shape.m), 1.0, shape.act)
    else:
        g = torch.Generator(device=device)
        g.manual_seed(seed * 1000003 + 7 + T)
        x = _normal_torch(g, (T, shape.m), 1.0, shape.act, device)
    if locality > 0.0 and T > 1:
        coin = _rng(seed, 8 + T).random(T)
        for t in range(1, T):
            if coin[t] < locality:
                x[t] = x[t - 1]
    return x


def make_topk_trace(E: int, k: int, steps: int, layers: int, batch: int, seed: int = 0,
                    p_layer: float = 0.44, p_token: float = 0.5):
    """Seeded routing trace for the paged decode run.

    Returns (ids [steps, layers, batch, k] int32, weights [steps, layers, batch, k]
    float32).  Within a row the ids are distinct and in no particular order;
    weights are a softmax of k N(0,1) logits, largest first.
    """
    rng = _rng(seed, 11)
    ids = np.empty((steps, layers, batch, k), np.int32)
    for s in range(steps):
        for l in range(layers):
            for b in range(batch):
                if l > 0 and rng.random() < p_layer:
                    ids[s, l, b] = ids[s, l - 1, b]
                elif s > 0 and rng.random() < p_token:
                    ids[s, l, b] = ids[s - 1, l, b]
                else:
                    ids[s, l, b] = rng.choice(E, size=k, replace=False)
    logits = rng.standard_normal((steps, layers, batch, k)).astype(np.float32)
    logits = -np.sort(-logits, axis=-1)
    ex = np.exp(logits - logits[..., :1])
    weights = (ex / ex.sum(axis=-1, keepdims=True)).astype(np.float32)
    return ids, weights

