"""Seeded synthetic inputs for the routed-expert MoE block.

This module is the one thing the oracle and the CUDA path share: it draws
random bytes and numbers and hands the same arrays to both.  It holds none of
the method's arithmetic (no decoding, routing, GEMV or rounding of results).

Every tensor has its own stream, addressed by (seed, layer, expert, tensor), so
any expert of any layer can be regenerated on its own without drawing the rest
of the model.  Draws follow the workloads' stated distributions:

* codes: uniform bytes (both nibbles uniform over all 16 codes);
* MXFP4 scales: E8M0 bytes uniform over [e_lo, e_hi];
* int4 scales: |N(0, sigma)| drawn in fp64 and stored as fp16 (numpy's
  round-to-nearest-even conversion);
* biases, activations, residuals: N(0, sigma) drawn in fp32 and stored as
  bfloat16 bit patterns (round-to-nearest-even on the fp32 bits);
* router logits: N(0, 1) fp32, plus an optional bias on "hot" experts.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

FMT_MXFP4 = 1
FMT_INT4 = 2

# tensor ids of the per-(layer, expert) streams
_T_GU_CODES, _T_GU_SCALES, _T_GU_BIAS, _T_DN_CODES, _T_DN_SCALES, _T_DN_BIAS = range(6)
# tensor ids of per-step streams
_T_X, _T_R, _T_LOGITS = 100, 101, 102
_T_ROUTER_W, _T_ROUTER_B = 200, 201


@dataclass(frozen=True)
class Shape:
    """Geometry and value distributions of one expert layer / stack."""
    name: str
    hidden: int
    intermediate: int
    experts: int
    top_k: int
    fmt: int = FMT_MXFP4
    group: int = 32              # 32 for MXFP4 blocks, 64 for int4 groups
    layers: int = 1
    has_bias: bool = True
    e8m0_lo: int = 119           # MXFP4 scale bytes uniform in [lo, hi]
    e8m0_hi: int = 123
    int4_scale_sigma: float = 0.02
    bias_sigma: float = 1.0
    tokens: int = 1
    seed: int = 0
    hot_experts: tuple = field(default_factory=tuple)
    hot_bias: float = 0.0

    @property
    def scale_dtype(self):
        return np.uint8 if self.fmt == FMT_MXFP4 else np.uint16

    def scales_per_row(self, K: int) -> int:
        return K // 32 if self.fmt == FMT_MXFP4 else K // self.group

    def expert_bytes(self) -> int:
        """Packed bytes of one expert: codes + scales + biases."""
        H, I = self.hidden, self.intermediate
        sb = 1 if self.fmt == FMT_MXFP4 else 2
        gu = 2 * I * (H // 2 + self.scales_per_row(H) * sb)
        dn = H * (I // 2 + self.scales_per_row(I) * sb)
        bias = (2 * I + H) * 2 if self.has_bias else 0
        return gu + dn + bias


# The workloads (sizes and distributions as stated for each).
TINY = Shape("tiny MXFP4 layer H=I=256 E=8 top-2", 256, 256, 8, 2,
             e8m0_lo=119, e8m0_hi=123, bias_sigma=0.02, seed=0)
GPTOSS_LAYER = Shape("gpt-oss-20B-shaped MXFP4 layer H=I=2880 E=32 top-4", 2880, 2880, 32, 4,
                     e8m0_lo=117, e8m0_hi=124, bias_sigma=1.0, seed=1)
GPTOSS_STACK = Shape("gpt-oss-20B-shaped 24-layer MXFP4 stack", 2880, 2880, 32, 4, layers=24,
                     e8m0_lo=117, e8m0_hi=124, bias_sigma=1.0, seed=2)
INT4_STACK = Shape("int4 48-layer stack H=2048 I=768 E=128 top-8", 2048, 768, 128, 8,
                   fmt=FMT_INT4, group=64, layers=48, has_bias=False,
                   int4_scale_sigma=0.02, seed=3)
BATCHED = Shape("batched MXFP4 layer H=I=2880 E=128 top-4 M=512", 2880, 2880, 128, 4,
                e8m0_lo=117, e8m0_hi=124, bias_sigma=1.0, tokens=512, seed=4)
BATCHED_SKEWED = Shape("batched MXFP4 layer, +2 logit bias on experts 0..7", 2880, 2880, 128, 4,
                       e8m0_lo=117, e8m0_hi=124, bias_sigma=1.0, tokens=512, seed=4,
                       hot_experts=tuple(range(8)), hot_bias=2.0)


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence(entropy=seed, spawn_key=tuple(key)))


def bf16_bits_from_f32(v: np.ndarray) -> np.ndarray:
    """fp32 -> bfloat16 bit patterns, round to nearest even (input encoding)."""
    u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def _bytes(rng: np.random.Generator, n: int) -> np.ndarray:
    return np.frombuffer(rng.bytes(n), dtype=np.uint8).copy()


@dataclass
class LayerTensors:
    """One layer, all experts, in the caller-facing packed layout:
    gu_codes [E][2I][H/2] u8, gu_scales [E][2I][H/blk], gu_bias [E][2I] bf16 bits,
    dn_codes [E][H][I/2] u8, dn_scales [E][H][I/blk], dn_bias [E][H] bf16 bits."""
    gu_codes: np.ndarray
    gu_scales: np.ndarray
    gu_bias: np.ndarray | None
    dn_codes: np.ndarray
    dn_scales: np.ndarray
    dn_bias: np.ndarray | None


def _scales(shape: Shape, rng: np.random.Generator, n: int) -> np.ndarray:
    if shape.fmt == FMT_MXFP4:
        return rng.integers(shape.e8m0_lo, shape.e8m0_hi + 1, size=n, dtype=np.uint8)
    v = np.abs(rng.normal(0.0, shape.int4_scale_sigma, size=n))
    return v.astype(np.float16).view(np.uint16)


def expert_tensors(shape: Shape, layer: int, expert: int):
    """The six tensors of one expert (no leading E axis)."""
    H, I, s = shape.hidden, shape.intermediate, shape.seed
    gu_codes = _bytes(_rng(s, layer, expert, _T_GU_CODES), 2 * I * H // 2).reshape(2 * I, H // 2)
    gu_scales = _scales(shape, _rng(s, layer, expert, _T_GU_SCALES),
                        2 * I * shape.scales_per_row(H)).reshape(2 * I, -1)
    dn_codes = _bytes(_rng(s, layer, expert, _T_DN_CODES), H * I // 2).reshape(H, I // 2)
    dn_scales = _scales(shape, _rng(s, layer, expert, _T_DN_SCALES),
                        H * shape.scales_per_row(I)).reshape(H, -1)
    if shape.has_bias:
        gu_bias = bf16_bits_from_f32(_rng(s, layer, expert, _T_GU_BIAS)
                                     .normal(0.0, shape.bias_sigma, 2 * I).astype(np.float32))
        dn_bias = bf16_bits_from_f32(_rng(s, layer, expert, _T_DN_BIAS)
                                     .normal(0.0, shape.bias_sigma, H).astype(np.float32))
    else:
        gu_bias = dn_bias = None
    return gu_codes, gu_scales, gu_bias, dn_codes, dn_scales, dn_bias


def layer_tensors(shape: Shape, layer: int = 0, experts=None) -> LayerTensors:
    """All E experts of one layer; with ``experts`` given, only those are drawn
    and the others are left zero (for a caller that reads only those)."""
    if experts is None:
        parts = [expert_tensors(shape, layer, e) for e in range(shape.experts)]

        def stackp(i):
            if parts[0][i] is None:
                return None
            return np.stack([p[i] for p in parts])

        return LayerTensors(*[stackp(i) for i in range(6)])
    H, I, E = shape.hidden, shape.intermediate, shape.experts
    sd = shape.scale_dtype
    t = LayerTensors(
        np.zeros((E, 2 * I, H // 2), np.uint8), np.zeros((E, 2 * I, shape.scales_per_row(H)), sd),
        np.zeros((E, 2 * I), np.uint16) if shape.has_bias else None,
        np.zeros((E, H, I // 2), np.uint8), np.zeros((E, H, shape.scales_per_row(I)), sd),
        np.zeros((E, H), np.uint16) if shape.has_bias else None)
    names = ("gu_codes", "gu_scales", "gu_bias", "dn_codes", "dn_scales", "dn_bias")
    for e in sorted(set(int(v) for v in experts)):
        for name, part in zip(names, expert_tensors(shape, layer, e)):
            if part is not None:
                getattr(t, name)[e] = part
    return t


def router_tensors(shape: Shape, layer: int = 0):
    """Router weights of one layer: W bf16 bits [E][H] ~N(0, 1/H) (so that a
    normalised input gives logits of unit spread, as the given-logits inputs
    have) and bias bf16 bits [E] ~N(0, 0.1)."""
    H, E, s = shape.hidden, shape.experts, shape.seed
    w = _rng(s, layer, _T_ROUTER_W).normal(0.0, 1.0 / np.sqrt(H), (E, H)).astype(np.float32)
    b = _rng(s, layer, _T_ROUTER_B).normal(0.0, 0.1, E).astype(np.float32)
    return bf16_bits_from_f32(w), bf16_bits_from_f32(b)


def step_inputs(shape: Shape, step: int, M: int | None = None, layers: int | None = None):
    """Per-step inputs: x bf16 bits [M][H] ~N(0,1), residual bf16 bits [M][H] ~N(0,1),
    router logits fp32 [L][M][E] ~N(0,1) (+hot_bias on the hot experts)."""
    M = shape.tokens if M is None else M
    L = shape.layers if layers is None else layers
    H, E, s = shape.hidden, shape.experts, shape.seed
    x = bf16_bits_from_f32(_rng(s, step, _T_X).standard_normal((M, H), dtype=np.float32))
    r = bf16_bits_from_f32(_rng(s, step, _T_R).standard_normal((M, H), dtype=np.float32))
    logits = _rng(s, step, _T_LOGITS).standard_normal((L, M, E), dtype=np.float32)
    if shape.hot_experts:
        logits[:, :, list(shape.hot_experts)] += np.float32(shape.hot_bias)
    return x, r, logits
