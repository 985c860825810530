"""Seeded synthetic inputs for the routed-expert MoE layer.

This module is shared by the CUDA path's tests/bench and by the oracle's tests.
It draws random numbers and stores them in the layer's storage formats; it
holds none of the layer's arithmetic (no dequantisation, no router, no top-k,
no FFN, no combine).  Everything is numpy on the host.

Layer shapes follow the qwen3_5_moe routed-expert layer described on the page
"Qwen3.6-35B-A3B (qwen3_5_moe) on the native Metal engine: proposal and gate"
(section "What it is": 256 experts, 8 picked, plus a shared expert) and on
"r9700-vllm-blogs part 13" (hidden size 2048, moe_intermediate 512).  The
storage format is the MLX affine rule quoted in the same proposal (experts at
4 bits in groups of 64, router at 8 bits): a group of 64 consecutive inputs of
one output row shares one bf16 scale and one bf16 bias.  The same page's slice
"8-bit experts" names the variant with 8-bit expert codes (same rule, q in
0..255); the WORKLOADS_B8 list draws it.  WORKLOADS_NVFP4 draws the
block-scaled variant: experts in NVFP4, the checkpoint format named on the
"Qwen-3.6-35B-A3B-SIQ-K6-K4K3" model card (4-bit E2M1 codes, one E4M3 scale
per 16 inputs of a row, one fp32 scale per matrix; router unchanged).

Storage layout (all little-endian, rows dense):
  x        bf16 bits, uint16 [T, H]
  router   codes uint8 [E, H], scales/biases bf16 bits uint16 [E, H/64]
  v        shared-expert gate vector, bf16 bits uint16 [H]
  gate, up codes uint8 [E, I, H/2] (4-bit: element j of a row is byte j//2,
           low nibble for even j; 8-bit: [E, I, H], element j is byte j),
           scales/biases uint16 [E, I, H/64]
  down     codes uint8 [E, H, I/2] (8-bit: [E, H, I]), scales/biases uint16 [E, H, I/64]
  s_gate, s_up, s_down: the shared expert, same layouts with a leading dim of 1
  NVFP4 experts: codes as the 4-bit codes (E2M1: bit 3 sign, bits 2-1 exponent,
           bit 0 mantissa), scales uint8 E4M3 [E, rows, in/16], no biases (an
           empty array), gscale float32 [E] (one per matrix)
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

GROUP = 64


@dataclasses.dataclass(frozen=True)
class LayerShape:
    hidden: int
    inter: int
    n_experts: int
    top_k: int
    has_shared: int = 1
    bits: int = 4
    router_bits: int = 8
    group: int = GROUP
    fmt: str = "affine"        # "affine" (MLX, bits 4 or 8) or "nvfp4" (bits 4)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One named workload: a layer shape, a token count and the input recipe."""
    name: str
    shape: LayerShape
    tokens: int
    seed: int
    zipf_s: float = 0.0        # > 0: per-expert log-Zipf logit bias
    tie_every: int = 0         # > 0: every n-th row of supplied logits is snapped to 1/8


QWEN_SHAPE = LayerShape(hidden=2048, inter=512, n_experts=256, top_k=8)
QWEN_SHAPE_B8 = dataclasses.replace(QWEN_SHAPE, bits=8)
QWEN_SHAPE_NVFP4 = dataclasses.replace(QWEN_SHAPE, fmt="nvfp4")
TINY_SHAPE = LayerShape(hidden=256, inter=64, n_experts=16, top_k=2)

WORKLOADS = [
    Workload("tiny_T4_H256_E16_k2", TINY_SHAPE, 4, seed=0),
    Workload("decode_T1_H2048_E256_k8", QWEN_SHAPE, 1, seed=1),
    Workload("decode_T16_H2048_E256_k8", QWEN_SHAPE, 16, seed=2),
    Workload("prefill_T512_H2048_E256_k8", QWEN_SHAPE, 512, seed=3),
    Workload("prefill_T4096_zipf1.1_H2048_E256_k8", QWEN_SHAPE, 4096, seed=4,
             zipf_s=1.1, tie_every=20),
]

# The same layer with 8-bit expert codes (router unchanged).
WORKLOADS_B8 = [
    Workload("decode_T1_H2048_E256_k8_b8", QWEN_SHAPE_B8, 1, seed=11),
    Workload("decode_T16_H2048_E256_k8_b8", QWEN_SHAPE_B8, 16, seed=12),
    Workload("prefill_T512_H2048_E256_k8_b8", QWEN_SHAPE_B8, 512, seed=13),
]


# The same layer with NVFP4 experts (router unchanged).
WORKLOADS_NVFP4 = [
    Workload("decode_T1_H2048_E256_k8_nvfp4", QWEN_SHAPE_NVFP4, 1, seed=21),
    Workload("decode_T16_H2048_E256_k8_nvfp4", QWEN_SHAPE_NVFP4, 16, seed=22),
    Workload("prefill_T512_H2048_E256_k8_nvfp4", QWEN_SHAPE_NVFP4, 512, seed=23),
]


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); returns uint16 bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class QMat:
    codes: np.ndarray    # uint8 [..., rows, in*bits/8]
    scales: np.ndarray   # uint16 [..., rows, in/64]
    biases: np.ndarray   # uint16 [..., rows, in/64] (NVFP4: empty)
    gscale: np.ndarray | None = None   # NVFP4: float32 [...], one per matrix


@dataclasses.dataclass
class LayerWeights:
    shape: LayerShape
    router: QMat
    gate: QMat
    up: QMat
    down: QMat
    s_gate: QMat
    s_up: QMat
    s_down: QMat
    shared_gate_vec: np.ndarray   # uint16 [H]

    def nbytes(self) -> int:
        tot = self.shared_gate_vec.nbytes
        for m in (self.router, self.gate, self.up, self.down, self.s_gate, self.s_up, self.s_down):
            tot += m.codes.nbytes + m.scales.nbytes + m.biases.nbytes + (0 if m.gscale is None else m.gscale.nbytes)
        return tot


def _expert_qmat(rng: np.random.Generator, n: int, rows: int, cols: int) -> QMat:
    """4-bit codes uniform in 0..15, scale ~ U(0.005, 0.02) rounded to bf16, bias = -8*scale."""
    codes = rng.integers(0, 256, size=(n, rows, cols // 2), dtype=np.uint8)
    s = f32_to_bf16_bits(rng.uniform(0.005, 0.02, size=(n, rows, cols // GROUP)).astype(np.float32))
    # -8 * s is exact in bf16 (power-of-two scaling of a bf16 value).
    b = f32_to_bf16_bits(-8.0 * bf16_bits_to_f32(s))
    return QMat(codes, s, b)


def _expert_qmat8(rng: np.random.Generator, n: int, rows: int, cols: int) -> QMat:
    """8-bit codes uniform in 0..255, scale ~ U(0.005, 0.02) / 16 rounded to bf16, bias = -128*scale.

    The same weight spread as the 4-bit draw (|w| up to about 0.16), over 256 levels.
    """
    codes = rng.integers(0, 256, size=(n, rows, cols), dtype=np.uint8)
    s = f32_to_bf16_bits(rng.uniform(0.005 / 16, 0.02 / 16, size=(n, rows, cols // GROUP)).astype(np.float32))
    # -128 * s is exact in bf16 (power-of-two scaling of a bf16 value).
    b = f32_to_bf16_bits(-128.0 * bf16_bits_to_f32(s))
    return QMat(codes, s, b)


def _expert_qmat_nvfp4(rng: np.random.Generator, n: int, rows: int, cols: int) -> QMat:
    """NVFP4: E2M1 codes uniform over all 16 (so -0 too); E4M3 block scales with exponent field
    uniform in 9..13 and mantissa uniform (values 4 to 120, never NaN); per-matrix fp32 scale
    ~ U(3e-4, 6e-4).  |w| up to about 0.4, mean about 0.04, near the affine draws' spread."""
    codes = rng.integers(0, 256, size=(n, rows, cols // 2), dtype=np.uint8)
    e = rng.integers(9, 14, size=(n, rows, cols // 16), dtype=np.uint8)
    m = rng.integers(0, 8, size=(n, rows, cols // 16), dtype=np.uint8)
    scales = ((e << 3) | m).astype(np.uint8)
    g = rng.uniform(3e-4, 6e-4, size=(n,)).astype(np.float32)
    return QMat(codes, scales, np.zeros((n, rows, 0), dtype=np.uint16), g)


def _quantise_8bit(w: np.ndarray) -> QMat:
    """Generator-side 8-bit affine quantiser for the router (group 64 along the input dim).

    Per group: bias = min, scale = (max - min) / 255, both rounded to bf16;
    code = clamp(rint((w - bias) / scale), 0, 255).  Only the code
    distribution depends on this rule: both the kernels and the oracle read
    the stored codes, scales and biases.
    """
    rows, cols = w.shape
    g = w.reshape(rows, cols // GROUP, GROUP).astype(np.float32)
    lo = g.min(axis=2)
    hi = g.max(axis=2)
    b_bits = f32_to_bf16_bits(lo)
    s_bits = f32_to_bf16_bits((hi - lo) / 255.0)
    b = bf16_bits_to_f32(b_bits)[..., None]
    s = bf16_bits_to_f32(s_bits)[..., None]
    s_safe = np.where(s > 0, s, 1.0)
    q = np.clip(np.rint((g - b) / s_safe), 0, 255).astype(np.uint8)
    return QMat(q.reshape(rows, cols), s_bits, b_bits)


def make_weights(shape: LayerShape, seed: int) -> LayerWeights:
    """Draw one layer's weights.  Draw order: router, v, gate, up, down, shared gate/up/down."""
    assert shape.bits in (4, 8) and shape.router_bits == 8 and shape.group == GROUP
    assert shape.fmt in ("affine", "nvfp4") and (shape.fmt == "affine" or shape.bits == 4)
    H, I, E = shape.hidden, shape.inter, shape.n_experts
    rng = np.random.default_rng([seed, 1])
    router = _quantise_8bit(rng.normal(0.0, 0.02, size=(E, H)).astype(np.float32))
    v = f32_to_bf16_bits(rng.normal(0.0, 0.02, size=(H,)).astype(np.float32))
    qmat = _expert_qmat_nvfp4 if shape.fmt == "nvfp4" else _expert_qmat8 if shape.bits == 8 else _expert_qmat
    gate = qmat(rng, E, I, H)
    up = qmat(rng, E, I, H)
    down = qmat(rng, E, H, I)
    ns = 1 if shape.has_shared else 0
    s_gate = qmat(rng, ns, I, H)
    s_up = qmat(rng, ns, I, H)
    s_down = qmat(rng, ns, H, I)
    return LayerWeights(shape, router, gate, up, down, s_gate, s_up, s_down, v)


def make_x(shape: LayerShape, tokens: int, seed: int, stream: int = 0) -> np.ndarray:
    """x ~ N(0, 1) rounded to bf16, [T, H] uint16 bits."""
    rng = np.random.default_rng([seed, 2, stream])
    return f32_to_bf16_bits(rng.normal(0.0, 1.0, size=(tokens, shape.hidden)).astype(np.float32))


def zipf_bias(shape: LayerShape, s: float, seed: int) -> np.ndarray:
    """Per-expert logit bias -s*ln(r_e), r_e = 1 + pi(e) for a seeded permutation pi.

    Adding ln of a Zipf(s) prior to the logits makes expert popularity follow
    that prior: a few experts take most tokens.
    """
    rng = np.random.default_rng([seed, 3])
    ranks = 1 + rng.permutation(shape.n_experts)
    return (-s * np.log(ranks.astype(np.float64))).astype(np.float32)


def snap_rows_to_eighths(logits: np.ndarray, every: int) -> np.ndarray:
    """Return a copy of fp32 logits with rows t % every == 0 snapped to multiples of 1/8.

    Snapping to a coarse grid makes exact equal logits common, which exercises
    the lower-id tie rule of the top-k.
    """
    out = np.array(logits, dtype=np.float32, copy=True)
    rows = np.arange(0, out.shape[0], every)
    out[rows] = (np.rint(out[rows].astype(np.float64) * 8.0) / 8.0).astype(np.float32)
    return out


def workload_inputs(wl: Workload, stream: int = 0):
    """(weights, x, router_bias or None) for a named workload."""
    w = make_weights(wl.shape, wl.seed)
    x = make_x(wl.shape, wl.tokens, wl.seed, stream)
    bias = zipf_bias(wl.shape, wl.zipf_s, wl.seed) if wl.zipf_s > 0 else None
    return w, x, bias


def active_expert_bytes(shape: LayerShape) -> int:
    """Bytes of one expert's gate+up+down codes, scales and biases (NVFP4: codes, block scales and
    the per-matrix scale)."""
    H, I = shape.hidden, shape.inter
    if shape.fmt == "nvfp4":
        per = lambda rows, cols: rows * cols // 2 + rows * (cols // 16) + 4
    else:
        per = lambda rows, cols: rows * cols * shape.bits // 8 + 2 * 2 * rows * (cols // GROUP)
    return 2 * per(I, H) + per(H, I)


def router_bytes(shape: LayerShape) -> int:
    H, E = shape.hidden, shape.n_experts
    return E * H * shape.router_bits // 8 + 2 * 2 * E * (H // GROUP) + 2 * H


def expert_flops_per_token(shape: LayerShape) -> int:
    """Multiply-adds x2 of the k routed + shared expert FFNs for one token."""
    slots = shape.top_k + (1 if shape.has_shared else 0)
    return slots * 3 * 2 * shape.hidden * shape.inter


def nominal_tokens_per_expert(wl: Workload) -> float:
    return wl.tokens * wl.shape.top_k / wl.shape.n_experts


if __name__ == "__main__":
    for wl in WORKLOADS + WORKLOADS_B8 + WORKLOADS_NVFP4:
        print(wl.name, active_expert_bytes(wl.shape), router_bytes(wl.shape),
              expert_flops_per_token(wl.shape), math.ceil(nominal_tokens_per_expert(wl)))
