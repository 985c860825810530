"""Pins for the oracle's NVFP4 experts, each against something other than the oracle.

The pages name NVFP4 as a checkpoint format of the layer (model card
"Qwen-3.6-35B-A3B-SIQ-K6-K4K3", served by a fused FP4 MoE backend) but print
none of its numbers.  Its definition is the public one: E2M1 elements, one E4M3
scale per 16 consecutive inputs of a row, one fp32 scale per matrix.  The pins:
the E2M1 value table of that definition written out as literals, torch's own
float8_e4m3fn decoding for every scale code, a hand-computed row, a dense torch
SwiGLU over an independently dequantised expert, and an NVFP4 layer equal to an
affine layer with the same weights.
"""
import copy

import numpy as np
import pytest
import torch

from quantised_moe_expert_gb300 import synth

# The 16 E2M1 values, code 0 .. 15 (bit 3 sign, two exponent bits with bias 1, one mantissa bit).
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]

SHAPE = synth.LayerShape(hidden=192, inter=128, n_experts=6, top_k=2, fmt="nvfp4")


def _e4m3_torch(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def _dequant_independent(codes, scales, g):
    """[rows, in/2] codes, [rows, in/16] E4M3 codes, fp32 g -> fp64 [rows, in], without the oracle."""
    q = np.empty(codes.shape[:-1] + (2 * codes.shape[-1],), np.uint8)
    q[..., 0::2] = codes & 0x0F
    q[..., 1::2] = codes >> 4
    v = np.asarray(E2M1_TABLE, np.float64)[q]
    return v * np.repeat(_e4m3_torch(scales), 16, axis=-1) * np.float64(g)


def test_e2m1_value_table(orc):
    got = [orc.e2m1_to_f64(c) for c in range(16)]
    assert got == E2M1_TABLE
    assert np.signbit(got[8]) and not np.signbit(got[0])


def test_e4m3_matches_torch_for_every_code(orc):
    ref = _e4m3_torch(np.arange(256))
    got = np.array([orc.e4m3_to_f64(c) for c in range(256)])
    nan = np.isnan(ref)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.all(np.isnan(got[nan]))
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6 and got[0x38] == 1.0


def test_nvfp4_hand_row(orc):
    """32 inputs, two blocks.  Byte i holds inputs 2i (low nibble) and 2i+1 (high nibble).
    Block 0 scale 0x38 = 1.0, block 1 scale 0x01 = 2^-9; matrix scale 0.5 (exact in fp32)."""
    codes = np.array([0x21, 0x7F, 0x98, 0x00] + [0x00] * 4 + [0x17, 0xE5, 0x00, 0x00] + [0x00] * 4, np.uint8)
    scales = np.array([0x38, 0x01], np.uint8)
    got = orc.dequant_row_nvfp4(codes, scales, 0.5, 32)
    a = [0.5, 1.0, -6.0, 6.0, -0.0, -0.5, 0.0, 0.0] + [0.0] * 8            # codes 1,2 F,7 8,9 0,0
    b = [6.0, 0.5, 3.0, -4.0, 0.0, 0.0, 0.0, 0.0] + [0.0] * 8              # codes 7,1 5,E
    expect = np.array(a, np.float64) * 0.5
    expect = np.concatenate([expect, np.array(b, np.float64) * 2.0 ** -9 * 0.5])
    assert np.array_equal(got, expect)
    assert np.signbit(got[4])


def _silu(v):
    return v / (1.0 + torch.exp(-v))


@pytest.mark.parametrize("e", [-1, 0, 3, 5])
def test_nvfp4_expert_matches_dense_torch(orc, e):
    """silu(Wg x) * (Wu x) and Wd h of an expert, with Wg, Wu, Wd dequantised by the literal E2M1
    table, torch's E4M3 decoding and the matrix scale of that expert (a block, row, expert or scale
    index slip in the oracle fails this)."""
    w = synth.make_weights(SHAPE, 41)
    mats = (w.s_gate, w.s_up, w.s_down) if e < 0 else (w.gate, w.up, w.down)
    i = 0 if e < 0 else e
    Wg, Wu, Wd = (torch.from_numpy(_dequant_independent(m.codes[i], m.scales[i], m.gscale[i])) for m in mats)
    x = torch.from_numpy(synth.bf16_bits_to_f32(synth.make_x(SHAPE, 1, 41)[0]).astype(np.float64))
    h_ref = _silu(Wg @ x) * (Wu @ x)
    y_ref = Wd @ h_ref
    h, y = orc.expert_ffn(SHAPE, w, e, x.numpy())
    assert np.max(np.abs(h - h_ref.numpy())) <= 1e-12 * max(1.0, float(h_ref.abs().max()))
    assert np.max(np.abs(y - y_ref.numpy())) <= 1e-12 * max(1.0, float(y_ref.abs().max()))
    yd = orc.expert_down(SHAPE, w, e, h_ref.numpy())
    assert np.max(np.abs(yd - y_ref.numpy())) <= 1e-12 * max(1.0, float(y_ref.abs().max()))


def test_nvfp4_layer_equals_affine_layer_with_the_same_weights(orc):
    """Codes restricted to the E2M1 values 0.5 k (|k| <= 4), the four blocks of each group of 64 given
    one E4M3 scale and the matrix scale a power of two: w = 0.5 k S g, which the affine rule stores as
    q = k + 8, s = 0.5 S g, b = -8 s (all exact in bf16).  The two layers then hold the same weights and
    the oracle gives them the same output, routing and stages bit for bit."""
    shape_a = synth.LayerShape(hidden=192, inter=128, n_experts=6, top_k=2)
    wn = synth.make_weights(SHAPE, 43)
    wa = copy.deepcopy(synth.make_weights(shape_a, 43))
    wa.router, wa.shared_gate_vec = wn.router, wn.shared_gate_vec
    rng = np.random.default_rng(43)
    k_to_code = {0: 0x0, 1: 0x1, 2: 0x2, 3: 0x3, 4: 0x4, -1: 0x9, -2: 0xA, -3: 0xB, -4: 0xC}
    for name in ("gate", "up", "down", "s_gate", "s_up", "s_down"):
        mn, ma = getattr(wn, name), getattr(wa, name)
        n, rows, half = mn.codes.shape
        k = rng.integers(-4, 5, size=(n, rows, 2 * half))
        q = np.vectorize(k_to_code.get)(k).astype(np.uint8)
        mn.codes = (q[..., 0::2] | (q[..., 1::2] << 4)).astype(np.uint8)
        a = (k + 8).astype(np.uint8)
        ma.codes = (a[..., 0::2] | (a[..., 1::2] << 4)).astype(np.uint8)
        sg = mn.scales[..., ::4]                                   # one E4M3 code per group of 64
        mn.scales = np.repeat(sg, 4, axis=-1)
        mn.gscale = np.full(n, 2.0 ** -10, np.float32)
        s = 0.5 * _e4m3_torch(sg) * 2.0 ** -10
        ma.scales = synth.f32_to_bf16_bits(s.astype(np.float32))
        assert np.array_equal(synth.bf16_bits_to_f32(ma.scales).astype(np.float64), s)
        ma.biases = synth.f32_to_bf16_bits((-8.0 * s).astype(np.float32))
    x = synth.make_x(shape_a, 5, 43)
    ra, rn = orc.forward(shape_a, wa, x), orc.forward(SHAPE, wn, x)
    for key in ("y", "y_exact", "ids", "p", "w_s", "logits"):
        assert np.array_equal(ra[key], rn[key]), key
    xf = synth.bf16_bits_to_f32(x[1]).astype(np.float64)
    for e in (-1, 0, 5):
        ha, ya = orc.expert_ffn(shape_a, wa, e, xf)
        hn, yn = orc.expert_ffn(SHAPE, wn, e, xf)
        assert np.array_equal(ha, hn) and np.array_equal(ya, yn), e
