"""Pins for the FP64 oracle: each checks it against something other than itself.

The pages print no worked numerical example of the layer, so the pins are
hand-built fixtures (tests/golden), closed forms, textbook special cases
computed with torch/numpy float64 library routines, brute force, and
invariants of the method.  Each names the rule it pins.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from quantised_moe_expert_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits_of(vals):
    return synth.f32_to_bf16_bits(np.asarray(vals, dtype=np.float32))


# ----------------------------------------------------------------- bf16 rounding

def test_bf16_rne_matches_torch_on_fp32_values(orc):
    rng = np.random.default_rng(11)
    v = np.concatenate([rng.normal(0, 1, 4000), rng.normal(0, 1e-3, 500), rng.normal(0, 1e3, 500)]).astype(np.float32)
    expect = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.bf16_rne(v.astype(np.float64))
    assert np.array_equal(got, expect)


def test_bf16_rne_ties_and_single_rounding(orc):
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties go to the even mantissa (1.0).
    assert orc.bf16_rne([1.0 + 2.0 ** -8])[0] == 0x3F80
    # 1 + 3*2^-8 lies halfway between 1 + 2^-7 (odd) and 1 + 2^-6 (even).
    assert orc.bf16_rne([1.0 + 3 * 2.0 ** -8])[0] == 0x3F82
    # Just above the tie: an fp64 value that a detour through fp32 would round to the tie.
    assert orc.bf16_rne([1.0 + 2.0 ** -8 + 2.0 ** -40])[0] == 0x3F81
    assert orc.bf16_rne([-(1.0 + 2.0 ** -8 + 2.0 ** -40)])[0] == 0xBF81
    assert orc.bf16_rne([0.0])[0] == 0 and orc.bf16_rne([-0.0])[0] == 0x8000


# ----------------------------------------------------------------- dequant

def test_dequant_hand_built_groups(orc):
    with open(os.path.join(GOLDEN, "dequant_groups.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        codes = np.frombuffer(bytes.fromhex(c["codes_hex"]), dtype=np.uint8)
        n = c["in_dim"]
        got = orc.dequant_row(codes, bits_of(c["scales"]), bits_of(c["biases"]), c["bits"], n)
        if "expected_repeat" in c:
            exp = np.full(n, c["expected_repeat"])
        elif "expected_pattern" in c:
            pat = c["expected_pattern"]
            exp = np.array([pat[j % len(pat)] for j in range(n)], dtype=np.float64)
        elif "expected_groups" in c:
            exp = np.repeat(np.array(c["expected_groups"], dtype=np.float64), 64)
        else:
            s, b = c["expected_affine_of_index"]
            exp = s * np.arange(n) + b
        assert np.array_equal(got, exp), c["name"]


def test_dequant_round_trip_requantise(orc):
    """Codes drawn at random, dequantised, re-quantised with the same scale/bias: identical codes."""
    rng = np.random.default_rng(5)
    H = 256
    q = rng.integers(0, 16, size=H).astype(np.uint8)
    codes = (q[0::2] | (q[1::2] << 4)).astype(np.uint8)
    s = bits_of(rng.uniform(0.005, 0.02, H // 64))
    b = synth.f32_to_bf16_bits(-8 * synth.bf16_bits_to_f32(s))
    w = orc.dequant_row(codes, s, b, 4, H)
    sf = np.repeat(synth.bf16_bits_to_f32(s).astype(np.float64), 64)
    bf = np.repeat(synth.bf16_bits_to_f32(b).astype(np.float64), 64)
    assert np.array_equal(np.rint((w - bf) / sf).astype(np.uint8), q)


# ----------------------------------------------------------------- top-k

def brute_topk(logits, k):
    """Full sort by (-logit, id) with numpy lexsort: a different algorithm from the oracle's selection."""
    T, E = logits.shape
    out = np.empty((T, k), np.int32)
    ids = np.arange(E)
    for t in range(T):
        order = np.lexsort((ids, -logits[t].astype(np.float64)))
        out[t] = order[:k]
    return out


@pytest.mark.parametrize("E,k", [(16, 2), (256, 8), (8, 8), (5, 1)])
def test_topk_matches_brute_force_random(orc, E, k):
    rng = np.random.default_rng(E * 10 + k)
    logits = rng.normal(0, 1, size=(64, E)).astype(np.float32)
    assert np.array_equal(orc.topk(logits, k), brute_topk(logits, k))


def test_topk_ties_go_to_lower_id(orc):
    E, k = 32, 8
    rng = np.random.default_rng(3)
    rows = [np.zeros(E, np.float32),                                    # all equal -> ids 0..k-1
            np.where(np.arange(E) % 2 == 0, 0.0, -0.0).astype(np.float32),  # +0 == -0
            np.round(rng.normal(0, 1, E) * 2) / 2,                       # many ties at the boundary
            np.repeat(np.array([3.0, 1.0, 1.0, 1.0], np.float32), E // 4)]
    logits = np.stack(rows).astype(np.float32)
    ids = orc.topk(logits, k)
    assert np.array_equal(ids[0], np.arange(k))
    assert np.array_equal(ids[1], np.arange(k))
    assert np.array_equal(ids, brute_topk(logits, k))
    snapped = synth.snap_rows_to_eighths(rng.normal(0, 0.9, size=(200, 256)).astype(np.float32), 1)
    assert np.array_equal(orc.topk(snapped, 8), brute_topk(snapped, 8))


# ----------------------------------------------------------------- pick weights

def test_pick_weights_sum_to_one_and_order(orc):
    rng = np.random.default_rng(9)
    logits = rng.normal(0, 1, size=(128, 256)).astype(np.float32)
    ids = orc.topk(logits, 8)
    pe, pb = orc.pick_weights(logits, ids)
    assert np.all(np.abs(pe.sum(1) - 1.0) < 1e-15)
    assert np.all(np.diff(pe, axis=1) <= 0)
    assert np.all(pe > 0)
    assert np.array_equal(pb, orc.bf16_rne(pe))


def test_pick_weights_closed_forms(orc):
    # k = 1: the only pick has weight exactly 1.
    logits = np.array([[0.3, -1.0, 2.5, 0.0]], np.float32)
    ids = orc.topk(logits, 1)
    pe, pb = orc.pick_weights(logits, ids)
    assert pe[0, 0] == 1.0 and pb[0, 0] == 0x3F80
    # k equal logits: each weight is 1/k (exact in bf16 for k = 8).
    logits = np.zeros((1, 16), np.float32)
    pe, pb = orc.pick_weights(logits, orc.topk(logits, 8))
    assert np.all(pb == bits_of([0.125]))
    # two picks whose logits differ by ln 3: weights 3/4 and 1/4.
    l2 = np.float32(1.0 - math.log(3.0))
    logits = np.array([[1.0, l2, -5.0]], np.float32)
    pe, pb = orc.pick_weights(logits, orc.topk(logits, 2))
    d = float(np.float64(1.0) - np.float64(l2))
    assert abs(pe[0, 0] - 1 / (1 + math.exp(-d))) < 1e-15
    assert np.array_equal(pb[0], bits_of([0.75, 0.25]))


def test_pick_weights_translation_invariant(orc):
    rng = np.random.default_rng(4)
    logits = (rng.integers(-64, 64, size=(32, 64)) / 16).astype(np.float32)
    shifted = (logits + np.float32(3.0)).astype(np.float32)   # exact: multiples of 1/16 in range
    ids = orc.topk(logits, 8)
    assert np.array_equal(ids, orc.topk(shifted, 8))
    assert np.array_equal(orc.pick_weights(logits, ids)[0], orc.pick_weights(shifted, ids)[0])


# ----------------------------------------------------------------- shared weight

def test_shared_weight_closed_forms(orc):
    H = 128
    rng = np.random.default_rng(2)
    x = bits_of(rng.normal(0, 1, size=(3, H)))
    gamma, ws = orc.shared_weight(x, np.zeros(H, np.uint16))
    assert np.all(gamma == 0) and np.all(ws == bits_of([0.5]))
    # one-hot x and v[0] = 2: gamma = 2, weight = bf16(1 / (1 + e^-2)).
    x1 = np.zeros((1, H), np.uint16)
    x1[0, 0] = bits_of([1.0])[0]
    v = np.zeros(H, np.uint16)
    v[0] = bits_of([2.0])[0]
    gamma, ws = orc.shared_weight(x1, v)
    assert gamma[0] == 2.0
    assert ws[0] == bits_of([1.0 / (1.0 + math.exp(-2.0))])[0]
    # bf16 rounding of the gate logit before the sigmoid: gamma = 1 + 2^-8 + 2^-12 rounds to 1 + 2^-7.
    v[0] = bits_of([1.0])[0]
    v[1] = bits_of([2.0 ** -8])[0]
    v[2] = bits_of([2.0 ** -12])[0]
    x1[0, :3] = bits_of([1.0, 1.0, 1.0])
    gamma, ws = orc.shared_weight(x1, v)
    assert ws[0] == bits_of([1.0 / (1.0 + math.exp(-(1.0 + 2.0 ** -7)))])[0]


# ----------------------------------------------------------------- router logits

def test_router_logits_match_float64_matmul(orc):
    shape = synth.TINY_SHAPE
    w = synth.make_weights(shape, 0)
    x = synth.make_x(shape, 6, 0)
    R = orc.dequant_matrix(w.router.codes, w.router.scales, w.router.biases, 8, shape.hidden)
    ref = torch.from_numpy(synth.bf16_bits_to_f32(x).astype(np.float64)) @ torch.from_numpy(R).T
    assert np.array_equal(orc.router_logits(shape, w, x), ref.numpy().astype(np.float32))
    bias = np.linspace(-1, 1, shape.n_experts).astype(np.float32)
    got = orc.router_logits(shape, w, x, bias)
    exp = (ref.numpy().astype(np.float32).astype(np.float64) + bias.astype(np.float64)).astype(np.float32)
    assert np.array_equal(got, exp)


# ----------------------------------------------------------------- layer: dense special case

def _one_expert_layer(shared_zero=True, seed=7):
    shape = synth.LayerShape(hidden=128, inter=64, n_experts=1, top_k=1)
    w = synth.make_weights(shape, seed)
    if shared_zero:
        # codes all 8 with bias = -8*scale make every shared weight exactly 0.
        for m in (w.s_gate, w.s_up, w.s_down):
            m.codes[...] = 0x88
    return shape, w


def _dense_swiglu(orc, shape, m_gate, m_up, m_down, x_f64):
    """Textbook SwiGLU MLP with torch float64 library routines on the dequantised matrices."""
    Wg = torch.from_numpy(orc.dequant_matrix(m_gate[0], m_gate[1], m_gate[2], 4, shape.hidden))
    Wu = torch.from_numpy(orc.dequant_matrix(m_up[0], m_up[1], m_up[2], 4, shape.hidden))
    Wd = torch.from_numpy(orc.dequant_matrix(m_down[0], m_down[1], m_down[2], 4, shape.inter))
    x = torch.from_numpy(x_f64)
    h = torch.nn.functional.silu(x @ Wg.T) * (x @ Wu.T)
    return (h @ Wd.T).numpy()


def test_one_expert_top1_equals_dense_swiglu(orc):
    shape, w = _one_expert_layer()
    x = synth.make_x(shape, 5, 1)
    out = orc.forward(shape, w, x)
    assert np.all(out["ids"] == 0) and np.all(out["p"] == 0x3F80)
    ref = _dense_swiglu(orc, shape, (w.gate.codes[0], w.gate.scales[0], w.gate.biases[0]),
                        (w.up.codes[0], w.up.scales[0], w.up.biases[0]),
                        (w.down.codes[0], w.down.scales[0], w.down.biases[0]),
                        synth.bf16_bits_to_f32(x).astype(np.float64))
    assert np.max(np.abs(out["y_exact"] - ref) / (1 + np.abs(ref))) < 1e-12
    assert np.array_equal(out["y"], orc.bf16_rne(ref))


def test_shared_slot_weight_half_when_gate_vector_zero(orc):
    """Shared expert identical to the routed one and v = 0: y = (1 + 0.5) * y_e, rounded once."""
    shape, w = _one_expert_layer(shared_zero=False, seed=8)
    for src, dst in ((w.gate, w.s_gate), (w.up, w.s_up), (w.down, w.s_down)):
        dst.codes[...] = src.codes
        dst.scales[...] = src.scales
        dst.biases[...] = src.biases
    w.shared_gate_vec[...] = 0
    x = synth.make_x(shape, 3, 2)
    out = orc.forward(shape, w, x)
    ref = _dense_swiglu(orc, shape, (w.gate.codes[0], w.gate.scales[0], w.gate.biases[0]),
                        (w.up.codes[0], w.up.scales[0], w.up.biases[0]),
                        (w.down.codes[0], w.down.scales[0], w.down.biases[0]),
                        synth.bf16_bits_to_f32(x).astype(np.float64))
    assert np.all(out["w_s"] == bits_of([0.5]))
    assert np.max(np.abs(out["y_exact"] - 1.5 * ref) / (1 + np.abs(ref))) < 1e-12


# ----------------------------------------------------------------- layer invariants

def test_identical_experts_give_sum_of_pick_weights(orc):
    shape = synth.LayerShape(hidden=128, inter=64, n_experts=6, top_k=3)
    w = synth.make_weights(shape, 12)
    for m in (w.gate, w.up, w.down):
        m.codes[1:] = m.codes[0]
        m.scales[1:] = m.scales[0]
        m.biases[1:] = m.biases[0]
    for m in (w.s_gate, w.s_up, w.s_down):
        m.codes[...] = 0x88
    x = synth.make_x(shape, 4, 12)
    out = orc.forward(shape, w, x)
    for t in range(4):
        _, ye = orc.expert_ffn(shape, w, 0, synth.bf16_bits_to_f32(x[t]).astype(np.float64))
        psum = orc.bf16_to_f64(out["p"][t]).sum()
        assert np.max(np.abs(out["y_exact"][t] - psum * ye) / (1 + np.abs(ye))) < 1e-12


def test_expert_relabelling_invariance(orc):
    shape = synth.LayerShape(hidden=128, inter=64, n_experts=8, top_k=3)
    w = synth.make_weights(shape, 21)
    x = synth.make_x(shape, 6, 21)
    base = orc.forward(shape, w, x)
    pi = np.random.default_rng(0).permutation(8)     # expert e moves to slot pi[e]
    inv = np.argsort(pi)
    import copy
    w2 = copy.deepcopy(w)
    for m2, m in ((w2.router, w.router), (w2.gate, w.gate), (w2.up, w.up), (w2.down, w.down)):
        m2.codes[...] = m.codes[inv]
        m2.scales[...] = m.scales[inv]
        m2.biases[...] = m.biases[inv]
    out = orc.forward(shape, w2, x)
    assert np.array_equal(out["y"], base["y"])
    assert np.array_equal(out["ids"], pi[base["ids"]])
    assert np.array_equal(out["p"], base["p"])


def test_eight_bit_layer_equals_four_bit_layer_with_the_same_weights(orc):
    """Every 4-bit code written as one byte (q in 0..15), same scales and biases: the same weights, so
    the 8-bit layer's output, routing and every stage equal the 4-bit layer's bit for bit.  Several
    experts and both matrix orientations: an 8-bit row or expert stride taken as the 4-bit one fails."""
    import copy
    shape4 = synth.LayerShape(hidden=192, inter=128, n_experts=6, top_k=3)
    shape8 = synth.LayerShape(hidden=192, inter=128, n_experts=6, top_k=3, bits=8)
    w4 = synth.make_weights(shape4, 31)
    w8 = copy.deepcopy(w4)
    for name in ("gate", "up", "down", "s_gate", "s_up", "s_down"):
        c4 = getattr(w4, name).codes
        c8 = np.empty(c4.shape[:-1] + (2 * c4.shape[-1],), np.uint8)
        c8[..., 0::2] = c4 & 0x0F            # element 2i: low nibble of byte i
        c8[..., 1::2] = c4 >> 4
        getattr(w8, name).codes = c8
    x = synth.make_x(shape4, 7, 31)
    a, b = orc.forward(shape4, w4, x), orc.forward(shape8, w8, x)
    for key in ("y", "y_exact", "ids", "p", "w_s", "logits"):
        assert np.array_equal(a[key], b[key]), key
    xf = synth.bf16_bits_to_f32(x[2]).astype(np.float64)
    for e in (-1, 0, 5):
        h4, y4 = orc.expert_ffn(shape4, w4, e, xf)
        h8, y8 = orc.expert_ffn(shape8, w8, e, xf)
        assert np.array_equal(h4, h8) and np.array_equal(y4, y8), e


def test_rows_are_independent(orc):
    shape = synth.TINY_SHAPE
    w = synth.make_weights(shape, 0)
    x = synth.make_x(shape, 5, 3)
    full = orc.forward(shape, w, x)
    for t in range(5):
        one = orc.forward(shape, w, x, rows=[t])
        for key in ("y", "ids", "p", "w_s", "logits"):
            assert np.array_equal(one[key][0], full[key][t]), key


def test_logits_in_overrides_router(orc):
    shape = synth.TINY_SHAPE
    w = synth.make_weights(shape, 0)
    x = synth.make_x(shape, 4, 0)
    lg = np.zeros((4, shape.n_experts), np.float32)
    lg[:, 5] = 1.0
    lg[:, 3] = 1.0
    out = orc.forward(shape, w, x, logits_in=lg)
    assert np.all(out["ids"] == np.array([3, 5]))
    assert np.all(out["p"] == bits_of([0.5]))


# ----------------------------------------------------------------- permutation

def test_permutation_matches_stable_argsort(orc):
    rng = np.random.default_rng(1)
    for T, k, E in ((4, 2, 16), (512, 8, 256), (37, 8, 256), (0, 8, 256)):
        logits = rng.normal(0, 1, size=(T, E)).astype(np.float32)
        ids = orc.topk(logits, k) if T else np.zeros((0, k), np.int32)
        counts, offsets, perm, inv = orc.permute(ids, E)
        flat = ids.reshape(-1)
        assert np.array_equal(counts, np.bincount(flat, minlength=E))
        assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts) and offsets[-1] == T * k
        assert np.array_equal(perm, np.argsort(flat, kind="stable"))
        assert np.array_equal(inv[perm], np.arange(T * k))


# ----------------------------------------------------------------- expert down projection

def test_expert_down_equals_float64_matmul_and_one_hot_columns(orc):
    """oracle_expert_down against a torch float64 matmul of the dequantised down matrix, a one-hot
    h (which must pick out column j of that matrix: pins the [H, I] orientation and the column
    index), and linearity in h."""
    shape = synth.TINY_SHAPE
    w = synth.make_weights(shape, 5)
    rng = np.random.default_rng(17)
    for e in (0, 7, -1):
        m = w.s_down if e < 0 else w.down
        i = 0 if e < 0 else e
        Wd = orc.dequant_matrix(m.codes[i], m.scales[i], m.biases[i], 4, shape.inter)
        assert Wd.shape == (shape.hidden, shape.inter)
        h = rng.normal(0, 2, shape.inter)
        got = orc.expert_down(shape, w, e, h)
        ref = (torch.from_numpy(Wd) @ torch.from_numpy(h)).numpy()
        assert np.max(np.abs(got - ref)) <= 1e-12 * (1 + np.abs(ref).max())
        for j in (0, 1, 33, shape.inter - 1):
            onehot = np.zeros(shape.inter)
            onehot[j] = 1.0
            assert np.array_equal(orc.expert_down(shape, w, e, onehot), Wd[:, j])
        h2 = rng.normal(0, 1, shape.inter)
        lin = orc.expert_down(shape, w, e, 3.0 * h + h2)
        assert np.max(np.abs(lin - (3.0 * got + orc.expert_down(shape, w, e, h2)))) <= 1e-11


def test_expert_ffn_h_equals_float64_swiglu_of_dequantised_rows(orc):
    """The h that oracle_expert_ffn returns is silu(Wg x) * (Wu x) of the dequantised matrices."""
    shape = synth.TINY_SHAPE
    w = synth.make_weights(shape, 6)
    x = synth.bf16_bits_to_f32(synth.make_x(shape, 1, 6)).astype(np.float64)[0]
    for e in (3, -1):
        mg, mu = (w.s_gate, w.s_up) if e < 0 else (w.gate, w.up)
        i = 0 if e < 0 else e
        Wg = torch.from_numpy(orc.dequant_matrix(mg.codes[i], mg.scales[i], mg.biases[i], 4, shape.hidden))
        Wu = torch.from_numpy(orc.dequant_matrix(mu.codes[i], mu.scales[i], mu.biases[i], 4, shape.hidden))
        xt = torch.from_numpy(x)
        ref = (torch.nn.functional.silu(Wg @ xt) * (Wu @ xt)).numpy()
        h, y = orc.expert_ffn(shape, w, e, x)
        assert np.max(np.abs(h - ref)) <= 1e-12 * (1 + np.abs(ref).max())
        assert np.max(np.abs(y - orc.expert_down(shape, w, e, h))) <= 1e-12 * (1 + np.abs(y).max())
