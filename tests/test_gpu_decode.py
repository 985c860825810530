"""GPU parity of the routing kernels and the decode (T <= 16) path against the FP64 oracle.

Every call goes through the C ABI (libmoe.so) via the thin Python binding.
"""
import numpy as np
import pytest
import torch

import oracle
import quantised_moe_expert_gb300 as qm
from quantised_moe_expert_gb300 import synth

from . import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    qm.load()
    oracle.build()


def _check_routing_against_oracle(layer, wl, x, got, ref, logits_gpu=None):
    """ids bit-exact on unambiguous rows; p and w_s within one bf16 ulp."""
    k = wl.shape.top_k
    gap = H.oracle_gap(ref["logits"], k)
    clear = gap >= H.AMBIGUOUS_GAP
    assert np.array_equal(got["ids"][clear], ref["ids"][clear])
    same = np.all(got["ids"] == ref["ids"], axis=1)
    assert H.ulp_diff_bf16(got["p"][same], ref["p"][same]).max(initial=0) <= 1
    if wl.shape.has_shared:
        assert H.ulp_diff_bf16(got["w_s"], ref["w_s"]).max(initial=0) <= 1
    # rows whose picks differ must be near-ties of the oracle's own logits: every pick's
    # oracle logit is within the logit tolerance of the k-th largest.
    for t in np.nonzero(~same)[0]:
        lt = ref["logits"][t].astype(np.float64)
        kth = -np.sort(-lt)[k - 1]
        assert np.all(lt[got["ids"][t]] >= kth - 2 * H.LOGIT_TOL), t
    return same


@pytest.mark.parametrize("wl_index", [0, 1, 2])
def test_router_logits_and_topk(wl_index):
    wl, w, layer = H.device_layer(wl_index)
    x = synth.make_x(wl.shape, wl.tokens, wl.seed)
    got = H.run_route(layer, x)
    ref = oracle.forward(wl.shape, w, x)
    assert np.max(np.abs(got["logits"] - ref["logits"])) <= H.LOGIT_TOL
    _check_routing_against_oracle(layer, wl, x, got, ref)


@pytest.mark.parametrize("wl_index", [0, 1, 2])
def test_decode_forward_matches_oracle(wl_index):
    wl, w, layer = H.device_layer(wl_index)
    x = synth.make_x(wl.shape, wl.tokens, wl.seed)
    got = H.run_forward(layer, x, path=qm.MOE_PATH_AUTO)
    assert got["status"] == 0
    ref = oracle.forward(wl.shape, w, x)
    same = _check_routing_against_oracle(layer, wl, x, got, ref)
    stats = H.check_y(got["y"], ref["y"], rows=np.nonzero(same)[0])
    if wl_index == 0:
        # the small layer's outputs are O(1): the plain 2e-2 max-abs bound applies too
        assert stats["max_abs"] <= 2e-2, stats


def test_supplied_logits_route_bit_exact_with_forced_ties():
    """Identical fp32 logits on both sides: ids, pick weights and shared weights bit-exact."""
    wl, w, layer = H.device_layer(2)
    x = synth.make_x(wl.shape, 16, wl.seed)
    lg = oracle.router_logits(wl.shape, w, x)
    rng = np.random.default_rng(7)
    lg = synth.snap_rows_to_eighths(lg + rng.normal(0, 0.5, lg.shape).astype(np.float32), 2)
    lg[3, :] = 0.0                   # a row of all-equal logits: ids 0..7
    lg[5, ::2] = -0.0                # signed zeros compare equal
    lg[5, 1::2] = 0.0
    got = H.run_route(layer, x, logits_in=lg)
    ref = oracle.forward(wl.shape, w, x, logits_in=lg)
    gaps = H.oracle_gap(lg, wl.shape.top_k)
    assert (gaps == 0).sum() >= 2   # exact ties at the top-k boundary are present
    assert np.array_equal(got["ids"], ref["ids"])
    assert np.array_equal(got["p"], ref["p"])
    assert np.array_equal(got["w_s"], ref["w_s"])
    assert np.array_equal(got["logits"], lg)
    y = H.run_forward(layer, x, logits_in=lg)
    assert np.array_equal(y["ids"], ref["ids"])
    H.check_y(y["y"], ref["y"])


def test_decode_windows_equal_single_row_steps():
    """Rows of every window of 1..16 tokens are byte-equal to T = 1 steps of the same rows."""
    wl, w, layer = H.device_layer(2)
    x = synth.make_x(wl.shape, 16, wl.seed)
    solo = [H.run_forward(layer, x[t:t + 1]) for t in range(16)]
    for n in range(1, 17):
        win = H.run_forward(layer, x[:n])
        for t in range(n):
            for key in ("y", "ids", "p", "w_s"):
                assert np.array_equal(win[key][t], solo[t][key][0]), (n, t, key)


def test_router_bias_is_added_once_in_fp32():
    wl, w, layer = H.device_layer(0)
    x = synth.make_x(wl.shape, 4, wl.seed)
    bias = synth.zipf_bias(wl.shape, 1.1, wl.seed)
    got = H.run_route(layer, x, router_bias=bias)
    ref = oracle.forward(wl.shape, w, x, bias=bias)
    assert np.max(np.abs(got["logits"] - ref["logits"])) <= H.LOGIT_TOL
    _check_routing_against_oracle(layer, wl, x, got, ref)


def test_permute_matches_oracle():
    wl, w, layer = H.device_layer(3)
    rng = np.random.default_rng(3)
    for T in (1, 16, 130, 512, 1000):
        ids = oracle.topk(rng.normal(0, 1, (T, 256)).astype(np.float32), 8)
        ws = qm.workspace(layer.cfg, T)
        d_ids = torch.from_numpy(ids).cuda()
        counts = torch.empty(256, dtype=torch.int32, device="cuda")
        offsets = torch.empty(257, dtype=torch.int32, device="cuda")
        perm = torch.empty(T * 8, dtype=torch.int32, device="cuda")
        inv = torch.empty(T * 8, dtype=torch.int32, device="cuda")
        qm.moe_permute(layer.cfg, d_ids, T, counts, offsets, perm, inv, ws)
        torch.cuda.synchronize()
        rc, ro, rp, ri = oracle.permute(ids, 256)
        assert np.array_equal(counts.cpu().numpy(), rc)
        assert np.array_equal(offsets.cpu().numpy(), ro)
        assert np.array_equal(perm.cpu().numpy(), rp)
        assert np.array_equal(inv.cpu().numpy(), ri)
        assert qm.moe_get_device_status(ws) == 0


def test_staged_entry_points_equal_forward_decode():
    """moe_route -> moe_permute -> moe_expert_ffn (decode) -> moe_combine equals moe_forward."""
    wl, w, layer = H.device_layer(2)
    T = 16
    x_bits = synth.make_x(wl.shape, T, wl.seed, stream=1)
    full = H.run_forward(layer, x_bits, path=qm.MOE_PATH_DECODE)
    x = H.to_dev_u16(x_bits)
    ws = qm.workspace(layer.cfg, T)
    sh = wl.shape
    ids = torch.empty((T, sh.top_k), dtype=torch.int32, device="cuda")
    p = torch.empty((T, sh.top_k), dtype=torch.int16, device="cuda")
    w_s = torch.empty((T,), dtype=torch.int16, device="cuda")
    qm.moe_route(layer.cfg, layer.w, x, T, None, None, None, ids, p, w_s, ws)
    counts = torch.empty(256, dtype=torch.int32, device="cuda")
    offsets = torch.empty(257, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * 8, dtype=torch.int32, device="cuda")
    inv = torch.empty(T * 8, dtype=torch.int32, device="cuda")
    qm.moe_permute(layer.cfg, ids, T, counts, offsets, perm, inv, ws)
    acc = torch.zeros((T, sh.hidden), dtype=torch.float32, device="cuda")
    qm.moe_expert_ffn(layer.cfg, layer.w, x, T, ids, p, w_s, counts, offsets, perm, acc, qm.MOE_PATH_DECODE, ws)
    y = torch.empty((T, sh.hidden), dtype=torch.int16, device="cuda")
    qm.moe_combine(layer.cfg, T, acc, y)
    torch.cuda.synchronize()
    assert qm.moe_get_device_status(ws) == 0
    assert np.array_equal(H.u16(y), full["y"])
    assert np.array_equal(ids.cpu().numpy(), full["ids"])


def test_outputs_leave_guard_regions_untouched():
    wl, w, layer = H.device_layer(1)
    T, Hd = 3, wl.shape.hidden
    x = H.to_dev_u16(synth.make_x(wl.shape, T, wl.seed))
    guard = 4096
    buf = torch.full((T * Hd + 2 * guard,), 0x5A5A, dtype=torch.int16, device="cuda")
    y = buf[guard:guard + T * Hd].view(T, Hd)
    ws_need = qm.moe_workspace_size(layer.cfg, T)
    wsbuf = torch.full((ws_need + 2 * guard,), 0x33, dtype=torch.uint8, device="cuda")
    ws = wsbuf[guard:guard + ws_need]
    qm.moe_forward(layer.cfg, layer.w, x, T, None, None, y, None, None, None, qm.MOE_PATH_DECODE, ws)
    torch.cuda.synchronize()
    b = buf.cpu()
    assert torch.all(b[:guard] == 0x5A5A) and torch.all(b[guard + T * Hd:] == 0x5A5A)
    wb = wsbuf.cpu()
    assert torch.all(wb[:guard] == 0x33) and torch.all(wb[guard + ws_need:] == 0x33)
    assert qm.moe_get_device_status(ws) == 0
