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
    print(f"y vs oracle {wl.name} T={wl.tokens}: {stats}")
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
    ws[:512].zero_()                      # the header (status word and counters) starts zero
    qm.moe_forward(layer.cfg, layer.w, x, T, None, None, y, None, None, None, qm.MOE_PATH_DECODE, ws)
    torch.cuda.synchronize()
    b = buf.cpu()
    assert torch.all(b[:guard] == 0x5A5A) and torch.all(b[guard + T * Hd:] == 0x5A5A)
    wb = wsbuf.cpu()
    assert torch.all(wb[:guard] == 0x33) and torch.all(wb[guard + ws_need:] == 0x33)
    assert qm.moe_get_device_status(ws) == 0


def test_fused_routing_equals_route_kernel():
    """The fused decode kernel's router and top-k give the same ids and bits of p as moe_route."""
    wl, w, layer = H.device_layer(2)
    x = synth.make_x(wl.shape, 16, wl.seed, stream=4)
    r = H.run_route(layer, x)
    f = H.run_forward(layer, x, path=qm.MOE_PATH_DECODE)
    assert f["status"] == 0
    assert np.array_equal(r["ids"], f["ids"])
    assert np.array_equal(r["p"], f["p"])
    assert np.array_equal(r["w_s"], f["w_s"])


@pytest.mark.parametrize("wl_index,T", [(0, 4), (1, 1), (2, 16)])
def test_decode_stages_against_fp64(wl_index, T):
    wl, w, layer = H.device_layer(wl_index)
    x = synth.make_x(wl.shape, T, wl.seed, stream=6)
    H.check_stages_against_fp64(wl, w, layer, x, qm.MOE_PATH_DECODE)


@pytest.mark.parametrize("wl_index", [0, 1])
def test_decode_rows_beyond_fp16_range(wl_index):
    """x far above the fp16 range, or entirely below its normal range: per-token power-of-two
    scaling keeps every 16-bit intermediate in range (routing pinned with the oracle's logits)."""
    wl, w, layer = H.device_layer(wl_index)
    x = H.range_rows(wl.shape, wl.seed)
    lg = oracle.router_logits(wl.shape, w, x)
    got = H.run_forward(layer, x, path=qm.MOE_PATH_DECODE, logits_in=lg)
    assert got["status"] == 0
    ref = oracle.forward(wl.shape, w, x, logits_in=lg)
    assert np.array_equal(got["ids"], ref["ids"])
    H.check_rows_scale_free(got["y"], ref["y"])


@pytest.mark.parametrize("nstreams", [2, 4])
def test_concurrent_streams_equal_solo(nstreams):
    """Two and four decode calls in flight on separate streams and workspaces give the solo bytes."""
    wl, w, layer = H.device_layer(2)
    Ts = [1, 16, 5, 3][:nstreams]
    xs = [synth.make_x(wl.shape, T, wl.seed, stream=30 + i) for i, T in enumerate(Ts)]
    solo = [H.run_forward(layer, x, path=qm.MOE_PATH_DECODE) for x in xs]
    streams = [torch.cuda.Stream() for _ in Ts]
    outs = []
    torch.cuda.synchronize()
    for rep in range(3):
        outs = []
        for x, st in zip(xs, streams):
            xd = H.to_dev_u16(x)
            ws = qm.workspace(layer.cfg, x.shape[0])
            torch.cuda.synchronize()
            outs.append((xd, ws))
        res = []
        for (xd, ws), st in zip(outs, streams):
            res.append(qm.forward(layer, xd, ws, path=qm.MOE_PATH_DECODE, stream=st, with_routing=True))
        torch.cuda.synchronize()
        for i, (y, ids, p, w_s) in enumerate(res):
            assert qm.moe_get_device_status(outs[i][1]) == 0
            assert np.array_equal(H.u16(y), solo[i]["y"]), (nstreams, rep, i)
            assert np.array_equal(ids.cpu().numpy(), solo[i]["ids"])
            assert np.array_equal(H.u16(p), solo[i]["p"])


def test_decode_timeline_is_ordered():
    """The per-CTA stamps of one launch are non-decreasing through the kernel's phases."""
    wl, w, layer = H.device_layer(1)
    x = H.to_dev_u16(synth.make_x(wl.shape, 1, wl.seed))
    ws = qm.workspace(layer.cfg, 1)
    qm.forward(layer, x, ws, path=qm.MOE_PATH_DECODE)
    st = qm.moe_decode_timeline(layer.cfg, 1, ws)
    assert st.shape[0] >= 1
    d = np.diff(st.astype(np.int64), axis=1)
    assert np.all(d >= 0), d.min()
    assert qm.moe_get_device_status(ws) == 0


@pytest.mark.parametrize("wl_index,T", [(0, 4), (2, 16)])
def test_packed_and_gathered_down_codes_give_the_same_bytes(wl_index, T):
    """The decode kernel's two ways of reading the down codes (the packed copy, one block per
    slice, or 16-byte pieces of the MLX rows) feed the same arithmetic: identical outputs."""
    wl, w, layer = H.device_layer(wl_index)
    x = synth.make_x(wl.shape, T, wl.seed, stream=40)
    a = H.run_forward(layer, x, path=qm.MOE_PATH_DECODE)
    b = H.run_forward(layer.unpacked(), x, path=qm.MOE_PATH_DECODE)
    assert a["status"] == 0 and b["status"] == 0
    for key in ("y", "ids", "p", "w_s"):
        assert np.array_equal(a[key], b[key]), key


def test_pack_down_layout():
    """moe_pack_down writes byte b of row r, column slice c of expert e at ((e * I/32 + c) * H + r) * 16 + b."""
    wl, w, layer = H.device_layer(0)
    sh = wl.shape
    got = layer.tensors["down.packed"].cpu().numpy().view(np.uint8)
    src = w.down.codes
    E, Hd, half = src.shape
    ref = src.reshape(E, Hd, half // 16, 16).transpose(0, 2, 1, 3).reshape(-1)
    assert np.array_equal(got.reshape(-1), ref)
    sgot = layer.tensors["s_down.packed"].cpu().numpy().view(np.uint8)
    sref = w.s_down.codes.reshape(1, Hd, half // 16, 16).transpose(0, 2, 1, 3).reshape(-1)
    assert np.array_equal(sgot.reshape(-1), sref)
