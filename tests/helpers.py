"""Shared helpers of the GPU parity tests: device upload, C-ABI calls, comparisons."""
import numpy as np
import torch

import quantised_moe_expert_gb300 as qm
from quantised_moe_expert_gb300 import synth

# Output tolerance against the bf16-rounded oracle.  Every element must be within the plain
# ABS_TOL of the oracle or be its bf16 neighbour (one rounding flip: the kernels' fp32 value and
# the oracle's fp64 value straddle a bf16 rounding boundary), and within ELEM_TOL * max(1, |y|);
# the whole output within REL_RMS_TOL relative RMS.
ABS_TOL = 2e-2
ELEM_TOL = 2e-2          # |y - y_ref| <= ELEM_TOL * max(1, |y_ref|)
REL_RMS_TOL = 1e-2       # ||y - y_ref||_2 / ||y_ref||_2
# Router logits: the kernels sum in fp32, the oracle in fp64 then rounds once; the largest
# difference measured on the five workloads is below 2e-6 (logits of magnitude up to ~5).
LOGIT_TOL = 4e-6
AMBIGUOUS_GAP = 1e-5     # ids must equal the oracle's on every row whose k-th / (k+1)-th gap is at least this
# Stage checks, |gpu - fp64| / max(1, |fp64|): h is rounded to fp16 (relative 2^-11 = 4.9e-4) after
# fp32 sums of g and u; the down projection sums exact products (signed codes times fp16 h) in fp32.
STAGE_H_TOL = 1e-3
STAGE_DOWN_TOL = 1e-4

_layers = {}


def device_layer(wl_index: int):
    """(workload, host weights, device layer) for a named workload, cached per session."""
    if wl_index not in _layers:
        wl = synth.WORKLOADS[wl_index]
        w = synth.make_weights(wl.shape, wl.seed)
        _layers[wl_index] = (wl, w, qm.DeviceLayer(w))
    return _layers[wl_index]


def to_dev_u16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def u16(t):
    return t.cpu().numpy().view(np.uint16)


def bf16_to_f64(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def ulp_diff_bf16(a, b):
    """|a - b| in bf16 units in the last place (sign-magnitude ordering)."""
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    return np.abs(ordered(a) - ordered(b))


def run_forward(layer, x_bits, path=qm.MOE_PATH_AUTO, router_bias=None, logits_in=None, cfg=None):
    x = to_dev_u16(x_bits)
    T = x_bits.shape[0]
    ws = qm.workspace(layer.cfg, T)
    rb = None if router_bias is None else torch.from_numpy(router_bias).cuda()
    li = None if logits_in is None else torch.from_numpy(np.ascontiguousarray(logits_in, np.float32)).cuda()
    y, ids, p, w_s = qm.forward(layer, x, ws, router_bias=rb, logits_in=li, path=path, with_routing=True, cfg=cfg)
    torch.cuda.synchronize()
    status = qm.moe_get_device_status(ws)
    return dict(y=u16(y), ids=ids.cpu().numpy(), p=u16(p), w_s=u16(w_s)[:T], status=status)


def run_route(layer, x_bits, router_bias=None, logits_in=None):
    x = to_dev_u16(x_bits)
    T = x_bits.shape[0]
    sh = layer.shape
    ws = qm.workspace(layer.cfg, T)
    logits = torch.empty((T, sh.n_experts), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, sh.top_k), dtype=torch.int32, device="cuda")
    p = torch.empty((T, sh.top_k), dtype=torch.int16, device="cuda")
    w_s = torch.empty((T,), dtype=torch.int16, device="cuda")
    rb = None if router_bias is None else torch.from_numpy(router_bias).cuda()
    li = None if logits_in is None else torch.from_numpy(np.ascontiguousarray(logits_in, np.float32)).cuda()
    qm.moe_route(layer.cfg, layer.w, x, T, rb, li, logits, ids, p, w_s, ws)
    torch.cuda.synchronize()
    return dict(logits=logits.cpu().numpy(), ids=ids.cpu().numpy(), p=u16(p), w_s=u16(w_s))


def oracle_gap(logits, k):
    """k-th minus (k+1)-th largest logit per row (inf when k == E)."""
    s = -np.sort(-logits.astype(np.float64), axis=1)
    if s.shape[1] <= k:
        return np.full(s.shape[0], np.inf)
    return s[:, k - 1] - s[:, k]


def check_y(y_gpu, y_ref, rows=None):
    """Element-wise and relative-RMS output tolerance; returns the stats."""
    yg = y_gpu if rows is None else y_gpu[rows]
    yr = y_ref if rows is None else y_ref[rows]
    g = bf16_to_f64(yg)
    r = bf16_to_f64(yr)
    err = np.abs(g - r)
    ulp = ulp_diff_bf16(yg, yr)
    scaled = err / np.maximum(1.0, np.abs(r))
    rel_rms = np.sqrt((err ** 2).sum() / max((r ** 2).sum(), 1e-300))
    beyond_abs = err > ABS_TOL
    stats = dict(max_abs=float(err.max(initial=0)), max_scaled=float(scaled.max(initial=0)), rel_rms=float(rel_rms),
                 max_ulp=int(ulp.max(initial=0)), n_beyond_abs=int(beyond_abs.sum()),
                 max_ulp_beyond_abs=int(ulp[beyond_abs].max(initial=0)))
    assert stats["max_ulp_beyond_abs"] <= 1, stats      # |err| <= 2e-2, or one bf16 rounding flip
    assert stats["max_scaled"] <= ELEM_TOL, stats
    assert stats["rel_rms"] <= REL_RMS_TOL, stats
    return stats
