"""Shared helpers of the GPU parity tests: device upload, C-ABI calls, comparisons."""
import concurrent.futures
import os

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
# The prefill path's tensor-memory GEMMs (experts with more than 32 tokens) dequantise each weight to
# fp16, w = fp16(s q + b): one more rounding of 2^-11 relative per weight, in both projections, so
# the errors of h and of the down output grow to a few 2^-11 of the row's terms (measured on GB300
# over every slot: h 1.5e-3 and down 1.9e-3 at T = 512, 9.7e-4 and 1.5e-3 at T = 4096; the
# small-tile kernels, exact codes, 4.7e-4 and 9.7e-5 at T = 40).
PREFILL_STAGE_H_TOL = 4e-3
PREFILL_STAGE_DOWN_TOL = 4e-3
# With 8-bit codes that rounding is real for every weight: s (q - 128) needs up to 16 significant bits
# (the synthetic 4-bit weights s (q - 8) need at most 11 and are exact in fp16), so each weight carries
# up to 2^-11 relative error and a row's sum up to 2^-11 sum_j |w_j x_j|, some 1e-2 of max(1, |g|) at
# the worst of 2.4 million elements (measured on GB300 at T = 512: h 1.7e-2, down 1.0e-2).  The
# relative RMS over all slots stays near 2^-11 / sqrt(3) of the typical term and is checked tightly.
PREFILL_B8_STAGE_TOL = 4e-2
PREFILL_B8_STAGE_REL_RMS = 2e-3
STAGE_REL_RMS = 1e-3

_layers = {}


def device_layer(wl):
    """(workload, host weights, device layer) for a named workload (a synth.Workload, or an index
    into synth.WORKLOADS), cached per session."""
    if isinstance(wl, int):
        wl = synth.WORKLOADS[wl]
    if wl.name not in _layers:
        w = synth.make_weights(wl.shape, wl.seed)
        _layers[wl.name] = (wl, w, qm.DeviceLayer(w))
    return _layers[wl.name]


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


def range_rows(shape, seed):
    """Rows of x whose magnitudes leave the fp16 range: max |x| of 1e3, 7e4 and 1e6, a row entirely
    below 2^-14 (the smallest fp16 normal), and an ordinary row."""
    base = synth.bf16_bits_to_f32(synth.make_x(shape, 5, seed, stream=21)).astype(np.float64)
    scale = np.array([1e3, 7e4, 1e6, 2.0 ** -20, 1.0])
    rows = base / np.abs(base).max(axis=1, keepdims=True) * scale[:, None]
    rows[4] = base[4]
    return synth.f32_to_bf16_bits(rows.astype(np.float32))


def check_rows_scale_free(y_gpu, y_ref):
    """The output rule of check_y made independent of each row's scale: per-row relative RMS, and every
    element within 4e-3 of the row's RMS (the plain 2e-2 bound at the workloads' output RMS of ~5) or
    one bf16 rounding flip from the oracle."""
    for t in range(y_ref.shape[0]):
        g, r = bf16_to_f64(y_gpu[t]), bf16_to_f64(y_ref[t])
        assert np.all(np.isfinite(g)), t
        rms = np.sqrt((r ** 2).mean())
        rel = np.sqrt(((g - r) ** 2).sum() / (r ** 2).sum())
        assert rel <= REL_RMS_TOL, (t, rel)
        beyond = np.abs(g - r) > 4e-3 * rms
        assert ulp_diff_bf16(y_gpu[t][beyond], y_ref[t][beyond]).max(initial=0) <= 1, (t, rms)


def stages(layer, x_bits, ids, path):
    """h and the unweighted expert output of every slot from moe_expert_stages (fp64 copies)."""
    sh = layer.shape
    T = x_bits.shape[0]
    nslot = T * (sh.top_k + sh.has_shared)
    x = to_dev_u16(x_bits)
    ws = qm.workspace(layer.cfg, T)
    d_ids = torch.from_numpy(np.ascontiguousarray(ids, np.int32)).cuda()
    counts = torch.empty(sh.n_experts, dtype=torch.int32, device="cuda")
    offsets = torch.empty(sh.n_experts + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * sh.top_k, dtype=torch.int32, device="cuda")
    inv = torch.empty(T * sh.top_k, dtype=torch.int32, device="cuda")
    qm.moe_permute(layer.cfg, d_ids, T, counts, offsets, perm, inv, ws)
    h = torch.full((nslot, sh.inter), float("nan"), dtype=torch.float32, device="cuda")
    # both paths write every element of the slot outputs once: NaN marks an element never written
    ys = torch.full((nslot, sh.hidden), float("nan"), dtype=torch.float32, device="cuda")
    qm.moe_expert_stages(layer.cfg, layer.w, x, T, d_ids, counts, offsets, perm, h, ys, path, ws)
    torch.cuda.synchronize()
    assert qm.moe_get_device_status(ws) == 0
    return h.cpu().numpy().astype(np.float64), ys.cpu().numpy().astype(np.float64)


def check_stages_against_fp64(wl, w, layer, x_bits, path, bias=None):
    """Each projection class on its own against an FP64 restatement fed the same inputs, on every slot.

    gate/up pair: h from the GPU against the oracle's h for the same x (the GPU rounds h to fp16: 11
    significant bits).  down: the GPU's slot output against the oracle's down projection of the GPU's
    own h.  The oracle calls run in threads (its C routines release the interpreter lock)."""
    import oracle
    sh = wl.shape
    T, k = x_bits.shape[0], sh.top_k
    ids = oracle.topk(oracle.router_logits(sh, w, x_bits, bias), k)
    h_gpu, y_gpu = stages(layer, x_bits, ids, path)
    xs = bf16_to_f64(x_bits)
    slots = [(t, t * k + j, int(ids[t, j])) for t in range(T) for j in range(k)]
    if sh.has_shared:
        slots += [(t, T * k + t, -1) for t in range(T)]

    def one(slot):
        t, f, e = slot
        h_ref, _ = oracle.expert_ffn(sh, w, e, xs[t])
        dh = float((np.abs(h_gpu[f] - h_ref) / np.maximum(1.0, np.abs(h_ref))).max())
        y_ref = oracle.expert_down(sh, w, e, h_gpu[f])
        dy = float((np.abs(y_gpu[f] - y_ref) / np.maximum(1.0, np.abs(y_ref))).max())
        # squared error and squared reference sums, for the relative RMS over all slots
        return (dh, dy, float(((h_gpu[f] - h_ref) ** 2).sum()), float((h_ref ** 2).sum()),
                float(((y_gpu[f] - y_ref) ** 2).sum()), float((y_ref ** 2).sum()))

    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1))) as ex:
        errs = np.array(list(ex.map(one, slots, chunksize=64)))
    assert not np.isnan(errs).any(), "a stage output holds NaN (not written)"
    worst_h, worst_y = float(errs[:, 0].max()), float(errs[:, 1].max())
    rms_h = float(np.sqrt(errs[:, 2].sum() / errs[:, 3].sum()))
    rms_y = float(np.sqrt(errs[:, 4].sum() / errs[:, 5].sum()))
    prefill = path == qm.MOE_PATH_PREFILL
    print(f"stage errors T={T} bits={sh.bits} path={path}: h {worst_h:.3e} (rel RMS {rms_h:.3e}), "
          f"down {worst_y:.3e} (rel RMS {rms_y:.3e}) over {len(slots)} slots")
    if getattr(sh, "fmt", "affine") == "nvfp4":
        # NVFP4 weights are exact in fp16 (e2m1 * e4m3: at most 6 significant bits) on both paths: h
        # carries its fp16 rounding, the down projection sums exact products
        tol_h, tol_y, tol_rms = STAGE_H_TOL, STAGE_DOWN_TOL, STAGE_REL_RMS
    elif prefill and sh.bits == 8:
        tol_h = tol_y = PREFILL_B8_STAGE_TOL
        tol_rms = PREFILL_B8_STAGE_REL_RMS
    elif prefill:
        tol_h, tol_y, tol_rms = PREFILL_STAGE_H_TOL, PREFILL_STAGE_DOWN_TOL, STAGE_REL_RMS
    else:
        tol_h, tol_y, tol_rms = STAGE_H_TOL, STAGE_DOWN_TOL, STAGE_REL_RMS
    assert worst_h <= tol_h, worst_h
    assert worst_y <= tol_y, worst_y
    assert rms_h <= tol_rms and rms_y <= tol_rms, (rms_h, rms_y)
    return worst_h, worst_y


def compare_rows(wl, w, x, got, rows, bias=None, logits_in=None):
    """ids (outside near-ties), p and y of the given rows against the oracle; returns (y stats, oracle)."""
    import oracle
    ref = oracle.forward(wl.shape, w, x, bias=bias, logits_in=logits_in, rows=rows)
    g = {key: got[key][rows] for key in ("y", "ids", "p", "w_s")}
    gap = oracle_gap(ref["logits"], wl.shape.top_k)
    clear = gap >= (0 if logits_in is not None else AMBIGUOUS_GAP)
    assert np.array_equal(g["ids"][clear], ref["ids"][clear])
    same = np.nonzero(np.all(g["ids"] == ref["ids"], axis=1))[0]
    assert ulp_diff_bf16(g["p"][same], ref["p"][same]).max(initial=0) <= 1
    stats = check_y(g["y"], ref["y"], rows=same)
    print(f"y vs oracle {wl.name} T={x.shape[0]} rows={len(same)}: {stats}")
    return stats, ref


def compare_all_rows(wl, w, layer, x, got, bias=None, logits_in=None):
    """Every row: ids, p, w_s and y against the oracle; near-tie rows under the GPU's own logits."""
    import oracle
    T = x.shape[0]
    stats, ref = compare_rows(wl, w, x, got, np.arange(T), bias=bias, logits_in=logits_in)
    if wl.shape.has_shared:
        assert ulp_diff_bf16(got["w_s"], ref["w_s"]).max(initial=0) <= 1
    diff = np.nonzero(np.any(got["ids"] != ref["ids"], axis=1))[0]
    if len(diff):
        assert logits_in is None
        r = run_route(layer, x, router_bias=bias)
        assert np.array_equal(r["ids"], got["ids"])
        ref2 = oracle.forward(wl.shape, w, x, logits_in=r["logits"], rows=diff)
        assert np.array_equal(ref2["ids"], got["ids"][diff])
        assert np.array_equal(ref2["p"], got["p"][diff])
        check_y(got["y"][diff], ref2["y"])
    return stats, len(diff)
