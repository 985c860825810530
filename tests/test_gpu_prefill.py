"""GPU parity of the prefill (tcgen05 grouped GEMM) path against the FP64 oracle.

Every case is compared element by element on every row, the T = 512 and
T = 4096 layers included.  Rows whose ids differ from the oracle's (only
allowed where the oracle's k-th and (k+1)-th logits are within 1e-5) are
compared with the oracle run on the GPU's own fp32 logits for those rows.
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


def test_prefill_tiny_all_rows():
    wl, w, layer = H.device_layer(0)
    x = synth.make_x(wl.shape, wl.tokens, wl.seed)
    got = H.run_forward(layer, x, path=qm.MOE_PATH_PREFILL)
    assert got["status"] == 0
    stats, _ = H.compare_rows(wl, w, x, got, np.arange(wl.tokens))
    assert stats["max_abs"] <= 2e-2, stats


@pytest.mark.parametrize("T", [1, 3, 17, 40, 129, 2000])
def test_prefill_ragged_token_counts_small_layer(T):
    """Token counts that leave ragged N tiles, several tiles per expert and tiny experts (T = 2000:
    every routed expert above 32 tokens, on the tensor-memory GEMMs)."""
    wl, w, layer = H.device_layer(0)
    x = synth.make_x(wl.shape, T, wl.seed, stream=T)
    got = H.run_forward(layer, x, path=qm.MOE_PATH_PREFILL)
    assert got["status"] == 0
    H.compare_rows(wl, w, x, got, np.arange(T))


def test_prefill_t512_every_row():
    wl, w, layer = H.device_layer(3)
    x = synth.make_x(wl.shape, wl.tokens, wl.seed)
    got = H.run_forward(layer, x, path=qm.MOE_PATH_AUTO)
    assert got["status"] == 0
    r = H.run_route(layer, x)
    ref_logits = oracle.router_logits(wl.shape, w, x)
    assert np.abs(r["logits"].astype(np.float64) - ref_logits).max() <= H.LOGIT_TOL
    _, ndiff = H.compare_all_rows(wl, w, layer, x, got)
    assert ndiff <= 2


def test_prefill_t4096_zipf_every_row():
    wl, w, layer = H.device_layer(4)
    x = synth.make_x(wl.shape, wl.tokens, wl.seed)
    bias = synth.zipf_bias(wl.shape, wl.zipf_s, wl.seed)
    got = H.run_forward(layer, x, path=qm.MOE_PATH_AUTO, router_bias=bias)
    assert got["status"] == 0
    ref_logits = oracle.router_logits(wl.shape, w, x, bias)
    r = H.run_route(layer, x, router_bias=bias)
    err = np.abs(r["logits"].astype(np.float64) - ref_logits)
    assert err.max() <= H.LOGIT_TOL, (err.max(), np.unravel_index(err.argmax(), err.shape))
    _, ndiff = H.compare_all_rows(wl, w, layer, x, got, bias=bias)
    assert ndiff <= 2
    counts = np.bincount(got["ids"].ravel(), minlength=wl.shape.n_experts)
    assert counts.max() > 8 * wl.tokens * wl.shape.top_k / wl.shape.n_experts   # the skew is real


def test_prefill_t4096_forced_ties_bit_exact_routing():
    """Supplied logits with 5% of rows snapped to 1/8: ids, p, w_s, permutation bit-exact on all rows."""
    wl, w, layer = H.device_layer(4)
    x = synth.make_x(wl.shape, wl.tokens, wl.seed)
    bias = synth.zipf_bias(wl.shape, wl.zipf_s, wl.seed)
    lg = synth.snap_rows_to_eighths(oracle.router_logits(wl.shape, w, x, bias), wl.tie_every)
    gaps = H.oracle_gap(lg, wl.shape.top_k)
    assert (gaps == 0).sum() >= 1
    r = H.run_route(layer, x, logits_in=lg)
    ref_ids = oracle.topk(lg, wl.shape.top_k)
    assert np.array_equal(r["ids"], ref_ids)
    _, ref_p = oracle.pick_weights(lg, ref_ids)
    assert np.array_equal(r["p"], ref_p)
    _, ref_ws = oracle.shared_weight(x, w.shared_gate_vec)
    assert H.ulp_diff_bf16(r["w_s"], ref_ws).max() <= 1
    # permutation of the full batch
    T, k = wl.tokens, wl.shape.top_k
    ws = qm.workspace(layer.cfg, T)
    counts = torch.empty(256, dtype=torch.int32, device="cuda")
    offsets = torch.empty(257, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * k, dtype=torch.int32, device="cuda")
    inv = torch.empty(T * k, dtype=torch.int32, device="cuda")
    qm.moe_permute(layer.cfg, torch.from_numpy(ref_ids).cuda(), T, counts, offsets, perm, inv, ws)
    torch.cuda.synchronize()
    rc, ro, rp, ri = oracle.permute(ref_ids, 256)
    assert np.array_equal(perm.cpu().numpy(), rp) and np.array_equal(inv.cpu().numpy(), ri)
    assert np.array_equal(counts.cpu().numpy(), rc) and np.array_equal(offsets.cpu().numpy(), ro)
    # the whole layer on the forced-tie logits, every row: routing bit-exact, y within tolerance
    got = H.run_forward(layer, x, logits_in=lg)
    assert got["status"] == 0
    assert np.array_equal(got["ids"], ref_ids) and np.array_equal(got["p"], ref_p)
    H.compare_all_rows(wl, w, layer, x, got, logits_in=lg)


def test_decode_and_prefill_paths_agree():
    wl, w, layer = H.device_layer(2)
    x = synth.make_x(wl.shape, 16, wl.seed, stream=3)
    a = H.run_forward(layer, x, path=qm.MOE_PATH_DECODE)
    b = H.run_forward(layer, x, path=qm.MOE_PATH_PREFILL)
    assert np.array_equal(a["ids"], b["ids"]) and np.array_equal(a["p"], b["p"])
    H.check_y(b["y"], a["y"])


def test_staged_prefill_expert_ffn_accumulates():
    """moe_expert_ffn on the prefill path adds into a caller accumulator (twice = 2x)."""
    wl, w, layer = H.device_layer(0)
    T = 40
    sh = wl.shape
    x_bits = synth.make_x(sh, T, wl.seed, stream=5)
    x = H.to_dev_u16(x_bits)
    ws = qm.workspace(layer.cfg, T)
    ids = torch.empty((T, sh.top_k), dtype=torch.int32, device="cuda")
    p = torch.empty((T, sh.top_k), dtype=torch.int16, device="cuda")
    w_s = torch.empty((T,), dtype=torch.int16, device="cuda")
    qm.moe_route(layer.cfg, layer.w, x, T, None, None, None, ids, p, w_s, ws)
    counts = torch.empty(sh.n_experts, dtype=torch.int32, device="cuda")
    offsets = torch.empty(sh.n_experts + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * sh.top_k, dtype=torch.int32, device="cuda")
    inv = torch.empty(T * sh.top_k, dtype=torch.int32, device="cuda")
    qm.moe_permute(layer.cfg, ids, T, counts, offsets, perm, inv, ws)
    acc = torch.zeros((T, sh.hidden), dtype=torch.float32, device="cuda")
    qm.moe_expert_ffn(layer.cfg, layer.w, x, T, ids, p, w_s, counts, offsets, perm, acc, qm.MOE_PATH_PREFILL, ws)
    once = acc.clone()
    qm.moe_expert_ffn(layer.cfg, layer.w, x, T, ids, p, w_s, counts, offsets, perm, acc, qm.MOE_PATH_PREFILL, ws)
    torch.cuda.synchronize()
    assert qm.moe_get_device_status(ws) == 0
    assert torch.equal(acc, 2 * once)            # one fixed-order sum per element: exactly twice
    y = torch.empty((T, sh.hidden), dtype=torch.int16, device="cuda")
    qm.moe_combine(layer.cfg, T, once, y)
    torch.cuda.synchronize()
    ref = oracle.forward(sh, w, x_bits)
    H.check_y(H.u16(y), ref["y"])
    # the fused forward sums the same slot outputs in the same order: the same bytes
    got = H.run_forward(layer, x_bits, path=qm.MOE_PATH_PREFILL)
    assert np.array_equal(got["y"], H.u16(y))


@pytest.mark.parametrize("wl_index", [3, 4])
def test_prefill_is_bit_reproducible(wl_index):
    """Two forwards of the same batch give the same bytes (every slot output written once, summed in
    slot order)."""
    wl, w, layer = H.device_layer(wl_index)
    x = synth.make_x(wl.shape, wl.tokens, wl.seed, stream=9)
    bias = synth.zipf_bias(wl.shape, wl.zipf_s, wl.seed) if wl.zipf_s > 0 else None
    a = H.run_forward(layer, x, path=qm.MOE_PATH_PREFILL, router_bias=bias)
    b = H.run_forward(layer, x, path=qm.MOE_PATH_PREFILL, router_bias=bias)
    assert a["status"] == 0 and b["status"] == 0
    for key in ("y", "ids", "p", "w_s"):
        assert np.array_equal(a[key], b[key]), key


@pytest.mark.parametrize("forced", [False, True])
def test_prefill_rows_beyond_fp16_range(forced):
    """x far above the fp16 range, or entirely below its normal range, on the prefill path.  Five rows
    alone take the small-tile kernels (a few tokens per expert); the same rows repeated 40 times with
    every token routed to experts 0..7 make tiles of up to 128 tokens of the tensor-memory GEMMs, each
    tile mixing rows of max |x| 1e6 and 2^-20.  Per-token power-of-two scaling keeps every 16-bit
    intermediate in range; routing is pinned with supplied logits."""
    wl, w, layer = H.device_layer(1)
    x = H.range_rows(wl.shape, wl.seed)
    if forced:
        x = np.tile(x, (40, 1))
        lg = np.zeros((x.shape[0], wl.shape.n_experts), dtype=np.float32)
        lg[:, :8] = np.arange(8, 0, -1, dtype=np.float32)
    else:
        lg = oracle.router_logits(wl.shape, w, x).astype(np.float32)
    got = H.run_forward(layer, x, path=qm.MOE_PATH_PREFILL, logits_in=lg)
    assert got["status"] == 0
    ref = oracle.forward(wl.shape, w, x, logits_in=lg)
    assert np.array_equal(got["ids"], ref["ids"])
    H.check_rows_scale_free(got["y"], ref["y"])


@pytest.mark.parametrize("wl_index,T", [(0, 40), (3, 512), (4, 4096)])
def test_prefill_stages_against_fp64(wl_index, T):
    """h and the down projection of every slot on the prefill path against FP64 (the T = 4096 layer with
    its Zipf router bias: hot experts go through the tensor-memory GEMMs, cold ones through the
    small-tile kernels)."""
    wl, w, layer = H.device_layer(wl_index)
    x = synth.make_x(wl.shape, T, wl.seed, stream=6)
    bias = synth.zipf_bias(wl.shape, wl.zipf_s, wl.seed) if getattr(wl, "zipf_s", None) else None
    H.check_stages_against_fp64(wl, w, layer, x, qm.MOE_PATH_PREFILL, bias=bias)
