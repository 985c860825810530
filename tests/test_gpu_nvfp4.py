"""GPU parity of the layer with NVFP4 experts against the FP64 oracle.

NVFP4 is the checkpoint format of the model card "Qwen-3.6-35B-A3B-SIQ-K6-K4K3"
(served there by a fused FP4 MoE backend): E2M1 codes, an E4M3 scale per 16
inputs of a row, an fp32 scale per matrix; the router stays 8-bit affine.  At
every T the experts run on the tensor-memory grouped GEMMs (every item; a
decode path request selects them too).  Every row is compared, and each
projection class on its own against FP64.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import quantised_moe_expert_gb300 as qm
from quantised_moe_expert_gb300 import synth

from . import helpers as H

pytestmark = pytest.mark.gpu

TINY_NV = synth.Workload("tiny_T4_H256_E16_k2_nvfp4", dataclasses.replace(synth.TINY_SHAPE, fmt="nvfp4"), 4, seed=20)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    qm.load()
    oracle.build()


@pytest.mark.parametrize("i", range(len(synth.WORKLOADS_NVFP4)), ids=[wl.name for wl in synth.WORKLOADS_NVFP4])
def test_nvfp4_forward_every_row(i):
    """T = 1, 16 and 512: ids, p, w_s and y on every row."""
    wl, w, layer = H.device_layer(synth.WORKLOADS_NVFP4[i])
    x = synth.make_x(wl.shape, wl.tokens, wl.seed)
    got = H.run_forward(layer, x, path=qm.MOE_PATH_AUTO)
    assert got["status"] == 0
    stats, ndiff = H.compare_all_rows(wl, w, layer, x, got)
    print(wl.name, stats, "near-tie rows", ndiff)
    assert ndiff <= 2


@pytest.mark.parametrize("path", [qm.MOE_PATH_DECODE, qm.MOE_PATH_PREFILL], ids=["decode", "prefill"])
@pytest.mark.parametrize("T", [1, 3, 17, 40, 129])
def test_nvfp4_ragged_token_counts_small_layer(T, path):
    """A small NVFP4 layer (I = 64: a weight tile half past the expert's rows) at ragged token counts."""
    wl, w, layer = H.device_layer(TINY_NV)
    x = synth.make_x(wl.shape, T, wl.seed, stream=T)
    got = H.run_forward(layer, x, path=path)
    assert got["status"] == 0
    H.compare_rows(wl, w, x, got, np.arange(T))


@pytest.mark.parametrize("path", [qm.MOE_PATH_DECODE, qm.MOE_PATH_PREFILL], ids=["decode", "prefill"])
def test_nvfp4_edge_scales_and_codes(path):
    """Block scales at the ends of E4M3 (subnormals 2^-9 .. 7 2^-9, zero, the largest normal 448, the
    smallest normal 2^-6), negative scales, and blocks of -0 codes, in every expert matrix."""
    wl = TINY_NV
    w = synth.make_weights(wl.shape, 77)
    rng = np.random.default_rng(77)
    special = np.array([0x01, 0x02, 0x07, 0x00, 0x7E, 0x08, 0xB8, 0x80], np.uint8)
    for name in ("gate", "up", "down", "s_gate", "s_up", "s_down"):
        m = getattr(w, name)
        sel = rng.random(m.scales.shape) < 0.25
        m.scales[sel] = special[rng.integers(0, len(special), size=int(sel.sum()))]
        zero = rng.random(m.codes.shape) < 0.05
        m.codes[zero] = 0x88
    layer = qm.DeviceLayer(w)
    x = synth.make_x(wl.shape, 24, 77)
    got = H.run_forward(layer, x, path=path)
    assert got["status"] == 0
    H.compare_rows(wl, w, x, got, np.arange(24))


@pytest.mark.parametrize("T", [1, 16])
def test_nvfp4_prefill_path_at_decode_sizes(T):
    """The grouped GEMMs at one 16-column tile per expert give the oracle's rows too."""
    wl, w, layer = H.device_layer(synth.WORKLOADS_NVFP4[1])
    x = synth.make_x(wl.shape, T, wl.seed, stream=50 + T)
    got = H.run_forward(layer, x, path=qm.MOE_PATH_PREFILL)
    assert got["status"] == 0
    H.compare_all_rows(wl, w, layer, x, got)


@pytest.mark.parametrize("i", [1, 2], ids=["T16", "T512"])
def test_nvfp4_stages_against_fp64(i):
    """h and the down projection of every slot, each against FP64 fed the same inputs."""
    wl, w, layer = H.device_layer(synth.WORKLOADS_NVFP4[i])
    x = synth.make_x(wl.shape, wl.tokens, wl.seed)
    H.check_stages_against_fp64(wl, w, layer, x, qm.MOE_PATH_PREFILL)


@pytest.mark.parametrize("path", [qm.MOE_PATH_DECODE, qm.MOE_PATH_PREFILL], ids=["decode", "prefill"])
def test_nvfp4_rows_beyond_fp16_range(path):
    """Rows with max |x| of 1e3, 7e4 and 1e6, one below 2^-14 and an ordinary one."""
    wl, w, layer = H.device_layer(synth.WORKLOADS_NVFP4[1])
    x = H.range_rows(wl.shape, wl.seed)
    lg = oracle.router_logits(wl.shape, w, x)           # routing pinned: the rows' logits are large
    got = H.run_forward(layer, x, path=path, logits_in=lg)
    assert got["status"] == 0
    ref = oracle.forward(wl.shape, w, x, logits_in=lg)
    assert np.array_equal(got["ids"], ref["ids"])
    H.check_rows_scale_free(got["y"], ref["y"])
