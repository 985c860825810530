"""GPU parity of the layer with 8-bit expert codes against the FP64 oracle.

8-bit experts are the slice "8-bit experts" of the page "Qwen3.6-35B-A3B
(qwen3_5_moe) on the native Metal engine: proposal and gate": the same MLX
affine rule (group 64, bf16 scale and bias) with codes q in 0..255.  At
T <= 16 the layer runs on the weight-streaming decode kernels (the fused decode
kernel takes 4-bit codes only), above on the tensor-memory grouped GEMMs (all
items, the small-tile kernels take 4-bit codes only).  Every row is compared.
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

TINY_B8 = synth.Workload("tiny_T4_H256_E16_k2_b8", dataclasses.replace(synth.TINY_SHAPE, bits=8), 4, seed=10)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    qm.load()
    oracle.build()


@pytest.mark.parametrize("i", range(len(synth.WORKLOADS_B8)), ids=[wl.name for wl in synth.WORKLOADS_B8])
def test_b8_forward_every_row(i):
    """T = 1, 16 (decode kernels) and 512 (grouped GEMMs): ids, p, w_s and y on every row."""
    wl, w, layer = H.device_layer(synth.WORKLOADS_B8[i])
    x = synth.make_x(wl.shape, wl.tokens, wl.seed)
    got = H.run_forward(layer, x, path=qm.MOE_PATH_AUTO)
    assert got["status"] == 0
    stats, ndiff = H.compare_all_rows(wl, w, layer, x, got)
    print(wl.name, stats, "near-tie rows", ndiff)
    assert ndiff <= 2


@pytest.mark.parametrize("path", [qm.MOE_PATH_DECODE, qm.MOE_PATH_PREFILL], ids=["decode", "prefill"])
@pytest.mark.parametrize("T", [1, 3, 17, 40, 129])
def test_b8_ragged_token_counts_small_layer(T, path):
    """A small 8-bit layer (I = 64: a weight tile half past the expert's rows) at ragged token counts."""
    wl, w, layer = H.device_layer(TINY_B8)
    x = synth.make_x(wl.shape, T, wl.seed, stream=T)
    got = H.run_forward(layer, x, path=path)
    assert got["status"] == 0
    H.compare_rows(wl, w, x, got, np.arange(T))


@pytest.mark.parametrize("T", [1, 16])
def test_b8_prefill_path_at_decode_sizes(T):
    """The grouped GEMMs at one 16-column tile per expert give the oracle's rows too."""
    wl, w, layer = H.device_layer(synth.WORKLOADS_B8[1])
    x = synth.make_x(wl.shape, T, wl.seed, stream=50 + T)
    got = H.run_forward(layer, x, path=qm.MOE_PATH_PREFILL)
    assert got["status"] == 0
    H.compare_all_rows(wl, w, layer, x, got)


def test_b8_prefill_stages_against_fp64():
    """h and the down projection of every slot of the 8-bit T = 512 layer, each against FP64."""
    wl, w, layer = H.device_layer(synth.WORKLOADS_B8[2])
    x = synth.make_x(wl.shape, wl.tokens, wl.seed)
    H.check_stages_against_fp64(wl, w, layer, x, qm.MOE_PATH_PREFILL)


@pytest.mark.parametrize("path", [qm.MOE_PATH_DECODE, qm.MOE_PATH_PREFILL], ids=["decode", "prefill"])
def test_b8_rows_beyond_fp16_range(path):
    """Rows with max |x| of 1e3, 7e4 and 1e6, one below 2^-14 and an ordinary one."""
    wl, w, layer = H.device_layer(synth.WORKLOADS_B8[1])
    x = H.range_rows(wl.shape, wl.seed)
    lg = oracle.router_logits(wl.shape, w, x)           # routing pinned: the rows' logits are large
    got = H.run_forward(layer, x, path=path, logits_in=lg)
    assert got["status"] == 0
    ref = oracle.forward(wl.shape, w, x, logits_in=lg)
    assert np.array_equal(got["ids"], ref["ids"])
    H.check_rows_scale_free(got["y"], ref["y"])
