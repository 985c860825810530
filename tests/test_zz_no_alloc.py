"""The decode entry point without a workspace, for callers that cannot allocate.

Runs through the C ABI and compares with moe_forward (which takes a caller
workspace) on two calls in a row, within the parity tolerance of the other
tests.  The file sorts last so that a run stopping at its first failure has
already run every other test.
"""
import numpy as np
import pytest
import torch

import quantised_moe_expert_gb300 as qm
from quantised_moe_expert_gb300 import synth

from . import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    qm.load()


@pytest.mark.parametrize("wl_index,T", [(1, 1), (2, 16), (2, 5)])
def test_static_scratch_decode_matches_workspace_decode(wl_index, T):
    wl, w, layer = H.device_layer(wl_index)
    sh = wl.shape
    x = H.to_dev_u16(synth.make_x(sh, T, wl.seed, stream=11))
    ws = qm.workspace(layer.cfg, T)
    y_ref = torch.empty((T, sh.hidden), dtype=torch.int16, device="cuda")
    ids_ref = torch.empty((T, sh.top_k), dtype=torch.int32, device="cuda")
    qm.moe_forward(layer.cfg, layer.w, x, T, None, None, y_ref, ids_ref, None, None, qm.MOE_PATH_DECODE, ws)
    torch.cuda.synchronize()
    assert qm.moe_get_device_status(ws) == 0
    for _ in range(2):                                  # two calls in a row share the static scratch
        y = torch.full((T, sh.hidden), -1, dtype=torch.int16, device="cuda")
        ids = torch.full((T, sh.top_k), -1, dtype=torch.int32, device="cuda")
        qm.moe_forward_decode_static(layer.cfg, layer.w, x, T, None, None, y, ids, None, None)
        torch.cuda.synchronize()
        assert np.array_equal(ids.cpu().numpy(), ids_ref.cpu().numpy())
        H.check_y(H.u16(y), H.u16(y_ref))


def test_static_scratch_refuses_layers_beyond_its_size():
    """A layer whose decode scratch exceeds the fixed array is refused before anything is enqueued."""
    wl, w, layer = H.device_layer(1)
    big = qm.moe_config(8192, 4096, 256, 16, 64, 4, 8, 1, 0)
    assert qm.moe_workspace_size(big, 16) > 24 << 20
    x = torch.zeros((16, 8192), dtype=torch.int16, device="cuda")
    y = torch.full((16, 8192), 7, dtype=torch.int16, device="cuda")
    with pytest.raises(qm.MoeError) as e:
        qm.moe_forward_decode_static(big, layer.w, x, 16, None, None, y, None, None, None)
    assert e.value.status == qm.MOE_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(y == 7)


def test_static_scratch_zero_tokens_is_a_no_op():
    wl, w, layer = H.device_layer(1)
    x = torch.zeros((1, wl.shape.hidden), dtype=torch.int16, device="cuda")
    y = torch.full((1, wl.shape.hidden), 7, dtype=torch.int16, device="cuda")
    qm.moe_forward_decode_static(layer.cfg, layer.w, x, 0, None, None, y, None, None, None)
    torch.cuda.synchronize()
    assert torch.all(y == 7)


def test_static_scratch_refuses_prefill_sizes():
    wl, w, layer = H.device_layer(1)
    x = torch.zeros((17, wl.shape.hidden), dtype=torch.int16, device="cuda")
    y = torch.empty_like(x)
    with pytest.raises(qm.MoeError) as e:
        qm.moe_forward_decode_static(layer.cfg, layer.w, x, 17, None, None, y, None, None, None)
    assert e.value.status == qm.MOE_ERR_INVALID_ARG
