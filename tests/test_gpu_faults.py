"""Device-side failure handling without a GPU fault.

The in-kernel waits are bounded by the call's moe_config.wait_polls (in the
fused decode kernel: its waits on other CTAs; a CTA's waits on its own copies
keep a fixed bound).  A bound of one poll makes those waits run out before the
other CTAs arrive: the kernels must record MOE_ERR_TIMEOUT in the workspace
status word, drain what they issued, free their TMEM and return, leaving the
context usable.  Nothing here traps, faults or hangs the GPU.
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


def test_prefill_wait_limit_runs_out_then_recovers():
    wl, w, layer = H.device_layer(0)
    x = synth.make_x(wl.shape, 40, wl.seed, stream=9)
    got = H.run_forward(layer, x, path=qm.MOE_PATH_PREFILL, cfg=qm.config_of(wl.shape, wait_polls=1))
    assert got["status"] == qm.MOE_ERR_TIMEOUT
    again = H.run_forward(layer, x, path=qm.MOE_PATH_PREFILL)
    assert again["status"] == 0
    ref = oracle.forward(wl.shape, w, x)
    assert np.array_equal(again["ids"], ref["ids"])
    H.check_y(again["y"], ref["y"])


@pytest.mark.parametrize("T", [1, 16])
def test_decode_wait_limit_runs_out_then_recovers(T):
    """One poll: the first CTAs at the router counter cannot find every other CTA there yet."""
    wl, w, layer = H.device_layer(2)
    x = synth.make_x(wl.shape, T, wl.seed, stream=9)
    got = H.run_forward(layer, x, path=qm.MOE_PATH_DECODE, cfg=qm.config_of(wl.shape, wait_polls=1))
    assert got["status"] == qm.MOE_ERR_TIMEOUT
    again = H.run_forward(layer, x, path=qm.MOE_PATH_DECODE)
    assert again["status"] == 0
    ref = oracle.forward(wl.shape, w, x)
    same = np.all(again["ids"] == ref["ids"], axis=1)
    H.check_y(again["y"], ref["y"], rows=np.nonzero(same)[0])


def test_decode_workspace_reused_after_timeout():
    """A call that timed out leaves the workspace's counters zero: the next call on it is correct."""
    wl, w, layer = H.device_layer(1)
    x = H.to_dev_u16(synth.make_x(wl.shape, 1, wl.seed, stream=10))
    ws = qm.workspace(layer.cfg, 1)
    qm.forward(layer, x, ws, path=qm.MOE_PATH_DECODE, cfg=qm.config_of(wl.shape, wait_polls=1))
    torch.cuda.synchronize()
    hdr = ws[:512].view(torch.int32).cpu().numpy()
    assert hdr[0] == qm.MOE_ERR_TIMEOUT                             # status set
    assert hdr[64] == 0 and hdr[96] == 0                            # counters back to zero
    assert hdr[120] == 1                                            # the launch's epoch, advanced at exit
    y1 = qm.forward(layer, x, ws, path=qm.MOE_PATH_DECODE)
    torch.cuda.synchronize()
    assert qm.moe_get_device_status(ws) == qm.MOE_ERR_TIMEOUT     # the earlier call's status, kept until read
    y2 = qm.forward(layer, x, ws, path=qm.MOE_PATH_DECODE)
    torch.cuda.synchronize()
    assert qm.moe_get_device_status(ws) == 0
    assert torch.equal(y1, y2)


def test_decode_dirty_header_is_reported():
    """A workspace whose header was not zero-filled is reported, not silently used."""
    wl, w, layer = H.device_layer(0)
    x = H.to_dev_u16(synth.make_x(wl.shape, 2, wl.seed, stream=12))
    ws = qm.workspace(layer.cfg, 2)
    ws[:512].view(torch.int32)[1:].fill_(0x33333333)
    qm.forward(layer, x, ws, path=qm.MOE_PATH_DECODE, cfg=qm.config_of(wl.shape, wait_polls=64))
    assert qm.moe_get_device_status(ws) in (qm.MOE_ERR_WORKSPACE, qm.MOE_ERR_TIMEOUT)
    y = qm.forward(layer, x, ws, path=qm.MOE_PATH_DECODE)            # the status read reset the header
    assert qm.moe_get_device_status(ws) == 0


def test_bad_expert_ids_are_reported_not_trapped():
    """Out-of-range ids given to moe_permute set MOE_ERR_DEVICE; nothing is written out of bounds."""
    wl, w, layer = H.device_layer(0)
    T, k, E = 8, wl.shape.top_k, wl.shape.n_experts
    ids = np.tile(np.arange(k, dtype=np.int32), (T, 1))
    ids[3, 1] = E + 5
    ids[5, 0] = -2
    ws = qm.workspace(layer.cfg, T)
    guard = 1024
    buf = torch.full((T * k + 2 * guard,), -7, dtype=torch.int32, device="cuda")
    perm = buf[guard:guard + T * k]
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    inv = torch.empty(T * k, dtype=torch.int32, device="cuda")
    qm.moe_permute(layer.cfg, torch.from_numpy(ids).cuda(), T, counts, offsets, perm, inv, ws)
    torch.cuda.synchronize()
    assert qm.moe_get_device_status(ws) == qm.MOE_ERR_DEVICE
    b = buf.cpu()
    assert torch.all(b[:guard] == -7) and torch.all(b[guard + T * k:] == -7)
