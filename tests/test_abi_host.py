"""Host-side checks of the C ABI: the library builds and loads, exports every
declared entry point, and refuses bad arguments before touching the GPU.

No test here enqueues GPU work: every call below fails validation (or has
T == 0) and returns before any CUDA call, so the suite runs without a GPU.
The fake device pointers are never dereferenced.
"""
import ctypes
import os
import re
import subprocess

import pytest

import quantised_moe_expert_gb300 as qm
from quantised_moe_expert_gb300 import synth

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe.h")
FAKE = 0x7f0000010000          # 16-byte aligned, never dereferenced
MISALIGNED = FAKE + 8


@pytest.fixture(scope="module")
def lib():
    return qm.load()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"MOE_API\s+[\w\s\*]*?\b(moe_\w+)\s*\(", text)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10
    assert set(names) == set(qm.EXPORTED)
    out = subprocess.run(["nm", "-D", "--defined-only", qm.library_path()], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (moe_\w+)", out))
    for n in names:
        assert n in exported, n
        assert hasattr(lib, n)


def test_status_strings(lib):
    for code in range(7):
        assert lib.moe_status_string(code)
    assert lib.moe_status_string(99) == b"unknown status"


def cfg_from(**kw):
    d = dict(hidden=2048, inter=512, n_experts=256, top_k=8, group=64, bits=4, router_bits=8, has_shared=1,
             wait_polls=0)
    d.update(kw)
    return qm.moe_config(**d)


@pytest.mark.parametrize("kw,expect", [
    ({}, qm.MOE_OK),
    (dict(hidden=256, inter=64, n_experts=16, top_k=2), qm.MOE_OK),
    (dict(has_shared=0), qm.MOE_OK),
    (dict(bits=8), qm.MOE_OK),
    (dict(bits=2), qm.MOE_ERR_UNSUPPORTED),
    (dict(bits=6), qm.MOE_ERR_UNSUPPORTED),
    (dict(group=32), qm.MOE_ERR_UNSUPPORTED),
    (dict(router_bits=4), qm.MOE_ERR_UNSUPPORTED),
    (dict(hidden=100), qm.MOE_ERR_UNSUPPORTED),
    (dict(inter=96), qm.MOE_ERR_UNSUPPORTED),
    (dict(n_experts=300), qm.MOE_ERR_UNSUPPORTED),
    (dict(top_k=17), qm.MOE_ERR_UNSUPPORTED),
    (dict(n_experts=4, top_k=5), qm.MOE_ERR_UNSUPPORTED),
    (dict(has_shared=2), qm.MOE_ERR_UNSUPPORTED),
    (dict(format=qm.MOE_FORMAT_NVFP4), qm.MOE_OK),
    (dict(format=qm.MOE_FORMAT_NVFP4, bits=8), qm.MOE_ERR_UNSUPPORTED),
    (dict(format=2), qm.MOE_ERR_UNSUPPORTED),
    (dict(format=-1), qm.MOE_ERR_UNSUPPORTED),
    (dict(hidden=0), qm.MOE_ERR_INVALID_ARG),
    (dict(top_k=-1), qm.MOE_ERR_INVALID_ARG),
])
def test_check_config(lib, kw, expect):
    assert lib.moe_check_config(ctypes.byref(cfg_from(**kw))) == expect


def test_workspace_size(lib):
    cfg = cfg_from()
    n = ctypes.c_size_t()
    sizes = []
    for T in (0, 1, 16, 512, 4096, 65536):
        assert lib.moe_workspace_size(ctypes.byref(cfg), T, ctypes.byref(n)) == qm.MOE_OK
        sizes.append(n.value)
    assert sizes == sorted(sizes) and sizes[0] > 0
    assert lib.moe_workspace_size(ctypes.byref(cfg), -1, ctypes.byref(n)) == qm.MOE_ERR_INVALID_ARG
    assert lib.moe_workspace_size(ctypes.byref(cfg), 65537, ctypes.byref(n)) == qm.MOE_ERR_INVALID_ARG
    assert lib.moe_workspace_size(ctypes.byref(cfg), 1, None) == qm.MOE_ERR_INVALID_ARG
    assert lib.moe_workspace_size(None, 1, ctypes.byref(n)) == qm.MOE_ERR_INVALID_ARG


def fake_weights(misalign=None):
    q = lambda: qm.moe_qmat(FAKE, FAKE, FAKE)
    w = qm.moe_weights(q(), q(), q(), q(), q(), q(), q(), FAKE)
    if misalign:
        getattr(w, misalign).codes = MISALIGNED
    return w


def forward(lib, cfg, w, T=1, x=FAKE, y=FAKE, ws=FAKE, ws_bytes=1 << 40, path=0, logits_in=None):
    return lib.moe_forward(ctypes.byref(cfg), ctypes.byref(w) if w is not None else None, x, T, None, logits_in,
                           y, None, None, None, path, ws, ws_bytes, None)


def test_forward_rejects_bad_arguments(lib):
    cfg, w = cfg_from(), fake_weights()
    assert forward(lib, cfg, None) == qm.MOE_ERR_INVALID_ARG
    assert forward(lib, cfg, w, x=None) == qm.MOE_ERR_INVALID_ARG
    assert forward(lib, cfg, w, x=MISALIGNED) == qm.MOE_ERR_INVALID_ARG
    assert forward(lib, cfg, w, y=MISALIGNED) == qm.MOE_ERR_INVALID_ARG
    assert forward(lib, cfg, w, ws=MISALIGNED) == qm.MOE_ERR_INVALID_ARG
    assert forward(lib, cfg, w, T=-3) == qm.MOE_ERR_INVALID_ARG
    assert forward(lib, cfg, w, path=7) == qm.MOE_ERR_INVALID_ARG
    for m in ("gate", "up", "down", "s_gate", "router"):
        assert forward(lib, cfg, fake_weights(m)) == qm.MOE_ERR_INVALID_ARG, m
    # the router is not needed when logits are supplied
    assert forward(lib, cfg, fake_weights("router"), T=0, logits_in=FAKE) == qm.MOE_OK
    assert forward(lib, cfg_from(bits=3), w) == qm.MOE_ERR_UNSUPPORTED


def test_nvfp4_weights_need_the_matrix_scales(lib):
    """NVFP4 expert matrices carry a 4-byte aligned fp32 scale per matrix; biases may be NULL."""
    cfg = cfg_from(format=qm.MOE_FORMAT_NVFP4)
    q = lambda g: qm.moe_qmat(FAKE, FAKE, None, g)
    w = qm.moe_weights(qm.moe_qmat(FAKE, FAKE, FAKE), q(FAKE), q(FAKE), q(FAKE), q(FAKE), q(FAKE), q(FAKE), FAKE)
    assert forward(lib, cfg, w, T=0) == qm.MOE_OK                          # checks pass, nothing enqueued
    for m in ("gate", "up", "down", "s_gate", "s_up", "s_down"):
        bad = qm.moe_weights(*[getattr(w, n) for n in ("router", "gate", "up", "down", "s_gate", "s_up", "s_down")],
                             FAKE)
        getattr(bad, m).gscale = None
        assert forward(lib, cfg, bad, T=0) == qm.MOE_ERR_INVALID_ARG, m
        getattr(bad, m).gscale = FAKE + 2
        assert forward(lib, cfg, bad, T=0) == qm.MOE_ERR_INVALID_ARG, m
    # the affine rule still wants its biases
    assert forward(lib, cfg_from(), w, T=0) == qm.MOE_ERR_INVALID_ARG


def test_forward_workspace_too_small(lib):
    cfg, w = cfg_from(), fake_weights()
    need = qm.moe_workspace_size(cfg, 16)
    assert forward(lib, cfg, w, T=16, ws_bytes=need - 1) == qm.MOE_ERR_WORKSPACE
    assert forward(lib, cfg, w, T=0, ws_bytes=need) == qm.MOE_OK      # T == 0 enqueues nothing


def test_other_entry_points_reject_bad_arguments(lib):
    cfg, w = cfg_from(), fake_weights()
    big = 1 << 40
    assert lib.moe_route(ctypes.byref(cfg), ctypes.byref(w), FAKE, 4, None, None, None, None, FAKE, FAKE, FAKE,
                         big, None) == qm.MOE_ERR_INVALID_ARG                     # ids missing
    assert lib.moe_route(ctypes.byref(cfg), ctypes.byref(w), FAKE, 4, MISALIGNED, None, None, FAKE, FAKE, FAKE,
                         FAKE, big, None) == qm.MOE_ERR_INVALID_ARG               # misaligned bias
    assert lib.moe_route(ctypes.byref(cfg), ctypes.byref(w), FAKE, 4, None, None, None, FAKE, FAKE, FAKE,
                         FAKE, 16, None) == qm.MOE_ERR_WORKSPACE
    assert lib.moe_permute(ctypes.byref(cfg), None, 4, FAKE, FAKE, FAKE, FAKE, FAKE, big, None) == \
        qm.MOE_ERR_INVALID_ARG
    assert lib.moe_expert_ffn(ctypes.byref(cfg), ctypes.byref(w), FAKE, 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                              MISALIGNED, 0, FAKE, big, None) == qm.MOE_ERR_INVALID_ARG
    assert lib.moe_expert_ffn(ctypes.byref(cfg), ctypes.byref(w), FAKE, 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                              FAKE, 3, FAKE, big, None) == qm.MOE_ERR_INVALID_ARG
    assert lib.moe_combine(ctypes.byref(cfg), 4, None, FAKE, None) == qm.MOE_ERR_INVALID_ARG
    assert lib.moe_combine(ctypes.byref(cfg), 0, FAKE, FAKE, None) == qm.MOE_OK
    st = ctypes.c_int()
    assert lib.moe_get_device_status(None, big, None, ctypes.byref(st)) == qm.MOE_ERR_INVALID_ARG
    assert lib.moe_get_device_status(FAKE, 8, None, ctypes.byref(st)) == qm.MOE_ERR_INVALID_ARG
    assert lib.moe_get_device_status(FAKE, 256, None, ctypes.byref(st)) == qm.MOE_ERR_INVALID_ARG   # header is 512 B
    # stage outputs: misaligned h_out, bad path, too small a workspace; T == 0 or no outputs enqueue nothing
    assert lib.moe_expert_stages(ctypes.byref(cfg), ctypes.byref(w), FAKE, 4, FAKE, FAKE, FAKE, FAKE, MISALIGNED,
                                 None, 0, FAKE, big, None) == qm.MOE_ERR_INVALID_ARG
    assert lib.moe_expert_stages(ctypes.byref(cfg), ctypes.byref(w), FAKE, 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 9,
                                 FAKE, big, None) == qm.MOE_ERR_INVALID_ARG
    assert lib.moe_expert_stages(ctypes.byref(cfg), ctypes.byref(w), FAKE, 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0,
                                 FAKE, 16, None) == qm.MOE_ERR_WORKSPACE
    assert lib.moe_expert_stages(ctypes.byref(cfg), ctypes.byref(w), FAKE, 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0,
                                 FAKE, big, None) == qm.MOE_OK
    assert lib.moe_expert_stages(ctypes.byref(cfg), ctypes.byref(w), FAKE, 4, FAKE, FAKE, FAKE, FAKE, None, None, 0,
                                 FAKE, big, None) == qm.MOE_OK
    assert lib.moe_pack_down(ctypes.byref(cfg), ctypes.byref(w), MISALIGNED, None, None) == qm.MOE_ERR_INVALID_ARG
    assert lib.moe_pack_down(ctypes.byref(cfg), ctypes.byref(fake_weights("down")), FAKE, None, None) == \
        qm.MOE_ERR_INVALID_ARG
    # the decode layout of the down codes is for 4-bit codes (the fused decode kernel reads it)
    assert lib.moe_pack_down(ctypes.byref(cfg_from(bits=8)), ctypes.byref(w), FAKE, None, None) == \
        qm.MOE_ERR_UNSUPPORTED
    bad = fake_weights()
    bad.down_packed = MISALIGNED
    assert forward(lib, cfg, bad) == qm.MOE_ERR_INVALID_ARG
    n = ctypes.c_int()
    assert lib.moe_decode_timeline(ctypes.byref(cfg), 1, FAKE, big, None, None, 4, ctypes.byref(n)) == \
        qm.MOE_ERR_INVALID_ARG
    assert lib.moe_decode_timeline(ctypes.byref(cfg), 1, FAKE, 16, None, FAKE, 4, ctypes.byref(n)) == \
        qm.MOE_ERR_WORKSPACE


def test_wait_limit_is_a_field_of_the_call_config(lib):
    """The bound on in-kernel waits travels with each call (no process-wide setting)."""
    names = [f[0] for f in qm.moe_config._fields_]
    assert "wait_polls" in names
    assert lib.moe_check_config(ctypes.byref(cfg_from(wait_polls=1))) == qm.MOE_OK
    assert lib.moe_check_config(ctypes.byref(cfg_from(wait_polls=-5))) == qm.MOE_OK
    assert "moe_set_wait_limit" not in open(HEADER).read()


def test_python_binding_has_every_entry_point():
    for n in qm.EXPORTED:
        if n not in ("moe_status_string",):
            assert callable(getattr(qm, n)), n


def test_workloads_match_layer_shapes():
    assert [wl.tokens for wl in synth.WORKLOADS] == [4, 1, 16, 512, 4096]
    s = synth.QWEN_SHAPE
    assert (s.hidden, s.inter, s.n_experts, s.top_k) == (2048, 512, 256, 8)
    assert synth.active_expert_bytes(s) == 1769472
    assert synth.router_bytes(s) == 524288 + 32768 + 4096
