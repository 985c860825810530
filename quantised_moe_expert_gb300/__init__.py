"""GB300 (sm_103a) routed-expert MoE layer of the qwen3_5_moe family.

This package is a thin Python binding of ``libmoe.so`` (the C ABI declared in
``include/moe.h``).  Every function named ``moe_*`` here marshals torch tensors
(device memory and streams only) into the C call of the same name; all of the
layer's arithmetic runs in the library's CUDA kernels.  There is no CPU
fallback: without the built library or a CUDA device the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import numpy as np
import torch

from . import _build

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_DEVICE = 6

MOE_PATH_AUTO = 0
MOE_PATH_DECODE = 1
MOE_PATH_PREFILL = 2

MOE_FORMAT_AFFINE = 0
MOE_FORMAT_NVFP4 = 1

EXPORTED = ("moe_status_string", "moe_check_config", "moe_workspace_size", "moe_route", "moe_permute",
            "moe_expert_ffn", "moe_combine", "moe_forward", "moe_get_device_status", "moe_pack_down",
            "moe_expert_stages",
            "moe_decode_timeline", "moe_forward_decode_static")


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {status_string(status)} (status {status})")
        self.status = status


class moe_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("hidden", "inter", "n_experts", "top_k", "group", "bits", "router_bits", "has_shared",
                 "wait_polls", "format")]


class moe_qmat(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("biases", ctypes.c_void_p),
                ("gscale", ctypes.c_void_p)]


class moe_weights(ctypes.Structure):
    _fields_ = [(n, moe_qmat) for n in ("router", "gate", "up", "down", "s_gate", "s_up", "s_down")] + \
               [("shared_gate_vec", ctypes.c_void_p), ("down_packed", ctypes.c_void_p),
                ("s_down_packed", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None

_VP = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t


def library_path() -> str:
    return _build.LIB


def load(build: bool = True):
    """Load libmoe.so (building it with nvcc first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build:
            _build.build()
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"libmoe.so not built ({_build.LIB}); run quantised_moe_expert_gb300._build")
        lib = ctypes.CDLL(_build.LIB)
        P = ctypes.POINTER
        lib.moe_status_string.restype = ctypes.c_char_p
        lib.moe_status_string.argtypes = [_I]
        lib.moe_check_config.argtypes = [P(moe_config)]
        lib.moe_workspace_size.argtypes = [P(moe_config), _I, P(ctypes.c_size_t)]
        lib.moe_route.argtypes = [P(moe_config), P(moe_weights), _VP, _I, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]
        lib.moe_permute.argtypes = [P(moe_config), _VP, _I, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]
        lib.moe_expert_ffn.argtypes = [P(moe_config), P(moe_weights), _VP, _I, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                       _I, _VP, _SZ, _VP]
        lib.moe_combine.argtypes = [P(moe_config), _I, _VP, _VP, _VP]
        lib.moe_forward.argtypes = [P(moe_config), P(moe_weights), _VP, _I, _VP, _VP, _VP, _VP, _VP, _VP, _I, _VP,
                                    _SZ, _VP]
        lib.moe_get_device_status.argtypes = [_VP, _SZ, _VP, P(ctypes.c_int)]
        lib.moe_pack_down.argtypes = [P(moe_config), P(moe_weights), _VP, _VP, _VP]
        lib.moe_expert_stages.argtypes = [P(moe_config), P(moe_weights), _VP, _I, _VP, _VP, _VP, _VP, _VP, _VP, _I,
                                          _VP, _SZ, _VP]
        lib.moe_decode_timeline.argtypes = [P(moe_config), _I, _VP, _SZ, _VP, _VP, _I, P(ctypes.c_int)]
        lib.moe_forward_decode_static.argtypes = [P(moe_config), P(moe_weights), _VP, _I, _VP, _VP, _VP, _VP, _VP,
                                                  _VP, _VP]
        for name in EXPORTED:
            if name != "moe_status_string":
                getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load(build=False).moe_status_string(status).decode() if _lib is not None else f"status {status}"


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(fn: str, rc: int):
    if rc != MOE_OK:
        raise MoeError(fn, rc)


def config_of(shape, wait_polls: int = 0) -> moe_config:
    """moe_config from any object with the layer-shape attributes (e.g. synth.LayerShape)."""
    fmt = MOE_FORMAT_NVFP4 if getattr(shape, "fmt", "affine") == "nvfp4" else MOE_FORMAT_AFFINE
    return moe_config(shape.hidden, shape.inter, shape.n_experts, shape.top_k, shape.group, shape.bits,
                      shape.router_bits, shape.has_shared, wait_polls, fmt)


def _ptr(t):
    return None if t is None or t.numel() == 0 else t.data_ptr()


class DeviceLayer:
    """One layer's weights resident on a CUDA device, plus the C weight struct.

    pack=True also makes the decode layout of the down codes (moe_pack_down) and hands it to the
    library in moe_weights.down_packed / s_down_packed (4-bit experts only: the layout and the fused
    decode kernel that reads it are for 4-bit codes)."""

    def __init__(self, host, device="cuda", pack: bool = True):
        self.shape = host.shape
        self.cfg = config_of(host.shape)
        self.tensors = {}

        def up(name, arr):
            arr = np.ascontiguousarray(arr)
            if arr.dtype == np.uint16:
                arr = arr.view(np.int16)
            t = torch.from_numpy(arr).to(device)
            self.tensors[name] = t
            return t

        def q(name, m):
            c = up(name + ".codes", m.codes)
            s = up(name + ".scales", m.scales)
            b = up(name + ".biases", m.biases)
            g = None if m.gscale is None else up(name + ".gscale", m.gscale)
            return moe_qmat(c.data_ptr(), s.data_ptr(), _ptr(b), _ptr(g))

        self.w = moe_weights(q("router", host.router), q("gate", host.gate), q("up", host.up),
                             q("down", host.down), q("s_gate", host.s_gate), q("s_up", host.s_up),
                             q("s_down", host.s_down), up("v", host.shared_gate_vec).data_ptr(), None, None)
        if pack and host.shape.bits == 4 and getattr(host.shape, "fmt", "affine") == "affine":
            self.pack()

    def pack(self):
        """The decode layout of the down codes, made on the device by moe_pack_down."""
        d, sd = self.tensors["down.codes"], self.tensors["s_down.codes"]
        dp = torch.empty_like(d)
        sdp = torch.empty_like(sd) if self.shape.has_shared else None
        moe_pack_down(self.cfg, self.w, dp, sdp)
        self.tensors["down.packed"] = dp
        self.w.down_packed = dp.data_ptr()
        if sdp is not None:
            self.tensors["s_down.packed"] = sdp
            self.w.s_down_packed = sdp.data_ptr()

    def unpacked(self) -> "DeviceLayer":
        """The same layer without the packed down codes (the decode kernel gathers from the MLX layout)."""
        t = {k: v for k, v in self.tensors.items() if not k.endswith(".packed")}
        return DeviceLayer.from_tensors(self.shape, t)

    @staticmethod
    def from_tensors(shape, tensors):
        """Wrap device tensors already laid out as the C ABI expects (same keys as ``tensors``)."""
        obj = DeviceLayer.__new__(DeviceLayer)
        obj.shape = shape
        obj.cfg = config_of(shape)
        obj.tensors = tensors

        def q(name):
            return moe_qmat(tensors[name + ".codes"].data_ptr(), tensors[name + ".scales"].data_ptr(),
                            _ptr(tensors[name + ".biases"]), _ptr(tensors.get(name + ".gscale")))
        opt = lambda name: tensors[name].data_ptr() if name in tensors else None
        obj.w = moe_weights(q("router"), q("gate"), q("up"), q("down"), q("s_gate"), q("s_up"), q("s_down"),
                            tensors["v"].data_ptr(), opt("down.packed"), opt("s_down.packed"))
        return obj


# ---------------------------------------------------------------- C ABI, same names

def moe_check_config(cfg: moe_config) -> int:
    return load().moe_check_config(ctypes.byref(cfg))


def moe_workspace_size(cfg: moe_config, T: int) -> int:
    n = ctypes.c_size_t(0)
    _check("moe_workspace_size", load().moe_workspace_size(ctypes.byref(cfg), T, ctypes.byref(n)))
    return n.value


def moe_route(cfg, w, x, T, router_bias, logits_in, logits_out, ids, p, w_shared, ws, stream=None):
    rc = load().moe_route(ctypes.byref(cfg), ctypes.byref(w), _ptr(x), T, _ptr(router_bias), _ptr(logits_in),
                          _ptr(logits_out), _ptr(ids), _ptr(p), _ptr(w_shared), _ptr(ws),
                          ws.numel() * ws.element_size(), _stream(stream))
    _check("moe_route", rc)


def moe_permute(cfg, ids, T, counts, offsets, perm, inv_perm, ws, stream=None):
    rc = load().moe_permute(ctypes.byref(cfg), _ptr(ids), T, _ptr(counts), _ptr(offsets), _ptr(perm),
                            _ptr(inv_perm), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check("moe_permute", rc)


def moe_expert_ffn(cfg, w, x, T, ids, p, w_shared, counts, offsets, perm, acc, path, ws, stream=None):
    rc = load().moe_expert_ffn(ctypes.byref(cfg), ctypes.byref(w), _ptr(x), T, _ptr(ids), _ptr(p), _ptr(w_shared),
                               _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(acc), path, _ptr(ws),
                               ws.numel() * ws.element_size(), _stream(stream))
    _check("moe_expert_ffn", rc)


def moe_combine(cfg, T, acc, y, stream=None):
    _check("moe_combine", load().moe_combine(ctypes.byref(cfg), T, _ptr(acc), _ptr(y), _stream(stream)))


def moe_forward(cfg, w, x, T, router_bias, logits_in, y, ids_out, p_out, w_shared_out, path, ws, stream=None):
    rc = load().moe_forward(ctypes.byref(cfg), ctypes.byref(w), _ptr(x), T, _ptr(router_bias), _ptr(logits_in),
                            _ptr(y), _ptr(ids_out), _ptr(p_out), _ptr(w_shared_out), path, _ptr(ws),
                            ws.numel() * ws.element_size(), _stream(stream))
    _check("moe_forward", rc)


def moe_forward_decode_static(cfg, w, x, T, router_bias, logits_in, y, ids_out, p_out, w_shared_out, stream=None):
    """Decode layer (T <= 16) without a workspace, for callers that cannot allocate device memory.

    The scratch is a fixed array inside libmoe.so's device memory, shared by
    every call: keep calls ordered on the GPU (overlapping calls race).  The
    first call on a device must come before any stream capture.
    """
    rc = load().moe_forward_decode_static(ctypes.byref(cfg), ctypes.byref(w), _ptr(x), T, _ptr(router_bias),
                                          _ptr(logits_in), _ptr(y), _ptr(ids_out), _ptr(p_out), _ptr(w_shared_out),
                                          _stream(stream))
    _check("moe_forward_decode_static", rc)


def moe_get_device_status(ws, stream=None) -> int:
    st = ctypes.c_int(0)
    _check("moe_get_device_status", load().moe_get_device_status(_ptr(ws), ws.numel() * ws.element_size(),
                                                                 _stream(stream), ctypes.byref(st)))
    return st.value


def moe_pack_down(cfg, w, down_packed, s_down_packed=None, stream=None):
    rc = load().moe_pack_down(ctypes.byref(cfg), ctypes.byref(w), _ptr(down_packed), _ptr(s_down_packed),
                              _stream(stream))
    _check("moe_pack_down", rc)


def moe_expert_stages(cfg, w, x, T, ids, counts, offsets, perm, h_out, yslot_out, path, ws, stream=None):
    rc = load().moe_expert_stages(ctypes.byref(cfg), ctypes.byref(w), _ptr(x), T, _ptr(ids), _ptr(counts),
                                  _ptr(offsets), _ptr(perm), _ptr(h_out), _ptr(yslot_out), path, _ptr(ws),
                                  ws.numel() * ws.element_size(), _stream(stream))
    _check("moe_expert_stages", rc)


def moe_decode_timeline(cfg, T, ws, stream=None, max_ctas: int = 256) -> np.ndarray:
    """Per-CTA %globaltimer stamps (ns) of the last fused decode launch on ws: [n_ctas, 14] uint64."""
    buf = np.zeros((max_ctas, 14), dtype=np.uint64)
    n = ctypes.c_int(0)
    rc = load().moe_decode_timeline(ctypes.byref(cfg), T, _ptr(ws), ws.numel() * ws.element_size(),
                                    _stream(stream), ctypes.c_void_p(buf.ctypes.data), max_ctas, ctypes.byref(n))
    _check("moe_decode_timeline", rc)
    return buf[:min(n.value, max_ctas)]


# ---------------------------------------------------------------- conveniences

def workspace(cfg: moe_config, T: int, device="cuda") -> torch.Tensor:
    """A zero-filled device workspace of moe_workspace_size bytes (uint8, 256-byte aligned by the allocator)."""
    return torch.zeros(moe_workspace_size(cfg, T), dtype=torch.uint8, device=device)


def forward(layer: DeviceLayer, x: torch.Tensor, ws: torch.Tensor, router_bias=None, logits_in=None,
            path: int = MOE_PATH_AUTO, stream=None, with_routing: bool = False, cfg: Optional[moe_config] = None):
    """y (int16 view of bf16 bits) = layer(x); optionally also (ids, p, w_s).  cfg overrides layer.cfg
    (e.g. to set wait_polls for one call)."""
    T = x.shape[0]
    dev = x.device
    y = torch.empty((T, layer.shape.hidden), dtype=torch.int16, device=dev)
    ids = p = w_s = None
    if with_routing:
        ids = torch.empty((T, layer.shape.top_k), dtype=torch.int32, device=dev)
        p = torch.empty((T, layer.shape.top_k), dtype=torch.int16, device=dev)
        w_s = torch.empty((max(T, 1),), dtype=torch.int16, device=dev)
    moe_forward(cfg if cfg is not None else layer.cfg, layer.w, x, T, router_bias, logits_in, y, ids, p, w_s, path,
                ws, stream)
    return (y, ids, p, w_s) if with_routing else y
