"""FP64 CPU oracle for the routed-expert MoE layer (test infrastructure).

Only the tests, the package smoke check and the bench's CPU-baseline leg may
import this package.  The library path never loads it: it is the independent
reference the CUDA kernels are checked against, and it shares no code with
them.  The arithmetic lives in ``moe_oracle.c`` (plain C, fp64 accumulation);
this module compiles it with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so (gcc, OpenMP, no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Cfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("hidden", "inter", "n_experts", "top_k", "group", "bits", "router_bits", "has_shared", "format")]


class _QMat(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("biases", ctypes.c_void_p),
                ("bscales", ctypes.c_void_p), ("gscale", ctypes.c_void_p)]


class _Weights(ctypes.Structure):
    _fields_ = [(n, _QMat) for n in ("router", "gate", "up", "down", "s_gate", "s_up", "s_down")] + \
               [("shared_gate_vec", ctypes.c_void_p)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            _lib.oracle_bf16_rne.restype = ctypes.c_uint16
            _lib.oracle_bf16_rne.argtypes = [ctypes.c_double]
            _lib.oracle_bf16_to_double.restype = ctypes.c_double
            _lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            _lib.oracle_f32_rne.restype = ctypes.c_float
            _lib.oracle_f32_rne.argtypes = [ctypes.c_double]
            _lib.oracle_num_threads.restype = ctypes.c_int
            for f in ("oracle_e2m1_to_double", "oracle_e4m3_to_double"):
                getattr(_lib, f).restype = ctypes.c_double
                getattr(_lib, f).argtypes = [ctypes.c_int]
        return _lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _cfg(shape) -> _Cfg:
    return _Cfg(shape.hidden, shape.inter, shape.n_experts, shape.top_k, shape.group, shape.bits,
                shape.router_bits, shape.has_shared, 1 if is_nvfp4(shape) else 0)


def is_nvfp4(shape) -> bool:
    return getattr(shape, "fmt", "affine") == "nvfp4"


def num_threads() -> int:
    return lib().oracle_num_threads()


def bf16_rne(v) -> np.ndarray:
    """fp64 values -> bf16 bits (uint16), round to nearest even, one rounding."""
    v = np.asarray(v, dtype=np.float64)
    f = lib().oracle_bf16_rne
    return np.array([f(float(a)) for a in v.ravel()], dtype=np.uint16).reshape(v.shape)


def bf16_to_f64(b) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def dequant_row(codes_row, scales_row, biases_row, bits: int, in_dim: int, group: int = 64) -> np.ndarray:
    out = np.empty(in_dim, dtype=np.float64)
    codes_row, scales_row, biases_row = _c(codes_row, np.uint8), _c(scales_row, np.uint16), _c(biases_row, np.uint16)
    lib().oracle_dequant_row(_p(codes_row), _p(scales_row), _p(biases_row), ctypes.c_int(bits),
                             ctypes.c_int(in_dim), ctypes.c_int(group), _p(out))
    return out


def e2m1_to_f64(code: int) -> float:
    return lib().oracle_e2m1_to_double(int(code))


def e4m3_to_f64(code: int) -> float:
    return lib().oracle_e4m3_to_double(int(code))


def dequant_row_nvfp4(codes_row, bscales_row, gscale: float, in_dim: int) -> np.ndarray:
    out = np.empty(in_dim, dtype=np.float64)
    codes_row, bscales_row = _c(codes_row, np.uint8), _c(bscales_row, np.uint8)
    lib().oracle_dequant_row_nvfp4(_p(codes_row), _p(bscales_row), ctypes.c_float(gscale), ctypes.c_int(in_dim),
                                   _p(out))
    return out


def dequant_matrix(codes, scales, biases, bits: int, in_dim: int, group: int = 64) -> np.ndarray:
    """Dequantise a [rows, in] matrix row by row with ``dequant_row``."""
    rows = codes.shape[0]
    return np.stack([dequant_row(codes[r], scales[r], biases[r], bits, in_dim, group) for r in range(rows)])


def router_logits(shape, weights, x, bias=None) -> np.ndarray:
    x = _c(x, np.uint16)
    T = x.shape[0]
    out = np.empty((T, shape.n_experts), dtype=np.float32)
    r = weights.router
    bias_c = None if bias is None else _c(bias, np.float32)
    cfg = _cfg(shape)
    codes, s, b = _c(r.codes, np.uint8), _c(r.scales, np.uint16), _c(r.biases, np.uint16)
    lib().oracle_router_logits(ctypes.byref(cfg), _p(codes), _p(s), _p(b), _p(x), ctypes.c_int(T),
                               _p(bias_c), _p(out))
    return out


def topk(logits, k: int) -> np.ndarray:
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), dtype=np.int32)
    lib().oracle_topk(_p(logits), ctypes.c_int(T), ctypes.c_int(E), ctypes.c_int(k), _p(ids))
    return ids


def pick_weights(logits, ids):
    logits, ids = _c(logits, np.float32), _c(ids, np.int32)
    T, E = logits.shape
    k = ids.shape[1]
    pe = np.empty((T, k), dtype=np.float64)
    pb = np.empty((T, k), dtype=np.uint16)
    lib().oracle_pick_weights(_p(logits), _p(ids), ctypes.c_int(T), ctypes.c_int(E), ctypes.c_int(k),
                              _p(pe), _p(pb))
    return pe, pb


def shared_weight(x, v):
    x, v = _c(x, np.uint16), _c(v, np.uint16)
    T, H = x.shape
    gamma = np.empty(T, dtype=np.float32)
    ws = np.empty(T, dtype=np.uint16)
    lib().oracle_shared_weight(_p(x), _p(v), ctypes.c_int(T), ctypes.c_int(H), _p(gamma), _p(ws))
    return gamma, ws


def _qmat_struct(m, keep, e=None, nvfp4=False):
    """ctypes view of a stacked QMat (or of its expert e): affine codes/scales/biases, or NVFP4
    codes, E4M3 block scales (stored in ``scales``) and the fp32 per-matrix scales."""
    sel = (lambda a: a) if e is None else (lambda a: a[e:e + 1])
    if nvfp4:
        arrs = (_c(sel(m.codes), np.uint8), _c(sel(m.scales), np.uint8), _c(sel(m.gscale), np.float32))
        keep.extend(arrs)
        return _QMat(arrs[0].ctypes.data, None, None, arrs[1].ctypes.data, arrs[2].ctypes.data)
    arrs = (_c(sel(m.codes), np.uint8), _c(sel(m.scales), np.uint16), _c(sel(m.biases), np.uint16))
    keep.extend(arrs)
    return _QMat(arrs[0].ctypes.data, arrs[1].ctypes.data, arrs[2].ctypes.data, None, None)


def _expert_mats(shape, weights, e, keep):
    """(gate, up, down) structs of expert e; e == -1 selects the shared expert."""
    mats = (weights.s_gate, weights.s_up, weights.s_down) if e < 0 else (weights.gate, weights.up, weights.down)
    return tuple(_qmat_struct(m, keep, 0 if e < 0 else e, is_nvfp4(shape)) for m in mats)


def expert_ffn(shape, weights, e: int, x_f64):
    """One expert (e == -1: shared) on one token given as fp64 [H]; returns (h [I], y [H])."""
    keep = []
    mg, mu, md = _expert_mats(shape, weights, e, keep)
    x_f64 = _c(x_f64, np.float64)
    h = np.empty(shape.inter, dtype=np.float64)
    y = np.empty(shape.hidden, dtype=np.float64)
    cfg = _cfg(shape)
    lib().oracle_expert_ffn_m(ctypes.byref(cfg), ctypes.byref(mg), ctypes.byref(mu), ctypes.byref(md), _p(x_f64),
                              _p(h), _p(y))
    return h, y


def expert_down(shape, weights, e: int, h_f64):
    keep = []
    md = _expert_mats(shape, weights, e, keep)[2]
    h_f64 = _c(h_f64, np.float64)
    y = np.empty(shape.hidden, dtype=np.float64)
    cfg = _cfg(shape)
    lib().oracle_expert_down_m(ctypes.byref(cfg), ctypes.byref(md), _p(h_f64), _p(y))
    return y


def _weights_struct(weights, keep):
    nv = is_nvfp4(weights.shape)

    def q(m, expert=True):
        return _qmat_struct(m, keep, None, nv and expert)
    v = _c(weights.shared_gate_vec, np.uint16)
    keep.append(v)
    return _Weights(q(weights.router, False), q(weights.gate), q(weights.up), q(weights.down),
                    q(weights.s_gate), q(weights.s_up), q(weights.s_down), v.ctypes.data)


def forward(shape, weights, x, bias=None, logits_in=None, rows=None):
    """The whole layer on the tokens of ``x`` (or on ``rows`` of it: rows are independent).

    Returns a dict with y (bf16 bits [T,H]), y_exact (fp64 before the final
    rounding), ids [T,k], p (bf16 bits), w_s (bf16 bits) and logits (fp32).
    """
    x = _c(x, np.uint16)
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        x = _c(x[rows], np.uint16)
        if logits_in is not None:
            logits_in = np.asarray(logits_in)[rows]
    T = x.shape[0]
    H, E, k = shape.hidden, shape.n_experts, shape.top_k
    keep = []
    ws_struct = _weights_struct(weights, keep)
    out = dict(y=np.empty((T, H), np.uint16), y_exact=np.empty((T, H), np.float64),
               ids=np.empty((T, k), np.int32), p=np.empty((T, k), np.uint16),
               w_s=np.empty(T, np.uint16), logits=np.empty((T, E), np.float32))
    bias_c = None if bias is None else _c(bias, np.float32)
    lin = None if logits_in is None else _c(logits_in, np.float32)
    cfg = _cfg(shape)
    rc = lib().oracle_forward(ctypes.byref(cfg), ctypes.byref(ws_struct), _p(x), ctypes.c_int(T), _p(bias_c),
                              _p(lin), _p(out["y"]), _p(out["y_exact"]), _p(out["ids"]), _p(out["p"]),
                              _p(out["w_s"]), _p(out["logits"]))
    assert rc == 0
    return out


def permute(ids, n_experts: int):
    ids = _c(ids, np.int32)
    T, k = ids.shape
    counts = np.empty(n_experts, np.int32)
    offsets = np.empty(n_experts + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    inv = np.empty(T * k, np.int32)
    lib().oracle_permute(_p(ids), ctypes.c_int(T), ctypes.c_int(k), ctypes.c_int(n_experts), _p(counts),
                         _p(offsets), _p(perm), _p(inv))
    return counts, offsets, perm, inv
