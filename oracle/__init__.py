"""moeq oracle -- TEST INFRASTRUCTURE ONLY.

A numpy/ctypes front end for ``moeq_oracle.c``, the plain single-threaded CPU
statement of the FP8 live-quant MoE expert path (see the header of that file
for what is computed and which reading of the source page each step follows).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It never imports the CUDA package
``bandwidth_bound_fp8_gb300`` and the CUDA package never imports it.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, exhaustive codec checks, library routines on special
cases (torch's float8_e4m3fn decode, numpy matmul, numpy stable argsort,
scipy softmax) and brute force on tiny shapes.  No function is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moeq_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_vpp = ctypes.POINTER(ctypes.c_void_p)


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (-O2, IEEE semantics, no contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call([
            "gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", "-Wall", "-Wextra", "-Wno-unused-parameter",
            "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        L.orc_set_fault.argtypes = [ctypes.c_int]
        L.orc_e4m3_decode.restype = ctypes.c_double
        L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_e4m3_encode.argtypes = [ctypes.c_double]
        L.orc_e4m3_encode_scan.restype = ctypes.c_uint8
        L.orc_e4m3_encode_scan.argtypes = [ctypes.c_double]
        L.orc_f64_to_bf16.restype = ctypes.c_uint16
        L.orc_f64_to_bf16.argtypes = [ctypes.c_double]
        L.orc_bf16_to_f32.restype = ctypes.c_float
        L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_quant_act_f32.argtypes = [_f32p, ctypes.c_int, ctypes.c_int, _u8p, _f32p]
        L.orc_quant_act_bf16.argtypes = [_u16p, ctypes.c_int, ctypes.c_int, _u8p, _f32p]
        L.orc_quant_weight.argtypes = [_f32p, ctypes.c_int, ctypes.c_int, _u8p, _f32p]
        L.orc_gemm.argtypes = [_u8p, _f32p, ctypes.c_int, _u8p, _f32p, ctypes.c_int,
                               ctypes.c_int, _f64p, ctypes.c_void_p]
        L.orc_route.argtypes = [_f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                _i32p, _f64p, _i32p, _i32p, _i32p, _i32p, _i32p]
        L.orc_swiglu.restype = ctypes.c_float
        L.orc_swiglu.argtypes = [ctypes.c_double, ctypes.c_double]
        L.orc_swiglu_vec.argtypes = [_f64p, _f64p, ctypes.c_int, _f32p]
        L.orc_moe_layer.argtypes = [
            _u16p, _f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            _vpp, _vpp, _vpp, _vpp,
            _u16p, _f64p, _f64p, _f32p, _f64p, _f64p, _u8p, _f32p, _u8p, _f32p,
            _i32p, _f64p, _i32p, _i32p, _i32p, _i32p, _i32p]
        _lib = L
    return _lib


def set_fault(f: int) -> None:
    """Plant mistake number f in the oracle (0 restores it); mutation tests only."""
    lib().orc_set_fault(int(f))


# --------------------------------------------------------------------------
# codec
# --------------------------------------------------------------------------
def e4m3_decode(c: int) -> float:
    return lib().orc_e4m3_decode(int(c) & 0xFF)


def e4m3_decode_table() -> np.ndarray:
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def e4m3_encode(v: float) -> int:
    return int(lib().orc_e4m3_encode(float(v)))


def e4m3_encode_scan(v: float) -> int:
    return int(lib().orc_e4m3_encode_scan(float(v)))


def f64_to_bf16_bits(v: float) -> int:
    return int(lib().orc_f64_to_bf16(float(v)))


def bf16_bits_to_f32(b: int) -> float:
    return float(lib().orc_bf16_to_f32(int(b) & 0xFFFF))


# --------------------------------------------------------------------------
# quantisation
# --------------------------------------------------------------------------
def quant_act(x: np.ndarray):
    """x: [M, K] float32 or bf16 bit patterns (uint16).  Returns (q [M,K] u8, s [M,K/128] f32)."""
    x = np.ascontiguousarray(x)
    M, K = x.shape
    q = np.zeros((M, K), np.uint8)
    s = np.zeros((M, K // 128), np.float32)
    if x.dtype == np.uint16:
        rc = lib().orc_quant_act_bf16(x, M, K, q, s)
    else:
        rc = lib().orc_quant_act_f32(np.ascontiguousarray(x, np.float32), M, K, q, s)
    if rc:
        raise ValueError(f"orc_quant_act: rc={rc}")
    return q, s


def quant_weight(w: np.ndarray):
    """w: [N, K] float32.  Returns (q [N,K] u8, s [N/128, K/128] f32)."""
    w = np.ascontiguousarray(w, np.float32)
    N, K = w.shape
    q = np.zeros((N, K), np.uint8)
    s = np.zeros((N // 128, K // 128), np.float32)
    if lib().orc_quant_weight(w, N, K, q, s):
        raise ValueError("orc_quant_weight: shape not a multiple of 128")
    return q, s


# --------------------------------------------------------------------------
# GEMM, routing, SwiGLU, layer
# --------------------------------------------------------------------------
def gemm(qa, sa, qw, sw, with_T: bool = True):
    """Block-scaled FP8 GEMM in fp64.  Returns y [M,N] (and T [M,N])."""
    qa = np.ascontiguousarray(qa, np.uint8)
    sa = np.ascontiguousarray(sa, np.float32)
    qw = np.ascontiguousarray(qw, np.uint8)
    sw = np.ascontiguousarray(sw, np.float32)
    M, K = qa.shape
    N = qw.shape[0]
    y = np.zeros((M, N), np.float64)
    T = np.zeros((M, N), np.float64) if with_T else None
    rc = lib().orc_gemm(qa, sa, M, qw, sw, N, K, y,
                        T.ctypes.data_as(ctypes.c_void_p) if with_T else None)
    if rc:
        raise ValueError("orc_gemm: shape not a multiple of 128")
    return (y, T) if with_T else y


class Route:
    """Routing plan as the oracle states it (see orc_route)."""

    def __init__(self, topk_id, topk_w, uniq, offs, pair_tok, pair_of):
        self.topk_id, self.topk_w = topk_id, topk_w
        self.uniq, self.offs, self.pair_tok, self.pair_of = uniq, offs, pair_tok, pair_of

    @property
    def n_uniq(self):
        return len(self.uniq)

    @property
    def n_pairs(self):
        return len(self.pair_tok)


def route(logits: np.ndarray, k: int) -> Route:
    logits = np.ascontiguousarray(logits, np.float32)
    M, E = logits.shape
    P_max = M * k + M
    topk_id = np.zeros((M, k), np.int32)
    topk_w = np.zeros((M, k), np.float64)
    n_uniq = np.zeros(1, np.int32)
    uniq = np.zeros(E + 1, np.int32)
    offs = np.zeros(E + 2, np.int32)
    pair_tok = np.zeros(P_max, np.int32)
    pair_of = np.zeros((M, k + 1), np.int32)
    P = lib().orc_route(logits, M, E, k, topk_id, topk_w, n_uniq, uniq, offs, pair_tok, pair_of)
    if P < 0:
        raise ValueError(f"orc_route rc={P}")
    U = int(n_uniq[0])
    return Route(topk_id, topk_w, uniq[:U].copy(), offs[:U + 1].copy(), pair_tok[:P].copy(), pair_of)


def swiglu(gate: float, up: float) -> float:
    return float(lib().orc_swiglu(float(gate), float(up)))


def swiglu_vec(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    g = np.ascontiguousarray(gate, np.float64).ravel()
    u = np.ascontiguousarray(up, np.float64).ravel()
    h = np.zeros(g.size, np.float32)
    lib().orc_swiglu_vec(g, u, g.size, h)
    return h.reshape(np.shape(gate))


class LayerResult:
    pass


def moe_layer(x_bf16: np.ndarray, logits: np.ndarray, k: int, experts: dict, H: int, I: int):
    """One MoE layer.  ``experts[e] = (qgu [2I,H] u8, sgu f32, qd [H,I] u8, sd f32)``
    for every expert the routing touches (e = E_routed is the shared expert)."""
    x_bf16 = np.ascontiguousarray(x_bf16, np.uint16)
    logits = np.ascontiguousarray(logits, np.float32)
    M, E = logits.shape
    P_max = M * k + M
    keep = []

    def ptrs(idx):
        arr = (ctypes.c_void_p * (E + 1))()
        for e, t in experts.items():
            a = np.ascontiguousarray(t[idx])
            keep.append(a)
            arr[e] = a.ctypes.data
        return ctypes.cast(arr, _vpp), arr

    pqgu, a0 = ptrs(0)
    psgu, a1 = ptrs(1)
    pqd, a2 = ptrs(2)
    psd, a3 = ptrs(3)
    r = LayerResult()
    r.out_bf16 = np.zeros((M, H), np.uint16)
    r.out64 = np.zeros((M, H), np.float64)
    r.Tout = np.zeros((M, H), np.float64)
    r.h = np.zeros((P_max, I), np.float32)
    r.y64 = np.zeros((P_max, H), np.float64)
    r.Ty = np.zeros((P_max, H), np.float64)
    r.qx = np.zeros((M, H), np.uint8)
    r.sx = np.zeros((M, H // 128), np.float32)
    r.qh = np.zeros((P_max, I), np.uint8)
    r.sh = np.zeros((P_max, I // 128), np.float32)
    topk_id = np.zeros((M, k), np.int32)
    topk_w = np.zeros((M, k), np.float64)
    n_uniq = np.zeros(1, np.int32)
    uniq = np.zeros(E + 1, np.int32)
    offs = np.zeros(E + 2, np.int32)
    pair_tok = np.zeros(P_max, np.int32)
    pair_of = np.zeros((M, k + 1), np.int32)
    P = lib().orc_moe_layer(x_bf16, logits, M, H, I, E, k, pqgu, psgu, pqd, psd,
                            r.out_bf16, r.out64, r.Tout, r.h, r.y64, r.Ty,
                            r.qx, r.sx, r.qh, r.sh,
                            topk_id, topk_w, n_uniq, uniq, offs, pair_tok, pair_of)
    if P < 0:
        raise ValueError(f"orc_moe_layer rc={P} (missing expert weights?)")
    U = int(n_uniq[0])
    r.route = Route(topk_id, topk_w, uniq[:U].copy(), offs[:U + 1].copy(), pair_tok[:P].copy(), pair_of)
    r.h, r.y64, r.Ty, r.qh, r.sh = r.h[:P], r.y64[:P], r.Ty[:P], r.qh[:P], r.sh[:P]
    return r


def bf16_bits_to_f32_array(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (a bit shift, no arithmetic)."""
    return (np.ascontiguousarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)
