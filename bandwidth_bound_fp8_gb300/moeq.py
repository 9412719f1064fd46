"""Thin ctypes binding of libmoeq (include/moeq.h), same names as the C ABI.

Argument marshalling only: every step of the path runs in the CUDA kernels of
libmoeq.so.  Tensors are torch tensors on the current CUDA device; the stream
defaults to torch's current stream.  A non-zero status raises MoeqError.
There is no fallback: if libmoeq.so is missing the import of the library
raises, loudly.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoeq.so")

MOEQ_OK = 0
MOEQ_ERR_INVALID_ARG = 1
MOEQ_ERR_UNSUPPORTED_SHAPE = 2
MOEQ_ERR_WORKSPACE = 3
MOEQ_ERR_CUDA = 4
MOEQ_ERR_TIMEOUT = 5
MOEQ_ERR_DEVICE = 6
MOEQ_BF16 = 0
MOEQ_F32 = 1
MOEQ_GROUP = 128
MOEQ_MAX_TOKENS = 16
MOEQ_MAX_LAYERS = 256
MOEQ_STACK_EAGER = 1

# Every symbol include/moeq.h declares (checked by the tests against the header).
EXPORTS = [
    "moeq_status_string", "moeq_abi_version", "moeq_max_uniq", "moeq_max_pairs",
    "moeq_route_plan_bytes", "moeq_route_plan_carve", "moeq_workspace_size",
    "moeq_gemm_workspace_size", "moeq_workspace_init", "moeq_read_device_status",
    "moeq_quant_act", "moeq_quant_weight", "moeq_pack_weight", "moeq_route", "moeq_expert_gemm_gateup_swiglu",
    "moeq_expert_gemm_down", "moeq_combine", "moeq_moe_layer", "moeq_expert_gemm_down_noalloc",
    "moeq_dense_ffn_workspace_size", "moeq_dense_ffn", "moeq_stack_workspace_size", "moeq_moe_stack",
    "moeq_stack_plan", "moeq_stack_release_graphs", "moeq_tp_shard_weights", "moeq_moe_layer_shard",
    "moeq_tp_reduce", "moeq_layer_ws_count_offset", "moeq_gemm_ws_count_offset",
]


class MoeqError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: status {status} ({status_string(status)})")


class moeq_route_plan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("topk_id", "topk_w", "n_uniq", "uniq", "offs", "pair_tok", "pair_of")]


_lib = None
_vp = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t


def load(path: str = LIB_PATH):
    """Load libmoeq.so (raises if it is not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libmoeq.so not found at {path}: build it with __graft_entry__.build()")
    L = ctypes.CDLL(path)
    sig = {
        "moeq_status_string": (ctypes.c_char_p, [_i]),
        "moeq_abi_version": (_i, []),
        "moeq_max_uniq": (_i, [_i, _i, _i]),
        "moeq_max_pairs": (_i, [_i, _i]),
        "moeq_route_plan_bytes": (_sz, [_i, _i, _i]),
        "moeq_route_plan_carve": (_i, [_vp, _sz, _i, _i, _i, ctypes.POINTER(moeq_route_plan)]),
        "moeq_workspace_size": (_sz, [_i, _i, _i, _i, _i]),
        "moeq_gemm_workspace_size": (_sz, [_i, _i, _i, _i, _i]),
        "moeq_workspace_init": (_i, [_vp, _sz, _vp]),
        "moeq_read_device_status": (_i, [_vp, _sz, ctypes.POINTER(_i)]),
        "moeq_quant_act": (_i, [_vp, _i, _i, _i, _vp, _vp, _vp]),
        "moeq_quant_weight": (_i, [_vp, _i, _i, _i, _vp, _vp, _vp]),
        "moeq_pack_weight": (_i, [_vp, _i, _i, _i, _vp, _vp]),
        "moeq_route": (_i, [_vp, _i, _i, _i, ctypes.POINTER(moeq_route_plan), _vp]),
        "moeq_expert_gemm_gateup_swiglu": (_i, [_vp, _i, _i, _i, _i, _vp, _vp, _i, _vp, _vp, _vp, _vp,
                                                _i, _i, _vp, _vp, _vp, _vp, _sz, _vp]),
        "moeq_expert_gemm_down": (_i, [_vp, _i, _i, _i, _vp, _vp, _i, _vp, _vp, _vp, _i, _i,
                                       _vp, _vp, _vp, _vp, _sz, _vp]),
        "moeq_combine": (_i, [_vp, _i, ctypes.POINTER(moeq_route_plan), _i, _i, _vp, _vp]),
        "moeq_expert_gemm_down_noalloc": (_i, [_vp, _i, _i, _i, _vp, _vp, _i, _vp, _vp, _vp, _i, _i,
                                               _vp, _vp, _vp, _vp, _vp]),
        "moeq_dense_ffn_workspace_size": (_sz, [_i, _i, _i]),
        "moeq_dense_ffn": (_i, [_vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
        "moeq_stack_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i]),
        "moeq_tp_shard_weights": (_i, [_i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
        "moeq_moe_layer_shard": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp,
                                      ctypes.POINTER(moeq_route_plan), _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
        "moeq_tp_reduce": (_i, [_vp, _i, _i, _i, _vp, _vp]),
        "moeq_layer_ws_count_offset": (_sz, [_i, _i, _i, _i, _i, _i]),
        "moeq_gemm_ws_count_offset": (_sz, [_i, _i, _i, _i, _i, _i]),
        "moeq_moe_stack": (_i, [_i, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _i, _vp, _sz, _vp]),
        "moeq_stack_plan": (_i, [_vp, _sz, _i, _i, _i, _i, _i, _i, _i, ctypes.POINTER(moeq_route_plan)]),
        "moeq_stack_release_graphs": (_i, []),
        "moeq_moe_layer": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp,
                                ctypes.POINTER(moeq_route_plan), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                _sz, _vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def status_string(status: int) -> str:
    return load().moeq_status_string(int(status)).decode()


def _check(fn: str, status: int) -> None:
    if status != MOEQ_OK:
        raise MoeqError(fn, status)


def _p(t):
    """Device (or host) pointer of a tensor, None for None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype(t) -> int:
    if t.dtype == torch.bfloat16:
        return MOEQ_BF16
    if t.dtype == torch.float32:
        return MOEQ_F32
    raise TypeError(f"unsupported activation dtype {t.dtype}")


# ----------------------------------------------------------------- sizes
def moeq_abi_version() -> int:
    return load().moeq_abi_version()


def moeq_max_uniq(M, E_routed, top_k) -> int:
    return load().moeq_max_uniq(M, E_routed, top_k)


def moeq_max_pairs(M, top_k) -> int:
    return load().moeq_max_pairs(M, top_k)


def moeq_route_plan_bytes(M, E_routed, top_k) -> int:
    return load().moeq_route_plan_bytes(M, E_routed, top_k)


def moeq_workspace_size(M, H, I, n_experts_incl_shared, top_k) -> int:
    return load().moeq_workspace_size(M, H, I, n_experts_incl_shared, top_k)


def moeq_gemm_workspace_size(rows_out, K, rows_in, max_uniq, is_gate_up) -> int:
    return load().moeq_gemm_workspace_size(rows_out, K, rows_in, max_uniq, int(bool(is_gate_up)))


class RoutePlan:
    """A route plan in one device buffer, with torch views of its members.
    `within` = (uint8 tensor, moeq_route_plan) views a plan already carved
    inside that buffer (e.g. a stack workspace's) instead of allocating one."""

    def __init__(self, M: int, E_routed: int, top_k: int, device="cuda", within=None):
        L = load()
        self.M, self.E, self.k = M, E_routed, top_k
        if within is None:
            nbytes = L.moeq_route_plan_bytes(M, E_routed, top_k)
            if not nbytes:
                raise MoeqError("moeq_route_plan_bytes", MOEQ_ERR_INVALID_ARG)
            self.buf = torch.zeros(nbytes, dtype=torch.uint8, device=device)
            self.c = moeq_route_plan()
            _check("moeq_route_plan_carve",
                   L.moeq_route_plan_carve(self.buf.data_ptr(), nbytes, M, E_routed, top_k, ctypes.byref(self.c)))
        else:
            self.buf, self.c = within
        self.max_uniq = L.moeq_max_uniq(M, E_routed, top_k)
        self.max_pairs = L.moeq_max_pairs(M, top_k)
        base = self.buf.data_ptr()

        def view(field, n, dt):
            off = getattr(self.c, field) - base
            assert 0 <= off and off + 4 * n <= self.buf.numel(), "plan outside its buffer"
            return self.buf[off:off + 4 * n].view(dt)

        self.topk_id = view("topk_id", M * top_k, torch.int32).view(M, top_k)
        self.topk_w = view("topk_w", M * top_k, torch.float32).view(M, top_k)
        self.n_uniq = view("n_uniq", 1, torch.int32)
        self.uniq = view("uniq", self.max_uniq, torch.int32)
        self.offs = view("offs", self.max_uniq + 1, torch.int32)
        self.pair_tok = view("pair_tok", self.max_pairs, torch.int32)
        self.pair_of = view("pair_of", M * (top_k + 1), torch.int32).view(M, top_k + 1)


class Workspace:
    """Caller-owned workspace (a torch uint8 buffer), zeroed once."""

    def __init__(self, nbytes: int, device="cuda", stream=None):
        if not nbytes:
            raise MoeqError("workspace size", MOEQ_ERR_WORKSPACE)
        self.nbytes = int(nbytes)
        self.buf = torch.empty(self.nbytes + 256, dtype=torch.uint8, device=device)
        off = (-self.buf.data_ptr()) % 256
        self.t = self.buf[off:off + self.nbytes]
        moeq_workspace_init(self.t, self.nbytes, stream)

    @property
    def ptr(self):
        return self.t.data_ptr()


# ----------------------------------------------------------------- calls
def moeq_workspace_init(ws, ws_bytes, stream=None) -> None:
    _check("moeq_workspace_init", load().moeq_workspace_init(_p(ws), ws_bytes, _stream(stream)))


def moeq_read_device_status(ws, ws_bytes) -> int:
    out = ctypes.c_int(0)
    _check("moeq_read_device_status", load().moeq_read_device_status(_p(ws), ws_bytes, ctypes.byref(out)))
    return out.value


def moeq_quant_act(x, q, s, stream=None) -> None:
    M, K = x.shape
    _check("moeq_quant_act", load().moeq_quant_act(_p(x), _dtype(x), M, K, _p(q), _p(s), _stream(stream)))


def moeq_quant_weight(w, q, s, stream=None) -> None:
    E, N, K = w.shape
    _check("moeq_quant_weight", load().moeq_quant_weight(_p(w), E, N, K, _p(q), _p(s), _stream(stream)))


def moeq_pack_weight(q_rows, q_tiles, stream=None) -> None:
    E, N, K = q_rows.shape
    _check("moeq_pack_weight", load().moeq_pack_weight(_p(q_rows), E, N, K, _p(q_tiles), _stream(stream)))


def moeq_route(logits, plan: RoutePlan, top_k: int, stream=None) -> None:
    M, E = logits.shape
    _check("moeq_route", load().moeq_route(_p(logits), M, E, top_k, ctypes.byref(plan.c), _stream(stream)))


def moeq_expert_gemm_gateup_swiglu(x, H, I, w_gu, s_gu, n_experts, uniq, offs, pair_tok, n_uniq,
                                   max_uniq, max_pairs, h, ws: Workspace, q_x=None, s_x=None,
                                   stream=None) -> None:
    M = x.shape[0]
    _check("moeq_expert_gemm_gateup_swiglu", load().moeq_expert_gemm_gateup_swiglu(
        _p(x), _dtype(x), M, H, I, _p(w_gu), _p(s_gu), n_experts, _p(uniq), _p(offs), _p(pair_tok),
        _p(n_uniq), max_uniq, max_pairs, _p(h), _p(q_x), _p(s_x), ws.ptr, ws.nbytes, _stream(stream)))


def moeq_expert_gemm_down_noalloc(a, K, N, w_d, s_d, n_experts, uniq, offs, n_uniq, max_uniq, max_pairs, y,
                                  q_a=None, s_a=None, device_status=None, stream=None) -> None:
    """moeq_expert_gemm_down on the library's static scratch (no workspace);
    device_status: optional device int32 tensor that receives the status word."""
    _check("moeq_expert_gemm_down_noalloc", load().moeq_expert_gemm_down_noalloc(
        _p(a), _dtype(a), K, N, _p(w_d), _p(s_d), n_experts, _p(uniq), _p(offs), _p(n_uniq),
        max_uniq, max_pairs, _p(y), _p(q_a), _p(s_a), _p(device_status), _stream(stream)))


def moeq_expert_gemm_down(a, K, N, w_d, s_d, n_experts, uniq, offs, n_uniq, max_uniq, max_pairs, y,
                          ws: Workspace, q_a=None, s_a=None, stream=None) -> None:
    _check("moeq_expert_gemm_down", load().moeq_expert_gemm_down(
        _p(a), _dtype(a), K, N, _p(w_d), _p(s_d), n_experts, _p(uniq), _p(offs), _p(n_uniq),
        max_uniq, max_pairs, _p(y), _p(q_a), _p(s_a), ws.ptr, ws.nbytes, _stream(stream)))


def moeq_dense_ffn_workspace_size(M, H, I) -> int:
    return int(load().moeq_dense_ffn_workspace_size(M, H, I))


def moeq_dense_ffn(x, H, I, w_gu, s_gu, w_d, s_d, out, ws: Workspace, h=None, q_x=None, s_x=None, q_h=None,
                   s_h=None, stream=None) -> None:
    M = x.shape[0]
    _check("moeq_dense_ffn", load().moeq_dense_ffn(
        _p(x), M, H, I, _p(w_gu), _p(s_gu), _p(w_d), _p(s_d), _p(out), _p(h), _p(q_x), _p(s_x), _p(q_h), _p(s_h),
        ws.ptr, ws.nbytes, _stream(stream)))


def moeq_combine(y, N, plan: RoutePlan, M, top_k, out, stream=None) -> None:
    _check("moeq_combine", load().moeq_combine(_p(y), N, ctypes.byref(plan.c), M, top_k, _p(out),
                                               _stream(stream)))


def moeq_moe_layer(x, logits, H, I, E_routed, top_k, w_gu, s_gu, w_d, s_d, out, ws: Workspace,
                   plan: RoutePlan | None = None, h=None, y=None, q_x=None, s_x=None, q_h=None, s_h=None,
                   events=None, stream=None) -> None:
    M = x.shape[0]
    ev = None
    if events is not None:
        handles = [e.cuda_event for e in events]
        if not all(handles):
            raise ValueError("moeq_moe_layer: events must be created (recorded once) before use")
        if len(handles) != 2:
            raise ValueError("moeq_moe_layer: events must be two created events (before, after)")
        ev = (ctypes.c_void_p * 2)(*handles)
    _check("moeq_moe_layer", load().moeq_moe_layer(
        _p(x), _p(logits), M, H, I, E_routed, top_k, _p(w_gu), _p(s_gu), _p(w_d), _p(s_d), _p(out),
        ctypes.byref(plan.c) if plan is not None else None, _p(h), _p(y), _p(q_x), _p(s_x), _p(q_h), _p(s_h),
        ev, ws.ptr, ws.nbytes, _stream(stream)))


def moeq_stack_workspace_size(L, M, H, I, n_experts_incl_shared, top_k) -> int:
    return int(load().moeq_stack_workspace_size(L, M, H, I, n_experts_incl_shared, top_k))


def moeq_moe_stack(x, logits, H, I, E_routed, top_k, w_gu, s_gu, w_d, s_d, out, ws: Workspace, flags=0,
                   stream=None) -> None:
    """L layers in sequence (L = len(w_gu)); logits [L, M, E_routed], out
    [L, M, H]; w_gu .. s_d: sequences of L tensors (or device pointers)."""
    Ln, M = len(w_gu), x.shape[0]
    if not (len(s_gu) == len(w_d) == len(s_d) == Ln):
        raise ValueError("moeq_moe_stack: one weight set per layer")
    arr = lambda ts: (ctypes.c_void_p * Ln)(*[_p(t) for t in ts])
    _check("moeq_moe_stack", load().moeq_moe_stack(
        Ln, _p(x), _p(logits), M, H, I, E_routed, top_k, arr(w_gu), arr(s_gu), arr(w_d), arr(s_d), _p(out),
        int(flags), ws.ptr, ws.nbytes, _stream(stream)))


def moeq_stack_plan(ws: Workspace, L, M, H, I, E_routed, top_k, layer) -> RoutePlan:
    """Layer `layer`'s route plan inside a stack workspace, as a RoutePlan view."""
    c = moeq_route_plan()
    _check("moeq_stack_plan", load().moeq_stack_plan(ws.ptr, ws.nbytes, L, M, H, I, E_routed, top_k, layer,
                                                     ctypes.byref(c)))
    return RoutePlan(M, E_routed, top_k, within=(ws.t, c))


def moeq_stack_release_graphs() -> None:
    _check("moeq_stack_release_graphs", load().moeq_stack_release_graphs())


def moeq_tp_shard_weights(E, H, I, R, rank, w_gu, s_gu, w_d, s_d, w_gu_shard, s_gu_shard, w_d_shard, s_d_shard,
                          stream=None) -> None:
    _check("moeq_tp_shard_weights", load().moeq_tp_shard_weights(
        E, H, I, R, rank, _p(w_gu), _p(s_gu), _p(w_d), _p(s_d), _p(w_gu_shard), _p(s_gu_shard), _p(w_d_shard),
        _p(s_d_shard), _stream(stream)))


def moeq_moe_layer_shard(x, logits, H, I_shard, E_routed, top_k, w_gu, s_gu, w_d, s_d, out_partial, ws: Workspace,
                         plan: RoutePlan | None = None, h=None, q_x=None, s_x=None, q_h=None, s_h=None,
                         stream=None) -> None:
    M = x.shape[0]
    _check("moeq_moe_layer_shard", load().moeq_moe_layer_shard(
        _p(x), _p(logits), M, H, I_shard, E_routed, top_k, _p(w_gu), _p(s_gu), _p(w_d), _p(s_d), _p(out_partial),
        ctypes.byref(plan.c) if plan is not None else None, _p(h), _p(q_x), _p(s_x), _p(q_h), _p(s_h),
        ws.ptr, ws.nbytes, _stream(stream)))


def moeq_tp_reduce(partials, out, stream=None) -> None:
    R, M, H = partials.shape
    _check("moeq_tp_reduce", load().moeq_tp_reduce(_p(partials), R, M, H, _p(out), _stream(stream)))


def moeq_layer_ws_count_offset(M, H, I, n_experts_incl_shared, top_k, which) -> int:
    return int(load().moeq_layer_ws_count_offset(M, H, I, n_experts_incl_shared, top_k, which))


def moeq_gemm_ws_count_offset(rows_out, K, rows_in, max_uniq, is_gate_up, which) -> int:
    return int(load().moeq_gemm_ws_count_offset(rows_out, K, rows_in, max_uniq, is_gate_up, which))
