"""Host-side checks of the C ABI (no GPU): the library builds and loads,
exports every symbol include/moeq.h declares, and rejects bad arguments
before touching a device."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "moeq.h")


@pytest.fixture(scope="module")
def lib():
    from bandwidth_bound_fp8_gb300 import build, moeq
    build.build()
    return moeq.load()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moeq_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_four_path_calls():
    names = _declared()
    for n in ("moeq_quant_act", "moeq_expert_gemm_gateup_swiglu", "moeq_expert_gemm_down", "moeq_moe_layer"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from bandwidth_bound_fp8_gb300 import moeq
    names = _declared()
    assert sorted(moeq.EXPORTS) == names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    from bandwidth_bound_fp8_gb300 import moeq
    assert moeq.moeq_abi_version() == 2
    for s in range(7):
        assert moeq.status_string(s)
    assert moeq.status_string(99) == "unknown status"


def test_plan_sizes(lib):
    from bandwidth_bound_fp8_gb300 import moeq
    assert moeq.moeq_max_uniq(1, 256, 8) == 9
    assert moeq.moeq_max_uniq(16, 256, 8) == 129
    assert moeq.moeq_max_uniq(64, 256, 8) == 257
    assert moeq.moeq_max_pairs(16, 8) == 144
    assert moeq.moeq_route_plan_bytes(1, 256, 8) > 0
    assert moeq.moeq_route_plan_bytes(17, 256, 8) == 0      # M above the limit
    assert moeq.moeq_route_plan_bytes(1, 256, 0) == 0
    assert moeq.moeq_route_plan_bytes(1, 4, 8) == 0         # k > E


def test_plan_carve_layout(lib):
    from bandwidth_bound_fp8_gb300 import moeq
    M, E, k = 4, 256, 8
    n = moeq.moeq_route_plan_bytes(M, E, k)
    buf = ctypes.create_string_buffer(n + 16)
    base = (ctypes.addressof(buf) + 15) // 16 * 16
    plan = moeq.moeq_route_plan()
    assert lib.moeq_route_plan_carve(base, n, M, E, k, ctypes.byref(plan)) == 0
    fields = [plan.topk_id, plan.topk_w, plan.n_uniq, plan.uniq, plan.offs, plan.pair_tok, plan.pair_of]
    assert all(f % 16 == 0 for f in fields)
    assert fields == sorted(fields) and fields[0] == base and fields[-1] + 4 * M * (k + 1) <= base + n
    assert lib.moeq_route_plan_carve(base, n - 1, M, E, k, ctypes.byref(plan)) == 3   # too small
    assert lib.moeq_route_plan_carve(base + 4, n, M, E, k, ctypes.byref(plan)) == 1   # misaligned


def test_argument_validation_without_device(lib):
    """Bad arguments are rejected on the host before any device query."""
    buf = ctypes.create_string_buffer(1 << 16)
    p = (ctypes.addressof(buf) + 255) // 256 * 256
    plan_bad = None
    # null / misaligned pointers, bad dtype, bad M
    assert lib.moeq_quant_act(None, 0, 1, 128, p, p, None) == 1
    assert lib.moeq_quant_act(p + 2, 0, 1, 128, p, p, None) == 1
    assert lib.moeq_quant_act(p, 7, 1, 128, p, p, None) == 1
    assert lib.moeq_quant_act(p, 0, 0, 128, p, p, None) == 1
    # K not a multiple of 128
    assert lib.moeq_quant_act(p, 0, 1, 100, p, p, None) == 2
    assert lib.moeq_quant_weight(p, 1, 128, 200, p, p, None) == 2
    assert lib.moeq_route(p, 1, 256, 8, plan_bad, None) == 1
    # gate_up: M above 16, H not a multiple of 128, half-given dump
    args = [p, 0, 17, 256, 128, p, p, 1, p, p, p, p, 1, 1, p, None, None, p, 1 << 16, None]
    assert lib.moeq_expert_gemm_gateup_swiglu(*args) == 1
    args[2], args[3] = 1, 200
    assert lib.moeq_expert_gemm_gateup_swiglu(*args) == 2
    args[3], args[15] = 256, p
    assert lib.moeq_expert_gemm_gateup_swiglu(*args) == 1
    # down: N not a multiple of 128
    assert lib.moeq_expert_gemm_down(p, 0, 256, 100, p, p, 1, p, p, p, 1, 1, p, None, None, p, 1 << 16, None) == 2
    # layer: k > E, then M = 0
    assert lib.moeq_moe_layer(p, p, 1, 256, 128, 4, 8, p, p, p, p, p, None, None, None, None, None, None, None,
                              None, p, 1 << 16, None) == 1
    assert lib.moeq_moe_layer(p, p, 0, 256, 128, 8, 2, p, p, p, p, p, None, None, None, None, None, None, None,
                              None, p, 1 << 16, None) == 1
    # combine with top_k > 0 but no weights
    plan = __import__("bandwidth_bound_fp8_gb300.moeq", fromlist=["x"]).moeq_route_plan()
    plan.pair_of = p
    assert lib.moeq_combine(p, 256, ctypes.byref(plan), 1, 8, p, None) == 1
    # workspace init: null or tiny
    assert lib.moeq_workspace_init(None, 1024, None) == 3
    assert lib.moeq_workspace_init(p, 16, None) == 3


def test_dense_ffn_workspace_size_rejects_shapes(lib):
    """moeq_dense_ffn serves 1..16 tokens, H a multiple of 256 up to 6144, I
    a multiple of 128: other shapes get a zero workspace size (and the call
    MOEQ_ERR_UNSUPPORTED_SHAPE)."""
    assert lib.moeq_dense_ffn_workspace_size(0, 512, 256) == 0
    assert lib.moeq_dense_ffn_workspace_size(17, 512, 256) == 0
    assert lib.moeq_dense_ffn_workspace_size(1, 384, 256) == 0
    assert lib.moeq_dense_ffn_workspace_size(1, 8192, 256) == 0
    assert lib.moeq_dense_ffn_workspace_size(1, 512, 200) == 0


def test_stack_rejects_layer_count_before_the_device(lib):
    """moeq_moe_stack checks L (1 .. MOEQ_MAX_LAYERS) before it looks for a
    device; the workspace size is 0 outside that range."""
    assert lib.moeq_stack_workspace_size(0, 1, 512, 256, 17, 4) == 0
    assert lib.moeq_stack_workspace_size(257, 1, 512, 256, 17, 4) == 0
    arr = (ctypes.c_void_p * 1)(16)
    st = lib.moeq_moe_stack(0, 16, 16, 1, 512, 256, 16, 4, arr, arr, arr, arr, 16, 0, 16, 1 << 20, None)
    assert st == 1   # MOEQ_ERR_INVALID_ARG
