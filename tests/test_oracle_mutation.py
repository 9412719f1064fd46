"""Planted mistakes: each plausible slip planted in the ORACLE (CPU only)
must make at least one pin fail.  This checks the pins, not the GPU path."""
import pytest

import test_oracle_codec as tc
import test_oracle_gemm as tg
import test_oracle_layer as tl
import test_oracle_quant as tq
import test_oracle_route as tr

PINS = [
    tc.test_decode_matches_torch_all_codes, tc.test_midpoints_round_to_even,
    tc.test_encode_matches_torch_in_range, tq.test_quant_hand_cases,
    tg.test_gemm_hand_case, tg.test_gemm_brute_force_numpy, tg.test_gemm_single_block_isolation,
    tg.test_gemm_is_the_sum_of_its_k_groups,
    tr.test_route_hand_cases, tr.test_swiglu_closed_forms, tl.test_layer_brute_force,
]

FAULTS = {
    1: "subnormal decode off by 2x",
    2: "ties rounded away from even",
    3: "scale constant 447 instead of 448",
    4: "last product of each group dropped",
    5: "weight block scales transposed",
    6: "routing ties to the higher id",
    7: "wrong sign in silu",
    8: "weight operand transposed",
    9: "shared expert dropped from the combine",
}


def _needs_golden(fn):
    return fn.__code__.co_varnames[: fn.__code__.co_argcount]


@pytest.mark.parametrize("fault", sorted(FAULTS))
def test_planted_mistake_is_caught(orc, golden_dir, fault):
    caught = []
    orc.set_fault(fault)
    try:
        for fn in PINS:
            args = {"orc": orc, "golden_dir": golden_dir}
            try:
                fn(**{a: args[a] for a in _needs_golden(fn)})
            except AssertionError:
                caught.append(fn.__name__)
            except ValueError:
                caught.append(fn.__name__)
    finally:
        orc.set_fault(0)
    assert caught, f"planted mistake {fault} ({FAULTS[fault]}) passed every pin"
