"""The oracle's pins catch plausible mistakes planted in the oracle (on the CPU).

Each mutant (see ORACLE_MUTANT in oracle/cake_oracle.c) plants one mistake --
a dropped term, a transposed operand, a reduction that runs past its expert,
the wrong expert's weights, a wrong sign, a router split without its low
part.  Every mutant must fail at least one of the pins in test_oracle_pins.py
and test_oracle_router.py.
"""
import pytest

import oracle
import test_oracle_pins as pins
import test_oracle_router as rpins

PIN_CALLS = [
    lambda lib: pins.test_hand_worked_golden(lib),
    lambda lib: pins.test_e1_is_one_dense_gemm(lib, 48, 64, 37),
    lambda lib: pins.test_per_expert_blocks_are_dense_gemms(lib),
    lambda lib: pins.test_wgrad_sum_over_experts_identity(lib),
    lambda lib: pins.test_exact_integer_inputs(lib),
    lambda lib: pins.test_one_hot_inputs_select_weights(lib),
    lambda lib: pins.test_zero_inputs_and_empty_expert(lib),
    lambda lib: pins.test_rows_beyond_last_offset_do_not_contribute(lib),
    lambda lib: pins.test_pure_python_brute_force(lib),
    lambda lib: rpins.test_hand_worked_product(lib),
    lambda lib: rpins.test_pure_python_restatement(lib),
    lambda lib: rpins.test_emulation_error_bound(lib),
]


def test_unmutated_oracle_passes_every_pin(oracle_lib):
    for call in PIN_CALLS:
        call(oracle_lib)


@pytest.mark.parametrize("mutant", [1, 2, 3, 4, 5, 6])
def test_each_planted_mistake_fails_a_pin(mutant):
    lib = oracle.load(mutant=mutant)
    failures = 0
    for call in PIN_CALLS:
        try:
            call(lib)
        except (AssertionError, ValueError):
            failures += 1
    assert failures >= 1, f"mutant {mutant} passed every pin"
