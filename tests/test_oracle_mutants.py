"""Every deliberately wrong oracle build must fail at least one pin (CPU only).

The wrong variants are compiled from the oracle source with ORACLE_PLANT=k:
1 scale dropped, 2 causal diagonal excluded, 3 GQA head map h % Hkv,
4 query/key operands transposed, 5 LSE without the row maximum,
6 sign of the max shift flipped.
"""
import pytest

import oracle
import oracle_pins as P


@pytest.mark.parametrize("plant", [1, 2, 3, 4, 5, 6])
def test_planted_mistake_is_caught(plant, golden_dir):
    oracle.build(plant)
    failed = []
    for name in P.ALL_PINS:
        fn = getattr(P, name)
        try:
            if name == "pin_worked_example":
                fn(golden_dir, plant=plant)
            else:
                fn(plant=plant)
        except AssertionError:
            failed.append(name)
    assert failed, f"planted mistake {plant} passed every pin"
    print(f"plant {plant} caught by {failed}")


def test_real_oracle_is_not_a_plant():
    assert oracle._load(0).oracle_plant() == 0
