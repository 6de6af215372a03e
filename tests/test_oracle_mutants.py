"""Planted mistakes in the oracle (built on the CPU) must each fail a pin.

Each variant of ``oracle/msgl_oracle.c`` compiled with ORACLE_MUTANT=n
carries one plausible slip: 1 drops the diagonal key, 2 maps q heads to kv
heads interleaved instead of grouped, 3 drops the softmax scale, 4 returns
a base-2 LSE, 5 uses the page id as a slot base, 7 reads V from the K pool,
8 forgets the softmax normaliser.  If one of them passed every pin, the
pins would not be tight enough to trust the oracle.
"""
import pytest

import oracle
from tests.test_oracle import PINS

MUTANTS = [1, 2, 3, 4, 5, 7, 8]


@pytest.mark.parametrize("mutant", MUTANTS)
def test_mutant_fails_some_pin(mutant):
    assert oracle.mutant_id(mutant) == mutant
    failed = []
    for pin in PINS:
        try:
            pin(mutant)
        except (AssertionError, oracle.OracleError):
            failed.append(pin.__name__)
    assert failed, f"planted mistake {mutant} passed every pin"
