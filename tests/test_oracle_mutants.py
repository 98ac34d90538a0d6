"""Each planted mistake of the pages' pitfalls table (s01..s15), built into its
own copy of the oracle on the CPU, must be rejected by the pin the table names,
while the unmodified oracle passes every pin."""
import pytest

import oracle
import pins


@pytest.mark.parametrize("mutant", sorted(pins.KILLS))
def test_planted_mistake_is_rejected(mutant):
    bad = oracle.Oracle(mutant)
    killer = pins.KILLS[mutant]
    with pytest.raises(AssertionError):
        pins.PINS[killer](bad)


def test_unmodified_oracle_is_not_a_mutant(orc):
    assert orc.lib.orc_mutant() == 0
