"""Each planted mistake in the oracle (compiled with -DORACLE_MUTATION=k, on the
CPU) must be caught by at least one pin; the unmutated oracle passes all.

Mutations: 1 drops 1/sqrt(d); 2 starts the recurrence at m=0; 3 uses floor 1
in the stabilized normalizer; 4 shifts the forget-sum index; 5 leaves the
input gate unrescaled in the step; 6 drops |.| on the row sum; 7 uses an
exponential forget activation; 8 transposes q and k.  In the backward: 9
takes eq (90)'s printed sign(n) literally; 10 drops the db term of eq (92);
11 lets eq (102)'s inner sum include j = k; 12 uses K instead of Q in eq (99).
In the recurrent backward: 13 drops Omega's negative branch; 14 takes
sigma for sigma' in eq (68).
"""
import pytest

import oracle
import pins


@pytest.mark.parametrize("mutation", range(1, 15))
def test_mutation_is_caught(mutation):
    assert oracle._lib(mutation).oracle_mutation() == mutation
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(mutation)
        except AssertionError as e:
            caught.append(f"{pin.__name__}: {e}")
    assert caught, f"mutation {mutation} passed every pin"
