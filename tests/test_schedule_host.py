"""Host logic of the stale-factor schedule (no GPU): KfacStep.refresh_due
against the oracle's schedule predicate, and argument checks."""
import pytest

import oracle
from second_order_optimisation_gb300.step import KfacStep


@pytest.mark.parametrize("warmup,every", [(0, 1), (0, 5), (3, 2), (10, 20), (1, 7)])
def test_refresh_due_matches_oracle(warmup, every):
    st = KfacStep([], 32, device="cpu", update_every=every, warmup=warmup)
    assert [st.refresh_due(t) for t in range(60)] == [bool(oracle.is_refresh_step(t, warmup, every))
                                                     for t in range(60)]
    # refresh steps in the steady state are exactly every-th apart
    ref = [t for t in range(warmup, 60) if st.refresh_due(t)]
    assert all(b - a == every for a, b in zip(ref, ref[1:]))


def test_schedule_arguments_checked():
    with pytest.raises(ValueError):
        KfacStep([], 32, device="cpu", update_every=0)
    with pytest.raises(ValueError):
        KfacStep([], 32, device="cpu", warmup=-1)
    with pytest.raises(ValueError):
        KfacStep([], 32, device="cpu", weights=[None])
