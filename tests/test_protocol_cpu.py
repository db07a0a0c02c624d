"""The prefill kernel's barrier protocol, run as a discrete-event model under
many random timings: every parity wait and probe must pass only on the phase
it means and never be overtaken, and every schedule must finish. The model
also finds the missed-speculation race an earlier version of the kernel had
(the MMA warp waiting for the speculative phase 0 by parity).

The failure path is run the same way: the producer stops issuing loads at a
key tile (the debug library's injected stall), every wait is bounded, and
each schedule must end with some wait having given up, no copy in flight
when the CTA exits and no MMA in flight when the tensor memory is freed."""
import random

import pytest

from _pipeline_model import Model, ProtocolError


@pytest.mark.parametrize("rope", [False, True])
@pytest.mark.parametrize("NT", [1, 2])
@pytest.mark.parametrize("STAGES", [2, 3])
@pytest.mark.parametrize("spec_miss", [False, True])
def test_every_schedule_is_sound(NT, STAGES, spec_miss, rope):
    for nk in range(0, 7):
        for seed in range(60):
            rng = random.Random(1000003 * seed + 7919 * nk + 31 * NT + STAGES + (5 if spec_miss else 0))
            Model(NT, STAGES, nk, spec_miss, rng, rope=rope).run()


def test_model_finds_the_old_speculation_race():
    found = []
    for seed in range(400):
        rng = random.Random(seed)
        try:
            Model(2, 2, 4, True, rng, variant="old-speculation").run()
        except ProtocolError as e:
            found.append(str(e))
    assert found, "the old protocol passed every schedule"
    assert any("two phases past" in f or "older phase" in f for f in found), found[:3]


@pytest.mark.parametrize("rope", [False, True])
@pytest.mark.parametrize("NT", [1, 2])
@pytest.mark.parametrize("STAGES", [2, 3])
@pytest.mark.parametrize("spec_miss", [False, True])
def test_stalled_producer_ends_cleanly(NT, STAGES, spec_miss, rope):
    for nk in range(2, 7):
        for stop in range(1, nk):
            for seed in range(25):
                rng = random.Random(7919 * seed + 131 * nk + 17 * stop + NT + STAGES)
                m = Model(NT, STAGES, nk, spec_miss, rng, stop_at=stop, rope=rope)
                m.run()
                assert m.timeouts, "the stall was not noticed"


def test_model_finds_a_missing_failure_drain():
    found = []
    for seed in range(200):
        try:
            Model(2, 2, 4, False, random.Random(seed), variant="no-failure-drain", stop_at=2).run()
        except ProtocolError as e:
            found.append(str(e))
    assert any("MMA is still in flight" in f for f in found), found[:3]
