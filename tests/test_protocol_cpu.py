"""The prefill kernel's barrier protocol, run as a discrete-event model under
many random timings: every parity wait and probe must pass only on the phase
it means and never be overtaken, and every schedule must finish. The model
also finds the missed-speculation race an earlier version of the kernel had
(the MMA warp waiting for the speculative phase 0 by parity)."""
import random

import pytest

from _pipeline_model import Model, ProtocolError


@pytest.mark.parametrize("NT", [1, 2])
@pytest.mark.parametrize("STAGES", [2, 3])
@pytest.mark.parametrize("spec_miss", [False, True])
def test_every_schedule_is_sound(NT, STAGES, spec_miss):
    for nk in range(0, 7):
        for seed in range(60):
            rng = random.Random(1000003 * seed + 7919 * nk + 31 * NT + STAGES + (5 if spec_miss else 0))
            Model(NT, STAGES, nk, spec_miss, rng).run()


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
