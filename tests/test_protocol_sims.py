"""The tensor-core kernels' mbarrier protocols, modelled on the CPU
(tests/protocol_sims) and run under seeded random interleavings of their
roles and of the asynchronous work (TMA loads landing in any order, the
tensor pipe in issue order, bulk reductions reading shared memory late):
no buffer may be overwritten before its reader is done, and no schedule may
leave every role waiting.  Each model also carries planted protocol mistakes
(a missing wait, a release before the read), and each must fail."""
import random

import pytest

from protocol_sims import dkdv_kernel, dq_kernel, fwd_kernel, onepass_kernel

CLEAN_SCHEDULES = 400
MUTANT_SCHEDULES = 2000


def draws(n, seed, choices):
    rng = random.Random(seed)
    return [[rng.choice(choices) for _ in range(rng.randint(1, 5))] for _ in range(n)]


MODELS = {
    # tiles per work item: K/V tiles of a query tile (dQ kernel), query tiles
    # of a K/V tile (dK / dV and one-pass kernels); 0 covers an item with
    # nothing visible.
    "dkdv_kernel": (dkdv_kernel, [0, 1, 1, 2, 3, 5, 7]),
    # forward: the use masks of an item's K/V tiles (1: query tile 0, 2: query
    # tile 1, 3: both), including items where one query tile sees nothing.
    "fwd_kernel": (fwd_kernel, [[], [3], [3, 3], [3, 3, 3, 2], [1], [2, 3], [3, 1],
                                [3, 3, 3, 3, 3], [2], [1, 1], [3, 3, 3, 3, 3, 3, 3]]),
    "dq_kernel": (dq_kernel, [0, 1, 1, 2, 3, 5, 7]),
    "onepass_kernel": (onepass_kernel, [0, 1, 1, 2, 3, 5]),
}


@pytest.mark.parametrize("name", sorted(MODELS))
def test_protocol_holds_under_random_schedules(name):
    model, choices = MODELS[name]
    for seed, items in enumerate(draws(CLEAN_SCHEDULES, 11, choices)):
        model.run(items, seed)


@pytest.mark.parametrize("name,mutation", [(n, m) for n in sorted(MODELS) for m in (1, 2, 3)])
def test_planted_protocol_mistake_is_caught(name, mutation):
    model, choices = MODELS[name]
    for seed, items in enumerate(draws(MUTANT_SCHEDULES, 13, choices)):
        try:
            model.run(items, seed, mutation=mutation)
        except AssertionError:
            return
    pytest.fail(f"{name} mutation {mutation} survived {MUTANT_SCHEDULES} schedules")
