"""Host model of the tile-barrier protocol of the prefill kernels (CPU).

The TMA producer loads chunk j of a key (value) stream into ring slot j % R
once chunk j - R has been consumed; the chunks of tile u complete on tile
barrier u % NB; the MMA issuer waits once per tile, then consumes and frees
the tile's chunks in order.  A barrier may be re-armed only after its
previous phase has been waited for, or the two phases mix.  With NB = R
barriers this holds for every tile size the kernels use (1-4 key chunks of a
5-slot ring, 1-2 value chunks of a 3-slot ring); with only two barriers it
breaks for tiles of one or two chunks, which this model must detect."""
import random

import pytest


def _first_violation(R, kc, NB, ntiles=40, seeds=200):
    for seed in range(seeds):
        rng = random.Random(seed)
        nchunks = ntiles * kc
        loaded = consumed = 0
        waited = -1
        while consumed < nchunks:
            t_cons = consumed // kc
            acts = []
            if loaded < nchunks and loaded - R < consumed:
                acts.append("load")
            if waited < t_cons and loaded >= (t_cons + 1) * kc:
                acts.append("wait")
            if waited >= t_cons:
                acts.append("consume")
            assert acts, "the protocol deadlocked"
            a = rng.choice(acts)
            if a == "load":
                u, c = divmod(loaded, kc)
                if c == 0 and u >= NB and waited < u - NB:
                    return (seed, u)
                loaded += 1
            elif a == "wait":
                waited = t_cons
            else:
                consumed += 1
    return None


@pytest.mark.parametrize("R,kc", [(5, 1), (5, 2), (5, 3), (5, 4), (3, 1), (3, 2)])
def test_one_barrier_per_ring_slot_is_safe(R, kc):
    assert _first_violation(R, kc, NB=R) is None


@pytest.mark.parametrize("R,kc", [(5, 1), (5, 2), (3, 1)])
def test_two_barriers_are_unsafe_for_short_tiles(R, kc):
    assert _first_violation(R, kc, NB=2) is not None
