"""The mbarrier ring protocol of the TMA producers, restated and checked on the CPU.

Every kernel streams operand tiles through a ring of S shared-memory stages:
copy number i goes to stage i mod S and completes phase i // S of that stage's
`full` barrier; a wait for "parity p" on a barrier returns once the most recent
phase with that parity has completed.  After its loop a producer calls
`drain_ring(full, S, issued)`, which for each stage s < min(S, issued) waits on
parity (fills(s) - 1) & 1 with fills(s) = issued // S + (s < issued % S).  The
tests below check, against a brute-force simulation of the ring, that this is
the parity of the last phase armed on each stage (so the CTA cannot exit while
any copy it issued is still landing) and that the consumers' running
(stage, parity) pair and the producer's refill condition agree with it.
"""
import pytest


def drain_targets(stages, issued):
    """(stage, parity) pairs drain_ring waits on, as the device code computes them."""
    out = []
    for s in range(min(stages, issued)):
        fills = issued // stages + (1 if s < issued % stages else 0)
        out.append((s, (fills - 1) & 1))
    return out


def simulated_last_phases(stages, issued):
    """Brute force: issue copies one by one, remember the last phase armed on each stage."""
    last = {}
    for i in range(issued):
        last[i % stages] = i // stages
    return sorted((s, ph & 1) for s, ph in last.items())


@pytest.mark.parametrize("stages", [1, 3, 4, 8])
def test_drain_waits_for_the_last_phase_of_every_stage(stages):
    for issued in range(0, 5 * stages + 3):
        assert drain_targets(stages, issued) == simulated_last_phases(stages, issued), (stages, issued)


@pytest.mark.parametrize("stages", [3, 4, 8])
def test_consumer_and_producer_parities_agree(stages):
    # consumer: running (s, phase) flipped every time s wraps; producer: before
    # copy i >= S it waits on `empty` parity (i // S - 1) & 1, the phase the
    # consumers completed when they released copy i - S of the same stage.
    s, phase = 0, 0
    released = {}
    for i in range(6 * stages):
        assert (s, phase) == (i % stages, (i // stages) & 1)
        released[i] = (s, phase)           # consumers arrive on empty[s] for copy i
        if (s := s + 1) == stages:
            s, phase = 0, phase ^ 1
    for i in range(stages, 6 * stages):
        stage, parity = i % stages, (i // stages - 1) & 1
        assert released[i - stages] == (stage, parity)
