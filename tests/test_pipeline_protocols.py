"""CPU model check of the kernels' mbarrier pipelines (tests/protocol_model.py): the forward
(128-key steps, block-sparse streams with gaps, the d = 64 half steps), the dK/dV kernel (its
d = 128 and d = 64 layouts, with the dQ claims and, at d = 64, the staged TMA additions) and the
deterministic dQ kernel run their roles' waits, arrivals
and buffer reads and writes under many random interleavings (and the dK/dV kernel's CTAs their
claims on the shared dQ accumulator), for every per-tile step count up to
a few stages past the ring's length; no deadlock, no wait on a wrong phase, no read of a stage
before its copy or after its release.  Planted protocol errors (among them the dO race once found in
the dK/dV kernel) must fail."""

import pytest

from protocol_model import dkdv, dq_claims, dq_kernel, forward


def _tile_steps(nmax):
    # tile 1 never has steps without tile 0 (its rows come after tile 0's); under a causal mask
    # it has more, without one the same
    return [(a, b) for a in range(nmax + 1) for b in range(nmax + 1) if not (a == 0 and b > 0)]


@pytest.mark.parametrize("half,S", [(False, 2), (False, 4), (True, 2)],
                         ids=["128-key-2-stages", "128-key-4-stages", "half-step-2-stages"])
def test_forward_protocol(half, S):
    for n0, n1 in _tile_steps(9):
        for seed in range(8):
            forward((n0, n1), S, half, seed)


@pytest.mark.parametrize("S", [2, 4])
def test_block_sparse_forward_protocol(S):
    """Block-sparse K/V streams: each position is kept by tile 0, tile 1 or both, with gaps."""
    import random

    rng = random.Random(5)
    for length in range(1, 9):
        for _ in range(20):
            uses = [rng.choice((1, 2, 3)) for _ in range(length)]
            for seed in range(4):
                forward(None, S, False, seed, uses=uses)


@pytest.mark.parametrize("d64", [False, True], ids=["d128", "d64"])
@pytest.mark.parametrize("groups", [2, 4])
@pytest.mark.parametrize("with_dq", [True, False])
def test_dkdv_protocol(d64, groups, with_dq):
    for nit in range(0, 9):
        for seed in range(12):
            dkdv(nit, seed, d64=d64, groups=groups, with_dq=with_dq)


def test_deterministic_dq_protocol():
    for nb in range(0, 10):
        for seed in range(12):
            dq_kernel(nb, seed)


def _fails(fn):
    for seed in range(200):
        try:
            fn(seed)
        except AssertionError:
            return True
    return False


@pytest.mark.parametrize("d64,bug", [(False, "dv_before_do"), (False, "early_q_release"),
                                     (True, "early_q_release"), (True, "no_stage_wait"),
                                     (True, "no_mode_wait")])
def test_checker_catches_dkdv_protocol_errors(d64, bug):
    assert _fails(lambda seed: dkdv(6, seed, d64=d64, bug=bug))


def test_early_do_release_is_harmless_under_this_producer_order():
    for seed in range(100):
        dkdv(6, seed, bug="early_do_release")


@pytest.mark.parametrize("half", [False, True])
def test_checker_catches_an_early_stage_release(half):
    assert _fails(lambda seed: forward((5, 7), 2, half, seed, bug="early_k_release"))


def test_checker_catches_an_overwrite_of_unread_scores():
    assert _fails(lambda seed: dq_kernel(6, seed, bug="s_before_read"))


def _abort_runs(half, S, conditional_drain=False):
    """Sims of forward runs in which one wait, at many points of many runs, times out."""
    import random

    rng = random.Random(11)
    for n0, n1 in [(1, 1), (3, 4), (6, 8), (7, 7)]:
        for seed in range(6):
            spins = forward((n0, n1), S, half, seed).spins
            for abort_at in sorted(rng.sample(range(1, max(2, spins + 1)), min(8, spins))):
                yield forward((n0, n1), S, half, seed, abort_at=abort_at,
                              conditional_drain=conditional_drain)


@pytest.mark.parametrize("half,S", [(False, 2), (False, 4), (True, 2)],
                         ids=["128-key-2-stages", "128-key-4-stages", "half-step-2-stages"])
def test_forward_timeout_every_role_leaves(half, S):
    """A wait that runs past its limit, at any point of any role: every role leaves (no
    deadlock), and when the CTA exits no MMA is queued and no copy is in flight (the producer
    waits for its last copies whether or not the CTA has aborted)."""
    for sim in _abort_runs(half, S):
        assert sim.abort and sim.exit_ops == 0 and sim.exit_copies == 0


def test_checker_catches_a_drain_only_when_already_aborted():
    """The kernels' producers once waited for their last copies only if the abort flag was
    already set when they left their loop; if another role timed out after that, a copy issued
    just before could still be in flight when the CTA exited and land in the shared memory of
    the SM's next CTA.  The checker finds that form in all three kernels."""
    assert any(sim.exit_copies > 0 for sim in _abort_runs(False, 2, conditional_drain=True))
    assert any(sim.exit_copies > 0 for sim in _dkdv_abort_runs(True, conditional_drain=True))
    assert any(sim.exit_copies > 0 for sim in _dq_abort_runs(conditional_drain=True))


def _dkdv_abort_runs(with_dq, conditional_drain=False, d64=False):
    import random

    rng = random.Random(13)
    for nit in (1, 2, 5, 8):
        for seed in range(5):
            spins = dkdv(nit, seed, d64=d64, with_dq=with_dq).spins
            for abort_at in sorted(rng.sample(range(1, max(2, spins + 1)), min(8, spins))):
                yield dkdv(nit, seed, d64=d64, with_dq=with_dq, abort_at=abort_at,
                           conditional_drain=conditional_drain)


def _dq_abort_runs(conditional_drain=False):
    import random

    rng = random.Random(17)
    for nb in (1, 2, 5, 8):
        for seed in range(5):
            spins = dq_kernel(nb, seed).spins
            for abort_at in sorted(rng.sample(range(1, max(2, spins + 1)), min(8, spins))):
                yield dq_kernel(nb, seed, abort_at=abort_at, conditional_drain=conditional_drain)


@pytest.mark.parametrize("d64", [False, True], ids=["d128", "d64"])
@pytest.mark.parametrize("with_dq", [True, False])
def test_dkdv_timeout_every_role_leaves(with_dq, d64):
    """The dK/dV kernel's timeout path: a wait runs out at any point of any role; every role
    leaves, and the CTA exits with no MMA queued and no copy (or TMA addition) in flight."""
    for sim in _dkdv_abort_runs(with_dq, d64=d64):
        assert sim.abort and sim.exit_ops == 0 and sim.exit_copies == 0


def test_deterministic_dq_timeout_every_role_leaves():
    """The same for the deterministic dQ kernel."""
    for sim in _dq_abort_runs():
        assert sim.abort and sim.exit_ops == 0 and sim.exit_copies == 0


@pytest.mark.parametrize("causal", [True, False])
def test_dq_claims_across_ctas(causal):
    """The dK/dV kernel's CTAs sharing the dQ accumulator: whatever the interleaving, the memory
    delays and the number of CTAs resident at a time (down to one: no CTA may wait for one that
    cannot start), every query tile ends with each contribution exactly once, the first partial
    stored before any addition reaches it."""
    for nkt in (1, 2, 3, 5, 8):
        for resident in (1, 2, 3, 8):
            for seed in range(8):
                dq_claims(nkt, causal, seed, resident=resident)


def test_dq_claims_in_any_claim_order():
    """Claims made out of the drains' order (all at a CTA's start) only make later claimants wait
    longer; the result is the same."""
    for causal in (True, False):
        for seed in range(20):
            dq_claims(6, causal, seed, resident=3, bug="claim_at_start")


@pytest.mark.parametrize("bug", ["no_wait", "no_fence"])
def test_checker_catches_dq_claim_errors(bug):
    assert _fails(lambda seed: dq_claims(5, True, seed, resident=5, bug=bug))
    assert _fails(lambda seed: dq_claims(5, False, seed, resident=5, bug=bug))


def test_dq_claims_timeout_every_role_leaves():
    """A wait (of any CTA) that runs past its limit: every role of every CTA leaves."""
    import random

    rng = random.Random(19)
    for causal in (True, False):
        for seed in range(6):
            spins = dq_claims(5, causal, seed, resident=3).spins
            for abort_at in sorted(rng.sample(range(1, max(2, spins + 1)), min(6, spins))):
                assert dq_claims(5, causal, seed, resident=3, abort_at=abort_at).abort
