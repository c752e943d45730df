"""Pins of the schedule-planner oracle (oracle/schedule.py) to the TIDE paper:
the exhaustive validation counts Appendix D prints, Proposition 4.1, the
paper's own colliding example, the Latin square of Figure 6b and the
recursive-doubling rounds of Figure 5a."""
import functools

import pytest

from oracle import schedule as sch

L8 = 8


@functools.lru_cache(maxsize=None)
def _accepted(M, L, w_wave):
    return sch.plan_accepted(M, L, w_wave)


def test_appendix_d_counts():
    """Appendix D: over M in [2, 1024] at L = 8, 458,304 base plans
    (M, W_wave, k, me) are accepted and 65,472 colliding plans rejected.
    Plan space (the one reading that gives both counts): W_wave in 1..8,
    k in 1..32 concurrent rail transfers, me in {0, 1}; acceptance depends
    on (M, W_wave) only."""
    accepted = rejected = 0
    for M in range(2, 1025):
        for w_wave in range(1, L8 + 1):
            ok = _accepted(M, L8, w_wave)
            n = 32 * 2  # k, me
            accepted += n if ok else 0
            rejected += 0 if ok else n
    assert (accepted, rejected) == (458_304, 65_472)


def test_proposition_4_1_divisor_widths_never_collide():
    for L in (2, 4, 8):
        for w_wave in [d for d in range(1, L + 1) if L % d == 0]:
            for M in range(2, 300):
                assert _accepted(M, L, w_wave), (M, L, w_wave)


def test_paper_collision_example():
    """M = 9, L = 8, W_wave = 3: wave 2 holds c in {7, 8, 9}; c = 8 and the
    own node c = 9 both have (c mod 9) mod 8 = 0, so they collide."""
    ws = sch.waves(9, 3)
    assert ws[2] == [7, 8, 9]
    assert sch.wave_collides(ws[2], 9, 8)
    assert not sch.wave_collides(ws[2][:2], 9, 8)
    assert not sch.plan_accepted(9, 8, 3)


def test_figure_6b_latin_square():
    """Figure 6b (L = 4): destination D (own node, c_bar = 0) and contributors
    A, B, C with c_bar = 1, 2, 3; GPU j holds, for sub-slices s = 0..3,
    GPU0: D A B C, GPU1: C D A B, GPU2: B C D A, GPU3: A B C D."""
    L, M = 4, 4
    name = {0: "D", 1: "A", 2: "B", 3: "C"}
    rows = {}
    for j in range(L):
        row = []
        for s in range(L):
            cbar = [cb for cb in range(L) if sch.landing_gpu(s, cb if cb else M, M, L) == j]
            assert len(cbar) == 1
            row.append(name[cbar[0]])
        rows[j] = "".join(row)
    assert rows == {0: "DABC", 1: "CDAB", 2: "BCDA", 3: "ABCD"}


def test_equations_6_to_8_are_consistent():
    """Eq. (7) and Eq. (8) are inverse: local rank j of a contributor picks
    sub-slice s = (j + c_bar) mod L, which lands on GPU j."""
    for M in (2, 5, 9, 64):
        for L in (2, 4, 8):
            for m in range(M):
                for n in range(M):
                    c = sch.contributor_index(m, n, M)
                    assert 1 <= c <= M and (c == M) == (n == m)
                    for j in range(L):
                        assert sch.landing_gpu(sch.sub_slice(j, c, M, L), c, M, L) == j


def test_stale_blocks_zeroed():
    """Appendix D: accepted plans are stale-block free (with zeroing)."""
    for M in range(2, 70):
        for w_wave in range(1, L8 + 1):
            if _accepted(M, L8, w_wave):
                for me in (0, 1):
                    assert sch.stale_block_free(M, L8, w_wave, me), (M, w_wave, me)


def test_figure_5a_recursive_doubling():
    """Figure 5a, M = 5: three rounds adding 1, 2 and 1 shards; node 0 holds
    0 1, then 0 1 2 3, then 0 1 2 3 4."""
    assert [(d, c) for d, c, _ in sch.bruck_rounds(5)] == [(0, 1), (1, 2), (2, 1)]
    held = [[n] for n in range(5)]
    seen = []
    for d, c, step in sch.bruck_rounds(5):
        held = [held[n] + held[(n + step) % 5][:c] for n in range(5)]
        seen.append(held[0])
    assert seen == [[0, 1], [0, 1, 2, 3], [0, 1, 2, 3, 4]]


@pytest.mark.parametrize("M", list(range(1, 70)) + [127, 128, 129, 1000, 1024])
def test_recursive_doubling_covers_every_node(M):
    """Section 3.1: the c_d sum to M - 1, so every node ends with all M shards
    exactly once, in ceil(log2 M) rounds."""
    rounds = sch.bruck_rounds(M)
    assert sum(c for _, c, _ in rounds) == M - 1
    assert len(rounds) == (M - 1).bit_length()
    for n, held in enumerate(sch.bruck_simulate(M)):
        assert sorted(held) == list(range(M)), n
