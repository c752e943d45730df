"""The library's schedule planners (host C++ in libtide) against the
schedule oracle: Equations (6)-(8), Appendix D acceptance (including its
printed counts, through the C ABI), network rounds, stale-block zeroing and
recursive doubling.  CPU only."""
import random

import pytest

from oracle import schedule as sch


@pytest.fixture(scope="module")
def tide():
    from all_gather_gb300 import build
    build.build()
    import all_gather_gb300
    all_gather_gb300.load_library()
    return all_gather_gb300


def test_latin_square_matches_equations(tide):
    rnd = random.Random(3)
    for _ in range(20000):
        M, L = rnd.randint(1, 300), rnd.choice([1, 2, 3, 4, 7, 8, 16, 64])
        m, n, s = rnd.randrange(M), rnd.randrange(M), rnd.randrange(L)
        want = sch.landing_gpu(s, sch.contributor_index(m, n, M), M, L)
        assert tide.tide_latin_square_gpu(s, m, n, M, L) == want
    assert tide.tide_latin_square_gpu(0, 0, 0, 0, 8) == -1
    assert tide.tide_latin_square_gpu(8, 0, 0, 4, 8) == -1


def test_appendix_d_counts_through_the_library(tide):
    accepted = rejected = 0
    for M in range(2, 1025):
        for w_wave in range(1, 9):
            for k in range(1, 33):
                for me in (0, 1):
                    st, _ = tide.tide_rs_wave_plan(M, 8, w_wave, k, me)
                    if st == tide.TIDE_OK:
                        accepted += 1
                    else:
                        rejected += 1
    assert (accepted, rejected) == (458_304, 65_472)


def test_acceptance_and_rounds_match_oracle(tide):
    for L in (2, 4, 8):
        for M in range(1, 200):
            for w_wave in range(1, L + 3):
                for k in (1, 3, 8):
                    st, info = tide.tide_rs_wave_plan(M, L, w_wave, k, 0)
                    assert (st == tide.TIDE_OK) == sch.plan_accepted(M, L, w_wave), (M, L, w_wave)
                    assert info["waves"] == len(sch.waves(M, w_wave))
                    if st == tide.TIDE_OK:
                        assert info["network_rounds"] == sch.network_rounds(M, w_wave, k)
                        assert info["generations"] == (1 if len(sch.waves(M, w_wave)) == 1 else 2)


def test_zero_masks_match_oracle(tide):
    for L in (4, 8):
        for M in range(1, 40):
            for w_wave in range(1, L + 1):
                for me in (0, 1):
                    for entry in sch.inbox_schedule(M, L, w_wave, me):
                        got = tide.tide_rs_wave_zero_mask(M, L, w_wave, me, entry["wave"])
                        want = [0] * L
                        for gpu, s in entry["zero"]:
                            want[gpu] |= 1 << s
                        assert got == want, (M, L, w_wave, me, entry["wave"])


def test_rejection_explains_the_collision(tide):
    st, _ = tide.tide_rs_wave_plan(9, 8, 3, 1, 0)
    assert st == tide.TIDE_ERR_UNSUPPORTED
    assert "contributors 8 and 9" in tide.tide_last_error()
    with pytest.raises(tide.TideError):
        tide.tide_rs_wave_plan(9, 65, 3, 1, 0)


def test_bruck_matches_oracle(tide):
    for M in list(range(1, 300)) + [511, 512, 513, 1024]:
        assert tide.tide_bruck_schedule(M) == sch.bruck_rounds(M)
    with pytest.raises(ValueError):
        tide.tide_bruck_schedule(0)
