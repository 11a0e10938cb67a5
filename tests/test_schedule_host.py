"""The library's host-side schedule calls (indexshare_schedule_score / _search) against the
oracle's plain walk and exhaustive enumeration, on seeded random overlap matrices: the best
score is unique, the returned schedule must be one of the oracle's best ones (CPU only)."""
import numpy as np
import pytest

import long_context_sparse_tcgen05_gb300 as dsa
import oracle
from long_context_sparse_tcgen05_gb300 import build as dsa_build


@pytest.fixture(scope="module", autouse=True)
def _lib():
    dsa_build.build()
    dsa.load_library()


def _matrices(n, seed):
    rng = np.random.default_rng(seed)
    a = rng.uniform(0.2, 1.0, (n, n))
    sym = (a + a.T) / 2
    np.fill_diagonal(sym, 1.0)
    np.fill_diagonal(a, 1.0)
    # block structure: clusters of layers overlap strongly inside, weakly across
    c = rng.integers(0, 3, n)
    blk = np.where(c[:, None] == c[None, :], 0.9, 0.4) + rng.uniform(-0.05, 0.05, (n, n))
    np.fill_diagonal(blk, 1.0)
    return [sym, a, blk]


@pytest.mark.parametrize("n", [1, 2, 5, 9, 12])
def test_schedule_search_matches_enumeration(n):
    for M in _matrices(n, 100 + n):
        for n_full in range(1, n + 1):
            sched, score = dsa.indexshare_schedule_search(M.tolist(), n_full)
            best, arg = oracle.schedule_search(M, n_full)
            assert sched.count("F") == n_full and sched[0] == "F" and len(sched) == n
            assert score == pytest.approx(best, abs=1e-12)
            assert sched in arg
            assert dsa.indexshare_schedule_score(M.tolist(), sched) == pytest.approx(
                oracle.schedule_score(M, sched), abs=1e-12)


def test_schedule_score_matches_oracle_on_random_schedules():
    rng = np.random.default_rng(7)
    M = _matrices(16, 7)[2]
    for _ in range(200):
        s = "F" + "".join(rng.choice(["F", "S"], 15))
        assert dsa.indexshare_schedule_score(M.tolist(), s) == pytest.approx(
            oracle.schedule_score(M, s), abs=1e-12)
