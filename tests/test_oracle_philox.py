"""Oracle pins: Philox4x32-10 and the uniform / Gumbel conversion."""
import numpy as np
import pytest
from scipy import stats

from conftest import load_golden


def test_philox_known_answers(oracle_mod):
    kat = load_golden("philox_kat.json")
    for v in kat["vectors"]:
        ctr = [int(x, 16) for x in v["ctr"]]
        key = [int(x, 16) for x in v["key"]]
        out = oracle_mod.philox(ctr, key)
        assert [int(x) for x in out] == [int(x, 16) for x in v["out"]]


def test_uniform_uses_the_stated_counter_and_word(oracle_mod):
    # u is built from word (e & 3) of Philox((e >> 2, pos, req, (round << 3) | purpose), (seed lo, seed hi))
    seed, rnd, purpose, req, pos = 0x0123456789ABCDEF, 5, 3, 17, 9
    for e in range(12):
        ctr = [e >> 2, pos, req, ((rnd << 3) | purpose) & 0xFFFFFFFF]
        key = [seed & 0xFFFFFFFF, seed >> 32]
        x = int(oracle_mod.philox(ctr, key)[e & 3])
        expect = ((x >> 9) * 2 + 1) / 2.0 ** 24
        assert oracle_mod.uniform(seed, rnd, purpose, req, pos, e) == expect


def test_uniform_range_and_histogram(oracle_mod):
    n = 200_000
    u = np.array([oracle_mod.uniform(7, 1, 0, 3, 2, e) for e in range(n)])
    assert u.min() >= 2.0 ** -24 and u.max() <= 1 - 2.0 ** -24
    # the values are odd multiples of 2^-24, so they are exact in binary32
    assert np.all(u.astype(np.float32).astype(np.float64) == u)
    counts, _ = np.histogram(u, bins=64, range=(0.0, 1.0))
    assert stats.chisquare(counts).pvalue > 1e-3
    # Gumbel(0,1) transform: mean = Euler-Mascheroni constant, var = pi^2/6
    g = -np.log(-np.log(u))
    assert abs(g.mean() - np.euler_gamma) < 5 * np.sqrt(np.pi ** 2 / 6 / n)
    assert abs(g.var() - np.pi ** 2 / 6) < 0.05


def test_purposes_and_positions_are_distinct_streams(oracle_mod):
    a = [oracle_mod.uniform(1, 0, 0, 0, 0, e) for e in range(64)]
    b = [oracle_mod.uniform(1, 0, 3, 0, 0, e) for e in range(64)]
    c = [oracle_mod.uniform(1, 0, 0, 0, 1, e) for e in range(64)]
    d = [oracle_mod.uniform(1, 1, 0, 0, 0, e) for e in range(64)]
    for x in (b, c, d):
        assert len(set(a) & set(x)) == 0
