"""Oracle pins: the hardware-aware prefix scheduler (Algorithm 1) against the
pages' worked examples, exhaustive enumeration on tiny batches, and invariants."""
import itertools

import numpy as np
import pytest

from conftest import load_golden


def _sps_from(b0, vals, n):
    """SPS table indexed by B-1, given values starting at B = b0 (earlier entries unused)."""
    t = [1e9] * (b0 - 1) + list(vals)
    assert len(t) >= n
    return np.array(t, dtype=np.float64)


def test_single_request_worked_example(oracle_mod):
    ex = load_golden("worked_examples.json")["single_request"]
    c = np.array(ex["c"])
    s = np.cumprod(c)
    assert np.allclose(s, ex["s_printed"], atol=5.0001e-4)
    out = oracle_mod.schedule(s[None, :], ex["sps"], oracle_mod.SCHED_SYNC)
    assert int(out["keep"][0]) == ex["keep"] == int(out["admitted"])
    # Theta column of the table: theta_m = SPS(1+m) * E_m, E_m = 1 + s_1 + ... + s_m
    theta = out["theta_curve"][: len(ex["theta_printed"])]
    assert np.allclose(theta, ex["theta_printed"], atol=0.05 + 1e-9)
    E = theta / np.array(ex["sps"][: len(theta)])
    assert np.allclose(E, ex["E_printed"], atol=5.0001e-4)
    assert out["theta_best"] == pytest.approx(theta[3])
    # the full scan finds the same maximum on this unimodal curve
    full = oracle_mod.schedule(s[None, :], ex["sps"], oracle_mod.SCHED_FULL_SCAN)
    assert int(full["keep"][0]) == 3


def test_two_request_worked_example(oracle_mod):
    ex = load_golden("worked_examples.json")["two_requests"]
    a = np.cumprod(np.array(ex["c"]), axis=1)
    assert np.allclose(a, ex["a_printed"], atol=1e-12)
    sps = _sps_from(2, ex["sps_from_B2"], 6)
    for mode in (oracle_mod.SCHED_SYNC, oracle_mod.SCHED_FULL_SCAN):
        out = oracle_mod.schedule(a, sps, mode)
        assert out["keep"].tolist() == ex["keep"]
        assert out["theta_best"] == pytest.approx(ex["theta_best"], abs=1e-12)
    curve = oracle_mod.schedule(a, sps, oracle_mod.SCHED_FULL_SCAN)["theta_curve"]
    assert np.allclose(curve, ex["theta_curve_printed"], atol=1e-12)
    # the printed order follows from the curve: tau increments are the sorted a's
    tau = curve / sps[1:6]
    inc = np.diff(tau)
    order = [tuple(p) for p in ex["order_printed"]]
    assert np.allclose(inc, [a[r - 1, j - 1] for r, j in order])


def test_three_request_walkthrough(oracle_mod):
    ex = load_golden("worked_examples.json")["three_requests"]
    a = np.cumprod(np.array(ex["c"]), axis=1)
    assert np.allclose(a, ex["a_printed"], atol=5.0001e-4)
    sps = _sps_from(3, ex["sps_from_B3"], 12)
    out = oracle_mod.schedule(a, sps, oracle_mod.SCHED_SYNC)
    assert out["keep"].tolist() == ex["keep"]
    assert out["theta_best"] == pytest.approx(ex["theta_best"], abs=5.0001e-4)
    curve = oracle_mod.schedule(a, sps, oracle_mod.SCHED_FULL_SCAN)["theta_curve"]
    # the page sums survivals already rounded to 3 decimals (up to 4 of them here), so its
    # printed Theta carries up to 4 * 5e-4 of display rounding on top of its own last digit
    assert np.allclose(curve[:5], ex["theta_printed_first"], atol=2.5e-3)
    tau = curve / sps[2:12]
    order = [tuple(p) for p in ex["order_printed"]]
    assert np.allclose(np.diff(tau), [a[r - 1, j - 1] for r, j in order])


def test_appendix_a_thresholds(oracle_mod):
    ex = load_golden("worked_examples.json")["appendix_a"]
    sps = ex["sps"]
    # causal scheduler: Theta_1 = 0.9 <= Theta_0 = 1.0 -> l = 0 whatever a_2 is
    for a2 in (0.72, 1e-9):
        out = oracle_mod.schedule(np.array([[ex["a1"], a2]]), sps, oracle_mod.SCHED_SYNC)
        assert int(out["keep"][0]) == 0
    hi = oracle_mod.schedule(np.array([[0.8, 0.72]]), sps, oracle_mod.SCHED_FULL_SCAN)
    assert np.allclose(hi["theta_curve"], [ex["theta0"], ex["theta1"], ex["theta2_if_c2_0.9"]])
    assert int(hi["keep"][0]) == 2
    lo = oracle_mod.schedule(np.array([[0.8, 1e-300]]), sps, oracle_mod.SCHED_FULL_SCAN)
    assert lo["theta_curve"][2] == pytest.approx(ex["theta2_if_c2_0"])
    assert int(lo["keep"][0]) == 0


def _exhaustive(a, gam, sps):
    """max over every length vector l (0 <= l_r <= gamma_r) of (R + sum a) * SPS(R + sum l),
    and the best tau for each total batch size."""
    R = a.shape[0]
    best = -np.inf
    best_tau = {}
    for ell in itertools.product(*[range(g + 1) for g in gam]):
        tau = R + sum(a[r, :ell[r]].sum() for r in range(R))
        B = R + sum(ell)
        best_tau[B] = max(best_tau.get(B, -np.inf), tau)
        best = max(best, tau * sps[B - 1])
    return best, best_tau


def test_greedy_matches_exhaustive_enumeration(oracle_mod):
    rng = np.random.default_rng(11)
    for trial in range(300):
        R = int(rng.integers(1, 4))
        G = int(rng.integers(1, 4))
        gam = rng.integers(0, G + 1, size=R)
        c = rng.uniform(0.05, 1.0, size=(R, G))
        if trial % 5 == 0:
            c = np.round(c, 1)  # force ties between requests
        a = np.cumprod(c, axis=1)
        n = R * (1 + G)
        if trial % 2:
            sps = np.cumprod(rng.uniform(0.5, 1.0, size=n)) * 100  # monotone, jagged
        else:
            sps = 100.0 / (1.0 + rng.uniform(0.01, 0.5) * np.arange(1, n + 1))  # smooth
        best, best_tau = _exhaustive(a, gam, sps)
        full = oracle_mod.schedule(a, sps, oracle_mod.SCHED_FULL_SCAN, gamma=gam)
        assert full["theta_best"] == pytest.approx(best, rel=1e-12)
        # Lemmas 1-2: the sorted prefix of size m attains the best tau for batch R + m
        curve = full["theta_curve"]
        for m in range(int(full["pool"]) + 1):
            assert curve[m] / sps[R + m - 1] == pytest.approx(best_tau[R + m], rel=1e-12)
        # early stop equals the global optimum when Theta is unimodal along the sweep
        th = curve[: int(full["pool"]) + 1]
        d = np.diff(th)
        unimodal = not np.any((d[1:] > 0) & (d[:-1] <= 0))
        sync = oracle_mod.schedule(a, sps, oracle_mod.SCHED_SYNC, gamma=gam)
        if unimodal:
            assert sync["theta_best"] == pytest.approx(best, rel=1e-12)
        # invariants
        for out in (full, sync):
            keep = out["keep"]
            assert np.all(keep >= 0) and np.all(keep <= gam)
            assert keep.sum() == out["admitted"]
            assert out["theta_best"] >= R * sps[R - 1] * (1 - 1e-15)


def test_async_capacity_uses_old_survivals_for_K_and_current_for_ranking(oracle_mod):
    rng = np.random.default_rng(5)
    R, G = 6, 4
    sps = 100.0 / (1.0 + 0.08 * np.arange(1, R * (1 + G) + 1))
    cur = np.cumprod(rng.uniform(0.2, 1.0, (R, G)), axis=1)
    old = np.cumprod(rng.uniform(0.2, 1.0, (R, G)), axis=1)
    full_old = oracle_mod.schedule(old, sps, oracle_mod.SCHED_FULL_SCAN)
    out = oracle_mod.schedule(cur, sps, oracle_mod.SCHED_ASYNC_CAPACITY, surv_capacity=old)
    K = int(full_old["admitted"])
    assert int(out["capacity"]) == K
    assert int(out["admitted"]) == min(K, R * G)
    # the admitted set is the top-K of the current survivals
    flat = sorted(((-cur[r, j], r, j) for r in range(R) for j in range(G)))[:K]
    expect = np.zeros(R, int)
    for _, r, j in flat:
        expect[r] = max(expect[r], j + 1)
    assert out["keep"].tolist() == expect.tolist()
    # with identical old and current survivals it is the full scan
    same = oracle_mod.schedule(cur, sps, oracle_mod.SCHED_ASYNC_CAPACITY, surv_capacity=cur)
    full = oracle_mod.schedule(cur, sps, oracle_mod.SCHED_FULL_SCAN)
    assert same["keep"].tolist() == full["keep"].tolist()


def test_zero_survivals_never_admitted_and_ties_keep_prefixes(oracle_mod):
    R, G = 3, 4
    a = np.array([[1.0, 1.0, 1.0, 0.0], [1.0, 1.0, 0.5, 0.25], [0.0, 0.0, 0.0, 0.0]])
    sps = np.full(R * (1 + G), 10.0)  # flat: every positive key raises Theta
    out = oracle_mod.schedule(a, sps, oracle_mod.SCHED_SYNC)
    assert out["keep"].tolist() == [3, 4, 0]
    assert int(out["pool"]) == 7


def test_sync_stop_comes_by_the_first_forced_decrease(oracle_mod):
    # Admitting an m-th key adds a <= 1 to tau >= R, so once SPS(R + m - 1) * R >= SPS(R + m) * (R + 1)
    # Theta cannot rise at m whatever the keys are: the sync scan admits fewer than that m. The GPU
    # scheduler relies on this to take only the top keys; check the bound on random survivals and
    # tables with drops of every size, including drops just below and above the forcing ratio.
    rng = np.random.default_rng(5)
    n_checked = 0
    for trial in range(300):
        R = int(rng.integers(1, 40))
        G = int(rng.integers(1, 9))
        n = R * (1 + G)
        sps = np.full(n, 1000.0)
        B = np.arange(1, n + 1)
        for _ in range(int(rng.integers(1, 4))):
            b0 = int(rng.integers(R + 1, R + R * G + 2))
            ratio = 1.0 + float(rng.choice([0.2, 0.9, 1.0, 1.1, 5.0])) / R
            sps = np.where(B >= b0, sps / ratio, sps)
        c = rng.uniform(0.05, 1.0, size=(R, G))
        surv = np.cumprod(c, axis=1)
        surv[rng.random((R, G)) < 0.1] = 0.0
        out = oracle_mod.schedule(surv, sps, oracle_mod.SCHED_SYNC)
        forced = [m for m in range(1, R * G + 1) if sps[R + m - 2] * R >= sps[R + m - 1] * (R + 1)]
        if forced:
            assert int(out["admitted"]) < forced[0]
            n_checked += 1
    assert n_checked > 100
