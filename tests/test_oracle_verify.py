"""Oracle pins: rejection-sampling verification and the losslessness of a whole
round (sample -> schedule -> verify), including the Appendix A negative control.

The pins are distributional: the acceptance rate equals 1 - TV (eq. 8a-8c), and
the emitted tokens follow the target distribution (chi-square), which a wrong
accept rule, residual or bonus row would break."""
import numpy as np
import pytest
from scipy import special, stats

from conftest import load_golden


def _chi2(counts, p):
    n = counts.sum()
    exp = p * n
    keep = exp >= 5
    obs = np.append(counts[keep], counts[~keep].sum())
    ex = np.append(exp[keep], exp[~keep].sum())
    if ex[-1] == 0:
        obs, ex = obs[:-1], ex[:-1]
    return stats.chisquare(obs, ex * obs.sum() / ex.sum()).pvalue


def _draft_setup(n, G, V, logp_draft, seed=17):
    """Requests whose draft distribution is exactly softmax(logp_draft[k]) (no bias)."""
    U = np.ascontiguousarray(np.broadcast_to(np.asarray(logp_draft, np.float64)[None], (n, G, V)))
    E = np.zeros((V, 1))
    W = np.zeros((1, V))
    h = np.zeros((n, G, 1))
    T = np.ones(n, np.float32)
    anchor = np.zeros(n, np.int32)
    return U, E, W, h, T, anchor


def test_acceptance_rate_is_one_minus_tv(oracle_mod):
    ex = load_golden("worked_examples.json")["tv_identity"]
    n = 1_000_000
    U, E, W, h, T, anchor = _draft_setup(n, 1, 2, np.log([ex["p_d"]]))
    s = oracle_mod.sample_block(U, E, W, h, [0.0], [0.0], 0.0, T, anchor, 3, 0, threads=8)
    target = np.ascontiguousarray(np.broadcast_to(np.log([ex["p_t"], [0.5, 0.5]])[None], (n, 2, 2)))
    keep = np.ones(n, np.int32)
    v = oracle_mod.verify(target, U, E, W, anchor, s["tokens"], s["lse"], s["logit"], keep, T, 3, 0,
                          threads=8)
    rate = v["accepted"].mean()
    assert abs(rate - ex["accept"]) < 5 * np.sqrt(0.16 / n)
    # y_1 follows p_t
    y1 = np.where(v["accepted"] >= 1, s["tokens"][:, 0], v["next_token"])
    assert abs((y1 == 0).mean() - ex["p_t"][0]) < 5 * np.sqrt(0.21 / n)


def test_verify_alone_is_lossless(oracle_mod):
    """V=16, two admitted positions, 10^6 requests: y_1 ~ p_t(row 0); given x_1 was
    accepted, y_2 ~ p_t(row 1); with nothing admitted the bonus is ~ p_t(row 0)."""
    rng = np.random.default_rng(8)
    n, G, V = 1_000_000, 2, 16
    ld = rng.normal(0, 1.5, (G, V))
    lt = rng.normal(0, 1.5, (G + 1, V))
    U, E, W, h, T, anchor = _draft_setup(n, G, V, ld)
    s = oracle_mod.sample_block(U, E, W, h, [0.0], [0.0], 0.0, T, anchor, 21, 4, threads=8)
    target = np.ascontiguousarray(np.broadcast_to(lt[None], (n, G + 1, V)))
    v = oracle_mod.verify(target, U, E, W, anchor, s["tokens"], s["lse"], s["logit"],
                          np.full(n, 2, np.int32), T, 21, 4, threads=8)
    acc, nxt, tok = v["accepted"], v["next_token"], s["tokens"]
    y1 = np.where(acc >= 1, tok[:, 0], nxt)
    pt = special.softmax(lt, axis=1)
    assert _chi2(np.bincount(y1, minlength=V), pt[0]) > 1e-3
    sel = acc >= 1
    y2 = np.where(acc[sel] >= 2, tok[sel, 1], nxt[sel])
    assert _chi2(np.bincount(y2, minlength=V), pt[1]) > 1e-3
    # acceptance of position 1 = 1 - TV(p_d, p_t)
    pd = special.softmax(ld, axis=1)
    c1 = 1 - 0.5 * np.abs(pd[0] - pt[0]).sum()
    assert abs(sel.mean() - c1) < 5 * np.sqrt(c1 * (1 - c1) / n)
    # residual flag marks exactly the rejected rounds
    assert np.array_equal(v["resampled"] == 1, acc < 2)
    # nothing admitted: bonus token from row 0
    b = oracle_mod.verify(target[:200_000], U[:200_000], E, W, anchor[:200_000], tok[:200_000],
                          s["lse"][:200_000], s["logit"][:200_000], np.zeros(200_000, np.int32),
                          T[:200_000], 22, 0, threads=8)
    assert np.all(b["accepted"] == 0) and np.all(b["resampled"] == 0)
    assert _chi2(np.bincount(b["next_token"], minlength=V), pt[0]) > 1e-3


def _appendix_a_round(oracle_mod, mode, sps, n=1_000_000, seed=31):
    """Appendix A setup: tokens A=0, B=1 and an anchor C=2 that is never drawn.
    p_d = (0.5, 0.5), p_t(row 0) = (0.7, 0.3). An identity embedding feeds eq. (7):
    c_1 = sigmoid(b) = 0.8 (anchor), c_2 = 0.9 after A and ~0 after B."""
    V, G, r = 3, 2, 3
    ld = np.log(np.array([[0.5, 0.5, 1e-300]] * G))
    U, _, _, h, T, _ = _draft_setup(n, G, V, ld)
    E = np.eye(V)
    W = np.zeros((r, V))
    b = np.log(4.0)
    w_e = np.array([special.logit(0.9) - b, -80.0, 0.0], np.float32)
    anchor = np.full(n, 2, np.int32)
    s = oracle_mod.sample_block(U, E, W, h, [0.0], w_e, b, T, anchor, seed, 0, threads=8)
    assert np.allclose(s["conf"][:, 0], 0.8, atol=1e-6)
    sc = oracle_mod.schedule(s["surv"].reshape(n, 1, G), sps, mode)
    keep = sc["keep"].reshape(n)
    lt = np.log(np.array([[0.7, 0.3, 1e-300], [0.5, 0.5, 1e-300], [0.5, 0.5, 1e-300]]))
    target = np.ascontiguousarray(np.broadcast_to(lt[None], (n, G + 1, V)))
    v = oracle_mod.verify(target, U, E, W, anchor, s["tokens"], s["lse"], s["logit"], keep, T, seed, 0,
                          threads=8)
    y1 = np.where(v["accepted"] >= 1, s["tokens"][:, 0], v["next_token"])
    return y1, keep


def test_full_round_sync_scheduler_is_lossless(oracle_mod):
    ex = load_golden("worked_examples.json")["appendix_a"]
    n = 1_000_000
    # Appendix A curve: the causal scheduler never admits x_1
    y1, keep = _appendix_a_round(oracle_mod, oracle_mod.SCHED_SYNC, ex["sps"], n)
    assert np.all(keep == 0)
    assert abs((y1 == 0).mean() - ex["P_Y_A_target"]) < 5 * np.sqrt(0.21 / n)
    # a curve on which admission of x_2 depends on x_1 (through c_2) -- still lossless
    y1, keep = _appendix_a_round(oracle_mod, oracle_mod.SCHED_SYNC, [1.0, 0.6, 0.5], n, seed=32)
    assert set(np.unique(keep)) == {1, 2}
    assert abs((y1 == 0).mean() - ex["P_Y_A_target"]) < 5 * np.sqrt(0.21 / n)


def test_appendix_a_lookahead_is_not_lossless(oracle_mod):
    """Negative control: the unconstrained full scan looks at c_2, which depends on x_1,
    before admitting x_1; the first emitted token is then A with probability 0.85."""
    ex = load_golden("worked_examples.json")["appendix_a"]
    n = 1_000_000
    y1, keep = _appendix_a_round(oracle_mod, oracle_mod.SCHED_FULL_SCAN, ex["sps"], n)
    assert set(np.unique(keep)) == {0, 2}
    p = (y1 == 0).mean()
    assert abs(p - ex["P_Y_A_lookahead"]) < 5 * np.sqrt(0.13 / n)
    assert abs(p - ex["P_Y_A_target"]) > 0.1


def test_residual_reads_the_bias_of_the_rejected_position(oracle_mod):
    """With a Markov bias, the residual at a rejected position k must use W_1[x_{k-1}] W_2.
    Check the residual token law against norm(max(0, p_t - p_d)) built from numpy."""
    rng = np.random.default_rng(12)
    n, G, V, r = 400_000, 2, 12, 3
    U1 = rng.normal(0, 1.0, (G, V))
    E = rng.normal(0, 0.8, (V, r))
    W = rng.normal(0, 0.8, (r, V))
    U = np.ascontiguousarray(np.broadcast_to(U1[None], (n, G, V)))
    h = np.zeros((n, G, 1))
    T = np.full(n, 0.9, np.float32)
    anchor = np.full(n, 5, np.int32)
    s = oracle_mod.sample_block(U, E, W, h, [0.0], np.zeros(r), 0.0, T, anchor, 41, 2, threads=8)
    lt = rng.normal(0, 1.0, (G + 1, V))
    target = np.ascontiguousarray(np.broadcast_to(lt[None], (n, G + 1, V)))
    v = oracle_mod.verify(target, U, E, W, anchor, s["tokens"], s["lse"], s["logit"],
                          np.full(n, 2, np.int32), T, 41, 2, threads=8)
    # rounds that accepted x_1 = t and rejected x_2: residual at position 1 given prev = t
    t = int(np.bincount(s["tokens"][:, 0]).argmax())
    sel = (v["accepted"] == 1) & (s["tokens"][:, 0] == t)
    pd = special.softmax((U1[1] + E[t] @ W) / 0.9)
    pt = special.softmax(lt[1] / 0.9)
    res = np.maximum(pt - pd, 0)
    res /= res.sum()
    assert sel.sum() > 5000
    assert _chi2(np.bincount(v["next_token"][sel], minlength=V), res) > 1e-3


def test_residual_margins_under_relative_errors(oracle_mod):
    """The residual draw's robust margins (rgap): equal to the exact top-two gaps when no error
    is assumed; never larger when one is; and their sign agrees with a brute-force search over
    perturbed probabilities (each p_t(v), p_d(v) moved by at most the relative error e, in the
    direction that helps the runner-up) on a three-token residual max(0, p_t - p_d)."""
    V = 3
    pd = np.array([0.2, 0.3, 0.5])
    pt = np.array([0.5, 0.35, 0.15])
    n = 64
    U = np.ascontiguousarray(np.broadcast_to(np.log(pd)[None, None], (n, 1, V)))
    E, W = np.zeros((V, 1)), np.zeros((1, V))
    T = np.ones(n, np.float32)
    anchor = np.zeros(n, np.int32)
    tokens = np.full((n, 1), 2, np.int32)            # p_t(2) / p_d(2) = 0.3: mostly rejected
    lse = np.zeros((n, 1))
    logit = np.full((n, 1), np.log(0.5))
    target = np.ascontiguousarray(np.broadcast_to(np.log(np.stack([pt, pt]))[None], (n, 2, V)))
    keep = np.ones(n, np.int32)
    base = oracle_mod.verify(target, U, E, W, anchor, tokens, lse, logit, keep, T, 5, 1)
    rej = base["resampled"] == 1
    assert rej.sum() > 20
    np.testing.assert_array_equal(base["rgap2"], base["gap2"])
    res = pt - pd
    for e in (1e-3, 0.05, 0.1, 0.2):
        o = oracle_mod.verify(target, U, E, W, anchor, tokens, lse, logit, keep, T, 5, 1, res_rel_eps=e)
        assert np.all(o["rgap2"][rej] <= base["gap2"][rej])
        for q in np.where(rej)[0]:
            g = np.array([-np.log(-np.log(oracle_mod.uniform(5, 1, 2, q, 0, v))) for v in range(V)])
            w = int(o["next_token"][q])
            # brute force: the winner's p_t down and p_d up, one rival's p_t up and p_d down, by e
            lo = pt[w] * (1 - e) - pd[w] * (1 + e)
            beaten = False
            for v in range(V):
                if v == w:
                    continue
                hi = pt[v] * (1 + e) - pd[v] * (1 - e)
                if hi > 0 and (lo <= 0 or np.log(hi) + g[v] >= np.log(lo) + g[w]):
                    beaten = True
            assert beaten == (o["rgap2"][q] <= 0), (e, q, o["rgap2"][q])
    assert res[2] < 0
