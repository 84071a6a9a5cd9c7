"""Pins of the oracle's widening functions: the flattened verify batch, the static
confidence-threshold admission and sequential temperature scaling of the confidences.

Each is pinned to something other than the oracle: a hand-worked flattening, the single-request
worked example's printed survivals and Theta, closed forms of the threshold rule on monotone
survivals, and the invariants temperature scaling must keep."""
import numpy as np
import pytest

import oracle

from conftest import load_golden


# ------------------------------------------------------------------ ragged verify batch

def test_assemble_hand_example():
    # zhongzhuzhou.org notes, physical execution without padding: every request contributes its
    # anchor and its admitted draft tokens to one stream, with request id and causal position
    keep = [2, 0, 3]
    anchor = [10, 20, 30]
    tokens = [[1, 2, 3], [4, 5, 6], [7, 8, 9]]
    o = oracle.assemble(keep, anchor, tokens)
    assert o["flat_tokens"].tolist() == [10, 1, 2, 20, 30, 7, 8, 9, -1, -1, -1, -1]
    assert o["flat_request"].tolist() == [0, 0, 0, 1, 2, 2, 2, 2, -1, -1, -1, -1]
    assert o["flat_position"].tolist() == [0, 1, 2, 0, 0, 1, 2, 3, -1, -1, -1, -1]
    assert o["offsets"].tolist() == [0, 3, 4, 8]


def test_assemble_invariants_and_bounds():
    rng = np.random.default_rng(5)
    R, G = 37, 6
    keep = rng.integers(0, G + 1, R)
    anchor = rng.integers(0, 1000, R)
    tokens = rng.integers(0, 1000, (R, G))
    o = oracle.assemble(keep, anchor, tokens)
    off = o["offsets"]
    assert off[0] == 0 and np.all(np.diff(off) == keep + 1) and off[-1] == (keep + 1).sum()
    for q in range(R):
        run = slice(off[q], off[q + 1])
        assert o["flat_tokens"][run].tolist() == [anchor[q]] + tokens[q, :keep[q]].tolist()
        assert np.all(o["flat_request"][run] == q)
        assert o["flat_position"][run].tolist() == list(range(keep[q] + 1))
    assert np.all(o["flat_tokens"][off[-1]:] == -1)
    # the degenerate batch: nothing admitted anywhere leaves the anchors alone
    o0 = oracle.assemble(np.zeros(R, np.int32), anchor, tokens)
    assert o0["flat_tokens"][:R].tolist() == anchor.tolist() and o0["offsets"][-1] == R
    with pytest.raises(ValueError):
        oracle.assemble([G + 1] + [0] * (R - 1), anchor, tokens)


# ------------------------------------------------------------------ static threshold admission

def test_threshold_on_the_worked_example():
    ex = load_golden("worked_examples.json")["single_request"]
    c = np.array(ex["c"])
    surv = np.cumprod(c)[None, :]
    np.testing.assert_allclose(surv[0], ex["s_printed"], atol=5.0001e-4)
    sps = np.array(ex["sps"] + [ex["sps"][-1] * 0.9 ** i for i in range(1, 16)], dtype=np.float64)
    # admitted = the positions whose survival reaches the threshold
    for thr, keep in ((0.96, 0), (0.9, 1), (0.8, 2), (0.5, 3), (0.2, 4)):
        o = oracle.schedule(surv, sps, oracle.SCHED_THRESHOLD, threshold=thr)
        assert o["keep"].tolist() == [keep] and o["admitted"] == keep
        assert o["capacity"] == -1 and o["pool"] == 4
    # keep 3 reproduces the page's Theta at B = 4 (E = 3.567, Theta = 1212.7)
    o = oracle.schedule(surv, sps, oracle.SCHED_THRESHOLD, threshold=0.5)
    assert abs(o["theta_best"] - ex["theta_printed"][3]) <= 0.051


def test_threshold_closed_form_on_monotone_survivals():
    rng = np.random.default_rng(11)
    P, R, G = 20, 9, 5
    c = rng.uniform(0.2, 1.0, (P, R, G))
    surv = np.cumprod(c, axis=2)
    gamma = rng.integers(0, G + 1, R)
    sps = 1.0 / (1e-3 + 2e-6 * np.arange(1, R * (G + 1) + 1))
    thr = 0.45
    o = oracle.schedule(surv, sps, oracle.SCHED_THRESHOLD, gamma=gamma, threshold=thr)
    in_gamma = np.arange(G)[None, None, :] < gamma[None, :, None]
    admit = (surv >= thr) & in_gamma
    np.testing.assert_array_equal(o["keep"], admit.sum(axis=2))   # prefix-closed: a count
    np.testing.assert_array_equal(o["admitted"], admit.sum(axis=(1, 2)))
    tau = R + (surv * admit).sum(axis=(1, 2))
    np.testing.assert_allclose(o["theta_best"], tau * sps[R + admit.sum(axis=(1, 2)) - 1], rtol=1e-12)
    # threshold 0 admits the whole pool, i.e. every in-range position
    o0 = oracle.schedule(surv, sps, oracle.SCHED_THRESHOLD, gamma=gamma, threshold=0.0)
    np.testing.assert_array_equal(o0["keep"], np.broadcast_to(gamma, (P, R)))


def test_threshold_literal_rule_on_non_monotone_survivals():
    # l_r is the largest admitted position (Algorithm 1 sets l_r = j), also when a dips
    surv = np.array([[0.9, 0.3, 0.6, 0.1]])
    sps = np.linspace(10, 1, 10)
    o = oracle.schedule(surv, sps, oracle.SCHED_THRESHOLD, threshold=0.5)
    assert o["keep"].tolist() == [3] and o["admitted"] == 2


# ------------------------------------------------------------------ sequential temperature scaling

def _round(seed=3, R=5, G=4, V=40, r=8, d=12):
    rng = np.random.default_rng(seed)
    return dict(U=rng.normal(0, 2, (R, G, V)), E=rng.normal(0, 0.2, (V, r)), W=rng.normal(0, 0.2, (r, V)),
                h=rng.normal(0, 1, (R, G, d)), w_h=rng.normal(0, 0.3, d), w_e=rng.normal(0, 0.3, r), b=0.4,
                temperature=np.ones(R, np.float32), anchor=rng.integers(0, V, R), seed=7, rnd=2)


def test_sts_unit_temperatures_change_nothing():
    a = _round()
    base = oracle.sample_block(**a)
    ones = oracle.sample_block(**a, sts_temp=np.ones(4))
    for k in ("tokens", "conf", "surv", "lse", "logit"):
        np.testing.assert_array_equal(base[k], ones[k])


def test_sts_scales_the_logit_and_keeps_the_order():
    a = _round()
    base = oracle.sample_block(**a)
    t = np.array([0.5, 1.0, 2.0, 4.0])
    sts = oracle.sample_block(**a, sts_temp=t, forced_tokens=base["tokens"])
    logit = lambda c: np.log(c) - np.log1p(-c)
    # temperature scaling divides the head's logit by t_k ...
    np.testing.assert_allclose(logit(sts["conf"]) * t[None, :], logit(base["conf"]), rtol=1e-9, atol=1e-9)
    # ... so it is monotone at each position: the ranking across requests is unchanged
    for k in range(4):
        assert np.argsort(sts["conf"][:, k], kind="stable").tolist() == \
            np.argsort(base["conf"][:, k], kind="stable").tolist()
    # and the survival is the running product of the scaled confidences; the draws do not move
    np.testing.assert_allclose(sts["surv"], np.cumprod(sts["conf"], axis=1), rtol=1e-12)
    np.testing.assert_array_equal(sts["tokens"], base["tokens"])


def test_controlled_tv_rows_have_the_asked_distance():
    """Input shaping of the controlled-distance workload: rows built from a draft distribution
    p_d sit at exactly the asked total-variation distance from it (before rounding), the mass
    moves to the least likely token, and T log p_t recovers p_t."""
    import torch
    from speculative_decoding_draft_round_gb300 import workloads as wl
    g = torch.Generator().manual_seed(3)
    n, G, V = 5, 4, 300
    logits = torch.randn((n, G, V), generator=g, dtype=torch.float64) * 2.0
    lp = torch.log_softmax(logits, dim=2)
    T = torch.tensor([0.3, 0.7, 1.0, 1.2, 0.5], dtype=torch.float64)
    delta = 0.05 + 0.55 * torch.rand((n, G), generator=g, dtype=torch.float64)
    rows = wl.tv_target_rows(lp, T, delta, floor=-1e9).double()
    p_t = torch.softmax(rows / T.view(-1, 1, 1), dim=2)
    p_d = torch.exp(lp)
    tv = 0.5 * (p_t - p_d).abs().sum(dim=2)
    assert torch.allclose(tv, delta, atol=1e-5)
    assert torch.equal((p_t - p_d).argmax(dim=2), p_d.argmin(dim=2))
