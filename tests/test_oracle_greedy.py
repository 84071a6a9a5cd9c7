"""Pins of the oracle's temperature-0 (greedy) decoding: the draft takes the arg-max of its
logits and verification is an exact match with the target's arg-max (zhongzhuzhou.org notes,
FAQ on greedy decoding). Pinned to numpy's argmax, to hand-built targets, and to the limit of
the stochastic sampler and verifier as the temperature goes to zero."""
import numpy as np

import oracle


def _inputs(seed, R=6, G=4, V=50, r=8, d=10, zero_bias=False):
    rng = np.random.default_rng(seed)
    E = np.zeros((V, r)) if zero_bias else rng.normal(0, 0.3, (V, r))
    W = np.zeros((r, V)) if zero_bias else rng.normal(0, 0.3, (r, V))
    return dict(U=rng.normal(0, 3, (R, G, V)), E=E, W=W, h=rng.normal(0, 1, (R, G, d)),
                w_h=rng.normal(0, 0.3, d), w_e=rng.normal(0, 0.3, r), b=0.3,
                anchor=rng.integers(0, V, R), seed=9, rnd=4)


def test_greedy_draft_without_bias_is_numpy_argmax():
    a = _inputs(1, zero_bias=True)
    R = a["U"].shape[0]
    o = oracle.sample_block(temperature=np.zeros(R, np.float32), **a)
    np.testing.assert_array_equal(o["tokens"], np.argmax(a["U"], axis=2))
    np.testing.assert_allclose(o["logit"], a["U"].max(axis=2), rtol=0, atol=1e-12)
    np.testing.assert_array_equal(o["lse"], o["logit"])   # point mass: log p_d(x_k) = 0


def test_greedy_draft_is_the_zero_temperature_limit_of_sampling():
    a = _inputs(2)
    R = a["U"].shape[0]
    greedy = oracle.sample_block(temperature=np.zeros(R, np.float32), **a)
    cold = oracle.sample_block(temperature=np.full(R, 1e-6, np.float32), **a)
    # where the greedy top-two gap is not tiny, the Gumbel draw at T -> 0 is the arg-max
    clear = greedy["gap1"] > 1e-3
    assert clear.mean() > 0.9
    np.testing.assert_array_equal(greedy["tokens"][clear], cold["tokens"][clear])


def _target(R, G, V, best, rng):
    """Target logits whose row (q, j) has its maximum at best[q][j] by a margin of 5."""
    t = rng.normal(0, 1, (R, G + 1, V))
    for q in range(R):
        for j in range(G + 1):
            t[q, j, best[q, j]] = t[q, j].max() + 5.0
    return t


def test_greedy_verify_hand_cases():
    rng = np.random.default_rng(3)
    R, G, V, r = 4, 3, 12, 4
    best = rng.integers(0, V, (R, G + 1))
    target = _target(R, G, V, best, rng)
    tokens = best[:, :G].copy()
    tokens[0, 2] = (best[0, 2] + 1) % V        # request 0: two matches, then a mismatch
    tokens[1, 0] = (best[1, 0] + 1) % V        # request 1: mismatch at once
    keep = np.array([3, 2, 3, 0])              # request 2: all three match; request 3: nothing admitted
    U = rng.normal(0, 1, (R, G, V))
    o = oracle.verify(target, U, rng.normal(0, 1, (V, r)), rng.normal(0, 1, (r, V)), rng.integers(0, V, R),
                      tokens, np.zeros((R, G)), np.zeros((R, G)), keep, np.zeros(R, np.float32), 5, 1)
    assert o["accepted"].tolist() == [2, 0, 3, 0]
    assert o["next_token"].tolist() == [best[0, 2], best[1, 0], best[2, 3], best[3, 0]]
    assert o["resampled"].tolist() == [1, 1, 0, 0]


def test_greedy_verify_is_the_zero_temperature_limit():
    # draft and target both at a tiny temperature: the stochastic test accepts exactly the
    # arg-max matches, and the residual / bonus draw lands on the target's arg-max
    rng = np.random.default_rng(4)
    a = _inputs(5, R=8, G=4, V=30)
    R, G, V = a["U"].shape
    t_cold = np.full(R, 1e-5, np.float32)
    s = oracle.sample_block(temperature=t_cold, **a)
    best = rng.integers(0, V, (R, G + 1))
    best[:, :G] = np.where(rng.random((R, G)) < 0.6, s["tokens"], best[:, :G])   # mostly matching
    target = _target(R, G, V, best, rng)
    keep = rng.integers(0, G + 1, R)
    common = (target, a["U"], a["E"], a["W"], a["anchor"], s["tokens"], s["lse"], s["logit"], keep)
    cold = oracle.verify(*common, t_cold, 11, 2)
    greedy = oracle.verify(*common, np.zeros(R, np.float32), 11, 2)
    np.testing.assert_array_equal(cold["accepted"], greedy["accepted"])
    np.testing.assert_array_equal(cold["next_token"], greedy["next_token"])
    np.testing.assert_array_equal(cold["resampled"], greedy["resampled"])
