"""Pins of the oracle's RNN sequential head (zhongzhuzhou.org notes, eq. 6):
  z_k = [s_{k-1}; W_1[x_{k-1}]; h_k],  s_k = g s_{k-1} + (1 - g) tanh(W_c z_k),  g = sigmoid(W_g z_k),
  s_0 = 0,  B_k = W_2^T tanh(W_o z_k),  W_rnn = [W_g; W_c; W_o] packed as [3r][2r + d].
Each pin ties the head to something outside it: independent sampling when its weights vanish,
the Markov head of eq. (5) when W_o passes a tiny multiple of W_1[x_{k-1}] through, and a
hand-written recurrence read back through greedy decoding."""
import numpy as np

import oracle


def _inputs(seed, R=5, G=5, V=60, r=6, d=7):
    rng = np.random.default_rng(seed)
    return dict(U=rng.normal(0, 2, (R, G, V)), E=rng.normal(0, 0.4, (V, r)), W=rng.normal(0, 0.4, (r, V)),
                h=rng.normal(0, 1, (R, G, d)), w_h=rng.normal(0, 0.3, d), w_e=rng.normal(0, 0.3, r), b=0.2,
                temperature=np.full(R, 0.8, np.float32), anchor=rng.integers(0, V, R), seed=13, rnd=3)


def test_vanishing_weights_give_independent_sampling():
    a = _inputs(1)
    V, r = a["E"].shape
    d = a["h"].shape[2]
    rnn = oracle.sample_block(head=oracle.HEAD_RNN, W_rnn=np.zeros((3 * r, 2 * r + d)), **a)
    indep = dict(a, E=np.zeros_like(a["E"]))   # Markov head without bias: B = 0
    ref = oracle.sample_block(**indep)
    for k in ("tokens", "lse", "logit"):
        np.testing.assert_array_equal(rnn[k], ref[k])
    assert np.all(rnn["a_rows"] == 0.0)


def test_small_identity_output_reproduces_the_markov_head():
    a = _inputs(2)
    V, r = a["E"].shape
    d = a["h"].shape[2]
    eps = 1e-3
    W_rnn = np.zeros((3 * r, 2 * r + d))
    W_rnn[2 * r:, r:2 * r] = eps * np.eye(r)          # W_o reads W_1[x_{k-1}] only
    rnn = oracle.sample_block(head=oracle.HEAD_RNN, W_rnn=W_rnn, **dict(a, W=a["W"] / eps))
    markov = oracle.sample_block(**a)
    # tanh(eps e) / eps = e (1 - eps^2 e^2 / 3 + ...): the logits agree to ~1e-7 relative
    clear = (markov["gap1"] > 1e-5) & (markov["gap2"] > 1e-5)
    assert clear.mean() > 0.95
    np.testing.assert_array_equal(rnn["tokens"][clear], markov["tokens"][clear])
    forced = oracle.sample_block(head=oracle.HEAD_RNN, W_rnn=W_rnn, forced_tokens=markov["tokens"],
                                 **dict(a, W=a["W"] / eps))
    np.testing.assert_allclose(forced["lse"], markov["lse"], rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(forced["a_rows"] / eps, a["E"][np.concatenate(
        [a["anchor"][:, None], markov["tokens"][:, :-1]], axis=1)], rtol=1e-5)


def test_gated_recurrence_through_greedy_decoding():
    a = _inputs(3, G=6)
    R, G, V = a["U"].shape
    r = a["E"].shape[1]
    d = a["h"].shape[2]
    rng = np.random.default_rng(4)
    M = rng.normal(0, 0.8, (r, d))
    eps = 1e-3
    W_rnn = np.zeros((3 * r, 2 * r + d))              # W_g = 0: the gate is 1/2
    W_rnn[r:2 * r, 2 * r:] = M                        # candidate from h_k only
    W_rnn[2 * r:, :r] = eps * np.eye(r)               # output from the previous state only
    a = dict(a, temperature=np.zeros(R, np.float32), W=a["W"] / eps)
    o = oracle.sample_block(head=oracle.HEAD_RNN, W_rnn=W_rnn, **a)
    # the same recurrence by hand: x_k = argmax(U_k + W^T s_{k-1}), s_k = s_{k-1}/2 + tanh(M h_k)/2
    W = a["W"] * eps
    tok = np.zeros((R, G), np.int64)
    for q in range(R):
        s = np.zeros(r)
        for k in range(G):
            tok[q, k] = np.argmax(a["U"][q, k] + s @ W)
            s = 0.5 * s + 0.5 * np.tanh(M @ a["h"][q, k])
    clear = o["gap1"] > 1e-5
    assert clear.mean() > 0.95
    np.testing.assert_array_equal(o["tokens"][clear], tok[clear])


def test_verifier_recomputes_the_rnn_bias_from_the_rows():
    # the residual of a rejected position uses the sampler's bias operand rows: with rows
    # equal to W_1[x_{k-1}], the result is the Markov head's verification
    a = _inputs(5)
    R, G, V = a["U"].shape
    rng = np.random.default_rng(6)
    s = oracle.sample_block(**a)
    target = rng.normal(0, 2, (R, G + 1, V))
    keep = np.full(R, G)
    common = (target, a["U"], a["E"], a["W"], a["anchor"], s["tokens"], s["lse"], s["logit"], keep,
              a["temperature"], 21, 4)
    ref = oracle.verify(*common)
    got = oracle.verify(*common, a_rows=s["a_rows"])
    for k in ("accepted", "next_token", "resampled"):
        np.testing.assert_array_equal(got[k], ref[k])
