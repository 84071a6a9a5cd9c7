"""Oracle pins: Markov-head serial sampling, confidence head and survival products.

Each check is fixed by something other than the oracle's own code: the
softmax distribution (chi-square against scipy), library log-sum-exp, special
cases that reduce to the flat Gumbel-max or to a constant sigmoid, and a
one-hot embedding that exposes which token the confidence head reads."""
import numpy as np
import pytest
from scipy import special, stats

PUR_DRAFT_ELEM = 0


def _inputs(R, G, V, r, d, rng, u_std=2.0, ew_std=0.3):
    U = rng.normal(0, u_std, (R, G, V)).astype(np.float32)
    E = rng.normal(0, ew_std, (V, r)).astype(np.float32)
    W = rng.normal(0, ew_std, (r, V)).astype(np.float32)
    h = rng.normal(0, 1, (R, G, d)).astype(np.float32)
    w_h = rng.normal(0, 0.3, d).astype(np.float32)
    w_e = rng.normal(0, 0.3, r).astype(np.float32)
    T = rng.uniform(0.5, 1.5, R).astype(np.float32)
    anchor = rng.integers(0, V, R).astype(np.int32)
    return U, E, W, h, w_h, w_e, T, anchor


def _logits(U, E, W, T, q, k, prev, use_bias=True):
    bias = E[prev].astype(np.float64) @ W.astype(np.float64) if use_bias else 0.0
    return (U[q, k].astype(np.float64) + bias) / float(T[q])


def test_flat_gumbel_max_when_vocab_fits_one_block(oracle_mod):
    rng = np.random.default_rng(0)
    R, G, V, r, d = 5, 4, 100, 6, 3
    U, E, W, h, w_h, w_e, T, anchor = _inputs(R, G, V, r, d, rng)
    seed, rnd = 99, 7
    out = oracle_mod.sample_block(U, E, W, h, w_h, w_e, 0.5, T, anchor, seed, rnd)
    for q in range(R):
        prev = anchor[q]
        for k in range(G):
            l = _logits(U, E, W, T, q, k, prev)
            g = np.array([-np.log(-np.log(oracle_mod.uniform(seed, rnd, PUR_DRAFT_ELEM, q, k, v)))
                          for v in range(V)])
            assert out["tokens"][q, k] == int(np.argmax(l + g))
            assert out["lse"][q, k] == pytest.approx(special.logsumexp(l), rel=1e-13)
            assert out["logit"][q, k] == pytest.approx(l[out["tokens"][q, k]], rel=1e-13)
            prev = out["tokens"][q, k]


def _chi2_ok(counts, p, min_expected=5.0):
    n = counts.sum()
    exp = p * n
    keep = exp >= min_expected
    obs = np.append(counts[keep], counts[~keep].sum())
    ex = np.append(exp[keep], exp[~keep].sum())
    if ex[-1] == 0:
        obs, ex = obs[:-1], ex[:-1]
    return stats.chisquare(obs, ex * obs.sum() / ex.sum()).pvalue


@pytest.mark.parametrize("V", [16, 1000])
def test_draws_follow_softmax_of_biased_logits(oracle_mod, V):
    """10^6 (V=16) / 2*10^5 (V=1000, eight blocks with a ragged tail) draws of position 0
    and of position 1 given the drawn position-0 token."""
    rng = np.random.default_rng(1)
    n = 1_000_000 if V == 16 else 200_000
    r, d, G = 4, 2, 2
    U1 = rng.normal(0, 1.0, (1, G, V)).astype(np.float32)
    E = rng.normal(0, 0.5, (V, r)).astype(np.float32)
    W = rng.normal(0, 0.5, (r, V)).astype(np.float32)
    U = np.ascontiguousarray(np.broadcast_to(U1, (n, G, V)))
    h = np.zeros((n, G, d), np.float32)
    T = np.full(n, 0.8, np.float32)
    anchor = np.full(n, 3, np.int32)
    out = oracle_mod.sample_block(U, E, W, h, np.zeros(d), np.zeros(r), 0.0, T, anchor, 1234, 0,
                                  threads=8)
    tok = out["tokens"]
    p0 = special.softmax(_logits(U1, E, W, T, 0, 0, 3))
    assert _chi2_ok(np.bincount(tok[:, 0], minlength=V), p0) > 1e-3
    t = int(np.bincount(tok[:, 0]).argmax())
    sel = tok[:, 0] == t
    p1 = special.softmax(_logits(U1, E, W, T, 0, 1, t))
    assert _chi2_ok(np.bincount(tok[sel, 1], minlength=V), p1) > 1e-3


def test_low_temperature_picks_argmax_of_biased_logits(oracle_mod):
    rng = np.random.default_rng(2)
    R, G, V, r, d = 4, 3, 300, 5, 2
    U, E, W, h, w_h, w_e, T, anchor = _inputs(R, G, V, r, d, rng, u_std=3.0)
    T = np.full(R, 1e-4, np.float32)
    out = oracle_mod.sample_block(U, E, W, h, w_h, w_e, 0.0, T, anchor, 5, 0)
    for q in range(R):
        prev = anchor[q]
        for k in range(G):
            l = _logits(U, E, W, T, q, k, prev)
            assert out["tokens"][q, k] == int(np.argmax(l))
            prev = out["tokens"][q, k]


def test_bias_first_off_leaves_first_position_unbiased(oracle_mod):
    rng = np.random.default_rng(3)
    R, G, V, r, d = 3, 2, 50, 4, 2
    U, E, W, h, w_h, w_e, T, anchor = _inputs(R, G, V, r, d, rng)
    T = np.full(R, 1e-4, np.float32)
    out = oracle_mod.sample_block(U, E, W, h, w_h, w_e, 0.0, T, anchor, 5, 0, bias_first=0)
    for q in range(R):
        assert out["tokens"][q, 0] == int(np.argmax(U[q, 0]))
        l1 = _logits(U, E, W, T, q, 1, out["tokens"][q, 0])
        assert out["tokens"][q, 1] == int(np.argmax(l1))


def test_confidence_head_special_cases(oracle_mod):
    """w = 0 gives sigmoid(b); one-hot h gives sigmoid(w_h[j] + b); an identity embedding
    exposes which token eq. (7) reads (x_{k-1}) versus the x_k variant."""
    rng = np.random.default_rng(4)
    R, G, V = 6, 5, 16
    r, d = V, 4
    U = rng.normal(0, 1, (R, G, V)).astype(np.float32)
    E = np.eye(V, dtype=np.float32)             # W_1[x] = e_x
    W = np.zeros((r, V), np.float32)            # no Markov bias
    T = np.ones(R, np.float32)
    anchor = rng.integers(0, V, R).astype(np.int32)
    # constant: c = sigmoid(b) = 0.8 for b = ln 4
    h = rng.normal(0, 1, (R, G, d)).astype(np.float32)
    out = oracle_mod.sample_block(U, E, W, h, np.zeros(d), np.zeros(r), np.log(4.0), T, anchor, 1, 0)
    assert np.allclose(out["conf"], 0.8, atol=1e-7)
    assert np.allclose(out["surv"], 0.8 ** np.arange(1, G + 1)[None, :], rtol=1e-6)
    # one-hot h_k picks w_h[j]
    h = np.zeros((R, G, d), np.float32)
    h[:, :, 2] = 1.0
    w_h = np.array([0.0, 0.0, 1.25, 0.0], np.float32)
    out = oracle_mod.sample_block(U, E, W, h, w_h, np.zeros(r), -0.5, T, anchor, 1, 0)
    assert np.allclose(out["conf"], special.expit(1.25 - 0.5), rtol=1e-7)
    # identity embedding: c_k = sigmoid(w_e[x] + b)
    w_e = np.linspace(-3, 3, V).astype(np.float32)
    for conf_token in (0, 1):
        out = oracle_mod.sample_block(U, E, W, np.zeros((R, G, d), np.float32), np.zeros(d), w_e, 0.25,
                                      T, anchor, 1, 0, conf_token=conf_token)
        tok = out["tokens"]
        prev = np.concatenate([anchor[:, None], tok[:, :-1]], axis=1)
        x = prev if conf_token == 0 else tok
        assert np.allclose(out["conf"], special.expit(w_e[x].astype(np.float64) + 0.25), rtol=1e-7)
        assert np.allclose(out["surv"], np.cumprod(out["conf"], axis=1), rtol=1e-12)


def test_per_request_gamma_and_forced_tokens(oracle_mod):
    rng = np.random.default_rng(6)
    R, G, V, r, d = 4, 5, 40, 3, 2
    U, E, W, h, w_h, w_e, T, anchor = _inputs(R, G, V, r, d, rng)
    gam = np.array([0, 2, 5, 3], np.int32)
    out = oracle_mod.sample_block(U, E, W, h, w_h, w_e, 0.1, T, anchor, 8, 3, gamma=gam)
    for q in range(R):
        assert np.all(out["tokens"][q, gam[q]:] == -1)
        assert np.all(out["surv"][q, gam[q]:] == 0) and np.all(out["surv"][q, :gam[q]] > 0)
    # conditioning on the oracle's own draws reproduces every output
    same = oracle_mod.sample_block(U, E, W, h, w_h, w_e, 0.1, T, anchor, 8, 3, gamma=gam,
                                   forced_tokens=np.where(out["tokens"] < 0, 0, out["tokens"]))
    for k in ("tokens", "conf", "surv", "lse", "logit"):
        assert np.array_equal(same[k], out[k])
    # conditioning on other tokens changes the bias of the next position only
    forced = rng.integers(0, V, (R, G)).astype(np.int32)
    f = oracle_mod.sample_block(U, E, W, h, w_h, w_e, 0.1, T, anchor, 8, 3, forced_tokens=forced)
    for q in range(R):
        prev = anchor[q]
        for k in range(G):
            l = _logits(U, E, W, T, q, k, prev)
            assert f["lse"][q, k] == pytest.approx(special.logsumexp(l), rel=1e-13)
            assert f["logit"][q, k] == pytest.approx(l[forced[q, k]], rel=1e-13)
            prev = forced[q, k]


def test_bf16_inputs_are_read_exactly(oracle_mod):
    rng = np.random.default_rng(7)
    R, G, V, r, d = 2, 2, 64, 4, 8
    U, E, W, h, w_h, w_e, T, anchor = _inputs(R, G, V, r, d, rng)

    def to_bf16_bits(x):
        b = x.astype(np.float32).view(np.uint32)
        return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)

    def from_bits(x):
        return (x.astype(np.uint32) << 16).view(np.float32)

    Ub, Eb, Wb, hb = (to_bf16_bits(x) for x in (U, E, W, h))
    a = oracle_mod.sample_block(Ub, Eb, Wb, hb, w_h, w_e, 0.3, T, anchor, 4, 1)
    b = oracle_mod.sample_block(from_bits(Ub), from_bits(Eb), from_bits(Wb), from_bits(hb), w_h, w_e, 0.3,
                                T, anchor, 4, 1)
    for k in ("tokens", "conf", "surv", "lse", "logit"):
        assert np.array_equal(a[k], b[k])
