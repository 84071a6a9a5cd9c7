"""GPU parity at the full workload sizes, in the launch configuration the bench
times: the whole round runs on the GPU, then every request is checked
stage-wise against the oracle (sampler, scheduler on every survival, verifier),
on two consecutive rounds, and size-independent invariants are checked too.
The excusal counts of each workload are printed (pytest -s) and must stay rare."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_draft_round_gb300 as ds
from speculative_decoding_draft_round_gb300 import workloads as wl
from parity import _threads, add_counts, check_sample, check_schedule, check_verify, new_counts, report, rows, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    ds.lib()
    oracle.build()


def _capacity_survivals(rnd, rnd_idx):
    old = ds.sample_block(rnd.U, rnd.E, rnd.W, rnd.h, rnd.w_h, rnd.w_e, rnd.b, rnd.temperature, rnd.anchor,
                          rnd.seed, rnd_idx, gamma=rnd.gamma)
    return old["surv"].clone()


def _check_acceptance_is_one_minus_tv(rnd, tv, o_tok):
    """[P3] eq. 8a-8c: a draft token drawn from p_d is accepted with probability
    sum_v min(p_t, p_d) = 1 - TV(p_t, p_d). The round's draft is verified with every drafted
    position admitted; over every position the verifier tests (up to and including the first
    rejection) on requests whose draft equals the oracle's, the number accepted must match the
    sum of 1 - TV within 5 standard deviations."""
    keep = rnd.gamma.clone() if rnd.gamma is not None else torch.full((rnd.R,), rnd.gamma_max, dtype=torch.int32,
                                                                       device=DEV)
    v = ds.verify(rnd.target, rnd.U, rnd.E, rnd.W, rnd.anchor, _last["tokens"].clamp(min=0), _last["draft_lse"],
                  _last["draft_logit"], keep, rnd.temperature, rnd.seed, rnd.round, gamma=rnd.gamma)
    assert ds.check(v["workspace"]) == 0
    tok, kp, acc = to_np(_last["tokens"]), to_np(keep), to_np(v["accepted"])
    acc_sum, exp_sum, var, n_tested = 0.0, 0.0, 0.0, 0
    for q in range(rnd.R):
        kq, aq = int(kp[q]), int(acc[q])
        if kq == 0 or not np.array_equal(tok[q, :kq], o_tok[q, :kq]):
            continue
        for j in range(min(aq + 1, kq)):
            acc_sum += 1.0 if j < aq else 0.0
            exp_sum += 1.0 - tv[q, j]
            var += tv[q, j] * (1.0 - tv[q, j])
            n_tested += 1
    z = (acc_sum - exp_sum) / max(np.sqrt(var), 1e-9)
    print("acceptance vs 1 - TV: %d tested positions, %.0f accepted, %.1f expected, z = %.2f" % (
        n_tested, acc_sum, exp_sum, z))
    assert n_tested >= 500
    assert abs(z) < 5


_last = {}


def _check_round(rnd, workload, t):
    cap = _capacity_survivals(rnd, t - 2) if rnd.mode == wl.SCHED_ASYNC_CAPACITY else None
    runner = ds.RoundRunner(rnd, surv_capacity=cap)
    rnd.round = t
    runner.set_round(t)
    runner.run()
    assert runner.check() == 0
    res = runner.results()
    _last.clear()
    _last.update(res)
    R, G = rnd.R, rnd.gamma_max
    counts = new_counts()
    # every request, in chunks that keep the oracle's copies of U and the target small
    step = 64
    for s0 in range(0, R, step):
        ids = np.arange(s0, min(R, s0 + step))
        add_counts(counts, check_sample(rnd, res, ids))
        v = check_verify(rnd, res, res["keep"], res, ids)
        counts["accept"] += v["accept"]
        counts["residual_fp32"] += v["residual_fp32"]
        counts["draw"] += v["draw"]
    counts["theta"] += check_schedule(res["surv"], rnd.sps, rnd.mode, res, gamma=rnd.gamma,
                                      surv_capacity=cap)["theta"]
    report("workload %d round %d" % (workload, t), counts)

    # invariants on every request
    tok = to_np(res["tokens"])
    g = np.full(R, G) if rnd.gamma is None else to_np(rnd.gamma)
    active = np.arange(G)[None, :] < g[:, None]
    assert np.all((tok[active] >= 0) & (tok[active] < rnd.V)) and np.all(tok[~active] == -1)
    surv = to_np(res["surv"])
    conf = to_np(res["conf"])
    assert np.all((conf[active] > 0) & (conf[active] < 1))
    assert np.all(np.diff(np.where(active, surv, 0), axis=1) <= 1e-7)
    keep = to_np(res["keep"])
    acc = to_np(res["accepted"])
    nxt = to_np(res["next_token"])
    assert np.all((keep >= 0) & (keep <= g))
    assert np.all((acc >= 0) & (acc <= keep))
    assert np.all((nxt >= 0) & (nxt < rnd.V))
    st = ds.decode_stats(res["stats"])
    assert st["admitted"] == keep.sum()
    lse = to_np(res["draft_lse"])
    logit = to_np(res["draft_logit"])
    assert np.all(logit[active] <= lse[active] + 1e-4)
    return counts


def _fill_tv_target(rnd, t):
    """Target rows of the controlled-distance workload from the oracle's own draft at round t
    (its draft distribution of every drafted position); returns TV(p_t, p_d) [R][G] recomputed
    after the rows were rounded to bf16, and the oracle's tokens."""
    G, R = rnd.gamma_max, rnd.R
    tv = np.zeros((R, G))
    tokens = np.zeros((R, G), np.int32)
    g = to_np(rnd.gamma)
    for s0 in range(0, R, 32):
        ids = np.arange(s0, min(R, s0 + 32))
        o = oracle.sample_block(rows(rnd.U, ids), to_np(rnd.E), to_np(rnd.W), rows(rnd.h, ids), to_np(rnd.w_h),
                                to_np(rnd.w_e), rnd.b, to_np(rnd.temperature)[ids], to_np(rnd.anchor)[ids], rnd.seed,
                                t, gamma=g[ids], req_ids=ids, logp=True, threads=_threads())
        tokens[ids] = o["tokens"]
        lp = torch.from_numpy(o["logp"]).to(DEV)
        idx = torch.as_tensor(ids, device=DEV)
        new = wl.tv_target_rows(lp, rnd.temperature[idx], rnd.extra["tv_delta"][idx])
        for j, q in enumerate(ids):
            n = int(g[q])
            rnd.target[q, :n] = new[j, :n].to(rnd.target.dtype)
        # the distance the verifier sees: p_t from the rounded rows at temperature T
        zt = rnd.target[idx, :G].double() / rnd.temperature[idx].double().view(-1, 1, 1)
        p_t = torch.softmax(zt, dim=2)
        tv[ids] = (0.5 * (p_t - torch.exp(lp.double())).abs().sum(dim=2)).cpu().numpy()
    return tv, tokens


@pytest.mark.parametrize("workload", [2, 3, 4, 5])
def test_full_size_round(workload):
    torch.cuda.empty_cache()
    rnd = wl.WORKLOADS[workload](device=DEV)
    total = new_counts()
    if workload == 5:
        # the target is scored on the drafted prefix: build it from round 2's draft
        tv, o_tok = _fill_tv_target(rnd, 2)
    for t in (2, 3):
        add_counts(total, _check_round(rnd, workload, t))
        if workload == 5 and t == 2:
            _check_acceptance_is_one_minus_tv(rnd, tv, o_tok)
    report("workload %d, two rounds" % workload, total)
    # every request of both rounds was compared; excusals stay rare
    assert total["checked_requests"] == 2 * rnd.R
    assert total["draw"] + total["residual_fp32"] <= max(2, total["checked_tokens"] // 1000)
    assert total["accept"] <= max(2, total["checked_requests"] // 100)
    assert total["theta"] <= 1


@pytest.mark.parametrize("workload", [2, 3])
def test_full_size_round_resident_loop(workload):
    """The resident loop (one persistent launch for every draft step, W held on chip between
    steps) at the full sizes it takes, every request compared with the oracle."""
    torch.cuda.empty_cache()
    rnd = wl.WORKLOADS[workload](device=DEV)
    rnd.round = 4
    out = ds.sample_block(rnd.U, rnd.E, rnd.W, rnd.h, rnd.w_h, rnd.w_e, rnd.b, rnd.temperature, rnd.anchor,
                          rnd.seed, rnd.round, gamma=rnd.gamma, path=ds.PATH_RESIDENT)
    assert ds.check(out["workspace"]) == 0
    total = new_counts()
    for s0 in range(0, rnd.R, 64):
        add_counts(total, check_sample(rnd, out, np.arange(s0, min(rnd.R, s0 + 64))))
    report("resident loop, workload %d" % workload, total)
    assert total["checked_requests"] == rnd.R
    assert total["draw"] <= max(2, total["checked_tokens"] // 1000)


def test_round_replays_from_a_cuda_graph():
    """A whole round (sampler, scheduler, verifier) captured into a CUDA graph on a side stream and
    replayed gives the eager round's outputs bit for bit: the calls allocate nothing and never wait
    on the host, and their programmatic-launch edges survive capture."""
    torch.cuda.empty_cache()
    rnd = wl.WORKLOADS[2](device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        runner = ds.RoundRunner(rnd)
        runner.set_round(9)
        runner.run(stream=s)
        s.synchronize()
        assert runner.check(s) == 0
        eager = {k: v.clone() for k, v in runner.results().items()
                 if torch.is_tensor(v) and k != "workspace" and v.device.type == "cuda"}
        for k, v in runner.results().items():   # poison every output before the replay
            if k in eager:
                v.fill_(float("nan") if v.is_floating_point() else -7)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            runner.run(stream=s)
        g.replay()
        s.synchronize()
        assert runner.check(s) == 0
        out = runner.results()
    for k, v in eager.items():
        assert torch.equal(out[k], v), "%s differs after graph replay" % k
