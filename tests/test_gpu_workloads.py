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
from parity import add_counts, check_sample, check_schedule, check_verify, new_counts, report, to_np

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


def _check_round(rnd, workload, t):
    cap = _capacity_survivals(rnd, t - 2) if rnd.mode == wl.SCHED_ASYNC_CAPACITY else None
    runner = ds.RoundRunner(rnd, surv_capacity=cap)
    rnd.round = t
    runner.set_round(t)
    runner.run()
    assert runner.check() == 0
    res = runner.results()
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


@pytest.mark.parametrize("workload", [2, 3, 4, 5])
def test_full_size_round(workload):
    torch.cuda.empty_cache()
    rnd = wl.WORKLOADS[workload](device=DEV)
    total = new_counts()
    for t in (2, 3):
        add_counts(total, _check_round(rnd, workload, t))
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
