"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the same
seeded inputs, at sizes that span several vocabulary blocks, several request
tiles and ragged tails, and the degenerate cases of the method."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_draft_round_gb300 as ds
from speculative_decoding_draft_round_gb300 import workloads as wl
from parity import add_counts, check_sample, check_schedule, check_verify, new_counts, report, to_np
from conftest import load_golden

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    ds.lib()
    oracle.build()


def _paths(rnd):
    """The contraction paths these inputs support: CUDA cores always; the per-step tensor-core
    kernels and the resident loop when the shape allows."""
    paths = [ds.PATH_CUDA_CORE]
    for path in (ds.PATH_TENSOR_CORE, ds.PATH_RESIDENT):
        a, _ = ds.sample_args(rnd.U, rnd.E, rnd.W, rnd.h, rnd.w_h, rnd.w_e, rnd.b, rnd.temperature, rnd.anchor,
                              rnd.seed, rnd.round, gamma=rnd.gamma, path=path)
        try:
            if ds.sample_path(a) == path:
                paths.append(path)
        except ds.DsparkError:
            pass
    return paths


SMALL = [
    dict(name="c1", R=4, G=4, V=64, r=8, d=32, dtype="f32", u_std=2.0, t_std=2.0, ew_std=0.1, wh_std=0.3),
    dict(name="ragged_f32", R=11, G=5, V=300, r=24, d=20, dtype="f32", ew_std=0.2,
         gamma=[5, 0, 3, 5, 1, 2, 5, 4, 5, 0, 5]),
    dict(name="tiles_bf16", R=160, G=3, V=1000, r=64, d=96, dtype="bf16", ew_std=0.15,
         temperature=lambda R, g, dev: 0.4 + torch.rand((R,), generator=g, device=dev)),
    dict(name="wide_bf16", R=37, G=4, V=2056, r=256, d=64, dtype="bf16", ew_std=0.05,
         gamma=[4, 2] * 18 + [3]),
    # the resident loop with W tiles in tensor memory, in shared memory and streamed (6 blocks per
    # CTA on 152 SMs), two request halves with a ragged second one
    dict(name="resident_bf16", R=100, G=3, V=100000, r=256, d=64, dtype="bf16", ew_std=0.05,
         temperature=lambda R, g, dev: 0.5 + torch.rand((R,), generator=g, device=dev)),
]


def _make(spec, seed=123, **over):
    spec = dict(spec)
    spec.update(over)
    name = spec.pop("name")
    R, G, V, r, d, dtype = (spec.pop(k) for k in ("R", "G", "V", "r", "d", "dtype"))
    sps = spec.pop("sps", None)
    if sps is None:
        sps = wl.sps_hyperbolic(R * (1 + G), a=1e-3, b=4e-5)
    return wl.make_round(name, R, G, V, r, d, dtype, seed=seed, device=DEV, sps=sps, **spec)


@pytest.mark.parametrize("spec", SMALL, ids=[s["name"] for s in SMALL])
@pytest.mark.parametrize("conf_token", [0, 1])
def test_sample_block_matches_oracle(spec, conf_token):
    rnd = _make(spec, conf_token=conf_token)
    ids = np.arange(rnd.R)
    for path in _paths(rnd):
        total = new_counts()
        for rnd_idx in (0, 7):
            out = ds.sample_block(rnd.U, rnd.E, rnd.W, rnd.h, rnd.w_h, rnd.w_e, rnd.b, rnd.temperature,
                                  rnd.anchor, rnd.seed, rnd_idx, gamma=rnd.gamma, conf_token=conf_token,
                                  path=path)
            assert ds.check(out["workspace"]) == 0
            rnd.round = rnd_idx
            add_counts(total, check_sample(rnd, out, ids))
        report("sample %s conf_token=%d path=%d" % (spec["name"], conf_token, path), total)
        assert total["draw"] <= max(2, total["checked_tokens"] // 1000)


def test_bias_first_off_and_tiny_vocab():
    rnd = _make(dict(name="v5", R=6, G=3, V=5, r=4, d=8, dtype="f32", ew_std=0.5), bias_first=0)
    out = ds.sample_block(rnd.U, rnd.E, rnd.W, rnd.h, rnd.w_h, rnd.w_e, rnd.b, rnd.temperature, rnd.anchor,
                          rnd.seed, 0, bias_first=0)
    check_sample(rnd, out, np.arange(rnd.R))


def _rand_surv(R, G, gen, zero_frac=0.1, ties=False):
    c = torch.rand((R, G), generator=gen) * 0.95 + 0.05
    if ties:
        c = torch.round(c * 10) / 10
    a = torch.cumprod(c, dim=1)
    a[torch.rand((R, G), generator=gen) < zero_frac] = 0.0
    return a.to(torch.float32)


@pytest.mark.parametrize("mode", [ds.SCHED_SYNC, ds.SCHED_FULL_SCAN, ds.SCHED_ASYNC_CAPACITY])
def test_schedule_matches_oracle(mode):
    gen = torch.Generator().manual_seed(77)
    cases = [(1, 1), (3, 2), (4, 4), (32, 16), (128, 16), (100, 7), (512, 16), (8192, 1), (256, 32)]
    n_exc = 0
    for R, G in cases:
        for sps_kind in ("hyper", "stair", "steep"):
            n = R * (1 + G)
            if sps_kind == "hyper":
                sps = wl.sps_hyperbolic(n, a=1e-3, b=2e-6 * 32 / R)
            elif sps_kind == "stair":
                sps = wl.sps_staircase(n)
            else:
                sps = wl.sps_hyperbolic(n, a=1e-3, b=1e-4)
            for ties in (False, True):
                surv = _rand_surv(R, G, gen, ties=ties).to(DEV)
                old = _rand_surv(R, G, gen).to(DEV) if mode == ds.SCHED_ASYNC_CAPACITY else None
                gamma = torch.randint(0, G + 1, (R,), generator=gen, dtype=torch.int32).to(DEV) if ties else None
                out = ds.schedule(surv, sps.to(DEV), mode, gamma=gamma, surv_capacity=old)
                assert ds.check(out["workspace"]) == 0
                n_exc += check_schedule(surv, sps, mode, out, gamma=gamma, surv_capacity=old)["theta"]
    assert n_exc <= 2


@pytest.mark.parametrize("mode", [ds.SCHED_SYNC, ds.SCHED_FULL_SCAN, ds.SCHED_ASYNC_CAPACITY])
def test_schedule_monotone_runs_match_oracle(mode):
    # survivals that never increase along a request (the sampler's running products, zeros only
    # as a tail) take the kernel's merge of per-request runs instead of the radix sort
    gen = torch.Generator().manual_seed(78)
    cases = [(1, 1), (3, 2), (5, 3), (32, 16), (128, 16), (100, 7), (512, 16), (8192, 1), (256, 32), (37, 5)]
    n_exc = 0
    for R, G in cases:
        sps = wl.sps_hyperbolic(R * (1 + G), a=1e-3, b=2e-6 * 32 / R)
        for ties in (False, True):
            surv = _rand_surv(R, G, gen, zero_frac=0.0, ties=ties)
            tail = torch.randint(0, G + 1, (R,), generator=gen)
            surv[torch.arange(G)[None, :] >= tail[:, None]] = 0.0   # underflowed tails
            surv = surv.to(DEV)
            old = _rand_surv(R, G, gen, zero_frac=0.0).to(DEV) if mode == ds.SCHED_ASYNC_CAPACITY else None
            gamma = torch.randint(0, G + 1, (R,), generator=gen, dtype=torch.int32).to(DEV) if ties else None
            out = ds.schedule(surv, sps.to(DEV), mode, gamma=gamma, surv_capacity=old)
            assert ds.check(out["workspace"]) == 0
            n_exc += check_schedule(surv, sps, mode, out, gamma=gamma, surv_capacity=old)["theta"]
    assert n_exc <= 2


def _sps_drops(n, drops, base=1000.0):
    """SPS(B) for B = 1..n: `base`, multiplied by f at every B >= B0 for each (B0, f) in drops."""
    B = torch.arange(1, n + 1, dtype=torch.float64)
    v = torch.full((n,), base, dtype=torch.float64)
    for b0, f in drops:
        v = torch.where(B >= b0, v * f, v)
    return v.to(torch.float32)


def test_schedule_sync_forced_stop_matches_oracle():
    # sync mode with a table whose drop at some B forces Theta down whatever the keys (a ratio of at
    # least 1 + 1/R): the kernel then takes only the top keys, merged from the sorted request runs.
    # Drops land before, inside and past the pool; a mild earlier drop may stop the scan first;
    # R past the fast path's limit and unsorted runs take the full sort.
    gen = torch.Generator().manual_seed(79)
    cases = [(1, 1), (3, 2), (5, 3), (37, 5), (64, 4), (100, 7), (128, 16), (512, 16), (600, 2)]
    n_exc = 0
    for R, G in cases:
        n = R * (1 + G)
        stop_at = sorted({1, 2, min(63, R * G), max(1, R * G // 2), min(256, R * G), min(300, R * G)})
        for m0 in stop_at:
            for mild in (False, True):
                drops = [(R + m0, 0.9 * R / (R + 1.0))]           # forced: ratio above 1 + 1/R
                if mild and m0 > 2:
                    drops.append((R + m0 // 2, 1.0 / (1.0 + 0.4 / R)))   # may or may not stop first
                sps = _sps_drops(n, drops)
                for variant in ("ties", "tails", "sparse", "unsorted"):
                    # confidences of at least 0.5 keep every a above 1e-5, so no admission changes
                    # Theta by less than the tie band
                    c = torch.rand((R, G), generator=gen) * 0.5 + 0.5
                    if variant == "ties":
                        c = torch.round(c * 10) / 10
                    surv = torch.cumprod(c, dim=1).to(torch.float32)
                    if variant == "tails":
                        tail = torch.randint(0, G + 1, (R,), generator=gen)
                        surv[torch.arange(G)[None, :] >= tail[:, None]] = 0.0
                    elif variant == "sparse":   # most requests empty: the pool can end before the drop
                        surv[torch.rand((R,), generator=gen) < 0.8] = 0.0
                    elif variant == "unsorted" and G > 1:
                        surv[:, [0, G - 1]] = surv[:, [G - 1, 0]]
                    surv = surv.to(DEV)
                    gamma = torch.randint(0, G + 1, (R,), generator=gen, dtype=torch.int32).to(DEV) \
                        if variant == "ties" else None
                    out = ds.schedule(surv, sps.to(DEV), ds.SCHED_SYNC, gamma=gamma)
                    assert ds.check(out["workspace"]) == 0
                    n_exc += check_schedule(surv, sps, ds.SCHED_SYNC, out, gamma=gamma)["theta"]
    assert n_exc <= 2


def test_schedule_worked_examples_on_gpu():
    ex = load_golden("worked_examples.json")
    s = ex["single_request"]
    surv = torch.tensor([np.cumprod(s["c"])], dtype=torch.float32, device=DEV)
    out = ds.schedule(surv, torch.tensor(s["sps"], dtype=torch.float32, device=DEV), ds.SCHED_SYNC)
    assert out["keep"].tolist() == [3]
    assert ds.decode_stats(out["stats"])["theta_best"] == pytest.approx(1212.746, abs=1e-3)
    t = ex["two_requests"]
    surv = torch.tensor(np.cumprod(t["c"], axis=1), dtype=torch.float32, device=DEV)
    sps = torch.tensor([9.0] + t["sps_from_B2"], dtype=torch.float32, device=DEV)
    for mode in (ds.SCHED_SYNC, ds.SCHED_FULL_SCAN):
        out = ds.schedule(surv, sps, mode)
        assert out["keep"].tolist() == t["keep"]
    h = ex["three_requests"]
    surv = torch.tensor(np.cumprod(h["c"], axis=1), dtype=torch.float32, device=DEV)
    sps = torch.tensor([9.0, 9.0] + h["sps_from_B3"], dtype=torch.float32, device=DEV)
    out = ds.schedule(surv, sps, ds.SCHED_SYNC)
    assert out["keep"].tolist() == h["keep"]
    a = ex["appendix_a"]
    sps = torch.tensor(a["sps"], dtype=torch.float32, device=DEV)
    assert ds.schedule(torch.tensor([[0.8, 0.72]], device=DEV), sps, ds.SCHED_SYNC)["keep"].tolist() == [0]
    assert ds.schedule(torch.tensor([[0.8, 0.72]], device=DEV), sps, ds.SCHED_FULL_SCAN)["keep"].tolist() == [2]


@pytest.mark.parametrize("spec", SMALL, ids=[s["name"] for s in SMALL])
def test_verify_matches_oracle(spec):
    rnd = _make(spec, seed=321)
    ids = np.arange(rnd.R)
    gen = torch.Generator().manual_seed(5)
    for path in _paths(rnd):
        total = new_counts()
        sout = ds.sample_block(rnd.U, rnd.E, rnd.W, rnd.h, rnd.w_h, rnd.w_e, rnd.b, rnd.temperature,
                               rnd.anchor, rnd.seed, rnd.round, gamma=rnd.gamma, path=path)
        g = torch.full((rnd.R,), rnd.gamma_max) if rnd.gamma is None else rnd.gamma.cpu()
        for trial in range(3):
            if trial == 0:
                keep = g.clone()                                  # verify everything drafted
            elif trial == 1:
                keep = torch.zeros_like(g)                        # bonus only
            else:
                keep = (torch.rand(rnd.R, generator=gen) * (g + 1)).floor().to(torch.int32)
            keep = keep.to(torch.int32).to(DEV)
            vpath = ds.PATH_TENSOR_CORE if path == ds.PATH_RESIDENT else path   # the verifier's residual path
            vout = ds.verify(rnd.target, rnd.U, rnd.E, rnd.W, rnd.anchor, sout["tokens"], sout["draft_lse"],
                             sout["draft_logit"], keep, rnd.temperature, rnd.seed, rnd.round, gamma=rnd.gamma,
                             path=vpath)
            assert ds.check(vout["workspace"]) == 0
            add_counts(total, check_verify(rnd, sout, keep, vout, ids))
        report("verify %s path=%d" % (spec["name"], path), total)
        assert total["draw"] + total["accept"] + total["residual_fp32"] <= max(2, 3 * rnd.R // 100)


def test_verify_rows_past_the_prewait_items():
    """verify_rows forms at most 16 row-0 items per CTA before its dependency wait (a CTA per SM
    slot, about 600 on this part); R = 2048 requests of V = 65536 hold 2048 x 8 row-0 items, so
    the rest, and every later row, come after the wait. Sampled requests (both ends of the range
    and random ones) are compared with the oracle; every request's outputs are checked for range."""
    rnd = wl.make_round("R2048_g2_V65536_bf16", 2048, 2, 65536, 64, 32, "bf16", seed=99, device=DEV,
                        sps=wl.sps_hyperbolic(2048 * 3))
    rnd.round = 5
    sout = ds.sample_block(rnd.U, rnd.E, rnd.W, rnd.h, rnd.w_h, rnd.w_e, rnd.b, rnd.temperature,
                           rnd.anchor, rnd.seed, rnd.round, gamma=rnd.gamma)
    assert ds.check(sout["workspace"]) == 0
    gen = torch.Generator().manual_seed(6)
    keep = (torch.rand(rnd.R, generator=gen) * 3).floor().to(torch.int32).to(DEV)
    vout = ds.verify(rnd.target, rnd.U, rnd.E, rnd.W, rnd.anchor, sout["tokens"], sout["draft_lse"],
                     sout["draft_logit"], keep, rnd.temperature, rnd.seed, rnd.round)
    assert ds.check(vout["workspace"]) == 0
    kp = to_np(keep)
    acc = to_np(vout["accepted"])
    nxt = to_np(vout["next_token"])
    assert np.all((acc >= 0) & (acc <= kp)) and np.all((nxt >= 0) & (nxt < rnd.V))
    ids = np.unique(np.concatenate([np.arange(32), np.arange(rnd.R - 32, rnd.R),
                                    np.random.default_rng(7).choice(rnd.R, 96, replace=False)]))
    total = check_verify(rnd, sout, keep, vout, ids)
    report("verify R=2048 V=65536", total)
    assert total["checked_requests"] == len(ids)
    assert total["draw"] + total["accept"] + total["residual_fp32"] <= 2


def test_tiny_round_end_to_end():
    """The tiny round exactly: the oracle runs alone from the inputs (its own draws feed its
    scheduler and verifier) and every output must equal the GPU's. A round in which one of the
    oracle's own decisions lies within the tolerance of a tie is counted, not compared; at
    least 18 of the 20 rounds must be compared in full."""
    rnd = wl.tiny(device=DEV)
    runner = ds.RoundRunner(rnd)
    skipped = {"draw": 0, "theta": 0, "verify": 0}
    compared = 0
    for rnd_idx in range(20):
        runner.set_round(rnd_idx)
        runner.run()
        assert runner.check() == 0
        res = runner.results()
        o_s = oracle.sample_block(to_np(rnd.U), to_np(rnd.E), to_np(rnd.W), to_np(rnd.h), to_np(rnd.w_h),
                                  to_np(rnd.w_e), rnd.b, to_np(rnd.temperature), to_np(rnd.anchor), rnd.seed,
                                  rnd_idx)
        gap = np.minimum(o_s["gap1"], o_s["gap2"])
        if np.any(gap < 1e-4):
            skipped["draw"] += 1
            continue
        assert np.array_equal(to_np(res["tokens"]), o_s["tokens"])
        assert np.allclose(to_np(res["surv"]), o_s["surv"], atol=1e-5)
        o_c = oracle.schedule(o_s["surv"], to_np(rnd.sps).astype(np.float64), rnd.mode)
        if o_c["min_margin"] <= 1e-12:
            skipped["theta"] += 1
            continue
        assert to_np(res["keep"]).tolist() == o_c["keep"].tolist()
        o_v = oracle.verify(to_np(rnd.target), to_np(rnd.U), to_np(rnd.E), to_np(rnd.W), to_np(rnd.anchor),
                            o_s["tokens"], o_s["lse"], o_s["logit"], o_c["keep"], to_np(rnd.temperature),
                            rnd.seed, rnd_idx)
        if np.nanmin(o_v["accept_margin"], initial=1.0) < 1e-4 or np.min(o_v["gap1"]) < 1e-4 or \
                np.min(o_v["gap2"]) < 1e-4:
            skipped["verify"] += 1
            continue
        assert to_np(res["accepted"]).tolist() == o_v["accepted"].tolist()
        assert to_np(res["next_token"]).tolist() == o_v["next_token"].tolist()
        assert to_np(res["resampled"]).tolist() == o_v["resampled"].tolist()
        compared += 1
    print("tiny round end to end: %d of 20 rounds compared in full, near-ties %s" % (compared, skipped))
    assert compared >= 18


def test_out_of_range_device_inputs_are_clamped_and_reported():
    rnd = _make(SMALL[0])
    bad = rnd.anchor.clone()
    bad[1] = rnd.V + 5
    out = ds.sample_block(rnd.U, rnd.E, rnd.W, rnd.h, rnd.w_h, rnd.w_e, rnd.b, rnd.temperature, bad, rnd.seed, 0)
    assert ds.check(out["workspace"]) == 6
    assert ds.check(out["workspace"]) == 0     # the word is cleared by the check
    toks = to_np(out["tokens"])
    assert np.all((toks >= 0) & (toks < rnd.V))
    keep = torch.tensor([9, 0, 1, 2], dtype=torch.int32, device=DEV)   # 9 > gamma
    v = ds.verify(rnd.target, rnd.U, rnd.E, rnd.W, rnd.anchor, out["tokens"], out["draft_lse"],
                  out["draft_logit"], keep, rnd.temperature, rnd.seed, 0)
    assert ds.check(v["workspace"]) == 6
    assert int(v["accepted"][0]) <= rnd.gamma_max


@pytest.mark.parametrize("n", [1_000_000])
def test_gpu_acceptance_rate_and_losslessness(n):
    """TV identity (0.8 at p_t = (0.7, 0.3), p_d = (0.5, 0.5)) and the law of the first
    emitted token over 10^6 rounds run on the GPU."""
    from scipy import special, stats
    ex = load_golden("worked_examples.json")["tv_identity"]
    R = 8192
    rounds = n // R + 1
    V, G = 16, 2
    rng = np.random.default_rng(3)
    ld = rng.normal(0, 1.5, (G, V))
    lt = rng.normal(0, 1.5, (G + 1, V))
    U = torch.tensor(ld, dtype=torch.float32, device=DEV).expand(R, G, V).contiguous()
    E = torch.zeros((V, 8), device=DEV)
    W = torch.zeros((8, V), device=DEV)
    h = torch.zeros((R, G, 8), device=DEV)
    z8 = torch.zeros(8, device=DEV)
    T = torch.ones(R, device=DEV)
    anchor = torch.zeros(R, dtype=torch.int32, device=DEV)
    target = torch.tensor(lt, dtype=torch.float32, device=DEV).expand(R, G + 1, V).contiguous()
    keep = torch.full((R,), 2, dtype=torch.int32, device=DEV)
    y1 = []
    for t in range(rounds):
        s = ds.sample_block(U, E, W, h, z8, z8, 0.0, T, anchor, 11, t)
        v = ds.verify(target, U, E, W, anchor, s["tokens"], s["draft_lse"], s["draft_logit"], keep, T, 11, t)
        y1.append(torch.where(v["accepted"] >= 1, s["tokens"][:, 0], v["next_token"]).cpu().numpy())
    y1 = np.concatenate(y1)
    pt = special.softmax(lt[0])
    counts = np.bincount(y1, minlength=V)
    assert stats.chisquare(counts, pt * counts.sum()).pvalue > 1e-3
    # two-point TV identity
    U2 = torch.tensor(np.log(ex["p_d"]), dtype=torch.float32, device=DEV).view(1, 1, 2).expand(R, 1, 2).contiguous()
    t2 = torch.tensor(np.log([ex["p_t"], [0.5, 0.5]]), dtype=torch.float32, device=DEV).view(1, 2, 2)
    t2 = t2.expand(R, 2, 2).contiguous()
    E2, W2 = torch.zeros((2, 8), device=DEV), torch.zeros((8, 2), device=DEV)
    h2 = torch.zeros((R, 1, 8), device=DEV)
    k1 = torch.ones(R, dtype=torch.int32, device=DEV)
    acc = 0
    for t in range(rounds):
        s = ds.sample_block(U2, E2, W2, h2, z8, z8, 0.0, T, anchor, 12, t)
        v = ds.verify(t2, U2, E2, W2, anchor, s["tokens"], s["draft_lse"], s["draft_logit"], k1, T, 12, t)
        acc += int(v["accepted"].sum())
    rate = acc / (rounds * R)
    assert abs(rate - ex["accept"]) < 5 * np.sqrt(0.16 / (rounds * R))
