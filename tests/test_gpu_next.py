"""GPU parity of the widening calls through the C ABI against the CPU oracle: the flattened
verify batch (dspark_assemble), the static confidence-threshold admission (scheduler mode 3),
sequential temperature scaling of the confidences (dspark_sample_block's sts_temp) and the RNN
sequential head (head = HEAD_RNN, with the verifier rebuilding rejected positions from a_rows)."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_draft_round_gb300 as ds
from speculative_decoding_draft_round_gb300 import workloads as wl
from parity import check_sample, to_np
from conftest import load_golden

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    ds.lib()
    oracle.build()


def _i32(a):
    return torch.as_tensor(np.asarray(a), dtype=torch.int32, device=DEV)


# ------------------------------------------------------------------ flattened verify batch

def _check_assemble(keep, anchor, tokens):
    out = ds.assemble(_i32(keep), _i32(anchor), _i32(tokens))
    torch.cuda.synchronize()
    assert ds.check(out["workspace"]) == 0
    o = oracle.assemble(keep, anchor, tokens)
    for k in ("flat_tokens", "flat_request", "flat_position", "offsets"):
        np.testing.assert_array_equal(to_np(out[k]), o[k], err_msg=k)   # index work: bit-exact


@pytest.mark.parametrize("R,G", [(1, 1), (3, 3), (37, 6), (1000, 7), (8192, 1), (512, 16)])
def test_assemble_matches_oracle(R, G):
    rng = np.random.default_rng(R * 31 + G)
    keep = rng.integers(0, G + 1, R)
    anchor = rng.integers(0, 151936, R)
    tokens = rng.integers(0, 151936, (R, G))
    _check_assemble(keep, anchor, tokens)
    _check_assemble(np.zeros(R, np.int64), anchor, tokens)        # nothing admitted
    _check_assemble(np.full(R, G), anchor, tokens)                # everything admitted


def test_assemble_clamps_out_of_range_keep():
    R, G = 5, 4
    keep = np.array([1, -3, 9, 4, 0])
    anchor, tokens = np.arange(R), np.arange(R * G).reshape(R, G) + 100
    out = ds.assemble(_i32(keep), _i32(anchor), _i32(tokens))
    torch.cuda.synchronize()
    assert ds.check(out["workspace"]) == 6   # DSPARK_ERR_DEVICE_INPUT: clamped
    o = oracle.assemble(np.clip(keep, 0, G), anchor, tokens)
    np.testing.assert_array_equal(to_np(out["flat_tokens"]), o["flat_tokens"])
    np.testing.assert_array_equal(to_np(out["offsets"]), o["offsets"])


def test_assemble_after_a_full_round():
    rnd = wl.WORKLOADS[3](device=DEV)
    runner = ds.RoundRunner(rnd)
    runner.set_round(4)
    runner.run()
    assert runner.check() == 0
    res = runner.results()
    tokens = to_np(res["tokens"])
    keep = to_np(res["keep"])
    anchor = to_np(rnd.anchor)
    _check_assemble(keep, anchor, np.where(tokens < 0, 0, tokens))


# ------------------------------------------------------------------ static threshold admission

def _check_threshold(surv, sps, thr, gamma=None):
    s32 = torch.as_tensor(surv, dtype=torch.float32, device=DEV)
    g = None if gamma is None else _i32(gamma)
    sp = torch.as_tensor(sps, dtype=torch.float32, device=DEV)
    out = ds.schedule(s32, sp, ds.SCHED_THRESHOLD, gamma=g, threshold=thr)
    torch.cuda.synchronize()
    assert ds.check(out["workspace"]) == 0
    thr32 = float(np.float32(thr))   # the call compares against the fp32 threshold
    o = oracle.schedule(to_np(s32).astype(np.float64), to_np(sp).astype(np.float64), oracle.SCHED_THRESHOLD,
                        gamma=None if gamma is None else np.asarray(gamma), threshold=thr32)
    st = ds.decode_stats(out["stats"])
    np.testing.assert_array_equal(to_np(out["keep"]), o["keep"])   # exact comparisons: bit-exact
    assert st["admitted"] == o["admitted"] and st["pool"] == o["pool"] and st["capacity"] == -1
    assert st["batch"] == s32.shape[0] + o["admitted"]
    assert abs(st["theta_best"] - o["theta_best"]) <= 1e-9 * abs(o["theta_best"])
    return st


def test_threshold_worked_example_on_gpu():
    ex = load_golden("worked_examples.json")["single_request"]
    surv = np.cumprod(np.array(ex["c"]))[None, :]
    sps = np.array(ex["sps"] + [ex["sps"][-1] * 0.9 ** i for i in range(1, 16)])
    for thr, keep in ((0.96, 0), (0.9, 1), (0.8, 2), (0.5, 3), (0.2, 4)):
        st = _check_threshold(surv, sps, thr)
        assert st["admitted"] == keep


@pytest.mark.parametrize("R,G", [(9, 5), (128, 16), (512, 16)])
def test_threshold_matches_oracle(R, G):
    rng = np.random.default_rng(R + G)
    surv = np.cumprod(rng.uniform(0.3, 1.0, (R, G)), axis=1)
    gamma = rng.integers(0, G + 1, R)
    sps = wl.sps_staircase(R * (1 + G)).numpy()
    for thr in (0.0, 0.25, 0.6, 0.95, 1.5):
        _check_threshold(surv, sps, thr, gamma)
    # survivals exactly at the threshold are admitted (>=)
    surv[0, :] = np.float32(0.5)
    _check_threshold(surv, sps, 0.5, gamma)


# ------------------------------------------------------------------ sequential temperature scaling

@pytest.mark.parametrize("spec", [
    dict(name="sts_f32", R=11, G=5, V=300, r=24, d=20, dtype="f32", ew_std=0.2, gamma=[5, 0, 3, 5, 1, 2, 5, 4, 5, 0, 5]),
    dict(name="sts_bf16", R=160, G=3, V=1000, r=64, d=96, dtype="bf16", ew_std=0.15),
], ids=["cuda_core_f32", "tensor_core_bf16"])
def test_sts_temperatures_match_oracle(spec):
    spec = dict(spec)
    name = spec.pop("name")
    R, G, V, r, d, dtype = (spec.pop(k) for k in ("R", "G", "V", "r", "d", "dtype"))
    rnd = wl.make_round(name, R, G, V, r, d, dtype, seed=77, device=DEV, sps=wl.sps_hyperbolic(R * (1 + G)),
                        **spec)
    rnd.round = 3
    t = torch.tensor([0.5, 1.7, 3.0, 0.8, 1.1][:G], dtype=torch.float32, device=DEV)
    out = ds.sample_block(rnd.U, rnd.E, rnd.W, rnd.h, rnd.w_h, rnd.w_e, rnd.b, rnd.temperature, rnd.anchor,
                          rnd.seed, rnd.round, gamma=rnd.gamma, sts_temp=t)
    torch.cuda.synchronize()
    assert ds.check(out["workspace"]) == 0
    check_sample(rnd, out, np.arange(R), sts_temp=t)   # the oracle gets the same temperatures


# ------------------------------------------------------------------ greedy decoding (temperature 0)

GREEDY_SPECS = [
    dict(name="greedy_f32", R=11, G=5, V=300, r=24, d=20, dtype="f32", ew_std=0.2),
    dict(name="greedy_bf16", R=160, G=3, V=1000, r=64, d=96, dtype="bf16", ew_std=0.15),
]


def _greedy_round(spec, seed):
    spec = dict(spec)
    name = spec.pop("name")
    R, G, V, r, d, dtype = (spec.pop(k) for k in ("R", "G", "V", "r", "d", "dtype"))
    # every third request decodes greedily, the others sample at T in [0.5, 1.5)
    temp = lambda R_, g, dev: torch.where(torch.arange(R_, device=dev) % 3 == 0, torch.zeros(R_, device=dev),
                                          0.5 + torch.rand((R_,), generator=g, device=dev))
    rnd = wl.make_round(name, R, G, V, r, d, dtype, seed=seed, device=DEV, temperature=temp,
                        sps=wl.sps_hyperbolic(R * (1 + G)), **spec)
    rnd.round = 5
    return rnd


@pytest.mark.parametrize("spec", GREEDY_SPECS, ids=["cuda_core_f32", "tensor_core_bf16"])
def test_greedy_draft_matches_oracle(spec):
    rnd = _greedy_round(spec, 31)
    out = ds.sample_block(rnd.U, rnd.E, rnd.W, rnd.h, rnd.w_h, rnd.w_e, rnd.b, rnd.temperature, rnd.anchor,
                          rnd.seed, rnd.round, gamma=rnd.gamma)
    torch.cuda.synchronize()
    assert ds.check(out["workspace"]) == 0
    check_sample(rnd, out, np.arange(rnd.R))
    g = to_np(rnd.temperature) == 0
    np.testing.assert_array_equal(to_np(out["draft_lse"])[g], to_np(out["draft_logit"])[g])


@pytest.mark.parametrize("spec", GREEDY_SPECS, ids=["cuda_core_f32", "tensor_core_bf16"])
def test_greedy_verify_matches_oracle(spec):
    from parity import check_verify
    rnd = _greedy_round(spec, 32)
    out = ds.sample_block(rnd.U, rnd.E, rnd.W, rnd.h, rnd.w_h, rnd.w_e, rnd.b, rnd.temperature, rnd.anchor,
                          rnd.seed, rnd.round, gamma=rnd.gamma)
    torch.cuda.synchronize()
    R, G, V = rnd.R, rnd.gamma_max, rnd.V
    # make the target's arg-max agree with the draft on about 60% of the positions
    tok = out["tokens"].long()
    agree = torch.rand((R, G), device=DEV) < 0.6
    tgt = rnd.target.float()
    rowmax = tgt[:, :G].amax(dim=2)
    bump = torch.where(agree, rowmax + 4.0, tgt[:, :G].gather(2, tok.unsqueeze(2)).squeeze(2))
    tgt[:, :G].scatter_(2, tok.unsqueeze(2), bump.unsqueeze(2))
    rnd.target = tgt.to(rnd.target.dtype)
    keep = torch.randint(0, G + 1, (R,), device=DEV, dtype=torch.int32)
    v = ds.verify(rnd.target, rnd.U, rnd.E, rnd.W, rnd.anchor, out["tokens"], out["draft_lse"],
                  out["draft_logit"], keep, rnd.temperature, rnd.seed, rnd.round, gamma=rnd.gamma)
    torch.cuda.synchronize()
    assert ds.check(v["workspace"]) == 0
    n_exc = check_verify(rnd, out, keep, v, np.arange(R))
    # greedy verification compares raw target values exactly: no excusal on those requests
    g = np.where(to_np(rnd.temperature) == 0)[0]
    o = oracle.verify(to_np(rnd.target)[g], to_np(rnd.U)[g], to_np(rnd.E), to_np(rnd.W), to_np(rnd.anchor)[g],
                      to_np(out["tokens"])[g], to_np(out["draft_lse"])[g].astype(np.float64),
                      to_np(out["draft_logit"])[g].astype(np.float64), to_np(keep)[g],
                      to_np(rnd.temperature)[g], rnd.seed, rnd.round, req_ids=g)
    np.testing.assert_array_equal(to_np(v["accepted"])[g], o["accepted"])
    np.testing.assert_array_equal(to_np(v["next_token"])[g], o["next_token"])
    np.testing.assert_array_equal(to_np(v["resampled"])[g], o["resampled"])


# ------------------------------------------------------------------ RNN sequential head (eq. 6)

RNN_SPECS = [
    dict(name="rnn_f32", R=11, G=5, V=300, r=24, d=20, dtype="f32", ew_std=0.2, gamma=[5, 0, 3, 5, 1, 2, 5, 4, 5, 0, 5]),
    dict(name="rnn_tiles_bf16", R=160, G=3, V=1000, r=64, d=96, dtype="bf16", ew_std=0.15),
    dict(name="rnn_wide_bf16", R=37, G=4, V=2056, r=256, d=64, dtype="bf16", ew_std=0.05, gamma=[4, 2] * 18 + [3]),
    # 2r + d = 228 is not a multiple of 8: W_rnn rows do not meet the copy engine's 16-byte pitch, so the
    # step runs on CUDA cores beside the tensor-core statistics kernel
    dict(name="rnn_pitch_bf16", R=40, G=3, V=1024, r=64, d=100, dtype="bf16", ew_std=0.15),
]


def _rnn_round(spec, seed):
    spec = dict(spec)
    name = spec.pop("name")
    R, G, V, r, d, dtype = (spec.pop(k) for k in ("R", "G", "V", "r", "d", "dtype"))
    rnd = wl.make_round(name, R, G, V, r, d, dtype, seed=seed, device=DEV, sps=wl.sps_hyperbolic(R * (1 + G)),
                        **spec)
    rnd.round = 6
    return rnd, wl.rnn_weights(rnd)


@pytest.mark.parametrize("spec", RNN_SPECS, ids=[s["name"] for s in RNN_SPECS])
def test_rnn_head_matches_oracle(spec):
    from parity import check_verify
    rnd, W_rnn = _rnn_round(spec, 41)
    paths = [ds.PATH_CUDA_CORE] + ([ds.PATH_TENSOR_CORE] if rnd.dtype == "bf16" else [])
    for path in paths:
        out = ds.sample_block(rnd.U, rnd.E, rnd.W, rnd.h, rnd.w_h, rnd.w_e, rnd.b, rnd.temperature, rnd.anchor,
                              rnd.seed, rnd.round, gamma=rnd.gamma, path=path, head=ds.HEAD_RNN, W_rnn=W_rnn,
                              a_rows=True)
        torch.cuda.synchronize()
        assert ds.check(out["workspace"]) == 0
        check_sample(rnd, out, np.arange(rnd.R), head=ds.HEAD_RNN, W_rnn=W_rnn)
        # verification rebuilds a rejected position's draft with the reported operands
        g = np.full(rnd.R, rnd.gamma_max) if rnd.gamma is None else to_np(rnd.gamma)
        keep = _i32(g)
        v = ds.verify(rnd.target, rnd.U, rnd.E, rnd.W, rnd.anchor, out["tokens"].clamp(min=0), out["draft_lse"],
                      out["draft_logit"], keep, rnd.temperature, rnd.seed, rnd.round, gamma=rnd.gamma,
                      a_rows=out["a_rows"])
        torch.cuda.synchronize()
        assert ds.check(v["workspace"]) == 0
        check_verify(rnd, out, keep, v, np.arange(rnd.R), a_rows=out["a_rows"])


def test_markov_head_reports_its_operand_rows():
    rnd, _ = _rnn_round(RNN_SPECS[1], 42)
    out = ds.sample_block(rnd.U, rnd.E, rnd.W, rnd.h, rnd.w_h, rnd.w_e, rnd.b, rnd.temperature, rnd.anchor,
                          rnd.seed, rnd.round, gamma=rnd.gamma, a_rows=True)
    torch.cuda.synchronize()
    check_sample(rnd, out, np.arange(rnd.R))   # compares a_rows with W_1[x_{k-1}]


def test_static_entry_runs_the_rnn_head():
    # no library handle or allocation on the RNN head's path: the static entry takes it when its
    # scratch fits the array, and matches the workspace entry
    rnd, W_rnn = _rnn_round(RNN_SPECS[2], 43)
    ref = ds.sample_block(rnd.U, rnd.E, rnd.W, rnd.h, rnd.w_h, rnd.w_e, rnd.b, rnd.temperature, rnd.anchor,
                          rnd.seed, rnd.round, gamma=rnd.gamma, head=ds.HEAD_RNN, W_rnn=W_rnn)
    assert ds.check(ref["workspace"]) == 0
    got = ds.sample_block_static(rnd.U, rnd.E, rnd.W, rnd.h, rnd.w_h, rnd.w_e, rnd.b, rnd.temperature, rnd.anchor,
                                 rnd.seed, rnd.round, gamma=rnd.gamma, head=ds.HEAD_RNN, W_rnn=W_rnn)
    assert ds.check_static() == 0
    assert torch.equal(got["tokens"], ref["tokens"])
    for k in ("conf", "surv", "draft_lse", "draft_logit"):
        assert torch.allclose(got[k], ref[k], rtol=0, atol=1e-5 * max(1.0, float(ref[k].abs().max()))), k


def test_step_ready_events_keep_the_results():
    # the sampler waits on per-step events (inputs still arriving); the draws do not change
    rnd, _ = _rnn_round(RNN_SPECS[1], 44)
    runner = ds.RoundRunner(rnd)
    runner.set_round(3)
    runner.run()
    torch.cuda.synchronize()
    ref = {k: v.clone() for k, v in runner.results().items() if torch.is_tensor(v)}
    side = torch.cuda.Stream()
    events = [torch.cuda.Event() for _ in range(rnd.gamma_max)]
    side.wait_stream(torch.cuda.current_stream())
    for ev in events:
        ev.record(side)
    runner.run_draft(step_ready=events)
    runner.run_verify()
    torch.cuda.synchronize()
    assert runner.check() == 0
    got = runner.results()
    for k in ("tokens", "conf", "surv", "keep", "accepted", "next_token"):
        assert torch.equal(got[k], ref[k]), k


# ------------------------------------------------------------------ the resident loop's variants

def test_resident_loop_variants_match_oracle():
    """Greedy requests mixed with sampled ones, per-position confidence temperatures, no bias at the
    first step, the conditioning-token choice of eq. 7, reported operand rows and ragged draft
    lengths, on the persistent W-resident path (one CTA per vocabulary block here)."""
    temp = lambda R_, g, dev: torch.where(torch.arange(R_, device=dev) % 3 == 0, torch.zeros(R_, device=dev),
                                          0.5 + torch.rand((R_,), generator=g, device=dev))
    for conf_token, bias_first in ((0, 0), (1, 1)):
        rnd = wl.make_round("loop_var", 96, 5, 12800, 256, 64, "bf16", seed=51, device=DEV, temperature=temp,
                            sps=wl.sps_hyperbolic(96 * 6), conf_token=conf_token, bias_first=bias_first,
                            gamma=[5, 3, 0, 4, 5, 1] * 16)
        rnd.round = 7
        t = torch.tensor([0.7, 1.3, 2.0, 0.9, 1.1], dtype=torch.float32, device=DEV)
        out = ds.sample_block(rnd.U, rnd.E, rnd.W, rnd.h, rnd.w_h, rnd.w_e, rnd.b, rnd.temperature, rnd.anchor,
                              rnd.seed, rnd.round, gamma=rnd.gamma, conf_token=conf_token, bias_first=bias_first,
                              path=ds.PATH_RESIDENT, sts_temp=t, a_rows=True)
        torch.cuda.synchronize()
        assert ds.check(out["workspace"]) == 0
        check_sample(rnd, out, np.arange(rnd.R), sts_temp=t)
        g = to_np(rnd.temperature) == 0
        np.testing.assert_array_equal(to_np(out["draft_lse"])[g], to_np(out["draft_logit"])[g])
