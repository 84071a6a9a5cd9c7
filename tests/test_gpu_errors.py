"""Device-side error paths, made to happen without faulting the GPU: non-finite inputs are
flagged in the status word (never trapped), and a bounded wait that runs out (its bound set to
almost nothing through dspark_set_wait_limit) records a timeout, lets the kernel's own copies
and MMAs land, frees its tensor memory and returns, so that the next call runs normally."""
import numpy as np
import pytest
import torch

import speculative_decoding_draft_round_gb300 as ds
from speculative_decoding_draft_round_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    ds.lib()


def _round(dtype):
    if dtype == "bf16":   # tensor-core path: several request tiles, a ragged vocabulary tail
        return wl.make_round("err_bf16", 160, 3, 1000, 64, 96, "bf16", seed=61, device=DEV, ew_std=0.15)
    return wl.make_round("err_f32", 11, 4, 300, 24, 20, "f32", seed=62, device=DEV, ew_std=0.2)


def _sample(rnd, U=None, h=None, path=ds.PATH_AUTO, rnd_idx=3):
    return ds.sample_block(rnd.U if U is None else U, rnd.E, rnd.W, rnd.h if h is None else h, rnd.w_h, rnd.w_e,
                           rnd.b, rnd.temperature, rnd.anchor, rnd.seed, rnd_idx, gamma=rnd.gamma, path=path)


def _paths(rnd):
    return [ds.PATH_CUDA_CORE] + ([ds.PATH_TENSOR_CORE] if rnd.dtype == "bf16" else [])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("bad", [float("nan"), float("inf")])
def test_nonfinite_draft_logit_is_flagged(dtype, bad):
    rnd = _round(dtype)
    for path in _paths(rnd):
        U = rnd.U.clone()
        U[5 % rnd.R, 1, 17] = bad
        out = _sample(rnd, U=U, path=path)
        assert ds.check(out["workspace"]) == ds.ERR_NONFINITE_INPUT, "path %d" % path
        out = _sample(rnd, path=path)   # the same call on clean inputs
        assert ds.check(out["workspace"]) == 0, "path %d" % path


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_minus_infinity_is_a_zero_weight(dtype):
    rnd = _round(dtype)
    for path in _paths(rnd):
        ref = _sample(rnd, path=path)
        U = rnd.U.clone()
        # mask the token each request drafted at position 0: it can no longer be drawn there
        tok0 = ref["tokens"][:, 0].long()
        U[torch.arange(rnd.R, device=DEV), 0, tok0] = float("-inf")
        out = _sample(rnd, U=U, path=path)
        assert ds.check(out["workspace"]) == 0
        assert not torch.any(out["tokens"][:, 0] == ref["tokens"][:, 0])
        assert torch.all(torch.isfinite(out["draft_lse"]))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_nonfinite_hidden_state_is_flagged(dtype):
    rnd = _round(dtype)
    h = rnd.h.clone()
    h[2, 0, 3] = float("nan")
    out = _sample(rnd, h=h)
    assert ds.check(out["workspace"]) == ds.ERR_NONFINITE_INPUT


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_nonfinite_target_logit_is_flagged(dtype):
    rnd = _round(dtype)
    s = _sample(rnd)
    keep = torch.full((rnd.R,), rnd.gamma_max, dtype=torch.int32, device=DEV)
    for bad in (float("nan"), float("inf")):
        tgt = rnd.target.clone()
        tgt[1, 0, 40] = bad
        v = ds.verify(tgt, rnd.U, rnd.E, rnd.W, rnd.anchor, s["tokens"], s["draft_lse"], s["draft_logit"], keep,
                      rnd.temperature, rnd.seed, 3)
        assert ds.check(v["workspace"]) == ds.ERR_NONFINITE_INPUT
    v = ds.verify(rnd.target, rnd.U, rnd.E, rnd.W, rnd.anchor, s["tokens"], s["draft_lse"], s["draft_logit"], keep,
                  rnd.temperature, rnd.seed, 3)
    assert ds.check(v["workspace"]) == 0


def test_wait_that_runs_out_records_a_timeout_and_the_next_call_recovers():
    rnd = _round("bf16")
    ref = _sample(rnd, path=ds.PATH_TENSOR_CORE)
    assert ds.check(ref["workspace"]) == 0
    codes = []
    old = ds.set_wait_limit(1)   # 1 ns: any wait that is not satisfied at once runs out
    try:
        for _ in range(3):
            out = _sample(rnd, path=ds.PATH_TENSOR_CORE)
            codes.append(ds.check(out["workspace"]))
            if codes[-1] == ds.ERR_TIMEOUT:
                break
    finally:
        ds.set_wait_limit(0)
    assert old == 4_000_000_000
    assert ds.ERR_TIMEOUT in codes, codes
    # the aborted kernels released their tensor memory and drained their copies: the same call
    # now runs normally and reproduces the reference exactly
    again = _sample(rnd, path=ds.PATH_TENSOR_CORE)
    assert ds.check(again["workspace"]) == 0
    for k in ("tokens", "conf", "surv", "draft_lse", "draft_logit"):
        assert torch.equal(again[k], ref[k]), k
