"""dspark_sample_block_static: the sampler entry point that takes no workspace.

It exists for callers that cannot allocate device memory where they run a round (code inside
another framework's memory pool without access to its allocator, code that must not grow the
device footprint after start-up, runtimes that only pass input and output buffers). Its
scratch lives in a fixed device array of the library. This file is collected last so that a
run stopping at the first failure has already run every other test; it passes alone in a fresh
process and after the other tests."""
import numpy as np
import pytest
import torch

import speculative_decoding_draft_round_gb300 as ds
from speculative_decoding_draft_round_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

CONF_TOL = 1e-5   # the tolerance the parity tests use for c_k and a_k


def _compare(a, b):
    assert torch.equal(a["tokens"], b["tokens"])
    for k in ("conf", "surv", "draft_lse", "draft_logit"):
        assert torch.allclose(a[k], b[k], rtol=0, atol=CONF_TOL * max(1.0, float(b[k].abs().max()))), k


@pytest.mark.parametrize("shape", ["tensor_core", "fp32"])
def test_static_entry_matches_workspace_entry_twice(shape):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    if shape == "tensor_core":
        rnd = wl.make_round("nalloc_bf16", 160, 3, 1000, 64, 96, "bf16", seed=9, device="cuda", ew_std=0.15,
                            gamma=[3, 1, 2, 0] * 40)
    else:
        rnd = wl.make_round("nalloc_f32", 6, 4, 300, 24, 20, "f32", seed=10, device="cuda", ew_std=0.2)
    for rnd_idx in (4, 5):   # two calls in a row: the array keeps the previous call's contents
        ref = ds.sample_block(rnd.U, rnd.E, rnd.W, rnd.h, rnd.w_h, rnd.w_e, rnd.b, rnd.temperature, rnd.anchor,
                              rnd.seed, rnd_idx, gamma=rnd.gamma)
        assert ds.check(ref["workspace"]) == 0
        got = ds.sample_block_static(rnd.U, rnd.E, rnd.W, rnd.h, rnd.w_h, rnd.w_e, rnd.b, rnd.temperature,
                                     rnd.anchor, rnd.seed, rnd_idx, gamma=rnd.gamma)
        assert ds.check_static() == 0   # synchronises; no clamped input, timeout or non-finite value
        _compare(got, ref)


def test_static_entry_rejects_shapes_beyond_its_array():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    # the call is refused on the host before any launch, so uninitialised inputs suffice
    R, G, V, r, d = 8192, 1, 32768, 64, 8
    dev = "cuda"
    bf = torch.bfloat16
    args = (torch.empty((R, G, V), dtype=bf, device=dev), torch.empty((V, r), dtype=bf, device=dev),
            torch.empty((r, V), dtype=bf, device=dev), torch.empty((R, G, d), dtype=bf, device=dev),
            torch.zeros(d, device=dev), torch.zeros(r, device=dev), 0.0, torch.ones(R, device=dev),
            torch.zeros(R, dtype=torch.int32, device=dev), 1, 0)
    a, _ = ds.sample_args(*args)
    assert ds.workspace_bytes("sample", a) > ds.STATIC_WORKSPACE_BYTES
    with pytest.raises(ds.DsparkError) as err:
        ds.sample_block_static(*args)
    assert err.value.code == 2


@pytest.mark.parametrize("workload", [1, 2, 3, 4, 5])
def test_static_array_holds_each_workload(workload):
    """The scratch each of the five workload shapes needs, from dspark_sample_workspace_size on
    this device (the tensor-core layout depends on the SM count), fits the static array."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    R, G, V, r, d, dt = wl.SHAPES[workload]
    dev = "cuda"
    args = (torch.empty((R, G, V), dtype=dt, device=dev), torch.empty((V, r), dtype=dt, device=dev),
            torch.empty((r, V), dtype=dt, device=dev), torch.empty((R, G, d), dtype=dt, device=dev),
            torch.zeros(d, device=dev), torch.zeros(r, device=dev), 0.0, torch.ones(R, device=dev),
            torch.zeros(R, dtype=torch.int32, device=dev), 1, 0)
    a, _ = ds.sample_args(*args)
    need = ds.workspace_bytes("sample", a)
    print("workload %d (R=%d G=%d V=%d r=%d): sampler scratch %.2f MiB of %.0f MiB" % (
        workload, R, G, V, r, need / 2**20, ds.STATIC_WORKSPACE_BYTES / 2**20))
    assert need <= ds.STATIC_WORKSPACE_BYTES
    del args
    torch.cuda.empty_cache()
