"""C ABI checks that need no GPU: the library builds and loads, exports every
function include/dspark.h declares, its argument structs have the layout the
Python binding assumes, and host-side validation rejects bad arguments before
any launch."""
import ctypes as C
import os
import re
import subprocess
import tempfile

import pytest

import speculative_decoding_draft_round_gb300 as ds
from speculative_decoding_draft_round_gb300 import build as dsbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dspark.h")


@pytest.fixture(scope="module")
def L():
    dsbuild.build()
    return ds.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(dspark_\w+)\s*\(", text, flags=re.M)))


def test_every_declared_function_is_exported(L):
    names = _declared()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(ds.EXPORTS) | set(n for n in names if n not in ds.EXPORTS)
    for n in ds.EXPORTS:
        assert n in names


def test_struct_layouts_match_c(L):
    prog = r'''
#include <stdio.h>
#include <stddef.h>
#include "dspark.h"
int main(void) {
  printf("%zu %zu %zu %zu\n", sizeof(dspark_sample_args), sizeof(dspark_schedule_args),
         sizeof(dspark_verify_args), sizeof(dspark_schedule_stats));
  printf("%zu %zu %zu\n", offsetof(dspark_sample_args, seed), offsetof(dspark_sample_args, draft_logit),
         offsetof(dspark_sample_args, b));
  printf("%zu %zu\n", offsetof(dspark_verify_args, seed), offsetof(dspark_verify_args, resampled));
  printf("%zu %zu\n", offsetof(dspark_schedule_args, gamma), offsetof(dspark_schedule_args, stats));
  return 0;
}
'''
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "t.c")
        exe = os.path.join(d, "t")
        open(src, "w").write(prog)
        subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), src, "-o", exe], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split()
    vals = [int(x) for x in out]
    assert vals[0] == C.sizeof(ds.SampleArgs)
    assert vals[1] == C.sizeof(ds.ScheduleArgs)
    assert vals[2] == C.sizeof(ds.VerifyArgs)
    assert vals[3] == C.sizeof(ds.ScheduleStats)
    assert vals[4] == ds.SampleArgs.seed.offset and vals[5] == ds.SampleArgs.draft_logit.offset
    assert vals[6] == ds.SampleArgs.b.offset
    assert vals[7] == ds.VerifyArgs.seed.offset and vals[8] == ds.VerifyArgs.resampled.offset
    assert vals[9] == ds.ScheduleArgs.gamma.offset and vals[10] == ds.ScheduleArgs.stats.offset


def test_version_and_status_strings(L):
    assert L.dspark_abi_version() == 1
    for code in range(7):
        assert L.dspark_status_string(code)
    assert L.dspark_status_string(99) == b"unknown status"


def _fake_sample_args(**kw):
    a = ds.SampleArgs()
    a.struct_size = C.sizeof(ds.SampleArgs)
    a.R, a.gamma_max, a.V, a.r, a.d, a.dtype = 4, 4, 64, 8, 32, ds.F32
    fake = 0x10000
    for f in ("U", "E", "W", "h", "w_h", "w_e", "temperature", "anchor", "tokens", "conf", "surv",
              "draft_lse", "draft_logit"):
        setattr(a, f, fake)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_sample_validation_happens_before_any_launch(L):
    n = C.c_size_t(0)
    assert L.dspark_sample_workspace_size(C.byref(_fake_sample_args()), C.byref(n)) == 0
    assert n.value >= 256
    bad = [dict(struct_size=7), dict(R=0), dict(gamma_max=33), dict(V=0), dict(r=0), dict(dtype=5),
           dict(conf_token=2), dict(bias_first=3), dict(path=9), dict(round=1 << 29), dict(U=None),
           dict(tokens=None)]
    for kw in bad:
        assert L.dspark_sample_workspace_size(C.byref(_fake_sample_args(**kw)), C.byref(n)) == 1, kw
    # too-small workspace is refused before launching anything
    assert L.dspark_sample_block(C.byref(_fake_sample_args()), 0x20000, 16, None) == 3
    assert L.dspark_sample_block(C.byref(_fake_sample_args()), None, 1 << 20, None) == 3
    # the tensor-core path needs bf16; forcing it on fp32 is an unsupported shape
    assert L.dspark_sample_block(C.byref(_fake_sample_args(path=2)), 0x20000, 1 << 30, None) == 2


def test_schedule_validation(L):
    a = ds.ScheduleArgs()
    a.struct_size = C.sizeof(ds.ScheduleArgs)
    a.R, a.gamma_max, a.mode, a.n_sps = 512, 16, 0, 512 * 17
    a.surv = a.sps = a.keep = a.stats = 0x10000
    n = C.c_size_t(0)
    assert L.dspark_schedule_workspace_size(C.byref(a), C.byref(n)) == 0
    a.R = 513
    assert L.dspark_schedule_workspace_size(C.byref(a), C.byref(n)) == 2   # > 8192 slots
    a.R, a.n_sps = 512, 100
    assert L.dspark_schedule_workspace_size(C.byref(a), C.byref(n)) == 1   # SPS table too short
    a.n_sps, a.mode = 512 * 17, 1
    assert L.dspark_schedule_workspace_size(C.byref(a), C.byref(n)) == 1   # async needs old survivals
    a.mode = 3                                                                 # static threshold
    assert L.dspark_schedule_workspace_size(C.byref(a), C.byref(n)) == 0
    a.threshold = float("nan")
    assert L.dspark_schedule_workspace_size(C.byref(a), C.byref(n)) == 1
    a.mode, a.threshold = 4, 0.5
    assert L.dspark_schedule_workspace_size(C.byref(a), C.byref(n)) == 1


def test_assemble_validation(L):
    a = ds.AssembleArgs()
    a.struct_size = C.sizeof(ds.AssembleArgs)
    a.R, a.gamma_max = 128, 16
    for f in ("keep", "anchor", "tokens", "flat_tokens", "flat_request", "flat_position", "offsets"):
        setattr(a, f, 0x10000)
    n = C.c_size_t(0)
    assert L.dspark_assemble_workspace_size(C.byref(a), C.byref(n)) == 0 and n.value == 256
    # refused on the host before any launch
    assert L.dspark_assemble(C.byref(a), None, 0, None) == 3                  # no workspace
    a.R = 8193
    assert L.dspark_assemble(C.byref(a), C.c_void_p(0x10000), 256, None) == 2
    a.R, a.gamma_max = 128, 33
    assert L.dspark_assemble(C.byref(a), C.c_void_p(0x10000), 256, None) == 1
    a.gamma_max, a.offsets = 16, 0
    assert L.dspark_assemble(C.byref(a), C.c_void_p(0x10000), 256, None) == 1
    a.struct_size = 4
    assert L.dspark_assemble_workspace_size(C.byref(a), C.byref(n)) == 1


def test_verify_validation(L):
    a = ds.VerifyArgs()
    a.struct_size = C.sizeof(ds.VerifyArgs)
    a.R, a.gamma_max, a.V, a.r, a.dtype = 8, 4, 100, 16, ds.BF16
    for f in ("target", "U", "E", "W", "anchor", "tokens", "draft_lse", "draft_logit", "keep", "temperature",
              "accepted", "next_token", "resampled"):
        setattr(a, f, 0x10000)
    n = C.c_size_t(0)
    assert L.dspark_verify_workspace_size(C.byref(a), C.byref(n)) == 0
    a.keep = None
    assert L.dspark_verify_workspace_size(C.byref(a), C.byref(n)) == 1


def test_library_links_no_vendor_math_library(L):
    """Every contraction on the path runs in this library's own kernels: the shared object
    links the CUDA runtime only, no cuBLAS / cuDNN."""
    out = subprocess.run(["ldd", ds.LIB_PATH], capture_output=True, text=True).stdout
    for lib in ("cublas", "cudnn", "cusparse"):
        assert lib not in out, out
