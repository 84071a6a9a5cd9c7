"""Plain CPU oracle for one DSpark draft round -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package. The CUDA
library never links, loads or calls it, and it shares no code with it.

The arithmetic lives in ``dspark_oracle.c`` (IEEE double, literal loops, its
own Philox4x32-10); this module only builds that file with gcc and marshals
numpy arrays through ctypes. Requests are independent in the sampler and the
verifier, so calls may be split over threads (ctypes releases the GIL while a
foreign function runs).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dspark_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libdspark_oracle.so")

F32, BF16, F64 = 0, 1, 2
SCHED_SYNC, SCHED_ASYNC_CAPACITY, SCHED_FULL_SCAN, SCHED_THRESHOLD = 0, 1, 2, 3
HEAD_MARKOV, HEAD_RNN = 0, 1

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libdspark_oracle.so`` (gcc, no fast-math,
    no floating-point contraction, so x86 and Arm give the same doubles)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "dspark_oracle.h"))
    ):
        return _LIB_PATH
    tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _SampleArgs(C.Structure):
    _fields_ = [
        ("R", C.c_int), ("gamma_max", C.c_int), ("V", C.c_int), ("r", C.c_int), ("d", C.c_int),
        ("dtype", C.c_int),
        ("gamma", C.c_void_p), ("req_ids", C.c_void_p),
        ("U", C.c_void_p), ("E", C.c_void_p), ("W", C.c_void_p), ("h", C.c_void_p),
        ("w_h", C.c_void_p), ("w_e", C.c_void_p), ("b", C.c_float),
        ("temperature", C.c_void_p), ("anchor", C.c_void_p),
        ("seed", C.c_uint64), ("round", C.c_uint64),
        ("conf_token", C.c_int), ("bias_first", C.c_int), ("noise_block", C.c_int),
        ("forced_tokens", C.c_void_p),
        ("tokens", C.c_void_p), ("conf", C.c_void_p), ("surv", C.c_void_p), ("lse", C.c_void_p),
        ("logit", C.c_void_p), ("gap1", C.c_void_p), ("gap2", C.c_void_p),
        ("sts_temp", C.c_void_p), ("head", C.c_int), ("W_rnn", C.c_void_p), ("a_rows", C.c_void_p),
        ("logp", C.c_void_p),
    ]


class _ScheduleArgs(C.Structure):
    _fields_ = [
        ("P", C.c_int), ("R", C.c_int), ("gamma_max", C.c_int),
        ("gamma", C.c_void_p), ("surv", C.c_void_p), ("surv_capacity", C.c_void_p),
        ("sps", C.c_void_p), ("n_sps", C.c_int), ("mode", C.c_int),
        ("keep", C.c_void_p), ("theta_best", C.c_void_p), ("admitted", C.c_void_p),
        ("capacity", C.c_void_p), ("pool", C.c_void_p), ("min_margin", C.c_void_p),
        ("theta_curve", C.c_void_p), ("threshold", C.c_double),
    ]


class _AssembleArgs(C.Structure):
    _fields_ = [
        ("R", C.c_int), ("gamma_max", C.c_int),
        ("keep", C.c_void_p), ("anchor", C.c_void_p), ("tokens", C.c_void_p),
        ("flat_tokens", C.c_void_p), ("flat_request", C.c_void_p), ("flat_position", C.c_void_p),
        ("offsets", C.c_void_p),
    ]


class _VerifyArgs(C.Structure):
    _fields_ = [
        ("R", C.c_int), ("gamma_max", C.c_int), ("V", C.c_int), ("r", C.c_int), ("dtype", C.c_int),
        ("gamma", C.c_void_p), ("req_ids", C.c_void_p),
        ("target", C.c_void_p), ("U", C.c_void_p), ("E", C.c_void_p), ("W", C.c_void_p),
        ("anchor", C.c_void_p), ("tokens", C.c_void_p),
        ("draft_lse", C.c_void_p), ("draft_logit", C.c_void_p),
        ("keep", C.c_void_p), ("temperature", C.c_void_p),
        ("seed", C.c_uint64), ("round", C.c_uint64),
        ("bias_first", C.c_int), ("noise_block", C.c_int), ("a_rows", C.c_void_p),
        ("res_rel_eps", C.c_double),
        ("accepted", C.c_void_p), ("next_token", C.c_void_p), ("resampled", C.c_void_p),
        ("accept_margin", C.c_void_p), ("lse_t", C.c_void_p),
        ("gap1", C.c_void_p), ("gap2", C.c_void_p), ("rgap1", C.c_void_p), ("rgap2", C.c_void_p),
    ]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = C.CDLL(_LIB_PATH)
            L.dso_philox4x32_10.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p]
            L.dso_philox4x32_10.restype = None
            L.dso_uniform.argtypes = [C.c_uint64, C.c_uint64, C.c_uint32, C.c_uint32, C.c_uint32, C.c_uint32]
            L.dso_uniform.restype = C.c_double
            L.dso_sample_block.argtypes = [C.POINTER(_SampleArgs)]
            L.dso_sample_block.restype = C.c_int
            L.dso_schedule.argtypes = [C.POINTER(_ScheduleArgs)]
            L.dso_schedule.restype = C.c_int
            L.dso_verify.argtypes = [C.POINTER(_VerifyArgs)]
            L.dso_assemble.argtypes = [C.POINTER(_AssembleArgs)]
            L.dso_assemble.restype = C.c_int
            L.dso_verify.restype = C.c_int
            _lib = L
    return _lib


# ----------------------------------------------------------------- helpers

def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:  # raw bf16 bit patterns
        return BF16
    if a.dtype == np.float64:
        return F64
    raise TypeError("oracle tensors must be float32, float64 or uint16 (bf16 bits), got %s" % a.dtype)


def _c(a, dtype=None):
    a = np.ascontiguousarray(a if dtype is None else np.asarray(a, dtype=dtype))
    return a


def _p(a):
    return None if a is None else a.ctypes.data


def philox(ctr, key):
    """Philox4x32-10 of one 4-word counter and 2-word key."""
    c = np.asarray(ctr, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    out = np.zeros(4, dtype=np.uint32)
    lib().dso_philox4x32_10(c.ctypes.data, k.ctypes.data, out.ctypes.data)
    return out


def uniform(seed, rnd, purpose, req, pos, elem) -> float:
    return lib().dso_uniform(seed, rnd, purpose, req, pos, elem)


def _chunks(n, threads):
    threads = max(1, min(int(threads), n))
    bounds = np.linspace(0, n, threads + 1).astype(int)
    return [(int(bounds[i]), int(bounds[i + 1])) for i in range(threads) if bounds[i + 1] > bounds[i]]


def _run(fn, parts, threads):
    if threads <= 1 or len(parts) <= 1:
        return [fn(p) for p in parts]
    with ThreadPoolExecutor(max_workers=len(parts)) as ex:
        return list(ex.map(fn, parts))


# ----------------------------------------------------------------- sampler

def sample_block(U, E, W, h, w_h, w_e, b, temperature, anchor, seed, rnd, *, gamma=None,
                 req_ids=None, conf_token=0, bias_first=1, noise_block=128, forced_tokens=None,
                 sts_temp=None, head=HEAD_MARKOV, W_rnn=None, threads=1, logp=False):
    """Markov-head serial sampling, confidence head and survival products for R requests.

    U [R][G][V], E [V][r], W [r][V], h [R][G][d] share one element type
    (float32, float64 or uint16 bf16 bits). Returns a dict of numpy arrays; with logp=True
    also "logp" [R][G][V] float32, the draft distribution log p_d of every active position."""
    U, E, W, h = _c(U), _c(E), _c(W), _c(h)
    dt = _dtype_code(U)
    if not (_dtype_code(E) == dt and _dtype_code(W) == dt and _dtype_code(h) == dt):
        raise TypeError("U, E, W, h must share one element type")
    R, G, V = U.shape
    r = E.shape[1]
    d = h.shape[2]
    w_h, w_e = _c(w_h, np.float32), _c(w_e, np.float32)
    temperature, anchor = _c(temperature, np.float32), _c(anchor, np.int32)
    gamma = None if gamma is None else _c(gamma, np.int32)
    req_ids = np.arange(R, dtype=np.int32) if req_ids is None else _c(req_ids, np.int32)
    forced = None if forced_tokens is None else _c(forced_tokens, np.int32)
    sts = None if sts_temp is None else _c(sts_temp, np.float64)
    if head == HEAD_RNN:
        W_rnn = _c(W_rnn)
        if _dtype_code(W_rnn) != dt or W_rnn.shape != (3 * r, 2 * r + d):
            raise TypeError("W_rnn must be [3r][2r+d] of the inputs' element type")
    out = {
        "tokens": np.zeros((R, G), np.int32), "conf": np.zeros((R, G)), "surv": np.zeros((R, G)),
        "lse": np.zeros((R, G)), "logit": np.zeros((R, G)), "gap1": np.zeros((R, G)),
        "gap2": np.zeros((R, G)), "a_rows": np.zeros((R, G, r)),
    }
    if logp:
        out["logp"] = np.zeros((R, G, V), np.float32)

    def part(se):
        s, e = se
        a = _SampleArgs()
        a.R, a.gamma_max, a.V, a.r, a.d, a.dtype = e - s, G, V, r, d, dt
        a.gamma = _p(None if gamma is None else gamma[s:e])
        a.req_ids = _p(req_ids[s:e])
        a.U, a.E, a.W, a.h = _p(U[s:e]), _p(E), _p(W), _p(h[s:e])
        a.w_h, a.w_e, a.b = _p(w_h), _p(w_e), float(b)
        a.temperature, a.anchor = _p(temperature[s:e]), _p(anchor[s:e])
        a.seed, a.round = int(seed), int(rnd)
        a.conf_token, a.bias_first, a.noise_block = int(conf_token), int(bias_first), int(noise_block)
        a.forced_tokens = _p(None if forced is None else forced[s:e])
        a.sts_temp = _p(sts)
        a.head = int(head)
        a.W_rnn = _p(W_rnn if head == HEAD_RNN else None)
        for k, arr in out.items():
            setattr(a, k, _p(arr[s:e]))
        rc = lib().dso_sample_block(C.byref(a))
        if rc:
            raise RuntimeError("dso_sample_block failed: %d" % rc)

    _run(part, _chunks(R, threads), threads)
    return out


# ----------------------------------------------------------------- scheduler

def schedule(surv, sps, mode=SCHED_SYNC, *, gamma=None, surv_capacity=None, threshold=0.0):
    """Algorithm 1 over P independent problems. surv: [R][G] or [P][R][G] (any float),
    sps: [n_sps] with sps[B-1] = SPS(B). SCHED_THRESHOLD admits every candidate whose survival
    reaches `threshold`."""
    surv = np.asarray(surv, dtype=np.float64)
    squeeze = surv.ndim == 2
    if squeeze:
        surv = surv[None]
    surv = np.ascontiguousarray(surv)
    P, R, G = surv.shape
    sps = _c(sps, np.float64)
    if gamma is not None:
        gamma = np.ascontiguousarray(np.broadcast_to(np.asarray(gamma, dtype=np.int32), (P, R)))
    cap = None
    if surv_capacity is not None:
        cap = np.ascontiguousarray(np.broadcast_to(np.asarray(surv_capacity, dtype=np.float64), (P, R, G)))
    elif mode == SCHED_ASYNC_CAPACITY:
        raise ValueError("asynchronous capacity scheduling needs surv_capacity")
    out = {
        "keep": np.zeros((P, R), np.int32), "theta_best": np.zeros(P), "admitted": np.zeros(P, np.int32),
        "capacity": np.zeros(P, np.int32), "pool": np.zeros(P, np.int32), "min_margin": np.zeros(P),
        "theta_curve": np.zeros((P, R * G + 1)),
    }
    a = _ScheduleArgs()
    a.P, a.R, a.gamma_max = P, R, G
    a.gamma, a.surv, a.surv_capacity = _p(gamma), _p(surv), _p(cap)
    a.sps, a.n_sps, a.mode = _p(sps), int(sps.shape[0]), int(mode)
    a.threshold = float(threshold)
    for k, arr in out.items():
        setattr(a, k, _p(arr))
    rc = lib().dso_schedule(C.byref(a))
    if rc:
        raise RuntimeError("dso_schedule failed: %d" % rc)
    if squeeze:
        out = {k: v[0] for k, v in out.items()}
    return out


# ----------------------------------------------------------------- verifier

def verify(target, U, E, W, anchor, tokens, draft_lse, draft_logit, keep, temperature, seed, rnd, *,
           gamma=None, req_ids=None, bias_first=1, noise_block=128, a_rows=None, threads=1, res_rel_eps=0.0):
    """Rejection-sampling verification of the admitted prefixes of R requests.

    res_rel_eps: the relative error of the probabilities assumed by the residual draw's robust
    margins rgap1 / rgap2 (equal to gap1 / gap2 when 0)."""
    target, U, E, W = _c(target), _c(U), _c(E), _c(W)
    dt = _dtype_code(U)
    if not (_dtype_code(target) == dt and _dtype_code(E) == dt and _dtype_code(W) == dt):
        raise TypeError("target, U, E, W must share one element type")
    R, G, V = U.shape
    r = E.shape[1]
    anchor, tokens, keep = _c(anchor, np.int32), _c(tokens, np.int32), _c(keep, np.int32)
    draft_lse, draft_logit = _c(draft_lse, np.float64), _c(draft_logit, np.float64)
    temperature = _c(temperature, np.float32)
    gamma = None if gamma is None else _c(gamma, np.int32)
    req_ids = np.arange(R, dtype=np.int32) if req_ids is None else _c(req_ids, np.int32)
    arows = None if a_rows is None else _c(a_rows, np.float64)
    out = {
        "accepted": np.zeros(R, np.int32), "next_token": np.zeros(R, np.int32),
        "resampled": np.zeros(R, np.int32), "accept_margin": np.zeros((R, G)),
        "lse_t": np.zeros((R, G + 1)), "gap1": np.zeros(R), "gap2": np.zeros(R),
        "rgap1": np.zeros(R), "rgap2": np.zeros(R),
    }

    def part(se):
        s, e = se
        a = _VerifyArgs()
        a.R, a.gamma_max, a.V, a.r, a.dtype = e - s, G, V, r, dt
        a.gamma = _p(None if gamma is None else gamma[s:e])
        a.req_ids = _p(req_ids[s:e])
        a.target, a.U, a.E, a.W = _p(target[s:e]), _p(U[s:e]), _p(E), _p(W)
        a.anchor, a.tokens = _p(anchor[s:e]), _p(tokens[s:e])
        a.draft_lse, a.draft_logit = _p(draft_lse[s:e]), _p(draft_logit[s:e])
        a.keep, a.temperature = _p(keep[s:e]), _p(temperature[s:e])
        a.seed, a.round = int(seed), int(rnd)
        a.bias_first, a.noise_block = int(bias_first), int(noise_block)
        a.a_rows = _p(None if arows is None else arows[s:e])
        a.res_rel_eps = float(res_rel_eps)
        for k, arr in out.items():
            setattr(a, k, _p(arr[s:e]))
        rc = lib().dso_verify(C.byref(a))
        if rc:
            raise RuntimeError("dso_verify failed: %d" % rc)

    _run(part, _chunks(R, threads), threads)
    return out


# ----------------------------------------------------------------- ragged verify batch

def assemble(keep, anchor, tokens):
    """Flatten the admitted prefixes: per request its anchor, then keep[r] draft tokens."""
    keep, anchor, tokens = _c(keep, np.int32), _c(anchor, np.int32), _c(tokens, np.int32)
    R, G = tokens.shape
    cap = R * (G + 1)
    out = {"flat_tokens": np.zeros(cap, np.int32), "flat_request": np.zeros(cap, np.int32),
           "flat_position": np.zeros(cap, np.int32), "offsets": np.zeros(R + 1, np.int32)}
    a = _AssembleArgs()
    a.R, a.gamma_max = R, G
    a.keep, a.anchor, a.tokens = _p(keep), _p(anchor), _p(tokens)
    for k, arr in out.items():
        setattr(a, k, _p(arr))
    rc = lib().dso_assemble(C.byref(a))
    if rc:
        raise ValueError("dso_assemble: keep outside [0, gamma_max]")
    return out
