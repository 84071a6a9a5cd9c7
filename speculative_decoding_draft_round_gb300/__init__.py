"""Python binding of libdspark, the GB300 hot path of one DSpark draft round.

The binding only marshals arguments: it checks tensor devices, dtypes and
shapes, allocates output tensors and workspaces with torch, and passes raw
device pointers and the current CUDA stream to the C ABI in
``include/dspark.h``. Every step of the round runs in the library's CUDA
kernels; there is no CPU or PyTorch fallback, and a missing library raises.

Calls (same names as the C ABI):
  sample_block  Markov-head serial sampling, confidence head, survival products
  schedule      hardware-aware prefix scheduler (sync / async capacity / full scan)
  verify        rejection-sampling verification, residual or bonus token
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdspark.so")

F32, BF16 = 0, 1
SCHED_SYNC, SCHED_ASYNC_CAPACITY, SCHED_FULL_SCAN, SCHED_THRESHOLD = 0, 1, 2, 3
PATH_AUTO, PATH_CUDA_CORE, PATH_TENSOR_CORE, PATH_RESIDENT = 0, 1, 2, 3
HEAD_MARKOV, HEAD_RNN = 0, 1
NOISE_BLOCK = 128
MAX_GAMMA = 32
MAX_SLOTS = 8192

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported shape", 3: "workspace", 4: "CUDA error",
          5: "timeout", 6: "out-of-range device input", 7: "non-finite input"}
ERR_TIMEOUT, ERR_DEVICE_INPUT, ERR_NONFINITE_INPUT = 5, 6, 7

_vp = C.c_void_p


class SampleArgs(C.Structure):
    _fields_ = [
        ("struct_size", C.c_uint32), ("R", C.c_int32), ("gamma_max", C.c_int32), ("V", C.c_int32),
        ("r", C.c_int32), ("d", C.c_int32), ("dtype", C.c_int32), ("conf_token", C.c_int32),
        ("bias_first", C.c_int32), ("path", C.c_int32),
        ("gamma", _vp), ("U", _vp), ("E", _vp), ("W", _vp), ("h", _vp), ("w_h", _vp), ("w_e", _vp),
        ("b", C.c_float), ("temperature", _vp), ("anchor", _vp),
        ("seed", C.c_uint64), ("round", C.c_uint64),
        ("tokens", _vp), ("conf", _vp), ("surv", _vp), ("draft_lse", _vp), ("draft_logit", _vp),
        ("sts_temp", _vp), ("head", C.c_int32), ("W_rnn", _vp), ("a_rows", _vp), ("step_ready", _vp),
    ]


class ScheduleStats(C.Structure):
    _fields_ = [("theta_best", C.c_double), ("admitted", C.c_int32), ("capacity", C.c_int32),
                ("batch", C.c_int32), ("pool", C.c_int32)]


class ScheduleArgs(C.Structure):
    _fields_ = [
        ("struct_size", C.c_uint32), ("R", C.c_int32), ("gamma_max", C.c_int32), ("mode", C.c_int32),
        ("n_sps", C.c_int32),
        ("gamma", _vp), ("surv", _vp), ("surv_capacity", _vp), ("sps", _vp), ("keep", _vp), ("stats", _vp),
        ("threshold", C.c_float),
    ]


class VerifyArgs(C.Structure):
    _fields_ = [
        ("struct_size", C.c_uint32), ("R", C.c_int32), ("gamma_max", C.c_int32), ("V", C.c_int32),
        ("r", C.c_int32), ("dtype", C.c_int32), ("bias_first", C.c_int32), ("path", C.c_int32),
        ("gamma", _vp), ("target", _vp), ("U", _vp), ("E", _vp), ("W", _vp), ("anchor", _vp), ("tokens", _vp),
        ("draft_lse", _vp), ("draft_logit", _vp), ("keep", _vp), ("temperature", _vp),
        ("seed", C.c_uint64), ("round", C.c_uint64),
        ("accepted", _vp), ("next_token", _vp), ("resampled", _vp), ("a_rows", _vp),
    ]


class AssembleArgs(C.Structure):
    _fields_ = [
        ("struct_size", C.c_uint32), ("R", C.c_int32), ("gamma_max", C.c_int32),
        ("keep", _vp), ("anchor", _vp), ("tokens", _vp),
        ("flat_tokens", _vp), ("flat_request", _vp), ("flat_position", _vp), ("offsets", _vp),
    ]


EXPORTS = ("dspark_sample_workspace_size", "dspark_sample_block", "dspark_schedule_workspace_size",
           "dspark_schedule", "dspark_verify_workspace_size", "dspark_verify", "dspark_check",
           "dspark_status_string", "dspark_abi_version", "dspark_launch_count", "dspark_time_kernel",
           "dspark_last_error", "dspark_sample_path", "dspark_sample_block_static", "dspark_check_static",
           "dspark_set_wait_limit",
           "dspark_assemble_workspace_size", "dspark_assemble")

KERNELS = {"draft_setup": 0, "draft_stats": 1, "draft_commit": 2, "schedule": 3, "verify_rows": 4,
           "verify_decide": 5, "residual_stats": 6, "residual_pick": 7, "assemble": 8, "rnn_step": 9,
           "rnn_hidden": 10, "draft_loop": 11}


class EventPair(C.Structure):
    _fields_ = [("start", C.c_void_p), ("stop", C.c_void_p)]

_lib = None


class DsparkError(RuntimeError):
    def __init__(self, fn, code, detail=""):
        msg = "%s failed: %s (%d)" % (fn, STATUS.get(code, "unknown"), code)
        if detail:
            msg += ": " + detail
        super().__init__(msg)
        self.code = code


def lib():
    """Load libdspark.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libdspark.so is missing: build it with __graft_entry__.build() "
                               "or python -m speculative_decoding_draft_round_gb300.build")
        L = C.CDLL(LIB_PATH)
        for name, argt in (("dspark_sample_workspace_size", [C.POINTER(SampleArgs), C.POINTER(C.c_size_t)]),
                           ("dspark_sample_block", [C.POINTER(SampleArgs), _vp, C.c_size_t, _vp]),
                           ("dspark_schedule_workspace_size", [C.POINTER(ScheduleArgs), C.POINTER(C.c_size_t)]),
                           ("dspark_schedule", [C.POINTER(ScheduleArgs), _vp, C.c_size_t, _vp]),
                           ("dspark_verify_workspace_size", [C.POINTER(VerifyArgs), C.POINTER(C.c_size_t)]),
                           ("dspark_verify", [C.POINTER(VerifyArgs), _vp, C.c_size_t, _vp]),
                           ("dspark_assemble_workspace_size", [C.POINTER(AssembleArgs), C.POINTER(C.c_size_t)]),
                           ("dspark_assemble", [C.POINTER(AssembleArgs), _vp, C.c_size_t, _vp]),
                           ("dspark_check", [_vp, _vp])):
            f = getattr(L, name)
            f.argtypes = argt
            f.restype = C.c_int32
        L.dspark_status_string.argtypes = [C.c_int32]
        L.dspark_status_string.restype = C.c_char_p
        L.dspark_abi_version.argtypes = []
        L.dspark_abi_version.restype = C.c_int32
        L.dspark_sample_block_static.argtypes = [C.POINTER(SampleArgs), _vp]
        L.dspark_sample_block_static.restype = C.c_int32
        L.dspark_check_static.argtypes = [_vp]
        L.dspark_check_static.restype = C.c_int32
        L.dspark_set_wait_limit.argtypes = [C.c_uint64]
        L.dspark_set_wait_limit.restype = C.c_uint64
        L.dspark_sample_path.argtypes = [C.POINTER(SampleArgs)]
        L.dspark_sample_path.restype = C.c_int32
        L.dspark_last_error.argtypes = []
        L.dspark_last_error.restype = C.c_char_p
        L.dspark_launch_count.argtypes = []
        L.dspark_launch_count.restype = C.c_uint64
        L.dspark_time_kernel.argtypes = [C.c_int32, C.c_void_p, C.c_int32, C.POINTER(C.c_int32)]
        L.dspark_time_kernel.restype = C.c_int32
        _lib = L
    return _lib


# ----------------------------------------------------------------- marshalling helpers

def _ptr(t):
    return None if t is None else t.data_ptr()


def _dev(t, name, dtype=None, shape=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    return t


def _dtype_code(t):
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError("tensor dtype must be float32 or bfloat16, got %s" % t.dtype)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _call(fn, *args):
    rc = getattr(lib(), fn)(*args)
    if rc != 0:
        detail = lib().dspark_last_error().decode() if rc == 4 else ""
        raise DsparkError(fn, rc, detail)


def _workspace(fn_size, args, workspace, device):
    n = C.c_size_t(0)
    _call(fn_size, C.byref(args), C.byref(n))
    if workspace is None:
        workspace = torch.zeros(n.value, dtype=torch.uint8, device=device)
    elif workspace.numel() < n.value:
        raise ValueError("workspace has %d bytes, needs %d" % (workspace.numel(), n.value))
    return workspace


def workspace_bytes(kind: str, args) -> int:
    n = C.c_size_t(0)
    _call("dspark_%s_workspace_size" % kind, C.byref(args), C.byref(n))
    return n.value


def sample_path(args) -> int:
    """PATH_CUDA_CORE or PATH_TENSOR_CORE: the contraction path dspark_sample_block takes for `args`."""
    p = int(lib().dspark_sample_path(C.byref(args)))
    if p < 0:
        raise DsparkError("dspark_sample_path", -p)
    return p


def launch_count() -> int:
    """Kernels launched by libdspark in this process."""
    return int(lib().dspark_launch_count())


class KernelTimer:
    """Records CUDA events around every launch of one kernel family (dspark_time_kernel)."""

    def __init__(self, kernel: str, capacity: int):
        self.kernel = KERNELS[kernel]
        self.events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(capacity)]
        # torch creates the underlying cudaEvent_t on first record: record once so the handles exist
        for a, b in self.events:
            a.record()
            b.record()
        torch.cuda.synchronize()
        self.pairs = (EventPair * capacity)()
        for i, (a, b) in enumerate(self.events):
            self.pairs[i].start = a.cuda_event
            self.pairs[i].stop = b.cuda_event
        self.count = C.c_int32(0)

    def __enter__(self):
        rc = lib().dspark_time_kernel(self.kernel, self.pairs, len(self.events), C.byref(self.count))
        if rc:
            raise DsparkError("dspark_time_kernel", rc)
        return self

    def __exit__(self, *exc):
        lib().dspark_time_kernel(-1, None, 0, None)

    def durations_ms(self):
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in self.events[: self.count.value]]


def check(workspace, stream=None) -> int:
    """Synchronise the stream and return (and clear) the workspace's device status word."""
    return lib().dspark_check(_ptr(workspace), _stream(stream))


# ----------------------------------------------------------------- calls

def sample_args(U, E, W, h, w_h, w_e, b, temperature, anchor, seed, rnd, *, gamma=None, conf_token=0,
                bias_first=1, path=PATH_AUTO, out=None, sts_temp=None, head=HEAD_MARKOV, W_rnn=None,
                a_rows=False):
    R, G, V = U.shape
    r = E.shape[1]
    d = h.shape[2]
    dt = U.dtype
    _dev(U, "U", dt)
    _dev(E, "E", dt, (V, r))
    _dev(W, "W", dt, (r, V))
    _dev(h, "h", dt, (R, G, d))
    _dev(w_h, "w_h", torch.float32, (d,))
    _dev(w_e, "w_e", torch.float32, (r,))
    _dev(temperature, "temperature", torch.float32, (R,))
    _dev(anchor, "anchor", torch.int32, (R,))
    _dev(gamma, "gamma", torch.int32, (R,))
    _dev(sts_temp, "sts_temp", torch.float32, (G,))
    if head == HEAD_RNN:
        _dev(W_rnn, "W_rnn", dt, (3 * r, 2 * r + d))
    dev = U.device
    if out is None:
        out = {"tokens": torch.empty((R, G), dtype=torch.int32, device=dev)}
        for k in ("conf", "surv", "draft_lse", "draft_logit"):
            out[k] = torch.empty((R, G), dtype=torch.float32, device=dev)
        if a_rows:
            out["a_rows"] = torch.empty((R, G, r), dtype=torch.float32, device=dev)
    a = SampleArgs()
    a.struct_size = C.sizeof(SampleArgs)
    a.R, a.gamma_max, a.V, a.r, a.d = R, G, V, r, d
    a.dtype = _dtype_code(U)
    a.conf_token, a.bias_first, a.path = int(conf_token), int(bias_first), int(path)
    a.gamma, a.U, a.E, a.W, a.h = _ptr(gamma), _ptr(U), _ptr(E), _ptr(W), _ptr(h)
    a.w_h, a.w_e, a.b = _ptr(w_h), _ptr(w_e), float(b)
    a.temperature, a.anchor = _ptr(temperature), _ptr(anchor)
    a.seed, a.round = int(seed), int(rnd)
    a.tokens, a.conf, a.surv = _ptr(out["tokens"]), _ptr(out["conf"]), _ptr(out["surv"])
    a.draft_lse, a.draft_logit = _ptr(out["draft_lse"]), _ptr(out["draft_logit"])
    a.sts_temp = _ptr(sts_temp)
    a.head = int(head)
    a.W_rnn = _ptr(W_rnn if head == HEAD_RNN else None)
    a.a_rows = _ptr(out.get("a_rows"))
    return a, out


def sample_block(U, E, W, h, w_h, w_e, b, temperature, anchor, seed, rnd, *, gamma=None, conf_token=0,
                 bias_first=1, path=PATH_AUTO, out=None, workspace=None, stream=None, sts_temp=None,
                 head=HEAD_MARKOV, W_rnn=None, a_rows=False):
    """dspark_sample_block on the current (or given) stream; returns the output tensors (with
    a_rows=True also each step's bias operand, which dspark_verify needs for an RNN-head draft)."""
    a, out = sample_args(U, E, W, h, w_h, w_e, b, temperature, anchor, seed, rnd, gamma=gamma,
                         conf_token=conf_token, bias_first=bias_first, path=path, out=out, sts_temp=sts_temp,
                         head=head, W_rnn=W_rnn, a_rows=a_rows)
    ws = _workspace("dspark_sample_workspace_size", a, workspace, U.device)
    _call("dspark_sample_block", C.byref(a), _ptr(ws), ws.numel(), _stream(stream))
    out["workspace"] = ws
    return out


STATIC_WORKSPACE_BYTES = 8 << 20


def sample_block_static(U, E, W, h, w_h, w_e, b, temperature, anchor, seed, rnd, *, gamma=None, conf_token=0,
                        bias_first=1, path=PATH_AUTO, out=None, stream=None, sts_temp=None, head=HEAD_MARKOV,
                        W_rnn=None):
    """dspark_sample_block_static: the sampler with its scratch in the library's static device
    array (for callers that cannot allocate device memory). Only the output tensors are
    allocated here, by torch, when `out` is not given. Shapes whose scratch exceeds the array
    are refused."""
    a, out = sample_args(U, E, W, h, w_h, w_e, b, temperature, anchor, seed, rnd, gamma=gamma,
                         conf_token=conf_token, bias_first=bias_first, path=path, out=out, sts_temp=sts_temp,
                         head=head, W_rnn=W_rnn)
    _call("dspark_sample_block_static", C.byref(a), _stream(stream))
    return out


def set_wait_limit(ns: int) -> int:
    """Bound (ns) of every device-side wait of the calls made after this one (0: the default of
    4 s); returns the previous bound. A wait that runs out records ERR_TIMEOUT (for tests)."""
    return int(lib().dspark_set_wait_limit(int(ns)))


def check_static(stream=None) -> int:
    """Synchronise the stream and return (and clear) the status word of the static array that
    sample_block_static uses on the current device."""
    return lib().dspark_check_static(_stream(stream))


def schedule_args(surv, sps, mode=SCHED_SYNC, *, gamma=None, surv_capacity=None, out=None, threshold=0.0):
    R, G = surv.shape
    _dev(surv, "surv", torch.float32)
    _dev(sps, "sps", torch.float32)
    _dev(gamma, "gamma", torch.int32, (R,))
    _dev(surv_capacity, "surv_capacity", torch.float32, (R, G))
    dev = surv.device
    if out is None:
        out = {"keep": torch.empty(R, dtype=torch.int32, device=dev),
               "stats": torch.empty(C.sizeof(ScheduleStats), dtype=torch.uint8, device=dev)}
    a = ScheduleArgs()
    a.struct_size = C.sizeof(ScheduleArgs)
    a.R, a.gamma_max, a.mode, a.n_sps = R, G, int(mode), int(sps.numel())
    a.gamma, a.surv, a.surv_capacity, a.sps = _ptr(gamma), _ptr(surv), _ptr(surv_capacity), _ptr(sps)
    a.keep, a.stats = _ptr(out["keep"]), _ptr(out["stats"])
    a.threshold = float(threshold)
    return a, out


def schedule(surv, sps, mode=SCHED_SYNC, *, gamma=None, surv_capacity=None, out=None, workspace=None,
             stream=None, threshold=0.0):
    """dspark_schedule; returns {"keep": [R] int32, "stats": raw device bytes of dspark_schedule_stats}.
    SCHED_THRESHOLD admits every candidate whose survival reaches `threshold`."""
    a, out = schedule_args(surv, sps, mode, gamma=gamma, surv_capacity=surv_capacity, out=out,
                           threshold=threshold)
    ws = _workspace("dspark_schedule_workspace_size", a, workspace, surv.device)
    _call("dspark_schedule", C.byref(a), _ptr(ws), ws.numel(), _stream(stream))
    out["workspace"] = ws
    return out


def assemble_args(keep, anchor, tokens, out=None):
    R, G = tokens.shape
    _dev(keep, "keep", torch.int32, (R,))
    _dev(anchor, "anchor", torch.int32, (R,))
    _dev(tokens, "tokens", torch.int32, (R, G))
    dev = tokens.device
    if out is None:
        n = R * (G + 1)
        out = {k: torch.empty(n, dtype=torch.int32, device=dev)
               for k in ("flat_tokens", "flat_request", "flat_position")}
        out["offsets"] = torch.empty(R + 1, dtype=torch.int32, device=dev)
    a = AssembleArgs()
    a.struct_size = C.sizeof(AssembleArgs)
    a.R, a.gamma_max = R, G
    a.keep, a.anchor, a.tokens = _ptr(keep), _ptr(anchor), _ptr(tokens)
    a.flat_tokens, a.flat_request = _ptr(out["flat_tokens"]), _ptr(out["flat_request"])
    a.flat_position, a.offsets = _ptr(out["flat_position"]), _ptr(out["offsets"])
    return a, out


def assemble(keep, anchor, tokens, *, out=None, workspace=None, stream=None):
    """dspark_assemble: the admitted prefixes as one flat token stream with request ids, causal
    positions and per-request offsets (entries past offsets[R] are -1)."""
    a, out = assemble_args(keep, anchor, tokens, out=out)
    ws = _workspace("dspark_assemble_workspace_size", a, workspace, tokens.device)
    _call("dspark_assemble", C.byref(a), _ptr(ws), ws.numel(), _stream(stream))
    out["workspace"] = ws
    return out


def decode_stats(stats_bytes) -> dict:
    """Host copy of a dspark_schedule_stats device struct."""
    raw = bytes(stats_bytes.cpu().numpy().tobytes())
    s = ScheduleStats.from_buffer_copy(raw)
    return {"theta_best": s.theta_best, "admitted": s.admitted, "capacity": s.capacity, "batch": s.batch,
            "pool": s.pool}


def verify_args(target, U, E, W, anchor, tokens, draft_lse, draft_logit, keep, temperature, seed, rnd, *,
                gamma=None, bias_first=1, path=PATH_AUTO, out=None, a_rows=None):
    R, G, V = U.shape
    r = E.shape[1]
    dt = U.dtype
    _dev(target, "target", dt, (R, G + 1, V))
    _dev(U, "U", dt)
    _dev(E, "E", dt, (V, r))
    _dev(W, "W", dt, (r, V))
    _dev(anchor, "anchor", torch.int32, (R,))
    _dev(tokens, "tokens", torch.int32, (R, G))
    _dev(draft_lse, "draft_lse", torch.float32, (R, G))
    _dev(draft_logit, "draft_logit", torch.float32, (R, G))
    _dev(keep, "keep", torch.int32, (R,))
    _dev(temperature, "temperature", torch.float32, (R,))
    _dev(gamma, "gamma", torch.int32, (R,))
    _dev(a_rows, "a_rows", torch.float32, (R, G, r))
    dev = U.device
    if out is None:
        out = {"accepted": torch.empty(R, dtype=torch.int32, device=dev),
               "next_token": torch.empty(R, dtype=torch.int32, device=dev),
               "resampled": torch.empty(R, dtype=torch.uint8, device=dev)}
    a = VerifyArgs()
    a.struct_size = C.sizeof(VerifyArgs)
    a.R, a.gamma_max, a.V, a.r = R, G, V, r
    a.dtype, a.bias_first, a.path = _dtype_code(U), int(bias_first), int(path)
    a.gamma, a.target, a.U, a.E, a.W = _ptr(gamma), _ptr(target), _ptr(U), _ptr(E), _ptr(W)
    a.anchor, a.tokens, a.draft_lse, a.draft_logit = _ptr(anchor), _ptr(tokens), _ptr(draft_lse), _ptr(draft_logit)
    a.keep, a.temperature = _ptr(keep), _ptr(temperature)
    a.seed, a.round = int(seed), int(rnd)
    a.accepted, a.next_token, a.resampled = _ptr(out["accepted"]), _ptr(out["next_token"]), _ptr(out["resampled"])
    a.a_rows = _ptr(a_rows)
    return a, out


def verify(target, U, E, W, anchor, tokens, draft_lse, draft_logit, keep, temperature, seed, rnd, *,
           gamma=None, bias_first=1, path=PATH_AUTO, out=None, workspace=None, stream=None, a_rows=None):
    """dspark_verify; returns accepted lengths, next tokens and residual flags (a_rows: the
    sampler's bias operands, needed for an RNN-head draft)."""
    a, out = verify_args(target, U, E, W, anchor, tokens, draft_lse, draft_logit, keep, temperature, seed, rnd,
                         gamma=gamma, bias_first=bias_first, path=path, out=out, a_rows=a_rows)
    ws = _workspace("dspark_verify_workspace_size", a, workspace, U.device)
    _call("dspark_verify", C.byref(a), _ptr(ws), ws.numel(), _stream(stream))
    out["workspace"] = ws
    return out


class RoundRunner:
    """Runs sample_block -> schedule -> verify for one workload with persistent
    argument structs, outputs and workspaces (the launch sequence a serving
    loop would replay every round). path selects the sampler's contraction path; the verifier
    has no resident loop and takes the per-step tensor-core kernels for PATH_RESIDENT."""

    def __init__(self, rnd, *, path=PATH_AUTO, surv_capacity=None, device=None):
        self.rnd = rnd
        self.path = path
        dev = device or rnd.U.device
        self.sa, self.sout = sample_args(rnd.U, rnd.E, rnd.W, rnd.h, rnd.w_h, rnd.w_e, rnd.b, rnd.temperature,
                                         rnd.anchor, rnd.seed, rnd.round, gamma=rnd.gamma,
                                         conf_token=rnd.conf_token, bias_first=rnd.bias_first, path=path)
        self.sws = torch.zeros(workspace_bytes("sample", self.sa), dtype=torch.uint8, device=dev)
        self.surv_capacity = surv_capacity
        self.ca, self.cout = schedule_args(self.sout["surv"], rnd.sps, rnd.mode, gamma=rnd.gamma,
                                           surv_capacity=surv_capacity)
        self.cws = torch.zeros(workspace_bytes("schedule", self.ca), dtype=torch.uint8, device=dev)
        self.va, self.vout = verify_args(rnd.target, rnd.U, rnd.E, rnd.W, rnd.anchor, self.sout["tokens"],
                                         self.sout["draft_lse"], self.sout["draft_logit"], self.cout["keep"],
                                         rnd.temperature, rnd.seed, rnd.round, gamma=rnd.gamma,
                                         bias_first=rnd.bias_first,
                                         path=PATH_TENSOR_CORE if path == PATH_RESIDENT else path)
        self.vws = torch.zeros(workspace_bytes("verify", self.va), dtype=torch.uint8, device=dev)

    def set_round(self, rnd_index: int):
        self.sa.round = int(rnd_index)
        self.va.round = int(rnd_index)

    def run(self, stream=None):
        self.run_draft(stream)
        self.run_verify(stream)

    def run_draft(self, stream=None, step_ready=None):
        """The sampler and the scheduler: keep is known (on the device) when these have run.
        step_ready: optional list of gamma_max torch.cuda.Event; step k's kernels wait for
        step_ready[k] (for inputs still being copied in)."""
        s = _stream(stream)
        if step_ready is not None:
            handles = (C.c_void_p * len(step_ready))(*[ev.cuda_event for ev in step_ready])
            self.sa.step_ready = C.cast(handles, C.c_void_p)
        try:
            _call("dspark_sample_block", C.byref(self.sa), _ptr(self.sws), self.sws.numel(), s)
        finally:
            self.sa.step_ready = None
        _call("dspark_schedule", C.byref(self.ca), _ptr(self.cws), self.cws.numel(), s)

    def run_verify(self, stream=None):
        _call("dspark_verify", C.byref(self.va), _ptr(self.vws), self.vws.numel(), _stream(stream))

    def check(self, stream=None) -> int:
        codes = [check(w, stream) for w in (self.sws, self.cws, self.vws)]
        return next((c for c in codes if c), 0)

    def results(self) -> dict:
        out = dict(self.sout)
        out.update(self.cout)
        out.update(self.vout)
        return out
