"""Helpers shared by the GPU parity tests: move workload tensors to numpy for
the oracle and compare the CUDA results with the oracle stage by stage.

Stage-wise parity feeds each oracle stage the GPU's own upstream outputs
(draft tokens for the sampler's later positions, GPU survivals for the
scheduler, GPU tokens / log-normalisers / keep lengths for the verifier).
Integer decisions must then agree exactly, except where the oracle's own
floating-point margin is below the stated tolerance:
  - a draw whose top-two perturbed values (block level or element level)
    differ by < 1e-4 ("draw");
  - an accept test with |log u - log(p_t/p_d)| < 1e-4 ("accept");
  - a scheduler decision whose relative Theta margin is <= 1e-12 ("theta");
  - a residual draw whose oracle margin is >= 1e-4 but which another candidate
    could win when every probability carries the relative error RES_REL_EPS of
    the GPU's fp32 residual ("residual_fp32"; derived beside RES_REL_EPS).
Excusals are counted per kind, returned as a dict and printed by the tests."""
from __future__ import annotations

import numpy as np
import torch

import oracle

TOK_TOL = 1e-4      # top-two gap below which a draw is excused
ACC_TOL = 1e-4      # accept-test margin below which a decision is excused
THETA_TOL = 1e-12   # relative Theta margin below which a scheduler decision is excused
CONF_TOL = 1e-5     # c_k and a_k, absolute
LSE_TOL = 1e-5      # log-normalisers and logits, relative to max(1, |value|)
ROW_TOL = 1e-5      # bias operand rows (W_1 rows, or tanh outputs of the RNN head), absolute
# Relative error of each probability p_t(v), p_d(v) in the GPU's fp32 residual max(0, p_t - p_d):
# each is 2^(z*s - L) with L an fp32 log-normaliser in log2 units (draft_lse from the sampler,
# lse_t from the verify rows) and z = U + B or the target logit rounded to fp32. For magnitudes
# below 128 each of these three fp32 roundings is at most 2^-18 (half an ulp), the exponential
# adds 2^-22, so the relative error is below ln 2 * 3 * 2^-18 + 2^-21 = 8.4e-6.
RES_REL_EPS = 1e-5


def new_counts():
    return {"draw": 0, "accept": 0, "theta": 0, "residual_fp32": 0, "checked_tokens": 0, "checked_requests": 0}


def add_counts(total, part):
    for k, v in part.items():
        total[k] = total.get(k, 0) + v
    return total


def report(label, counts):
    """Print one line of excusal counts (pytest -s or the captured output of a failure)."""
    print("parity %s: %s" % (label, " ".join("%s=%d" % kv for kv in sorted(counts.items()))), flush=True)


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def rows(t: torch.Tensor, ids) -> np.ndarray:
    idx = torch.as_tensor(np.asarray(ids), dtype=torch.long, device=t.device)
    return to_np(t.index_select(0, idx))


def _threads():
    import os
    return max(1, min(16, os.cpu_count() or 1))


def check_sample(rnd, out, ids, threads=None, sts_temp=None, head=0, W_rnn=None):
    """Compare dspark_sample_block outputs with the oracle on requests `ids` (sts_temp: the
    per-position confidence temperatures the call was given, if any). Returns the excusal
    counts."""
    threads = threads or _threads()
    ids = np.asarray(ids)
    tok = to_np(out["tokens"])[ids]
    gamma = None if rnd.gamma is None else to_np(rnd.gamma)[ids]
    o = oracle.sample_block(rows(rnd.U, ids), to_np(rnd.E), to_np(rnd.W), rows(rnd.h, ids), to_np(rnd.w_h),
                            to_np(rnd.w_e), rnd.b, to_np(rnd.temperature)[ids], to_np(rnd.anchor)[ids],
                            rnd.seed, rnd.round, gamma=gamma, req_ids=ids, conf_token=rnd.conf_token,
                            bias_first=rnd.bias_first, forced_tokens=np.where(tok < 0, 0, tok),
                            sts_temp=None if sts_temp is None else to_np(sts_temp).astype(np.float64),
                            head=head, W_rnn=None if W_rnn is None else to_np(W_rnn), threads=threads)
    if "a_rows" in out:   # the bias operand of each step
        g_rows = to_np(out["a_rows"])[ids].astype(np.float64)
        np.testing.assert_allclose(g_rows, o["a_rows"], rtol=0, atol=ROW_TOL)
    G = rnd.gamma_max
    g = np.full(len(ids), G) if gamma is None else gamma
    active = np.arange(G)[None, :] < g[:, None]
    assert np.all(tok[~active] == -1)
    mism = (tok != o["tokens"]) & active
    excused = mism & ((o["gap1"] < TOK_TOL) | (o["gap2"] < TOK_TOL))
    bad = mism & ~excused
    assert not bad.any(), "token mismatch at %s (gpu %s oracle %s gaps %s %s)" % (
        np.argwhere(bad)[:5].tolist(), tok[bad][:5], o["tokens"][bad][:5], o["gap1"][bad][:5], o["gap2"][bad][:5])
    for key, okey, tol, rel in (("conf", "conf", CONF_TOL, False), ("surv", "surv", CONF_TOL, False),
                                ("draft_lse", "lse", LSE_TOL, True), ("draft_logit", "logit", LSE_TOL, True)):
        g_ = to_np(out[key])[ids].astype(np.float64)
        err = np.abs(g_ - o[okey])
        lim = tol * (np.maximum(1.0, np.abs(o[okey])) if rel else 1.0)
        worst = np.max(np.where(active, err - lim, -1.0))
        assert worst <= 0, "%s differs by %.3g (limit %.3g)" % (key, np.max(np.where(active, err, 0)), tol)
    c = new_counts()
    c["draw"] = int(excused.sum())
    c["checked_tokens"] = int(active.sum())
    c["checked_requests"] = len(ids)
    return c


def check_schedule(surv, sps, mode, out, *, gamma=None, surv_capacity=None):
    """Compare dspark_schedule on GPU survivals with the oracle. Returns the excusal counts
    (theta = 1 when the oracle's own Theta margin lies inside the tie band, so that the
    decision is not compared; the stats that do not depend on it still are)."""
    import speculative_decoding_draft_round_gb300 as ds
    s = to_np(surv).astype(np.float64)
    gam = None if gamma is None else to_np(gamma)
    cap = None if surv_capacity is None else to_np(surv_capacity).astype(np.float64)
    o = oracle.schedule(s, to_np(sps).astype(np.float64), mode, gamma=gam, surv_capacity=cap)
    keep = to_np(out["keep"])
    st = ds.decode_stats(out["stats"])
    c = new_counts()
    assert st["pool"] == int(o["pool"])
    if o["min_margin"] <= THETA_TOL:
        c["theta"] = 1
        return c
    assert keep.tolist() == o["keep"].tolist(), "keep differs: gpu %s oracle %s" % (
        keep[keep != o["keep"]][:8], o["keep"][keep != o["keep"]][:8])
    assert st["admitted"] == int(o["admitted"])
    assert st["pool"] == int(o["pool"])
    assert st["batch"] == s.shape[0] + int(o["admitted"])
    assert st["capacity"] == int(o["capacity"])
    assert abs(st["theta_best"] - o["theta_best"]) <= 1e-9 * abs(o["theta_best"])
    return c


def check_verify(rnd, sout, keep, vout, ids, threads=None, a_rows=None):
    """Compare dspark_verify with the oracle on requests `ids`, fed the GPU's draft outputs.
    Returns the excusal counts."""
    threads = threads or _threads()
    ids = np.asarray(ids)
    gamma = None if rnd.gamma is None else to_np(rnd.gamma)[ids]
    tok = to_np(sout["tokens"])[ids]
    kp = to_np(keep)[ids]
    o = oracle.verify(rows(rnd.target, ids), rows(rnd.U, ids), to_np(rnd.E), to_np(rnd.W),
                      to_np(rnd.anchor)[ids], np.where(tok < 0, 0, tok),
                      to_np(sout["draft_lse"])[ids].astype(np.float64),
                      to_np(sout["draft_logit"])[ids].astype(np.float64), kp, to_np(rnd.temperature)[ids],
                      rnd.seed, rnd.round, gamma=gamma, req_ids=ids, bias_first=rnd.bias_first,
                      a_rows=None if a_rows is None else to_np(a_rows)[ids].astype(np.float64), threads=threads,
                      res_rel_eps=RES_REL_EPS)
    acc = to_np(vout["accepted"])[ids]
    nxt = to_np(vout["next_token"])[ids]
    res = to_np(vout["resampled"])[ids]
    c = new_counts()
    c["checked_requests"] = len(ids)
    for i in range(len(ids)):
        a_o = int(o["accepted"][i])
        if acc[i] != a_o:
            j = min(acc[i], a_o)
            assert o["accept_margin"][i, j] < ACC_TOL, "accepted differs for request %d: gpu %d oracle %d" % (
                ids[i], acc[i], a_o)
            c["accept"] += 1
            continue
        assert res[i] == o["resampled"][i]
        c["checked_tokens"] += 1
        if nxt[i] != o["next_token"][i]:
            if o["gap1"][i] < TOK_TOL or o["gap2"][i] < TOK_TOL:
                c["draw"] += 1
                continue
            # a residual draw decided inside the fp32 error of its probabilities
            assert res[i] == 1 and (o["rgap1"][i] < TOK_TOL or o["rgap2"][i] < TOK_TOL), (
                "next token differs for request %d: gpu %d oracle %d (gaps %g %g, fp32 margins %g %g)" % (
                    ids[i], nxt[i], o["next_token"][i], o["gap1"][i], o["gap2"][i], o["rgap1"][i], o["rgap2"][i]))
            c["residual_fp32"] += 1
    assert np.all((acc >= 0) & (acc <= kp))
    return c
