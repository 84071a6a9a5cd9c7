"""Seeded synthetic inputs for one DSpark draft round.

This module holds no step of the method: it only draws random tensors with the
shapes and value distributions of the workloads the round is measured on, so
that the CUDA library and the CPU oracle read the same bits. The pages measure
on benchmark suites and trained DeepSeek / Qwen3 weights; none of those are
used. The synthetic distributions stand in for their shape: independent
Gaussian logits (`small`), structured high-acceptance logits with a shared
boosted top-1 (`structured`), a mix of low- and high-entropy requests
(`mixed_entropy`), and a target that differs from the draft by a controlled
total-variation distance (`controlled_tv`). WORKLOADS numbers them 1-5 from
`tiny` up, the order of their sizes.

Distribution notation N(mu, s) means mean mu and standard deviation s.
bf16 tensors are drawn in fp32 and rounded to nearest-even by torch.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

SCHED_SYNC, SCHED_ASYNC_CAPACITY, SCHED_FULL_SCAN = 0, 1, 2


@dataclass
class Round:
    name: str
    R: int
    gamma_max: int
    V: int
    r: int
    d: int
    dtype: str                      # "f32" or "bf16"
    U: torch.Tensor                 # [R][G][V]
    E: torch.Tensor                 # [V][r]
    W: torch.Tensor                 # [r][V]
    h: torch.Tensor                 # [R][G][d]
    w_h: torch.Tensor               # [d] fp32
    w_e: torch.Tensor               # [r] fp32
    b: float
    temperature: torch.Tensor       # [R] fp32
    anchor: torch.Tensor            # [R] int32
    target: torch.Tensor            # [R][G+1][V]
    sps: torch.Tensor               # [n_sps] fp32, sps[B-1] = SPS(B)
    gamma: Optional[torch.Tensor]   # [R] int32 or None
    mode: int
    seed: int
    round: int = 0
    conf_token: int = 0
    bias_first: int = 1
    extra: dict = field(default_factory=dict)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def draft_tokens(self) -> int:
        if self.gamma is None:
            return self.R * self.gamma_max
        return int(self.gamma.sum().item())


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, std, g, device, mean=0.0):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std + mean


def sps_tiny(n: int = 20) -> torch.Tensor:
    """SPS(1..5) = 1000, 520, 400, 340, 280, then x0.9 per extra B."""
    v = [1000.0, 520.0, 400.0, 340.0, 280.0]
    while len(v) < n:
        v.append(v[-1] * 0.9)
    return torch.tensor(v[:n], dtype=torch.float32)


def sps_hyperbolic(n: int, a: float = 1e-3, b: float = 2e-6) -> torch.Tensor:
    """Monotone SPS(B) = 1 / (a + b B), B = 1..n."""
    B = torch.arange(1, n + 1, dtype=torch.float64)
    return (1.0 / (a + b * B)).to(torch.float32)


def sps_staircase(n: int, base: float = 1000.0, drop: float = 0.92, step: int = 64) -> torch.Tensor:
    """Staircase SPS(B) = base * drop^floor(B / step), B = 1..n."""
    B = torch.arange(1, n + 1, dtype=torch.float64)
    return (base * drop ** torch.floor(B / step)).to(torch.float32)


def make_round(name: str, R: int, gamma_max: int, V: int, r: int, d: int, dtype: str, *, seed: int,
               device="cpu", u_std=3.0, t_std=3.0, ew_std=0.05, wh_std=None, we_std=0.3, b=1.5,
               temperature=None, gamma=None, sps=None, mode=SCHED_SYNC, boost=None, entropy_split=None,
               tv_range=None, conf_token=0, bias_first=1) -> Round:
    """Generic generator; the named configurations below call it.

    boost=(p, delta): on a fraction p of positions add delta to the top-1 of U_k
      (before the bias) and to the same token in target row k; the bonus row gets its
      own top-1 boosted with probability p.
    entropy_split=(n_low, scale): requests r < n_low have U and target scaled by `scale`.
    tv_range=(lo, hi): delta ~ U[lo, hi] per position, kept in extra["tv_delta"]; the target
      rows are then built by fill_controlled_tv_target from the realised draft distribution.
    """
    dev = torch.device(device)
    g = _gen(seed, dev)
    G = gamma_max
    U = _normal((R, G, V), u_std, g, dev)
    E = _normal((V, r), ew_std, g, dev)
    W = _normal((r, V), ew_std, g, dev)
    h = _normal((R, G, d), 1.0, g, dev)
    w_h = _normal((d,), wh_std if wh_std is not None else 1.0 / math.sqrt(d), g, dev)
    w_e = _normal((r,), we_std, g, dev)
    target = _normal((R, G + 1, V), t_std, g, dev)
    anchor = torch.randint(0, V, (R,), generator=g, device=dev, dtype=torch.int64).to(torch.int32)
    if temperature is None:
        temp = torch.ones(R, device=dev)
    elif callable(temperature):
        temp = temperature(R, g, dev).to(torch.float32)
    else:
        temp = torch.as_tensor(temperature, dtype=torch.float32, device=dev).expand(R).clone()
    if entropy_split is not None:
        n_low, scale = entropy_split
        U[:n_low] *= scale
        target[:n_low] *= scale
    if boost is not None:
        p, delta = boost
        hit = torch.rand((R, G), generator=g, device=dev) < p
        top = U.argmax(dim=2)                                     # [R][G]
        add = hit.to(torch.float32) * delta
        U.scatter_add_(2, top.unsqueeze(2), add.unsqueeze(2))
        target[:, :G].scatter_add_(2, top.unsqueeze(2), add.unsqueeze(2))
        hit_b = (torch.rand((R,), generator=g, device=dev) < p).to(torch.float32) * delta
        top_b = target[:, G].argmax(dim=1)
        target[:, G].scatter_add_(1, top_b.unsqueeze(1), hit_b.unsqueeze(1))
    if tv_range is not None:
        # the target rows of the drafted positions are built from the realised draft distribution
        # once it is known (fill_controlled_tv_target); until then they keep their N(0, t_std) draw
        lo, hi = tv_range
        delta_out = lo + (hi - lo) * torch.rand((R, G), generator=g, device=dev)
    else:
        delta_out = None
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    gamma_t = None if gamma is None else torch.as_tensor(gamma, dtype=torch.int32, device=dev)
    if sps is None:
        sps = sps_hyperbolic(R * (1 + G))
    rnd = Round(name=name, R=R, gamma_max=G, V=V, r=r, d=d, dtype=dtype,
                U=U.to(tdt), E=E.to(tdt), W=W.to(tdt), h=h.to(tdt), w_h=w_h, w_e=w_e, b=float(b),
                temperature=temp, anchor=anchor, target=target.to(tdt), sps=sps.to(dev), gamma=gamma_t,
                mode=mode, seed=int(seed), conf_token=conf_token, bias_first=bias_first)
    if delta_out is not None:
        rnd.extra["tv_delta"] = delta_out
    return rnd


def tv_target_rows(logp_d: torch.Tensor, temperature: torch.Tensor, delta: torch.Tensor,
                   floor: float = -30.0) -> torch.Tensor:
    """Target logit rows at a controlled total-variation distance from a given distribution.

    logp_d [n][G][V]: log p_d of the positions' draft distributions; temperature [n] (> 0);
    delta [n][G] in [0, 1). With v0 = argmin p_d and lam = delta / (1 - p_d(v0)),
    p_t = (1 - lam) p_d + lam e_v0, so that TV(p_t, p_d) = lam (1 - p_d(v0)) = delta; returns
    T log p_t [n][G][V] (fp32), clamped below at floor * T. Input shaping only: the draft
    distribution comes from whoever drafted."""
    p_d = torch.exp(logp_d.float())
    v0 = p_d.argmin(dim=2, keepdim=True)
    pv0 = p_d.gather(2, v0)
    lam = (delta.unsqueeze(2) / (1.0 - pv0)).clamp(max=1.0)
    p_t = (1.0 - lam) * p_d
    p_t.scatter_add_(2, v0, lam)
    T = temperature.view(-1, 1, 1)
    return torch.maximum(T * torch.log(p_t), floor * T)


def fill_controlled_tv_target(rnd: Round, draft_logp, chunk: int = 32) -> None:
    """Replace target rows 0..gamma_r - 1 of every request with rows at the controlled distance
    rnd.extra["tv_delta"] from the realised draft distribution: draft_logp(ids) returns log p_d
    [len(ids)][G][V] of those requests' drafted positions. Rows past gamma_r and the bonus row
    keep their draw. The rows are rounded to the round's element type like every input."""
    delta = rnd.extra["tv_delta"]
    G = rnd.gamma_max
    g = None if rnd.gamma is None else rnd.gamma.cpu().tolist()
    for s0 in range(0, rnd.R, chunk):
        ids = list(range(s0, min(rnd.R, s0 + chunk)))
        lp = draft_logp(ids).to(rnd.target.device)
        rows = tv_target_rows(lp, rnd.temperature[ids], delta[ids].to(lp.device))
        for j, q in enumerate(ids):
            n = G if g is None else int(g[q])
            rnd.target[q, :n] = rows[j, :n].to(rnd.target.dtype)


def tiny(device="cpu") -> Round:
    """R=4, gamma=4, V=64, r=8, d=32, fp32; U, target ~N(0,2); E, W ~N(0,0.1);
    w_h, w_e ~N(0,0.3), b=1.5; T=1; SPS 1000,520,400,340,280 then x0.9 to B=20."""
    return make_round("R4_g4_V64_f32", 4, 4, 64, 8, 32, "f32", seed=0, device=device,
                      u_std=2.0, t_std=2.0, ew_std=0.1, wh_std=0.3, we_std=0.3, b=1.5,
                      sps=sps_tiny(20), mode=SCHED_SYNC)


def small(device="cpu") -> Round:
    """R=32, gamma=16, V=32768, r=256, d=2048, bf16; U, target ~N(0,3); E, W ~N(0,0.05);
    T=1; SPS(B) = 1/(1e-3 + 2e-6 B), 544 entries."""
    return make_round("R32_g16_V32768_bf16", 32, 16, 32768, 256, 2048, "bf16", seed=1,
                      device=device, sps=sps_hyperbolic(544), mode=SCHED_SYNC)


def _temp_structured(R, g, dev):
    return torch.where(torch.arange(R, device=dev) % 2 == 0, torch.tensor(0.6, device=dev),
                       torch.tensor(1.0, device=dev))


def structured(device="cpu") -> Round:
    """R=128, gamma=16, V=151936, r=256, d=4096, bf16; U, target ~N(0,3) with the top-1
    boosted by +6 on 70% of positions; T in {0.6, 1.0}; staircase SPS, 2176 entries."""
    return make_round("R128_g16_V151936_bf16", 128, 16, 151936, 256, 4096, "bf16", seed=2,
                      device=device, boost=(0.7, 6.0), temperature=_temp_structured,
                      sps=sps_staircase(2176), mode=SCHED_SYNC)


def mixed_entropy(device="cpu") -> Round:
    """R=256, gamma=16, V=129280, r=256, d=7168, bf16; requests r<128 have logits x4;
    staircase SPS, 4352 entries; asynchronous capacity scheduling."""
    return make_round("R256_g16_V129280_bf16", 256, 16, 129280, 256, 7168, "bf16", seed=3,
                      device=device, entropy_split=(128, 4.0), sps=sps_staircase(4352),
                      mode=SCHED_ASYNC_CAPACITY)


def _temp_controlled_tv(R, g, dev):
    return 0.3 + 0.9 * torch.rand((R,), generator=g, device=dev)


def controlled_tv(device="cpu") -> Round:
    """R=512, gamma 8 (r < 256) or 16, V=129280, r=256, d=7168, bf16; target differs from
    the draft by TV ~U[0.05, 0.6] per position once fill_controlled_tv_target has built its
    rows from the realised draft; T ~U[0.3, 1.2]; staircase SPS, 8704 entries; full-scan
    scheduling over 8192 slots."""
    R = 512
    gamma = [8] * (R // 2) + [16] * (R // 2)
    return make_round("R512_g8-16_V129280_bf16", R, 16, 129280, 256, 7168, "bf16", seed=4,
                      device=device, temperature=_temp_controlled_tv, gamma=gamma, tv_range=(0.05, 0.6),
                      sps=sps_staircase(8704), mode=SCHED_FULL_SCAN)


WORKLOADS = {1: tiny, 2: small, 3: structured, 4: mixed_entropy, 5: controlled_tv}

# (R, gamma_max, V, r, d, element type) of each workload, without drawing its tensors
SHAPES = {1: (4, 4, 64, 8, 32, torch.float32), 2: (32, 16, 32768, 256, 2048, torch.bfloat16),
          3: (128, 16, 151936, 256, 4096, torch.bfloat16), 4: (256, 16, 129280, 256, 7168, torch.bfloat16),
          5: (512, 16, 129280, 256, 7168, torch.bfloat16)}


def rnn_weights(rnd: Round, seed: int = 99) -> torch.Tensor:
    """Seeded weights W_rnn [3r][2r+d] (rows W_g, W_c, W_o) for the RNN head, N(0, 1/sqrt(2r+d)) so
    that the projections of z = [s; W_1[x]; h] are of order one; the element type of the round."""
    g = _gen(seed, rnd.U.device)
    Z = 2 * rnd.r + rnd.d
    w = _normal((3 * rnd.r, Z), 1.0 / math.sqrt(Z), g, rnd.U.device)
    return w.to(rnd.U.dtype)
