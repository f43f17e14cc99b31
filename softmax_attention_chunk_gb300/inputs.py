"""Seeded synthetic inputs for PaTH attention (shared by the tests, the bench and smoke()).

This module only draws random numbers and rounds them to the storage dtype; it holds none of
the attention arithmetic.  Every (batch, head) slice of every tensor comes from its own
``torch.Generator('cpu')`` whose seed is a fixed function of (config seed, tensor name, flat
head index).  A test can therefore regenerate only the heads it samples, and get bit-identical
values to the full tensor that was copied to the GPU.

Distributions (PaTH reading notes, cc.laoqi.cc/papers/2505.16381, §2.1 symbol table and the
parameterisation of beta; PaTH-FoX forget gate in §2.5):

* q, k, v ~ N(0, 1)/sqrt(d), rounded to the storage dtype;
* w = w_raw/||w_raw|| with w_raw ~ N(0, I_d) (normalised in fp64, then rounded);
* beta = 2*sigmoid(x), x ~ N(0, 1), kept in fp32; optionally a fraction of positions get
  beta ~ U[1.95, 2) clipped to the largest fp32 below 2 (near-reflection stress);
* log f = log(sigmoid(x_f)), x_f ~ N(2, 1), fp32 (forget gate, optional);
* dO ~ N(0, 1) in the storage dtype (upstream gradient, optional).
"""
from __future__ import annotations

import math

import torch

TORCH_DTYPES = {"bf16": torch.bfloat16, "fp32": torch.float32}

# largest float32 strictly below 2.0
BETA_MAX_BELOW_2 = float(torch.tensor(2.0, dtype=torch.float32).nextafter(torch.tensor(0.0)).item())

_TENSOR_IDS = {
    "q": 1, "k": 2, "v": 3, "w": 4, "xbeta": 5, "near2_mask": 6, "near2_val": 7, "xf": 8, "dO": 9,
    "kc": 11, "vc": 12, "sq": 13, "sk": 14, "sv": 15, "sw": 16, "sxbeta": 17, "xfc": 18, "sxf": 19,
}

# The five workloads (sizes and distributions).  Index 1 is run at L=4096 by default; the
# L=2048 variant is "fig1_fwd_l2048".
CONFIGS = {
    "pr1_tiny_fwd": dict(seed=1000, batch=1, heads=2, seqlen=128, head_dim=64, dtype="fp32",
                         near2_frac=0.0, fox=False, scale=1.0),
    "fig1_fwd_l2048": dict(seed=1001, batch=32, heads=32, seqlen=2048, head_dim=64, dtype="bf16",
                           near2_frac=0.05, fox=False, scale=1.0),
    "fig1_fwd_l4096": dict(seed=1001, batch=32, heads=32, seqlen=4096, head_dim=64, dtype="bf16",
                           near2_frac=0.05, fox=False, scale=1.0),
    "train_b8h16_l4096": dict(seed=1002, batch=8, heads=16, seqlen=4096, head_dim=64, dtype="bf16",
                              near2_frac=0.0, fox=False, scale=1.0),
    "fox_long_l16384": dict(seed=1003, batch=1, heads=32, seqlen=16384, head_dim=64, dtype="bf16",
                            near2_frac=0.0, fox=True, scale=1.0),
    "decode_b32h32_t32768": dict(seed=1004, batch=32, heads=32, head_dim=64, dtype="bf16",
                                 t0=32768, steps=256, scale=1.0),
}


def _gen(seed: int, name: str, bh: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed((seed * 1_000_003 + _TENSOR_IDS[name] * 65_537 + bh) % (2**63 - 1))
    return g


def _heads(batch: int, heads: int, heads_subset):
    return list(range(batch * heads)) if heads_subset is None else [int(h) for h in heads_subset]


def _normal_rows(seed, name, bh, rows, d, dtype, scale=1.0, mean=0.0):
    x = torch.randn(rows, d, generator=_gen(seed, name, bh), dtype=torch.float32)
    if mean != 0.0:
        x = x + mean
    return (x * scale).to(dtype)


def _unit_rows(seed, name, bh, rows, d, dtype):
    x = torch.randn(rows, d, generator=_gen(seed, name, bh), dtype=torch.float32).double()
    x = x / x.norm(dim=-1, keepdim=True)
    return x.to(dtype)


def _beta_row(seed, bh, rows, near2_frac, prefix=""):
    x = torch.randn(rows, generator=_gen(seed, prefix + "xbeta", bh), dtype=torch.float64)
    beta = (2.0 * torch.sigmoid(x)).to(torch.float32)
    if near2_frac > 0.0:
        m = torch.rand(rows, generator=_gen(seed, "near2_mask", bh), dtype=torch.float64) < near2_frac
        u = torch.rand(rows, generator=_gen(seed, "near2_val", bh), dtype=torch.float64)
        nv = (1.95 + 0.05 * u).clamp(max=BETA_MAX_BELOW_2).to(torch.float32)
        beta = torch.where(m, nv, beta)
    return beta.clamp(max=BETA_MAX_BELOW_2)


def _parallel(fn, n):
    """Runs fn(i) for i < n on a thread pool (torch kernels release the GIL)."""
    if n <= 8:
        for i in range(n):
            fn(i)
        return
    import concurrent.futures as cf
    import os
    with cf.ThreadPoolExecutor(max_workers=min(32, os.cpu_count() or 4)) as ex:
        list(ex.map(fn, range(n)))


def gen_path_inputs(batch, heads, seqlen, head_dim, dtype="bf16", seed=1000, near2_frac=0.0,
                    fox=False, with_dO=False, heads_subset=None, **_unused):
    """Inputs of the forward/backward workload.

    Returns a dict of CPU tensors.  Without ``heads_subset`` the shapes are [B,H,L,d] and
    [B,H,L]; with it (a list of flat head indices b*H+h) they are [n,L,d] and [n,L], holding
    exactly the values those heads have in the full tensors.
    """
    tdt = TORCH_DTYPES[dtype]
    d, L = head_dim, seqlen
    sd = 1.0 / math.sqrt(d)
    hs = _heads(batch, heads, heads_subset)
    n = len(hs)
    res = {key: torch.empty(n, L, d, dtype=tdt) for key in ("q", "k", "v", "w")}
    res["beta"] = torch.empty(n, L, dtype=torch.float32)
    res["log_f"] = torch.empty(n, L, dtype=torch.float32) if fox else None
    res["dO"] = torch.empty(n, L, d, dtype=tdt) if with_dO else None

    def one(idx):
        bh = hs[idx]
        res["q"][idx] = _normal_rows(seed, "q", bh, L, d, tdt, sd)
        res["k"][idx] = _normal_rows(seed, "k", bh, L, d, tdt, sd)
        res["v"][idx] = _normal_rows(seed, "v", bh, L, d, tdt, sd)
        res["w"][idx] = _unit_rows(seed, "w", bh, L, d, tdt)
        res["beta"][idx] = _beta_row(seed, bh, L, near2_frac)
        if fox:
            xf = torch.randn(L, generator=_gen(seed, "xf", bh), dtype=torch.float64) + 2.0
            res["log_f"][idx] = torch.log(torch.sigmoid(xf)).to(torch.float32)
        if with_dO:
            res["dO"][idx] = _normal_rows(seed, "dO", bh, L, d, tdt, 1.0)

    _parallel(one, n)
    if heads_subset is None:
        for key, t in list(res.items()):
            if t is not None:
                res[key] = t.reshape(batch, heads, *t.shape[1:])
    return res


def _log_f_row(seed, name, bh, rows):
    """log f = log sigmoid(N(2, 1)), computed in fp64, stored fp32."""
    xf = torch.randn(rows, generator=_gen(seed, name, bh), dtype=torch.float64) + 2.0
    return torch.log(torch.sigmoid(xf)).to(torch.float32)


def gen_decode_inputs(batch, heads, head_dim, t0, steps, dtype="bf16", seed=1004, capacity=None,
                      heads_subset=None, fox=False, **_unused):
    """Inputs of the decode workload: a cache pre-filled with ``t0`` random entries and
    ``steps`` new tokens per head.

    Returns k_cache/v_cache of shape [B,H,capacity,d] (entries >= t0 are zero), per-step
    q,k,v,w of shape [steps,B,H,d] and beta of shape [steps,B,H].  With ``fox`` also a_cache
    [B,H,capacity] (fp32 running sums of the pre-filled entries' log f, summed in fp64) and the
    per-step log_f [steps,B,H].  With ``heads_subset`` the head axes collapse to one axis of the
    selected flat head indices.
    """
    tdt = TORCH_DTYPES[dtype]
    d = head_dim
    cap = t0 + steps if capacity is None else capacity
    sd = 1.0 / math.sqrt(d)
    hs = _heads(batch, heads, heads_subset)
    n = len(hs)
    kc = torch.zeros(n, cap, d, dtype=tdt)
    vc = torch.zeros(n, cap, d, dtype=tdt)
    sq, sk, sv, sw = (torch.empty(n, steps, d, dtype=tdt) for _ in range(4))
    sb = torch.empty(n, steps, dtype=torch.float32)
    ac = torch.zeros(n, cap, dtype=torch.float32) if fox else None
    sf = torch.empty(n, steps, dtype=torch.float32) if fox else None

    def one(idx):
        bh = hs[idx]
        if t0 > 0:
            kc[idx, :t0] = _normal_rows(seed, "kc", bh, t0, d, tdt, sd)
            vc[idx, :t0] = _normal_rows(seed, "vc", bh, t0, d, tdt, sd)
        sq[idx] = _normal_rows(seed, "sq", bh, steps, d, tdt, sd)
        sk[idx] = _normal_rows(seed, "sk", bh, steps, d, tdt, sd)
        sv[idx] = _normal_rows(seed, "sv", bh, steps, d, tdt, sd)
        sw[idx] = _unit_rows(seed, "sw", bh, steps, d, tdt)
        sb[idx] = _beta_row(seed, bh, steps, 0.0, prefix="s")
        if fox:
            if t0 > 0:
                ac[idx, :t0] = torch.cumsum(_log_f_row(seed, "xfc", bh, t0).double(), 0).to(torch.float32)
            sf[idx] = _log_f_row(seed, "sxf", bh, steps)

    _parallel(one, n)
    step = lambda x: x.transpose(0, 1).contiguous()  # [steps, n, ...]
    res = dict(k_cache=kc, v_cache=vc, q=step(sq), k=step(sk), v=step(sv), w=step(sw), beta=step(sb))
    if fox:
        res["a_cache"] = ac
        res["log_f"] = step(sf)
    if heads_subset is None:
        res["k_cache"] = kc.reshape(batch, heads, cap, d)
        res["v_cache"] = vc.reshape(batch, heads, cap, d)
        for key in ("q", "k", "v", "w"):
            res[key] = res[key].reshape(steps, batch, heads, d)
        res["beta"] = res["beta"].reshape(steps, batch, heads)
        if fox:
            res["a_cache"] = ac.reshape(batch, heads, cap)
            res["log_f"] = res["log_f"].reshape(steps, batch, heads)
    return res
