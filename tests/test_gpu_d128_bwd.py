"""Head-dim-128 backward (bf16 inputs: the CUDA-core kernels with their products on TF32 warp MMAs,
operands fetched by asynchronous copies, 16 warps per persistent CTA) against the oracle.

* a ragged length with the forget gate (dlog f included), every gradient in full;
* more query tiles than the grid's persistent CTAs (1280 tiles of 32 rows against a cap of 1216), so
  that some CTAs run two tiles back to back, on sampled heads.

Tolerance: 2e-2 * max(1, max|ref|) max abs per gradient and 3e-2 relative Frobenius, as for the
other bf16 backward paths.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from softmax_attention_chunk_gb300.inputs import gen_path_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def np64(x):
    return x.detach().double().cpu().numpy()


def flat(x):
    return None if x is None else x.reshape(-1, *x.shape[2:])


def compare(case, g, ref, keys, record_margin, heads=None):
    for key in keys:
        got = np64(flat(g[key]))
        if heads is not None:
            got = got[heads]
        r = ref[key]
        bound = 2e-2 * max(1.0, np.abs(r).max())
        e = np.abs(got - r).max()
        rr = np.linalg.norm(got - r) / max(np.linalg.norm(r), 1e-30)
        record_margin(case, key, e, bound, rel=rr)
        assert e <= bound and rr <= 3e-2, (key, e, bound, rr)


def test_bwd_d128_bf16_fox_ragged(cuda_lib, record_margin):
    from softmax_attention_chunk_gb300 import path_attn as pa

    inp = gen_path_inputs(2, 3, 333, 128, "bf16", seed=3501, with_dO=True, near2_frac=0.05, fox=True)
    t = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    o, lse = pa.fwd(t["q"], t["k"], t["v"], t["w"], t["beta"], t["log_f"], scale=1.0)
    g = pa.bwd(t["q"], t["k"], t["v"], t["w"], t["beta"], o, lse, t["dO"], scale=1.0, log_f=t["log_f"])
    torch.cuda.synchronize()
    args = [flat(inp[n]) for n in ("q", "k", "v", "w", "beta", "log_f")]
    ref = orc.bwd(*args, 1.0, flat(inp["dO"]), want_dlogf=True)
    compare("d128 backward B2 H3 L333 FoX", g, ref, ("dq", "dk", "dv", "dw", "dbeta", "dlog_f"), record_margin)


def test_bwd_d128_bf16_two_tiles_per_cta(cuda_lib, record_margin):
    from softmax_attention_chunk_gb300 import path_attn as pa

    B, H, L = 1, 80, 512
    cfg = dict(batch=B, heads=H, seqlen=L, head_dim=128, dtype="bf16", seed=3502, with_dO=True, near2_frac=0.05)
    inp = gen_path_inputs(**cfg)
    t = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    o, lse = pa.fwd(t["q"], t["k"], t["v"], t["w"], t["beta"], None, scale=1.0)
    g = pa.bwd(t["q"], t["k"], t["v"], t["w"], t["beta"], o, lse, t["dO"], scale=1.0)
    torch.cuda.synchronize()
    heads = [0, 41, B * H - 1]
    sub = gen_path_inputs(**cfg, heads_subset=heads)
    ref = orc.bwd(sub["q"], sub["k"], sub["v"], sub["w"], sub["beta"], None, 1.0, sub["dO"])
    compare(f"d128 backward B{B} H{H} L{L} (1280 tiles, heads {heads})", g, ref, ("dq", "dk", "dv", "dw", "dbeta"),
            record_margin, heads=heads)
