"""A seeded sweep of shapes through the bf16 tensor-core paths against the oracle: batch, heads,
length (ragged, one to several query tiles), scale (either sign), near-reflection fraction and
forget gate drawn from one generator, the forward and every gradient compared in full.  Head
counts are chosen so that the scans' 16-head groups end in a partial group.  Also the head-dim-128
forward across a partial head group, the one-shard (degenerate) context-parallel chain, and a
backward with more query tiles than SMs (several tiles per persistent CTA)."""
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


def sweep_cases(n=6, seed=2024):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        B = int(rng.integers(1, 3))
        H = int(rng.choice([1, 3, 9, 17]))
        L = int(rng.integers(1, 420))
        scale = float(rng.choice([-1.0, 1.0]) * rng.uniform(0.3, 1.2))
        near2 = float(rng.choice([0.0, 0.05, 0.3]))
        fox = bool(rng.integers(0, 2))
        cases.append((i, B, H, L, round(scale, 3), near2, fox))
    return cases


@pytest.mark.parametrize("i,B,H,L,scale,near2,fox", sweep_cases())
def test_sweep_tensor_core_fwd_bwd(cuda_lib, record_margin, i, B, H, L, scale, near2, fox):
    from softmax_attention_chunk_gb300 import path_attn as pa

    inp = gen_path_inputs(B, H, L, 64, "bf16", seed=3000 + i, with_dO=True, near2_frac=near2, fox=fox)
    t = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    o, lse = pa.fwd(t["q"], t["k"], t["v"], t["w"], t["beta"], t["log_f"], scale=scale)
    g = pa.bwd(t["q"], t["k"], t["v"], t["w"], t["beta"], o, lse, t["dO"], scale=scale, log_f=t["log_f"])
    torch.cuda.synchronize()
    args = [flat(inp[n]) for n in ("q", "k", "v", "w", "beta", "log_f")]
    o_ref, lse_ref = orc.fwd(*args, scale)
    case = f"sweep {i}: B{B} H{H} L{L} scale {scale} near2 {near2}{' FoX' if fox else ''}"
    err = np.abs(np64(flat(o)) - o_ref).max()
    rel = np.linalg.norm(np64(flat(o)) - o_ref) / max(np.linalg.norm(o_ref), 1e-30)
    lerr = np.abs(np64(flat(lse)) - lse_ref).max()
    record_margin(case, "o", err, 2e-2, rel=rel)
    assert err <= 2e-2 and rel <= 2e-2 and lerr <= 2e-2, (err, rel, lerr)
    ref = orc.bwd(*args, scale, flat(inp["dO"]), want_dlogf=fox)
    keys = ("dq", "dk", "dv", "dw", "dbeta") + (("dlog_f",) if fox else ())
    for key in keys:
        r, got = ref[key], np64(flat(g[key]))
        bound = 2e-2 * max(1.0, np.abs(r).max())
        e = np.abs(got - r).max()
        rr = np.linalg.norm(got - r) / max(np.linalg.norm(r), 1e-30)
        record_margin(case, key, e, bound, rel=rr)
        assert e <= bound and (rr <= 3e-2 or np.linalg.norm(r) < 1e-6), (key, e, bound, rr)


def test_fwd_d128_tc_partial_head_group(cuda_lib):
    """Head dim 128, batch 2 x 17 heads (34 heads: two full 16-head groups and a group of 2)."""
    from softmax_attention_chunk_gb300 import path_attn as pa

    inp = gen_path_inputs(2, 17, 260, 128, "bf16", seed=3101, near2_frac=0.05)
    t = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    o, lse = pa.fwd(t["q"], t["k"], t["v"], t["w"], t["beta"], None, scale=1.0)
    torch.cuda.synchronize()
    o_ref, lse_ref = orc.fwd(*[flat(inp[n]) for n in ("q", "k", "v", "w", "beta", "log_f")], 1.0)
    got = np64(flat(o))
    assert np.abs(got - o_ref).max() <= 2e-2
    assert np.linalg.norm(got - o_ref) / np.linalg.norm(o_ref) <= 2e-2
    assert np.abs(np64(flat(lse)) - lse_ref).max() <= 2e-2


def test_one_shard_chain_is_the_plain_forward(cuda_lib):
    """A chain of one shard: no messages, the shard's own preparation and scan give the forward."""
    from softmax_attention_chunk_gb300 import path_attn as pa
    from softmax_attention_chunk_gb300.context_parallel import ShardOps, emulate_ring

    inp = gen_path_inputs(1, 3, 384, 64, "bf16", seed=3201, near2_frac=0.05, fox=True)
    t = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    (o, lse), = emulate_ring([ShardOps(t["q"], t["k"], t["v"], t["w"], t["beta"], t["log_f"], 1.0)])
    o1, l1 = pa.fwd(t["q"], t["k"], t["v"], t["w"], t["beta"], t["log_f"], scale=1.0)
    torch.cuda.synchronize()
    assert torch.equal(o, o1)
    assert torch.equal(lse, l1)


@pytest.mark.parametrize("fox", [False, True])
def test_backward_with_several_tiles_per_cta(cuda_lib, record_margin, fox):
    """Batch 2 x 20 heads x 1024: 320 query tiles, more than the SMs, so the persistent backward
    scan runs two or three tiles per CTA (its rings and barrier phases carried from tile to tile);
    three whole heads against the oracle."""
    from softmax_attention_chunk_gb300 import path_attn as pa

    B, H, L = 2, 20, 1024
    cfg = dict(batch=B, heads=H, seqlen=L, head_dim=64, dtype="bf16", seed=3301 + fox, with_dO=True, near2_frac=0.05,
               fox=fox)
    inp = gen_path_inputs(**cfg)
    t = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    o, lse = pa.fwd(t["q"], t["k"], t["v"], t["w"], t["beta"], t["log_f"], scale=1.0)
    g = pa.bwd(t["q"], t["k"], t["v"], t["w"], t["beta"], o, lse, t["dO"], scale=1.0, log_f=t["log_f"])
    torch.cuda.synchronize()
    heads = [0, 17, B * H - 1]
    sub = gen_path_inputs(**cfg, heads_subset=heads)
    ref = orc.bwd(sub["q"], sub["k"], sub["v"], sub["w"], sub["beta"], sub["log_f"], 1.0, sub["dO"], want_dlogf=fox)
    keys = ("dq", "dk", "dv", "dw", "dbeta") + (("dlog_f",) if fox else ())
    case = f"backward B{B} H{H} L{L}{' FoX' if fox else ''}, several tiles per CTA (heads {heads})"
    for key in keys:
        got = np64(flat(g[key])[heads])
        r = ref[key]
        bound = 2e-2 * max(1.0, np.abs(r).max())
        e = np.abs(got - r).max()
        rr = np.linalg.norm(got - r) / max(np.linalg.norm(r), 1e-30)
        record_margin(case, key, e, bound, rel=rr)
        assert e <= bound and rr <= 3e-2, (key, e, bound, rr)
