"""The bf16 forward at head dim 128 on the tensor-core kernels (UT preparation and scan with every
head-dim-wide operand in two 64-column halves, F as a 128 x 128 tile pair), against the oracle:
ragged lengths across one and several 128-row query tiles (partial steps included), PaTH-FoX, a
negative scale, the chunk choices that select this path, the workspace status word, and sampled
rows at the bench's head-dim-128 shape (batch 4 x 16 heads x 2048)."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from softmax_attention_chunk_gb300.inputs import gen_path_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
D = 128


def np64(x):
    return x.detach().double().cpu().numpy()


def flat(x):
    return None if x is None else x.reshape(-1, *x.shape[2:])


def run(inp, scale, chunk=0):
    from softmax_attention_chunk_gb300 import path_attn as pa

    t = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    o, lse = pa.fwd(t["q"], t["k"], t["v"], t["w"], t["beta"], t["log_f"], scale=scale, chunk=chunk)
    torch.cuda.synchronize()
    return o, lse


def check_fwd(inp, o, lse, scale, record_margin=None, case=""):
    o_ref, lse_ref = orc.fwd(flat(inp["q"]), flat(inp["k"]), flat(inp["v"]), flat(inp["w"]), flat(inp["beta"]),
                             flat(inp["log_f"]), scale)
    got, gl = np64(flat(o)), np64(flat(lse))
    err = np.abs(got - o_ref).max()
    rel = np.linalg.norm(got - o_ref) / max(np.linalg.norm(o_ref), 1e-30)
    lerr = np.abs(gl - lse_ref).max()
    if record_margin:
        record_margin(case, "o", err, 2e-2, rel=rel)
        record_margin(case, "lse", lerr, 2e-2)
    assert err <= 2e-2 and rel <= 2e-2 and lerr <= 2e-2, (err, rel, lerr)


def test_the_bf16_forward_takes_the_tensor_core_path(cuda_lib):
    from softmax_attention_chunk_gb300 import path_attn as pa

    q = torch.zeros(1, 2, 300, D, dtype=torch.bfloat16, device=DEV)
    assert pa.path_attn_chunk(pa.make_desc(q, 1.0), 0) == 64
    assert pa.path_attn_chunk(pa.make_desc(q, 1.0), 1) == 32


@pytest.mark.parametrize("L", [1, 63, 64, 65, 128, 129, 300, 700])
def test_fwd_d128_tc_ragged(cuda_lib, record_margin, L):
    inp = gen_path_inputs(1, 2, L, D, "bf16", seed=1300 + L, near2_frac=0.05)
    o, lse = run(inp, 1.0)
    check_fwd(inp, o, lse, 1.0, record_margin, f"d128 tensor-core fwd B1 H2 L{L}")


@pytest.mark.parametrize("L", [65, 500])
def test_fwd_d128_tc_fox(cuda_lib, record_margin, L):
    inp = gen_path_inputs(2, 2, L, D, "bf16", seed=1400 + L, near2_frac=0.05, fox=True)
    o, lse = run(inp, 1.0)
    check_fwd(inp, o, lse, 1.0, record_margin, f"d128 tensor-core FoX fwd B2 H2 L{L}")


def test_fwd_d128_tc_negative_scale_and_chunk64(cuda_lib):
    inp = gen_path_inputs(1, 3, 257, D, "bf16", seed=1501, near2_frac=0.1)
    o, lse = run(inp, -0.7, chunk=64)
    check_fwd(inp, o, lse, -0.7)


def test_fwd_d128_tc_status_is_clean(cuda_lib):
    from softmax_attention_chunk_gb300 import path_attn as pa

    inp = gen_path_inputs(1, 2, 384, D, "bf16", seed=1601)
    t = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    desc = pa.make_desc(t["q"], 1.0)
    ws = pa.workspace(desc, 0, torch.device(DEV))
    pa.fwd(t["q"], t["k"], t["v"], t["w"], t["beta"], None, 1.0, ws=ws)
    cuda_lib.check_workspace(desc, 0, ws)


def test_fwd_d128_tc_bench_shape_sampled_rows(cuda_lib, record_margin):
    """Batch 4 x 16 heads x 2048 (the bench's head-dim-128 leg): sampled rows of three heads."""
    B, H, L = 4, 16, 2048
    cfg = dict(batch=B, heads=H, seqlen=L, head_dim=D, dtype="bf16", seed=1701, near2_frac=0.05)
    inp = gen_path_inputs(**cfg)
    o, lse = run(inp, 1.0)
    o, lse = o.reshape(-1, L, D), lse.reshape(-1, L)
    heads = [0, 29, B * H - 1]
    sub = gen_path_inputs(**cfg, heads_subset=heads)
    rng = np.random.default_rng(17)
    for n, h in enumerate(heads):
        rows = sorted(set([0, 1, 63, 64, 127, 128, 129, L // 2, L - 1] + rng.choice(L, 16, replace=False).tolist()))
        o_r, l_r = orc.fwd_rows(sub["q"][n], sub["k"][n], sub["v"][n], sub["w"][n], sub["beta"][n], None, 1.0, rows)
        got = np64(o[h, rows])
        err = np.abs(got - o_r).max()
        rel = np.linalg.norm(got - o_r) / np.linalg.norm(o_r)
        lerr = np.abs(np64(lse[h, rows]) - l_r).max()
        record_margin(f"d128 tensor-core fwd B{B} H{H} L{L} (sampled rows)", "o", err, 2e-2, rel=rel)
        assert err <= 2e-2 and rel <= 2e-2 and lerr <= 2e-2, (h, err, rel, lerr)
