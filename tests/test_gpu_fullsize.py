"""Parity at the full workload sizes, in the launch configuration bench.py times, on outputs
the oracle can compute one by one (sampled heads and rows; decode on sampled heads for all
steps).  Inputs are regenerated exactly for the sampled heads on the CPU."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from softmax_attention_chunk_gb300.inputs import CONFIGS, gen_decode_inputs, gen_path_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def np64(x):
    return x.detach().double().cpu().numpy()


def sample_rows(L, rng, n=24):
    fixed = [0, 1, 63, 64, 127, 128, 129, L // 2, L - 2, L - 1]
    extra = rng.choice(L, n, replace=False).tolist()
    return sorted(set(r for r in fixed + extra if 0 <= r < L))


def fwd_full(cfg):
    from softmax_attention_chunk_gb300 import path_attn as pa

    inp = gen_path_inputs(**cfg)
    t = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    o, lse = pa.fwd(t["q"], t["k"], t["v"], t["w"], t["beta"], t["log_f"], scale=cfg["scale"])
    torch.cuda.synchronize()
    return o.reshape(-1, cfg["seqlen"], cfg["head_dim"]), lse.reshape(-1, cfg["seqlen"])


@pytest.mark.parametrize("name", ["fig1_fwd_l2048", "fig1_fwd_l4096", "fox_long_l16384"])
def test_fwd_full_size_sampled(cuda_lib, name):
    cfg = CONFIGS[name]
    o, lse = fwd_full(cfg)
    BH = cfg["batch"] * cfg["heads"]
    heads = sorted({0, BH // 2 + 1, BH - 1})
    sub = gen_path_inputs(**cfg, heads_subset=heads)
    rng = np.random.default_rng(len(name))
    for n, h in enumerate(heads):
        rows = sample_rows(cfg["seqlen"], rng)
        o_r, l_r = orc.fwd_rows(sub["q"][n], sub["k"][n], sub["v"][n], sub["w"][n], sub["beta"][n],
                                None if sub["log_f"] is None else sub["log_f"][n], cfg["scale"], rows)
        got = np64(o[h, rows])
        err = np.abs(got - o_r).max()
        rel = np.linalg.norm(got - o_r) / np.linalg.norm(o_r)
        assert err <= 2e-2 and rel <= 2e-2, (h, err, rel)
        assert np.abs(np64(lse[h, rows]) - l_r).max() <= 2e-2


def test_train_fwd_bwd_full_size_sampled_heads(cuda_lib):
    from softmax_attention_chunk_gb300 import path_attn as pa

    cfg = CONFIGS["train_b8h16_l4096"]
    inp = gen_path_inputs(**cfg, with_dO=True)
    t = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    o, lse = pa.fwd(t["q"], t["k"], t["v"], t["w"], t["beta"], None, scale=cfg["scale"])
    g = pa.bwd(t["q"], t["k"], t["v"], t["w"], t["beta"], o, lse, t["dO"], scale=cfg["scale"])
    torch.cuda.synchronize()
    BH, L, d = cfg["batch"] * cfg["heads"], cfg["seqlen"], cfg["head_dim"]
    heads = [3, BH - 1]
    sub = gen_path_inputs(**cfg, with_dO=True, heads_subset=heads)
    ref = orc.bwd(sub["q"], sub["k"], sub["v"], sub["w"], sub["beta"], None, cfg["scale"], sub["dO"])
    for key in ("dq", "dk", "dv", "dw", "dbeta"):
        got = np64(g[key].reshape(BH, L, *g[key].shape[3:])[heads])
        r = ref[key]
        err = np.abs(got - r).max()
        rel = np.linalg.norm(got - r) / np.linalg.norm(r)
        assert err <= 2e-2 * max(1.0, np.abs(r).max()) and rel <= 3e-2, (key, err, rel)


def test_train_slice_l64_fp32_against_oracle_and_finite_differences(cuda_lib):
    """fp32 mode on an L=64 slice of the training workload: GPU gradients against the oracle's
    reverse mode (<= 1e-4) and against central differences of the oracle forward."""
    from softmax_attention_chunk_gb300 import path_attn as pa

    cfg = dict(CONFIGS["train_b8h16_l4096"])
    sub = gen_path_inputs(**cfg, with_dO=True, heads_subset=[5])
    L = 64
    x = {k: v[:, :L].float().contiguous() for k, v in sub.items() if v is not None}
    t = {k: v[None].to(DEV) for k, v in x.items()}
    o, lse = pa.fwd(t["q"], t["k"], t["v"], t["w"], t["beta"], None, scale=1.0)
    g = pa.bwd(t["q"], t["k"], t["v"], t["w"], t["beta"], o, lse, t["dO"], scale=1.0)
    torch.cuda.synchronize()
    ref = orc.bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], None, 1.0, x["dO"])
    for key in ("dq", "dk", "dv", "dw", "dbeta"):
        r = ref[key]
        assert np.abs(np64(g[key]).reshape(r[0].shape) - r[0]).max() <= 1e-4 * max(1.0, np.abs(r).max()), key
    q, k, v, w, beta, dO = (x[n].double().numpy()[0].copy() for n in ("q", "k", "v", "w", "beta", "dO"))
    rng = np.random.default_rng(0)

    def loss():
        oo, _ = orc.fwd(q[None], k[None], v[None], w[None], beta[None], None, 1.0)
        return float((oo[0] * dO).sum())

    h = 1e-6
    for name, arr, key in (("q", q, "dq"), ("k", k, "dk"), ("v", v, "dv"), ("w", w, "dw"), ("beta", beta, "dbeta")):
        gg = np64(g[key]).reshape(arr.shape)
        scale = max(1.0, np.abs(gg).max())
        for _ in range(12):
            idx = tuple(rng.integers(0, s) for s in arr.shape)
            old = arr[idx]
            arr[idx] = old + h
            fp = loss()
            arr[idx] = old - h
            fm = loss()
            arr[idx] = old
            fd = (fp - fm) / (2 * h)
            assert abs(fd - gg[idx]) <= 1e-4 * scale, (name, idx, fd, gg[idx])


def test_decode_full_size_sampled_heads(cuda_lib):
    from softmax_attention_chunk_gb300 import path_attn as pa

    cfg = CONFIGS["decode_b32h32_t32768"]
    B, H, d, t0, steps = cfg["batch"], cfg["heads"], cfg["head_dim"], cfg["t0"], cfg["steps"]
    di = gen_decode_inputs(**cfg)
    kc, vc = di["k_cache"].to(DEV), di["v_cache"].to(DEV)
    sx = {n: di[n].to(DEV) for n in ("q", "k", "v", "w", "beta")}
    del di
    heads = [7, B * H - 1]
    sub = gen_decode_inputs(**cfg, heads_subset=heads)
    kref = np64(sub["k_cache"]).copy()
    vref = np64(sub["v_cache"]).copy()
    desc = pa.make_decode_desc(kc, cfg["scale"])
    ws = pa.decode_workspace(desc, DEV)
    worst = 0.0
    for s in range(steps):
        o = pa.decode_step(kc, vc, t0 + s, *(sx[n][s] for n in ("q", "k", "v", "w", "beta")), scale=cfg["scale"],
                           ws=ws)
        o_r = orc.decode_step(kref, vref, t0 + s, *(sub[n][s] for n in ("q", "k", "v", "w", "beta")), cfg["scale"])
        got = np64(o.reshape(B * H, d)[heads])
        worst = max(worst, np.abs(got - o_r).max())
        assert np.linalg.norm(got - o_r) / np.linalg.norm(o_r) <= 2e-2, s
    assert worst <= 2e-2
    n = t0 + steps
    kg = np64(kc.reshape(B * H, -1, d)[heads, :n])
    assert np.abs(kg - kref[:, :n]).max() <= 2e-2


def test_prefill_full_length_sampled_rows(cuda_lib):
    """Hand-off of a prompt as long as the decode workload's cache (32768 tokens, bf16): sampled
    rows of every head against the oracle's one-key-at-a-time transport."""
    cfg = CONFIGS["decode_b32h32_t32768"]
    L = cfg["t0"]
    inp = gen_path_inputs(1, 4, L, cfg["head_dim"], "bf16", seed=cfg["seed"] + 5, near2_frac=0.05)
    from softmax_attention_chunk_gb300 import path_attn as pa

    cap = L + 16
    kc = torch.zeros(1, 4, cap, cfg["head_dim"], dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    t = {n: inp[n].to(DEV) for n in ("k", "v", "w", "beta")}
    pa.decode_prefill(kc, vc, t["k"], t["v"], t["w"], t["beta"])
    torch.cuda.synchronize()
    rows = sample_rows(L, np.random.default_rng(9))
    ref = orc.transport_keys(inp["k"].reshape(4, L, -1), inp["w"].reshape(4, L, -1), inp["beta"].reshape(4, L), rows)
    got = np64(kc.reshape(4, cap, -1)[:, rows])
    err = np.abs(got - ref).max()
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert err <= 2e-2 * np.abs(ref).max() and rel <= 2e-2, (err, rel)
    assert torch.equal(vc[:, :, :L], t["v"])
