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
def test_fwd_full_size_sampled(cuda_lib, name, record_margin):
    cfg = CONFIGS[name]
    o, lse = fwd_full(cfg)
    BH = cfg["batch"] * cfg["heads"]
    heads = sorted({0, BH // 2 + 1, BH - 1})
    sub = gen_path_inputs(**cfg, heads_subset=heads)
    rng = np.random.default_rng(len(name))
    worst = dict(o=0.0, lse=0.0, rel=0.0)
    for n, h in enumerate(heads):
        rows = sample_rows(cfg["seqlen"], rng)
        o_r, l_r = orc.fwd_rows(sub["q"][n], sub["k"][n], sub["v"][n], sub["w"][n], sub["beta"][n],
                                None if sub["log_f"] is None else sub["log_f"][n], cfg["scale"], rows)
        got = np64(o[h, rows])
        err = np.abs(got - o_r).max()
        rel = np.linalg.norm(got - o_r) / np.linalg.norm(o_r)
        lerr = np.abs(np64(lse[h, rows]) - l_r).max()
        worst = dict(o=max(worst["o"], err), lse=max(worst["lse"], lerr), rel=max(worst["rel"], rel))
        assert err <= 2e-2 and rel <= 2e-2, (h, err, rel)
        assert lerr <= 2e-2
    record_margin(f"{name} fwd", "o", worst["o"], 2e-2, rel=worst["rel"])
    record_margin(f"{name} fwd", "lse", worst["lse"], 2e-2)


def check_grads(case, got, ref, heads, BH, L, record_margin, keys=("dq", "dk", "dv", "dw", "dbeta")):
    """Gradients on sampled heads: max abs <= 2e-2 max(1, max|ref|) and relative Frobenius <= 3e-2
    per tensor; the unscaled errors and max|ref| are recorded."""
    for key in keys:
        g = np64(got[key].reshape(BH, L, *got[key].shape[3:])[heads])
        r = ref[key]
        err = np.abs(g - r).max()
        rel = np.linalg.norm(g - r) / np.linalg.norm(r)
        bound = 2e-2 * max(1.0, np.abs(r).max())
        record_margin(case, key, err, bound, ref_max=np.abs(r).max(), rel=rel)
        assert err <= bound and rel <= 3e-2, (case, key, err, rel)


def training_step(pa, t, scale, log_f=None):
    """The training step as bench.py runs it: the forward's PREPARE and SCAN (storing the transported
    query tiles) in the backward-sized workspace, then the backward's PREPARE (reusing the forward's
    preparation and tiles), SCAN and FINISH on the same workspace; the workspace status is checked."""
    desc = pa.make_desc(t["q"], scale)
    ws = pa.workspace(desc, 1, DEV)
    o = torch.empty_like(t["q"])
    lse = torch.empty(t["q"].shape[:3], dtype=torch.float32, device=DEV)
    grads = dict(dq=torch.empty_like(o), dk=torch.empty_like(o), dv=torch.empty_like(o), dw=torch.empty_like(o),
                 dbeta=torch.empty_like(t["beta"]))
    if log_f is not None:
        grads["dlog_f"] = torch.empty_like(t["beta"])
    args = (t["q"], t["k"], t["v"], t["w"], t["beta"])
    pa.fwd(*args, log_f, scale, ws=ws, out=(o, lse), phases=pa.PATH_FWD_PREPARE)
    pa.fwd(*args, log_f, scale, ws=ws, out=(o, lse), phases=pa.PATH_FWD_SCAN | pa.PATH_FWD_STORE_Z)
    for ph in (pa.PATH_BWD_PREPARE | pa.PATH_BWD_REUSE_FWD | pa.PATH_BWD_Z_FROM_FWD, pa.PATH_BWD_SCAN,
               pa.PATH_BWD_FINISH):
        pa.bwd(*args, o, lse, t["dO"], scale, ws=ws, log_f=log_f, out=grads, phases=ph)
    pa.check_workspace(desc, 1, ws)
    return o, lse, grads


def test_training_step_at_bench_shape_sampled_heads(cuda_lib, record_margin):
    """The exact step bench.py times (batch 32 x 32 heads, L 4096, bf16, 5 % near-reflection beta;
    forward storing its transported query tiles, backward reusing them and the preparation) on
    sampled heads against the oracle: o, lse and every gradient.  Heads 130, 517 and 1023 have
    their tiles more than 2^31 bytes into the tile store; 1023 is in the last 16-head group of the
    tile schedule."""
    pa = cuda_lib
    cfg = CONFIGS["fig1_fwd_l4096"]
    inp = gen_path_inputs(**cfg, with_dO=True)
    t = {k: v.to(DEV) for k, v in inp.items() if v is not None}
    del inp
    o, lse, g = training_step(pa, t, cfg["scale"])
    torch.cuda.synchronize()
    del t
    BH, L, d = cfg["batch"] * cfg["heads"], cfg["seqlen"], cfg["head_dim"]
    heads = [3, 130, 517, 1023]
    sub = gen_path_inputs(**cfg, with_dO=True, heads_subset=heads)
    o_r, l_r = orc.fwd(sub["q"], sub["k"], sub["v"], sub["w"], sub["beta"], None, cfg["scale"])
    got = np64(o.reshape(BH, L, d)[heads])
    err, rel = np.abs(got - o_r).max(), np.linalg.norm(got - o_r) / np.linalg.norm(o_r)
    lerr = np.abs(np64(lse.reshape(BH, L)[heads]) - l_r).max()
    record_margin("train step B32 H32 L4096", "o", err, 2e-2, rel=rel)
    record_margin("train step B32 H32 L4096", "lse", lerr, 2e-2)
    assert err <= 2e-2 and rel <= 2e-2 and lerr <= 2e-2, (err, rel, lerr)
    ref = orc.bwd(sub["q"], sub["k"], sub["v"], sub["w"], sub["beta"], None, cfg["scale"], sub["dO"])
    check_grads("train step B32 H32 L4096", g, ref, heads, BH, L, record_margin)


@pytest.mark.parametrize("shape", [(2, 16, 4096), (1, 32, 16384)])
def test_fox_training_step_long_sequences(cuda_lib, record_margin, shape):
    """PaTH-FoX training step (forget bias forward, dlog f backward, the bench's reuse path) at
    L 4096 (batch 2 x 16 heads) and at the long-context workload's shape (batch 1 x 32 heads,
    L 16384), sampled heads against the oracle including dlog f.  The backward forms the forget
    bias A_i - A_j from fp32 prefix sums over the whole sequence."""
    pa = cuda_lib
    Bt, H, L = shape
    cfg = dict(CONFIGS["fox_long_l16384"], batch=Bt, heads=H, seqlen=L)
    inp = gen_path_inputs(**cfg, with_dO=True)
    t = {k: v.to(DEV) for k, v in inp.items() if v is not None}
    del inp
    o, lse, g = training_step(pa, t, cfg["scale"], log_f=t["log_f"])
    torch.cuda.synchronize()
    del t
    BH, d = Bt * H, cfg["head_dim"]
    heads = [5, BH - 1]
    sub = gen_path_inputs(**cfg, with_dO=True, heads_subset=heads)
    case = f"FoX train step B{Bt} H{H} L{L}"
    o_r, l_r = orc.fwd(sub["q"], sub["k"], sub["v"], sub["w"], sub["beta"], sub["log_f"], cfg["scale"])
    got = np64(o.reshape(BH, L, d)[heads])
    err, rel = np.abs(got - o_r).max(), np.linalg.norm(got - o_r) / np.linalg.norm(o_r)
    lerr = np.abs(np64(lse.reshape(BH, L)[heads]) - l_r).max()
    record_margin(case, "o", err, 2e-2, rel=rel)
    record_margin(case, "lse", lerr, 2e-2)
    assert err <= 2e-2 and rel <= 2e-2 and lerr <= 2e-2, (err, rel, lerr)
    ref = orc.bwd(sub["q"], sub["k"], sub["v"], sub["w"], sub["beta"], sub["log_f"], cfg["scale"], sub["dO"],
                  want_dlogf=True)
    check_grads(case, g, ref, heads, BH, L, record_margin,
                keys=("dq", "dk", "dv", "dw", "dbeta", "dlog_f"))


def test_train_fwd_bwd_full_size_sampled_heads(cuda_lib, record_margin):
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
    check_grads("train B8 H16 L4096 (plain fwd + bwd)", g, ref, heads, BH, L, record_margin)


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


def test_decode_full_size_sampled_heads(cuda_lib, record_margin):
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
    kerr = np.abs(kg - kref[:, :n]).max()
    record_margin("decode B32 H32 t32768, 256 steps", "o_t (worst step)", worst, 2e-2)
    record_margin("decode B32 H32 t32768, 256 steps", "k_cache", kerr, 2e-2)
    assert kerr <= 2e-2


def test_prefill_full_length_sampled_rows(cuda_lib, record_margin):
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
    record_margin("prefill hand-off 4 heads x 32768", "k_cache rows", err, 2e-2 * np.abs(ref).max(), rel=rel)
    assert err <= 2e-2 * np.abs(ref).max() and rel <= 2e-2, (err, rel)
    assert torch.equal(vc[:, :, :L], t["v"])
