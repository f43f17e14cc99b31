"""GPU parity: the CUDA library (through the C ABI) against the fp64 CPU oracle, element by
element, on the same seeded inputs.  Sizes span several chunks and ragged tails.

Tolerances (stated by the workload definitions): max abs error <= 1e-4 in the fp32 mode and
<= 2e-2 on bf16 outputs.  Gradients use max abs <= tol * max(1, max |ref|) per tensor.  The
bf16 cases additionally require relative Frobenius error <= 2e-2 so that an error of the order of
the (small) outputs themselves cannot pass.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from softmax_attention_chunk_gb300.inputs import gen_decode_inputs, gen_path_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def flat(x):
    return None if x is None else x.reshape(-1, *x.shape[2:])


def np64(x):
    return x.detach().double().cpu().numpy()


def check(got, ref, tol, name, rel=None):
    got = np64(got).reshape(ref.shape)
    err = np.abs(got - ref).max()
    assert err <= tol, f"{name}: max abs err {err:.3e} > {tol:.1e}"
    if rel is not None and np.linalg.norm(ref) > 0:  # a zero reference leaves the max-abs bound
        r = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert r <= rel, f"{name}: rel fro err {r:.3e} > {rel:.1e}"
    return err


def run_fwd(inp, scale, chunk=0):
    from softmax_attention_chunk_gb300 import path_attn as pa

    t = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    o, lse = pa.fwd(t["q"], t["k"], t["v"], t["w"], t["beta"], t["log_f"], scale=scale, chunk=chunk)
    torch.cuda.synchronize()
    return o, lse


def oracle_fwd(inp, scale):
    return orc.fwd(flat(inp["q"]), flat(inp["k"]), flat(inp["v"]), flat(inp["w"]), flat(inp["beta"]),
                   flat(inp["log_f"]), scale)


@pytest.mark.parametrize("chunk", [0, 32, 64])
def test_fwd_pr1_tiny_fp32(cuda_lib, chunk):
    """Batch 1, 2 heads, L=128, d=64, fp32: max abs <= 1e-4."""
    from softmax_attention_chunk_gb300.inputs import CONFIGS

    cfg = CONFIGS["pr1_tiny_fwd"]
    inp = gen_path_inputs(**cfg)
    o, lse = run_fwd(inp, cfg["scale"], chunk)
    o_ref, lse_ref = oracle_fwd(inp, cfg["scale"])
    check(o, o_ref, 1e-4, "o")
    check(lse, lse_ref, 1e-4, "lse")


@pytest.mark.parametrize("L", [1, 2, 31, 33, 64, 65, 130, 257])
@pytest.mark.parametrize("fox", [False, True])
def test_fwd_ragged_fp32(cuda_lib, L, fox):
    inp = gen_path_inputs(2, 2, L, 64, "fp32", seed=100 + L, fox=fox)
    o, lse = run_fwd(inp, 1.0)
    o_ref, lse_ref = oracle_fwd(inp, 1.0)
    check(o, o_ref, 1e-4, "o")
    check(lse, lse_ref, 1e-4, "lse")


def test_fwd_large_logits_fp32(cuda_lib):
    """scale = 16 gives logits of std ~2: exercises the online-softmax rescaling."""
    inp = gen_path_inputs(1, 3, 300, 64, "fp32", seed=5, near2_frac=0.2)
    o, lse = run_fwd(inp, 16.0)
    o_ref, lse_ref = oracle_fwd(inp, 16.0)
    check(o, o_ref, 1e-4, "o")
    check(lse, lse_ref, 1e-4, "lse")


def test_fwd_beta_edges_fp32(cuda_lib):
    """beta = 0 (identity), exactly 2 (reflection), and out-of-range values (clamped to [0, 2])."""
    inp = gen_path_inputs(1, 2, 150, 64, "fp32", seed=6)
    b = inp["beta"].clone()
    b[..., 0::5] = 2.0
    b[..., 1::5] = 0.0
    b[..., 2::7] = 2.5
    b[..., 3::11] = -0.5
    inp["beta"] = b
    o, lse = run_fwd(inp, 1.0)
    o_ref, lse_ref = oracle_fwd(inp, 1.0)
    check(o, o_ref, 1e-4, "o")
    check(lse, lse_ref, 1e-4, "lse")


@pytest.mark.parametrize("fox", [False, True])
def test_fwd_bf16_near_reflection(cuda_lib, fox):
    inp = gen_path_inputs(2, 2, 700, 64, "bf16", seed=8, near2_frac=0.05, fox=fox)
    o, lse = run_fwd(inp, 1.0)
    o_ref, lse_ref = oracle_fwd(inp, 1.0)
    check(o, o_ref, 2e-2, "o", rel=2e-2)
    check(lse, lse_ref, 2e-2, "lse")


def run_bwd(inp, scale):
    from softmax_attention_chunk_gb300 import path_attn as pa

    t = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    o, lse = pa.fwd(t["q"], t["k"], t["v"], t["w"], t["beta"], None, scale=scale)
    g = pa.bwd(t["q"], t["k"], t["v"], t["w"], t["beta"], o, lse, t["dO"], scale=scale)
    torch.cuda.synchronize()
    return g


def check_grads(inp, g, scale, tol, rel=None):
    ref = orc.bwd(flat(inp["q"]), flat(inp["k"]), flat(inp["v"]), flat(inp["w"]), flat(inp["beta"]), None,
                  scale, flat(inp["dO"]))
    for key in ("dq", "dk", "dv", "dw", "dbeta"):
        r = ref[key]
        check(flat(g[key]), r, tol * max(1.0, np.abs(r).max()), key, rel=rel)


@pytest.mark.parametrize("L", [1, 31, 32, 33, 100, 129])
def test_bwd_fp32(cuda_lib, L):
    inp = gen_path_inputs(1, 2, L, 64, "fp32", seed=200 + L, with_dO=True, near2_frac=0.1)
    g = run_bwd(inp, 1.0)
    check_grads(inp, g, 1.0, 1e-4)


def test_bwd_fp32_scaled(cuda_lib):
    inp = gen_path_inputs(1, 2, 160, 64, "fp32", seed=31, with_dO=True)
    g = run_bwd(inp, 4.0)
    check_grads(inp, g, 4.0, 1e-4)


def test_bwd_bf16(cuda_lib):
    inp = gen_path_inputs(2, 2, 300, 64, "bf16", seed=32, with_dO=True, near2_frac=0.05)
    g = run_bwd(inp, 1.0)
    check_grads(inp, g, 1.0, 2e-2, rel=3e-2)


@pytest.mark.parametrize("L", [1, 40, 64, 65, 128, 129, 192, 257])
def test_bwd_bf16_ragged(cuda_lib, L):
    """bf16 tensor-core backward at lengths giving a lone partial chunk (1, 40), exact chunk and
    query-tile multiples (64, 128, 192), a tile whose only step is the partial one (65) and
    ragged tails after full tiles (129, 257)."""
    inp = gen_path_inputs(1, 3, L, 64, "bf16", seed=300 + L, with_dO=True, near2_frac=0.05)
    g = run_bwd(inp, 1.0)
    check_grads(inp, g, 1.0, 2e-2, rel=3e-2)


def test_bwd_bf16_more_heads_than_a_schedule_group(cuda_lib):
    """18 heads: the tile schedule takes heads 16 at a time, so the second group is partial."""
    inp = gen_path_inputs(2, 9, 200, 64, "bf16", seed=77, with_dO=True, near2_frac=0.05)
    g = run_bwd(inp, 1.0)
    check_grads(inp, g, 1.0, 2e-2, rel=3e-2)


def test_fwd_bf16_more_heads_than_a_schedule_group(cuda_lib):
    inp = gen_path_inputs(2, 9, 200, 64, "bf16", seed=78, near2_frac=0.05)
    o, lse = run_fwd(inp, 1.0)
    o_ref, lse_ref = oracle_fwd(inp, 1.0)
    check(flat(o), o_ref, 2e-2, "o", rel=2e-2)
    check(flat(lse), lse_ref, 2e-2, "lse")


@pytest.mark.parametrize("L,scale", [(1, 1.0), (31, 1.0), (33, 1.0), (129, 0.7), (200, 0.0)])
def test_bwd_fp32_fox(cuda_lib, L, scale):
    """Forget-gate backward on the fp32 path (32-row chunks): every gradient including dlog f
    within 1e-4 of the oracle, at a lone partial chunk, one chunk and one row, ragged tails and a
    zero scale (only the forget bias shapes the attention)."""
    from softmax_attention_chunk_gb300 import path_attn as pa

    inp = gen_path_inputs(1, 2, L, 64, "fp32", seed=600 + L, with_dO=True, near2_frac=0.1, fox=True)
    t = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    o, lse = pa.fwd(t["q"], t["k"], t["v"], t["w"], t["beta"], t["log_f"], scale=scale)
    g = pa.bwd(t["q"], t["k"], t["v"], t["w"], t["beta"], o, lse, t["dO"], scale=scale, log_f=t["log_f"])
    torch.cuda.synchronize()
    check_grads_fox(inp, g, scale, 1e-4, None)


def test_bwd_bf16_chunk32_fox(cuda_lib):
    """bf16 inputs on the 32-row-chunk (SIMT) path with the forget gate, within the bf16 bound."""
    from softmax_attention_chunk_gb300 import path_attn as pa

    inp = gen_path_inputs(2, 2, 150, 64, "bf16", seed=611, with_dO=True, near2_frac=0.05, fox=True)
    t = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    o, lse = pa.fwd(t["q"], t["k"], t["v"], t["w"], t["beta"], t["log_f"], scale=1.0, chunk=32)
    g = pa.bwd(t["q"], t["k"], t["v"], t["w"], t["beta"], o, lse, t["dO"], scale=1.0, chunk=32, log_f=t["log_f"])
    torch.cuda.synchronize()
    check_grads_fox(inp, g, 1.0, 2e-2, 3e-2)


@pytest.mark.parametrize("dtype,t0,steps,tol", [("fp32", 0, 40, 1e-4), ("fp32", 3000, 5, 1e-4),
                                                ("bf16", 0, 30, 2e-2), ("bf16", 5000, 6, 2e-2)])
def test_decode_steps(cuda_lib, dtype, t0, steps, tol):
    from softmax_attention_chunk_gb300 import path_attn as pa

    B, H, d = 2, 2, 64
    di = gen_decode_inputs(B, H, d, t0=t0, steps=steps, dtype=dtype, seed=40 + t0)
    kc, vc = di["k_cache"].to(DEV), di["v_cache"].to(DEV)
    kref = np64(di["k_cache"]).reshape(B * H, -1, d).copy()
    vref = np64(di["v_cache"]).reshape(B * H, -1, d).copy()
    for s in range(steps):
        args = [di[n][s].to(DEV) for n in ("q", "k", "v", "w", "beta")]
        o_t = pa.decode_step(kc, vc, t0 + s, *args, scale=1.0)
        torch.cuda.synchronize()
        o_r = orc.decode_step(kref, vref, t0 + s, *[flat(di[n][s]) for n in ("q", "k", "v", "w", "beta")], 1.0)
        check(o_t.reshape(B * H, d), o_r, tol, f"o_t step {s}", rel=2e-2 if dtype == "bf16" else None)
    n = t0 + steps
    check(kc.reshape(B * H, -1, d)[:, :n], kref[:, :n], tol, "rewritten keys")
    check(vc.reshape(B * H, -1, d)[:, :n], vref[:, :n], 0.0, "values")


def test_decode_matches_forward_rows(cuda_lib):
    """Decoding a sequence token by token from an empty cache gives the forward's rows."""
    from softmax_attention_chunk_gb300 import path_attn as pa

    L = 70
    inp = gen_path_inputs(1, 2, L, 64, "fp32", seed=77)
    o_f, _ = run_fwd(inp, 1.0)
    kc = torch.zeros(1, 2, L, 64, device=DEV)
    vc = torch.zeros_like(kc)
    rows = []
    for t in range(L):
        sl = lambda x: x[:, :, t].contiguous().to(DEV)
        rows.append(pa.decode_step(kc, vc, t, sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["w"]),
                                   sl(inp["beta"]), scale=1.0))
    o_d = torch.stack(rows, 2)
    assert (o_d - o_f).abs().max().item() <= 1e-4


def test_bwd_reusing_forward_preparation(cuda_lib):
    """PATH_BWD_REUSE_FWD: forward run in the backward's workspace, backward skips recomputing
    the preparation; gradients equal the plain backward's (up to reduction order) and the oracle's."""
    from softmax_attention_chunk_gb300 import path_attn as pa

    inp = gen_path_inputs(2, 2, 333, 64, "bf16", seed=44, with_dO=True, near2_frac=0.05)
    t = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    desc = pa.make_desc(t["q"], 1.0)
    ws = pa.workspace(desc, 1, DEV)
    o, lse = pa.fwd(t["q"], t["k"], t["v"], t["w"], t["beta"], None, 1.0, ws=ws)
    g_plain = pa.bwd(t["q"], t["k"], t["v"], t["w"], t["beta"], o, lse, t["dO"], 1.0)
    g_reuse = pa.bwd(t["q"], t["k"], t["v"], t["w"], t["beta"], o, lse, t["dO"], 1.0, ws=ws,
                     phases=pa.PATH_BWD_ALL | pa.PATH_BWD_REUSE_FWD)
    torch.cuda.synchronize()
    for key in ("dq", "dk", "dv", "dw", "dbeta"):
        a, b = g_plain[key].float(), g_reuse[key].float()
        assert (a - b).abs().max().item() <= 1e-2 * max(1.0, a.abs().max().item()), key
    check_grads(inp, g_reuse, 1.0, 2e-2, rel=3e-2)


@pytest.mark.parametrize("L", [65, 129, 333, 1000])
def test_training_step_with_stored_transported_queries(cuda_lib, L):
    """PATH_FWD_STORE_Z + PATH_BWD_Z_FROM_FWD: the forward stores every transported query tile, the
    backward skips recomputing them; gradients equal the plain backward's (the tiles are the same
    bf16 values up to MMA accumulation order) and the oracle's."""
    from softmax_attention_chunk_gb300 import path_attn as pa

    inp = gen_path_inputs(2, 2, L, 64, "bf16", seed=45 + L, with_dO=True, near2_frac=0.05)
    t = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    desc = pa.make_desc(t["q"], 1.0)
    o0, lse0 = pa.fwd(t["q"], t["k"], t["v"], t["w"], t["beta"], None, 1.0)
    g_plain = pa.bwd(t["q"], t["k"], t["v"], t["w"], t["beta"], o0, lse0, t["dO"], 1.0)
    ws = pa.workspace(desc, 1, DEV)
    o, lse = pa.fwd(t["q"], t["k"], t["v"], t["w"], t["beta"], None, 1.0, ws=ws,
                    phases=pa.PATH_FWD_ALL | pa.PATH_FWD_STORE_Z)
    g = pa.bwd(t["q"], t["k"], t["v"], t["w"], t["beta"], o, lse, t["dO"], 1.0, ws=ws,
               phases=pa.PATH_BWD_ALL | pa.PATH_BWD_REUSE_FWD | pa.PATH_BWD_Z_FROM_FWD)
    torch.cuda.synchronize()
    assert torch.equal(o, o0) and torch.equal(lse, lse0)  # storing Z leaves the outputs unchanged
    for key in ("dq", "dk", "dv", "dw", "dbeta"):
        a, b = g_plain[key].float(), g[key].float()
        assert (a - b).abs().max().item() <= 1e-2 * max(1.0, a.abs().max().item()), key
    check_grads(inp, g, 1.0, 2e-2, rel=3e-2)


# ---------------- prefill -> decode hand-off ----------------

def run_prefill(inp, dtype, cap, fill=7.0):
    from softmax_attention_chunk_gb300 import path_attn as pa

    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    B, H, L, d = inp["k"].shape
    kc = torch.full((B, H, cap, d), fill, dtype=tdt, device=DEV)
    vc = torch.full((B, H, cap, d), fill, dtype=tdt, device=DEV)
    t = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    pa.decode_prefill(kc, vc, t["k"], t["v"], t["w"], t["beta"])
    torch.cuda.synchronize()
    return kc, vc


@pytest.mark.parametrize("dtype,L", [("fp32", 1), ("fp32", 65), ("fp32", 333), ("bf16", 1), ("bf16", 64),
                                     ("bf16", 200), ("bf16", 1000)])
def test_prefill_cache_matches_oracle(cuda_lib, dtype, L):
    """Rows 0..L-1: keys transported to the prompt end (fp32 within 1e-4; bf16 within the bf16
    tolerance relative to the largest key), values copied exactly; rows >= L untouched."""
    inp = gen_path_inputs(1, 3, L, 64, dtype, seed=500 + L, near2_frac=0.05)
    cap = L + 7
    kc, vc = run_prefill(inp, dtype, cap)
    kref, vref = orc.prefill_cache(flat(inp["k"]), flat(inp["v"]), flat(inp["w"]), flat(inp["beta"]), cap)
    if dtype == "fp32":
        check(flat(kc)[:, :L], kref[:, :L], 1e-4, "k_cache")
    else:
        check(flat(kc)[:, :L], kref[:, :L], 2e-2 * np.abs(kref).max(), "k_cache", rel=2e-2)
    check(flat(vc)[:, :L], vref[:, :L], 0.0, "v_cache")
    assert bool((flat(kc)[:, L:] == 7).all()) and bool((flat(vc)[:, L:] == 7).all())


@pytest.mark.parametrize("dtype,L", [("fp32", 130), ("bf16", 300)])
def test_prefill_then_decode_matches_forward(cuda_lib, dtype, L):
    """Hand off L prompt tokens, decode four more: each output equals the forward oracle's row."""
    from softmax_attention_chunk_gb300 import path_attn as pa

    steps = 4
    inp = gen_path_inputs(1, 2, L + steps, 64, dtype, seed=600 + L, near2_frac=0.05)
    head = {n: inp[n][:, :, :L].contiguous() for n in ("k", "v", "w", "beta")}
    kc, vc = run_prefill(head, dtype, L + steps)
    o_ref, _ = orc.fwd(flat(inp["q"]), flat(inp["k"]), flat(inp["v"]), flat(inp["w"]), flat(inp["beta"]), None, 0.8)
    t = {n: inp[n].to(DEV) for n in ("q", "k", "v", "w", "beta")}
    for s in range(steps):
        pos = L + s
        o = pa.decode_step(kc, vc, pos, *(t[n][:, :, pos].contiguous() for n in ("q", "k", "v", "w", "beta")),
                           scale=0.8)
        torch.cuda.synchronize()
        if dtype == "fp32":
            check(flat(o), o_ref[:, pos], 1e-4, f"o[{pos}]")
        else:
            check(flat(o), o_ref[:, pos], 2e-2, f"o[{pos}]", rel=2e-2)


# ---------------- PaTH-FoX decode ----------------

@pytest.mark.parametrize("dtype,t0,steps,tol", [("fp32", 0, 30, 1e-4), ("fp32", 3000, 5, 1e-4), ("bf16", 2000, 5, 2e-2)])
def test_fox_decode_steps(cuda_lib, dtype, t0, steps, tol):
    """Forget-gate decode against the oracle step by step (outputs, rewritten keys, prefix cache)."""
    from softmax_attention_chunk_gb300 import path_attn as pa

    di = gen_decode_inputs(1, 3, 64, t0=t0, steps=steps, dtype=dtype, seed=71 + t0, fox=True)
    kc, vc, ac = di["k_cache"].to(DEV), di["v_cache"].to(DEV), di["a_cache"].to(DEV)
    kref, vref = np64(flat(di["k_cache"])).copy(), np64(flat(di["v_cache"])).copy()
    aref = np64(flat(di["a_cache"])).copy()
    for s in range(steps):
        x = {n: di[n][s].to(DEV) for n in ("q", "k", "v", "w", "beta", "log_f")}
        o = pa.decode_step_fox(kc, vc, ac, t0 + s, x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"], scale=1.0)
        torch.cuda.synchronize()
        o_r = orc.decode_step_fox(kref, vref, aref, t0 + s, *(flat(di[n][s]) for n in ("q", "k", "v", "w", "beta")),
                                  flat(di["log_f"][s]), 1.0)
        check(flat(o), o_r, tol, f"o[{s}]", rel=2e-2 if dtype == "bf16" else None)
    n = t0 + steps
    check(flat(kc)[:, :n], kref[:, :n], tol, "k_cache")
    check(flat(ac)[:, :n], aref[:, :n], 1e-3, "a_cache")


@pytest.mark.parametrize("dtype,L", [("fp32", 130), ("bf16", 300)])
def test_fox_prefill_then_decode_matches_forward(cuda_lib, dtype, L):
    """Hand off L FoX prompt tokens (keys and forget-gate prefix sums), decode four more: each
    output equals the FoX forward oracle's row."""
    from softmax_attention_chunk_gb300 import path_attn as pa

    steps = 4
    inp = gen_path_inputs(1, 2, L + steps, 64, dtype, seed=700 + L, near2_frac=0.05, fox=True)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    kc = torch.zeros(1, 2, L + steps, 64, dtype=tdt, device=DEV)
    vc = torch.zeros_like(kc)
    ac = torch.zeros(1, 2, L + steps, dtype=torch.float32, device=DEV)
    t = {n: inp[n].to(DEV) for n in ("q", "k", "v", "w", "beta", "log_f")}
    head = {n: t[n][:, :, :L].contiguous() for n in ("k", "v", "w", "beta", "log_f")}
    pa.decode_prefill(kc, vc, head["k"], head["v"], head["w"], head["beta"], log_f=head["log_f"], a_cache=ac)
    o_ref, _ = orc.fwd(flat(inp["q"]), flat(inp["k"]), flat(inp["v"]), flat(inp["w"]), flat(inp["beta"]),
                       flat(inp["log_f"]), 0.8)
    for s in range(steps):
        pos = L + s
        o = pa.decode_step_fox(kc, vc, ac, pos, *(t[n][:, :, pos].contiguous() for n in ("q", "k", "v", "w", "beta",
                                                                                           "log_f")), scale=0.8)
        torch.cuda.synchronize()
        if dtype == "fp32":
            check(flat(o), o_ref[:, pos], 1e-4, f"o[{pos}]")
        else:
            check(flat(o), o_ref[:, pos], 2e-2, f"o[{pos}]", rel=2e-2)



# ---------------- PaTH-FoX backward (bf16 tensor-core path) ----------------

def check_grads_fox(inp, g, scale, tol, rel):
    ref = orc.bwd(flat(inp["q"]), flat(inp["k"]), flat(inp["v"]), flat(inp["w"]), flat(inp["beta"]),
                  flat(inp["log_f"]), scale, flat(inp["dO"]), want_dlogf=True)
    for key in ("dq", "dk", "dv", "dw", "dbeta", "dlog_f"):
        r = ref[key]
        check(flat(g[key]), r, tol * max(1.0, np.abs(r).max()), key, rel=rel)


@pytest.mark.parametrize("L", [1, 64, 65, 200, 333])
def test_bwd_bf16_fox(cuda_lib, L):
    """Forget-gate backward: every gradient including dlog f against the oracle (whose dlog f is
    pinned by finite differences)."""
    from softmax_attention_chunk_gb300 import path_attn as pa

    inp = gen_path_inputs(2, 2, L, 64, "bf16", seed=800 + L, with_dO=True, near2_frac=0.05, fox=True)
    t = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    o, lse = pa.fwd(t["q"], t["k"], t["v"], t["w"], t["beta"], t["log_f"], scale=1.0)
    g = pa.bwd(t["q"], t["k"], t["v"], t["w"], t["beta"], o, lse, t["dO"], scale=1.0, log_f=t["log_f"])
    torch.cuda.synchronize()
    check_grads_fox(inp, g, 1.0, 2e-2, 3e-2)


def test_bwd_bf16_fox_training_step_reuse(cuda_lib):
    """Forget gate through the training-step path: the forward stores the transported queries and
    the backward reuses them and the preparation."""
    from softmax_attention_chunk_gb300 import path_attn as pa

    inp = gen_path_inputs(2, 9, 300, 64, "bf16", seed=901, with_dO=True, near2_frac=0.05, fox=True)
    t = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    desc = pa.make_desc(t["q"], 0.7)
    ws = pa.workspace(desc, 1, DEV)
    o, lse = pa.fwd(t["q"], t["k"], t["v"], t["w"], t["beta"], t["log_f"], 0.7, ws=ws,
                    phases=pa.PATH_FWD_ALL | pa.PATH_FWD_STORE_Z)
    g = pa.bwd(t["q"], t["k"], t["v"], t["w"], t["beta"], o, lse, t["dO"], 0.7, ws=ws, log_f=t["log_f"],
               phases=pa.PATH_BWD_ALL | pa.PATH_BWD_REUSE_FWD | pa.PATH_BWD_Z_FROM_FWD)
    torch.cuda.synchronize()
    check_grads_fox(inp, g, 0.7, 2e-2, 3e-2)


# ---------------- head dim 128 (fp32 SIMT kernels, 32-row chunks; decode) ----------------

@pytest.mark.parametrize("L,fox", [(1, False), (33, False), (100, False), (200, True)])
def test_fwd_d128_fp32(cuda_lib, L, fox):
    """Head dim 128 in the fp32 mode: outputs and lse within 1e-4 of the oracle (F is 128 x 128)."""
    inp = gen_path_inputs(1, 2, L, 128, "fp32", seed=700 + L, near2_frac=0.1, fox=fox)
    o, lse = run_fwd(inp, 1.0)
    o_ref, lse_ref = oracle_fwd(inp, 1.0)
    check(flat(o), o_ref, 1e-4, "o")
    check(flat(lse), lse_ref, 1e-4, "lse")


def test_fwd_d128_bf16(cuda_lib):
    inp = gen_path_inputs(2, 2, 300, 128, "bf16", seed=710, near2_frac=0.05)
    o, lse = run_fwd(inp, 1.0)
    o_ref, lse_ref = oracle_fwd(inp, 1.0)
    check(flat(o), o_ref, 2e-2, "o", rel=2e-2)
    check(flat(lse), lse_ref, 2e-2, "lse")


@pytest.mark.parametrize("L", [31, 100])
def test_bwd_d128_fp32(cuda_lib, L):
    inp = gen_path_inputs(1, 2, L, 128, "fp32", seed=720 + L, with_dO=True, near2_frac=0.1)
    g = run_bwd(inp, 1.0)
    check_grads(inp, g, 1.0, 1e-4)


def test_bwd_d128_fp32_fox(cuda_lib):
    from softmax_attention_chunk_gb300 import path_attn as pa

    inp = gen_path_inputs(1, 2, 90, 128, "fp32", seed=731, with_dO=True, near2_frac=0.1, fox=True)
    t = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    o, lse = pa.fwd(t["q"], t["k"], t["v"], t["w"], t["beta"], t["log_f"], scale=1.0)
    g = pa.bwd(t["q"], t["k"], t["v"], t["w"], t["beta"], o, lse, t["dO"], scale=1.0, log_f=t["log_f"])
    torch.cuda.synchronize()
    check_grads_fox(inp, g, 1.0, 1e-4, None)


def test_bwd_d128_bf16(cuda_lib):
    inp = gen_path_inputs(1, 2, 200, 128, "bf16", seed=740, with_dO=True, near2_frac=0.05)
    g = run_bwd(inp, 1.0)
    check_grads(inp, g, 1.0, 2e-2, rel=3e-2)


@pytest.mark.parametrize("dtype,t0,steps,tol", [("fp32", 0, 20, 1e-4), ("fp32", 3000, 4, 1e-4),
                                                ("bf16", 4000, 4, 2e-2)])
def test_decode_d128_steps(cuda_lib, dtype, t0, steps, tol):
    """Decode at head dim 128 (16 lanes per key) against the oracle step by step."""
    from softmax_attention_chunk_gb300 import path_attn as pa

    B, H, d = 2, 2, 128
    di = gen_decode_inputs(B, H, d, t0=t0, steps=steps, dtype=dtype, seed=750 + t0)
    kc, vc = di["k_cache"].to(DEV), di["v_cache"].to(DEV)
    kref = np64(di["k_cache"]).reshape(B * H, -1, d).copy()
    vref = np64(di["v_cache"]).reshape(B * H, -1, d).copy()
    for s in range(steps):
        args = [di[n][s].to(DEV) for n in ("q", "k", "v", "w", "beta")]
        o_t = pa.decode_step(kc, vc, t0 + s, *args, scale=1.0)
        torch.cuda.synchronize()
        o_r = orc.decode_step(kref, vref, t0 + s, *[flat(di[n][s]) for n in ("q", "k", "v", "w", "beta")], 1.0)
        check(o_t.reshape(B * H, d), o_r, tol, f"o_t step {s}", rel=2e-2 if dtype == "bf16" else None)
    n = t0 + steps
    check(kc.reshape(B * H, -1, d)[:, :n], kref[:, :n], tol, "rewritten keys")
    check(vc.reshape(B * H, -1, d)[:, :n], vref[:, :n], 0.0, "values")


def test_fox_decode_d128_steps(cuda_lib):
    from softmax_attention_chunk_gb300 import path_attn as pa

    t0, steps = 2000, 4
    di = gen_decode_inputs(1, 3, 128, t0=t0, steps=steps, dtype="fp32", seed=761, fox=True)
    kc, vc, ac = di["k_cache"].to(DEV), di["v_cache"].to(DEV), di["a_cache"].to(DEV)
    kref, vref = np64(flat(di["k_cache"])).copy(), np64(flat(di["v_cache"])).copy()
    aref = np64(flat(di["a_cache"])).copy()
    for s in range(steps):
        x = {n: di[n][s].to(DEV) for n in ("q", "k", "v", "w", "beta", "log_f")}
        o = pa.decode_step_fox(kc, vc, ac, t0 + s, x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"], scale=1.0)
        torch.cuda.synchronize()
        o_r = orc.decode_step_fox(kref, vref, aref, t0 + s, *(flat(di[n][s]) for n in ("q", "k", "v", "w", "beta")),
                                  flat(di["log_f"][s]), 1.0)
        check(flat(o), o_r, 1e-4, f"o[{s}]")
    check(flat(kc)[:, :t0 + steps], kref[:, :t0 + steps], 1e-4, "k_cache")


def test_decode_d128_matches_forward_rows(cuda_lib):
    """At head dim 128 too, decoding token by token from an empty cache gives the forward's rows."""
    from softmax_attention_chunk_gb300 import path_attn as pa

    L = 40
    inp = gen_path_inputs(1, 2, L, 128, "fp32", seed=771)
    o_f, _ = run_fwd(inp, 1.0)
    kc = torch.zeros(1, 2, L, 128, device=DEV)
    vc = torch.zeros_like(kc)
    rows = []
    for t in range(L):
        sl = lambda x: x[:, :, t].contiguous().to(DEV)
        rows.append(pa.decode_step(kc, vc, t, sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["w"]),
                                   sl(inp["beta"]), scale=1.0))
    o_d = torch.stack(rows, 2)
    assert (o_d - o_f).abs().max().item() <= 1e-4


@pytest.mark.parametrize("dtype,L", [("fp32", 1), ("fp32", 33), ("fp32", 200), ("bf16", 150)])
def test_prefill_d128_cache_matches_oracle(cuda_lib, dtype, L):
    """Hand-off at head dim 128 (fp32 preparation on 32-row chunks, 128 x 128 suffix products):
    keys transported to the prompt end, values copied, rows >= L untouched."""
    inp = gen_path_inputs(1, 2, L, 128, dtype, seed=800 + L, near2_frac=0.05)
    cap = L + 5
    kc, vc = run_prefill(inp, dtype, cap)
    kref, vref = orc.prefill_cache(flat(inp["k"]), flat(inp["v"]), flat(inp["w"]), flat(inp["beta"]), cap)
    if dtype == "fp32":
        check(flat(kc)[:, :L], kref[:, :L], 1e-4, "k_cache")
    else:
        check(flat(kc)[:, :L], kref[:, :L], 2e-2 * np.abs(kref).max(), "k_cache", rel=2e-2)
    check(flat(vc)[:, :L], vref[:, :L], 0.0, "v_cache")
    assert bool((flat(kc)[:, L:] == 7).all()) and bool((flat(vc)[:, L:] == 7).all())


def test_prefill_d128_then_decode_matches_forward(cuda_lib):
    from softmax_attention_chunk_gb300 import path_attn as pa

    L, steps = 70, 3
    inp = gen_path_inputs(1, 2, L + steps, 128, "fp32", seed=811, near2_frac=0.05)
    head = {n: inp[n][:, :, :L].contiguous() for n in ("k", "v", "w", "beta")}
    kc, vc = run_prefill(head, "fp32", L + steps)
    o_ref, _ = orc.fwd(flat(inp["q"]), flat(inp["k"]), flat(inp["v"]), flat(inp["w"]), flat(inp["beta"]), None, 1.0)
    t = {n: inp[n].to(DEV) for n in ("q", "k", "v", "w", "beta")}
    for s in range(steps):
        pos = L + s
        o = pa.decode_step(kc, vc, pos, *(t[n][:, :, pos].contiguous() for n in ("q", "k", "v", "w", "beta")),
                           scale=1.0)
        torch.cuda.synchronize()
        check(flat(o), o_ref[:, pos], 1e-4, f"o[{pos}]")
