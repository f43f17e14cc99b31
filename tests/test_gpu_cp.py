"""Context-parallel forward on the GPU, the ranks emulated in one process.

The shards of one sequence are prepared on the one device (ShardOps: the forward's PREPARE phase and
path_cp_shard_prepare through the C ABI), the chain's messages are copies of the sender's block
(emulate_ring: the schedule the multi-rank run uses, without collectives), and every shard's rows
must match the oracle's forward over the whole sequence within the bf16 tolerance.  The per-shard
transports are also checked on their own: the keys moved to the shard end against the oracle's
hand-off rows, the shard product against explicit products.
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


def shards(inp, world):
    L = inp["q"].shape[2]
    Ls = L // world
    out = []
    for r in range(world):
        sl = slice(r * Ls, (r + 1) * Ls)
        out.append({n: (None if t is None else t[:, :, sl].contiguous().to(DEV)) for n, t in inp.items()})
    return out


@pytest.mark.parametrize("B,H,L,world,fox", [(1, 2, 512, 4, False), (1, 2, 768, 3, True), (2, 4, 2048, 4, False),
                                             (1, 3, 1024, 2, True)])
def test_emulated_chain_matches_the_full_forward(cuda_lib, record_margin, B, H, L, world, fox):
    from softmax_attention_chunk_gb300.context_parallel import ShardOps, emulate_ring

    inp = gen_path_inputs(B, H, L, 64, "bf16", seed=900 + L + world, near2_frac=0.05, fox=fox)
    ops = [ShardOps(s["q"], s["k"], s["v"], s["w"], s["beta"], s["log_f"], 1.0) for s in shards(inp, world)]
    res = emulate_ring(ops)
    torch.cuda.synchronize()
    for op in ops:
        cuda_lib.check_workspace(op.desc, 0, op.ws)
    o = torch.cat([r[0] for r in res], dim=2)
    lse = torch.cat([r[1] for r in res], dim=2)
    o_ref, lse_ref = orc.fwd(flat(inp["q"]), flat(inp["k"]), flat(inp["v"]), flat(inp["w"]), flat(inp["beta"]),
                             flat(inp["log_f"]), 1.0)
    got, gl = np64(flat(o)), np64(flat(lse))
    err, rel = np.abs(got - o_ref).max(), np.linalg.norm(got - o_ref) / np.linalg.norm(o_ref)
    lerr = np.abs(gl - lse_ref).max()
    case = f"context parallel B{B} H{H} L{L} over {world} shards{' FoX' if fox else ''}"
    record_margin(case, "o", err, 2e-2, rel=rel)
    record_margin(case, "lse", lerr, 2e-2)
    assert err <= 2e-2 and rel <= 2e-2 and lerr <= 2e-2, (err, rel, lerr)
    # and the single-device forward over the whole sequence agrees row for row
    full = {n: (None if t is None else t.to(DEV)) for n, t in inp.items()}
    o1, l1 = cuda_lib.fwd(full["q"], full["k"], full["v"], full["w"], full["beta"], full["log_f"], 1.0)
    assert (o1.float() - o.float()).abs().max().item() <= 2e-2
    assert (l1 - lse).abs().max().item() <= 2e-2


def test_shard_transports_match_the_definitions(cuda_lib):
    from softmax_attention_chunk_gb300.context_parallel import ShardOps

    inp = gen_path_inputs(1, 2, 256, 64, "bf16", seed=931, near2_frac=0.1)
    s = {n: (None if t is None else t.to(DEV)) for n, t in inp.items()}
    op = ShardOps(s["q"], s["k"], s["v"], s["w"], s["beta"], None, 1.0)
    torch.cuda.synchronize()
    k, w, beta = flat(inp["k"]), flat(inp["w"]), flat(inp["beta"])
    kref, _ = orc.prefill_cache(k, flat(inp["v"]), w, beta, 256)  # rows H_{L-1} ... H_{j+1} k_j
    got = np64(flat(op.k_end))
    assert np.abs(got - kref).max() <= 2e-2 * np.abs(kref).max()
    assert np.linalg.norm(got - kref) / np.linalg.norm(kref) <= 2e-2
    wn, bn = np64(w), np64(beta).clip(0.0, 2.0)
    for h in range(2):
        M = np.eye(64)
        for t in range(256):
            M = M @ (np.eye(64) - bn[h, t] * np.outer(wn[h, t], wn[h, t]))
        assert np.abs(np64(op.t[0, h]) - M.T).max() <= 2e-2
