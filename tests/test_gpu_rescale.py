"""The forward scans' lazy rescale of the running output.

A query row starts the scan with the maximum of its own (diagonal) chunk's scores and lowers
the output's reference only when a key chunk visited later raises that maximum by more than
8 log2 units; the rescale then multiplies the row's running output in TMEM.  With scores of
about unit size (the workloads' q, k ~ N(0, 1)/sqrt(d) at scale 1) that never happens, so these
cases use a large score scale (score standard deviation 5 to 10 nats): rows whose own chunk holds few
keys then meet far larger scores in earlier chunks, at different steps for different rows of
one warp.  Each case first counts, from the oracle's explicit logits of one head, the rows that
must rescale, then compares the tensor-core forward (head dims 64 and 128, either sign of the
scale, with and without the forget gate, the training forward that stores Z, and the
context-parallel chain whose scan runs over the other shards' key blocks) with the oracle.

Tolerance: the scores here are |scale| times those of the same inputs at scale 1, and the bf16
rounding of the transported queries and keys perturbs each score by a relative amount, so the
absolute score error, and with it the lse error and the misweighting of the values in o, grow
in proportion to |scale|.  o is held to 2e-2 max abs (as every bf16 output) and to a relative
Frobenius error of 2e-2 * max(1, |scale| / 20); lse to 2e-2 * |scale| / 8.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from softmax_attention_chunk_gb300.inputs import gen_path_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
KTAU_NATS = 8.0 * math.log(2.0)  # the scans' rescale threshold, 8 log2 units


def np64(x):
    return x.detach().double().cpu().numpy()


def flat(x):
    return None if x is None else x.reshape(-1, *x.shape[2:])


def rows_that_rescale(inp, head, scale, chunk=64):
    """Rows of one head whose earlier keys score more than the threshold above the row's own
    chunk maximum (each rescales at least once)."""
    args = [flat(inp[n])[head] for n in ("q", "k", "w", "beta")]
    lf = None if inp["log_f"] is None else flat(inp["log_f"])[head]
    S = orc.logits(*args, log_f=lf, scale=scale)
    n = 0
    for i in range(S.shape[0]):
        c0 = (i // chunk) * chunk
        if c0 == 0:
            continue
        if S[i, :c0].max() > S[i, c0:i + 1].max() + KTAU_NATS:
            n += 1
    return n


def check_fwd(inp, o, lse, scale, case, record_margin):
    args = [flat(inp[n]) for n in ("q", "k", "v", "w", "beta", "log_f")]
    o_ref, lse_ref = orc.fwd(*args, scale)
    got = np64(flat(o))
    err = np.abs(got - o_ref).max()
    rel = np.linalg.norm(got - o_ref) / np.linalg.norm(o_ref)
    lerr = np.abs(np64(flat(lse)) - lse_ref).max()
    rbound = 2e-2 * max(1.0, abs(scale) / 20.0)
    lbound = 2e-2 * abs(scale) / 8.0
    record_margin(case, "o", err, 2e-2, rel=rel)
    record_margin(case, "lse", lerr, lbound)
    assert err <= 2e-2 and rel <= rbound, (err, rel, rbound)
    assert lerr <= lbound, (lerr, lbound)


@pytest.mark.parametrize("d,scale,fox", [(64, 40.0, False), (64, -40.0, False), (64, 60.0, True),
                                         (128, 56.0, False), (128, -84.0, True)])
def test_fwd_lazy_rescale(cuda_lib, record_margin, d, scale, fox):
    from softmax_attention_chunk_gb300 import path_attn as pa

    B, H, L = 1, 3, 392
    inp = gen_path_inputs(B, H, L, d, "bf16", seed=3400 + d + (scale < 0) + 2 * fox, near2_frac=0.05, fox=fox)
    nresc = rows_that_rescale(inp, 0, scale)
    assert nresc >= 8, f"the case exercises too few rescales ({nresc} rows)"
    t = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    o, lse = pa.fwd(t["q"], t["k"], t["v"], t["w"], t["beta"], t["log_f"], scale=scale, check=True)
    torch.cuda.synchronize()
    case = f"lazy rescale d{d} scale {scale}{' FoX' if fox else ''} ({nresc} rows of head 0 rescale)"
    check_fwd(inp, o, lse, scale, case, record_margin)


def test_training_forward_lazy_rescale(cuda_lib, record_margin):
    """The forward that also stores the transported query tiles (the training step's)."""
    from softmax_attention_chunk_gb300 import path_attn as pa

    B, H, L, scale = 1, 2, 456, 40.0
    inp = gen_path_inputs(B, H, L, 64, "bf16", seed=3411, near2_frac=0.05)
    assert rows_that_rescale(inp, 1, scale) >= 8
    t = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    desc = pa.make_desc(t["q"], scale)
    ws = pa.workspace(desc, 1, DEV)
    o, lse = pa.fwd(t["q"], t["k"], t["v"], t["w"], t["beta"], None, scale, ws=ws,
                    phases=pa.PATH_FWD_ALL | pa.PATH_FWD_STORE_Z, check=True)
    torch.cuda.synchronize()
    check_fwd(inp, o, lse, scale, f"lazy rescale, training forward (Z stored), scale {scale}", record_margin)


def test_context_parallel_chain_lazy_rescale(cuda_lib, record_margin):
    """The context-parallel chain (the scan in its block mode over the other shards' key blocks)."""
    from softmax_attention_chunk_gb300.context_parallel import ShardOps, emulate_ring

    B, H, L, world, scale = 1, 2, 512, 4, 40.0
    inp = gen_path_inputs(B, H, L, 64, "bf16", seed=3421, near2_frac=0.05)
    assert rows_that_rescale(inp, 0, scale) >= 8
    Ls = L // world
    ops = []
    for r in range(world):
        sl = slice(r * Ls, (r + 1) * Ls)
        s = {n: (None if t is None else t[:, :, sl].contiguous().to(DEV)) for n, t in inp.items()}
        ops.append(ShardOps(s["q"], s["k"], s["v"], s["w"], s["beta"], s["log_f"], scale))
    res = emulate_ring(ops)
    torch.cuda.synchronize()
    for op in ops:
        cuda_lib.check_workspace(op.desc, 0, op.ws)
    o = torch.cat([r[0] for r in res], dim=2)
    lse = torch.cat([r[1] for r in res], dim=2)
    check_fwd(inp, o, lse, scale, f"lazy rescale, context-parallel chain over {world} shards, scale {scale}",
              record_margin)
