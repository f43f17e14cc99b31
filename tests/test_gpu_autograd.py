"""The torch.autograd binding (softmax_attention_chunk_gb300.autograd.path_attention): gradients of a
scalar loss through the library's training forward and backward against the oracle's, on the
bf16 tensor-core path (plain and PaTH-FoX, dlog f included), the fp32 mode and head dim 128."""
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


@pytest.mark.parametrize("dtype,d,fox,tol", [("bf16", 64, False, 2e-2), ("bf16", 64, True, 2e-2),
                                             ("fp32", 64, False, 1e-4), ("bf16", 128, False, 2e-2)])
def test_autograd_gradients_match_the_oracle(cuda_lib, dtype, d, fox, tol):
    from softmax_attention_chunk_gb300.autograd import path_attention

    inp = gen_path_inputs(1, 2, 200, d, dtype, seed=3400 + d + fox, with_dO=True, near2_frac=0.05, fox=fox)
    names = ("q", "k", "v", "w", "beta") + (("log_f",) if fox else ())
    t = {n: inp[n].to(DEV).requires_grad_(True) for n in names}
    dO = inp["dO"].to(DEV)
    o = path_attention(t["q"], t["k"], t["v"], t["w"], t["beta"], t.get("log_f"), scale=0.9)
    loss = (o.float() * dO.float()).sum()
    grads = torch.autograd.grad(loss, [t[n] for n in names])
    torch.cuda.synchronize()
    o_ref, _ = orc.fwd(*[flat(inp[n]) for n in ("q", "k", "v", "w", "beta", "log_f")], 0.9)
    assert np.abs(np64(flat(o)) - o_ref).max() <= tol
    ref = orc.bwd(*[flat(inp[n]) for n in ("q", "k", "v", "w", "beta", "log_f")], 0.9, flat(inp["dO"]),
                  want_dlogf=fox)
    keys = {"q": "dq", "k": "dk", "v": "dv", "w": "dw", "beta": "dbeta", "log_f": "dlog_f"}
    for n, gr in zip(names, grads):
        r = ref[keys[n]]
        err = np.abs(np64(flat(gr)) - r).max()
        assert err <= tol * max(1.0, np.abs(r).max()), (n, err)
