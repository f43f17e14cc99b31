"""Failure path of the tensor-core kernels, made to run without a fault.

Every wait of those kernels on their pipeline barriers is bounded; a wait that gives up records a
code in the workspace, its kernel ends early, and path_attn_workspace_status reports
PATH_ERR_INTERNAL.  PATH_ATTN_DEBUG_STALL_NS makes the forward's preparation wait on a barrier
that nothing arrives at (a flag nobody sets) for a short limit, before any copy or MMA has been
issued, so nothing is left in flight when the kernel ends.  The context must stay usable: the
same workspace then runs a normal forward whose output matches the oracle.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from softmax_attention_chunk_gb300.inputs import gen_path_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_a_wait_that_gives_up_is_reported_and_the_context_survives(cuda_lib, monkeypatch):
    pa = cuda_lib
    inp = gen_path_inputs(1, 2, 300, 64, "bf16", seed=77)
    t = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    desc = pa.make_desc(t["q"], 1.0)
    ws = pa.workspace(desc, 0, DEV)
    stream = torch.cuda.current_stream().cuda_stream
    args = (t["q"], t["k"], t["v"], t["w"], t["beta"], None, 1.0)
    # a clean run reads PATH_OK
    pa.fwd(*args, ws=ws, check=True)
    assert pa.path_attn_workspace_status(desc, 0, ws.data_ptr(), ws.numel(), stream) == (pa.PATH_OK, 0)
    # the forced stall: every preparation CTA gives up after 2 ms and records code 99
    monkeypatch.setenv("PATH_ATTN_DEBUG_STALL_NS", "2000000")
    pa.fwd(*args, ws=ws, phases=pa.PATH_FWD_PREPARE)
    rc, code = pa.path_attn_workspace_status(desc, 0, ws.data_ptr(), ws.numel(), stream)
    assert (rc, code) == (pa.PATH_ERR_INTERNAL, 99), (pa.path_status_string(rc), code)
    with pytest.raises(RuntimeError, match="PATH_ERR_INTERNAL"):
        pa.check_workspace(desc, 0, ws)
    monkeypatch.delenv("PATH_ATTN_DEBUG_STALL_NS")
    # the next forward on the same workspace clears the word, runs normally and is correct
    o, lse = pa.fwd(*args, ws=ws, check=True)
    torch.cuda.synchronize()
    flat = lambda x: x.reshape(-1, *x.shape[2:])
    o_ref, lse_ref = orc.fwd(flat(inp["q"]), flat(inp["k"]), flat(inp["v"]), flat(inp["w"]), flat(inp["beta"]),
                             None, 1.0)
    assert np.abs(flat(o).double().cpu().numpy() - o_ref).max() <= 2e-2
    assert np.abs(flat(lse).double().cpu().numpy() - lse_ref).max() <= 2e-2


def test_prefill_status_reads_ok_after_a_normal_hand_off(cuda_lib):
    pa = cuda_lib
    inp = gen_path_inputs(1, 2, 200, 64, "bf16", seed=78)
    t = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    kc = torch.zeros(1, 2, 256, 64, dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    desc = pa.make_decode_desc(kc, 1.0)
    ws = torch.empty(pa.path_decode_prefill_workspace_size(desc, 200), dtype=torch.uint8, device=DEV)
    pa.decode_prefill(kc, vc, t["k"], t["v"], t["w"], t["beta"], ws=ws)
    stream = torch.cuda.current_stream().cuda_stream
    assert pa.path_decode_prefill_status(desc, 200, ws.data_ptr(), ws.numel(), stream) == (pa.PATH_OK, 0)
