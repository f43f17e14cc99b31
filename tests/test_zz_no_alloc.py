"""The decode step for callers that cannot allocate device memory.

Code that runs inside someone else's memory pool, plugins restricted to the buffers they are
handed, and serving loops that forbid allocation after start-up cannot provide the workspace
path_decode_step asks for.  path_decode_step_noalloc keeps that scratch in an array built into
the library.  These tests call it through the C ABI and check that it gives the same results as
path_decode_step on two calls in a row.  The file is named so that pytest collects it last.
"""
import pytest
import torch

from softmax_attention_chunk_gb300.inputs import gen_decode_inputs

FAKE = 1 << 20  # aligned address that is never dereferenced (the call is rejected first)


def test_noalloc_rejects_more_heads_than_its_scratch_holds():
    from softmax_attention_chunk_gb300 import build_lib

    build_lib.build()
    from softmax_attention_chunk_gb300 import path_attn as pa

    too_many = pa.path_decode_desc_t(1, pa.PATH_DECODE_NOALLOC_MAX_HEADS + 1, 64, 16, pa.PATH_BF16, 1.0)
    assert pa.path_decode_step_noalloc(too_many, *([FAKE] * 2), 3, *([FAKE] * 6), None) == 3  # WORKSPACE
    ok = pa.path_decode_desc_t(1, 2, 64, 16, pa.PATH_BF16, 1.0)
    assert pa.path_decode_step_noalloc(ok, None, FAKE, 3, *([FAKE] * 6), None) == 1
    assert pa.path_decode_step_noalloc(ok, FAKE, FAKE, 16, *([FAKE] * 6), None) == 4


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,tol", [("bf16", 2e-2), ("fp32", 1e-4)])
def test_noalloc_matches_workspace_decode_on_two_calls(dtype, tol):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from softmax_attention_chunk_gb300 import path_attn as pa

    dev = "cuda"
    B, H, d, t0 = 2, 3, 64, 3000
    di = gen_decode_inputs(B, H, d, t0=t0, steps=2, dtype=dtype, seed=123)
    kc_a, vc_a = di["k_cache"].to(dev), di["v_cache"].to(dev)
    kc_b, vc_b = kc_a.clone(), vc_a.clone()
    desc = pa.make_decode_desc(kc_a, 1.0)
    ws = pa.decode_workspace(desc, dev)
    stream = torch.cuda.current_stream().cuda_stream
    for s in range(2):
        q, k, v, w, beta = (di[n][s].to(dev) for n in ("q", "k", "v", "w", "beta"))
        o_ref = torch.empty(B, H, d, dtype=kc_a.dtype, device=dev)
        o_new = torch.full_like(o_ref, float("nan"))
        rc = pa.path_decode_step(desc, kc_a.data_ptr(), vc_a.data_ptr(), t0 + s, q.data_ptr(), k.data_ptr(),
                                 v.data_ptr(), w.data_ptr(), beta.data_ptr(), o_ref.data_ptr(), ws.data_ptr(),
                                 ws.numel(), stream)
        assert rc == 0, pa.path_status_string(rc)
        rc = pa.path_decode_step_noalloc(desc, kc_b.data_ptr(), vc_b.data_ptr(), t0 + s, q.data_ptr(),
                                         k.data_ptr(), v.data_ptr(), w.data_ptr(), beta.data_ptr(),
                                         o_new.data_ptr(), stream)
        assert rc == 0, pa.path_status_string(rc)
        torch.cuda.synchronize()
        assert torch.isfinite(o_new).all()
        assert (o_new.float() - o_ref.float()).abs().max().item() <= tol
        assert (kc_b.float() - kc_a.float()).abs().max().item() <= tol
        assert torch.equal(vc_b, vc_a)
