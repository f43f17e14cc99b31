"""Host-side checks of the C ABI that need no GPU: the library loads, exports every function
include/path_attn.h declares, and rejects bad arguments with the documented status before any
CUDA call.  Every call below fails validation, so nothing is ever launched (fake pointers are
never dereferenced)."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "path_attn.h")


@pytest.fixture(scope="module")
def pa():
    from softmax_attention_chunk_gb300 import build_lib

    build_lib.build()
    from softmax_attention_chunk_gb300 import path_attn

    return path_attn


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_]+\s*\**\s+(path_[a-z_]+)\s*\(", src, flags=re.M)))


def test_header_declares_the_three_path_calls():
    fns = declared_functions()
    for f in ("path_attn_fwd", "path_attn_bwd", "path_decode_step"):
        assert f in fns


def test_library_exports_every_declared_symbol(pa):
    lib = ctypes.CDLL(pa.LIB_PATH)
    for f in declared_functions():
        assert hasattr(lib, f), f
    assert sorted(pa.EXPORTED) == declared_functions()


def desc(pa, **kw):
    d = dict(batch=1, heads=2, seqlen=100, head_dim=64, dtype=pa.PATH_FP32, scale=1.0, chunk=0)
    d.update(kw)
    return pa.path_attn_desc_t(d["batch"], d["heads"], d["seqlen"], d["head_dim"], d["dtype"], d["scale"],
                               d["chunk"])


FAKE = 1 << 20  # aligned, never dereferenced


def test_status_strings(pa):
    for s in range(7):
        assert pa.path_status_string(s).startswith(pa.STATUS_NAMES[s])
    assert "unknown" in pa.path_status_string(99)


def test_descriptor_validation(pa):
    assert pa.path_attn_chunk(desc(pa), 0) == 64
    assert pa.path_attn_chunk(desc(pa, chunk=32), 0) == 32
    assert pa.path_attn_chunk(desc(pa), 1) > 0
    assert pa.path_attn_chunk(desc(pa, head_dim=96), 0) == -2           # unsupported head dim
    # head dim 128: fp32 (and every backward) runs the SIMT kernels, whose shared memory holds
    # 32-row chunks; the bf16 forward runs the head-dim-128 tensor-core kernels on 64-row chunks
    assert pa.path_attn_chunk(desc(pa, head_dim=128), 0) == 32
    assert pa.path_attn_chunk(desc(pa, head_dim=128, dtype=pa.PATH_BF16), 0) == 64
    assert pa.path_attn_chunk(desc(pa, head_dim=128, dtype=pa.PATH_BF16, chunk=32), 0) == 32
    assert pa.path_attn_chunk(desc(pa, head_dim=128, dtype=pa.PATH_BF16, chunk=64), 0) == 64
    assert pa.path_attn_chunk(desc(pa, head_dim=128, dtype=pa.PATH_BF16), 1) == 32
    assert pa.path_attn_chunk(desc(pa, head_dim=128, chunk=64), 0) == -2
    assert pa.path_attn_chunk(desc(pa, head_dim=128), 1) == 32
    assert pa.path_attn_workspace_size(desc(pa, head_dim=128), 1) > pa.path_attn_workspace_size(desc(pa), 1)
    assert pa.path_attn_chunk(desc(pa, head_dim=0), 0) == -1            # invalid
    assert pa.path_attn_chunk(desc(pa, seqlen=0), 0) == -1
    assert pa.path_attn_chunk(desc(pa, dtype=7), 0) == -1
    assert pa.path_attn_chunk(desc(pa, chunk=48), 0) == -2
    assert pa.path_attn_chunk(desc(pa, scale=float("nan")), 0) == -1
    assert pa.path_attn_workspace_size(desc(pa, head_dim=32), 0) == 0
    assert pa.path_attn_workspace_size(desc(pa), 0) > 0
    assert pa.path_attn_workspace_size(desc(pa), 1) > pa.path_attn_workspace_size(desc(pa), 0)
    # workspace grows with the problem
    assert pa.path_attn_workspace_size(desc(pa, seqlen=1000), 0) > pa.path_attn_workspace_size(desc(pa), 0)


def fwd_args(pa, d, ws_bytes=None, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, w=FAKE, beta=FAKE, log_f=None, o=FAKE, lse=FAKE, ws=FAKE,
             ws_bytes=pa.path_attn_workspace_size(d, 0) if ws_bytes is None else ws_bytes, stream=None)
    a.update(over)
    return a


def call_fwd(pa, d, **a):
    return pa.path_attn_fwd(d, a["q"], a["k"], a["v"], a["w"], a["beta"], a["log_f"], a["o"], a["lse"], a["ws"],
                            a["ws_bytes"], a["stream"])


def test_fwd_argument_errors(pa):
    d = desc(pa)
    ok_bytes = pa.path_attn_workspace_size(d, 0)
    assert call_fwd(pa, d, **fwd_args(pa, d, ws_bytes=ok_bytes - 1)) == 3          # workspace
    assert call_fwd(pa, d, **fwd_args(pa, d, q=None, ws_bytes=0)) == 1             # null
    assert call_fwd(pa, d, **fwd_args(pa, d, k=FAKE + 8, ws_bytes=0)) == 1         # misaligned
    assert call_fwd(pa, d, **fwd_args(pa, d, ws=FAKE + 16, ws_bytes=0)) == 1       # ws not 256-aligned
    assert call_fwd(pa, d, **fwd_args(pa, d, log_f=FAKE + 4, ws_bytes=0)) == 1
    assert call_fwd(pa, desc(pa, head_dim=96), **fwd_args(pa, d)) == 2
    d128 = desc(pa, head_dim=128)
    assert call_fwd(pa, d128, **fwd_args(pa, d128, ws_bytes=pa.path_attn_workspace_size(d128, 0) - 1)) == 3
    assert pa._lib.path_attn_fwd(None, *([FAKE] * 8), FAKE, 0, None) == 1
    for bad in (0, 4, 8):
        assert pa.path_attn_fwd_phases(bad, d, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, 0, None) in (1, 3)
    assert pa.path_attn_fwd_phases(0, d, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, ok_bytes, None) == 1


def test_bwd_argument_errors(pa):
    d = desc(pa)
    n = pa.path_attn_workspace_size(d, 1)
    args = [FAKE] * 6 + [None] + [FAKE] * 3 + [FAKE] * 5  # q k v w beta o? see order below
    # order: q,k,v,w,beta,log_f,o,lse,dO,dq,dk,dv,dw,dbeta,dlog_f,ws,ws_bytes,stream
    base = [FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE]
    assert pa.path_attn_bwd(d, *base, n - 1, None) == 3
    # forget gate: dlog f without log f, or a misaligned log f, is an argument error; the bf16
    # tensor-core path has no forget-gate backward at a zero scale (every check runs before any
    # launch: the pointers here are fake)
    with_dlogf = list(base); with_dlogf[14] = FAKE
    assert pa.path_attn_bwd(d, *with_dlogf, n, None) == 1
    with_logf = list(base); with_logf[5] = FAKE
    assert pa.path_attn_bwd(d, *with_logf, n - 1, None) == 3  # d is an fp32 descriptor
    odd_logf = list(with_logf); odd_logf[5] = FAKE + 4
    assert pa.path_attn_bwd(d, *odd_logf, n, None) == 1
    d0 = pa.path_attn_desc_t(d.batch, d.heads, d.seqlen, d.head_dim, pa.PATH_BF16, 0.0, d.chunk)
    assert pa.path_attn_bwd(d0, *with_logf, pa.path_attn_workspace_size(d0, 1), None) == 2
    null_dw = list(base); null_dw[12] = None
    assert pa.path_attn_bwd(d, *null_dw, n, None) == 1
    assert pa.path_attn_bwd_phases(8, d, *base, n, None) == 1
    del args


def test_decode_argument_errors(pa):
    dd = pa.path_decode_desc_t(2, 2, 64, 100, pa.PATH_BF16, 1.0)
    n = pa.path_decode_workspace_size(dd)
    assert n > 0
    vec = [FAKE] * 6
    assert pa.path_decode_step(dd, FAKE, FAKE, 100, *vec, FAKE, n, None) == 4     # t + 1 > capacity
    assert pa.path_decode_step(dd, FAKE, FAKE, -1, *vec, FAKE, n, None) == 1
    assert pa.path_decode_step(dd, FAKE, FAKE, 5, *vec, FAKE, n - 1, None) == 3
    assert pa.path_decode_step(dd, None, FAKE, 5, *vec, FAKE, n, None) == 1
    bad = pa.path_decode_desc_t(2, 2, 96, 100, pa.PATH_BF16, 1.0)
    assert pa.path_decode_workspace_size(bad) == 0
    assert pa.path_decode_step(bad, FAKE, FAKE, 5, *vec, FAKE, n, None) == 2
    # head dim 128: partials of 128 + 2 floats per split
    wide = pa.path_decode_desc_t(2, 2, 128, 100, pa.PATH_BF16, 1.0)
    n128 = pa.path_decode_workspace_size(wide)
    assert n128 > n
    assert pa.path_decode_step(wide, FAKE, FAKE, 5, *vec, FAKE, n128 - 1, None) == 3


def test_prefill_argument_errors(pa):
    """Prefill hand-off: every check runs before any CUDA call (FAKE pointers are never used)."""
    dd = pa.path_decode_desc_t(2, 2, 64, 100, pa.PATH_BF16, 1.0)
    n = pa.path_decode_prefill_workspace_size(dd, 70)
    assert n > 0 and n > pa.path_decode_prefill_workspace_size(dd, 10) > 0
    assert pa.path_decode_prefill_workspace_size(dd, 0) > 0            # an empty prompt is valid
    assert pa.path_decode_prefill_workspace_size(dd, 101) == 0         # longer than the cache
    assert pa.path_decode_prefill_workspace_size(dd, -1) == 0
    vec = [FAKE] * 4 + [None, None]
    assert pa.path_decode_prefill(dd, FAKE, FAKE, 101, *vec, FAKE, n, None) == 4   # prompt > capacity
    assert pa.path_decode_prefill(dd, FAKE, FAKE, -1, *vec, FAKE, n, None) == 1
    assert pa.path_decode_prefill(dd, FAKE, FAKE, 70, *vec, FAKE, n - 1, None) == 3
    assert pa.path_decode_prefill(dd, None, FAKE, 70, *vec, FAKE, n, None) == 1
    assert pa.path_decode_prefill(dd, FAKE, FAKE, 70, FAKE, FAKE, FAKE, None, None, None, FAKE, n, None) == 1
    assert pa.path_decode_prefill(dd, FAKE, FAKE, 70, *vec[:4], FAKE, None, FAKE, n, None) == 1  # log_f alone
    assert pa.path_decode_prefill(dd, FAKE, FAKE, 70, *vec[:4], None, FAKE, FAKE, n, None) == 1  # a_cache alone
    assert pa.path_decode_prefill(dd, FAKE, FAKE, 0, *vec, FAKE, n, None) == 0     # nothing to do
    bad = pa.path_decode_desc_t(2, 2, 96, 100, pa.PATH_BF16, 1.0)
    assert pa.path_decode_prefill_workspace_size(bad, 10) == 0
    assert pa.path_decode_prefill(bad, FAKE, FAKE, 10, *vec, FAKE, n, None) == 2
    wide = pa.path_decode_desc_t(2, 2, 128, 100, pa.PATH_BF16, 1.0)   # head dim 128: fp32 preparation
    n128 = pa.path_decode_prefill_workspace_size(wide, 70)
    assert n128 > n
    assert pa.path_decode_prefill(wide, FAKE, FAKE, 70, *vec, FAKE, n128 - 1, None) == 3


def test_fox_decode_argument_errors(pa):
    dd = pa.path_decode_desc_t(2, 2, 64, 100, pa.PATH_BF16, 1.0)
    n = pa.path_decode_workspace_size(dd)
    vec = [FAKE] * 7
    assert pa.path_decode_step_fox(dd, FAKE, FAKE, FAKE, 100, *vec, FAKE, n, None) == 4     # t + 1 > capacity
    assert pa.path_decode_step_fox(dd, FAKE, FAKE, FAKE, -1, *vec, FAKE, n, None) == 1
    assert pa.path_decode_step_fox(dd, FAKE, FAKE, FAKE, 5, *vec, FAKE, n - 1, None) == 3
    assert pa.path_decode_step_fox(dd, FAKE, FAKE, None, 5, *vec, FAKE, n, None) == 1      # no prefix cache
    assert pa.path_decode_step_fox(dd, FAKE, FAKE, FAKE, 5, *vec[:6], None, FAKE, n, None) == 1  # no o_t
    assert pa.path_decode_step_fox(dd, FAKE, FAKE, FAKE, 5, *vec[:5], None, FAKE, FAKE, n, None) == 1  # no log f


def test_torch_wrapper_rejects_bad_tensors(pa):
    q = torch.zeros(1, 1, 8, 64)
    with pytest.raises(ValueError):
        pa.fwd(q, q, q, q, torch.zeros(1, 1, 8), scale=1.0)  # CPU tensors are refused before any call


def test_input_generator_subsets_are_exact():
    from softmax_attention_chunk_gb300.inputs import gen_decode_inputs, gen_path_inputs

    full = gen_path_inputs(2, 3, 50, 64, "bf16", seed=4, near2_frac=0.3, fox=True, with_dO=True)
    sub = gen_path_inputs(2, 3, 50, 64, "bf16", seed=4, near2_frac=0.3, fox=True, with_dO=True,
                          heads_subset=[4, 1])
    for key in ("q", "k", "v", "w", "beta", "log_f", "dO"):
        f = full[key].reshape(6, *full[key].shape[2:])
        assert torch.equal(f[[4, 1]], sub[key]), key
    b = full["beta"]
    assert float(b.min()) > 0 and float(b.max()) < 2
    assert float(b.max()) >= 1.95  # the near-reflection tail is present
    w = full["w"].double()
    assert torch.allclose(w.norm(dim=-1), torch.ones(2, 3, 50, dtype=torch.float64), atol=1e-2)
    dfull = gen_decode_inputs(1, 3, 64, t0=10, steps=4, dtype="fp32", seed=2)
    dsub = gen_decode_inputs(1, 3, 64, t0=10, steps=4, dtype="fp32", seed=2, heads_subset=[2])
    assert torch.equal(dfull["k_cache"][0, 2], dsub["k_cache"][0])
    assert torch.equal(dfull["q"][:, 0, 2], dsub["q"][:, 0])
    assert torch.all(dfull["k_cache"][:, :, 10:] == 0)


def test_training_step_bits_are_validated(pa):
    """PATH_FWD_STORE_Z needs a backward-sized workspace on the bf16 tensor-core path; the new bits
    are accepted only next to a phase, and unknown bits are rejected."""
    d = desc(pa, dtype=pa.PATH_BF16)
    f_bytes = pa.path_attn_workspace_size(d, 0)
    b_bytes = pa.path_attn_workspace_size(d, 1)
    assert f_bytes < b_bytes
    fwd = lambda ph, n: pa.path_attn_fwd_phases(ph, d, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, n, None)
    assert fwd(pa.PATH_FWD_SCAN | pa.PATH_FWD_STORE_Z, b_bytes - 1) == 3   # forward-sized: too small
    assert fwd(pa.PATH_FWD_STORE_Z, b_bytes) == 1                         # no phase
    assert fwd(pa.PATH_FWD_ALL | 8, b_bytes) == 1                         # unknown bit
    base = [FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE]
    bwd = lambda ph, n: pa.path_attn_bwd_phases(ph, d, *base, n, None)
    assert bwd(pa.PATH_BWD_ALL | pa.PATH_BWD_REUSE_FWD | pa.PATH_BWD_Z_FROM_FWD, b_bytes - 1) == 3
    assert bwd(pa.PATH_BWD_Z_FROM_FWD, b_bytes) == 1
    assert bwd(pa.PATH_BWD_ALL | 32, b_bytes) == 1


def test_workspace_status_argument_errors(pa):
    """The status calls validate their arguments before any CUDA call; on the fp32 path (no bounded
    waits) and for an empty prompt they answer PATH_OK without touching the device."""
    code = ctypes.c_int(-1)
    d32 = desc(pa, dtype=pa.PATH_FP32)
    n32 = pa.path_attn_workspace_size(d32, 1)
    assert pa.path_attn_workspace_status(d32, 1, FAKE, n32, None) == (0, 0)   # fp32: nothing to read
    assert pa.path_attn_workspace_status(desc(pa, head_dim=96), 0, FAKE, n32, None)[0] == 2
    assert pa.path_attn_workspace_status(d32, 0, None, n32, None)[0] == 1
    assert pa.path_attn_workspace_status(d32, 0, FAKE + 16, n32, None)[0] == 1  # not 256-byte aligned
    dbf = desc(pa, dtype=pa.PATH_BF16)
    nb = pa.path_attn_workspace_size(dbf, 0)
    assert pa.path_attn_workspace_status(dbf, 0, FAKE, nb - 1, None)[0] == 3
    assert pa._lib.path_attn_workspace_status(None, 0, FAKE, nb, ctypes.byref(code), None) == 1
    dd = pa.path_decode_desc_t(2, 2, 64, 100, pa.PATH_BF16, 1.0)
    n = pa.path_decode_prefill_workspace_size(dd, 70)
    assert pa.path_decode_prefill_status(dd, 0, FAKE, n, None) == (0, 0)      # an empty prompt ran nothing
    assert pa.path_decode_prefill_status(dd, 101, FAKE, n, None)[0] == 4
    assert pa.path_decode_prefill_status(dd, 70, FAKE, n - 1, None)[0] == 3
    assert pa.path_decode_prefill_status(dd, 70, None, n, None)[0] == 1
    d32c = pa.path_decode_desc_t(2, 2, 64, 100, pa.PATH_FP32, 1.0)          # fp32 caches: SIMT preparation
    assert pa.path_decode_prefill_status(d32c, 70, FAKE, pa.path_decode_prefill_workspace_size(d32c, 70),
                                         None) == (0, 0)


def test_context_parallel_argument_errors(pa):
    """The context-parallel calls check scope and arguments before any CUDA call."""
    d = desc(pa, dtype=pa.PATH_BF16, seqlen=256)
    assert pa.path_cp_prepare_workspace_size(desc(pa, dtype=pa.PATH_FP32, seqlen=256)) == 0   # bf16 only
    assert pa.path_cp_prepare_workspace_size(desc(pa, dtype=pa.PATH_BF16, seqlen=200)) == 0   # not a 128 multiple
    n = pa.path_cp_prepare_workspace_size(d)
    assert n > 0
    F = [FAKE] * 7
    assert pa.path_cp_shard_prepare(desc(pa, dtype=pa.PATH_FP32, seqlen=256), *F[:4], None, *F[4:], None, None,
                                    None, FAKE, n, None) == 2
    assert pa.path_cp_shard_prepare(desc(pa, dtype=pa.PATH_BF16, seqlen=200), *F[:4], None, *F[4:], None, None,
                                    None, FAKE, n, None) == 2
    assert pa.path_cp_shard_prepare(desc(pa, dtype=pa.PATH_BF16, seqlen=256, head_dim=128), *F[:4], None, *F[4:],
                                    None, None, None, FAKE, n, None) == 2
    assert pa.path_cp_shard_prepare(d, None, *F[1:4], None, *F[4:], None, None, None, FAKE, n, None) == 1
    assert pa.path_cp_shard_prepare(d, *F[:4], FAKE, *F[4:], None, None, None, FAKE, n, None) == 1  # log_f alone
    assert pa.path_cp_shard_prepare(d, *F[:4], None, *F[4:], FAKE, None, None, FAKE, n, None) == 1  # a_q alone
    assert pa.path_cp_shard_prepare(d, *F[:4], None, *F[4:], None, None, None, FAKE, n - 1, None) == 3
    assert pa.path_cp_shard_prepare(d, *F[:4], None, *F[4:], None, None, None, FAKE + 16, n, None) == 1
    assert pa.path_cp_block_workspace_size(d, 100) == 0
    nb = pa.path_cp_block_workspace_size(d, 384)
    nf = pa.path_attn_workspace_size(d, 0)
    assert nb > 0
    att = lambda bl, a, b, fw, bw: pa.path_cp_attend_block(d, bl, FAKE, FAKE, FAKE, a, b, FAKE, fw, FAKE, bw, None)
    assert att(100, None, None, nf, nb) == 2
    assert att(0, None, None, nf, nb) == 1
    assert att(384, FAKE, None, nf, nb) == 1
    assert att(384, None, None, nf - 1, nb) == 3
    assert att(384, None, None, nf, nb - 1) == 3
    assert pa.path_cp_pass_block(d, 0, FAKE, None, FAKE, None, None) == 1
    assert pa.path_cp_pass_block(d, 100, FAKE, None, FAKE, None, None) == 2
    assert pa.path_cp_pass_block(d, 384, FAKE, FAKE, FAKE, None, None) == 1   # b_k without f_tot
    assert pa.path_cp_pass_block(d, 384, None, None, FAKE, None, None) == 1


def test_autograd_binding_rejects_host_tensors_before_any_launch(pa):
    """The autograd wrapper marshals through the same checks: CPU tensors are refused on the host."""
    import pytest as _pytest
    import torch as _torch

    from softmax_attention_chunk_gb300.autograd import path_attention

    q = _torch.zeros(1, 2, 64, 64, dtype=_torch.bfloat16)
    beta = _torch.zeros(1, 2, 64, dtype=_torch.float32)
    with _pytest.raises(ValueError):
        path_attention(q, q, q, q, beta)
