"""torch.autograd binding of the PaTH attention library.

path_attention(q, k, v, w, beta, log_f=None, scale=1.0) returns o [B, H, L, d] and is differentiable
in q, k, v, w, beta and (PaTH-FoX) log_f.  The forward runs the library's training forward
(PATH_FWD_STORE_Z) in a workspace sized for the backward, which the autograd graph keeps until the
backward; the backward then reuses the stored per-chunk preparation and transported query tiles
(PATH_BWD_REUSE_FWD | PATH_BWD_Z_FROM_FWD), as a training step does.  On the paths that do not
store them (fp32, head dim 128 backward) the flags are ignored and the backward recomputes.
The workspace holds the transported query tiles (16 KB per 128-row tile and earlier 64-row chunk:
16 GiB at batch 32 x 32 heads x 4096), kept alive like any saved activation.

Argument marshalling only (contiguous copies of the inputs where needed): every step of the
computation runs in the CUDA library.
"""
from __future__ import annotations

import torch

from . import path_attn as pa


class PathAttentionFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, w, beta, log_f, scale, chunk):
        q, k, v, w, beta = (t.contiguous() for t in (q, k, v, w, beta))
        log_f = None if log_f is None else log_f.contiguous()
        desc = pa.make_desc(q, scale, chunk)
        nbytes = max(pa.path_attn_workspace_size(desc, 0), pa.path_attn_workspace_size(desc, 1))
        if nbytes == 0:
            raise RuntimeError("path_attention: invalid descriptor (workspace size 0)")
        ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
        o, lse = pa.fwd(q, k, v, w, beta, log_f, scale, chunk, ws=ws, phases=pa.PATH_FWD_ALL | pa.PATH_FWD_STORE_Z)
        ctx.save_for_backward(q, k, v, w, beta, o, lse, *(() if log_f is None else (log_f,)))
        ctx.ws, ctx.scale, ctx.chunk, ctx.fox = ws, scale, chunk, log_f is not None
        ctx.mark_non_differentiable(lse)
        return o, lse

    @staticmethod
    def backward(ctx, do, _dlse):
        saved = ctx.saved_tensors
        q, k, v, w, beta, o, lse = saved[:7]
        log_f = saved[7] if ctx.fox else None
        g = pa.bwd(q, k, v, w, beta, o, lse, do.contiguous(), ctx.scale, ctx.chunk, ws=ctx.ws, log_f=log_f,
                   phases=pa.PATH_BWD_ALL | pa.PATH_BWD_REUSE_FWD | pa.PATH_BWD_Z_FROM_FWD)
        return g["dq"], g["dk"], g["dv"], g["dw"], g["dbeta"], g.get("dlog_f"), None, None


def path_attention(q, k, v, w, beta, log_f=None, scale=1.0, chunk=0, return_lse=False):
    """PaTH attention with autograd: q, k, v, w [B, H, L, d] (bf16 or fp32, one dtype), beta and
    log_f [B, H, L] float32 (log_f: the PaTH-FoX forget gate, or None).  Returns o (and lse, not
    differentiable, with return_lse)."""
    o, lse = PathAttentionFunction.apply(q, k, v, w, beta, log_f, scale, chunk)
    return (o, lse) if return_lse else o
