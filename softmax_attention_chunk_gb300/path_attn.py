"""Thin ctypes binding of the PaTH attention C ABI (include/path_attn.h).

Argument marshalling only: every step of the computation runs in the CUDA library.  PyTorch
supplies device memory and the current stream.  The functions named like the C entry points
(path_attn_fwd, ...) take raw integer pointers; fwd/bwd/decode_step take torch tensors,
allocate outputs/workspace with torch and raise RuntimeError on a non-zero status.

If the compiled library is missing this module raises at import: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build_lib

PATH_OK = 0
PATH_BF16, PATH_FP32 = 0, 1
STATUS_NAMES = {0: "PATH_OK", 1: "PATH_ERR_INVALID_ARG", 2: "PATH_ERR_UNSUPPORTED", 3: "PATH_ERR_WORKSPACE",
                4: "PATH_ERR_CAPACITY", 5: "PATH_ERR_CUDA", 6: "PATH_ERR_INTERNAL"}

LIB_PATH = build_lib.LIB
if not os.path.exists(LIB_PATH):
    raise ImportError(f"PaTH CUDA library not built ({LIB_PATH}); run __graft_entry__.build()")
_lib = ctypes.CDLL(LIB_PATH)


class path_attn_desc_t(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("heads", ctypes.c_int), ("seqlen", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("dtype", ctypes.c_int), ("scale", ctypes.c_float),
                ("chunk", ctypes.c_int)]


class path_decode_desc_t(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("capacity", ctypes.c_int), ("cache_dtype", ctypes.c_int), ("scale", ctypes.c_float)]


_vp, _sz, _i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
_DP = ctypes.POINTER(path_attn_desc_t)
_DDP = ctypes.POINTER(path_decode_desc_t)
_lib.path_status_string.restype = ctypes.c_char_p
_lib.path_status_string.argtypes = [_i]
_lib.path_attn_chunk.restype = _i
_lib.path_attn_chunk.argtypes = [_DP, _i]
_lib.path_attn_workspace_size.restype = _sz
_lib.path_attn_workspace_size.argtypes = [_DP, _i]
_lib.path_attn_fwd.restype = _i
_lib.path_attn_fwd.argtypes = [_DP] + [_vp] * 8 + [_vp, _sz, _vp]
_lib.path_attn_bwd.restype = _i
_lib.path_attn_bwd.argtypes = [_DP] + [_vp] * 15 + [_vp, _sz, _vp]
_lib.path_attn_fwd_phases.restype = _i
_lib.path_attn_fwd_phases.argtypes = [_i, _DP] + [_vp] * 8 + [_vp, _sz, _vp]
_lib.path_attn_bwd_phases.restype = _i
_lib.path_attn_bwd_phases.argtypes = [_i, _DP] + [_vp] * 15 + [_vp, _sz, _vp]
_lib.path_decode_workspace_size.restype = _sz
_lib.path_decode_workspace_size.argtypes = [_DDP]
_lib.path_decode_step.restype = _i
_lib.path_decode_step.argtypes = [_DDP, _vp, _vp, _i] + [_vp] * 6 + [_vp, _sz, _vp]
_lib.path_decode_step_noalloc.restype = _i
_lib.path_decode_step_noalloc.argtypes = [_DDP, _vp, _vp, _i] + [_vp] * 6 + [_vp]
_lib.path_decode_prefill_workspace_size.restype = _sz
_lib.path_decode_prefill_workspace_size.argtypes = [_DDP, _i]
_lib.path_decode_prefill.restype = _i
_lib.path_decode_prefill.argtypes = [_DDP, _vp, _vp, _i] + [_vp] * 6 + [_vp, _sz, _vp]
_lib.path_decode_step_fox.restype = _i
_lib.path_decode_step_fox.argtypes = [_DDP, _vp, _vp, _vp, _i] + [_vp] * 7 + [_vp, _sz, _vp]
_lib.path_attn_workspace_status.restype = _i
_lib.path_attn_workspace_status.argtypes = [_DP, _i, _vp, _sz, ctypes.POINTER(_i), _vp]
_lib.path_decode_prefill_status.restype = _i
_lib.path_decode_prefill_status.argtypes = [_DDP, _i, _vp, _sz, ctypes.POINTER(_i), _vp]
_lib.path_cp_prepare_workspace_size.restype = _sz
_lib.path_cp_prepare_workspace_size.argtypes = [_DP]
_lib.path_cp_shard_prepare.restype = _i
_lib.path_cp_shard_prepare.argtypes = [_DP] + [_vp] * 11 + [_vp, _sz, _vp]
_lib.path_cp_block_workspace_size.restype = _sz
_lib.path_cp_block_workspace_size.argtypes = [_DP, _i]
_lib.path_cp_attend_block.restype = _i
_lib.path_cp_attend_block.argtypes = [_DP, _i] + [_vp] * 5 + [_vp, _sz, _vp, _sz, _vp]
_lib.path_cp_pass_block.restype = _i
_lib.path_cp_pass_block.argtypes = [_DP, _i] + [_vp] * 4 + [_vp]
PATH_DECODE_NOALLOC_MAX_HEADS = 496
PATH_ERR_INTERNAL = 6

PATH_FWD_PREPARE, PATH_FWD_SCAN, PATH_FWD_ALL = 1, 2, 3
PATH_BWD_PREPARE, PATH_BWD_SCAN, PATH_BWD_FINISH, PATH_BWD_ALL = 1, 2, 4, 7
PATH_BWD_REUSE_FWD = 8
PATH_FWD_STORE_Z = 4
PATH_BWD_Z_FROM_FWD = 16

EXPORTED = ("path_status_string", "path_attn_chunk", "path_attn_workspace_size", "path_attn_fwd",
            "path_attn_bwd", "path_attn_fwd_phases", "path_attn_bwd_phases", "path_decode_workspace_size",
            "path_decode_step", "path_decode_step_noalloc", "path_decode_prefill_workspace_size",
            "path_decode_prefill", "path_decode_step_fox", "path_attn_workspace_status",
            "path_decode_prefill_status", "path_cp_prepare_workspace_size", "path_cp_shard_prepare",
            "path_cp_block_workspace_size", "path_cp_attend_block", "path_cp_pass_block")


# ---------------- raw entry points (same names as the C ABI) ----------------

def path_status_string(status: int) -> str:
    return _lib.path_status_string(int(status)).decode()


def path_attn_chunk(desc: path_attn_desc_t, for_backward: int) -> int:
    return _lib.path_attn_chunk(ctypes.byref(desc), int(for_backward))


def path_attn_workspace_size(desc: path_attn_desc_t, for_backward: int) -> int:
    return _lib.path_attn_workspace_size(ctypes.byref(desc), int(for_backward))


def path_attn_fwd(desc, q, k, v, w, beta, log_f, o, lse, ws, ws_bytes, stream) -> int:
    return _lib.path_attn_fwd(ctypes.byref(desc), q, k, v, w, beta, log_f, o, lse, ws, ws_bytes, stream)


def path_attn_bwd(desc, q, k, v, w, beta, log_f, o, lse, dO, dq, dk, dv, dw, dbeta, dlog_f, ws,
                  ws_bytes, stream) -> int:
    return _lib.path_attn_bwd(ctypes.byref(desc), q, k, v, w, beta, log_f, o, lse, dO, dq, dk, dv, dw,
                              dbeta, dlog_f, ws, ws_bytes, stream)


def path_attn_fwd_phases(phases, desc, q, k, v, w, beta, log_f, o, lse, ws, ws_bytes, stream) -> int:
    return _lib.path_attn_fwd_phases(int(phases), ctypes.byref(desc), q, k, v, w, beta, log_f, o, lse, ws,
                                     ws_bytes, stream)


def path_attn_bwd_phases(phases, desc, q, k, v, w, beta, log_f, o, lse, dO, dq, dk, dv, dw, dbeta, dlog_f,
                         ws, ws_bytes, stream) -> int:
    return _lib.path_attn_bwd_phases(int(phases), ctypes.byref(desc), q, k, v, w, beta, log_f, o, lse, dO, dq,
                                     dk, dv, dw, dbeta, dlog_f, ws, ws_bytes, stream)


def path_decode_workspace_size(desc: path_decode_desc_t) -> int:
    return _lib.path_decode_workspace_size(ctypes.byref(desc))


def path_decode_step(desc, k_cache, v_cache, t, q_t, k_t, v_t, w_t, beta_t, o_t, ws, ws_bytes, stream) -> int:
    return _lib.path_decode_step(ctypes.byref(desc), k_cache, v_cache, int(t), q_t, k_t, v_t, w_t, beta_t,
                                 o_t, ws, ws_bytes, stream)


def path_decode_step_noalloc(desc, k_cache, v_cache, t, q_t, k_t, v_t, w_t, beta_t, o_t, stream) -> int:
    return _lib.path_decode_step_noalloc(ctypes.byref(desc), k_cache, v_cache, int(t), q_t, k_t, v_t, w_t,
                                         beta_t, o_t, stream)


def path_decode_prefill_workspace_size(desc: path_decode_desc_t, prompt_len: int) -> int:
    return _lib.path_decode_prefill_workspace_size(ctypes.byref(desc), int(prompt_len))


def path_decode_prefill(desc, k_cache, v_cache, prompt_len, k, v, w, beta, log_f, a_cache, ws, ws_bytes,
                        stream) -> int:
    return _lib.path_decode_prefill(ctypes.byref(desc), k_cache, v_cache, int(prompt_len), k, v, w, beta, log_f,
                                    a_cache, ws, ws_bytes, stream)


def path_decode_step_fox(desc, k_cache, v_cache, a_cache, t, q_t, k_t, v_t, w_t, beta_t, log_f_t, o_t, ws, ws_bytes,
                         stream) -> int:
    return _lib.path_decode_step_fox(ctypes.byref(desc), k_cache, v_cache, a_cache, int(t), q_t, k_t, v_t, w_t,
                                     beta_t, log_f_t, o_t, ws, ws_bytes, stream)


def path_attn_workspace_status(desc, for_backward, ws, ws_bytes, stream):
    """(status, first recorded device code) of the passes that ran on the workspace; synchronises
    the stream."""
    code = _i(0)
    rc = _lib.path_attn_workspace_status(ctypes.byref(desc), int(for_backward), ws, ws_bytes, ctypes.byref(code),
                                         stream)
    return rc, code.value


def path_decode_prefill_status(desc, prompt_len, ws, ws_bytes, stream):
    """(status, first recorded device code) of a prefill hand-off's workspace; synchronises the stream."""
    code = _i(0)
    rc = _lib.path_decode_prefill_status(ctypes.byref(desc), int(prompt_len), ws, ws_bytes, ctypes.byref(code),
                                         stream)
    return rc, code.value


def path_cp_prepare_workspace_size(desc) -> int:
    return _lib.path_cp_prepare_workspace_size(ctypes.byref(desc))


def path_cp_shard_prepare(desc, q, k, w, beta, log_f, k_end, q_start, t_shard, a_q, b_k, f_tot, ws, ws_bytes,
                          stream) -> int:
    return _lib.path_cp_shard_prepare(ctypes.byref(desc), q, k, w, beta, log_f, k_end, q_start, t_shard, a_q, b_k,
                                      f_tot, ws, ws_bytes, stream)


def path_cp_block_workspace_size(desc, block_len) -> int:
    return _lib.path_cp_block_workspace_size(ctypes.byref(desc), int(block_len))


def path_cp_attend_block(desc, block_len, q_start, k_block, v_block, a_q, b_k, fwd_ws, fwd_ws_bytes, blk_ws,
                         blk_ws_bytes, stream) -> int:
    return _lib.path_cp_attend_block(ctypes.byref(desc), int(block_len), q_start, k_block, v_block, a_q, b_k, fwd_ws,
                                     fwd_ws_bytes, blk_ws, blk_ws_bytes, stream)


def path_cp_pass_block(desc, block_len, k_block, b_k, t_shard, f_tot, stream) -> int:
    return _lib.path_cp_pass_block(ctypes.byref(desc), int(block_len), k_block, b_k, t_shard, f_tot, stream)


# ---------------- torch-tensor wrappers ----------------

_DT = {torch.bfloat16: PATH_BF16, torch.float32: PATH_FP32}


def _p(t):
    return None if t is None else t.data_ptr()


def _check(rc, what):
    if rc != PATH_OK:
        raise RuntimeError(f"{what} failed: {path_status_string(rc)}")


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _need(t, dtype, shape, name):
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name}: expected contiguous cuda {dtype} {tuple(shape)}, got {t.dtype} "
                         f"{tuple(t.shape)} contiguous={t.is_contiguous()} device={t.device}")


def make_desc(q, scale, chunk=0) -> path_attn_desc_t:
    B, H, L, d = q.shape
    if q.dtype not in _DT:
        raise ValueError(f"unsupported dtype {q.dtype}")
    return path_attn_desc_t(B, H, L, d, _DT[q.dtype], float(scale), int(chunk))


def workspace(desc, for_backward, device):
    n = path_attn_workspace_size(desc, for_backward)
    if n == 0:
        raise RuntimeError("invalid descriptor (workspace size 0)")
    return torch.empty(n, dtype=torch.uint8, device=device)


def check_workspace(desc, for_backward, ws):
    """Raises RuntimeError if a tensor-core kernel that ran on `ws` gave up one of its bounded
    waits (its outputs are then incomplete).  Synchronises the current stream."""
    rc, code = path_attn_workspace_status(desc, for_backward, _p(ws), ws.numel(), _stream())
    if rc != PATH_OK:
        raise RuntimeError(f"device status of the workspace: {path_status_string(rc)} (code {code})")


def fwd(q, k, v, w, beta, log_f=None, scale=1.0, chunk=0, ws=None, out=None, phases=PATH_FWD_ALL, check=False):
    """o [B,H,L,d] (dtype of q) and lse [B,H,L] float32.  check=True synchronises and raises if a
    kernel gave up a bounded wait (the workspace status)."""
    desc = make_desc(q, scale, chunk)
    for name, t in (("k", k), ("v", v), ("w", w)):
        _need(t, q.dtype, q.shape, name)
    _need(q, q.dtype, q.shape, "q")
    _need(beta, torch.float32, q.shape[:3], "beta")
    if log_f is not None:
        _need(log_f, torch.float32, q.shape[:3], "log_f")
    if ws is None:
        ws = workspace(desc, 0, q.device)
    o, lse = out if out is not None else (torch.empty_like(q), torch.empty(q.shape[:3], dtype=torch.float32,
                                                                           device=q.device))
    rc = path_attn_fwd_phases(phases, desc, _p(q), _p(k), _p(v), _p(w), _p(beta), _p(log_f), _p(o), _p(lse),
                              _p(ws), ws.numel(), _stream())
    _check(rc, "path_attn_fwd")
    if check:
        check_workspace(desc, 1 if ws.numel() >= path_attn_workspace_size(desc, 1) else 0, ws)
    return o, lse


def bwd(q, k, v, w, beta, o, lse, dO, scale=1.0, chunk=0, ws=None, log_f=None, out=None,
        phases=PATH_BWD_ALL, check=False):
    """Gradients dict dq, dk, dv, dw (dtype of q) and dbeta (float32); with log_f (PaTH-FoX) also
    dlog_f (float32).  check=True synchronises and raises if a kernel gave up a bounded wait."""
    desc = make_desc(q, scale, chunk)
    for name, t in (("k", k), ("v", v), ("w", w), ("o", o), ("dO", dO)):
        _need(t, q.dtype, q.shape, name)
    _need(beta, torch.float32, q.shape[:3], "beta")
    _need(lse, torch.float32, q.shape[:3], "lse")
    if ws is None:
        ws = workspace(desc, 1, q.device)
    if log_f is not None:
        _need(log_f, torch.float32, q.shape[:3], "log_f")
    if out is None:
        out = dict(dq=torch.empty_like(q), dk=torch.empty_like(q), dv=torch.empty_like(q),
                   dw=torch.empty_like(q), dbeta=torch.empty_like(beta))
        if log_f is not None:
            out["dlog_f"] = torch.empty_like(beta)
    rc = path_attn_bwd_phases(phases, desc, _p(q), _p(k), _p(v), _p(w), _p(beta), _p(log_f), _p(o), _p(lse),
                              _p(dO), _p(out["dq"]), _p(out["dk"]), _p(out["dv"]), _p(out["dw"]),
                              _p(out["dbeta"]), _p(out.get("dlog_f")), _p(ws), ws.numel(), _stream())
    _check(rc, "path_attn_bwd")
    if check:
        check_workspace(desc, 1, ws)
    return out


def make_decode_desc(k_cache, scale) -> path_decode_desc_t:
    B, H, cap, d = k_cache.shape
    return path_decode_desc_t(B, H, d, cap, _DT[k_cache.dtype], float(scale))


def decode_workspace(desc, device):
    n = path_decode_workspace_size(desc)
    if n == 0:
        raise RuntimeError("invalid decode descriptor")
    return torch.empty(n, dtype=torch.uint8, device=device)


def decode_step(k_cache, v_cache, t, q_t, k_t, v_t, w_t, beta_t, scale=1.0, ws=None, out=None):
    """One decode step at position t (in place on the caches); returns o_t [B,H,d]."""
    desc = make_decode_desc(k_cache, scale)
    B, H, cap, d = k_cache.shape
    _need(v_cache, k_cache.dtype, k_cache.shape, "v_cache")
    for name, x in (("q_t", q_t), ("k_t", k_t), ("v_t", v_t), ("w_t", w_t)):
        _need(x, k_cache.dtype, (B, H, d), name)
    _need(beta_t, torch.float32, (B, H), "beta_t")
    if ws is None:
        ws = decode_workspace(desc, k_cache.device)
    o = torch.empty_like(q_t) if out is None else out
    rc = path_decode_step(desc, _p(k_cache), _p(v_cache), t, _p(q_t), _p(k_t), _p(v_t), _p(w_t), _p(beta_t),
                          _p(o), _p(ws), ws.numel(), _stream())
    _check(rc, "path_decode_step")
    return o


def decode_prefill(k_cache, v_cache, k, v, w, beta, ws=None, log_f=None, a_cache=None):
    """Prefill -> decode hand-off: rows 0..L-1 of the caches [B,H,cap,d] get the prompt keys
    k,v,w [B,H,L,d] (cache dtype), beta [B,H,L] fp32 transported to the prompt end; decoding then
    continues at t = L.  PaTH-FoX: log_f [B,H,L] and a_cache [B,H,cap] (fp32) together fill the
    forget-gate prefix cache."""
    desc = make_decode_desc(k_cache, 1.0)
    B, H, cap, d = k_cache.shape
    L = k.shape[2]
    _need(v_cache, k_cache.dtype, k_cache.shape, "v_cache")
    for name, x in (("k", k), ("v", v), ("w", w)):
        _need(x, k_cache.dtype, (B, H, L, d), name)
    _need(beta, torch.float32, (B, H, L), "beta")
    if (log_f is None) != (a_cache is None):
        raise ValueError("log_f and a_cache go together")
    if log_f is not None:
        _need(log_f, torch.float32, (B, H, L), "log_f")
        _need(a_cache, torch.float32, (B, H, cap), "a_cache")
    n = path_decode_prefill_workspace_size(desc, L)
    if n == 0:
        raise RuntimeError("invalid decode descriptor or prompt length")
    if ws is None:
        ws = torch.empty(n, dtype=torch.uint8, device=k_cache.device)
    rc = path_decode_prefill(desc, _p(k_cache), _p(v_cache), L, _p(k), _p(v), _p(w), _p(beta), _p(log_f),
                             _p(a_cache), _p(ws), ws.numel(), _stream())
    _check(rc, "path_decode_prefill")


def decode_step_fox(k_cache, v_cache, a_cache, t, q_t, k_t, v_t, w_t, beta_t, log_f_t, scale=1.0, ws=None, out=None):
    """One PaTH-FoX decode step at position t (in place on the caches and the forget-gate prefix
    cache a_cache [B,H,cap] fp32); returns o_t [B,H,d]."""
    desc = make_decode_desc(k_cache, scale)
    B, H, cap, d = k_cache.shape
    _need(v_cache, k_cache.dtype, k_cache.shape, "v_cache")
    _need(a_cache, torch.float32, (B, H, cap), "a_cache")
    for name, x in (("q_t", q_t), ("k_t", k_t), ("v_t", v_t), ("w_t", w_t)):
        _need(x, k_cache.dtype, (B, H, d), name)
    _need(beta_t, torch.float32, (B, H), "beta_t")
    _need(log_f_t, torch.float32, (B, H), "log_f_t")
    if ws is None:
        ws = decode_workspace(desc, k_cache.device)
    o = torch.empty_like(q_t) if out is None else out
    rc = path_decode_step_fox(desc, _p(k_cache), _p(v_cache), _p(a_cache), t, _p(q_t), _p(k_t), _p(v_t), _p(w_t),
                              _p(beta_t), _p(log_f_t), _p(o), _p(ws), ws.numel(), _stream())
    _check(rc, "path_decode_step_fox")
    return o
