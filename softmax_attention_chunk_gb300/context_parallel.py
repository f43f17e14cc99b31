"""Context-parallel (sequence-sharded) PaTH attention forward: one shard of the sequence per rank and
a chain of key blocks passed from rank to rank.

PaTH reading notes (cc.laoqi.cc/papers/2505.16381), §2.8, last paragraph (the paper's Sec. 3.5):
sequence parallelism passes the transported keys and values and the block transforms between devices
and accumulates right to left.  Rank r holds tokens [r Ls, (r+1) Ls).  For a query i of shard r and a
key j of an earlier shard r'

    logit(i, j) = scale k~_j . (M_{r'+1} ... M_{r-1}) z^_i  (+ a_i + b_j with a forget gate)

(k~_j: the key moved to the end of its shard; z^_i: the query moved to the start of its own; M_s: the
product of shard s's transitions).  Each rank prepares its shard (the forward's PREPARE phase and
path_cp_shard_prepare), then for s = 1 .. N-1:
  * rank r (s-1 <= r <= N-2) sends the block it holds to rank r+1 — at s = 1 its own keys (moved to
    its end), its values and key biases; later, the block it received at step s-1 after moving it
    through its own shard;
  * rank r (r >= s) receives the block of rank r-s, merges it into its queries' softmax state
    (path_cp_attend_block) and, unless it is the last rank, moves it through its shard
    (path_cp_pass_block) to send at step s+1.
After N-1 steps rank r has merged the blocks of ranks 0 .. r-1; the forward's SCAN phase adds the
rank's own earlier chunks and writes o and lse.  Merging order does not change the result.

Message passing and argument marshalling only: every piece of arithmetic runs in the CUDA library.
The schedule is written against a small ops interface (own_block, attend, pass_block, finish) so that
the same code drives the C ABI on GPUs (ShardOps, NCCL point-to-point) and, in the tests, an fp64
stand-in on CPU ranks (gloo).
"""
from __future__ import annotations

import torch

from . import path_attn as pa


def step_roles(rank: int, world: int, s: int):
    """(sends, receives) of `rank` at step s (1 <= s < world) of the chain."""
    return (s - 1 <= rank <= world - 2), (rank >= s)


class ShardOps:
    """The C-ABI operations on one rank's shard: q, k, v, w [B, H, Ls, 64] bf16 on the rank's GPU,
    beta (and log_f, for PaTH-FoX) [B, H, Ls] fp32; Ls a multiple of 128."""

    def __init__(self, q, k, v, w, beta, log_f=None, scale=1.0):
        self.desc = pa.make_desc(q, scale)
        B, H, L, d = q.shape
        dev = q.device
        self.shape, self.v, self.log_f, self.scale = (B, H, L, d), v, log_f, scale
        self.args = (q, k, v, w, beta)
        self.ws = pa.workspace(self.desc, 0, dev)
        self.o = torch.empty_like(q)
        self.lse = torch.empty(B, H, L, dtype=torch.float32, device=dev)
        # the local diagonal-chunk softmax state, which the remote blocks are merged into
        pa.fwd(*self.args, log_f, scale, ws=self.ws, out=(self.o, self.lse), phases=pa.PATH_FWD_PREPARE)
        self.k_end = torch.empty(B, H, L, d, dtype=torch.float32, device=dev)
        self.q_start = torch.empty_like(q)
        self.t = torch.empty(B, H, d, d, dtype=torch.float32, device=dev)
        fox = log_f is not None
        self.a = torch.empty(B, H, L, dtype=torch.float32, device=dev) if fox else None
        self.b = torch.empty(B, H, L, dtype=torch.float32, device=dev) if fox else None
        self.tot = torch.empty(B, H, dtype=torch.float32, device=dev) if fox else None
        prep_ws = torch.empty(pa.path_cp_prepare_workspace_size(self.desc), dtype=torch.uint8, device=dev)
        p = pa._p
        rc = pa.path_cp_shard_prepare(self.desc, p(q), p(k), p(w), p(beta), p(log_f), p(self.k_end), p(self.q_start),
                                      p(self.t), p(self.a), p(self.b), p(self.tot), p(prep_ws), prep_ws.numel(),
                                      pa._stream())
        pa._check(rc, "path_cp_shard_prepare")
        self.blk_ws = torch.empty(pa.path_cp_block_workspace_size(self.desc, L), dtype=torch.uint8, device=dev)

    def own_block(self):
        """This shard's block: keys moved to its end (fp32), values, key biases (FoX)."""
        return {"k": self.k_end, "v": self.v, "b": self.b}

    def attend(self, blk):
        p = pa._p
        rc = pa.path_cp_attend_block(self.desc, blk["k"].shape[2], p(self.q_start), p(blk["k"]), p(blk["v"]),
                                     p(self.a), p(blk["b"]), p(self.ws), self.ws.numel(), p(self.blk_ws),
                                     self.blk_ws.numel(), pa._stream())
        pa._check(rc, "path_cp_attend_block")

    def pass_block(self, blk):
        p = pa._p
        rc = pa.path_cp_pass_block(self.desc, blk["k"].shape[2], p(blk["k"]), p(blk["b"]), p(self.t), p(self.tot),
                                   pa._stream())
        pa._check(rc, "path_cp_pass_block")
        return blk

    def finish(self):
        """The forward's SCAN phase: o and lse of the shard's rows over the whole prefix."""
        pa.fwd(*self.args, self.log_f, self.scale, ws=self.ws, out=(self.o, self.lse), phases=pa.PATH_FWD_SCAN)
        return self.o, self.lse


def _exchange(send_blk, recv_like, rank, group):
    """One step's messages: the held block to rank+1, a block from rank-1 (tensors in sorted key order)."""
    import torch.distributed as dist

    ops, got = [], None
    if send_blk is not None:
        for key in sorted(send_blk):
            if send_blk[key] is not None:
                ops.append(dist.P2POp(dist.isend, send_blk[key].contiguous(), dist.get_global_rank(group, rank + 1)
                                      if group is not None else rank + 1, group))
    if recv_like is not None:
        got = {key: (None if t is None else torch.empty_like(t)) for key, t in recv_like.items()}
        for key in sorted(got):
            if got[key] is not None:
                ops.append(dist.P2POp(dist.irecv, got[key], dist.get_global_rank(group, rank - 1)
                                      if group is not None else rank - 1, group))
    if ops:
        for req in dist.batch_isend_irecv(ops):
            req.wait()
    return got


def ring_forward(ops, group=None):
    """The chain over the ranks of `group` (torch.distributed): returns this rank's (o, lse)."""
    import torch.distributed as dist

    rank, world = dist.get_rank(group), dist.get_world_size(group)
    like = ops.own_block()
    held = like
    for s in range(1, world):
        sends, receives = step_roles(rank, world, s)
        got = _exchange(held if sends else None, like if receives else None, rank, group)
        if got is not None:
            ops.attend(got)
            held = ops.pass_block(got) if rank <= world - 2 else None
    return ops.finish()


def emulate_ring(ops_list):
    """The same schedule in one process (a message is a copy of the sender's block): the shards of one
    sequence prepared on one device, for checking the arithmetic without a multi-GPU run."""
    world = len(ops_list)
    held = [ops.own_block() for ops in ops_list]
    for s in range(1, world):
        sent = [held[r] if step_roles(r, world, s)[0] else None for r in range(world)]
        for r in range(world):
            if step_roles(r, world, s)[1]:
                got = {key: (None if t is None else t.clone()) for key, t in sent[r - 1].items()}
                ops_list[r].attend(got)
                held[r] = ops_list[r].pass_block(got) if r <= world - 2 else None
    return [ops.finish() for ops in ops_list]
