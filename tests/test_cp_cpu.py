"""Context-parallel forward: the chain of key blocks between ranks, on CPU ranks (gloo).

The chain (softmax_attention_chunk_gb300.context_parallel) is driven here with an fp64 stand-in of
the shard operations written from the definitions (explicit Householder products, not the CUDA
library): keys moved to their shard's end, queries moved to their shard's start, the shard product
M, the forget-gate terms, the merge of a block into a softmax state by log-sum-exp.  Each rank's
rows after the chain must equal the oracle's forward over the whole sequence, which checks the
schedule (every earlier block reaches every rank once, moved through exactly the shards in between),
the direction of the transports and the bias bookkeeping.  World sizes 2 and 3 (3 has a block that
passes through a middle shard).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def problem(n, L, d, fox, seed=5):
    rng = np.random.default_rng(seed)
    q, k, v = (rng.standard_normal((n, L, d)) / np.sqrt(d) for _ in range(3))
    w = rng.standard_normal((n, L, d))
    w /= np.linalg.norm(w, axis=-1, keepdims=True)
    beta = rng.uniform(0.0, 2.0, (n, L))
    beta[:, ::7] = 1.999  # near-reflection tokens
    logf = np.log(1.0 / (1.0 + np.exp(-(rng.standard_normal((n, L)) + 2.0)))) if fox else None
    return q, k, v, w, beta, logf


class ExplicitShardOps:
    """fp64 stand-in of the shard operations (heads [n, Ls, d])."""

    def __init__(self, q, k, v, w, beta, logf, scale):
        from oracle import oracle as orc

        n, L, d = q.shape
        beta = np.clip(beta, 0.0, 2.0)
        self.o, self.lse = orc.fwd(q, k, v, w, beta, logf, scale)  # the shard's own causal rows
        H = lambda h, t: np.eye(d) - beta[h, t] * np.outer(w[h, t], w[h, t])
        self.k_end = np.zeros_like(k)
        self.q_start = np.zeros_like(q)
        self.M = np.zeros((n, d, d))
        for h in range(n):
            for j in range(L):
                x = k[h, j].copy()
                for t in range(j + 1, L):  # H_{j+1} first, H_{L-1} last
                    x = H(h, t) @ x
                self.k_end[h, j] = x
                z = q[h, j].copy()
                for t in range(j, -1, -1):  # H_i first, H_0 last
                    z = H(h, t) @ z
                self.q_start[h, j] = z
            M = np.eye(d)
            for t in range(L):
                M = M @ H(h, t)
            self.M[h] = M
        self.v, self.scale = v, scale
        if logf is not None:
            self.a = np.cumsum(logf, axis=1)
            self.tot = self.a[:, -1].copy()
            self.b = self.tot[:, None] - self.a
        else:
            self.a = self.b = self.tot = None

    def own_block(self):
        t = lambda x: None if x is None else torch.from_numpy(np.ascontiguousarray(x))
        return {"k": t(self.k_end), "v": t(self.v), "b": t(self.b)}

    def attend(self, blk):
        kb, vb = blk["k"].numpy(), blk["v"].numpy()
        s = self.scale * np.einsum("nid,njd->nij", self.q_start, kb)
        if self.a is not None:
            s = s + self.a[:, :, None] + blk["b"].numpy()[:, None, :]
        m = s.max(axis=2)
        lse_b = m + np.log(np.exp(s - m[:, :, None]).sum(axis=2))
        o_b = np.einsum("nij,njd->nid", np.exp(s - lse_b[:, :, None]), vb)
        lse_new = np.logaddexp(self.lse, lse_b)
        self.o = np.exp(self.lse - lse_new)[:, :, None] * self.o + np.exp(lse_b - lse_new)[:, :, None] * o_b
        self.lse = lse_new

    def pass_block(self, blk):
        blk["k"] = torch.from_numpy(np.einsum("njd,nde->nje", blk["k"].numpy(), self.M))
        if blk["b"] is not None:
            blk["b"] = blk["b"] + torch.from_numpy(self.tot)[:, None]
        return blk

    def finish(self):
        return self.o, self.lse


def _worker(rank, world, port, fox, out):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from softmax_attention_chunk_gb300.context_parallel import ring_forward

        Ls = 12
        q, k, v, w, beta, logf = problem(2, Ls * world, 6, fox)
        sl = slice(rank * Ls, (rank + 1) * Ls)
        ops = ExplicitShardOps(q[:, sl], k[:, sl], v[:, sl], w[:, sl], beta[:, sl],
                               None if logf is None else logf[:, sl], 0.9)
        o, lse = ring_forward(ops)
        out.put((rank, o.tolist(), lse.tolist()))
    finally:
        torch.distributed.destroy_process_group()


@pytest.mark.parametrize("world,fox", [(2, False), (3, False), (3, True)])
def test_chain_on_gloo_ranks_gives_the_full_forward(world, fox):
    import sys

    sys.path.insert(0, ROOT)
    from oracle import oracle as orc

    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, fox, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    Ls = 12
    q, k, v, w, beta, logf = problem(2, Ls * world, 6, fox)
    o_ref, lse_ref = orc.fwd(q, k, v, w, beta, logf, 0.9)
    for rank, o, lse in res:
        sl = slice(rank * Ls, (rank + 1) * Ls)
        np.testing.assert_allclose(np.array(o), o_ref[:, sl], rtol=0, atol=1e-12)
        np.testing.assert_allclose(np.array(lse), lse_ref[:, sl], rtol=0, atol=1e-12)


def test_schedule_delivers_every_earlier_block_once_through_the_shards_between():
    """Symbolic run of the schedule: a block is the list of shards it has been moved through."""
    from softmax_attention_chunk_gb300.context_parallel import step_roles

    for world in range(1, 7):
        held = [[r] for r in range(world)]  # origin first, then the shards passed
        seen = [[] for _ in range(world)]
        for s in range(1, world):
            sent = [held[r] if step_roles(r, world, s)[0] else None for r in range(world)]
            for r in range(world):
                if step_roles(r, world, s)[1]:
                    blk = list(sent[r - 1])
                    seen[r].append(blk)
                    held[r] = blk + [r] if r <= world - 2 else None
        for r in range(world):
            # rank r merges the blocks of ranks r-1, r-2, ..., 0, each moved through r'+1 .. r-1
            assert seen[r] == [[o] + list(range(o + 1, r)) for o in range(r - 1, -1, -1)]
