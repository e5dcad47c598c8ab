"""One graph partitioned over ranks by receiver ranges, with the halo exchanges of the
convolution (host logic; the convolution itself runs on each rank's own GPU).

A receiver-stationary convolution partitions naturally by receivers: rank r owns the
contiguous node range [n0, n1) of a receiver-sorted CSR and every edge into it, so its
messages m[n0:n1] are computed locally once it holds the rows x[a] of the senders a outside
its range (the halo). The backward is the transposed exchange: the dx partials that a rank
computes for its halo senders belong to their owners, which add them to their own. Edge
arrays (y, w, dy, dw) never move. This is the one exchange step of the data-parallel conv
(e3j, App. E.1 Eq. (12)-(16): the forward gathers sender rows, the backward scatters dx).

Local index space of rank r: its owned nodes first (global id - n0), then its halo nodes in
ascending global id. The local graph has one empty receiver segment per halo node, so local
node arrays have n_owned + n_halo rows and the library's calls take it as any other graph.
The exchanges go through torch.distributed point-to-point operations (NCCL between GPUs,
gloo on CPU); the order of every sum is fixed, so results are deterministic. A padding node
(e3j, Sec. 4) keeps its role on every rank: pass local_index([pad]) as the calls' pad_node
(its owner's local id, a halo id where it sends into other ranks, -1 elsewhere).
"""
from __future__ import annotations

import numpy as np


def receiver_cuts(rowptr, world: int) -> np.ndarray:
    """Node boundaries [0 = c_0 <= ... <= c_world = N] balancing the edges: c_r is the node
    boundary nearest to r * E / world."""
    rp = np.asarray(rowptr, dtype=np.int64)
    N, E = rp.shape[0] - 1, int(rp[-1])
    cuts = [0]
    for r in range(1, world):
        t = r * E / world
        b = int(np.searchsorted(rp, t))
        if b > 0 and (b > N or t - rp[b - 1] <= rp[b] - t):
            b -= 1
        cuts.append(min(max(b, cuts[-1]), N))
    cuts.append(N)
    return np.array(cuts, dtype=np.int64)


class HaloPartition:
    """Rank `rank`'s part of a receiver-sorted CSR (rowptr [N+1], sender [E]) split over
    `world` ranks by receiver_cuts. Attributes: n0, n1 (owned nodes), e0, e1 (owned edges),
    halo (global ids of the halo senders, ascending), n_owned, n_local, rowptr and sender of
    the local graph (int32, local ids), and per peer the local positions it sends and
    receives. Call setup(group) once before the exchanges."""

    def __init__(self, rowptr, sender, world: int, rank: int):
        rp = np.asarray(rowptr, dtype=np.int64)
        sd = np.asarray(sender, dtype=np.int64)
        if world < 1 or not 0 <= rank < world:
            raise ValueError(f"rank {rank} outside world {world}")
        N = rp.shape[0] - 1
        if rp[0] != 0 or np.any(np.diff(rp) < 0) or sd.shape[0] != int(rp[-1]):
            raise ValueError("rowptr / sender do not form a CSR")
        if sd.size and (sd.min() < 0 or sd.max() >= N):
            raise ValueError("sender id outside [0, N)")
        self.world, self.rank, self.N = world, rank, N
        self.cuts = receiver_cuts(rp, world)
        self.n0, self.n1 = int(self.cuts[rank]), int(self.cuts[rank + 1])
        self.e0, self.e1 = int(rp[self.n0]), int(rp[self.n1])
        s_loc = sd[self.e0:self.e1]
        outside = (s_loc < self.n0) | (s_loc >= self.n1)
        self.halo = np.unique(s_loc[outside])
        self.n_owned = self.n1 - self.n0
        self.n_local = self.n_owned + self.halo.shape[0]
        local = np.empty_like(s_loc)
        local[~outside] = s_loc[~outside] - self.n0
        local[outside] = self.n_owned + np.searchsorted(self.halo, s_loc[outside])
        self.sender = local.astype(np.int32)
        self.rowptr = np.concatenate([rp[self.n0:self.n1 + 1] - self.e0,
                                      np.full(self.halo.shape[0], self.e1 - self.e0, np.int64)]).astype(np.int32)
        owner = np.searchsorted(self.cuts, self.halo, side="right") - 1
        # halo rows this rank receives from each peer: local positions, in ascending global id
        self.recv_pos = {r: self.n_owned + np.nonzero(owner == r)[0] for r in range(world) if r != rank}
        self._need = {r: self.halo[owner == r] for r in range(world) if r != rank}
        self.send_pos = None

    def local_index(self, global_ids):
        """Local ids of global node ids (owned nodes, then halo nodes); -1 where a node is
        neither (for example, to pass a padding node's id to the library's pad_node)."""
        g = np.asarray(global_ids, dtype=np.int64)
        out = np.full(g.shape, -1, dtype=np.int64)
        own = (g >= self.n0) & (g < self.n1)
        out[own] = g[own] - self.n0
        pos = np.searchsorted(self.halo, g)
        hit = ~own & (pos < self.halo.shape[0])
        hit[hit] = self.halo[pos[hit]] == g[hit]
        out[hit] = self.n_owned + pos[hit]
        return out

    def setup(self, group=None):
        """Exchange the halo lists once: afterwards send_pos[r] holds the local (owned)
        positions of the rows peer r needs, in the order r expects them."""
        import torch.distributed as dist
        needs = [None] * self.world
        dist.all_gather_object(needs, {r: v.tolist() for r, v in self._need.items()}, group=group)
        self.send_pos = {r: np.asarray(needs[r].get(self.rank, []), dtype=np.int64) - self.n0
                         for r in range(self.world) if r != self.rank}
        return self

    def _exchange(self, send, recv, group):
        import torch.distributed as dist
        ops = []
        for r, t in send.items():
            if t.shape[0]:
                ops.append(dist.P2POp(dist.isend, t, r, group))
        for r, t in recv.items():
            if t.shape[0]:
                ops.append(dist.P2POp(dist.irecv, t, r, group))
        if ops:
            for q in dist.batch_isend_irecv(ops):
                q.wait()

    def gather_halo(self, x_owned, group=None):
        """Forward exchange: x_local [n_local, ...] = the owned rows, then the halo rows
        received from their owners. x_owned: [n_owned, ...] (any device and dtype)."""
        import torch
        assert self.send_pos is not None, "call setup() first"
        x_local = torch.empty((self.n_local,) + tuple(x_owned.shape[1:]), dtype=x_owned.dtype, device=x_owned.device)
        x_local[:self.n_owned] = x_owned
        send = {r: x_owned[torch.from_numpy(p).to(x_owned.device)].contiguous() for r, p in self.send_pos.items()}
        recv = {r: torch.empty((p.shape[0],) + tuple(x_owned.shape[1:]), dtype=x_owned.dtype, device=x_owned.device)
                for r, p in self.recv_pos.items()}
        self._exchange(send, recv, group)
        for r, p in self.recv_pos.items():
            if p.shape[0]:
                x_local[torch.from_numpy(p).to(x_owned.device)] = recv[r]
        return x_local

    def scatter_halo_grad(self, dx_local, group=None):
        """Backward exchange: dx_owned [n_owned, ...] = this rank's partials of its owned rows
        plus, in ascending peer rank, the partials the peers computed for them."""
        import torch
        assert self.send_pos is not None, "call setup() first"
        dev = dx_local.device
        send = {r: dx_local[torch.from_numpy(p).to(dev)].contiguous() for r, p in self.recv_pos.items()}
        recv = {r: torch.empty((p.shape[0],) + tuple(dx_local.shape[1:]), dtype=dx_local.dtype, device=dev)
                for r, p in self.send_pos.items()}
        self._exchange(send, recv, group)
        dx = dx_local[:self.n_owned].clone()
        for r in sorted(self.send_pos):
            p = self.send_pos[r]
            if p.shape[0]:   # positions are distinct: one addition per row
                dx[torch.from_numpy(p).to(dev)] += recv[r]
        return dx
