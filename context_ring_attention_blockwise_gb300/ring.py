"""Ring attention across processes: one process per GPU, each holding R consecutive ranks of a
plan's n_cp ("Context and expert parallelism", "Pass them around a ring": every rank computes its
queries against the key/value block it holds while it sends that block to its right neighbour and
receives the next one from its left; "When the ring hides its communication": each transfer
overlaps a step of attention).

Each process keeps a two-slot stage. At step s it computes on slot s % 2 (on the compute stream)
while the copy stream fills slot (s + 1) % 2: the library moves the blocks between the process's own
ranks (``dist_shift``), and a transport moves the one block that crosses to the next process. The
transport is the only inter-process step:

* ``NcclTransport``: device-to-device send/receive with torch.distributed over NCCL (one GPU per
  process);
* ``HostTransport``: through host memory with any torch.distributed backend (gloo): the block is
  copied to page-locked host memory, exchanged, and copied into the receiving slot;
* with one process (R = n_cp) no transport is needed: the shift passes the last rank's block to the
  first (``wrap``).

Blocks carry their position tables with them ("In PyTorch": every position-indexed tensor is
sharded with the sequence). Every compute step runs in the library's kernels; this module only
orders streams, events and the transport.
"""
from __future__ import annotations

from dataclasses import dataclass, field

REGIONS = ("k", "v", "pos", "tiles")


@dataclass
class HopCounters:
    """Bytes each of this process's ranks received over the ring, split into key/value bytes
    (what the pages count) and the position tables that travel with each block."""
    kv: list = field(default_factory=list)
    tables: list = field(default_factory=list)
    steps: list = field(default_factory=list)   # (step, slot index computed on)


class HostTransport:
    """The block that leaves this process goes to the next process and the previous process's
    block arrives, through host memory: device -> page-locked host copy on the copy stream, then
    torch.distributed isend / irecv (any backend, e.g. gloo), then host -> device on the copy stream."""

    def __init__(self, rank: int, world: int, group=None):
        self.rank, self.world, self.group = rank, world, group
        self._send = self._recv = None

    def exchange(self, send, recv, stream):
        import torch
        import torch.distributed as dist
        on_gpu = send[0].is_cuda
        if self._send is None:
            self._send = [torch.empty(t.shape, dtype=t.dtype, pin_memory=on_gpu) for t in send]
            self._recv = [torch.empty(t.shape, dtype=t.dtype, pin_memory=on_gpu) for t in recv]
        if on_gpu:
            with torch.cuda.stream(stream):
                for h, t in zip(self._send, send):
                    h.copy_(t, non_blocking=True)
            stream.synchronize()
        else:
            for h, t in zip(self._send, send):
                h.copy_(t)
        nxt, prv = (self.rank + 1) % self.world, (self.rank - 1) % self.world
        reqs = [dist.isend(h, nxt, group=self.group) for h in self._send]
        reqs += [dist.irecv(h, prv, group=self.group) for h in self._recv]
        for r in reqs:
            r.wait()
        if on_gpu:
            with torch.cuda.stream(stream):
                for t, h in zip(recv, self._recv):
                    t.copy_(h, non_blocking=True)
        else:
            for t, h in zip(recv, self._recv):
                t.copy_(h)


class NcclTransport:
    """Device-to-device send / receive of the crossing block with torch.distributed over NCCL,
    ordered after the copy stream's earlier work and before its later work."""

    def __init__(self, rank: int, world: int, group=None):
        self.rank, self.world, self.group = rank, world, group

    def exchange(self, send, recv, stream):
        import torch
        import torch.distributed as dist
        nxt, prv = (self.rank + 1) % self.world, (self.rank - 1) % self.world
        ops = [dist.P2POp(dist.isend, t, nxt, self.group) for t in send]
        ops += [dist.P2POp(dist.irecv, t, prv, self.group) for t in recv]
        with torch.cuda.stream(stream):
            for w in dist.batch_isend_irecv(ops):
                w.wait()


class LibraryBackend:
    """The device side of one process: the library's cpattn_dist_* calls on CUDA streams."""

    def __init__(self, plan, B: int, rank0: int, R: int, device):
        import torch
        from . import alloc_workspace
        self.plan, self.B, self.rank0, self.R = plan, B, rank0, R
        ws_bytes, slot_bytes, self.offsets, self.blocks = plan.dist_sizes(B, R)
        self.ws = alloc_workspace(ws_bytes, device)
        self.slots = [alloc_workspace(slot_bytes, device), alloc_workspace(slot_bytes, device)]
        self.device = torch.device(device)

    def region(self, slot, x: int, i: int):
        """Local rank i's block in region x of a slot, as a byte tensor."""
        o = self.offsets[x] + i * self.blocks[x]
        return slot[o:o + self.blocks[x]]

    def event(self, stream):
        import torch
        e = torch.cuda.Event()
        e.record(stream)
        return e

    @staticmethod
    def wait(stream, event):
        if event is not None:
            stream.wait_event(event)

    def begin(self, q, k, v, pos, slot, stream, lo=None):
        from . import dist_begin
        dist_begin(self.plan, self.B, self.rank0, self.R, q, k, v, self.ws, slot, pos=pos, stream=stream, lo=lo)

    def step(self, s, slot, scale, stream):
        from . import dist_step
        dist_step(self.plan, self.B, self.rank0, self.R, s, slot, self.ws, scale=scale, stream=stream)

    def shift(self, src, dst, wrap, stream):
        from . import dist_shift
        dist_shift(self.plan, self.B, self.R, src, dst, wrap, stream=stream)

    def step_shift(self, s, slot, next_slot, wrap, scale, stream):
        from . import dist_step_shift
        dist_step_shift(self.plan, self.B, self.rank0, self.R, s, slot, next_slot, wrap, self.ws, scale=scale,
                        stream=stream)

    def finalize(self, out, lse, stream):
        from . import dist_finalize
        dist_finalize(self.plan, self.B, self.rank0, self.R, self.ws, out, lse, stream=stream)


class RingProcess:
    """This process's part of the ring: ranks rank * R .. rank * R + R - 1 of the plan's n_cp, with
    R = n_cp / world. ``forward`` takes the process's tokens (rank-major, each rank's local layout
    order) and returns their outputs in the same order."""

    def __init__(self, plan, B: int, rank: int = 0, world: int = 1, transport=None, backend=None, device=None):
        if plan.n_cp % world:
            raise ValueError("n_cp must be a multiple of the number of processes")
        self.plan, self.B, self.rank, self.world = plan, B, rank, world
        self.R = plan.n_cp // world
        self.rank0 = rank * self.R
        if backend is None:
            backend = LibraryBackend(plan, B, self.rank0, self.R, device if device is not None else "cuda")
        self.backend = backend
        if world > 1 and transport is None:
            raise ValueError("a ring over several processes needs a transport")
        self.transport = transport
        self.counters = HopCounters(kv=[0] * self.R, tables=[0] * self.R)

    def forward(self, q, k, v, pos=None, scale=None, out=None, lse=None, stream=None, copy_stream=None,
                timeline=None, lo=None, shift_in_kernel=True):
        """timeline: a list to which each step appends (end of its compute, end of the hop that
        runs beside it) as timing events on the two streams (device backend only). With
        shift_in_kernel (and a backend that has it) each step's kernel also moves the blocks
        between this process's own ranks, so only the block that crosses to the next process
        uses the copy stream; otherwise the whole shift runs there too. Without a copy_stream the
        hops go to a new high-priority stream: the next step waits on them, so they should not
        queue behind other copies the caller runs. lo: the tokens' per-query lower bounds
        (document masks of packed sequences), in the order of q."""
        import torch
        be, R, n_cp = self.backend, self.R, self.plan.n_cp
        B, h, n = self.B, self.plan.h, self.plan.T // n_cp
        on_gpu = getattr(be, "device", None) is not None and be.device.type == "cuda"
        in_kernel = bool(shift_in_kernel) and hasattr(be, "step_shift")
        if on_gpu:
            compute = stream if stream is not None else torch.cuda.current_stream(be.device)
            if in_kernel and self.world == 1 and copy_stream is None:
                copy = compute          # nothing runs beside the steps: the kernels move every block
            else:
                copy = copy_stream if copy_stream is not None else torch.cuda.Stream(device=be.device, priority=-1)
        else:
            compute = copy = None
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty((B, h, R * n), dtype=torch.float32, device=q.device)
        slots = be.slots
        kv_blk = be.blocks[0] + be.blocks[1]
        tab_blk = be.blocks[2] + be.blocks[3]
        if lo is None:
            be.begin(q, k, v, pos, slots[0], compute)
        else:
            be.begin(q, k, v, pos, slots[0], compute, lo=lo)
        placed = be.event(compute)
        used = [None, None]     # the step that last computed on each slot
        arrived = None          # the hop that filled the slot of the next step
        for s in range(n_cp):
            cur, nxt = slots[s % 2], slots[(s + 1) % 2]
            if s > 0:
                be.wait(compute, arrived)
            if in_kernel and s + 1 < n_cp:
                be.step_shift(s, cur, nxt, self.world == 1, scale, compute)
            else:
                be.step(s, cur, scale, compute)
            self.counters.steps.append((s, s % 2))
            used[s % 2] = be.event(compute)
            if s + 1 < n_cp:
                # slot nxt was read by step s - 1; slot cur was filled by the hop before this step
                # (or, at step 0, by the placement on the compute stream)
                be.wait(copy, placed if s == 0 else used[(s + 1) % 2])
                if not in_kernel:
                    be.shift(cur, nxt, self.world == 1, copy)
                if self.world > 1:
                    send = [be.region(cur, x, R - 1) for x in range(4)]
                    recv = [be.region(nxt, x, 0) for x in range(4)]
                    self.transport.exchange(send, recv, copy)
                for i in range(R):
                    self.counters.kv[i] += kv_blk
                    self.counters.tables[i] += tab_blk
                arrived = be.event(copy)
            if timeline is not None:
                ce, xe = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                ce.record(compute)
                xe.record(copy)
                timeline.append((ce, xe))
        be.finalize(out, lse, compute)
        return out, lse


def local_tokens(T: int, n_cp: int, layout: int, rank0: int, R: int):
    """Natural token ids of ranks rank0 .. rank0 + R - 1, rank-major, each rank in its local layout
    order (the order ``RingProcess.forward`` takes its tokens in). Host-side index arithmetic only."""
    import numpy as np
    n = T // n_cp
    j = np.arange(n, dtype=np.int64)
    out = []
    for r in range(rank0, rank0 + R):
        if layout == 0:
            out.append(r * n + j)
        elif layout == 1:
            m = T // (2 * n_cp)
            out.append(np.where(j < m, r * m + j, (2 * n_cp - 1 - r) * m + (j - m)))
        else:
            out.append(j * n_cp + r)
    return np.concatenate(out)
