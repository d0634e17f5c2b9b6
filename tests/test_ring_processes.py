"""The multi-process ring's host protocol on CPU ("Pass them around a ring": each rank sends the
block it holds to its right neighbour and receives the next from its left): gloo ranks, each
holding R of the plan's n_cp ranks, with a stand-in for the device side whose blocks are tagged
with their source rank. Checked at every step: which block each rank holds (source (r - s) mod
n_cp), that its position table travelled with it, which stage slot is computed on, and that each
rank received exactly the key/value bytes the oracle counts (4 B n d_kv (n_cp - 1)).
No kernel is launched; the library is loaded only for its slot layout (cpattn_dist_sizes)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from context_ring_attention_blockwise_gb300 import _build
import context_ring_attention_blockwise_gb300 as cp
from context_ring_attention_blockwise_gb300.ring import HostTransport, RingProcess, local_tokens

B, T, H, NKV, D = 2, 2048, 4, 2, 64


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()


class TaggedBlocks:
    """The device side of one process with CPU tensors: slots laid out as the library lays them
    out, every key/value block filled with a tag of its source rank, the position region with the
    source rank's natural positions (from the oracle's layout map). step() checks what each rank
    holds; shift() moves blocks between the process's ranks as cpattn_dist_shift does."""

    def __init__(self, plan, B, rank0, R):
        self.plan, self.B, self.rank0, self.R = plan, B, rank0, R
        ws_bytes, slot_bytes, self.offsets, self.blocks = plan.dist_sizes(B, R)
        self.slots = [torch.zeros(slot_bytes, dtype=torch.uint8), torch.zeros(slot_bytes, dtype=torch.uint8)]
        self.device = torch.device("cpu")
        self.map = oracle.get().layout_map(plan.T, plan.n_cp, plan.layout)   # [n_cp][n] natural tokens
        self.seen = []

    def region(self, slot, x, i):
        o = self.offsets[x] + i * self.blocks[x]
        return slot[o:o + self.blocks[x]]

    def event(self, stream):
        return None

    @staticmethod
    def wait(stream, event):
        pass

    def begin(self, q, k, v, pos, slot, stream):
        for i in range(self.R):
            r = self.rank0 + i
            self.region(slot, 0, i).fill_(1 + r)
            self.region(slot, 1, i).fill_(101 + r)
            self.region(slot, 2, i).view(torch.int32).copy_(torch.from_numpy(self.map[r].astype(np.int32)))
            self.region(slot, 3, i).fill_(201 + r)

    def step(self, s, slot, scale, stream):
        n_cp = self.plan.n_cp
        for i in range(self.R):
            r = self.rank0 + i
            src = (r - s) % n_cp
            k = self.region(slot, 0, i)
            assert int(k.min()) == int(k.max()) == 1 + src, f"rank {r} step {s}: holds K of {int(k[0]) - 1}, not {src}"
            assert int(self.region(slot, 1, i)[0]) == 101 + src
            pos = self.region(slot, 2, i).view(torch.int32).numpy()
            assert np.array_equal(pos, self.map[src]), f"rank {r} step {s}: positions did not travel with the block"
            assert int(self.region(slot, 3, i).max()) == 201 + src
            self.seen.append((s, r, src))

    def shift(self, src, dst, wrap, stream):
        R = self.R
        for x in range(4):
            o, b = self.offsets[x], self.blocks[x]
            if R > 1:
                dst[o + b:o + b * R] = src[o:o + b * (R - 1)].clone()
            if wrap:
                dst[o:o + b] = src[o + b * (R - 1):o + b * R]

    def finalize(self, out, lse, stream):
        out.zero_()
        lse.zero_()


class TaggedBlocksStepShift(TaggedBlocks):
    """The same stand-in with cpattn_dist_step_shift: the step, then the shift from its slot into
    the next, both regions and tables, leaving local rank 0's block alone unless wrap (the
    transport fills it)."""

    def step_shift(self, s, slot, next_slot, wrap, scale, stream):
        assert next_slot is not slot
        self.step(s, slot, scale, stream)
        if not wrap:   # the transport's block must come from the transport, not from this shift
            for x in range(4):
                self.region(next_slot, x, 0).fill_(255)
        self.shift(slot, next_slot, wrap, stream)


def _run_ring(plan, rank, world, transport, step_shift=False):
    R = plan.n_cp // world
    be = (TaggedBlocksStepShift if step_shift else TaggedBlocks)(plan, B, rank * R, R)
    ring = RingProcess(plan, B, rank=rank, world=world, transport=transport, backend=be)
    n = plan.T // plan.n_cp
    q = torch.zeros((B, R * n, H, D), dtype=torch.bfloat16)
    kv = torch.zeros((B, R * n, NKV, D), dtype=torch.bfloat16)
    ring.forward(q, kv, kv)
    return ring, be


def _check(plan, rank, world, ring, be):
    R, n_cp, n = plan.n_cp // world, plan.n_cp, plan.T // plan.n_cp
    expect = [(s, r, (r - s) % n_cp) for s in range(n_cp) for r in range(rank * R, rank * R + R)]
    assert be.seen == expect
    assert ring.counters.steps == [(s, s % 2) for s in range(n_cp)]
    want = oracle.get().kv_bytes_recv(B, n, NKV, D, n_cp)
    assert ring.counters.kv == [want] * R, (ring.counters.kv, want)
    n_qt = -(-n // 128)
    assert ring.counters.tables == [(n_cp - 1) * (4 * n + 16 * n_qt)] * R


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, n_cp, layout, step_shift=False):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        plan = cp.Plan(T, H, NKV, D, n_cp, layout, True)
        ring, be = _run_ring(plan, rank, world, HostTransport(rank, world), step_shift)
        _check(plan, rank, world, ring, be)
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "striped"])
def test_one_process_holds_the_whole_ring(layout):
    plan = cp.Plan(T, H, NKV, D, 8, layout, True)
    ring, be = _run_ring(plan, 0, 1, None)
    _check(plan, 0, 1, ring, be)


@pytest.mark.parametrize("world,n_cp,layout", [(2, 4, "zigzag"), (2, 2, "contiguous"), (4, 4, "striped"),
                                               (2, 8, "striped")])
def test_gloo_ranks_pass_blocks_around_the_ring(world, n_cp, layout):
    mp.spawn(_rank_main, args=(world, _free_port(), n_cp, layout), nprocs=world, join=True)


@pytest.mark.parametrize("layout", ["zigzag", "striped"])
def test_one_process_ring_with_the_shift_in_the_step(layout):
    """The step-and-shift protocol (cpattn_dist_step_shift) with one process holding the ring."""
    plan = cp.Plan(T, H, NKV, D, 8, layout, True)
    ring, be = _run_ring(plan, 0, 1, None, step_shift=True)
    _check(plan, 0, 1, ring, be)


@pytest.mark.parametrize("world,n_cp,layout", [(2, 4, "zigzag"), (4, 4, "striped"), (2, 8, "contiguous")])
def test_gloo_ranks_with_the_shift_in_the_step(world, n_cp, layout):
    """The step-and-shift protocol across gloo ranks: the shift leaves local rank 0's block to the
    transport, which must fill it before the next step reads it."""
    mp.spawn(_rank_main, args=(world, _free_port(), n_cp, layout, True), nprocs=world, join=True)


def test_local_tokens_follow_the_oracle_layout():
    for layout in (0, 1, 2):
        m = oracle.get().layout_map(T, 8, layout)
        for rank0, R in ((0, 8), (2, 2), (7, 1)):
            assert np.array_equal(local_tokens(T, 8, layout, rank0, R), m[rank0:rank0 + R].reshape(-1))


def test_ring_process_refuses_uneven_or_untransported_splits():
    plan = cp.Plan(T, H, NKV, D, 4, "zigzag", True)
    with pytest.raises(ValueError):
        RingProcess(plan, B, rank=0, world=3, backend=object())
    with pytest.raises(ValueError):
        RingProcess(plan, B, rank=0, world=2, backend=object())


def test_dist_sizes_and_host_checks():
    plan = cp.Plan(T, H, NKV, D, 4, "zigzag", True)
    n = T // 4
    ws, slot, off, blk = plan.dist_sizes(B, 2)
    assert blk[0] == blk[1] == 2 * B * n * NKV * D and blk[2] == 4 * n and blk[3] == 16 * ((n + 127) // 128)
    assert all(o % 1024 == 0 for o in off) and off[0] == 0
    assert slot >= off[3] + 2 * blk[3] and ws > 2 * B * 2 * n * H * D
    # R out of range, steps before begin: refused on the host before any launch
    L = cp.lib()
    import ctypes
    sz = ctypes.c_size_t()
    assert L.cpattn_dist_sizes(plan.handle, B, 5, ctypes.byref(sz), None, None, None) == 1
    assert L.cpattn_dist_sizes(plan.handle, B, 0, ctypes.byref(sz), None, None, None) == 1
    buf = ctypes.c_void_p(1 << 20)
    assert L.cpattn_dist_step(plan.handle, B, 0, 2, 0, 0.0, buf, slot, buf, ws, None) == 1
    assert "cpattn_dist_begin" in L.cpattn_last_error().decode()
    assert L.cpattn_dist_finalize(plan.handle, B, 0, 2, buf, buf, buf, ws, None) == 1
