"""The ring across processes on the GPU ("Pass them around a ring"): each process holds R of the
plan's n_cp ranks, computes its ranks' queries against the blocks they hold with the library's
kernels, and passes the block that crosses to the next process through a transport.

* One process holding the whole ring (the library's own shift passes the last block to the first
  rank): against the oracle, and bit-identical to the single-process ring-step path, which runs the
  same kernel over the same blocks in the same order.
* Two processes on one GPU exchanging the crossing block over gloo through host memory: each
  process's rows against the oracle and bit-identical to the ring-step path. The processes'
  kernels never wait on each other; only the host exchange orders them.
* Document masks (a per-query lower bound that stays with the queries) in one and two processes,
  against the oracle's document-id definition."""
import os
import socket
import tempfile

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import context_ring_attention_blockwise_gb300 as cp
from context_ring_attention_blockwise_gb300.ring import HostTransport, RingProcess, local_tokens
from tests.gpu_util import compare, inputs, to_device_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from context_ring_attention_blockwise_gb300 import _build
    _build.build()


def _shard(x, tokens):
    return np.ascontiguousarray(x[:, tokens])


def _run_process(plan, B, rank, world, q, k, v, pos, transport, scale=None, lo=None):
    """This process's rows: natural token ids, o [B, R n, h, d] fp32, lse [B, h, R n]."""
    R = plan.n_cp // world
    toks = local_tokens(plan.T, plan.n_cp, plan.layout, rank * R, R)
    ring = RingProcess(plan, B, rank=rank, world=world, transport=transport, device="cuda")
    posd = None if pos is None else torch.from_numpy(np.ascontiguousarray(pos[toks], dtype=np.int32)).cuda()
    lod = None if lo is None else torch.from_numpy(np.ascontiguousarray(lo[toks], dtype=np.int32)).cuda()
    o, lse = ring.forward(to_device_bf16(_shard(q, toks)), to_device_bf16(_shard(k, toks)),
                          to_device_bf16(_shard(v, toks)), pos=posd, scale=scale, lo=lod)
    torch.cuda.synchronize()
    cp.check(plan, ring.backend.ws)
    return toks, o.float().cpu().numpy(), lse.cpu().numpy(), ring


def _ring_step_reference(q, k, v, plan, pos=None, scale=None):
    posd = None if pos is None else torch.from_numpy(np.ascontiguousarray(pos, dtype=np.int32)).cuda()
    o, lse = cp.ring_forward(to_device_bf16(q), to_device_bf16(k), to_device_bf16(v), plan, pos=posd, scale=scale)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), lse.cpu().numpy()


CASES = [
    # B, T, h, n_kv, d, n_cp, layout, causal
    (1, 2048, 4, 2, 128, 4, "zigzag", True),
    (2, 1024, 2, 2, 64, 4, "contiguous", True),
    (1, 1536, 4, 1, 128, 4, "striped", True),
    (1, 1024, 4, 4, 128, 2, "contiguous", False),
    (1, 1560, 2, 2, 128, 4, "zigzag", True),     # 390 tokens per rank: a short last tile
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[6]}-T{c[1]}-d{c[4]}-{'causal' if c[7] else 'full'}" for c in CASES])
def test_one_process_ring_matches_oracle_and_ring_step_path(case):
    B, T, h, n_kv, d, n_cp, layout, causal = case
    q, k, v = inputs(77 + T, B, T, h, n_kv, d)
    plan = cp.Plan(T, h, n_kv, d, n_cp, layout, causal)
    toks, o, lse, ring = _run_process(plan, B, 0, 1, q, k, v, None, None)
    ref_o, ref_lse = oracle.get().attention(q, k, v, causal=causal, rows=toks)
    compare(o, lse, ref_o, ref_lse, what=f"one-process ring {case}")
    ro, rl = _ring_step_reference(q, k, v, plan)
    assert np.array_equal(o, ro[:, toks]) and np.array_equal(lse, rl[:, :, toks]), "differs from the ring-step path"
    n = T // n_cp
    assert ring.counters.kv == [oracle.get().kv_bytes_recv(B, n, n_kv, d, n_cp)] * n_cp


def test_one_process_ring_shift_in_kernel_or_on_copy_stream():
    """The shift between a process's own ranks done by the step kernels gives the same blocks as
    the shift by copies on a copy stream: bit-identical outputs."""
    B, T, h, n_kv, d, n_cp = 1, 1560, 2, 2, 128, 4
    q, k, v = inputs(95, B, T, h, n_kv, d)
    plan = cp.Plan(T, h, n_kv, d, n_cp, "zigzag", True)
    toks = local_tokens(plan.T, plan.n_cp, plan.layout, 0, n_cp)
    outs = []
    for in_kernel in (True, False):
        ring = RingProcess(plan, B, rank=0, world=1, device="cuda")
        o, lse = ring.forward(to_device_bf16(_shard(q, toks)), to_device_bf16(_shard(k, toks)),
                              to_device_bf16(_shard(v, toks)), shift_in_kernel=in_kernel)
        torch.cuda.synchronize()
        cp.check(plan, ring.backend.ws)
        outs.append((o.view(torch.int16).clone(), lse.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_one_process_ring_with_position_ids():
    B, T, h, n_kv, d, n_cp = 1, 1024, 2, 1, 128, 4
    q, k, v = inputs(91, B, T, h, n_kv, d)
    pos = np.random.default_rng(5).permutation(T).astype(np.int32)
    plan = cp.Plan(T, h, n_kv, d, n_cp, "zigzag", True)
    toks, o, lse, _ = _run_process(plan, B, 0, 1, q, k, v, pos, None)
    ref_o, ref_lse = oracle.get().attention(q, k, v, causal=True, pos=pos, rows=toks)
    compare(o, lse, ref_o, ref_lse, what="one-process ring, permuted positions")


def _documents(T, seed):
    """Document ids of a packed sequence (runs of 100..900 tokens) and each token's lower bound."""
    rng = np.random.default_rng(seed)
    lengths, left = [], T
    while left > 0:
        lengths.append(min(left, int(rng.integers(100, 900))))
        left -= lengths[-1]
    doc = np.repeat(np.arange(len(lengths)), lengths).astype(np.int32)
    lo = np.repeat(np.concatenate([[0], np.cumsum(lengths)[:-1]]), lengths).astype(np.int32)
    return doc, lo


@pytest.mark.parametrize("layout", ["zigzag", "striped"])
def test_one_process_ring_with_document_masks(layout):
    B, T, h, n_kv, d, n_cp = 1, 2048, 4, 2, 128, 4
    q, k, v = inputs(93, B, T, h, n_kv, d)
    doc, lo = _documents(T, 4)
    plan = cp.Plan(T, h, n_kv, d, n_cp, layout, True)
    toks, o, lse, _ = _run_process(plan, B, 0, 1, q, k, v, None, None, lo=lo)
    ref_o, ref_lse = oracle.get().attention_docs(q, k, v, doc, causal=True, rows=toks)
    compare(o, lse, ref_o, ref_lse, what=f"one-process ring, document masks, {layout}")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, case, outdir, with_docs=False):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        B, T, h, n_kv, d, n_cp, layout, causal = case
        torch.cuda.set_device(0)
        q, k, v = inputs(177 + T, B, T, h, n_kv, d)
        plan = cp.Plan(T, h, n_kv, d, n_cp, layout, causal)
        lo = _documents(T, 6)[1] if with_docs else None
        toks, o, lse, ring = _run_process(plan, B, rank, world, q, k, v, None, HostTransport(rank, world), lo=lo)
        np.savez(os.path.join(outdir, f"rank{rank}.npz"), toks=toks, o=o, lse=lse, kv=np.array(ring.counters.kv))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case", [CASES[0], CASES[2], CASES[4], (1, 1024, 2, 2, 128, 2, "zigzag", True)],
                         ids=["zigzag", "striped", "ragged", "one-rank-each"])
def test_two_processes_on_one_gpu_exchange_through_host_memory(case):
    B, T, h, n_kv, d, n_cp, layout, causal = case
    world = 2
    with tempfile.TemporaryDirectory() as outdir:
        mp.start_processes(_rank_main, args=(world, _free_port(), case, outdir), nprocs=world, join=True,
                           start_method="spawn")
        parts = [dict(np.load(os.path.join(outdir, f"rank{r}.npz"))) for r in range(world)]
    q, k, v = inputs(177 + T, B, T, h, n_kv, d)
    plan = cp.Plan(T, h, n_kv, d, n_cp, layout, causal)
    ro, rl = _ring_step_reference(q, k, v, plan)
    n = T // n_cp
    for r, part in enumerate(parts):
        toks = part["toks"]
        ref_o, ref_lse = oracle.get().attention(q, k, v, causal=causal, rows=toks)
        compare(part["o"], part["lse"], ref_o, ref_lse, what=f"process {r} of 2")
        assert np.array_equal(part["o"], ro[:, toks]) and np.array_equal(part["lse"], rl[:, :, toks])
        assert list(part["kv"]) == [oracle.get().kv_bytes_recv(B, n, n_kv, d, n_cp)] * (n_cp // world)


def test_two_processes_with_document_masks():
    B, T, h, n_kv, d, n_cp, layout, causal = CASES[0]
    world = 2
    with tempfile.TemporaryDirectory() as outdir:
        mp.start_processes(_rank_main, args=(world, _free_port(), CASES[0], outdir, True), nprocs=world, join=True,
                           start_method="spawn")
        parts = [dict(np.load(os.path.join(outdir, f"rank{r}.npz"))) for r in range(world)]
    q, k, v = inputs(177 + T, B, T, h, n_kv, d)
    doc, _ = _documents(T, 6)
    for r, part in enumerate(parts):
        ref_o, ref_lse = oracle.get().attention_docs(q, k, v, doc, causal=True, rows=part["toks"])
        compare(part["o"], part["lse"], ref_o, ref_lse, what=f"process {r} of 2, document masks")
