"""GPU parity of the backward as ring steps (cpattn_backward_begin, cpattn_backward_ring_step for
steps 0..n_cp-1, cpattn_backward_finalize) against the fp64 oracle's gradients, with the bound
of the fused backward's tests (the same roundings meet in each term; only the fp32 summation
order across ring steps differs). Each step's K/V blocks and the circulating fp32 dK/dV partial
sums hop between the ranks' slots on a copy stream, and the last hop returns every block's
gradient to its owner, so these tests also check that data movement."""
import numpy as np
import pytest
import torch

import oracle
import synth
import context_ring_attention_blockwise_gb300 as cp
from synth.configs import CONTIGUOUS, ZIGZAG, STRIPED
from tests.gpu_util import to_device_bf16
from tests.test_gpu_backward import _compare, _inputs, _run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from context_ring_attention_blockwise_gb300 import _build
    _build.build()


def _ring(q, k, v, do, n_cp, layout, causal, pos=None, scale=None, streams=None):
    B, T, h, d = q.shape
    plan = cp.Plan(T, h, k.shape[2], d, n_cp, layout, causal)
    qd, kd, vd, dod = (to_device_bf16(x) for x in (q, k, v, do))
    posd = torch.from_numpy(np.ascontiguousarray(pos, dtype=np.int32)).cuda() if pos is not None else None
    o, lse = cp.forward(qd, kd, vd, plan, pos=posd, scale=scale)
    ws = cp.alloc_workspace(plan.backward_ring_workspace_size(B))
    compute, copy = streams if streams is not None else (None, None)
    dq, dk, dv = cp.ring_backward(qd, kd, vd, o, lse, dod, plan, pos=posd, scale=scale, ws=ws, stream=compute,
                                  copy_stream=copy)
    torch.cuda.synchronize()
    cp.check(plan, ws)
    return tuple(x.float().cpu().numpy() for x in (dq, dk, dv))


CASES = [
    # T, h, n_kv, d, n_cp, layout, causal
    (512, 2, 2, 64, 4, CONTIGUOUS, True),
    (512, 4, 2, 128, 4, ZIGZAG, True),
    (768, 4, 1, 128, 4, STRIPED, True),
    (512, 2, 2, 128, 2, CONTIGUOUS, False),
    (600, 2, 1, 64, 2, CONTIGUOUS, True),        # ragged: 300 tokens per rank
    (1040, 4, 2, 128, 4, ZIGZAG, True),          # ragged: 260 tokens per rank
    (384, 2, 1, 128, 1, CONTIGUOUS, True),       # one rank: the return hop is the identity
    (1024, 8, 2, 64, 8, STRIPED, False),         # eight ranks, non-causal
]


@pytest.mark.parametrize("case", CASES, ids=[f"T{c[0]}_h{c[1]}_kv{c[2]}_d{c[3]}_cp{c[4]}_{synth.LAYOUT_NAMES[c[5]]}_"
                                             f"{'causal' if c[6] else 'full'}" for c in CASES])
def test_ring_backward_matches_oracle(case):
    T, h, n_kv, d, n_cp, layout, causal = case
    q, k, v, do = _inputs(31 + T + h, 1, T, h, n_kv, d)
    dq, dk, dv = _ring(q, k, v, do, n_cp, layout, causal)
    rq, rk, rv = oracle.get().backward(q, k, v, do, causal=causal)
    _compare(dq, rq, "dq")
    _compare(dk, rk, "dk")
    _compare(dv, rv, "dv")


def test_ring_backward_positions_scale_batch():
    B, T, h, n_kv, d = 2, 512, 4, 2, 64
    q, k, v, do = _inputs(79, B, T, h, n_kv, d)
    pos = np.sort(np.random.default_rng(6).integers(0, 3 * T, size=T)).astype(np.int32)
    dq, dk, dv = _ring(q, k, v, do, 4, ZIGZAG, True, pos=pos, scale=0.07)
    rq, rk, rv = oracle.get().backward(q, k, v, do, causal=True, pos=pos, scale=0.07)
    _compare(dq, rq, "dq")
    _compare(dk, rk, "dk")
    _compare(dv, rv, "dv")


def test_ring_backward_agrees_with_fused_and_repeats_exactly():
    """Against the fused backward: the same gradients up to the fp32 order of the per-step sums
    (a bf16 rounding apart at most). Run twice on explicit streams: bit-identical."""
    q, k, v, do = _inputs(80, 1, 1024, 8, 2, 128)
    fused = _run(q, k, v, do, 8, ZIGZAG, True)
    streams = (torch.cuda.Stream(), torch.cuda.Stream())
    a = _ring(q, k, v, do, 8, ZIGZAG, True, streams=streams)
    b = _ring(q, k, v, do, 8, ZIGZAG, True, streams=streams)
    for x, y, f, name in zip(a, b, fused, ("dq", "dk", "dv")):
        assert np.array_equal(x, y), f"{name}: repeated ring backward differs"
        # one bf16 ulp of the value, plus the fp32 order difference of sums of up to 8192 terms
        # (at most ~8192 * 2^-24 of the largest term, taken as 2^-10 of the largest gradient)
        tol = 2.0 ** -7 * np.abs(f) + 2.0 ** -10 * float(np.max(np.abs(f)))
        assert np.all(np.abs(x - f) <= tol), f"{name}: ring-step and fused backward differ by {np.max(np.abs(x - f)):.3e}"


def test_ring_backward_steps_one_by_one():
    """begin, each step as its own C-ABI call on a compute and a copy stream, finalize; a step out
    of order or a second finalize is refused on the host."""
    T, h, n_kv, d, n_cp = 512, 4, 1, 128, 4
    q, k, v, do = _inputs(81, 1, T, h, n_kv, d)
    plan = cp.Plan(T, h, n_kv, d, n_cp, ZIGZAG, True)
    qd, kd, vd, dod = (to_device_bf16(x) for x in (q, k, v, do))
    o, lse = cp.forward(qd, kd, vd, plan)
    ws = cp.alloc_workspace(plan.backward_ring_workspace_size(1))
    compute, copy = torch.cuda.current_stream(), torch.cuda.Stream()
    cp.backward_begin(qd, kd, vd, o, lse, dod, plan, ws, stream=compute)
    with pytest.raises(cp.CpattnError):
        cp.backward_ring_step(plan, 1, 1, ws, compute=compute, copy=copy)        # step 0 comes first
    for s in range(n_cp):
        cp.backward_ring_step(plan, 1, s, ws, compute=compute, copy=copy)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    cp.backward_finalize(plan, 1, ws, dq, dk, dv, stream=compute)
    with pytest.raises(cp.CpattnError):
        cp.backward_finalize(plan, 1, ws, dq, dk, dv, stream=compute)             # needs a new begin
    torch.cuda.synchronize()
    cp.check(plan, ws)
    rq, rk, rv = oracle.get().backward(q, k, v, do, causal=True)
    _compare(dq.float().cpu().numpy(), rq, "dq")
    _compare(dk.float().cpu().numpy(), rk, "dk")
    _compare(dv.float().cpu().numpy(), rv, "dv")


def test_ring_backward_workload_sampled():
    """The GQA 4:1 zigzag T=16384 workload (8 ranks): dq of sampled rows, dk/dv of the last 64
    keys, whose gradients travel through all eight ranks' slots before returning."""
    w = synth.workload("gqa_zigzag_T16k")
    q, k, v = synth.make_qkv(w)
    do = synth.normal_bf16(w.seed, 4, (w.B, w.T, w.h, w.d))
    dq, dk, dv = _ring(q, k, v, do, w.n_cp, w.layouts[0], w.causal)
    rows = synth.sample_rows(w.T, w.n_cp, 48, seed=w.seed)
    keys = np.arange(w.T - 64, w.T)
    rq, rk, rv = oracle.get().backward(q, k, v, do, causal=w.causal, rows=rows, keys=keys)
    _compare(dq[:, rows], rq, "dq (sampled rows)")
    _compare(dk[:, keys], rk, "dk (last keys)")
    _compare(dv[:, keys], rv, "dv (last keys)")


def test_ring_paths_refuse_another_batch():
    """The ring steps and finalize must use the batch size the placement used; another one is
    refused on the host (CPATTN_ERR_INVALID), even with a workspace large enough for it."""
    q, k, v, do = _inputs(82, 1, 512, 2, 1, 64)
    plan = cp.Plan(512, 2, 1, 64, 4, ZIGZAG, True)
    qd, kd, vd, dod = (to_device_bf16(x) for x in (q, k, v, do))
    o, lse = cp.forward(qd, kd, vd, plan)
    copy = torch.cuda.Stream()
    ws = cp.alloc_workspace(plan.backward_ring_workspace_size(2))
    cp.backward_begin(qd, kd, vd, o, lse, dod, plan, ws)
    with pytest.raises(cp.CpattnError) as e:
        cp.backward_ring_step(plan, 2, 0, ws, copy=copy)
    assert e.value.status == 1
    wsf = cp.alloc_workspace(plan.ring_workspace_size(2))
    cp.permute(qd, kd, vd, plan, wsf)
    with pytest.raises(cp.CpattnError) as e:
        cp.ring_step(plan, 2, 0, wsf, copy=copy)
    assert e.value.status == 1
    torch.cuda.synchronize()
    cp.check(plan, wsf)
