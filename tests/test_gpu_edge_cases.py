"""Degenerate shapes on the GPU: a handful of tokens per virtual rank (one query tile holding
1..16 valid rows), zigzag chunks of a single token, one rank, one head, GQA down to one KV head;
forward, backward and the Ulysses head split against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
import context_ring_attention_blockwise_gb300 as cp
from tests.gpu_util import compare, inputs, run, to_device_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from context_ring_attention_blockwise_gb300 import _build
    _build.build()


TINY = [
    # T, h, n_kv, d, n_cp
    (4, 1, 1, 64, 4),        # one token per rank
    (8, 2, 1, 64, 4),        # two per rank: zigzag chunks of one token
    (16, 4, 2, 128, 8),
    (64, 2, 2, 128, 16),     # four per rank over 16 ranks
    (1, 1, 1, 128, 1),       # a single token
    (24, 8, 1, 64, 2),       # GQA 8:1
]


def _layouts(T, n_cp):
    out = [0, 2]                                   # contiguous, striped
    if T % (2 * n_cp) == 0:
        out.append(1)                              # zigzag needs two chunks per rank
    return out


@pytest.mark.parametrize("case", TINY, ids=lambda c: "T{}_h{}_kv{}_d{}_cp{}".format(*c))
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
def test_tiny_forward(case, causal):
    T, h, n_kv, d, n_cp = case
    q, k, v = inputs(300 + T + h, 1, T, h, n_kv, d)
    ref_o, ref_lse = oracle.get().attention(q, k, v, causal=causal)
    for layout in _layouts(T, n_cp):
        o, lse, _, _ = run(q, k, v, n_cp, layout, causal)
        compare(o, lse, ref_o, ref_lse, what=f"tiny {case} layout {layout} causal {causal}")
        o, lse, _, _ = run(q, k, v, n_cp, layout, causal, path="ring")
        compare(o, lse, ref_o, ref_lse, what=f"tiny ring-step {case} layout {layout} causal {causal}")


@pytest.mark.parametrize("case", TINY, ids=lambda c: "T{}_h{}_kv{}_d{}_cp{}".format(*c))
def test_tiny_backward(case):
    from tests.test_gpu_backward import _compare, _run
    T, h, n_kv, d, n_cp = case
    q, k, v = inputs(310 + T + h, 1, T, h, n_kv, d)
    do = synth.normal_bf16(310 + T, 4, (1, T, h, d))
    rq, rk, rv = oracle.get().backward(q, k, v, do, causal=True)
    for layout in _layouts(T, n_cp):
        dq, dk, dv = _run(q, k, v, do, n_cp, layout, True)
        _compare(dq, rq, f"dq {case} layout {layout}")
        _compare(dk, rk, f"dk {case} layout {layout}")
        _compare(dv, rv, f"dv {case} layout {layout}")


@pytest.mark.parametrize("case", [(4, 4, 2, 64, 4), (8, 8, 1, 128, 8), (2, 2, 2, 64, 2)],
                         ids=lambda c: "T{}_h{}_kv{}_d{}_cp{}".format(*c))
def test_tiny_ulysses(case):
    T, h, n_kv, d, n_cp = case
    q, k, v = inputs(320 + T + h, 1, T, h, n_kv, d)
    plan = cp.UlyssesPlan(T, h, n_kv, d, n_cp, True)
    ws = cp.alloc_workspace(plan.workspace_size(1))
    o, lse = cp.ulysses_forward(*(to_device_bf16(x) for x in (q, k, v)), plan, ws=ws)
    torch.cuda.synchronize()
    cp.check(plan, ws)
    ref_o, ref_lse = oracle.get().attention(q, k, v, causal=True)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_lse, what=f"tiny ulysses {case}")


@pytest.mark.parametrize("bits,what", [(0x47C3, "99840"), (0x7F80, "inf"), (0xFFC0, "NaN")])
def test_v_outside_the_fp16_range_is_reported(bits, what):
    """The forward multiplies P by V in fp16: a V value beyond 65504 (or infinite, or NaN) cannot be
    converted, so the call computes nothing and cpattn_check says why; the next call with values in
    range clears the record."""
    T, h, n_kv, d, n_cp = 512, 2, 2, 128, 4
    q, k, v = inputs(7, 1, T, h, n_kv, d)
    bad = v.copy()
    bad[0, 100, 1, 5] = bits
    plan = cp.Plan(T, h, n_kv, d, n_cp, "zigzag", True)
    ws = cp.alloc_workspace(plan.workspace_size(1))
    qd, kd = to_device_bf16(q), to_device_bf16(k)
    cp.forward(qd, kd, to_device_bf16(bad), plan, ws=ws)
    torch.cuda.synchronize()
    with pytest.raises(cp.CpattnError) as e:
        cp.check(plan, ws)
    assert e.value.status == 1 and "fp16 range" in str(e.value), what
    o, lse = cp.forward(qd, kd, to_device_bf16(v), plan, ws=ws)
    torch.cuda.synchronize()
    cp.check(plan, ws)
    ref_o, ref_lse = oracle.get().attention(q, k, v, causal=True)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_lse, what="after an out-of-range call")


def test_v_at_the_fp16_limits_is_exact():
    """V values at 65504 (the largest fp16) and below 2^-14 (fp16 subnormals) go through."""
    T, h, n_kv, d, n_cp = 256, 2, 1, 64, 2
    q, k, v = inputs(8, 1, T, h, n_kv, d)
    v = v.copy()
    v[0, :, 0, 0] = 0x477F          # 65280, exact in fp16
    v[0, :, 0, 1] = 0x3880          # 2^-14 * 1.0 = 6.1e-5
    v[0, :, 0, 2] = 0x3400          # 2^-23: an fp16 subnormal
    o, lse, plan, ws = run(q, k, v, n_cp, 0)
    ref_o, ref_lse = oracle.get().attention(q, k, v, causal=True)
    compare(o, lse, ref_o, ref_lse, what="V at the fp16 limits")
