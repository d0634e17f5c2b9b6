"""Document masks for packed sequences (cpattn_forward_masked) against the oracle's document-id
definition: a query sees only keys of its own document, at or before it. The library takes the
mask as a lower bound per query (the first token of its document) with positions 0..T-1; the
tests build that bound from document ids, so parity here also checks that the two statements of
the mask agree."""
import numpy as np
import pytest
import torch

import oracle
import synth
import context_ring_attention_blockwise_gb300 as cp
from synth.configs import CONTIGUOUS, ZIGZAG, STRIPED
from tests.gpu_util import compare, to_device_bf16, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from context_ring_attention_blockwise_gb300 import _build
    _build.build()


def packed_documents(T, seed, min_len=1, max_len=300):
    """Seeded document lengths summing to T; returns (doc id per token, first token per token)."""
    rng = np.random.default_rng(seed)
    lengths = []
    while sum(lengths) < T:
        lengths.append(int(rng.integers(min_len, max_len + 1)))
    lengths[-1] -= sum(lengths) - T
    if lengths[-1] == 0:
        lengths.pop()
    doc = np.repeat(np.arange(len(lengths)), lengths).astype(np.int32)
    starts = np.concatenate([[0], np.cumsum(lengths)[:-1]]).astype(np.int32)
    return doc, starts[doc]


def _masked(q, k, v, lo, n_cp, layout):
    B, T, h, d = q.shape
    plan = cp.Plan(T, h, k.shape[2], d, n_cp, layout, True)
    qd, kd, vd = (to_device_bf16(x) for x in (q, k, v))
    ws = cp.alloc_workspace(plan.workspace_size(B))
    o, lse = cp.forward_masked(qd, kd, vd, plan, torch.from_numpy(lo).cuda(), ws=ws)
    torch.cuda.synchronize()
    cp.check(plan, ws)
    return o.float().cpu().numpy(), lse.cpu().numpy()


CASES = [
    # T, h, n_kv, d, n_cp, layout, max document length
    (1024, 2, 2, 64, 4, CONTIGUOUS, 300),
    (1024, 4, 2, 128, 4, ZIGZAG, 300),
    (1536, 4, 1, 128, 4, STRIPED, 500),
    (1040, 2, 1, 128, 4, ZIGZAG, 40),       # many short documents, ragged ranks
    (2048, 8, 2, 128, 8, ZIGZAG, 2048),     # a few long documents
]


@pytest.mark.parametrize("case", CASES, ids=[f"T{c[0]}_h{c[1]}_kv{c[2]}_d{c[3]}_cp{c[4]}_{synth.LAYOUT_NAMES[c[5]]}_"
                                             f"max{c[6]}" for c in CASES])
def test_document_mask_matches_oracle(case):
    T, h, n_kv, d, n_cp, layout, max_len = case
    q, k, v = inputs(50 + T + h, 1, T, h, n_kv, d)
    doc, lo = packed_documents(T, seed=T + max_len, max_len=max_len)
    o, lse = _masked(q, k, v, lo, n_cp, layout)
    ref_o, ref_lse = oracle.get().attention_docs(q, k, v, doc, causal=True)
    compare(o, lse, ref_o, ref_lse, what=f"documents {case}")


def test_lower_bound_zero_is_the_plain_forward():
    """lo = 0 everywhere removes no key: bit-identical to cpattn_forward."""
    q, k, v = inputs(61, 1, 1024, 4, 2, 128)
    lo = np.zeros(1024, dtype=np.int32)
    o, lse = _masked(q, k, v, lo, 4, ZIGZAG)
    plan = cp.Plan(1024, 4, 2, 128, 4, ZIGZAG, True)
    o2, lse2 = cp.forward(*(to_device_bf16(x) for x in (q, k, v)), plan)
    assert np.array_equal(o, o2.float().cpu().numpy()) and np.array_equal(lse, lse2.cpu().numpy())


def test_document_mask_rejects_non_causal_plan():
    plan = cp.Plan(512, 2, 2, 64, 4, CONTIGUOUS, False)
    q, k, v = inputs(62, 1, 512, 2, 2, 64)
    with pytest.raises(cp.CpattnError) as e:
        cp.forward_masked(*(to_device_bf16(x) for x in (q, k, v)), plan, torch.zeros(512, dtype=torch.int32).cuda())
    assert e.value.status == 2


def test_documents_gqa_16k_sampled():
    """The GQA 4:1 zigzag T=16384 shape with packed documents of 256..4096 tokens: sampled rows."""
    w = synth.workload("gqa_zigzag_T16k")
    q, k, v = synth.make_qkv(w)
    doc, lo = packed_documents(w.T, seed=7, min_len=256, max_len=4096)
    o, lse = _masked(q, k, v, lo, w.n_cp, w.layouts[0])
    rows = synth.sample_rows(w.T, w.n_cp, 256, seed=w.seed)
    ref_o, ref_lse = oracle.get().attention_docs(q, k, v, doc, causal=True, rows=rows)
    compare(o[:, rows], lse[:, :, rows], ref_o, ref_lse, what="16K documents")


# ---- the backward under document masks -------------------------------------------------------

def _masked_backward(q, k, v, do, lo, n_cp, layout):
    B, T, h, d = q.shape
    plan = cp.Plan(T, h, k.shape[2], d, n_cp, layout, True)
    qd, kd, vd, dod = (to_device_bf16(x) for x in (q, k, v, do))
    lod = torch.from_numpy(lo).cuda()
    o, lse = cp.forward_masked(qd, kd, vd, plan, lod)
    ws = cp.alloc_workspace(plan.backward_workspace_size(B))
    dq, dk, dv = cp.backward(qd, kd, vd, o, lse, dod, plan, ws=ws, lo=lod)
    torch.cuda.synchronize()
    cp.check(plan, ws)
    return tuple(x.float().cpu().numpy() for x in (dq, dk, dv))


BWD_CASES = [
    (1024, 4, 2, 128, 4, ZIGZAG, 300),
    (1040, 2, 1, 64, 4, CONTIGUOUS, 40),
    (1536, 4, 1, 128, 4, STRIPED, 700),
]


@pytest.mark.parametrize("case", BWD_CASES, ids=[f"T{c[0]}_h{c[1]}_kv{c[2]}_d{c[3]}_cp{c[4]}_"
                                                 f"{synth.LAYOUT_NAMES[c[5]]}_max{c[6]}" for c in BWD_CASES])
def test_document_mask_backward_matches_oracle(case):
    from tests.test_gpu_backward import _compare
    T, h, n_kv, d, n_cp, layout, max_len = case
    q, k, v = inputs(70 + T + h, 1, T, h, n_kv, d)
    do = synth.normal_bf16(70 + T, 4, (1, T, h, d))
    doc, lo = packed_documents(T, seed=T + 3 * max_len, max_len=max_len)
    dq, dk, dv = _masked_backward(q, k, v, do, lo, n_cp, layout)
    rq, rk, rv = oracle.get().backward(q, k, v, do, causal=True, doc=doc)
    _compare(dq, rq, "dq")
    _compare(dk, rk, "dk")
    _compare(dv, rv, "dv")


def test_document_mask_backward_lower_bound_zero_is_plain():
    q, k, v = inputs(71, 1, 1024, 4, 2, 128)
    do = synth.normal_bf16(71, 4, (1, 1024, 4, 128))
    a = _masked_backward(q, k, v, do, np.zeros(1024, dtype=np.int32), 4, ZIGZAG)
    plan = cp.Plan(1024, 4, 2, 128, 4, ZIGZAG, True)
    qd, kd, vd, dod = (to_device_bf16(x) for x in (q, k, v, do))
    o, lse = cp.forward(qd, kd, vd, plan)
    b = cp.backward(qd, kd, vd, o, lse, dod, plan)
    for x, y in zip(a, b):
        assert np.array_equal(x, y.float().cpu().numpy())


def test_document_mask_backward_gqa_16k_sampled():
    """The GQA 4:1 zigzag T=16384 shape with packed documents of 256..4096 tokens: dq of sampled
    rows, dk/dv of sampled keys (each sees only the queries of its own document)."""
    from tests.test_gpu_backward import _compare
    w = synth.workload("gqa_zigzag_T16k")
    q, k, v = synth.make_qkv(w)
    do = synth.normal_bf16(w.seed, 4, (w.B, w.T, w.h, w.d))
    doc, lo = packed_documents(w.T, seed=9, min_len=256, max_len=4096)
    dq, dk, dv = _masked_backward(q, k, v, do, lo, w.n_cp, w.layouts[0])
    rows = synth.sample_rows(w.T, w.n_cp, 32, seed=w.seed)
    keys = np.sort(np.random.default_rng(11).choice(w.T, size=64, replace=False))
    rq, rk, rv = oracle.get().backward(q, k, v, do, causal=True, doc=doc, rows=rows, keys=keys)
    _compare(dq[:, rows], rq, "dq (sampled rows)")
    _compare(dk[:, keys], rk, "dk (sampled keys)")
    _compare(dv[:, keys], rv, "dv (sampled keys)")
