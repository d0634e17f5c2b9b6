"""Document ids on the GPU ("What context parallelism communicates": masks "such as document masks
for packed sequences"): key u is visible to query t iff doc[u] == doc[t] (and pos[u] <= pos[t] for a
causal plan), with any ids in any order and documents split into pieces. Against the oracle's
document-id definition on every layout; bit-identical to the lower-bound form where documents are
contiguous (the two walks visit the same tiles with the same element masks); the all-gather form
bit-identical to the ring form."""
import numpy as np
import pytest
import torch

import oracle
import synth
import context_ring_attention_blockwise_gb300 as cp
from tests.gpu_util import compare, inputs, to_device_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from context_ring_attention_blockwise_gb300 import _build
    _build.build()


def pieces(T, seed, n_ids, lo=16, hi=400):
    """Runs of random length, each given one of n_ids ids at random: documents in pieces."""
    rng = np.random.default_rng(seed)
    out, left = [], T
    while left > 0:
        ln = min(left, int(rng.integers(lo, hi)))
        out.append(np.full(ln, int(rng.integers(0, n_ids)) * 13 + 7, dtype=np.int32))
        left -= ln
    return np.concatenate(out)


def run_docs(q, k, v, plan, doc, pos=None, allgather=False):
    posd = None if pos is None else torch.from_numpy(np.ascontiguousarray(pos, dtype=np.int32)).cuda()
    B = q.shape[0]
    ws = cp.alloc_workspace(plan.allgather_workspace_size(B) if allgather else plan.workspace_size(B))
    o, lse = cp.forward_docs(to_device_bf16(q), to_device_bf16(k), to_device_bf16(v), plan,
                             torch.from_numpy(doc).cuda(), pos=posd, ws=ws, allgather=allgather)
    torch.cuda.synchronize()
    cp.check(plan, ws)
    return o, lse


CASES = [
    # B, T, h, n_kv, d, n_cp, layout, causal
    (1, 2048, 4, 2, 128, 4, "zigzag", True),
    (2, 1024, 2, 2, 64, 4, "contiguous", True),
    (1, 2048, 4, 1, 128, 8, "striped", True),
    (1, 1024, 4, 4, 128, 2, "contiguous", False),
    (1, 1560, 2, 2, 128, 4, "zigzag", True),
    (1, 1536, 2, 2, 128, 3, "striped", False),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[6]}-T{c[1]}-d{c[4]}-{'causal' if c[7] else 'full'}" for c in CASES])
def test_document_pieces_match_oracle(case):
    B, T, h, n_kv, d, n_cp, layout, causal = case
    q, k, v = inputs(31 + T, B, T, h, n_kv, d)
    doc = pieces(T, T + n_cp, 5)
    plan = cp.Plan(T, h, n_kv, d, n_cp, layout, causal)
    o, lse = run_docs(q, k, v, plan, doc)
    ref_o, ref_lse = oracle.get().attention_docs(q, k, v, doc, causal=causal)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_lse, what=f"document pieces {case}")
    og, lg = run_docs(q, k, v, plan, doc, allgather=True)
    assert torch.equal(og.view(torch.int16), o.view(torch.int16)) and torch.equal(lg, lse), "all-gather differs"


def test_document_ids_with_permuted_positions():
    B, T, h, n_kv, d, n_cp = 1, 1024, 4, 2, 128, 4
    q, k, v = inputs(33, B, T, h, n_kv, d)
    doc = pieces(T, 4, 3)
    pos = np.random.default_rng(8).permutation(T).astype(np.int32)
    plan = cp.Plan(T, h, n_kv, d, n_cp, "zigzag", True)
    o, lse = run_docs(q, k, v, plan, doc, pos=pos)
    ref_o, ref_lse = oracle.get().attention_docs(q, k, v, doc, causal=True, pos=pos)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_lse, what="document ids, permuted positions")


def test_one_token_documents_return_their_own_values():
    B, T, h, n_kv, d, n_cp = 1, 512, 2, 2, 128, 4
    q, k, v = inputs(34, B, T, h, n_kv, d)
    doc = np.random.default_rng(1).permutation(T).astype(np.int32)     # every token its own document
    plan = cp.Plan(T, h, n_kv, d, n_cp, "striped", False)
    o, lse = run_docs(q, k, v, plan, doc)
    vb = synth.bf16_bits_to_f32(v)
    on = o.float().cpu().numpy()
    # O = P V / l with P = 1 and V in fp16: exact wherever V converts exactly (|v| >= 2^-14), within
    # the fp16 subnormal spacing below that
    exact = np.abs(vb) >= 2.0 ** -14
    assert np.array_equal(on[exact], vb[exact]), "a lone token must return its own value row"
    assert np.max(np.abs(on - vb)) <= 2.0 ** -24
    ref_o, ref_lse = oracle.get().attention_docs(q, k, v, doc, causal=False)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_lse, what="one-token documents")


@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "striped"])
def test_contiguous_documents_equal_the_lower_bound_form(layout):
    B, T, h, n_kv, d, n_cp = 1, 2048, 4, 2, 128, 4
    q, k, v = inputs(35, B, T, h, n_kv, d)
    rng = np.random.default_rng(2)
    lengths, left = [], T
    while left > 0:
        lengths.append(min(left, int(rng.integers(50, 600))))
        left -= lengths[-1]
    ids = rng.permutation(len(lengths)).astype(np.int32) * 3 + 1          # shuffled ids
    doc = np.repeat(ids, lengths).astype(np.int32)
    lo = np.repeat(np.concatenate([[0], np.cumsum(lengths)[:-1]]), lengths).astype(np.int32)
    plan = cp.Plan(T, h, n_kv, d, n_cp, layout, True)
    o, lse = run_docs(q, k, v, plan, doc)
    ol, ll = cp.forward_masked(to_device_bf16(q), to_device_bf16(k), to_device_bf16(v), plan,
                               torch.from_numpy(lo).cuda())
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), ol.view(torch.int16)) and torch.equal(lse, ll)


def test_gqa_16k_document_pieces_sampled_rows():
    w = synth.workload("gqa_zigzag_T16k")
    q, k, v = synth.make_qkv(w)
    doc = pieces(w.T, 16, 12, lo=256, hi=3000)
    plan = cp.Plan(w.T, w.h, w.n_kv, w.d, w.n_cp, w.layouts[0], True)
    o, lse = run_docs(q, k, v, plan, doc)
    rows = synth.sample_rows(w.T, w.n_cp, 256, seed=w.seed)
    idx = torch.from_numpy(rows).cuda()
    ref_o, ref_lse = oracle.get().attention_docs(q, k, v, doc, causal=True, rows=rows)
    compare(o.index_select(1, idx).float().cpu().numpy(), lse.index_select(2, idx).cpu().numpy(), ref_o, ref_lse,
            what="16K GQA document pieces")


def test_many_row_groups_are_ordered_by_their_masked_work():
    """2048 row groups (T = 262144 over 4 ranks): the device sort of the row groups by their masked
    tile counts handles two per thread; lower-bound and document-id forms against the oracle on
    sampled rows."""
    B, T, h, n_kv, d, n_cp = 1, 262144, 2, 1, 128, 4
    q, k, v = inputs(36, B, T, h, n_kv, d)
    doc = pieces(T, 37, 40, lo=2000, hi=20000)
    starts = np.concatenate([[0], np.flatnonzero(np.diff(doc)) + 1])
    lengths = np.diff(np.concatenate([starts, [T]]))
    lo = np.repeat(starts, lengths).astype(np.int32)
    plan = cp.Plan(T, h, n_kv, d, n_cp, "zigzag", True)
    rows = synth.sample_rows(T, n_cp, 96, seed=5)
    idx = torch.from_numpy(rows).cuda()
    # a run may continue the previous run's id: the lower bound follows runs, the ids follow documents
    run_id = np.cumsum(np.concatenate([[0], (np.diff(doc) != 0).astype(np.int64)])).astype(np.int32)
    ref_o, ref_lse = oracle.get().attention_docs(q, k, v, run_id, causal=True, rows=rows)
    ol, ll = cp.forward_masked(to_device_bf16(q), to_device_bf16(k), to_device_bf16(v), plan,
                               torch.from_numpy(lo).cuda())
    torch.cuda.synchronize()
    compare(ol.index_select(1, idx).float().cpu().numpy(), ll.index_select(2, idx).cpu().numpy(), ref_o, ref_lse,
            what="2048 row groups, lower bound")
    od, ld = run_docs(q, k, v, plan, doc)
    ref_o, ref_lse = oracle.get().attention_docs(q, k, v, doc, causal=True, rows=rows)
    compare(od.index_select(1, idx).float().cpu().numpy(), ld.index_select(2, idx).cpu().numpy(), ref_o, ref_lse,
            what="2048 row groups, document ids")
