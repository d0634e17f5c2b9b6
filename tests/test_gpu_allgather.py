"""The all-gather variant on the GPU ("Splitting the sequence, and the one layer that objects":
gather the keys and values so that every rank holds the full K and V, then compute attention for
the local queries; "What context parallelism communicates": the gather is exposed and any mask
works with one ordinary attention kernel): every virtual rank reads only its own gathered copy.
Checked against the oracle, bit-identical to cpattn_forward (same arithmetic in the same order),
and with document masks against the oracle's document-id definition, including documents whose ids
do not increase along the packed sequence."""
import numpy as np
import pytest
import torch

import oracle
import context_ring_attention_blockwise_gb300 as cp
from tests.gpu_util import compare, inputs, to_device_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from context_ring_attention_blockwise_gb300 import _build
    _build.build()


CASES = [
    (1, 2048, 4, 2, 128, 4, "zigzag", True),
    (2, 1024, 2, 2, 64, 4, "contiguous", True),
    (1, 2048, 4, 1, 128, 8, "striped", True),
    (1, 1024, 4, 4, 128, 2, "contiguous", False),
    (1, 1560, 2, 2, 128, 4, "zigzag", True),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[6]}-T{c[1]}-d{c[4]}-ncp{c[5]}" for c in CASES])
def test_allgather_matches_oracle_and_the_ring(case):
    B, T, h, n_kv, d, n_cp, layout, causal = case
    q, k, v = inputs(55 + T, B, T, h, n_kv, d)
    plan = cp.Plan(T, h, n_kv, d, n_cp, layout, causal)
    qd, kd, vd = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    ws = cp.alloc_workspace(plan.allgather_workspace_size(B))
    o, lse = cp.allgather_forward(qd, kd, vd, plan, ws=ws)
    of, lf = cp.forward(qd, kd, vd, plan)
    torch.cuda.synchronize()
    cp.check(plan, ws)
    ref_o, ref_lse = oracle.get().attention(q, k, v, causal=causal)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_lse, what=f"all-gather {case}")
    assert torch.equal(o.view(torch.int16), of.view(torch.int16)) and torch.equal(lse, lf)
    # the two phases alone, after a placement, give the same result
    o2, l2 = torch.empty_like(o), torch.empty_like(lse)
    cp.permute(qd, kd, vd, plan, ws)
    cp.allgather_gather(plan, B, ws)
    cp.allgather_attend(plan, B, ws, o2, l2)
    torch.cuda.synchronize()
    assert torch.equal(o2.view(torch.int16), o.view(torch.int16)) and torch.equal(l2, lse)


def test_allgather_gathered_copies_are_each_ranks_own():
    # a rank's gathered copy is the whole K and V: overwriting rank 1's copy of V with 2.0 must
    # change rank 1's rows alone, so every rank reads its own copy
    B, T, h, n_kv, d, n_cp = 1, 1024, 2, 2, 128, 4
    q, k, v = inputs(61, B, T, h, n_kv, d)
    plan = cp.Plan(T, h, n_kv, d, n_cp, "contiguous", True)
    qd, kd, vd = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    ws = cp.alloc_workspace(plan.allgather_workspace_size(B))
    o, lse = torch.empty_like(qd), torch.empty((B, h, T), dtype=torch.float32, device="cuda")
    cp.permute(qd, kd, vd, plan, ws)
    cp.allgather_gather(plan, B, ws)
    fwd = plan.workspace_size(B)
    per_rank = 2 * B * T * n_kv * d
    gv = fwd + n_cp * per_rank                           # the gathered K, then V, follow the forward regions
    ws[gv + per_rank:gv + 2 * per_rank].view(torch.int16).fill_(0x4000)   # rank 1's copy of V: bf16 2.0
    cp.allgather_attend(plan, B, ws, o, lse)
    torch.cuda.synchronize()
    ref_o, ref_lse = oracle.get().attention(q, k, v, causal=True)
    n = T // n_cp
    on, ln = o.float().cpu().numpy(), lse.cpu().numpy()
    for r in (0, 2, 3):
        rows = np.arange(r * n, (r + 1) * n)
        compare(on[:, rows], ln[:, :, rows], ref_o[:, rows], ref_lse[:, :, rows], what=f"rank {r}")
    assert np.all(on[:, n:2 * n] == 2.0), "rank 1 did not read its own (overwritten) copy"


def _docs(T, seed, shuffled):
    rng = np.random.default_rng(seed)
    lengths = []
    while sum(lengths) < T:
        lengths.append(int(rng.integers(64, 700)))
    lengths[-1] -= sum(lengths) - T
    lengths = [x for x in lengths if x > 0]
    ids = np.arange(len(lengths))
    if shuffled:
        ids = rng.permutation(len(lengths)) * 7 + 3      # ids that do not increase along the sequence
    doc = np.repeat(ids, lengths).astype(np.int32)
    starts = np.concatenate([[0], np.cumsum(lengths)[:-1]])
    lo = np.repeat(starts, lengths).astype(np.int32)
    return doc, lo


@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "striped"])
@pytest.mark.parametrize("shuffled", [False, True], ids=["ordered-ids", "shuffled-ids"])
def test_allgather_document_masks(layout, shuffled):
    B, T, h, n_kv, d, n_cp = 1, 2048, 4, 2, 128, 4
    q, k, v = inputs(63, B, T, h, n_kv, d)
    doc, lo = _docs(T, 9, shuffled)
    plan = cp.Plan(T, h, n_kv, d, n_cp, layout, True)
    qd, kd, vd = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    lod = torch.from_numpy(lo).cuda()
    ws = cp.alloc_workspace(plan.allgather_workspace_size(B))
    o, lse = cp.allgather_forward(qd, kd, vd, plan, lo=lod, ws=ws)
    om, lm = cp.forward_masked(qd, kd, vd, plan, lod)
    torch.cuda.synchronize()
    cp.check(plan, ws)
    ref_o, ref_lse = oracle.get().attention_docs(q, k, v, doc, causal=True)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_lse, what=f"all-gather documents {layout}")
    assert torch.equal(o.view(torch.int16), om.view(torch.int16)) and torch.equal(lse, lm)
