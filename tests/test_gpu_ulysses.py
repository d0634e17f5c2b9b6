"""The head split (cpattn_ulysses_forward, "Ulysses, splitting by heads instead") on the GPU: the
all-to-all, every rank's exact attention over all tokens of its heads, the all-to-all back.
Against the oracle's attention definition (the oracle's literal Ulysses run is pinned equal to
it), and bit-identical to the plain one-rank forward, since the split changes no arithmetic of a
head."""
import numpy as np
import pytest
import torch

import oracle
import synth
import context_ring_attention_blockwise_gb300 as cp
from synth.configs import CONTIGUOUS
from tests.gpu_util import compare, to_device_bf16, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from context_ring_attention_blockwise_gb300 import _build
    _build.build()


def _ulysses(q, k, v, n_cp, causal=True, pos=None, scale=None):
    B, T, h, d = q.shape
    plan = cp.UlyssesPlan(T, h, k.shape[2], d, n_cp, causal)
    qd, kd, vd = (to_device_bf16(x) for x in (q, k, v))
    posd = torch.from_numpy(np.ascontiguousarray(pos, dtype=np.int32)).cuda() if pos is not None else None
    ws = cp.alloc_workspace(plan.workspace_size(B))
    o, lse = cp.ulysses_forward(qd, kd, vd, plan, pos=posd, scale=scale, ws=ws)
    torch.cuda.synchronize()
    cp.check(plan, ws)
    return o.float().cpu().numpy(), lse.cpu().numpy()


CASES = [
    # B, T, h, n_kv, d, n_cp, causal
    (1, 1024, 8, 8, 128, 4, True),      # two KV heads per rank
    (1, 1024, 8, 2, 64, 8, True),       # KV heads replicated on 4 ranks each
    (2, 512, 4, 1, 128, 4, False),      # one KV head for all, non-causal, two sequences
    (1, 1040, 8, 4, 128, 4, True),      # ragged: 1040 tokens, 260 per rank
    (1, 768, 16, 8, 64, 16, True),      # one query head per rank
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}_T{c[1]}_h{c[2]}_kv{c[3]}_d{c[4]}_cp{c[5]}_"
                                             f"{'causal' if c[6] else 'full'}" for c in CASES])
def test_ulysses_matches_oracle(case):
    B, T, h, n_kv, d, n_cp, causal = case
    q, k, v = inputs(90 + T + h + n_cp, B, T, h, n_kv, d)
    o, lse = _ulysses(q, k, v, n_cp, causal)
    ref_o, ref_lse = oracle.get().attention(q, k, v, causal=causal)
    compare(o, lse, ref_o, ref_lse, what=f"ulysses {case}")


def test_ulysses_positions_and_scale():
    q, k, v = inputs(93, 1, 512, 8, 2, 128)
    pos = np.sort(np.random.default_rng(3).integers(0, 2048, size=512)).astype(np.int32)
    o, lse = _ulysses(q, k, v, 4, True, pos=pos, scale=0.05)
    ref_o, ref_lse = oracle.get().attention(q, k, v, causal=True, pos=pos, scale=0.05)
    compare(o, lse, ref_o, ref_lse, what="ulysses positions")


@pytest.mark.parametrize("n_cp", [2, 8])
def test_ulysses_is_the_one_rank_forward(n_cp):
    """Bit-identical to cpattn_forward with one rank: each head's tiles run in the same order."""
    q, k, v = inputs(94, 1, 1024, 16, 4, 128)
    o, lse = _ulysses(q, k, v, n_cp, True)
    plan = cp.Plan(1024, 16, 4, 128, 1, CONTIGUOUS, True)
    o1, lse1 = cp.forward(*(to_device_bf16(x) for x in (q, k, v)), plan)
    assert np.array_equal(o, o1.float().cpu().numpy()) and np.array_equal(lse, lse1.cpu().numpy())


def test_ulysses_gqa_16k_sampled():
    """The GQA 4:1 T=16384 shape split over 8 ranks (one KV head each): sampled rows."""
    w = synth.workload("gqa_zigzag_T16k")
    q, k, v = synth.make_qkv(w)
    o, lse = _ulysses(q, k, v, w.n_cp, w.causal)
    rows = synth.sample_rows(w.T, w.n_cp, 128, seed=w.seed)
    ref_o, ref_lse = oracle.get().attention(q, k, v, causal=w.causal, rows=rows)
    compare(o, lse, ref_o, ref_lse, rows=rows, what="16K ulysses")
