"""GPU parity of the backward pass (cpattn_backward) against the fp64 oracle's gradients.

The forward outputs o (bf16) and lse (fp32) the backward consumes come from the library's own
forward on the same inputs, as a caller would pass them.

Tolerance, from the arithmetic. Every gradient element is a sum of terms (P dO for dV,
scale dS q for dK, scale dS k for dQ). The kernels round P and dS to bf16 for the tensor cores,
read bf16 operands, take D = <dO, O> from the bf16 forward output, and round the result to bf16:
up to four relative errors of 2^-9 meet in one term, so a term is off by at most ~2^-7 of its
size. The terms carry both signs and cancel, so the reference scale is the largest gradient
magnitude of the tensor (b, head slice): |got - exact| <= 2^-6 * max|exact| + 2^-8 * |exact|.
When the cancellation is total the exact gradient is 0 (one visible key: dS = P (dP - D) with
D = dP) and what remains is the fp32 rounding difference between the tensor core's dP and the
prep kernel's D (~1e-7 here): the bound has an absolute floor of 2^-16 for that case.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import context_ring_attention_blockwise_gb300 as cp
from synth.configs import CONTIGUOUS, ZIGZAG, STRIPED
from tests.gpu_util import to_device_bf16

pytestmark = pytest.mark.gpu

ATOL_FRAC = 2.0 ** -6
RTOL = 2.0 ** -8
FLOOR = 2.0 ** -16


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from context_ring_attention_blockwise_gb300 import _build
    _build.build()


def _inputs(seed, B, T, h, n_kv, d):
    q = synth.normal_bf16(seed, synth.TAG_Q, (B, T, h, d))
    k = synth.normal_bf16(seed, synth.TAG_K, (B, T, n_kv, d))
    v = synth.normal_bf16(seed, synth.TAG_V, (B, T, n_kv, d))
    do = synth.normal_bf16(seed, 4, (B, T, h, d))
    return q, k, v, do


def _run(q, k, v, do, n_cp, layout, causal, pos=None, scale=None):
    B, T, h, d = q.shape
    plan = cp.Plan(T, h, k.shape[2], d, n_cp, layout, causal)
    qd, kd, vd, dod = (to_device_bf16(x) for x in (q, k, v, do))
    posd = torch.from_numpy(np.ascontiguousarray(pos, dtype=np.int32)).cuda() if pos is not None else None
    o, lse = cp.forward(qd, kd, vd, plan, pos=posd, scale=scale)
    ws = cp.alloc_workspace(plan.backward_workspace_size(B))
    dq, dk, dv = cp.backward(qd, kd, vd, o, lse, dod, plan, pos=posd, scale=scale, ws=ws)
    torch.cuda.synchronize()
    cp.check(plan, ws)
    return tuple(x.float().cpu().numpy() for x in (dq, dk, dv))


def _compare(got, exact, what):
    """Per (b, head) slice: |got - exact| <= ATOL_FRAC * max|exact| + RTOL * |exact| + FLOOR."""
    assert got.shape == exact.shape
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    B, T, H, d = exact.shape
    worst = 0.0
    for b in range(B):
        for hh in range(H):
            e = exact[b, :, hh]
            g = got[b, :, hh]
            scale = float(np.max(np.abs(e))) if e.size else 0.0
            err = np.abs(g - e)
            bound = ATOL_FRAC * scale + RTOL * np.abs(e) + FLOOR
            ratio = float(np.max(err / np.maximum(bound, 1e-30))) if e.size else 0.0
            worst = max(worst, ratio)
            if ratio > 1.0:
                idx = np.unravel_index(int(np.argmax(err - bound)), err.shape)
                raise AssertionError(f"{what}: b={b} head={hh} worst at {idx}: got {g[idx]:.6f}, exact {e[idx]:.6f} "
                                     f"(max|exact| {scale:.4f}, max|err| {float(err.max()):.3e})")
    return worst


CASES = [
    # T, h, n_kv, d, n_cp, layout, causal
    (512, 2, 2, 64, 4, CONTIGUOUS, True),
    (512, 4, 2, 128, 4, ZIGZAG, True),
    (768, 4, 1, 128, 4, STRIPED, True),
    (512, 2, 2, 128, 2, CONTIGUOUS, False),
    (600, 2, 1, 64, 2, CONTIGUOUS, True),        # ragged: 300 tokens per rank
    (1040, 4, 2, 128, 4, ZIGZAG, True),          # ragged: 260 tokens per rank
]


@pytest.mark.parametrize("case", CASES, ids=[f"T{c[0]}_h{c[1]}_kv{c[2]}_d{c[3]}_cp{c[4]}_{synth.LAYOUT_NAMES[c[5]]}_"
                                             f"{'causal' if c[6] else 'full'}" for c in CASES])
def test_backward_matches_oracle(case):
    T, h, n_kv, d, n_cp, layout, causal = case
    q, k, v, do = _inputs(21 + T + h, 1, T, h, n_kv, d)
    dq, dk, dv = _run(q, k, v, do, n_cp, layout, causal)
    rq, rk, rv = oracle.get().backward(q, k, v, do, causal=causal)
    _compare(dq, rq, "dq")
    _compare(dk, rk, "dk")
    _compare(dv, rv, "dv")


def test_backward_positions_scale_batch():
    B, T, h, n_kv, d = 2, 512, 4, 2, 64
    q, k, v, do = _inputs(77, B, T, h, n_kv, d)
    rng = np.random.default_rng(5)
    pos = np.sort(rng.integers(0, 3 * T, size=T)).astype(np.int32)     # ties: equal positions see each other
    dq, dk, dv = _run(q, k, v, do, 4, ZIGZAG, True, pos=pos, scale=0.07)
    rq, rk, rv = oracle.get().backward(q, k, v, do, causal=True, pos=pos, scale=0.07)
    _compare(dq, rq, "dq")
    _compare(dk, rk, "dk")
    _compare(dv, rv, "dv")


def test_backward_is_deterministic():
    q, k, v, do = _inputs(78, 1, 512, 2, 1, 128)
    a = _run(q, k, v, do, 4, ZIGZAG, True)
    b = _run(q, k, v, do, 4, ZIGZAG, True)
    for x, y in zip(a, b):
        assert np.array_equal(x, y), "the backward has no atomics: repeated runs are bit-identical"


def test_backward_workload_sampled():
    """The GQA 4:1 zigzag T=16384 workload at full size, in the launch configuration the bench
    times: dq of sampled rows, dk/dv of the last 64 keys (few queries see them, so the oracle
    stays cheap)."""
    w = synth.workload("gqa_zigzag_T16k")
    q, k, v = synth.make_qkv(w)
    do = synth.normal_bf16(w.seed, 4, (w.B, w.T, w.h, w.d))
    dq, dk, dv = _run(q, k, v, do, w.n_cp, w.layouts[0], w.causal)
    rows = synth.sample_rows(w.T, w.n_cp, 48, seed=w.seed)
    keys = np.arange(w.T - 64, w.T)
    rq, rk, rv = oracle.get().backward(q, k, v, do, causal=w.causal, rows=rows, keys=keys)
    _compare(dq[:, rows], rq, "dq (sampled rows)")
    _compare(dk[:, keys], rk, "dk (last keys)")
    _compare(dv[:, keys], rv, "dv (last keys)")


def test_backward_70b_128k_sampled():
    """The 70B-shaped zigzag T=131072 workload the bench's backward extra times (GQA 8:1, 16
    ranks): dq of sampled rows, dk/dv of the last 64 keys."""
    w = synth.workload("llama70b_zigzag_T128k")
    q, k, v = synth.make_qkv(w)
    do = synth.normal_bf16(w.seed, 4, (w.B, w.T, w.h, w.d))
    dq, dk, dv = _run(q, k, v, do, w.n_cp, w.layouts[0], w.causal)
    rows = synth.sample_rows(w.T, w.n_cp, 24, seed=w.seed)
    keys = np.arange(w.T - 64, w.T)
    rq, rk, rv = oracle.get().backward(q, k, v, do, causal=w.causal, rows=rows, keys=keys)
    _compare(dq[:, rows], rq, "dq (sampled rows)")
    _compare(dk[:, keys], rk, "dk (last keys)")
    _compare(dv[:, keys], rv, "dv (last keys)")
