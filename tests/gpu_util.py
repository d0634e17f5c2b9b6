"""Helpers for the GPU parity tests: seeded inputs from ``synth``, the library call through the
C ABI binding, and the comparison against the fp64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
import context_ring_attention_blockwise_gb300 as cp

O_TOL = 1e-2      # max-abs error on O (bf16 output from bf16 inputs, fp32 accumulation)
LSE_TOL = 1e-3    # max-abs error on lse (fp32)


def o_tolerance(ref_o: np.ndarray) -> np.ndarray:
    """Per-element bound on |O - O_exact|: 1e-2, except where |O_exact| >= 4. There the spacing
    of the bf16 grid (2^-5 in [4, 8)) is wider than twice 1e-2, so no bf16 value need lie within
    1e-2 of the exact one; such elements must instead be within one bf16 ulp of it."""
    a = np.abs(ref_o)
    ulp = np.exp2(np.floor(np.log2(np.maximum(a, 1e-30))) - 7)
    return np.where(a >= 4.0, ulp, O_TOL)


def to_device_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def inputs(seed, B, T, h, n_kv, d, k_mult=1.0, q_zero=False):
    q = synth.normal_bf16(seed, synth.TAG_Q, (B, T, h, d))
    if q_zero:
        q = np.zeros_like(q)
    k = synth.normal_bf16(seed, synth.TAG_K, (B, T, n_kv, d), mult=k_mult)
    v = synth.normal_bf16(seed, synth.TAG_V, (B, T, n_kv, d))
    return q, k, v


def run(q, k, v, n_cp, layout, causal=True, pos=None, scale=None, path="fused"):
    """Returns (o fp32 numpy [B,T,h,d], lse numpy [B,h,T], plan, ws)."""
    B, T, h, d = q.shape
    plan = cp.Plan(T, h, k.shape[2], d, n_cp, layout, causal)
    qd, kd, vd = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    posd = torch.from_numpy(np.ascontiguousarray(pos, dtype=np.int32)).cuda() if pos is not None else None
    if path == "fused":
        ws = cp.alloc_workspace(plan.workspace_size(B))
        o, lse = cp.forward(qd, kd, vd, plan, pos=posd, scale=scale, ws=ws)
    else:
        ws = cp.alloc_workspace(plan.ring_workspace_size(B))
        o, lse = cp.ring_forward(qd, kd, vd, plan, pos=posd, scale=scale, ws=ws)
    torch.cuda.synchronize()
    cp.check(plan, ws)
    return o.float().cpu().numpy(), lse.cpu().numpy(), plan, ws


def compare(o, lse, ref_o, ref_lse, rows=None, what=""):
    """Max-abs errors against the oracle; rows selects natural token ids of o/lse."""
    if rows is not None:
        o = o[:, rows]
        lse = lse[:, :, rows]
    assert o.shape == ref_o.shape and lse.shape == ref_lse.shape
    assert np.all(np.isfinite(o)), f"{what}: non-finite O"
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin), f"{what}: -inf pattern of lse differs"
    err = np.abs(o - ref_o)
    eo = float(np.max(err)) if o.size else 0.0
    el = float(np.max(np.abs(lse[fin] - ref_lse[fin]))) if fin.any() else 0.0
    over = err > o_tolerance(ref_o)
    if over.any() or el > LSE_TOL:
        idx = np.unravel_index(int(np.argmax(err - o_tolerance(ref_o))), err.shape)
        le = np.where(fin, np.abs(np.where(fin, lse, 0) - np.where(fin, ref_lse, 0)), 0)
        li = np.unravel_index(int(np.argmax(le)), le.shape)
        what += f" [worst lse at (b, head, row) {li}: got {lse[li]:.6f}, exact {ref_lse[li]:.6f}]"
        raise AssertionError(f"{what}: max|dO| = {eo:.3e} ({int(over.sum())} elements over tolerance; worst at "
                             f"{idx}: got {o[idx]:.6f}, exact {ref_o[idx]:.6f}), max|dlse| = {el:.3e} (tol {LSE_TOL})")
    return eo, el
