"""The five benchmark workloads at full size on the GPU, in the launch configuration the bench
times, against the fp64 oracle (all heads, every batch element): every row of the tiny and the
16K GQA workloads, 4096 rows of the 32K non-causal one (every chunk boundary among them), and 256
rows of the two 128K ones; and the kernel's block-skip decisions bit-exact against the plan."""
import numpy as np
import pytest
import torch

import oracle
import synth
import context_ring_attention_blockwise_gb300 as cp
from tests.gpu_util import compare, to_device_bf16

pytestmark = pytest.mark.gpu

WORKLOADS = [(name, layout) for name in synth.ORDER for layout in synth.workload(name).layouts]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from context_ring_attention_blockwise_gb300 import _build
    _build.build()


@pytest.mark.parametrize("name,layout", WORKLOADS, ids=[f"{n}-{synth.LAYOUT_NAMES[l]}" for n, l in WORKLOADS])
def test_workload_sampled_rows(name, layout):
    w = synth.workload(name)
    q, k, v = synth.make_qkv(w)
    plan = cp.Plan(w.T, w.h, w.n_kv, w.d, w.n_cp, layout, w.causal)
    ws = cp.alloc_workspace(plan.workspace_size(w.B))
    qd, kd, vd = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    o, lse = cp.forward(qd, kd, vd, plan, ws=ws)
    torch.cuda.synchronize()
    cp.check(plan, ws)
    full, diag = cp.tile_counts(plan, w.B, ws)
    pc = plan.counts(w.B)
    assert np.array_equal(full, w.B * w.h * pc["full"]) and np.array_equal(diag, w.B * w.h * pc["diag"])
    if w.sampled_rows:
        rows = synth.sample_rows(w.T, w.n_cp, w.sampled_rows, seed=w.seed)
        idx = torch.from_numpy(rows).cuda()
        o_s = o.index_select(1, idx).float().cpu().numpy()
        lse_s = lse.index_select(2, idx).cpu().numpy()
        ref_o, ref_lse = oracle.get().attention(q, k, v, causal=w.causal, rows=rows)
        compare(o_s, lse_s, ref_o, ref_lse, what=f"{name} sampled rows")
    else:
        ref_o, ref_lse = oracle.get().attention(q, k, v, causal=w.causal)
        compare(o.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_lse, what=name)
    # edge rows the sample always holds: the first token sees one key, the last sees all
    assert np.all(np.isfinite(lse.cpu().numpy()))


@pytest.mark.parametrize("name", ["gqa_zigzag_T16k", "llama405b_tp_T128k"])
def test_workload_ring_step_path(name):
    w = synth.workload(name)
    layout = w.layouts[-1]
    q, k, v = synth.make_qkv(w)
    plan = cp.Plan(w.T, w.h, w.n_kv, w.d, w.n_cp, layout, w.causal)
    ws = cp.alloc_workspace(plan.ring_workspace_size(w.B))
    qd, kd, vd = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    o, lse = cp.ring_forward(qd, kd, vd, plan, ws=ws)
    torch.cuda.synchronize()
    cp.check(plan, ws)
    rows = synth.sample_rows(w.T, w.n_cp, 128, seed=w.seed + 1)
    idx = torch.from_numpy(rows).cuda()
    ref_o, ref_lse = oracle.get().attention(q, k, v, causal=w.causal, rows=rows)
    compare(o.index_select(1, idx).float().cpu().numpy(), lse.index_select(2, idx).cpu().numpy(), ref_o, ref_lse,
            what=f"{name} ring-step path")
