"""The allocation-free forward, checked against the ordinary one.

Callers that cannot allocate device memory -- a host callback, an allocator hook, a plug-in that
must leave the process's memory pools alone -- cannot hand cpattn_forward a workspace.
cpattn_forward_noalloc serves them with the library's built-in 64 MiB device scratch. These tests
call it through the C ABI twice in a row on different inputs and compare each result with
cpattn_forward's on the same inputs, within the tolerances the parity tests use, and check that a
device-side timeout recorded in the built-in scratch reaches the caller through cpattn_check_noalloc.
The file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import context_ring_attention_blockwise_gb300 as cp
from tests.gpu_util import LSE_TOL, O_TOL, inputs, to_device_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from context_ring_attention_blockwise_gb300 import _build
    _build.build()


def test_noalloc_matches_forward_on_two_calls_in_a_row():
    T, h, n_kv, d, n_cp = 2048, 8, 2, 128, 4
    plan = cp.Plan(T, h, n_kv, d, n_cp, "zigzag", True)
    assert plan.workspace_size(1) < 64 << 20
    for seed in (901, 902):                      # the second call must not see the first call's state
        q, k, v = (to_device_bf16(x) for x in inputs(seed, 1, T, h, n_kv, d))
        o_na, l_na = cp.forward_noalloc(q, k, v, plan)
        o_ref, l_ref = cp.forward(q, k, v, plan)
        torch.cuda.synchronize()
        cp.check_noalloc(plan)
        do = (o_na.float() - o_ref.float()).abs().max().item()
        dl = (l_na - l_ref).abs().max().item()
        assert do <= O_TOL and dl <= LSE_TOL, f"seed {seed}: max|dO| = {do:.3e}, max|dlse| = {dl:.3e}"
        assert torch.isfinite(o_na.float()).all()


def test_noalloc_rejects_problems_beyond_its_scratch():
    plan = cp.Plan(131072, 64, 8, 128, 16, "zigzag", True)
    assert plan.workspace_size(1) > 64 << 20
    q = torch.empty((1, 131072, 64, 128), dtype=torch.bfloat16, device="cuda")
    kv = torch.empty((1, 131072, 8, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cp.CpattnError) as e:
        cp.forward_noalloc(q, kv, kv, plan)
    assert e.value.status == 3 and "64 MiB" in str(e.value)


def test_noalloc_reports_a_device_timeout_and_recovers():
    T, h, n_kv, d, n_cp = 1024, 4, 2, 128, 2
    plan = cp.Plan(T, h, n_kv, d, n_cp, "contiguous", True)
    q, k, v = (to_device_bf16(x) for x in inputs(903, 1, T, h, n_kv, d))
    cp.forward_noalloc(q, k, v, plan)
    torch.cuda.synchronize()
    cp.check_noalloc(plan)
    # a wait that nothing completes, run out after 50 ms, recorded in the built-in scratch
    cp.selftest_wait_timeout_noalloc(50_000_000)
    torch.cuda.synchronize()
    with pytest.raises(cp.CpattnError) as e:
        cp.check_noalloc(plan)
    assert e.value.status == 5 and "timed out" in str(e.value)
    # the next call clears the record and computes the same result as the ordinary forward
    o_na, l_na = cp.forward_noalloc(q, k, v, plan)
    o_ref, l_ref = cp.forward(q, k, v, plan)
    torch.cuda.synchronize()
    cp.check_noalloc(plan)
    do = (o_na.float() - o_ref.float()).abs().max().item()
    dl = (l_na - l_ref).abs().max().item()
    assert do <= O_TOL and dl <= LSE_TOL, f"after the timeout: max|dO| = {do:.3e}, max|dlse| = {dl:.3e}"
