"""GPU parity through the C ABI: the sm_103a path against the fp64 oracle, element by element,
on seeded inputs that span several tiles and ragged tails, every layout, causal and not, GQA,
both head widths, custom position ids, and the ring-step path against the fused path."""
import numpy as np
import pytest
import torch

import oracle
import synth
import context_ring_attention_blockwise_gb300 as cp
from tests.gpu_util import compare, inputs, run, to_device_bf16

pytestmark = pytest.mark.gpu

CASES = [
    # (T, h, n_kv, d, n_cp, B)
    (512, 2, 2, 64, 4, 1),       # the tiny MHA workload's shape
    (800, 4, 2, 128, 4, 1),      # 200 tokens per rank: a full tile and a ragged one
    (768, 4, 1, 64, 3, 1),       # GQA 4:1, three ranks
    (1024, 2, 2, 128, 2, 2),     # batch of 2
    (384, 3, 1, 128, 1, 1),      # one rank: plain attention
    (1040, 2, 1, 128, 8, 1),     # 130 tokens per rank: 128 + a 2-token tail
]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from context_ring_attention_blockwise_gb300 import _build
    _build.build()


@pytest.mark.parametrize("case", CASES, ids=lambda c: "T{}_h{}_kv{}_d{}_cp{}_B{}".format(*c))
@pytest.mark.parametrize("layout", [0, 1, 2], ids=["contiguous", "zigzag", "striped"])
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
def test_forward_matches_oracle(case, layout, causal):
    T, h, n_kv, d, n_cp, B = case
    if layout == 1 and T % (2 * n_cp):
        pytest.skip("zigzag needs T % 2n_cp")
    q, k, v = inputs(100 + T + d, B, T, h, n_kv, d, k_mult=1.0 if causal else 2.0)
    ref_o, ref_lse = oracle.get().attention(q, k, v, causal=causal)
    o, lse, plan, ws = run(q, k, v, n_cp, layout, causal)
    compare(o, lse, ref_o, ref_lse, what=f"fused {case} layout {layout} causal {causal}")


@pytest.mark.parametrize("layout", [0, 1, 2], ids=["contiguous", "zigzag", "striped"])
@pytest.mark.parametrize("path", ["fused", "ring"])
def test_uniform_scores_give_mean_of_values(layout, path):
    """Q = 0: every visible key has the same score, so O is the running mean of V (closed form);
    on the ring-step path every step after the first adds at the running maximum's own scale."""
    T, h, d, n_cp = 512, 2, 128, 4
    q, k, v = inputs(7, 1, T, h, h, d, q_zero=True)
    o, lse, _, _ = run(q, k, v, n_cp, layout, True, path=path)
    vf = synth.bf16_bits_to_f32(v).astype(np.float64)
    mean = np.cumsum(vf, axis=1) / np.arange(1, T + 1)[None, :, None, None]
    assert np.max(np.abs(o - mean)) < 1e-2
    assert np.max(np.abs(lse[0] - np.log(np.arange(1, T + 1))[None, :])) < 1e-3


def test_tiny_workload_exact_config():
    w = synth.workload("tiny_mha_contig_T512")
    q, k, v = synth.make_qkv(w)
    ref_o, ref_lse = oracle.get().attention(q, k, v, causal=True)
    for path in ("fused", "ring"):
        o, lse, plan, ws = run(q, k, v, w.n_cp, w.layouts[0], True, path=path)
        compare(o, lse, ref_o, ref_lse, what=f"tiny workload, {path} path")


@pytest.mark.parametrize("layout", [0, 1, 2], ids=["contiguous", "zigzag", "striped"])
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
def test_ring_step_path_matches_oracle_and_fused(layout, causal):
    T, h, n_kv, d, n_cp = 1024, 4, 2, 128, 4
    q, k, v = inputs(55, 1, T, h, n_kv, d, k_mult=2.0)
    ref_o, ref_lse = oracle.get().attention(q, k, v, causal=causal)
    of, lf, _, _ = run(q, k, v, n_cp, layout, causal, path="fused")
    orr, lr, _, _ = run(q, k, v, n_cp, layout, causal, path="ring")
    compare(orr, lr, ref_o, ref_lse, what="ring-step path")
    compare(of, lf, ref_o, ref_lse, what="fused path")
    assert np.max(np.abs(orr - of)) <= 2 * 2 ** -8 * max(1.0, float(np.max(np.abs(of))))


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
def test_ring_step_running_maximum_jumps(causal):
    """The ring-step merge keeps each row's output unnormalised against a running maximum and adds
    a step's output by reductions while the step's maximum stays within 2^8 of it; a larger jump
    takes the rescale path (the running row read back and scaled down). Rank 3's keys are scaled
    by 8, so every query meeting that block after its own step sees its scores jump by far more
    than 8 (log2 units): contiguous ranks 0..2 meet it at steps 1..3, after their own blocks. (For
    the causal case the positions are reversed, so that block holds the earliest positions and
    every query sees it.) Both paths against the oracle and against the fused forward."""
    T, h, n_kv, d, n_cp = 1024, 4, 2, 128, 4
    q, k, v = inputs(57, 1, T, h, n_kv, d)
    k8 = synth.normal_bf16(57, synth.TAG_K, (1, T, n_kv, d), mult=8.0)
    n = T // n_cp
    k[:, 3 * n:] = k8[:, 3 * n:]
    if causal:   # make the late block visible to earlier ranks: reverse the positions
        pos = np.arange(T)[::-1].astype(np.int32).copy()
    else:
        pos = None
    ref_o, ref_lse = oracle.get().attention(q, k, v, causal=causal, pos=pos)
    of, lf, _, _ = run(q, k, v, n_cp, 0, causal, pos=pos, path="fused")
    orr, lr, _, _ = run(q, k, v, n_cp, 0, causal, pos=pos, path="ring")
    compare(orr, lr, ref_o, ref_lse, what="ring-step path, running maximum jumps")
    compare(of, lf, ref_o, ref_lse, what="fused path, large keys")
    assert np.max(np.abs(orr - of)) <= 2 * 2 ** -8 * max(1.0, float(np.max(np.abs(of))))


@pytest.mark.parametrize("case", [(1024, 4, 2, 128, 4, 1, True, 1), (1560, 2, 2, 128, 4, 2, True, 1),
                                  (768, 4, 1, 64, 3, 0, False, 1), (1024, 2, 2, 64, 4, 1, True, 2),
                                  (512, 2, 1, 128, 2, 1, True, 1)],
                         ids=["zigzag", "striped-ragged", "contiguous-full", "zigzag-B2", "two-ranks"])
def test_ring_step_hop_in_kernel_equals_copy_stream(case):
    """The hop done by the step kernels' idle warps delivers the same blocks as the copy-stream
    hop: the two passes are bit-identical, and both match the oracle."""
    T, h, n_kv, d, n_cp, layout, causal, B = case
    q, k, v = inputs(61 + T, B, T, h, n_kv, d)
    plan = cp.Plan(T, h, n_kv, d, n_cp, layout, causal)
    qd, kd, vd = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    ws = cp.alloc_workspace(plan.ring_workspace_size(B))
    ok, lk = cp.ring_forward(qd, kd, vd, plan, ws=ws)                       # hops in the kernels
    torch.cuda.synchronize()
    cp.check(plan, ws)
    oc, lc = cp.ring_forward(qd, kd, vd, plan, ws=ws, copy_stream=torch.cuda.Stream())
    torch.cuda.synchronize()
    cp.check(plan, ws)
    assert torch.equal(ok.view(torch.int16), oc.view(torch.int16)) and torch.equal(lk, lc)
    ref_o, ref_lse = oracle.get().attention(q, k, v, causal=causal)
    compare(ok.float().cpu().numpy(), lk.cpu().numpy(), ref_o, ref_lse, what=f"in-kernel hops {case}")


def test_ring_step_hop_in_kernel_with_reserved_sms():
    """With SMs left free the step kernels have fewer CTAs, each moving a larger share of the
    blocks: the same results, bit for bit."""
    T, h, n_kv, d, n_cp = 2048, 4, 2, 128, 8
    q, k, v = inputs(67, 1, T, h, n_kv, d)
    plan = cp.Plan(T, h, n_kv, d, n_cp, 1, True)
    qd, kd, vd = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    ws = cp.alloc_workspace(plan.ring_workspace_size(1))
    o0, l0 = cp.ring_forward(qd, kd, vd, plan, ws=ws)
    torch.cuda.synchronize()
    plan.set_reserved_sms(148)              # a handful of CTAs copy every block
    o1, l1 = cp.ring_forward(qd, kd, vd, plan, ws=ws)
    torch.cuda.synchronize()
    plan.set_reserved_sms(0)
    cp.check(plan, ws)
    assert torch.equal(o0.view(torch.int16), o1.view(torch.int16)) and torch.equal(l0, l1)


def test_ring_pass_keeps_one_kind_of_hop():
    """A pass that starts with in-kernel hops refuses a copy stream at a later step (and the
    reverse), before any launch; a new permute starts a new pass."""
    T, h, n_kv, d, n_cp = 512, 2, 1, 64, 4
    q, k, v = inputs(63, 1, T, h, n_kv, d)
    plan = cp.Plan(T, h, n_kv, d, n_cp, 1, True)
    qd, kd, vd = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    ws = cp.alloc_workspace(plan.ring_workspace_size(1))
    copy = torch.cuda.Stream()
    for first, second in ((None, copy), (copy, None)):
        cp.permute(qd, kd, vd, plan, ws)
        cp.ring_step(plan, 1, 0, ws, copy=first)
        with pytest.raises(cp.CpattnError, match="one kind of hop"):
            cp.ring_step(plan, 1, 1, ws, copy=second)
        torch.cuda.synchronize()    # the refused pass's step 0 (and any hop it queued) is done
    o, lse = cp.ring_forward(qd, kd, vd, plan, ws=ws)
    torch.cuda.synchronize()
    ref_o, ref_lse = oracle.get().attention(q, k, v, causal=True)
    compare(o.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_lse, what="after refused passes")


def test_ring_step_calls_one_by_one():
    """permute, then each ring step as its own C-ABI call on a compute and a copy stream, then
    finalize: the result equals the oracle for every rank's rows."""
    T, h, n_kv, d, n_cp, layout = 512, 2, 1, 64, 4, 1
    q, k, v = inputs(77, 1, T, h, n_kv, d)
    orc = oracle.get()
    plan = cp.Plan(T, h, n_kv, d, n_cp, layout, True)
    qd, kd, vd = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    ws = cp.alloc_workspace(plan.ring_workspace_size(1))
    copy = torch.cuda.Stream()
    cp.permute(qd, kd, vd, plan, ws)
    out = torch.empty_like(qd)
    lse = torch.empty((1, h, T), dtype=torch.float32, device="cuda")
    for s in range(n_cp):
        cp.ring_step(plan, 1, s, ws, compute=torch.cuda.current_stream(), copy=copy)
    cp.finalize(plan, 1, ws, out, lse)
    torch.cuda.synchronize()
    cp.check(plan, ws)
    lay = orc.layout_map(T, n_cp, layout)
    for r in range(n_cp):
        rows = lay[r]
        ref_o, ref_lse = orc.attention(q, k, v, causal=True, rows=rows)
        compare(out.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_lse, rows=rows, what=f"rank {r} rows")


@pytest.mark.parametrize("layout", [0, 1, 2], ids=["contiguous", "zigzag", "striped"])
@pytest.mark.parametrize("path", ["fused", "ring"])
def test_position_ids_drive_the_mask(layout, path):
    T, h, d, n_cp = 768, 2, 64, 4
    q, k, v = inputs(31, 1, T, h, 1, d)
    rng = np.random.default_rng(9)
    for pos in (np.arange(T)[::-1].copy(), rng.permutation(T), rng.integers(0, 50, T), np.arange(T) // 7):
        pos = pos.astype(np.int32)
        ref_o, ref_lse = oracle.get().attention(q, k, v, causal=True, pos=pos)
        o, lse, _, _ = run(q, k, v, n_cp, layout, True, pos=pos, path=path)
        compare(o, lse, ref_o, ref_lse, what=f"custom positions, layout {layout}, {path}")


def test_explicit_scale():
    T, h, d, n_cp = 512, 2, 128, 2
    q, k, v = inputs(41, 1, T, h, 2, d)
    ref_o, ref_lse = oracle.get().attention(q, k, v, causal=True, scale=0.2)
    o, lse, _, _ = run(q, k, v, n_cp, 1, True, scale=0.2)
    compare(o, lse, ref_o, ref_lse, what="scale 0.2")


@pytest.mark.parametrize("case", [(512, 2, 2, 64, 4, 0), (16384, 32, 8, 128, 8, 1), (1040, 2, 1, 128, 8, 2),
                                  (800, 4, 2, 128, 4, 1)])
def test_block_skip_decisions_bit_exact(case):
    """Tiles the kernel computed, by (rank, step) and class, equal B*h times the plan's counts,
    which equal the oracle's brute-force classification."""
    T, h, n_kv, d, n_cp, layout = case
    B = 1
    q, k, v = inputs(3, B, T, h, n_kv, d)
    for path in ("fused", "ring"):
        _, _, plan, ws = run(q, k, v, n_cp, layout, True, path=path)
        full, diag = cp.tile_counts(plan, B, ws)
        want = oracle.get().plan_counts(T, n_cp, layout, True, 128, 128)
        assert np.array_equal(full, B * h * want["full"]), path
        assert np.array_equal(diag, B * h * want["diag"]), path


def test_merge_kernel_matches_oracle():
    orc = oracle.get()
    rng = np.random.default_rng(4)
    for S, rows, h, d in ((1, 37, 2, 64), (2, 300, 4, 128), (5, 129, 3, 128), (16, 64, 1, 64)):
        o_parts = rng.standard_normal((S, rows, h, d)).astype(np.float32)
        lse_parts = (rng.standard_normal((S, h, rows)) * 4).astype(np.float32)
        lse_parts[rng.random((S, h, rows)) < 0.2] = -np.inf          # empty partials
        lse_parts[:, 0, 0] = -np.inf                                   # a row empty everywhere
        ref_o, ref_lse = orc.merge(o_parts.astype(np.float64), lse_parts.astype(np.float64))
        o, lse = cp.merge(torch.from_numpy(o_parts).cuda(), torch.from_numpy(lse_parts).cuda())
        o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(lse), fin)
        assert np.max(np.abs(lse[fin] - ref_lse[fin])) < 1e-5
        assert np.max(np.abs(o - ref_o)) <= 2 ** -8 * max(1.0, float(np.max(np.abs(ref_o)))) + 1e-6


def test_wait_timeout_is_reported_not_hung():
    ws = cp.alloc_workspace(4096)
    cp.selftest_wait_timeout(ws, timeout_ns=50_000_000)
    torch.cuda.synchronize()
    with pytest.raises(cp.CpattnError) as e:
        cp.check(None, ws)
    assert e.value.status == 5
    # the context is still usable afterwards
    q, k, v = inputs(1, 1, 256, 1, 1, 64)
    o, lse, plan, ws2 = run(q, k, v, 2, 0, True)
    assert np.all(np.isfinite(o))


def test_reserved_sms_change_no_result():
    """Leaving SMs free only changes which CTA runs a unit, not a unit's arithmetic: the fused forward
    and the ring-step path give bit-identical results with 8 SMs left free."""
    B, T, h, n_kv, d, n_cp = 1, 2048, 4, 2, 128, 4
    q, k, v = inputs(71, B, T, h, n_kv, d)
    qd, kd, vd = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    plan = cp.Plan(T, h, n_kv, d, n_cp, "zigzag", True)
    o0, l0 = cp.forward(qd, kd, vd, plan)
    r0, rl0 = cp.ring_forward(qd, kd, vd, plan)
    plan.set_reserved_sms(8)
    o1, l1 = cp.forward(qd, kd, vd, plan)
    r1, rl1 = cp.ring_forward(qd, kd, vd, plan)
    torch.cuda.synchronize()
    assert torch.equal(o0.view(torch.int16), o1.view(torch.int16)) and torch.equal(l0, l1)
    assert torch.equal(r0.view(torch.int16), r1.view(torch.int16)) and torch.equal(rl0, rl1)
