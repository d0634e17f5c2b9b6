"""Host-side tests of the C ABI: exported symbols, argument checks and the plan's block decisions
and counters, bit-exact against the oracle's brute force (CPU only; no kernel is launched)."""
import ctypes
import re
import subprocess

import numpy as np
import pytest
import torch

import oracle
import synth
from context_ring_attention_blockwise_gb300 import _build
import context_ring_attention_blockwise_gb300 as cp

HEADER = "include/cpattn.h"


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()


def declared_symbols():
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:cpattn_status_t|const char\*)\s+(cpattn_\w+)\(", text, re.M)))


def test_library_exports_every_declared_symbol():
    names = declared_symbols()
    assert len(names) >= 15
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(cpattn_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    L = cp.lib()
    for n in names:
        assert hasattr(L, n)
    assert set(cp.SYMBOLS) == set(names), "binding and header disagree"
    assert cp.version().startswith("cpattn")


@pytest.mark.parametrize("args,status", [
    ((512, 3, 2, 64, 4, 0, 1), 1),       # h % n_kv
    ((512, 2, 2, 96, 4, 0, 1), 2),       # d_k unsupported
    ((513, 2, 2, 64, 4, 0, 1), 1),       # T % n_cp
    ((516, 2, 2, 64, 4, 1, 1), 1),       # zigzag T % 2n_cp
    ((512, 2, 2, 64, 4, 7, 1), 1),       # unknown layout
    ((512, 2, 2, 64, 0, 0, 1), 1),       # n_cp
])
def test_plan_rejects_bad_arguments(args, status):
    h = ctypes.c_void_p()
    assert cp.lib().cpattn_plan(*args, ctypes.byref(h)) == status
    assert cp.lib().cpattn_last_error().decode()
    assert not h.value


def test_workspace_sizes_and_tile_shape():
    p = cp.Plan(16384, 32, 8, 128, 8, "zigzag")
    fwd, ring = p.workspace_size(1), p.ring_workspace_size(1)
    qkv = 16384 * (32 + 16) * 128 * 2
    assert qkv < fwd < qkv + (1 << 20)
    assert ring > fwd + 2 * 16384 * 16 * 128 * 2 + 16384 * 32 * 128 * 4
    assert p.workspace_size(2) > fwd
    assert p.tile_shape() == (128, 128)


def test_calls_fail_before_launch_on_bad_arguments():
    L = cp.lib()
    p = cp.Plan(512, 2, 2, 64, 4, "contiguous")
    fake = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 8)
    ws_ok = p.workspace_size(1)
    # NULL inputs, misaligned input, small or misaligned workspace, bad merge shape, bad step order
    assert L.cpattn_forward(p.handle, 1, None, fake, fake, None, 0.0, fake, fake, fake, ws_ok, None) == 1
    assert L.cpattn_forward(p.handle, 1, odd, fake, fake, None, 0.0, fake, fake, fake, ws_ok, None) == 1
    assert L.cpattn_forward(p.handle, 1, fake, fake, fake, None, 0.0, fake, fake, fake, ws_ok - 1, None) == 3
    assert L.cpattn_forward(p.handle, 1, fake, fake, fake, None, 0.0, fake, fake, odd, ws_ok, None) == 3
    assert L.cpattn_forward(p.handle, 0, fake, fake, fake, None, 0.0, fake, fake, fake, ws_ok, None) == 1
    assert L.cpattn_merge(2, 10, 2, 6, fake, fake, fake, fake, None) == 1
    assert L.cpattn_merge(2, 10, 2, 12, fake, fake, fake, fake, None) == 1     # d must be a multiple of 8
    assert L.cpattn_ring_step(p.handle, 1, 0, 0.0, fake, p.ring_workspace_size(1), None, None) == 1   # permute first
    assert "permute" in L.cpattn_last_error().decode()
    assert L.cpattn_finalize(p.handle, 1, fake, fake, fake, p.ring_workspace_size(1), None) == 1


def test_backward_ring_calls_fail_before_launch():
    """The ring-step backward checks its order, step range, workspace and pointers on the host."""
    L = cp.lib()
    T, h, n_kv, d, n_cp = 512, 2, 2, 64, 4
    p = cp.Plan(T, h, n_kv, d, n_cp, "contiguous")
    fake = ctypes.c_void_p(1 << 20)
    wsb = p.backward_ring_workspace_size(1)
    # K/V stage slots (2 x bf16 K, V), circulating dK/dV sums (2 x fp32) that each step's
    # contribution is added into, the running fp32 dQ, on top of the fused backward's workspace
    kv = T * n_kv * d
    extra = 2 * 2 * 2 * kv + 2 * 2 * 4 * kv + 4 * T * h * d
    assert p.backward_workspace_size(1) + extra <= wsb < p.backward_workspace_size(1) + extra + 16 * 1024
    assert L.cpattn_backward_ring_step(p.handle, 1, 0, 0.0, fake, wsb, None, None) == 1       # begin first
    assert "cpattn_backward_begin" in L.cpattn_last_error().decode()
    assert L.cpattn_backward_ring_step(p.handle, 1, n_cp, 0.0, fake, wsb, None, None) == 1    # step out of range
    assert L.cpattn_backward_ring_step(p.handle, 1, 0, 0.0, fake, wsb - 1, None, None) == 3   # small workspace
    assert L.cpattn_backward_finalize(p.handle, 1, fake, fake, fake, fake, wsb, None) == 1    # steps first
    assert "ring steps first" in L.cpattn_last_error().decode()
    assert L.cpattn_backward_finalize(p.handle, 1, None, fake, fake, fake, wsb, None) == 1    # NULL dq
    assert L.cpattn_backward_begin(p.handle, 1, None, fake, fake, fake, fake, fake, None, fake, wsb, None) == 1
    assert L.cpattn_backward_begin(p.handle, 1, fake, fake, fake, fake, fake, fake, None, fake, wsb - 1, None) == 3
    u = cp.UlyssesPlan(T, h, n_kv, d, 2, True)
    assert L.cpattn_backward_ring_step(u.handle, 1, 0, 0.0, fake, wsb, None, None) == 1       # a Ulysses plan


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path; would touch fake pointers on a GPU")
def test_no_cpu_fallback_without_a_device():
    p = cp.Plan(512, 2, 2, 64, 4, "contiguous")
    fake = ctypes.c_void_p(1 << 20)
    st = cp.lib().cpattn_forward(p.handle, 1, fake, fake, fake, None, 0.0, fake, fake, fake, p.workspace_size(1), None)
    assert st == 4, "without a CUDA device the forward must fail, not fall back"


def _compare_counts(T, h, n_kv, d, n_cp, layout, causal, B=1):
    orc = oracle.get()
    p = cp.Plan(T, h, n_kv, d, n_cp, layout, causal)
    got = p.counts(B)
    want = orc.plan_counts(T, n_cp, layout, causal, 128, 128)
    for key in ("full", "diag", "skip", "pairs"):
        assert np.array_equal(got[key], want[key]), key
    n = T // n_cp
    assert got["kv_bytes_recv"].tolist() == [orc.kv_bytes_recv(B, n, n_kv, d, n_cp)] * n_cp
    assert np.array_equal(got["half_units"], orc.half_units(T, n_cp, layout, causal))
    return got


@pytest.mark.parametrize("name", ["tiny_mha_contig_T512", "gqa_zigzag_T16k", "mha_noncausal_T32k"])
def test_plan_counts_match_oracle_workloads(name):
    w = synth.workload(name)
    for layout in w.layouts:
        _compare_counts(w.T, w.h, w.n_kv, w.d, w.n_cp, layout, w.causal, w.B)


@pytest.mark.parametrize("layout", [0, 1, 2])
@pytest.mark.parametrize("T,n_cp", [(800, 4), (1200, 3), (384, 2), (2048, 8), (640, 1)])
@pytest.mark.parametrize("causal", [True, False])
def test_plan_counts_match_oracle_ragged(layout, T, n_cp, causal):
    if layout == 1 and T % (2 * n_cp):
        pytest.skip("zigzag needs T % 2n_cp")
    _compare_counts(T, 4, 2, 64, n_cp, layout, causal)


def test_plan_counts_128k_closed_forms():
    """The two 128K workloads: counters from closed forms (brute force over 1.7e10 pairs is
    left to the GPU machine's oracle run in the bench)."""
    T, n_cp = 131072, 16
    n, m = T // n_cp, T // (2 * n_cp)
    z = cp.Plan(T, 64, 8, 128, n_cp, "zigzag").counts()
    assert z["pairs"].tolist() == [m * (T + 1)] * n_cp == [536875008] * n_cp
    assert z["half_units"].tolist() == [4 * n_cp] * n_cp
    s = cp.Plan(T, 16, 1, 128, n_cp, "striped").counts()
    assert s["pairs"].tolist() == [n_cp * n * (n - 1) // 2 + n * (r + 1) for r in range(n_cp)]
    assert s["pairs"][0] == 536813568 and s["pairs"][-1] == 536936448
    z5 = cp.Plan(T, 16, 1, 128, n_cp, "zigzag").counts()
    assert z5["kv_bytes_recv"][0] == 62_914_560          # the page's 63 MB per GPU per layer
    # tiles: every (rank, step) covers the 64 x 64 tile grid of one block
    for c in (z, s, z5):
        assert np.all(c["full"] + c["diag"] + c["skip"] == 64 * 64)
    # zigzag, steps 1..15: two of the four chunk pairs are visible -> exactly half the tiles, all FULL
    assert np.all(z["full"][:, 1:] == 2 * 32 * 32) and np.all(z["diag"][:, 1:] == 0)
    # striped: only the 64 diagonal tiles of each block are partly visible
    assert np.all(s["diag"] == 64)


@pytest.mark.parametrize("shape", [(1, 131072, 64, 8, 128, 16), (2, 32768, 16, 16, 128, 4), (1, 1040, 8, 2, 64, 4)])
def test_backward_counts_match_oracle(shape):
    """Bytes each rank receives in the backward ring: the oracle's count with fp32 gradient blocks."""
    B, T, h, n_kv, d, n_cp = shape
    plan = cp.Plan(T, h, n_kv, d, n_cp, cp.ZIGZAG if T % (2 * n_cp) == 0 else cp.CONTIGUOUS, True)
    got = plan.backward_counts(B)["bytes_recv"]
    want = oracle.get().bwd_bytes_recv(B, T // n_cp, n_kv, d, n_cp, 4)
    assert np.all(got == want)
    fwd = plan.counts(B)["kv_bytes_recv"]
    assert np.all(got > 2 * fwd)


@pytest.mark.parametrize("T,h,n_kv,d,n_cp,layout,B", [
    (131072, 16, 1, 128, 16, "zigzag", 1),       # the 405B per-TP slice: the pages' 63 MB
    (16384, 32, 8, 128, 8, "zigzag", 1),
    (32768, 16, 16, 128, 4, "contiguous", 2),
    (1536, 4, 2, 64, 3, "striped", 3),
])
def test_allgather_bytes_match_the_oracle(T, h, n_kv, d, n_cp, layout, B):
    """All-gather bytes per rank ("What context parallelism communicates": each rank receives the
    other n_cp - 1 chunks of K and V) bit-exact against the oracle's count for method 1."""
    plan = cp.Plan(T, h, n_kv, d, n_cp, layout)
    got = plan.allgather_counts(B)["bytes_recv"]
    want = B * oracle.get().cp_comm_bytes(T, h * d, n_kv * d, n_cp, oracle.ALLGATHER)
    assert float(want).is_integer() and np.all(got == int(want))
    assert np.all(got == plan.counts(B)["kv_bytes_recv"])   # the same volume as the ring
    if T == 131072 and n_kv == 1:
        assert int(got[0]) == 62914560


def test_reserved_sms_host_checks():
    plan = cp.Plan(2048, 4, 2, 128, 4, "zigzag")
    plan.set_reserved_sms(8)
    plan.set_reserved_sms(0)
    L = cp.lib()
    assert L.cpattn_plan_set_reserved_sms(plan.handle, -1) == 1
    assert L.cpattn_plan_set_reserved_sms(None, 4) == 1
