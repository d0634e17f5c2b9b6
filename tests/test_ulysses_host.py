"""Host-side tests of the head split (Ulysses, "Ulysses, splitting by heads instead"): the library's
plan checks and per-rank all-to-all byte counts against the oracle's rank-pair count, and the
oracle's Ulysses pins against planted mistakes (CPU only; no kernel is launched)."""
import numpy as np
import pytest

import oracle
from context_ring_attention_blockwise_gb300 import _build
import context_ring_attention_blockwise_gb300 as cp
from tests import oracle_pins


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()


SHAPES = [
    # B, T, h, n_kv, d_k, n_cp
    (1, 131072, 64, 8, 128, 16),    # 70B-shaped, KV heads replicated on 2 ranks each
    (1, 131072, 64, 8, 128, 8),     # one KV head per rank
    (1, 16384, 32, 8, 128, 8),
    (2, 32768, 16, 16, 128, 4),     # MHA
    (1, 4096, 16, 1, 64, 16),       # one KV head for all
    (3, 1040, 8, 2, 64, 4),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"B{s[0]}_T{s[1]}_h{s[2]}_kv{s[3]}_d{s[4]}_cp{s[5]}" for s in SHAPES])
def test_ulysses_counts_match_oracle(shape):
    B, T, h, n_kv, d_k, n_cp = shape
    plan = cp.UlyssesPlan(T, h, n_kv, d_k, n_cp, True)
    got = plan.counts(B)["bytes_recv"]
    want = oracle.get().ulysses_bytes_recv(B, T, h, n_kv, d_k, n_cp)
    assert np.array_equal(got, want)


def test_ulysses_counts_against_ring_bytes():
    """The pages' comparison at the 70B shape: Ulysses moves fewer bytes than the ring at 16 ranks
    (above 1 + h / n_kv = 9) even with the KV heads replicated, and more at 4."""
    for n_cp, fewer in ((16, True), (4, False)):
        uly = cp.UlyssesPlan(131072, 64, 8, 128, n_cp, True).counts(1)["bytes_recv"][0]
        ring = cp.Plan(131072, 64, 8, 128, n_cp, cp.ZIGZAG, True).counts(1)["kv_bytes_recv"][0]
        assert (uly < ring) == fewer


@pytest.mark.parametrize("args", [
    (1024, 6, 2, 64, 4),      # heads not a multiple of n_cp
    (1024, 12, 3, 64, 2),     # KV heads neither split nor replicated evenly
    (1000, 8, 8, 64, 3),      # 8 heads over 3 ranks
    (1002, 8, 8, 64, 4),      # tokens not a multiple of n_cp
    (1024, 8, 8, 96, 4),      # head width
])
def test_ulysses_plan_rejects_bad_arguments(args):
    with pytest.raises(cp.CpattnError):
        cp.UlyssesPlan(*args)


def test_plans_do_not_cross():
    uly = cp.UlyssesPlan(1024, 8, 2, 64, 4)
    with pytest.raises(cp.CpattnError) as e:
        cp.Plan.workspace_size(uly, 1)
    assert e.value.status == 1
    ring = cp.Plan(1024, 8, 2, 64, 4, cp.ZIGZAG)
    out = np.zeros(4, dtype=np.int64)
    assert cp.lib().cpattn_ulysses_counts(ring.handle, 1, out.ctypes.data) == 1


class _WrongKvHeads(oracle.Oracle):
    """Each rank takes the KV heads of the next rank."""
    def ulysses_heads(self, h, n_kv, n_cp, r):
        heads, _ = oracle.Oracle.ulysses_heads(h, n_kv, n_cp, r)
        _, kvh = oracle.Oracle.ulysses_heads(h, n_kv, n_cp, (r + 1) % n_cp)
        return heads, kvh


class _SwappedHeads(oracle.Oracle):
    """Ranks 0 and 1 swap their query heads (but keep their KV heads)."""
    def ulysses_heads(self, h, n_kv, n_cp, r):
        heads, kvh = oracle.Oracle.ulysses_heads(h, n_kv, n_cp, r)
        if n_cp > 1 and r in (0, 1):
            heads = oracle.Oracle.ulysses_heads(h, n_kv, n_cp, 1 - r)[0]
        return heads, kvh


class _CountsOwnShard(oracle.Oracle):
    """The byte count also counts what a rank keeps."""
    def ulysses_bytes_recv(self, B, T, h, n_kv, d_k, n_cp):
        return oracle.Oracle.ulysses_bytes_recv(self, B, T, h, n_kv, d_k, n_cp) * n_cp // max(n_cp - 1, 1)


@pytest.mark.parametrize("mutant", [_WrongKvHeads, _SwappedHeads, _CountsOwnShard], ids=lambda c: c.__name__)
def test_ulysses_pins_catch_planted_mistakes(mutant):
    orc = mutant(oracle.get().lib)
    failed = False
    for pin in (oracle_pins.pin_ulysses_split_equals_definition, oracle_pins.pin_ulysses_bytes):
        try:
            pin(orc)
        except (AssertionError, ValueError):
            failed = True
    assert failed, f"{mutant.__name__} passed every Ulysses pin"
