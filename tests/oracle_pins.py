"""Pins for the oracle: checks against what the pages and the mathematics fix.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when it disagrees with
a fact that does not come from the oracle itself: a library softmax-attention routine
(PyTorch's scaled_dot_product_attention in float64), a closed form, a figure printed on the
pages (``golden/pages_figures.json``, each with its citation), or brute force on tiny
inputs. The pins run against the committed oracle in ``test_oracle_pins.py`` and against
deliberately broken copies of it in ``test_oracle_mutations.py``.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import synth

CONTIGUOUS, ZIGZAG, STRIPED = 0, 1, 2
FULL, DIAG, SKIP = 0, 1, 2
with open(os.path.join(os.path.dirname(__file__), "golden", "pages_figures.json")) as _f:
    GOLDEN = json.load(_f)


def _qkv(seed, B, T, h, n_kv, d, k_mult=1.0):
    q = synth.normal_bf16(seed, synth.TAG_Q, (B, T, h, d))
    k = synth.normal_bf16(seed, synth.TAG_K, (B, T, n_kv, d), mult=k_mult)
    v = synth.normal_bf16(seed, synth.TAG_V, (B, T, n_kv, d))
    return q, k, v


def _f64(bits):
    return torch.from_numpy(synth.bf16_bits_to_f32(bits).astype(np.float64))


def _sdpa(q, k, v, causal, scale=None, mask=None):
    """Library reference: torch SDPA in float64 on [B,T,h,d] inputs, K/V heads repeat-interleaved."""
    Q, K, V = (_f64(x).permute(0, 2, 1, 3) for x in (q, k, v))
    g = Q.shape[1] // K.shape[1]
    K = K.repeat_interleave(g, dim=1)
    V = V.repeat_interleave(g, dim=1)
    out = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, is_causal=causal and mask is None,
                                                           scale=scale)
    return out.permute(0, 2, 1, 3).numpy()


def _maxabs(a, b):
    # a NaN difference (a planted mistake meeting -inf) stays NaN and fails every "<= tol" check
    with np.errstate(invalid="ignore"):
        return float(np.max(np.abs(np.asarray(a) - np.asarray(b)))) if np.size(a) else 0.0


# --------------------------------------------------------------------------------------
# The attention definition against a library routine
# --------------------------------------------------------------------------------------

def pin_sdpa_mha(orc):
    q, k, v = _qkv(11, 2, 37, 3, 3, 16)
    for causal in (True, False):
        o, _ = orc.attention(q, k, v, causal=causal)
        assert _maxabs(o, _sdpa(q, k, v, causal)) < 1e-12, "MHA output differs from SDPA"
    o, _ = orc.attention(q, k, v, causal=True, scale=0.37)
    assert _maxabs(o, _sdpa(q, k, v, True, scale=0.37)) < 1e-12, "explicit scale not honoured"


def pin_sdpa_gqa(orc):
    q, k, v = _qkv(12, 1, 29, 6, 2, 16)
    for causal in (True, False):
        o, _ = orc.attention(q, k, v, causal=causal)
        assert _maxabs(o, _sdpa(q, k, v, causal)) < 1e-12, "GQA head map differs from repeat-interleave"


def pin_pos_mask(orc):
    """Position ids decide the causal mask: key u visible to query t iff pos[u] <= pos[t]."""
    q, k, v = _qkv(13, 1, 24, 2, 1, 16)
    rng = np.random.default_rng(5)
    for pos in (rng.permutation(24).astype(np.int32), rng.integers(0, 6, 24).astype(np.int32)):
        o, _ = orc.attention(q, k, v, causal=True, pos=pos)
        mask = torch.from_numpy(pos[None, :] <= pos[:, None])          # [t, u]
        assert _maxabs(o, _sdpa(q, k, v, False, mask=mask)) < 1e-12, "position-id mask wrong"


def pin_rows_and_keys(orc):
    q, k, v = _qkv(14, 1, 40, 2, 2, 16)
    full_o, full_l = orc.attention(q, k, v, causal=True)
    rows = np.array([39, 0, 17, 5])
    o, l = orc.attention(q, k, v, causal=True, rows=rows)
    assert _maxabs(o, full_o[:, rows]) == 0.0 and _maxabs(l, full_l[:, :, rows]) == 0.0, "row subset"
    keys = np.array([3, 9, 10, 11, 30, 31, 38])
    o, _ = orc.attention(q, k, v, causal=False, keys=keys)
    ref = _sdpa(q, k[:, keys], v[:, keys], False)
    assert _maxabs(o, ref) < 1e-12, "key subset differs from SDPA on the subset"


# --------------------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------------------

def pin_uniform_scores(orc):
    """Q = 0 gives equal scores: O[t] = mean of the visible V, lse = ln |V(t)|."""
    B, T, h, d = 1, 33, 2, 16
    _, k, v = _qkv(15, B, T, h, h, d)
    q = np.zeros((B, T, h, d), dtype=np.uint16)
    vf = synth.bf16_bits_to_f32(v).astype(np.float64)
    o, l = orc.attention(q, k, v, causal=True)
    cmean = np.cumsum(vf, axis=1) / np.arange(1, T + 1)[None, :, None, None]
    assert _maxabs(o, cmean) < 1e-12, "causal uniform-score mean"
    assert _maxabs(l[0, 0], np.log(np.arange(1, T + 1))) < 1e-12, "causal lse = ln(t+1)"
    o, l = orc.attention(q, k, v, causal=False)
    assert _maxabs(o, np.broadcast_to(vf.mean(axis=1, keepdims=True), o.shape)) < 1e-12, "non-causal mean"
    assert _maxabs(l, np.full(l.shape, math.log(T))) < 1e-12, "non-causal lse = ln T"


def pin_single_key(orc):
    """Causal token 0 sees only key 0: O = V[0], lse = scale * <q_0, k_0>."""
    q, k, v = _qkv(16, 1, 8, 2, 1, 32)
    o, l = orc.attention(q, k, v, causal=True)
    qf, kf, vf = (synth.bf16_bits_to_f32(x).astype(np.float64) for x in (q, k, v))
    scale = 1.0 / math.sqrt(32)
    for i in range(2):
        assert _maxabs(o[0, 0, i], vf[0, 0, 0]) < 1e-15, "O at t=0"
        assert abs(l[0, i, 0] - scale * float(qf[0, 0, i] @ kf[0, 0, 0])) < 1e-12, "lse at t=0"


# --------------------------------------------------------------------------------------
# The ring and the merge against the definition
# --------------------------------------------------------------------------------------

def pin_ring_equals_definition(orc):
    """The pages: blockwise online softmax around the ring is exact."""
    for layout in (CONTIGUOUS, ZIGZAG, STRIPED):
        for n_cp in (1, 2, 4):
            for causal in (True, False):
                q, k, v = _qkv(17 + n_cp, 1, 32, 4, 2, 16, k_mult=2.0)
                ref_o, ref_l = orc.attention(q, k, v, causal=causal)
                for block in (1, 3, 16):
                    o, l = orc.ring(q, k, v, n_cp, layout, causal=causal, block=block)
                    assert _maxabs(o, ref_o) < 1e-12 and _maxabs(l, ref_l) < 1e-12, \
                        f"ring != definition (layout {layout}, n_cp {n_cp}, causal {causal}, block {block})"


def pin_merge_partition(orc):
    """Merging partials over a partition of the keys gives the full result; empty parts are identities."""
    q, k, v = _qkv(21, 1, 30, 2, 2, 16)
    T = 30
    full_o, full_l = orc.attention(q, k, v, causal=True)
    rng = np.random.default_rng(3)
    label = rng.integers(0, 4, T)
    label[:3] = 0                                       # part 3 may be empty for early rows
    parts_o, parts_l = [], []
    for s in range(5):                                  # part 4 is empty for every row
        keys = np.nonzero(label == s)[0]
        if keys.size:
            o, l = orc.attention(q, k, v, causal=True, keys=keys)
        else:
            o = np.zeros_like(full_o)
            l = np.full_like(full_l, -np.inf)
        parts_o.append(o[0])
        parts_l.append(l[0])
    mo, ml = orc.merge(np.stack(parts_o), np.stack(parts_l))
    assert _maxabs(mo, full_o[0]) < 1e-12 and _maxabs(ml, full_l[0]) < 1e-12, "merge of a partition"
    so, sl = orc.merge(np.stack(parts_o[:1]), np.stack(parts_l[:1]))
    assert _maxabs(so, parts_o[0]) < 1e-15 and _maxabs(sl[np.isfinite(sl)], parts_l[0][np.isfinite(sl)]) < 1e-15
    eo, el = orc.merge(np.zeros((2, 3, 1, 4)), np.full((2, 1, 3), -np.inf))
    assert np.all(eo == 0) and np.all(el == -np.inf), "all-empty merge"
    # equal lse: plain average, lse + ln 2
    a = np.ones((1, 1, 1, 4)); b = 3 * np.ones((1, 1, 1, 4))
    mo, ml = orc.merge(np.concatenate([a, b]), np.array([[[0.5]], [[0.5]]]))
    assert _maxabs(mo, 2 * np.ones((1, 1, 4))) < 1e-15 and abs(ml[0, 0] - (0.5 + math.log(2))) < 1e-15


# --------------------------------------------------------------------------------------
# Placement, block classes, work and bytes
# --------------------------------------------------------------------------------------

def pin_layout_examples(orc):
    """T = 16 over 4 ranks, written out by hand from the pages' descriptions."""
    assert orc.layout_map(16, 4, CONTIGUOUS)[1].tolist() == [4, 5, 6, 7]
    assert orc.layout_map(16, 4, ZIGZAG)[1].tolist() == [2, 3, 12, 13]     # chunks 1 and 6 of 8
    assert orc.layout_map(16, 4, STRIPED)[1].tolist() == [1, 5, 9, 13]
    z0 = orc.layout_map(16, 4, ZIGZAG)[0].tolist()
    assert z0[:2] == [0, 1] and z0[2:] == [14, 15], "GPU 0 gets the first chunk and the last"
    assert orc.chunk_assignment(4, ZIGZAG, 1) == [1, 6]
    assert orc.chunk_assignment(4, CONTIGUOUS, 2) == [2]
    for layout in (CONTIGUOUS, ZIGZAG, STRIPED):
        for T, n_cp in ((16, 4), (48, 3), (64, 8), (10, 1)):
            m = orc.layout_map(T, n_cp, layout)
            assert sorted(m.ravel().tolist()) == list(range(T)), "layout is a bijection"
            assert all(orc.token_of(T, n_cp, layout, r, j) == m[r, j] for r in range(n_cp) for j in range(T // n_cp))


def pin_classify_small(orc):
    assert orc.classify([5, 6], [1, 2]) == FULL
    assert orc.classify([5, 6], [1, 5]) == FULL
    assert orc.classify([5, 6], [7, 8]) == SKIP
    assert orc.classify([5, 6], [5, 7]) == DIAG
    assert orc.classify([5, 6], [6, 7]) == DIAG
    assert orc.classify([5, 6], [7, 8], causal=False) == FULL


def pin_half_units(orc):
    """Contiguous causal: rank r does 2r+1 half blocks, so the last does 2n_cp-1 times the first;
    zigzag: every rank does the same (4 n_cp half chunks)."""
    fig = GOLDEN["causal_imbalance"]
    assert fig["printed_ratio_formula"] == "2*n_cp - 1" and fig["zigzag_equal"]
    for n_cp in (1, 2, 4, 8, 16):
        c = orc.half_units(n_cp * 8, n_cp, CONTIGUOUS)
        assert c.tolist() == [2 * r + 1 for r in range(n_cp)]
        assert c[-1] == (2 * n_cp - 1) * c[0]
        z = orc.half_units(n_cp * 8, n_cp, ZIGZAG)
        assert z.tolist() == [4 * n_cp] * n_cp
        s = orc.half_units(n_cp * 8, n_cp, STRIPED)
        assert len(set(s.tolist())) == 1
    assert orc.half_units(64, 4, CONTIGUOUS, causal=False).tolist() == [8] * 4


def pin_pairs_closed_forms(orc):
    T, n_cp = 512, 4
    n, m = T // n_cp, T // (2 * n_cp)
    c = orc.plan_counts(T, n_cp, CONTIGUOUS)["pairs"].tolist()
    assert c == [8256, 24640, 41024, 57408]                     # n^2 r + n(n+1)/2 at n = 128
    assert c == [n * n * r + n * (n + 1) // 2 for r in range(n_cp)]
    z = orc.plan_counts(T, n_cp, ZIGZAG)["pairs"].tolist()
    assert z == [m * (T + 1)] * n_cp
    s = orc.plan_counts(T, n_cp, STRIPED)["pairs"].tolist()
    assert s == [n_cp * n * (n - 1) // 2 + n * (r + 1) for r in range(n_cp)]
    for counts in (c, z, s):
        assert sum(counts) == T * (T + 1) // 2
    nc = orc.plan_counts(T, n_cp, ZIGZAG, causal=False)["pairs"].tolist()
    assert nc == [n * T] * n_cp


def pin_step_classes(orc):
    """Block classes per (rank, ring step) at block granularity. At step s rank r holds the block
    of (r - s) mod n_cp: its left neighbour's block arrives each step."""
    T, n_cp = 64, 4
    n, m = T // n_cp, T // (2 * n_cp)
    pc = orc.plan_counts(T, n_cp, CONTIGUOUS, bq=n, bk=n)
    for r in range(n_cp):
        for s in range(n_cp):
            want = DIAG if s == 0 else (FULL if s <= r else SKIP)
            got = [pc["full"][r, s], pc["diag"][r, s], pc["skip"][r, s]]
            assert got == [int(want == FULL), int(want == DIAG), int(want == SKIP)], f"contiguous r{r} s{s}"
    pz = orc.plan_counts(T, n_cp, ZIGZAG, bq=m, bk=m)
    for r in range(n_cp):
        assert [pz["full"][r, 0], pz["diag"][r, 0], pz["skip"][r, 0]] == [1, 2, 1], "zigzag own step"
        for s in range(1, n_cp):
            assert [pz["full"][r, s], pz["diag"][r, s], pz["skip"][r, s]] == [2, 0, 2], "zigzag foreign step"
    ps = orc.plan_counts(T, n_cp, STRIPED, bq=n, bk=n)
    assert np.all(ps["diag"] == 1), "striped blocks are all partly visible"
    tiles = orc.plan_counts(T, n_cp, CONTIGUOUS, bq=5, bk=7)
    nt = (-(-n // 5)) * (-(-n // 7))
    assert np.all(tiles["full"] + tiles["diag"] + tiles["skip"] == nt), "ragged tiles cover the block"


def pin_bytes_pages(orc):
    fig = GOLDEN["ring_kv_bytes_405b"]
    T, n_cp, d_k, n_kv, h = fig["T"], fig["n_cp"], fig["d_k"], fig["n_kv_per_gpu"], fig["h_per_gpu"]
    n = T // n_cp
    b = orc.kv_bytes_recv(1, n, n_kv, d_k, n_cp)
    assert b == 4 * n * n_kv * d_k * (n_cp - 1) == 62_914_560
    assert round(b / 1e6) == fig["printed_megabytes"]
    assert round(b / 50e9 * 1e3, 1) == fig["printed_ms"]                 # InfiniBand, 50 GB/s (reading)
    no_gqa = orc.kv_bytes_recv(1, n, h, d_k, n_cp)
    assert no_gqa == fig["printed_without_gqa_factor"] * b
    assert round(no_gqa / 50e9 * 1e3) == fig["printed_without_gqa_ms"]
    assert orc.kv_bytes_recv(3, n, n_kv, d_k, n_cp) == 3 * b
    for method in (0, 1):
        assert orc.cp_comm_bytes(T, h * d_k, n_kv * d_k, n_cp, method) == b, "ring == all-gather bytes"


def pin_overlap_pages(orc):
    fig = GOLDEN["overlap_bar_tokens"]
    F = 989e12                                  # H100 dense bf16 (reading; the page gives none)
    nvl = orc.overlap_min_tokens(F, 450e9, 1, 1)
    ib = orc.overlap_min_tokens(F, 50e9, 1, 1)
    assert abs(nvl - fig["printed_nvlink_tokens"]) / fig["printed_nvlink_tokens"] < 0.01
    assert abs(ib - fig["printed_ib_tokens"]) / fig["printed_ib_tokens"] < 0.02
    gqa = orc.overlap_min_tokens(F, 450e9, 64, 8)
    assert abs(nvl / gqa - fig["printed_gqa_factor"]) < 1e-12
    assert fig["printed_tokens_per_gpu_128k_cp16"] > nvl and fig["printed_tokens_per_gpu_128k_cp16"] > ib / 8


def pin_ulysses(orc):
    fig = GOLDEN["ulysses_breakeven"]
    assert orc.ulysses_breakeven(16, 16) == fig["printed_mha_group_larger_than"]
    assert orc.ulysses_breakeven(64, 8) == fig["printed_gqa8_group_larger_than"]
    T, d_k, h, n_kv = 4096, 128, 64, 8
    n_eq = orc.ulysses_breakeven(h, n_kv)
    ring = orc.cp_comm_bytes(T, h * d_k, n_kv * d_k, n_eq, 0)
    uly = orc.cp_comm_bytes(T, h * d_k, n_kv * d_k, n_eq, 2)
    assert abs(ring - uly) / ring < 1e-12
    assert orc.cp_comm_bytes(T, h * d_k, n_kv * d_k, 16, 2) < orc.cp_comm_bytes(T, h * d_k, n_kv * d_k, 16, 0)


def pin_ulysses_split_equals_definition(orc):
    """The head split run literally (token shards, all-to-all, per-rank attention, all-to-all
    back) gives plain attention: against the library routine, every head count, KV split or
    replication, mask and position case."""
    rng = np.random.default_rng(11)
    for (h, n_kv) in ((8, 8), (8, 2), (8, 1)):
        q, k, v = _qkv(40 + h + n_kv, 1, 32, h, n_kv, 16)
        for n_cp in (1, 2, 4, 8):
            for causal in (True, False):
                o, lse = orc.ulysses(q, k, v, n_cp, causal=causal)
                assert _maxabs(o, _sdpa(q, k, v, causal)) < 1e-12
                o2, lse2 = orc.attention(q, k, v, causal=causal)
                assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
        pos = np.sort(rng.integers(0, 64, size=32)).astype(np.int32)
        o, _ = orc.ulysses(q, k, v, 4, causal=True, pos=pos)
        mask = torch.from_numpy(pos[None, :] <= pos[:, None])
        assert _maxabs(o, _sdpa(q, k, v, False, mask=mask)) < 1e-12


def pin_ulysses_bytes(orc):
    """Per-rank all-to-all bytes counted rank pair by rank pair: the pages' closed form when the
    KV heads split evenly, a hand count when they are replicated, and more bytes than the closed
    form once replication sets in."""
    for (B, T, h, n_kv, d_k, n_cp) in ((1, 131072, 64, 8, 128, 8), (2, 4096, 16, 16, 64, 4), (1, 16384, 32, 8, 128, 2)):
        got = orc.ulysses_bytes_recv(B, T, h, n_kv, d_k, n_cp)
        closed = B * orc.cp_comm_bytes(T, h * d_k, n_kv * d_k, n_cp, 2)
        assert np.all(got == got[0]) and got[0] == closed
    # T = 4, h = 2, n_kv = 1, n_cp = 2, d_k = 1: each rank receives the other rank's 2 tokens of its
    # query head, of the shared KV head (K and V), and 2 tokens of the other rank's output head:
    # 8 numbers of 2 bytes
    assert list(orc.ulysses_bytes_recv(1, 4, 2, 1, 1, 2)) == [16, 16]
    rep = orc.ulysses_bytes_recv(1, 131072, 64, 8, 128, 16)[0]
    assert rep > orc.cp_comm_bytes(131072, 64 * 128, 8 * 128, 16, 2)


# --------------------------------------------------------------------------------------
# Gradients: a library's automatic differentiation, finite differences of the forward
# definition, closed forms, an invariant, and the ring simulation
# --------------------------------------------------------------------------------------

def _dout(seed, B, T, h, d):
    return synth.normal_bf16(seed, 4, (B, T, h, d))


def _autograd(q, k, v, dout, causal, scale=None, mask=None):
    """torch float64 autograd of SDPA (K/V heads repeat-interleaved) for L = sum(O * dO)."""
    Q, K, V = (_f64(x).permute(0, 2, 1, 3).clone().requires_grad_(True) for x in (q, k, v))
    g = Q.shape[1] // K.shape[1]
    out = torch.nn.functional.scaled_dot_product_attention(Q, K.repeat_interleave(g, dim=1),
                                                           V.repeat_interleave(g, dim=1), attn_mask=mask,
                                                           is_causal=causal and mask is None, scale=scale)
    (out * _f64(dout).permute(0, 2, 1, 3)).sum().backward()
    return tuple(x.grad.permute(0, 2, 1, 3).numpy() for x in (Q, K, V))


def pin_backward_autograd(orc):
    for (B, T, h, n_kv, d, causal) in ((1, 41, 4, 2, 16, True), (2, 23, 2, 2, 8, False), (1, 30, 6, 1, 8, True)):
        q, k, v = _qkv(31, B, T, h, n_kv, d)
        do = _dout(31, B, T, h, d)
        dq, dk, dv = orc.backward(q, k, v, do, causal=causal)
        rq, rk, rv = _autograd(q, k, v, do, causal)
        assert _maxabs(dq, rq) < 1e-11 and _maxabs(dk, rk) < 1e-11 and _maxabs(dv, rv) < 1e-11, \
            f"gradients differ from autograd (B={B} T={T} h={h} n_kv={n_kv} causal={causal})"
    # explicit scale and a mask from position ids
    q, k, v = _qkv(32, 1, 20, 2, 1, 8)
    do = _dout(32, 1, 20, 2, 8)
    pos = np.array([3, 1, 4, 1, 5, 9, 2, 6, 5, 3, 5, 8, 9, 7, 9, 3, 2, 3, 8, 4], dtype=np.int32)
    mask = torch.from_numpy(pos[None, :] <= pos[:, None])
    dq, dk, dv = orc.backward(q, k, v, do, causal=True, scale=0.3, pos=pos)
    rq, rk, rv = _autograd(q, k, v, do, False, scale=0.3, mask=mask)
    assert _maxabs(dq, rq) < 1e-11 and _maxabs(dk, rk) < 1e-11 and _maxabs(dv, rv) < 1e-11, \
        "gradients with position ids and an explicit scale differ from autograd"


def _loss(orc, q, k, v, do, causal):
    o, _ = orc.attention(q, k, v, causal=causal)
    return float(np.sum(o * synth.bf16_bits_to_f32(do).astype(np.float64)))


def _bf16_bits(x):
    return (np.array([x], dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)[0]


def pin_backward_finite_differences(orc):
    """Central differences of the forward definition. The probed element is set to 0.5, and
    0.5 +- 2^-7 are exact in bf16, so the perturbed inputs are representable exactly."""
    B, T, h, n_kv, d = 1, 12, 2, 1, 8
    q, k, v = _qkv(33, B, T, h, n_kv, d)
    do = _dout(33, B, T, h, d)
    eps = 2.0 ** -7
    for causal in (True, False):
        for name, arr, idx in (("q", q, (0, 7, 1, 3)), ("k", k, (0, 2, 0, 5)), ("v", v, (0, 4, 0, 1))):
            base = arr.copy()
            base[idx] = _bf16_bits(0.5)
            args = {"q": q, "k": k, "v": v}
            args[name] = base
            dq, dk, dv = orc.backward(args["q"], args["k"], args["v"], do, causal=causal)
            grad = {"q": dq, "k": dk, "v": dv}[name][idx]
            plus, minus = base.copy(), base.copy()
            plus[idx] = _bf16_bits(0.5 + eps)
            minus[idx] = _bf16_bits(0.5 - eps)
            a = dict(args); a[name] = plus
            lp = _loss(orc, a["q"], a["k"], a["v"], do, causal)
            a[name] = minus
            lm = _loss(orc, a["q"], a["k"], a["v"], do, causal)
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - grad) < 2e-3 * max(1.0, abs(grad)), f"d{name} {grad} vs finite difference {fd}"


def pin_backward_closed_forms(orc):
    """Q = 0: every visible key has weight 1/|V(t)|, so dK = 0 exactly and
    dV_u = sum over the queries t that see u of dO_t / |V(t)|."""
    B, T, h, n_kv, d = 1, 19, 2, 2, 8
    _, k, v = _qkv(34, B, T, h, n_kv, d)
    q = np.zeros((B, T, h, d), dtype=np.uint16)
    do = _dout(34, B, T, h, d)
    g = synth.bf16_bits_to_f32(do).astype(np.float64)
    for causal in (True, False):
        dq, dk, dv = orc.backward(q, k, v, do, causal=causal)
        assert _maxabs(dk, 0.0) < 1e-14, "dK must vanish when Q = 0"
        want = np.zeros_like(dv)
        for u in range(T):
            for t in range(T):
                if causal and u > t:
                    continue
                want[0, u] += g[0, t] / ((t + 1) if causal else T)
        assert _maxabs(dv, want) < 1e-12, "dV closed form for Q = 0"


def pin_backward_invariants(orc):
    """sum_u dS_tu = 0 for every query, hence sum_u dK_u = 0 for every KV head and column; and
    the rows/keys subsets agree with the full computation."""
    q, k, v = _qkv(35, 2, 33, 4, 2, 16)
    do = _dout(35, 2, 33, 4, 16)
    dq, dk, dv = orc.backward(q, k, v, do, causal=True)
    assert _maxabs(dk.sum(axis=1), 0.0) < 1e-12, "key gradients must sum to zero over the keys"
    rows = np.array([0, 5, 32, 17])
    keys = np.array([32, 0, 9])
    sq, sk, sv = orc.backward(q, k, v, do, causal=True, rows=rows, keys=keys)
    assert _maxabs(sq, dq[:, rows]) < 1e-13 and _maxabs(sk, dk[:, keys]) < 1e-13 and _maxabs(sv, dv[:, keys]) < 1e-13, \
        "row/key subsets differ from the full gradients"


def pin_ring_backward_equals_definition(orc):
    for layout in (CONTIGUOUS, ZIGZAG, STRIPED):
        for causal in (True, False):
            q, k, v = _qkv(36 + layout, 1, 48, 4, 2, 8)
            do = _dout(36 + layout, 1, 48, 4, 8)
            full = orc.backward(q, k, v, do, causal=causal)
            ring = orc.ring_backward(q, k, v, do, 4, layout, causal=causal, block=5)
            for a, b in zip(full, ring):
                assert _maxabs(a, b) < 1e-12, f"ring backward differs (layout {layout}, causal {causal})"


def pin_backward_bytes(orc):
    """The pages: the backward ring roughly doubles the forward's traffic. With bf16 gradients
    the gradient blocks add n_cp/(n_cp - 1) of the forward bytes: 2 + 1/15 times at n_cp = 16."""
    fwd = orc.kv_bytes_recv(1, 8192, 1, 128, 16)
    bwd = orc.bwd_bytes_recv(1, 8192, 1, 128, 16, 2)
    assert fwd == 62914560 and bwd == 62914560 + 16 * 2 * 8192 * 128 * 2, "backward ring bytes"
    assert abs(bwd / fwd - (2 + 1 / 15)) < 1e-12


# --------------------------------------------------------------------------------------
# Document masks (packed sequences)
# --------------------------------------------------------------------------------------

def pin_document_mask(orc):
    """A query sees only its own document: against SDPA with the boolean document mask, and
    against each document's attention computed on its own (the definition on a slice)."""
    B, T, h, n_kv, d = 1, 40, 4, 2, 8
    q, k, v = _qkv(41, B, T, h, n_kv, d)
    lengths = [7, 1, 12, 20]
    doc = np.repeat(np.arange(len(lengths)), lengths).astype(np.int32)
    for causal in (True, False):
        o, lse = orc.attention_docs(q, k, v, doc, causal=causal)
        same = doc[None, :] == doc[:, None]
        mask = same & (np.arange(T)[None, :] <= np.arange(T)[:, None]) if causal else same
        ref = _sdpa(q, k, v, False, mask=torch.from_numpy(mask))
        assert _maxabs(o, ref) < 1e-12, "document mask differs from SDPA with the same mask"
        start = 0
        for ln in lengths:
            sl = slice(start, start + ln)
            so, sl_lse = orc.attention(q[:, sl], k[:, sl], v[:, sl], causal=causal)
            assert _maxabs(o[:, sl], so) < 1e-13 and _maxabs(lse[:, :, sl], sl_lse) < 1e-13, \
                "a document's rows must equal attention over that document alone"
            start += ln


def pin_document_mask_any_ids(orc):
    """Document ids in any order, documents split into pieces: against SDPA with the boolean mask
    doc[u] == doc[t] (and pos[u] <= pos[t]) under permuted positions; and one token per document,
    where every query sees only itself, so O = v_t and lse = scale <q_t, k_t> (closed form)."""
    B, T, h, n_kv, d = 1, 48, 4, 2, 8
    q, k, v = _qkv(43, B, T, h, n_kv, d)
    doc = np.array([5, 5, 2, 2, 2, 9, 5, 5, 9, 9, 2, 0] * 4, dtype=np.int32)   # pieces, ids not increasing
    pos = np.random.default_rng(3).permutation(T).astype(np.int32)
    for causal in (True, False):
        o, lse = orc.attention_docs(q, k, v, doc, causal=causal, pos=pos)
        same = doc[None, :] == doc[:, None]
        mask = same & (pos[None, :] <= pos[:, None]) if causal else same
        ref = _sdpa(q, k, v, False, mask=torch.from_numpy(mask))
        assert _maxabs(o, ref) < 1e-12, "document ids in any order differ from SDPA with the same mask"
    one = np.arange(T, dtype=np.int32)[::-1].copy()
    o, lse = orc.attention_docs(q, k, v, one, causal=False)
    qf, kf, vf = (_f64(x).numpy() for x in (q, k, v))
    g = h // n_kv
    for i in range(h):
        assert _maxabs(o[:, :, i], vf[:, :, i // g]) == 0.0, "a lone token must return its own value row"
        s = np.einsum("btc,btc->bt", qf[:, :, i], kf[:, :, i // g]) / np.sqrt(d)
        assert _maxabs(lse[:, i], s) < 1e-12, "a lone token's lse is its own score"


def pin_document_mask_gradients(orc):
    """Gradients under a document mask: against autograd with the boolean mask, and each document's
    gradients computed on its own slice."""
    B, T, h, n_kv, d = 1, 30, 4, 2, 8
    q, k, v = _qkv(42, B, T, h, n_kv, d)
    do = _dout(42, B, T, h, d)
    lengths = [9, 1, 14, 6]
    doc = np.repeat(np.arange(len(lengths)), lengths).astype(np.int32)
    dq, dk, dv = orc.backward(q, k, v, do, causal=True, doc=doc)
    mask = (doc[None, :] == doc[:, None]) & (np.arange(T)[None, :] <= np.arange(T)[:, None])
    rq, rk, rv = _autograd(q, k, v, do, False, mask=torch.from_numpy(mask))
    assert _maxabs(dq, rq) < 1e-11 and _maxabs(dk, rk) < 1e-11 and _maxabs(dv, rv) < 1e-11, \
        "document-mask gradients differ from autograd with the same mask"
    start = 0
    for ln in lengths:
        sl = slice(start, start + ln)
        gq, gk, gv = orc.backward(q[:, sl], k[:, sl], v[:, sl], do[:, sl], causal=True)
        assert _maxabs(dq[:, sl], gq) < 1e-12 and _maxabs(dk[:, sl], gk) < 1e-12 and _maxabs(dv[:, sl], gv) < 1e-12, \
            "a document's gradients must equal the gradients of that document alone"
        start += ln


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
