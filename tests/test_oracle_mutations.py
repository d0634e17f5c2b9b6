"""Plausible mistakes planted in copies of the oracle must each fail at least one pin.

Each case copies ``oracle/oracle.c``, replaces one exact piece of source text (which must be
found, so a change to the oracle cannot make a case pass vacuously), compiles the copy into a
temporary library on the CPU and runs every pin against it. The committed oracle is never
modified.
"""
import os
import tempfile

import pytest

import oracle
from tests import oracle_pins

# (name, original text, replacement, which occurrence (0-based) or None for all)
MUTANTS = [
    ("causal_exclusive", "return pu <= pt;", "return pu < pt;", None),
    ("gqa_map_modulo", "int kv = i / g;", "int kv = i % n_kv;", None),
    ("lse_drops_max", "*lrow = mx + log(sum);", "*lrow = log(sum);", None),
    ("scale_dropped", "s[ki] = scale * dot;", "s[ki] = dot;", None),
    ("key_row_of_query", "const uint16_t* krow = k + (((int64_t)b * T + u) * n_kv + kv) * d;",
     "const uint16_t* krow = k + (((int64_t)b * T + t) * n_kv + kv) * d;", 0),
    ("value_row_of_query", "const uint16_t* vrow = v + (((int64_t)b * T + u) * n_kv + kv) * d;",
     "const uint16_t* vrow = v + (((int64_t)b * T + t) * n_kv + kv) * d;", 0),
    ("ring_value_row_transposed", "const uint16_t* vrow = v + (((int64_t)b * T + u) * n_kv + kv) * d;",
     "const uint16_t* vrow = v + (((int64_t)b * T + u) * n_kv + (i % n_kv)) * d;", 1),
    ("ring_direction_in_counts", "int src = ((r - s) % n_cp + n_cp) % n_cp;", "int src = (r + s) % n_cp;", 1),
    ("ring_skips_own_block", "for (int s = 0; s < n_cp; ++s) {", "for (int s = 1; s < n_cp; ++s) {", 0),
    ("zigzag_mirror_off_by_one", "return (int64_t)(2 * n_cp - 1 - r) * m + (j - m);",
     "return (int64_t)(2 * n_cp - 2 - r) * m + (j - m);", None),
    ("striped_as_contiguous", "if (layout == LAYOUT_STRIPED) return j * n_cp + r;",
     "if (layout == LAYOUT_STRIPED) return (int64_t)r * n + j;", None),
    ("contiguous_transposed", "if (layout == LAYOUT_CONTIGUOUS) return (int64_t)r * n + j;",
     "if (layout == LAYOUT_CONTIGUOUS) return j * n_cp + r;", None),
    ("diag_counts_full", "units += (cls == CLASS_FULL) ? 2 : (cls == CLASS_DIAG) ? 1 : 0;",
     "units += (cls == CLASS_FULL) ? 2 : (cls == CLASS_DIAG) ? 2 : 0;", None),
    ("online_sum_not_rescaled", "l *= alpha;", "", None),
    ("online_rescale_sign", "double alpha = exp(m - m_new);", "double alpha = exp(m_new - m);", None),
    ("merge_weight_vs_max", "a += exp(x - L) *", "a += exp(x - mx) *", None),
    ("merge_lse_drops_max", "double L = mx + log(sum);", "double L = log(sum);", None),
    ("classify_strict", "if (kpos[c] <= qpos[a]) any_vis = 1; else any_hidden = 1;",
     "if (kpos[c] < qpos[a]) any_vis = 1; else any_hidden = 1;", None),
    ("pairs_strict", "for (int64_t u = 0; u < T; ++u) cnt += (!causal || lpos[u] <= pq);",
     "for (int64_t u = 0; u < T; ++u) cnt += (!causal || lpos[u] < pq);", None),
    ("bytes_count_own_block", "return (int64_t)(n_cp - 1) * 2", "return (int64_t)(n_cp) * 2", None),
    ("overlap_ratio_inverted", "return flops_per_s / bytes_per_s * (n_kv / h);",
     "return flops_per_s / bytes_per_s * (h / n_kv);", None),
    ("ulysses_keeps_all", "return 4.0 * n * (d + d_kv) * (n_cp - 1.0) / n_cp;",
     "return 4.0 * n * (d + d_kv) * (n_cp - 1.0);", None),
    # gradients
    ("bwd_drops_D", "*ds_out = p * (dp - d_t);", "*ds_out = p * dp;", None),
    ("bwd_ds_sign", "*ds_out = p * (dp - d_t);", "*ds_out = p * (d_t - dp);", None),
    ("bwd_D_unnormalised", "dd += bf16_value(grow[c]) * (acc[c] / sum);", "dd += bf16_value(grow[c]) * acc[c];", None),
    ("bwd_lse_drops_max", "*lse_out = mx + log(sum);", "*lse_out = log(sum);", None),
    ("bwd_dq_no_scale", "out[c] += scale * ds * bf16_value(krow[c]);", "out[c] += ds * bf16_value(krow[c]);", None),
    ("bwd_dk_no_scale", "if (gk) gk[c] += scale * ds * bf16_value(qrow[c]);", "if (gk) gk[c] += ds * bf16_value(qrow[c]);",
     None),
    ("bwd_dv_uses_ds", "if (gv) gv[c] += p * bf16_value(grow[c]);", "if (gv) gv[c] += ds * bf16_value(grow[c]);", None),
    ("bwd_first_head_only", "for (int i = kvh * g; i < (kvh + 1) * g; ++i)\n            for (int64_t t = 0; t < T; ++t) {",
     "for (int i = kvh * g; i < kvh * g + 1; ++i)\n            for (int64_t t = 0; t < T; ++t) {", None),
    ("ring_bwd_own_block", "int src = ((r - s) % n_cp + n_cp) % n_cp;     /* block rank r holds at step s */",
     "int src = r;", None),
    ("doc_mask_ignored", "if (doc && doc[u] != doc[t]) return 0;", "if (0) return 0;", None),
    ("doc_mask_sees_earlier_docs", "if (doc && doc[u] != doc[t]) return 0;", "if (doc && doc[u] > doc[t]) return 0;", None),
    ("bwd_bytes_grad_hops", "(int64_t)n_cp * 2 * blk * grad_bytes", "(int64_t)(n_cp - 1) * 2 * blk * grad_bytes", None),
]


def _mutate(src: str, old: str, new: str, which):
    count = src.count(old)
    assert count >= 1, f"pattern not found in oracle.c: {old!r}"
    if which is None:
        return src.replace(old, new)
    assert which < count
    idx = -1
    for _ in range(which + 1):
        idx = src.index(old, idx + 1)
    return src[:idx] + new + src[idx + len(old):]


@pytest.mark.parametrize("name,old,new,which", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, which):
    with open(oracle.SOURCE) as f:
        src = f.read()
    mutated = _mutate(src, old, new, which)
    assert mutated != src
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "oracle_mutant.c")
        with open(path, "w") as f:
            f.write(mutated)
        lib = oracle.bind(oracle.compile_source(path, os.path.join(tmp, "lib", "liboracle_mutant.so")))
        orc = oracle.Oracle(lib)
        failed = []
        for pin in oracle_pins.ALL_PINS:
            try:
                pin(orc)
            except (AssertionError, ValueError) as e:
                failed.append((pin.__name__, str(e)[:80]))
        assert failed, f"mutant {name} passed every pin"
