"""The five benchmark workloads, by shape (Llama-3-style long-context attention layers).

Every workload draws Q, K and V i.i.d. N(0, 1) rounded to bf16 from its own seed; the
non-causal one multiplies K by 2 before rounding (exact in bf16) so that scores have
standard deviation about 2 and the running max moves often. Position ids are 0..T-1.
"""
from __future__ import annotations

from dataclasses import dataclass, field

CONTIGUOUS, ZIGZAG, STRIPED = 0, 1, 2
LAYOUT_NAMES = {CONTIGUOUS: "contiguous", ZIGZAG: "zigzag", STRIPED: "striped"}
LAYOUT_IDS = {v: k for k, v in LAYOUT_NAMES.items()}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    h: int
    n_kv: int
    d: int
    n_cp: int
    layouts: tuple
    causal: bool
    seed: int
    k_mult: float = 1.0
    sampled_rows: int = 0          # 0: the oracle computes every row
    note: str = field(default="", compare=False)

    @property
    def n(self) -> int:
        return self.T // self.n_cp


CONFIGS = {
    "tiny_mha_contig_T512": Workload("tiny_mha_contig_T512", 1, 512, 2, 2, 64, 4, (CONTIGUOUS,), True, 1001,
                                     note="causal MHA, 4 contiguous ranks of 128"),
    "gqa_zigzag_T16k": Workload("gqa_zigzag_T16k", 1, 16384, 32, 8, 128, 8, (ZIGZAG,), True, 1002,
                                note="causal GQA 4:1, 16 chunks of 1024"),
    "mha_noncausal_T32k": Workload("mha_noncausal_T32k", 2, 32768, 16, 16, 128, 4, (CONTIGUOUS,), False, 1003,
                                   k_mult=2.0, sampled_rows=4096, note="non-causal MHA, K scaled by 2"),
    "llama70b_zigzag_T128k": Workload("llama70b_zigzag_T128k", 1, 131072, 64, 8, 128, 16, (ZIGZAG,), True, 1004,
                                      sampled_rows=256, note="70B-shaped causal GQA 8:1, 32 chunks of 4096"),
    "llama405b_tp_T128k": Workload("llama405b_tp_T128k", 1, 131072, 16, 1, 128, 16, (ZIGZAG, STRIPED), True, 1005,
                                   sampled_rows=256, note="405B per-TP slice, one KV head"),
}

ORDER = list(CONFIGS)


def workload(name: str) -> Workload:
    return CONFIGS[name]
