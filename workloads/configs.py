"""The five synthetic workloads (sizes, distributions, sampling parameters).

``tiny`` is the small case the oracle finishes in seconds; ``booking_128k`` is
the 128256-token, 256-row workload the throughput metric is quoted on; the rest
are parity cases.
"""

from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Config:
    name: str
    grammars: tuple[str, ...]   # row b uses grammars[b % len(grammars)]
    vocab_kind: str
    V: int
    B: int
    dtype: str                  # "f32" | "bf16"
    sigma: float
    boost: float
    boost_frac: float
    temp: float                 # 0 -> greedy
    top_p: float                # >= 1 -> no truncation
    steps: int
    random_start: bool = False  # rows start in uniformly drawn states
    vocab_seed: int = 0
    logit_seed: int = 1
    sample_seed: int = 0x5EED_0001


CONFIGS: dict[str, Config] = {
    "tiny": Config("tiny", ("calc_call",), "tiny", 512, 4, "f32", 1.0, 0.0, 0.0,
                   0.0, 1.0, 64),
    "booking_32k": Config("booking_32k", ("booking",), "bpe", 32000, 64, "bf16", 2.0, 0.0, 0.0,
                          0.7, 1.0, 400),
    "booking_128k": Config("booking_128k", ("booking",), "bpe", 128256, 256, "bf16", 2.0, 4.0, 0.05,
                           0.7, 0.9, 400),
    "reasoning_152k": Config("reasoning_152k", ("reasoning_answer",), "bpe", 151936, 1024, "bf16",
                             2.0, 0.0, 0.0, 0.7, 1.0, 256, random_start=True),
    "mixed_eval_152k": Config("mixed_eval_152k",
                              ("calc_call", "booking", "booking_200", "reasoning_answer_1024",
                               "calc_eval", "json_eval", "extraction", "reasoned"),
                              "bpe", 151936, 512, "bf16", 2.0, 4.0, 0.05, 0.7, 0.9, 512),
}


def get_config(name: str) -> Config:
    return CONFIGS[name]
