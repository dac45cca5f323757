"""Seeded synthetic inputs shared by the CUDA path's tests/bench and by the oracle.

This package holds only input generation: vocabularies, logits, grammar source
texts, per-row random draws and the workload table.  It contains none of the
method's arithmetic (no automaton, no masking, no sampling), so both the
product path and the oracle may import it without sharing any computation.

The workloads stand in for the pages' own (Llama 3.1 8B / Qwen2.5 vocabularies,
booking-decision schema runs, GSM8K answers), none of which ships here.
"""

from .configs import CONFIGS, Config, get_config  # noqa: F401
from .grammars import GRAMMARS, PDA_GRAMMARS, GrammarSpec, Bounds  # noqa: F401
from .vocab import make_vocab, vocab_csr  # noqa: F401
from .logits import make_logits, make_start_draws  # noqa: F401
