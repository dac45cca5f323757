"""Session cache of oracle automata and vocabularies for the tests."""

import functools

from oracle.dfa import compile_grammar
from workloads import GRAMMARS, make_vocab


@functools.lru_cache(maxsize=None)
def oracle_dfa(name: str):
    g = GRAMMARS[name]
    return compile_grammar(g.kind, g.source, g.bounds)


@functools.lru_cache(maxsize=None)
def vocab(kind: str, V: int, seed: int = 0):
    return make_vocab(kind, V, seed)


def parse_marked(data: bytes) -> list[int]:
    """Bytes with \\x01...\\x02 around host-injected parts -> symbol list."""
    out, forced = [], False
    for b in data:
        if b == 1:
            forced = True
        elif b == 2:
            forced = False
        else:
            out.append(b + 256 if forced else b)
    return out
