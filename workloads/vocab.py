"""Synthetic tokenizer vocabularies (seeded).

Two families, matching the workload descriptions:

* ``tiny``: every printable single byte 0x20..0x7E (95 tokens), then random
  2..6-byte strings over digits, arithmetic operators, letters and JSON
  punctuation, deduplicated, until ``V`` tokens exist.
* ``bpe``: every single byte 0x00..0xFF (256 tokens), then random strings whose
  length is geometric with mean 4 (p = 1/4) capped at 16 bytes (a draw of 1 or
  above 16, or a duplicate, is redrawn); each byte is printable ASCII
  (0x20..0x7E, uniform) with probability 0.9 and uniform over 0..255 otherwise.

Token ids are positions in the returned list.
"""

from __future__ import annotations

import numpy as np

_TINY_ALPHABET = (b"0123456789+-*/() " + b"abcdefghijklmnopqrstuvwxyz"
                  + b"ABCDEFGHIJKLMNOPQRSTUVWXYZ" + b'{}[]:,"')


def make_vocab(kind: str, V: int, seed: int) -> list[bytes]:
    rng = np.random.default_rng(seed)
    seen: set[bytes] = set()
    toks: list[bytes] = []

    def add(t: bytes) -> bool:
        if t in seen:
            return False
        seen.add(t)
        toks.append(t)
        return True

    if kind == "tiny":
        for b in range(0x20, 0x7F):
            add(bytes([b]))
        alpha = np.frombuffer(_TINY_ALPHABET, dtype=np.uint8)
        while len(toks) < V:
            n = int(rng.integers(2, 7))
            add(bytes(alpha[rng.integers(0, len(alpha), n)].tolist()))
    elif kind == "bpe":
        for b in range(256):
            add(bytes([b]))
        while len(toks) < V:
            n = int(rng.geometric(0.25))
            if n < 2 or n > 16:
                continue
            printable = rng.random(n) < 0.9
            pr = rng.integers(0x20, 0x7F, n)
            an = rng.integers(0, 256, n)
            add(bytes(np.where(printable, pr, an).astype(np.uint8).tolist()))
    else:
        raise ValueError(f"unknown vocab kind {kind!r}")
    if len(toks) < V:
        raise ValueError("vocabulary smaller than requested")
    return toks[:V]


def vocab_csr(tokens: list[bytes]) -> tuple[np.ndarray, np.ndarray]:
    """(bytes u8[total], off u32[V+1]) -- the CSR layout every consumer takes."""
    off = np.zeros(len(tokens) + 1, dtype=np.uint32)
    off[1:] = np.cumsum([len(t) for t in tokens], dtype=np.uint64).astype(np.uint32)
    data = np.frombuffer(b"".join(tokens), dtype=np.uint8).copy()
    return data, off
