"""One decode step on the CPU: token mask, sampler, accept (oracle).

Mask (usetacet.com/docs/grammar, "The guarantee": the automaton masks the
logits at every step).  Token t is allowed in state s iff walking the bytes of
t, as model-written symbols, from s never reaches DEAD.  A state inside a
forced region has no model-symbol transitions, so a token can end on entering
one (the token that closes ``</calc>``) but never pass through one.  A row with
a host-forced token gets a mask holding exactly that token (labs.miniml.ai
"Evaluator aware decoding", "A concrete prototype on llama.cpp").

Sampler (it sees only masked logits: usetacet.com/docs/grammar, "The
guarantee"), per row,
in float64 on the exact logit values x:
  * no allowed token -> NO_TOKEN;
  * temperature 0 -> argmax x over allowed tokens, ties to the lowest id;
  * else z = x / T (T as the binary32 the kernel receives), m = max z,
    p = exp(z - m) / sum exp(z - m) over allowed tokens;
    top-p: sort allowed tokens by z descending, take the smallest prefix whose
    cumulative p reaches top_p, tau = z at its end, nucleus = {z >= tau}
    (ties at tau included); top_p >= 1 keeps every allowed token;
    Gumbel-max: tok = argmax over the nucleus of z + g, g = -log(-log u) with
    u from the Philox stream (oracle.philox), ties to the lowest id.
  Reported alongside: ``gap`` (best minus second-best Gumbel score in the
  nucleus) and ``margin`` (distance of top_p from the cumulative mass on
  either side of the chosen threshold) -- a faithful implementation may differ
  from this one only where one of them is below its rounding error.

Accept: walk the token's bytes from the row's state (as injected symbols when
the token was forced); flags DONE (accepting state without successors),
FORCED_NEXT (the new state continues only with injected bytes), REJECTED
(DEAD), NO_TOKEN (the row had no token).
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .dfa import DEAD, OracleDFA, walk
from .philox import gumbel, sampler_words, uniform_from_word

NO_TOKEN = 0xFFFFFFFF
FLAG_DONE = 1
FLAG_FORCED_NEXT = 2
FLAG_REJECTED = 4
FLAG_NO_TOKEN = 8


def token_allowed(dfa: OracleDFA, state: int, tok: bytes) -> bool:
    """The mask bit by its definition (scalar walk)."""
    return state >= 0 and walk(dfa, state, list(tok)) != DEAD


class VocabMatrix:
    """Tokens as a zero-padded byte matrix, for walking all tokens at once."""

    def __init__(self, tokens: list[bytes]):
        self.tokens = tokens
        self.V = len(tokens)
        self.lens = np.array([len(t) for t in tokens], dtype=np.int64)
        L = int(self.lens.max())
        self.mat = np.zeros((self.V, L), dtype=np.int64)
        for i, t in enumerate(tokens):
            self.mat[i, :len(t)] = np.frombuffer(t, dtype=np.uint8)


def token_mask(dfa: OracleDFA, vm: VocabMatrix, state: int) -> np.ndarray:
    """Mask of every token from ``state``: the walk of ``token_allowed`` applied
    to all tokens side by side, one byte position at a time."""
    alive = vm.lens > 0
    if state < 0:
        return np.zeros(vm.V, dtype=bool)
    st = np.full(vm.V, state, dtype=np.int64)
    for j in range(vm.mat.shape[1]):
        act = alive & (vm.lens > j)
        if not act.any():
            break
        nxt = dfa.next[st[act], vm.mat[act, j]]
        st[act] = np.maximum(nxt, 0)
        alive[np.flatnonzero(act)[nxt < 0]] = False
    return alive


def pack_bitmask(mask: np.ndarray) -> np.ndarray:
    """u32 words, bit (t & 31) of word (t >> 5) is token t; pad bits are zero."""
    V = mask.shape[0]
    W = (V + 31) // 32
    padded = np.zeros(W * 32, dtype=np.uint64)
    padded[:V] = mask.astype(np.uint64)
    weights = (np.uint64(1) << np.arange(32, dtype=np.uint64))
    return (padded.reshape(W, 32) * weights).sum(axis=1).astype(np.uint32)


def unpack_bitmask(words: np.ndarray, V: int) -> np.ndarray:
    w = np.asarray(words, dtype=np.uint64)
    bits = (w[:, None] >> np.arange(32, dtype=np.uint64)) & np.uint64(1)
    return bits.reshape(-1)[:V].astype(bool)


def onehot_mask(V: int, tok: int) -> np.ndarray:
    m = np.zeros(V, dtype=bool)
    m[tok] = True
    return m


@dataclass
class SampleResult:
    tok: int
    probs: np.ndarray     # float64 [V]
    gap: float            # best - second best Gumbel score (inf if unique)
    margin: float         # top-p threshold margin (inf when no truncation)
    nucleus_size: int


def sample_row(x: np.ndarray, allowed: np.ndarray, temp: float, top_p: float,
               seed: int, row: int, step: int) -> SampleResult:
    x = np.asarray(x, dtype=np.float64)
    V = x.shape[0]
    idx = np.flatnonzero(allowed)
    probs = np.zeros(V, dtype=np.float64)
    if idx.size == 0:
        return SampleResult(NO_TOKEN, probs, np.inf, np.inf, 0)
    xa = x[idx]
    if temp == 0.0:
        tok = int(idx[np.flatnonzero(xa == xa.max())[0]])
        probs[tok] = 1.0
        return SampleResult(tok, probs, np.inf, np.inf, 1)
    T = float(np.float32(temp))
    z = xa / T
    m = z.max()
    e = np.exp(z - m)
    p = e / e.sum()
    probs[idx] = p
    if float(np.float32(top_p)) >= 1.0:
        nuc = idx
        zn = z
        margin = np.inf
    else:
        tp = float(np.float32(top_p))
        vals, inv = np.unique(z, return_inverse=True)          # ascending distinct z
        mass = np.bincount(inv.reshape(-1), weights=p)[::-1]    # descending
        cum = np.cumsum(mass)
        hit = np.flatnonzero(cum >= tp)
        j = int(hit[0]) if hit.size else len(cum) - 1
        tau = vals[::-1][j]
        keep = z >= tau
        nuc = idx[keep]
        zn = z[keep]
        above = cum[j - 1] if j > 0 else 0.0
        margin = float(min(cum[j] - tp, tp - above))
    g = gumbel(uniform_from_word(sampler_words(nuc, row, step, seed)))
    score = zn + g
    best = score.max()
    tok = int(nuc[np.flatnonzero(score == best)[0]])
    if score.size > 1:
        second = np.partition(score, -2)[-2]
        gap = float(best - second)
    else:
        gap = np.inf
    return SampleResult(tok, probs, gap, margin, int(nuc.size))


def accept(dfa: OracleDFA, state: int, tok: int, tokens: list[bytes], forced: bool):
    """Returns (next state, flags)."""
    if tok == NO_TOKEN:
        return state, FLAG_NO_TOKEN
    data = tokens[tok]
    syms = [b + 256 for b in data] if forced else list(data)
    ns = walk(dfa, state, syms) if state >= 0 else DEAD
    if ns < 0:
        return DEAD, FLAG_REJECTED
    flags = 0
    if dfa.accept[ns] and (dfa.next[ns] < 0).all():
        flags |= FLAG_DONE
    if (dfa.next[ns, :256] < 0).all() and (dfa.next[ns, 256:] >= 0).any():
        flags |= FLAG_FORCED_NEXT
    return ns, flags


FLAG_CAPPED = 16
FLAG_DRAFT_CUT = 32


@dataclass
class DraftResult:
    n: int               # draft tokens accepted (a prefix of the draft)
    path: list[int]      # state before position 0 .. n (path[j + 1]: after draft token j)
    state: int           # the row's state afterwards (0 after DONE or CAPPED)
    flags: int
    count: int | None    # token count afterwards (when counts are kept)


def state_flags(dfa: OracleDFA, s: int) -> int:
    """DONE / FORCED_NEXT of a live state, as ``accept`` reports them."""
    flags = 0
    if dfa.accept[s] and (dfa.next[s] < 0).all():
        flags |= FLAG_DONE
    if (dfa.next[s, :256] < 0).all() and (dfa.next[s, 256:] >= 0).any():
        flags |= FLAG_FORCED_NEXT
    return flags


def accept_many(dfa: OracleDFA, state: int, draft: list[int], tokens: list[bytes],
                forced: list[int] | None = None, count: int | None = None,
                max_tokens: int | None = None) -> DraftResult:
    """Speculative verification of a draft against the grammar
    (labs.miniml.ai "Evaluator aware decoding", "Where XGrammar-2 could take
    this": once a draft token ends an evaluated span, the evaluator's result
    fixes the tokens after it, so checking them is a comparison of ids).

    Token j of the draft is accepted when ``accept`` of it from the state left
    by tokens 0..j-1 does not reach DEAD; where ``forced[j] >= 0`` the host has
    pinned position j, so the token must equal that id and is walked as
    injected bytes.  Verification stops at the first refused token (flag
    DRAFT_CUT; the state stays that of the accepted prefix), after a token that
    ends the grammar (DONE), when the token count reaches max_tokens (CAPPED),
    or after a token whose state continues only with injected bytes when
    position j+1 is not pinned (the host has to evaluate the span first).
    The flags also carry DONE / FORCED_NEXT of the final state.  When token
    counts are kept (``count`` given), a row whose accepted tokens end it
    (DONE) or reach the cap restarts from state 0 with count 0, as the device
    accept does with counts.  An empty draft reports NO_TOKEN; a DEAD row
    accepts nothing (REJECTED)."""
    forced = forced if forced is not None else [-1] * len(draft)
    path = [state]
    if not draft:
        return DraftResult(0, path, state, FLAG_NO_TOKEN, count)
    if state < 0:
        return DraftResult(0, path, state, FLAG_REJECTED, count)
    s, n, cut, capped, c = state, 0, 0, 0, count
    for j, t in enumerate(draft):
        f = forced[j]
        ns = DEAD if (f >= 0 and t != f) else accept(dfa, s, t, tokens, f >= 0)[0]
        if ns == DEAD:
            cut = FLAG_DRAFT_CUT
            break
        s, n = ns, n + 1
        path.append(s)
        if c is not None:
            c += 1
        if state_flags(dfa, s) & FLAG_DONE:
            break
        if c is not None and c >= max_tokens:
            capped = FLAG_CAPPED
            break
        if state_flags(dfa, s) & FLAG_FORCED_NEXT and not (j + 1 < len(draft) and forced[j + 1] >= 0):
            break
    flags = state_flags(dfa, s) | cut | capped
    if c is not None and n > 0 and flags & (FLAG_DONE | FLAG_CAPPED):
        s, c = 0, 0
    return DraftResult(n, path, s, flags, c)
