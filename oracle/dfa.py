"""Oracle automaton: regular-expression tree -> canonical minimal trimmed DFA.

Construction (deliberately unlike the product's NFA pipeline):
  1. Brzozowski derivatives.  The states are derivative expressions, kept in a
     normal form (associative concatenation, union/intersection as sets,
     symbol sets merged, nullable repetitions starting at 0).  Rules:
        d(empty) = d(eps) = empty;  d(S) = eps if a in S else empty
        d(rs) = d(r) s  |  (d(s) if r is nullable)
        d(r|s) = d(r)|d(s);   d(r&s) = d(r)&d(s)
        d(r{m,n}) = d(r) r{max(m-1,0), n-1}      (r not nullable, or m = 0)
     A state accepts iff its expression is nullable.  Derivatives are taken per
     class of the alphabet partition induced by the tree's symbol sets.
  2. Trimming: states from which no accepting state is reachable are removed;
     a transition into one becomes DEAD.
  3. Minimisation: for acyclic automata, classify states in order of height
     (equal languages <=> equal acceptance and equal successor blocks); for
     cyclic ones, Moore refinement of {accepting, non-accepting} by the blocks
     of each state's successors until stable.
  4. Canonical numbering: breadth-first from the start state, visiting symbols
     0..511 in order, numbering states on first discovery.  The minimal trimmed
     automaton is unique up to isomorphism, so this numbering is unique.

Result: ``next[s, a]`` (int32, -1 = DEAD) over the 512 symbols and
``accept[s]``; state 0 is the start state.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .grammar import NSYM, GrammarError, source_to_tree

DEAD = -1


class _Terms:
    def __init__(self):
        self.nodes: list[tuple] = []
        self.index: dict[tuple, int] = {}
        self.EMPTY = self._intern(('empty',))
        self.EPS = self._intern(('eps',))
        self._nullable: dict[int, bool] = {}
        self._deriv: dict[tuple[int, int], int] = {}

    def _intern(self, node) -> int:
        i = self.index.get(node)
        if i is None:
            i = len(self.nodes)
            self.nodes.append(node)
            self.index[node] = i
        return i

    # smart constructors (language-preserving normal form)
    def sym(self, mask: int) -> int:
        return self.EMPTY if mask == 0 else self._intern(('sym', mask))

    def cat(self, a: int, b: int) -> int:
        if a == self.EMPTY or b == self.EMPTY:
            return self.EMPTY
        if a == self.EPS:
            return b
        if b == self.EPS:
            return a
        na = self.nodes[a]
        if na[0] == 'cat':
            return self.cat(na[1], self.cat(na[2], b))
        return self._intern(('cat', a, b))

    def alt(self, items) -> int:
        flat: set[int] = set()
        mask = 0
        for i in items:
            n = self.nodes[i]
            if n[0] == 'alt':
                for j in n[1]:
                    nj = self.nodes[j]
                    if nj[0] == 'sym':
                        mask |= nj[1]
                    else:
                        flat.add(j)
            elif n[0] == 'sym':
                mask |= n[1]
            elif i != self.EMPTY:
                flat.add(i)
        if mask:
            flat.add(self.sym(mask))
        if not flat:
            return self.EMPTY
        if len(flat) == 1:
            return next(iter(flat))
        return self._intern(('alt', frozenset(flat)))

    def inter(self, items) -> int:
        flat: set[int] = set()
        mask = None
        for i in items:
            if i == self.EMPTY:
                return self.EMPTY
            n = self.nodes[i]
            members = n[1] if n[0] == 'and' else (i,)
            for j in members:
                nj = self.nodes[j]
                if nj[0] == 'sym':
                    mask = nj[1] if mask is None else (mask & nj[1])
                else:
                    flat.add(j)
        if mask is not None:
            if mask == 0:
                return self.EMPTY
            flat.add(self.sym(mask))
        if len(flat) == 1:
            return next(iter(flat))
        return self._intern(('and', frozenset(flat)))

    def rep(self, a: int, m: int, n) -> int:
        if n == 0:
            return self.EPS
        if a == self.EMPTY:
            return self.EPS if m == 0 else self.EMPTY
        if a == self.EPS:
            return self.EPS
        if m == 1 and n == 1:
            return a
        if self.nullable(a):
            m = 0
        return self._intern(('rep', a, m, n))

    def nullable(self, t: int) -> bool:
        r = self._nullable.get(t)
        if r is not None:
            return r
        n = self.nodes[t]
        k = n[0]
        if k == 'empty' or k == 'sym':
            r = False
        elif k == 'eps':
            r = True
        elif k == 'cat':
            r = self.nullable(n[1]) and self.nullable(n[2])
        elif k == 'alt':
            r = any(self.nullable(c) for c in n[1])
        elif k == 'and':
            r = all(self.nullable(c) for c in n[1])
        else:  # rep
            r = n[2] == 0 or self.nullable(n[1])
        self._nullable[t] = r
        return r

    def deriv(self, t: int, a: int) -> int:
        """Derivative of term t by symbol a."""
        key = (t, a)
        r = self._deriv.get(key)
        if r is not None:
            return r
        n = self.nodes[t]
        k = n[0]
        if k in ('empty', 'eps'):
            r = self.EMPTY
        elif k == 'sym':
            r = self.EPS if (n[1] >> a) & 1 else self.EMPTY
        elif k == 'cat':
            r = self.cat(self.deriv(n[1], a), n[2])
            if self.nullable(n[1]):
                r = self.alt([r, self.deriv(n[2], a)])
        elif k == 'alt':
            r = self.alt([self.deriv(c, a) for c in n[1]])
        elif k == 'and':
            r = self.inter([self.deriv(c, a) for c in n[1]])
        else:  # rep
            body, m, hi = n[1], n[2], n[3]
            rest = self.rep(body, max(m - 1, 0), None if hi is None else hi - 1)
            r = self.cat(self.deriv(body, a), rest)
        self._deriv[key] = r
        return r

    def from_tree(self, tree) -> int:
        k = tree[0]
        if k == 'empty':
            return self.EMPTY
        if k == 'eps':
            return self.EPS
        if k == 'sym':
            return self.sym(tree[1])
        if k == 'cat':
            out = self.EPS
            for c in reversed(tree[1]):
                out = self.cat(self.from_tree(c), out)
            return out
        if k == 'alt':
            return self.alt([self.from_tree(c) for c in tree[1]])
        if k == 'and':
            return self.inter([self.from_tree(c) for c in tree[1]])
        if k == 'rep':
            return self.rep(self.from_tree(tree[1]), tree[2], tree[3])
        raise ValueError(k)


def _symbol_classes(tree) -> np.ndarray:
    """Partition of the 512 symbols: two symbols share a class iff every symbol
    set of the tree contains both or neither.  Returns class id per symbol."""
    masks: set[int] = set()

    def walk(t):
        k = t[0]
        if k == 'sym':
            masks.add(t[1])
        elif k in ('cat', 'alt', 'and'):
            for c in t[1]:
                walk(c)
        elif k == 'rep':
            walk(t[1])
    walk(tree)
    sig = [tuple((m >> a) & 1 for m in sorted(masks)) for a in range(NSYM)]
    ids: dict[tuple, int] = {}
    cls = np.empty(NSYM, dtype=np.int64)
    for a in range(NSYM):
        cls[a] = ids.setdefault(sig[a], len(ids))
    return cls


def _row_ids(sig: np.ndarray) -> np.ndarray:
    """Id per row such that equal rows get equal ids (via a byte view of each row)."""
    sig = np.ascontiguousarray(sig, dtype=np.int64)
    view = sig.view(np.dtype((np.void, sig.dtype.itemsize * sig.shape[1]))).reshape(-1)
    _, inv = np.unique(view, return_inverse=True)
    return inv.reshape(-1)


def _heights(tr: np.ndarray):
    """Longest path to a state without successors; None if the graph has a cycle."""
    S = tr.shape[0]
    succ = [np.unique(tr[s][tr[s] >= 0]) for s in range(S)]
    preds: list[list[int]] = [[] for _ in range(S)]
    outdeg = np.zeros(S, dtype=np.int64)
    for s in range(S):
        outdeg[s] = len(succ[s])
        for d in succ[s]:
            preds[d].append(s)
    height = np.zeros(S, dtype=np.int64)
    stack = [s for s in range(S) if outdeg[s] == 0]
    done = 0
    while stack:
        s = stack.pop()
        done += 1
        for p in preds[s]:
            height[p] = max(height[p], height[s] + 1)
            outdeg[p] -= 1
            if outdeg[p] == 0:
                stack.append(p)
    return height if done == S else None


def _minimise(tr: np.ndarray, acc: np.ndarray) -> np.ndarray:
    """Block id per state; two states share a block iff their residual languages
    are equal.

    Acyclic automata: states are classified in order of height (longest path
    to a state without successors).  Equal languages have equal longest words,
    hence equal heights, and a state's language is fixed by its acceptance and
    its successors' languages, all of smaller height -- so equal (acceptance,
    successor blocks) signatures at one height are exactly the equal languages.
    Cyclic automata: Moore refinement of {accepting, non-accepting} by the
    successors' blocks until the number of blocks stops growing."""
    S = tr.shape[0]
    height = _heights(tr)
    block = np.full(S, -1, dtype=np.int64)
    if height is not None:
        nb = 0
        for h in range(int(height.max()) + 1):
            members = np.flatnonzero(height == h)
            succ = np.where(tr[members] >= 0, block[np.maximum(tr[members], 0)], -1)
            ids = _row_ids(np.concatenate([acc[members, None].astype(np.int64), succ], axis=1))
            block[members] = ids + nb
            nb += int(ids.max()) + 1
        return block
    block = acc.astype(np.int64)
    nblocks = len(np.unique(block))
    while True:
        succ = np.where(tr >= 0, block[np.maximum(tr, 0)], -1)
        block = _row_ids(np.concatenate([block[:, None], succ], axis=1))
        k = int(block.max()) + 1
        if k == nblocks:
            return block
        nblocks = k


@dataclass
class OracleDFA:
    next: np.ndarray      # int32 [S, 512], DEAD = -1
    accept: np.ndarray    # bool [S]

    @property
    def n_states(self) -> int:
        return self.next.shape[0]

    def sink(self) -> np.ndarray:
        """Accepting states with no outgoing transition (a finished generation)."""
        return self.accept & (self.next < 0).all(axis=1)

    def forced_only(self) -> np.ndarray:
        """States whose only continuations are host-injected bytes."""
        return (self.next[:, :256] < 0).all(axis=1) & (self.next[:, 256:] >= 0).any(axis=1)


def build_dfa(tree) -> OracleDFA:
    T = _Terms()
    root = T.from_tree(tree)
    cls = _symbol_classes(tree)
    ncls = int(cls.max()) + 1
    rep_sym = [int(np.flatnonzero(cls == c)[0]) for c in range(ncls)]

    # 1. derivative automaton over symbol classes
    state_of: dict[int, int] = {root: 0}
    terms = [root]
    trans: list[list[int]] = []
    i = 0
    while i < len(terms):
        t = terms[i]
        row = []
        for c in range(ncls):
            d = T.deriv(t, rep_sym[c])
            if d == T.EMPTY:
                row.append(DEAD)
            else:
                j = state_of.get(d)
                if j is None:
                    j = len(terms)
                    state_of[d] = j
                    terms.append(d)
                row.append(j)
        trans.append(row)
        i += 1
    tr = np.array(trans, dtype=np.int64).reshape(len(terms), ncls)
    acc = np.array([T.nullable(t) for t in terms], dtype=bool)

    # 2. trim: keep states that can reach an accepting state
    n = len(terms)
    preds: list[list[int]] = [[] for _ in range(n)]
    for s in range(n):
        for d in set(tr[s].tolist()):
            if d >= 0:
                preds[d].append(s)
    live = acc.copy()
    stack = list(np.flatnonzero(acc))
    while stack:
        s = stack.pop()
        for p in preds[s]:
            if not live[p]:
                live[p] = True
                stack.append(p)
    if not live[0]:
        raise GrammarError('empty', 'the grammar accepts no string')
    tr = np.where((tr >= 0) & live[np.maximum(tr, 0)], tr, DEAD)

    # 3. minimisation over live states
    keep = np.flatnonzero(live)
    remap = np.full(n, -1, dtype=np.int64)
    remap[keep] = np.arange(len(keep))
    tr = np.where(tr >= 0, remap[np.maximum(tr, 0)], DEAD)[keep]
    acc = acc[keep]
    block = _minimise(tr, acc)
    nblocks = int(block.max()) + 1

    # 4. canonical breadth-first numbering over symbols 0..511
    start_block = int(block[remap[0]])
    rep_state = np.zeros(nblocks, dtype=np.int64)
    rep_state[block] = np.arange(len(block))
    canon = {start_block: 0}
    order = [start_block]
    q = 0
    while q < len(order):
        b = order[q]
        s = rep_state[b]
        for a in range(NSYM):
            d = tr[s, cls[a]]
            if d >= 0:
                bd = int(block[d])
                if bd not in canon:
                    canon[bd] = len(order)
                    order.append(bd)
        q += 1
    S = len(order)
    nxt = np.full((S, NSYM), DEAD, dtype=np.int32)
    accept = np.zeros(S, dtype=bool)
    for b, cid in canon.items():
        s = rep_state[b]
        accept[cid] = acc[s]
        row = tr[s, cls]
        ok = row >= 0
        nxt[cid, ok] = [canon[int(block[d])] for d in row[ok]]
    return OracleDFA(nxt, accept)


def compile_grammar(kind: str, source: str, bounds) -> OracleDFA:
    return build_dfa(source_to_tree(kind, source, bounds))


def walk(dfa: OracleDFA, state: int, symbols) -> int:
    """Scalar walk; returns DEAD as soon as a symbol has no transition."""
    s = state
    for a in symbols:
        if s < 0:
            return DEAD
        s = int(dfa.next[s, a])
    return s


def is_acyclic(dfa: OracleDFA) -> bool:
    S = dfa.n_states
    indeg = np.zeros(S, dtype=np.int64)
    succ = [sorted(set(int(d) for d in dfa.next[s] if d >= 0)) for s in range(S)]
    for s in range(S):
        for d in succ[s]:
            indeg[d] += 1
    stack = [s for s in range(S) if indeg[s] == 0]
    seen = 0
    while stack:
        s = stack.pop()
        seen += 1
        for d in succ[s]:
            indeg[d] -= 1
            if indeg[d] == 0:
                stack.append(d)
    return seen == S
