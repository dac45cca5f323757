"""String-operation evaluator (oracle side; test infrastructure, never called by
the product path).

labs.miniml.ai "Evaluator aware decoding", "Not just arithmetic: string
operations": the span protocol that evaluates arithmetic handles any pure
function over a completed span; the page's example is
``<strop>count("strawberry", "r")</strop><result>3</result>`` and its registry
holds count, len, reverse, upper and substr.  The page fixes neither the span
syntax beyond that example nor the character model (its "Why isn't this in
production APIs yet?" section lists grapheme versus code point counting among
the open owner decisions).  The reading taken here:

  span   := sp NAME sp '(' sp arg (sp ',' sp arg)* sp ')' sp     (sp = spaces)
  arg    := STRING | INT
  STRING := '"' ( any byte but '"' and '\\' | '\\"' | '\\\\' )* '"'
  INT    := '-'? [0-9]{1,9}

  count(s, sub)   -> number of non-overlapping occurrences of sub in s, found
                     left to right (sub must not be empty)
  len(s)          -> number of bytes of s
  reverse(s)      -> the bytes of s in reverse order
  upper(s)        -> s with ASCII a-z raised to A-Z, other bytes unchanged
  substr(s, i, j) -> the slice s[i:j] with negative indices counted from the
                     end and both ends clamped to [0, len(s)] (empty if i >= j)

Strings are byte strings: the workload grammars keep them ASCII, where bytes,
code points and graphemes agree.  Integer results are written in decimal,
string results as their bytes.  Errors give a code: ``parse`` (not in the
span language), ``unknown_op``, ``arity`` (wrong number or kinds of
arguments), ``empty`` (count of an empty substring), ``overflow`` (a result
over 64 bytes or a span over 4096 bytes), ``bad_char`` (a result byte '<',
which would end the result tag).
"""

from __future__ import annotations

from .evaluator import EvalError

MAX_RESULT = 64


def _parse(span: bytes):
    i, n = 0, len(span)

    def skip():
        nonlocal i
        while i < n and span[i] == 0x20:
            i += 1

    skip()
    j = i
    while i < n and (0x61 <= span[i] <= 0x7A):   # a-z
        i += 1
    name = span[j:i]
    if not name:
        raise EvalError('parse')
    skip()
    if i >= n or span[i] != 0x28:                # (
        raise EvalError('parse')
    i += 1
    args = []
    while True:
        skip()
        if i < n and span[i] == 0x22:            # string literal
            i += 1
            buf = bytearray()
            while True:
                if i >= n:
                    raise EvalError('parse')
                c = span[i]
                if c == 0x22:
                    i += 1
                    break
                if c == 0x5C:                    # backslash escape
                    if i + 1 >= n or span[i + 1] not in (0x22, 0x5C):
                        raise EvalError('parse')
                    buf.append(span[i + 1])
                    i += 2
                    continue
                buf.append(c)
                i += 1
            args.append(bytes(buf))
        else:
            neg = i < n and span[i] == 0x2D
            k = i + 1 if neg else i
            d = k
            while d < n and 0x30 <= span[d] <= 0x39:
                d += 1
            if d == k or d - k > 9:
                raise EvalError('parse')
            v = 0
            for c in span[k:d]:
                v = v * 10 + (c - 0x30)
            args.append(-v if neg else v)
            i = d
        skip()
        if i < n and span[i] == 0x2C:            # ,
            i += 1
            continue
        if i < n and span[i] == 0x29:            # )
            i += 1
            break
        raise EvalError('parse')
    skip()
    if i != n:
        raise EvalError('parse')
    return name, args


def _count(s: bytes, sub: bytes) -> int:
    if not sub:
        raise EvalError('empty')
    c, i = 0, 0
    while i + len(sub) <= len(s):
        if s[i:i + len(sub)] == sub:
            c += 1
            i += len(sub)
        else:
            i += 1
    return c


def _upper(s: bytes) -> bytes:
    return bytes(c - 32 if 0x61 <= c <= 0x7A else c for c in s)


def _reverse(s: bytes) -> bytes:
    out = bytearray()
    for k in range(len(s) - 1, -1, -1):
        out.append(s[k])
    return bytes(out)


def _clamp_index(i: int, L: int) -> int:
    if i < 0:
        i += L
    return min(max(i, 0), L)


def _substr(s: bytes, i: int, j: int) -> bytes:
    a, b = _clamp_index(i, len(s)), _clamp_index(j, len(s))
    out = bytearray()
    for k in range(a, b):
        out.append(s[k])
    return bytes(out)


_KINDS = {b'count': (bytes, bytes), b'len': (bytes,), b'reverse': (bytes,), b'upper': (bytes,),
          b'substr': (bytes, int, int)}


def evaluate_strop(span: bytes) -> bytes:
    """The result's bytes (decimal text for integers), or EvalError(code)."""
    if len(span) > 4096:
        raise EvalError('overflow')
    name, args = _parse(span)
    kinds = _KINDS.get(name)
    if kinds is None:
        raise EvalError('unknown_op')
    if len(args) != len(kinds) or any(not isinstance(a, k) for a, k in zip(args, kinds)):
        raise EvalError('arity')
    if name == b'count':
        out = str(_count(args[0], args[1])).encode('ascii')
    elif name == b'len':
        out = str(len(args[0])).encode('ascii')
    elif name == b'reverse':
        out = _reverse(args[0])
    elif name == b'upper':
        out = _upper(args[0])
    else:
        out = _substr(args[0], args[1], args[2])
    if len(out) > MAX_RESULT:
        raise EvalError('overflow')
    if 0x3C in out:
        raise EvalError('bad_char')
    return out
