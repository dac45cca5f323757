"""Arithmetic evaluator and forced-token tokeniser (oracle side).

labs.miniml.ai "Evaluator aware decoding": when ``</calc>`` closes, the engine
"evaluate[s] it locally: 17 * 23 + 91 = 482", then "tokenize[s]
<result>482</result> and inject[s] those tokens"; "Failures inject
<result_error>...</result_error> instead" ("A concrete prototype on
llama.cpp").  The page leaves the operator set and the failure cases open
("Why isn't this in production APIs yet?" lists float formatting, overflow and
division by zero as owner decisions); the reading taken here:

  expr    := term (('+' | '-') term)*
  term    := unary (('*' | '/') unary)*
  unary   := '-' unary | primary
  primary := NUMBER | '(' expr ')'
  NUMBER  := [0-9]+ ('.' [0-9]*)? | '.' [0-9]+
  spaces are skipped between tokens; evaluation is exact over the rationals.

Outcomes: an integer result -> its decimal text; otherwise an error code:
``parse`` (not in the language), ``div_zero``, ``non_integer`` (result is not
an integer), ``overflow`` (more than 64 decimal digits, or a span longer than
4096 bytes).  The whole span is lexed before it is parsed.

Forced tokenisation: greedy longest match over the vocabulary at each
position, lowest id among equal strings (every single byte is a token in the
workload vocabularies, so it always succeeds).
"""

from __future__ import annotations

from fractions import Fraction


class EvalError(Exception):
    def __init__(self, code: str):
        super().__init__(code)
        self.code = code


def _lex(span: bytes):
    toks = []
    i = 0
    n = len(span)
    while i < n:
        c = span[i]
        if c == 0x20:
            i += 1
        elif c in b'+-*/()':
            toks.append(chr(c))
            i += 1
        elif 0x30 <= c <= 0x39 or c == 0x2E:
            j = i
            while j < n and 0x30 <= span[j] <= 0x39:
                j += 1
            int_part = span[i:j]
            frac_part = b''
            if j < n and span[j] == 0x2E:
                k = j + 1
                while k < n and 0x30 <= span[k] <= 0x39:
                    k += 1
                frac_part = span[j + 1:k]
                j = k
                if not int_part and not frac_part:
                    raise EvalError('parse')
            elif not int_part:
                raise EvalError('parse')
            value = Fraction(int(int_part or b'0'))
            if frac_part:
                value += Fraction(int(frac_part), 10 ** len(frac_part))
            toks.append(value)
            i = j
        else:
            raise EvalError('parse')
    return toks


def evaluate(span: bytes) -> int:
    if len(span) > 4096:
        # evaluators stay time bounded (same page, "Where XGrammar-2 could take this")
        raise EvalError('overflow')
    toks = _lex(span)
    pos = 0

    def peek():
        return toks[pos] if pos < len(toks) else None

    def expr():
        nonlocal pos
        v = term()
        while peek() in ('+', '-'):
            op = toks[pos]
            pos += 1
            w = term()
            v = v + w if op == '+' else v - w
        return v

    def term():
        nonlocal pos
        v = unary()
        while peek() in ('*', '/'):
            op = toks[pos]
            pos += 1
            w = unary()
            if op == '*':
                v = v * w
            else:
                if w == 0:
                    raise EvalError('div_zero')
                v = v / w
        return v

    def unary():
        nonlocal pos
        if peek() == '-':
            pos += 1
            return -unary()
        return primary()

    def primary():
        nonlocal pos
        t = peek()
        if isinstance(t, Fraction):
            pos += 1
            return t
        if t == '(':
            pos += 1
            v = expr()
            if peek() != ')':
                raise EvalError('parse')
            pos += 1
            return v
        raise EvalError('parse')

    if not toks:
        raise EvalError('parse')
    v = expr()
    if pos != len(toks):
        raise EvalError('parse')
    if v.denominator != 1:
        raise EvalError('non_integer')
    if len(str(abs(v.numerator))) > 64:
        raise EvalError('overflow')
    return int(v.numerator)


def format_result(span: bytes | None, fmt: str) -> bytes:
    """Bytes the host forces after the span closes (no span found -> parse error).
    ``strop_tag`` evaluates a string operation (oracle.strops) and writes the
    result as ``calc_tag`` does."""
    try:
        if span is None:
            raise EvalError('parse')
        if fmt == 'strop_tag':
            from .strops import evaluate_strop
            value = evaluate_strop(span)
        else:
            value = str(evaluate(span)).encode('ascii')
        ok = True
    except EvalError as e:
        value = e.code.encode('ascii')
        ok = False
    if fmt in ('calc_tag', 'strop_tag'):
        return (b'<result>' + value + b'</result>') if ok else \
               (b'<result_error>' + value + b'</result_error>')
    if fmt == 'json_answer':
        return (b', "answer": ' + value + b'}') if ok else \
               (b', "answer": null, "error": "' + value + b'"}')
    raise ValueError(fmt)


def tokenize_greedy(text: bytes, tokens: list[bytes]) -> list[int]:
    lowest: dict[bytes, int] = {}
    for i, t in enumerate(tokens):
        lowest.setdefault(t, i)
    maxlen = max(len(t) for t in tokens)
    out = []
    i = 0
    while i < len(text):
        for L in range(min(maxlen, len(text) - i), 0, -1):
            tid = lowest.get(text[i:i + L])
            if tid is not None:
                out.append(tid)
                i += L
                break
        else:
            raise ValueError(f'byte {text[i]:#x} has no token')
    return out
