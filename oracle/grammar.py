r"""Grammar front-ends of the oracle: source text -> regular-expression tree.

Alphabet: 512 symbols.  Symbol b in 0..255 is byte b written by the model;
symbol 256 + b is byte b injected by the host (a forced token).  Injected
bytes are a separate alphabet so that two rules of labs.miniml.ai "Evaluator
aware decoding" ("A concrete prototype on llama.cpp", item 2) -- the model
never writes the result block itself, and the automaton moves forward over the
injected result -- are plain automaton structure: a state inside a forced
region has transitions on injected symbols only.

Tree nodes are tuples:
  ('empty',)            the empty language
  ('eps',)              the empty string
  ('sym', mask)         one symbol out of the set ``mask`` (a 512-bit int)
  ('cat', (a, b, ...))  concatenation
  ('alt', (a, b, ...))  union
  ('and', (a, b, ...))  intersection
  ('rep', a, m, n)      m..n copies of a (n None = unbounded)

GBNF-style rule language (one reading of the pages' GBNF grammar, labs.miniml.ai
"This is a grammar problem"; the pages call the automaton a pushdown automaton,
read here as bounded nesting so that it stays finite, usetacet.com/docs/grammar
"The guarantee"):
  rule     NAME ::= alt            (a rule starts at every ``NAME ::=``)
  alt      inter ('|' inter)*
  inter    seq ('&' seq)*
  seq      post*
  post     atom ('?' | '*' | '+' | '{m}' | '{m,}' | '{m,n}')*
  atom     "literal" | [class] | NAME | ( alt ) | @forced( alt )
Escapes in literals and classes: \\ \" \] \[ \- \^ \n \r \t \xHH.  ``#``
comments run to end of line.  The start rule is ``root``.  References are
expanded by inlining; a rule may be active at most ``depth_max`` times on the
expansion stack, and a reference beyond that denotes the empty language.  The
pushdown reading (``gbnf_to_tree(..., nesting='stack')``) bounds instead the
number of frames of recursive rules open at once, the stack of the device's
pushdown automaton; under either bound the language is regular, so the
derivative construction of oracle.dfa builds its automaton.

JSON-schema subset: see ``schema_to_tree``.
"""

from __future__ import annotations

import json

NSYM = 512
ALL_BYTES = (1 << 256) - 1


class GrammarError(Exception):
    def __init__(self, code: str, msg: str):
        super().__init__(f"{code}: {msg}")
        self.code = code


EMPTY = ('empty',)
EPS = ('eps',)


def sym_of(byte_values) -> tuple:
    mask = 0
    for b in byte_values:
        mask |= 1 << b
    return ('sym', mask)


def lit(data: bytes) -> tuple:
    if not data:
        return EPS
    if len(data) == 1:
        return sym_of([data[0]])
    return ('cat', tuple(sym_of([b]) for b in data))


def rng(lo: int, hi: int) -> tuple:
    return sym_of(range(lo, hi + 1))


def cat(*xs) -> tuple:
    return ('cat', tuple(xs)) if len(xs) != 1 else xs[0]


def alt(*xs) -> tuple:
    return ('alt', tuple(xs)) if len(xs) != 1 else xs[0]


def rep(x, m, n) -> tuple:
    return ('rep', x, m, n)


def forced(tree) -> tuple:
    """Move every model byte of ``tree`` to the injected-byte half of the alphabet."""
    kind = tree[0]
    if kind == 'sym':
        mask = tree[1]
        return ('sym', ((mask & ALL_BYTES) << 256) | (mask & (ALL_BYTES << 256)))
    if kind in ('cat', 'alt', 'and'):
        return (kind, tuple(forced(c) for c in tree[1]))
    if kind == 'rep':
        return ('rep', forced(tree[1]), tree[2], tree[3])
    return tree


# ----------------------------------------------------------------------------
# GBNF-style rules
# ----------------------------------------------------------------------------

_ESC = {ord('n'): 0x0A, ord('r'): 0x0D, ord('t'): 0x09}


def _tokenize(src: bytes):
    toks = []
    i, n = 0, len(src)

    def hexval(j):
        h = src[j:j + 2]
        try:
            return int(h.decode('ascii'), 16)
        except (ValueError, UnicodeDecodeError):
            raise GrammarError('syntax', f'bad \\x escape at byte {j}')

    def escape(j):
        # src[j] == backslash; returns (byte value, next index)
        if j + 1 >= n:
            raise GrammarError('syntax', 'dangling backslash')
        c = src[j + 1]
        if c == ord('x'):
            if j + 4 > n:
                raise GrammarError('syntax', 'short \\x escape')
            return hexval(j + 2), j + 4
        if c in _ESC:
            return _ESC[c], j + 2
        return c, j + 2

    while i < n:
        c = src[i]
        if c in b' \t\r\n':
            i += 1
        elif c == ord('#'):
            while i < n and src[i] != 0x0A:
                i += 1
        elif c == ord('"'):
            j = i + 1
            out = bytearray()
            while True:
                if j >= n:
                    raise GrammarError('syntax', 'unterminated literal')
                if src[j] == ord('"'):
                    j += 1
                    break
                if src[j] == ord('\\'):
                    v, j = escape(j)
                    out.append(v)
                else:
                    out.append(src[j])
                    j += 1
            toks.append(('lit', bytes(out)))
            i = j
        elif c == ord('['):
            j = i + 1
            neg = False
            if j < n and src[j] == ord('^'):
                neg = True
                j += 1
            items = []  # list of (value, is_escaped)
            while True:
                if j >= n:
                    raise GrammarError('syntax', 'unterminated class')
                if src[j] == ord(']'):
                    j += 1
                    break
                if src[j] == ord('\\'):
                    v, j = escape(j)
                    items.append((v, True))
                else:
                    items.append((src[j], False))
                    j += 1
            chars = set()
            k = 0
            while k < len(items):
                v, _ = items[k]
                is_range = (k + 2 < len(items) and items[k + 1] == (ord('-'), False))
                if is_range:
                    hi = items[k + 2][0]
                    if hi < v:
                        raise GrammarError('syntax', 'reversed class range')
                    chars.update(range(v, hi + 1))
                    k += 3
                else:
                    chars.add(v)
                    k += 1
            if neg:
                chars = set(range(256)) - chars
            toks.append(('set', sym_of(sorted(chars))))
            i = j
        elif src.startswith(b'::=', i):
            toks.append(('def', None))
            i += 3
        elif src.startswith(b'@forced', i):
            toks.append(('forced', None))
            i += 7
        elif c in b'()|&?*+':
            toks.append((chr(c), None))
            i += 1
        elif c == ord('{'):
            j = src.find(b'}', i)
            if j < 0:
                raise GrammarError('syntax', 'unterminated repetition')
            body = src[i + 1:j].decode('ascii', 'replace').replace(' ', '')
            parts = body.split(',')
            try:
                if len(parts) == 1:
                    m = nn = int(parts[0])
                elif len(parts) == 2:
                    m = int(parts[0])
                    nn = None if parts[1] == '' else int(parts[1])
                else:
                    raise ValueError
            except ValueError:
                raise GrammarError('syntax', f'bad repetition {{{body}}}')
            if m < 0 or (nn is not None and nn < m):
                raise GrammarError('syntax', f'bad repetition bounds {{{body}}}')
            toks.append(('repeat', (m, nn)))
            i = j + 1
        elif c == ord('_') or (c < 0x80 and chr(c).isalpha()):
            j = i
            while j < n and (src[j] in b'_-' or (src[j] < 0x80 and chr(src[j]).isalnum())):
                j += 1
            toks.append(('name', src[i:j].decode('ascii')))
            i = j
        else:
            raise GrammarError('syntax', f'unexpected byte {c:#x} at {i}')
    return toks


class _Parser:
    def __init__(self, toks):
        self.t = toks
        self.i = 0

    def peek(self, k=0):
        j = self.i + k
        return self.t[j] if j < len(self.t) else ('eof', None)

    def at_rule_start(self):
        return self.peek()[0] == 'name' and self.peek(1)[0] == 'def'

    def rules(self):
        out = {}
        while self.peek()[0] != 'eof':
            if not self.at_rule_start():
                raise GrammarError('syntax', 'expected "name ::="')
            name = self.peek()[1]
            self.i += 2
            if name in out:
                raise GrammarError('syntax', f'rule {name} defined twice')
            out[name] = self.alt()
        return out

    def alt(self):
        xs = [self.inter()]
        while self.peek()[0] == '|':
            self.i += 1
            xs.append(self.inter())
        return xs[0] if len(xs) == 1 else ('alt', tuple(xs))

    def inter(self):
        xs = [self.seq()]
        while self.peek()[0] == '&':
            self.i += 1
            xs.append(self.seq())
        return xs[0] if len(xs) == 1 else ('and', tuple(xs))

    def seq(self):
        xs = []
        while True:
            k = self.peek()[0]
            if k in ('|', '&', ')', 'eof') or self.at_rule_start():
                break
            xs.append(self.post())
        if not xs:
            return EPS
        return xs[0] if len(xs) == 1 else ('cat', tuple(xs))

    def post(self):
        x = self.atom()
        while True:
            k, v = self.peek()
            if k == '?':
                x = ('rep', x, 0, 1)
            elif k == '*':
                x = ('rep', x, 0, None)
            elif k == '+':
                x = ('rep', x, 1, None)
            elif k == 'repeat':
                x = ('rep', x, v[0], v[1])
            else:
                return x
            self.i += 1

    def atom(self):
        k, v = self.peek()
        self.i += 1
        if k == 'lit':
            return lit(v)
        if k == 'set':
            return v
        if k == 'name':
            return ('ref', v)
        if k == '(':
            x = self.alt()
            if self.peek()[0] != ')':
                raise GrammarError('syntax', 'expected )')
            self.i += 1
            return x
        if k == 'forced':
            if self.peek()[0] != '(':
                raise GrammarError('syntax', 'expected ( after @forced')
            self.i += 1
            x = self.alt()
            if self.peek()[0] != ')':
                raise GrammarError('syntax', 'expected )')
            self.i += 1
            return ('forced', x)
        raise GrammarError('syntax', f'unexpected token {k}')


def gbnf_rules(src: str | bytes) -> dict:
    """Rule name -> rule body (with ('ref', NAME) nodes), as parsed."""
    if isinstance(src, str):
        src = src.encode('utf-8')
    rules = _Parser(_tokenize(src)).rules()
    if 'root' not in rules:
        raise GrammarError('syntax', 'no root rule')
    return rules


def _refs(node, out: set) -> set:
    if node[0] == 'ref':
        out.add(node[1])
    elif node[0] in ('cat', 'alt', 'and'):
        for c in node[1]:
            _refs(c, out)
    elif node[0] in ('rep', 'forced'):
        _refs(node[1], out)
    return out


def recursive_rules(rules: dict) -> set:
    """Rules that can reach themselves through references (a rule on a cycle of
    the reference graph), by a search from each rule."""
    succ = {name: _refs(body, set()) for name, body in rules.items()}
    for name, ss in succ.items():
        for r in ss:
            if r not in rules:
                raise GrammarError('undefined_rule', r)
    out = set()
    for name in rules:
        seen, stack = set(), list(succ[name])
        while stack:
            r = stack.pop()
            if r == name:
                out.add(name)
                break
            if r not in seen:
                seen.add(r)
                stack.extend(succ[r])
    return out


def gbnf_to_tree(src: str | bytes, depth_max: int, nesting: str = 'per_rule') -> tuple:
    """Expand the rules from ``root`` into one tree.

    nesting='per_rule': a rule may be active at most ``depth_max`` times on the
    expansion stack (the bound of every GBNF grammar in the workloads).
    nesting='stack': the bound of a pushdown automaton whose stack holds at most
    ``depth_max`` frames -- every reference to a recursive rule (one on a cycle
    of the reference graph) opens a frame, references to other rules are plain
    inlining, and a reference that would open frame depth_max + 1 denotes the
    empty language.  The start rule is the base and opens no frame."""
    rules = gbnf_rules(src)
    if nesting not in ('per_rule', 'stack'):
        raise ValueError(nesting)
    rec = recursive_rules(rules) if nesting == 'stack' else set()
    active: dict[str, int] = {}
    frames = [0]

    def expand(node):
        kind = node[0]
        if kind == 'ref':
            name = node[1]
            if name not in rules:
                raise GrammarError('undefined_rule', name)
            if nesting == 'stack':
                if name not in rec:
                    return expand(rules[name])
                if frames[0] >= depth_max:
                    return EMPTY
                frames[0] += 1
                body = expand(rules[name])
                frames[0] -= 1
                return body
            if active.get(name, 0) >= depth_max:
                return EMPTY
            active[name] = active.get(name, 0) + 1
            body = expand(rules[name])
            active[name] -= 1
            return body
        if kind == 'forced':
            return forced(expand(node[1]))
        if kind in ('cat', 'alt', 'and'):
            return (kind, tuple(expand(c) for c in node[1]))
        if kind == 'rep':
            return ('rep', expand(node[1]), node[2], node[3])
        return node

    if nesting == 'stack':
        return expand(rules['root'])
    return expand(('ref', 'root'))


# ----------------------------------------------------------------------------
# JSON-schema subset
# ----------------------------------------------------------------------------

_IGNORED = {"title", "description", "$schema", "$id", "$comment", "default", "examples"}
_KNOWN = {"type", "properties", "required", "additionalProperties", "enum", "const",
          "anyOf", "items", "minItems", "maxItems", "minLength", "maxLength", "x-maxBytes"}

_HEX = sym_of(b'0123456789abcdefABCDEF')
_DIGIT = rng(0x30, 0x39)
_DIGIT19 = rng(0x31, 0x39)
_CONT = rng(0x80, 0xBF)


def _json_char() -> tuple:
    """One JSON string character: a well-formed UTF-8 scalar other than '"', '\\'
    and controls below 0x20, or an escape (each escape is one character)."""
    plain = sym_of([b for b in range(0x20, 0x80) if b not in (0x22, 0x5C)])
    utf8 = alt(
        plain,
        cat(rng(0xC2, 0xDF), _CONT),
        cat(sym_of([0xE0]), rng(0xA0, 0xBF), _CONT),
        cat(sym_of(list(range(0xE1, 0xED)) + [0xEE, 0xEF]), _CONT, _CONT),
        cat(sym_of([0xED]), rng(0x80, 0x9F), _CONT),
        cat(sym_of([0xF0]), rng(0x90, 0xBF), _CONT, _CONT),
        cat(rng(0xF1, 0xF3), _CONT, _CONT, _CONT),
        cat(sym_of([0xF4]), rng(0x80, 0x8F), _CONT, _CONT),
    )
    esc = cat(sym_of([0x5C]), alt(sym_of(b'"\\/bfnrt'), cat(sym_of(b'u'), _HEX, _HEX, _HEX, _HEX)))
    return alt(utf8, esc)


def _json_string_literal(s: str) -> bytes:
    out = bytearray(b'"')
    for ch in s.encode('utf-8'):
        if ch == 0x22:
            out += b'\\"'
        elif ch == 0x5C:
            out += b'\\\\'
        elif ch < 0x20:
            out += b'\\u%04x' % ch
        else:
            out.append(ch)
    out += b'"'
    return bytes(out)


def _json_value_literal(v) -> bytes:
    if v is None:
        return b'null'
    if v is True:
        return b'true'
    if v is False:
        return b'false'
    if isinstance(v, int):
        return str(v).encode('ascii')
    if isinstance(v, str):
        return _json_string_literal(v)
    raise GrammarError('unsupported', f'enum/const value of type {type(v).__name__}')


def _count(v, what: str) -> int:
    """A length/count keyword: a non-negative integral JSON number (<= 10**7)."""
    if isinstance(v, bool) or not isinstance(v, (int, float)) or v != int(v) or not 0 <= v <= 10**7:
        raise GrammarError('unsupported', f'{what} out of range')
    return int(v)


def schema_to_tree(text: str, ws_max: int, max_len_default: int, max_items_default: int) -> tuple:
    r"""Lower a JSON-schema subset to a tree.

    WS = [ \t\n\r]{0,ws_max} sits between structural tokens only: after '{'
    and '[', around ':' and ',', before '}' and ']'; never before the root value
    nor after it.  Constructs:
      object  "{" WS ( "\\"k1\\"" WS ":" WS v1 ( WS "," WS "\\"k\\"" WS ":" WS v )* )? WS "}"
              -- properties in declared order, every property required,
                 additionalProperties false or absent (absent is read as false)
      string  '"' CHAR{minLength,maxLength} '"'  (maxLength default max_len_default;
              with x-maxBytes and no maxLength: CHAR* limited to x-maxBytes bytes)
      integer -?(0|[1-9][0-9]{0,18})
      number  -?(0|[1-9][0-9]{0,15})(\\.[0-9]{1,16})?([eE][+-]?[0-9]{1,3})?
      boolean true|false;  null null;  enum/const: alternation of JSON literals
      array   "[" WS ( "]" | v ( WS "," WS v ){0,max-1} WS "]" )   (minItems 0)
              "[" WS v ( WS "," WS v ){min-1,max-1} WS "]"          (minItems >= 1)
      anyOf / type list: union
    Any other keyword fails closed (dev.to "I found a runner bug...", "What
    exists beyond the experiment": typed fail-closed refusals)."""
    try:
        schema = json.loads(text)
    except json.JSONDecodeError as e:
        raise GrammarError('syntax', f'schema is not JSON: {e}')
    ws = rep(sym_of(b' \t\n\r'), 0, ws_max)
    char = _json_char()

    def lower(s) -> tuple:
        if s is True or s == {}:
            raise GrammarError('unsupported', 'unconstrained value')
        if not isinstance(s, dict):
            raise GrammarError('unsupported', 'schema must be an object')
        for k in s:
            if k not in _KNOWN and k not in _IGNORED:
                raise GrammarError('unsupported', f'keyword {k}')
        if 'anyOf' in s:
            others = [k for k in s if k not in _IGNORED and k != 'anyOf']
            if others:
                raise GrammarError('unsupported', 'anyOf with sibling keywords')
            if not s['anyOf']:
                raise GrammarError('unsupported', 'empty anyOf')
            return alt(*[lower(b) for b in s['anyOf']])
        if 'enum' in s or 'const' in s:
            vals = s['enum'] if 'enum' in s else [s['const']]
            if not vals:
                raise GrammarError('unsupported', 'empty enum')
            ty = s.get('type')
            if ty is not None and not isinstance(ty, str):
                raise GrammarError('unsupported', 'enum value does not match type')
            for v in vals:
                if isinstance(v, float):
                    raise GrammarError('unsupported', 'non-integer number in enum')
                if ty is not None:
                    ok = {'string': isinstance(v, str), 'integer': isinstance(v, int) and not isinstance(v, bool),
                          'boolean': isinstance(v, bool), 'null': v is None}.get(ty)
                    if not ok:
                        raise GrammarError('unsupported', 'enum value does not match type')
            # duplicate literals collapse; order is irrelevant to the language
            return alt(*[lit(_json_value_literal(v)) for v in vals])
        ty = s.get('type')
        if isinstance(ty, list):
            if not ty:
                raise GrammarError('unsupported', 'empty type list')
            return alt(*[lower({**s, 'type': t}) for t in ty])
        if ty == 'object':
            props = s.get('properties', {})
            req = s.get('required', [])
            if sorted(req) != sorted(props.keys()) or len(set(req)) != len(req):
                raise GrammarError('unsupported', 'optional properties')
            if s.get('additionalProperties', False) is not False:
                raise GrammarError('unsupported', 'additionalProperties')
            if not props:
                return cat(lit(b'{'), ws, lit(b'}'))
            parts = [lit(b'{'), ws]
            for i, (k, v) in enumerate(props.items()):
                if i:
                    parts += [ws, lit(b','), ws]
                parts += [lit(_json_string_literal(k)), ws, lit(b':'), ws, lower(v)]
            parts += [ws, lit(b'}')]
            return cat(*parts)
        if ty == 'string':
            lo = _count(s.get('minLength', 0), 'minLength')
            if 'maxLength' in s:
                hi = _count(s['maxLength'], 'maxLength')
            elif 'x-maxBytes' in s:
                hi = None
            else:
                hi = max_len_default
            if hi is not None and hi < lo:
                raise GrammarError('unsupported', 'maxLength < minLength')
            body = rep(char, lo, hi)
            if 'x-maxBytes' in s:
                body = ('and', (body, rep(sym_of(range(256)), 0, _count(s['x-maxBytes'], 'x-maxBytes'))))
            return cat(lit(b'"'), body, lit(b'"'))
        if ty == 'integer':
            return cat(rep(lit(b'-'), 0, 1), alt(lit(b'0'), cat(_DIGIT19, rep(_DIGIT, 0, 18))))
        if ty == 'number':
            return cat(rep(lit(b'-'), 0, 1), alt(lit(b'0'), cat(_DIGIT19, rep(_DIGIT, 0, 15))),
                       rep(cat(lit(b'.'), rep(_DIGIT, 1, 16)), 0, 1),
                       rep(cat(sym_of(b'eE'), rep(sym_of(b'+-'), 0, 1), rep(_DIGIT, 1, 3)), 0, 1))
        if ty == 'boolean':
            return alt(lit(b'true'), lit(b'false'))
        if ty == 'null':
            return lit(b'null')
        if ty == 'array':
            if 'items' not in s:
                raise GrammarError('unsupported', 'array without items')
            item = lower(s['items'])
            lo = _count(s.get('minItems', 0), 'minItems')
            hi = _count(s.get('maxItems', max_items_default), 'maxItems')
            if hi < lo:
                raise GrammarError('unsupported', 'maxItems < minItems')
            more = cat(ws, lit(b','), ws, item)
            if hi == 0:
                return cat(lit(b'['), ws, lit(b']'))
            if lo == 0:
                return cat(lit(b'['), ws, alt(lit(b']'), cat(item, rep(more, 0, hi - 1), ws, lit(b']'))))
            return cat(lit(b'['), ws, item, rep(more, lo - 1, hi - 1), ws, lit(b']'))
        raise GrammarError('unsupported', f'type {ty!r}')

    return lower(schema)


def source_to_tree(kind: str, source: str, bounds) -> tuple:
    if kind == 'gbnf':
        return gbnf_to_tree(source, bounds.depth_max)
    if kind == 'json':
        return schema_to_tree(source, bounds.ws_max, bounds.max_len_default, bounds.max_items_default)
    if kind == 'structtag':
        return structtag_to_tree(source, bounds.ws_max, bounds.max_len_default, bounds.max_items_default)
    raise GrammarError('syntax', f'unknown grammar kind {kind}')


# ----------------------------------------------------------------------------
# Structural tags
# ----------------------------------------------------------------------------
#
# labs.miniml.ai "Evaluator aware decoding", "Where XGrammar-2 could take
# this": a Structural Tag is a JSON description whose atomic types (JSON
# schema, regex, literal strings) nest, and an evaluated tag is a tag
# (begin, content, end) whose completed content goes to a registered evaluator
# with the result forced into a sibling span.  The page sketches one element
# only; the reading taken here:
#   {"type": "literal", "text": S}
#   {"type": "regex", "pattern": P}          P in the subset of regex_to_tree, its
#                                            match at most max_len_default bytes
#   {"type": "json_schema", "json_schema": J}   the JSON-schema subset above
#   {"type": "sequence", "elements": [E...]} {"type": "or", "elements": [E...]}
#   {"type": "tag", "begin": S, "content": E, "end": S}
#   {"type": "evaluated_tag", "begin": S, "content": E, "end": S,
#    "evaluator": "arithmetic" | "string",
#    "result": {"begin": "<result>", "end": "</result>"}}
# An evaluated tag is followed by a forced region: <result>V</result> (V an
# optional minus and 1..64 digits for arithmetic, 0..64 bytes other than '<'
# for string operations) or <result_error>[a-z_]{1,32}</result_error>, the
# forms the host injects.  Unknown types or keys, other result tags and empty
# alternatives fail closed.

_RE_SPECIAL = set(b'()[]{}|*+?.\\^$')
_RE_CLASS_ESC = {ord('d'): b'0123456789',
                 ord('w'): b'abcdefghijklmnopqrstuvwxyzABCDEFGHIJKLMNOPQRSTUVWXYZ0123456789_',
                 ord('s'): b' \t\n\r\x0b\x0c'}
_RE_CHAR_ESC = {ord('n'): 0x0A, ord('t'): 0x09, ord('r'): 0x0D, ord('f'): 0x0C, ord('v'): 0x0B}


def regex_to_tree(pattern: str) -> tuple:
    """Regex subset over model bytes: literals, '.', classes [..] with ranges and
    '^', escapes (\\d \\w \\s \\n \\t \\r \\f \\v and escaped punctuation), groups,
    '|', and the postfix operators * + ? {m} {m,} {m,n}.  '.' is any byte but
    a newline.  Anchors, backreferences, lookarounds and non-ASCII characters
    inside classes fail closed."""
    src = pattern.encode('utf-8')
    pos = [0]

    def peek():
        return src[pos[0]] if pos[0] < len(src) else None

    def take():
        c = peek()
        if c is None:
            raise GrammarError('syntax', 'regex: unexpected end')
        pos[0] += 1
        return c

    def escape_atom():
        c = take()
        if c in _RE_CLASS_ESC:
            return sym_of(_RE_CLASS_ESC[c])
        if c in _RE_CHAR_ESC:
            return sym_of([_RE_CHAR_ESC[c]])
        if c in _RE_SPECIAL or c in b'-/"\'':
            return sym_of([c])
        raise GrammarError('unsupported', f'regex escape \\{chr(c)}')

    def class_atom():
        neg = False
        if peek() == ord('^'):
            take()
            neg = True
        members = set()
        first = True
        while True:
            c = take()
            if c == ord(']') and not first:
                break
            first = False
            if c == ord('\\'):
                e = take()
                if e in _RE_CLASS_ESC:
                    members |= set(_RE_CLASS_ESC[e])
                    continue
                lo = _RE_CHAR_ESC.get(e, e)
            else:
                lo = c
            if lo >= 0x80:
                raise GrammarError('unsupported', 'regex: non-ASCII in a class')
            if peek() == ord('-') and pos[0] + 1 < len(src) and src[pos[0] + 1] != ord(']'):
                take()
                h = take()
                if h == ord('\\'):
                    h = take()
                    h = _RE_CHAR_ESC.get(h, h)
                if h >= 0x80 or h < lo:
                    raise GrammarError('syntax', 'regex: bad class range')
                members |= set(range(lo, h + 1))
            else:
                members.add(lo)
        if neg:
            members = set(range(256)) - members
        return sym_of(members)

    def atom():
        c = take()
        if c == ord('('):
            if peek() == ord('?'):
                raise GrammarError('unsupported', 'regex: group flags')
            x = alternation()
            if take() != ord(')'):
                raise GrammarError('syntax', 'regex: unbalanced (')
            return x
        if c == ord('['):
            return class_atom()
        if c == ord('.'):
            return sym_of(b for b in range(256) if b != 0x0A)
        if c == ord('\\'):
            return escape_atom()
        if c in b'^$':
            raise GrammarError('unsupported', 'regex: anchors')
        if c in b')|*+?{}]':
            raise GrammarError('syntax', f'regex: unexpected {chr(c)}')
        return sym_of([c])

    def postfix():
        x = atom()
        while True:
            c = peek()
            if c == ord('*'):
                take()
                x = rep(x, 0, None)
            elif c == ord('+'):
                take()
                x = rep(x, 1, None)
            elif c == ord('?'):
                take()
                x = rep(x, 0, 1)
            elif c == ord('{'):
                take()
                body = bytearray()
                while peek() is not None and peek() != ord('}'):
                    body.append(take())
                take()
                parts = body.decode('ascii').split(',')
                try:
                    m = int(parts[0])
                    n = m if len(parts) == 1 else (None if parts[1] == '' else int(parts[1]))
                except ValueError:
                    raise GrammarError('syntax', 'regex: bad {m,n}') from None
                if len(parts) > 2 or m < 0 or (n is not None and n < m):
                    raise GrammarError('syntax', 'regex: bad {m,n}')
                x = rep(x, m, n)
            else:
                return x

    def sequence():
        items = []
        while peek() is not None and peek() not in b'|)':
            items.append(postfix())
        if not items:
            return EPS
        return cat(*items)

    def alternation():
        xs = [sequence()]
        while peek() == ord('|'):
            take()
            xs.append(sequence())
        return alt(*xs)

    tree = alternation()
    if pos[0] != len(src):
        raise GrammarError('syntax', 'regex: unbalanced )')
    return tree


_ST_KEYS = {'literal': {'text'}, 'regex': {'pattern'}, 'json_schema': {'json_schema'},
            'sequence': {'elements'}, 'or': {'elements'}, 'tag': {'begin', 'content', 'end'},
            'evaluated_tag': {'begin', 'content', 'end', 'evaluator', 'result'}}


def structtag_to_tree(text: str, ws_max: int, max_len_default: int, max_items_default: int) -> tuple:
    try:
        doc = json.loads(text)
    except ValueError as e:
        raise GrammarError('syntax', f'structural tag: {e}') from None
    any_byte = sym_of(range(256))

    def text_of(e, k):
        v = e.get(k)
        if not isinstance(v, str):
            raise GrammarError('unsupported', f'structural tag: {k} must be a string')
        return v.encode('utf-8')

    def lower(e):
        if not isinstance(e, dict) or e.get('type') not in _ST_KEYS:
            raise GrammarError('unsupported', 'structural tag: unknown element')
        ty = e['type']
        if set(e) - {'type'} != _ST_KEYS[ty]:
            raise GrammarError('unsupported', f'structural tag: keys of {ty}')
        if ty == 'literal':
            return lit(text_of(e, 'text'))
        if ty == 'regex':
            return ('and', (regex_to_tree(e['pattern']) if isinstance(e['pattern'], str) else
                            _raise_unsupported('pattern'), rep(any_byte, 0, max_len_default)))
        if ty == 'json_schema':
            return schema_to_tree(json.dumps(e['json_schema']), ws_max, max_len_default, max_items_default)
        if ty in ('sequence', 'or'):
            els = e['elements']
            if not isinstance(els, list) or (ty == 'or' and not els):
                raise GrammarError('unsupported', f'structural tag: elements of {ty}')
            kids = [lower(x) for x in els]
            if ty == 'sequence':
                return cat(*kids) if kids else EPS
            return alt(*kids)
        body = cat(lit(text_of(e, 'begin')), lower(e['content']), lit(text_of(e, 'end')))
        if ty == 'tag':
            return body
        res = e['result']
        if res != {'begin': '<result>', 'end': '</result>'}:
            raise GrammarError('unsupported', 'structural tag: result tags other than <result>')
        if e['evaluator'] == 'arithmetic':
            value = cat(rep(lit(b'-'), 0, 1), rep(rng(0x30, 0x39), 1, 64))
        elif e['evaluator'] == 'string':
            value = rep(sym_of(b for b in range(256) if b != 0x3C), 0, 64)
        else:
            raise GrammarError('unsupported', 'structural tag: unknown evaluator')
        error = cat(lit(b'<result_error>'), rep(sym_of(b'abcdefghijklmnopqrstuvwxyz_'), 1, 32),
                    lit(b'</result_error>'))
        return cat(body, forced(alt(cat(lit(b'<result>'), value, lit(b'</result>')), error)))

    return lower(doc)


def _raise_unsupported(what):
    raise GrammarError('unsupported', f'structural tag: {what}')
