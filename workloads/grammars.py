"""Grammar source texts of the workloads (inputs only; nothing here compiles them).

Two source kinds are used:

* ``gbnf``: the GBNF-style rule language (``name ::= expr``; ``|``, ``&``
  (intersection), juxtaposition, ``? * + {m} {m,} {m,n}``, ``"literal"``,
  ``[class]``, ``( )`` and ``@forced( )`` for bytes the host injects).
* ``json``: a JSON-schema subset (object / string / integer / number /
  boolean / null / enum / const / anyOf / array), compiled with bounded
  whitespace runs and bounded open fields.

Sources:
* calc call -- the tool-call shape ``calculate({"expression":"125*8"})`` from
  usetacet.com/docs/grammar, "Reading the grammar for a tool".
* booking-decision schema -- seedpath.ai "Guided Decoding & Structured-Output
  Reliability", Design 1 (base schema); the elided appointment object is read as
  ``{"date": string <= 20, "time": string <= 10}`` (the extraction schema's
  bounds, same page, Design 5).
* reasoning + integer answer -- dev.to "I found a runner bug...", "The system
  boundary I am testing" (model-facing integer contract).
* ``<calc>`` evaluator shape -- labs.miniml.ai "Evaluator aware decoding",
  "This is a grammar problem" and "A concrete prototype on llama.cpp".
* JSON evaluator shape ``{"expression": "17 * 23 + 91", "answer": 482}`` --
  same page, "This is a grammar problem" (JSON form); the expression character
  set follows the page's Structural-Tag sketch (content regex
  ``[0-9+\\-*/(). ]+``).
* extraction and "reasoned" schemas -- seedpath.ai page, Designs 5 and 2.
"""

from __future__ import annotations

import json
from dataclasses import dataclass, field


@dataclass(frozen=True)
class Bounds:
    """Termination bounds (usetacet.com/docs/grammar, "A valid call also has to end")."""
    ws_max: int = 4              # longest run of JSON whitespace in one slot
    max_len_default: int = 256   # maxLength of a JSON string that states none
    depth_max: int = 5           # simultaneous activations of one GBNF rule
    max_items_default: int = 16  # maxItems of a JSON array that states none
    max_tokens: int = 2048       # host cap on one constrained generation


@dataclass(frozen=True)
class GrammarSpec:
    name: str
    kind: str                   # "gbnf" | "json" | "structtag"
    source: str
    bounds: Bounds = field(default_factory=Bounds)
    # Evaluator-aware grammars: the host evaluates the text between the last
    # ``span_open`` and the ``span_close`` that ends the generated text when
    # the automaton enters a forced region, and forces the formatted result.
    evaluator: str | None = None     # "arith", "strop" or None
    span_open: bytes = b""
    span_close: bytes = b""
    result_format: str = ""         # "calc_tag" | "json_answer" | "strop_tag"


CALC_CALL = r'''
# calculate({"expression":"<1..64 of [0-9+*/() -], at most 8 spaces in a row>"})
root ::= "calculate({\"expression\":\"" body "\"})"
body ::= [0-9+*/() \-]{1,64} & norun
norun ::= ( [^ ] | " "{1,8} [^ ] )* " "{0,8}
'''

_ENUM_REASON = ["eligible", "under_age", "over_limit", "insufficient_info"]
_ENUM_ACTION = ["book_appointment", "decline", "offer_alternative", "escalate_human"]


def _booking_props(response_max: int) -> dict:
    return {
        "eligibility": {
            "type": "object",
            "properties": {
                "criteria_met": {"type": "boolean"},
                "reason_code": {"type": "string", "enum": _ENUM_REASON},
            },
            "required": ["criteria_met", "reason_code"],
            "additionalProperties": False,
        },
        "action": {"type": "string", "enum": _ENUM_ACTION},
        "appointment": {"anyOf": [
            {"type": "object",
             "properties": {"date": {"type": "string", "maxLength": 20},
                            "time": {"type": "string", "maxLength": 10}},
             "required": ["date", "time"], "additionalProperties": False},
            {"type": "null"}]},
        "response_text": {"type": "string", "maxLength": response_max},
    }


def booking_schema(response_max: int = 700) -> str:
    props = _booking_props(response_max)
    return json.dumps({"type": "object", "properties": props,
                       "required": list(props), "additionalProperties": False})


def reasoned_schema(calc_max: int = 400, response_max: int = 700) -> str:
    props = {"calculation": {"type": "string", "maxLength": calc_max},
             "within_limit_banding": {"enum": ["within_limit", "reduced_scope_band", "over_limit"]}}
    props.update(_booking_props(response_max))
    return json.dumps({"type": "object", "properties": props,
                       "required": list(props), "additionalProperties": False})


def reasoning_answer_schema(max_bytes: int = 2048) -> str:
    props = {"reasoning": {"type": "string", "x-maxBytes": max_bytes},
             "answer": {"type": "integer"}}
    return json.dumps({"type": "object", "properties": props,
                       "required": list(props), "additionalProperties": False})


def extraction_schema() -> str:
    props = {
        "customer_age": {"anyOf": [{"type": "integer"}, {"type": "null"}]},
        "price_components": {"type": "array", "items": {"type": "number"}, "maxItems": 10},
        "requested_date": {"anyOf": [{"type": "string", "maxLength": 20}, {"type": "null"}]},
        "requested_time": {"anyOf": [{"type": "string", "maxLength": 10}, {"type": "null"}]},
    }
    return json.dumps({"type": "object", "properties": props,
                       "required": list(props), "additionalProperties": False})


CALC_EVAL = r'''
# The expression is <calc>EXPR</calc><result>V</result> then a short tail.
root ::= "The expression is <calc>" span "</calc>" @forced( result ) tail
span ::= expr & [0-9+\-*/(). ]{1,48}
expr ::= sp term ( sp op sp term )* sp
term ::= num | "(" expr ")"
num ::= "-"? [0-9]{1,6} ( "." [0-9]{1,3} )?
op ::= [+\-*/]
sp ::= " "?
result ::= "<result>" "-"? [0-9]{1,64} "</result>" | "<result_error>" [a-z_]{1,32} "</result_error>"
tail ::= [a-z ,]{0,24} "."
'''

JSON_EVAL = r'''
# {"expression": "EXPR", "answer": V}  -- the answer is forced by the host
root ::= "{\"expression\": \"" span "\"" @forced( answer )
span ::= [0-9+\-*/(). ]{1,64} & norun
norun ::= ( [^ ] | " "{1,8} [^ ] )* " "{0,8}
answer ::= ", \"answer\": " ( "-"? [0-9]{1,64} "}" | "null, \"error\": \"" [a-z_]{1,32} "\"}" )
'''

STROP_EVAL = r'''
# The answer is <strop>OP("...")</strop><result>V</result> then a short tail.
root ::= "The answer is <strop>" call "</strop>" @forced( result ) tail
call ::= "count(" str "," sp str ")" | "len(" str ")" | "reverse(" str ")" | "upper(" str ")"
       | "substr(" str "," sp int "," sp int ")"
str ::= "\"" ( [a-zA-Z0-9 .,!?'\-] | "\\\"" | "\\\\" ){0,24} "\""
int ::= "-"? [0-9]{1,2}
sp ::= " "?
result ::= "<result>" [^<]{0,64} "</result>" | "<result_error>" [a-z_]{1,32} "</result_error>"
tail ::= [a-z ,]{0,24} "."
'''

# The page's evaluated tag (labs.miniml.ai "Evaluator aware decoding", "Where
# XGrammar-2 could take this") inside a structural tag with the calc_eval
# framing: the same language as calc_eval's outer shape, written as nested
# structural-tag elements.
CALC_STRUCTTAG = json.dumps({
    "type": "sequence",
    "elements": [
        {"type": "literal", "text": "The expression is "},
        {"type": "evaluated_tag", "begin": "<calc>",
         "content": {"type": "regex", "pattern": "[0-9+\\-*/(). ]+"},
         "end": "</calc>", "evaluator": "arithmetic",
         "result": {"begin": "<result>", "end": "</result>"}},
        {"type": "regex", "pattern": "[a-z ,]{0,24}\\."},
    ],
})


# Any JSON value without whitespace: strings of printable ASCII other than '"'
# and '\\' (no escapes), integers.  value, object, member and array lie on a
# cycle of references, so each reference to them opens a frame of the
# pushdown automaton: an array costs two frames per level (value, array), an
# object three (value, object, member).
JSON_NESTED = r'''
root ::= value
value ::= object | array | string | number | "true" | "false" | "null"
object ::= "{" ( member ( "," member )* )? "}"
member ::= string ":" value
array ::= "[" ( value ( "," value )* )? "]"
string ::= "\"" [ !#-\[\]-~]* "\""
number ::= "-"? ( "0" | [1-9] [0-9]* )
'''

# Recursive grammars for the pushdown path: name -> (GBNF source, stack bound).
PDA_GRAMMARS: dict[str, tuple[str, int]] = {
    "json_nested": (JSON_NESTED, 32),
}


GRAMMARS: dict[str, GrammarSpec] = {
    "calc_call": GrammarSpec("calc_call", "gbnf", CALC_CALL),
    "booking": GrammarSpec("booking", "json", booking_schema(700)),
    "booking_200": GrammarSpec("booking_200", "json", booking_schema(200)),
    "reasoning_answer": GrammarSpec("reasoning_answer", "json", reasoning_answer_schema(2048)),
    "reasoning_answer_1024": GrammarSpec("reasoning_answer_1024", "json", reasoning_answer_schema(1024)),
    "calc_eval": GrammarSpec("calc_eval", "gbnf", CALC_EVAL, evaluator="arith",
                             span_open=b"<calc>", span_close=b"</calc>", result_format="calc_tag"),
    "json_eval": GrammarSpec("json_eval", "gbnf", JSON_EVAL, evaluator="arith",
                             span_open=b'{"expression": "', span_close=b'"',
                             result_format="json_answer"),
    "strop_eval": GrammarSpec("strop_eval", "gbnf", STROP_EVAL, evaluator="strop",
                              span_open=b"<strop>", span_close=b"</strop>", result_format="strop_tag"),
    "calc_structtag": GrammarSpec("calc_structtag", "structtag", CALC_STRUCTTAG, Bounds(max_len_default=48),
                                  evaluator="arith", span_open=b"<calc>", span_close=b"</calc>",
                                  result_format="calc_tag"),
    "extraction": GrammarSpec("extraction", "json", extraction_schema()),
    "reasoned": GrammarSpec("reasoned", "json", reasoned_schema()),
}
