// Structural-tag front-end.
//
// labs.miniml.ai "Evaluator aware decoding", "Where XGrammar-2 could take
// this": a Structural Tag is a JSON description whose atomic types (JSON
// schema, regex, literal strings) nest, and an evaluated tag is a tag whose
// completed content goes to a registered evaluator, with the result forced
// into a sibling span.  Elements read here:
//   {"type": "literal", "text": S}
//   {"type": "regex", "pattern": P}          (subset below; a match is at most
//                                            max_len_default bytes long)
//   {"type": "json_schema", "json_schema": J}   (the JSON-schema front-end)
//   {"type": "sequence", "elements": [E...]}, {"type": "or", "elements": [E...]}
//   {"type": "tag", "begin": S, "content": E, "end": S}
//   {"type": "evaluated_tag", "begin": S, "content": E, "end": S,
//    "evaluator": "arithmetic" | "string",
//    "result": {"begin": "<result>", "end": "</result>"}}
// An evaluated tag is followed by a forced region holding what the host
// injects: <result>V</result> (V: -?[0-9]{1,64} for arithmetic, [^<]{0,64}
// for string operations) or <result_error>[a-z_]{1,32}</result_error>.
// Regex subset: bytes, '.', [classes] with ranges and '^', escapes \d \w \s
// \n \t \r \f \v and escaped punctuation, ( ) groups, '|', and * + ? {m}
// {m,} {m,n}; '.' is any byte but a newline.  Anchors, group flags and
// non-ASCII inside classes fail closed (CG_E_UNSUPPORTED), as do unknown
// element types or keys, other result tags and evaluators.
#include <cstring>
#include <map>
#include <set>
#include <utility>

#include "../../../include/cg.h"
#include "ir.h"
#include "json.h"

namespace cg {
namespace {

[[noreturn]] void fail(int code, const std::string& m) { throw CompileError{code, m}; }

SymSet class_escape(unsigned char c, bool* ok) {
  SymSet s;
  *ok = true;
  if (c == 'd') s.set_range('0', '9');
  else if (c == 'w') { s.set_range('a', 'z'); s.set_range('A', 'Z'); s.set_range('0', '9'); s.set('_'); }
  else if (c == 's') { s.set(' '); s.set('\t'); s.set('\n'); s.set('\r'); s.set(0x0B); s.set(0x0C); }
  else *ok = false;
  return s;
}

int char_escape(unsigned char c) {
  switch (c) {
    case 'n': return 0x0A;
    case 't': return 0x09;
    case 'r': return 0x0D;
    case 'f': return 0x0C;
    case 'v': return 0x0B;
    default: return -1;
  }
}

bool is_special(unsigned char c) {
  return std::strchr("()[]{}|*+?.\\^$", c) != nullptr && c != 0;
}

class Regex {
 public:
  Regex(IR& ir, std::string p) : ir_(ir), p_(std::move(p)) {}
  int parse() {
    int x = alternation();
    if (i_ != p_.size()) fail(CG_E_SYNTAX, "regex: unbalanced )");
    return x;
  }

 private:
  IR& ir_;
  const std::string p_;  // owned: the caller's string may be a temporary
  size_t i_ = 0;

  bool more() const { return i_ < p_.size(); }
  unsigned char cur() const { return static_cast<unsigned char>(p_[i_]); }
  unsigned char next() {
    if (!more()) fail(CG_E_SYNTAX, "regex: unexpected end");
    return static_cast<unsigned char>(p_[i_++]);
  }

  int alternation() {
    std::vector<int> alts{sequence()};
    while (more() && cur() == '|') {
      ++i_;
      alts.push_back(sequence());
    }
    return ir_.alt(alts);
  }
  int sequence() {
    std::vector<int> items;
    while (more() && cur() != '|' && cur() != ')') items.push_back(postfix());
    if (items.empty()) return ir_.eps();
    return ir_.cat(items);
  }
  int postfix() {
    int x = atom();
    for (;;) {
      if (!more()) return x;
      const unsigned char c = cur();
      if (c == '*') { ++i_; x = ir_.rep(x, 0, -1); }
      else if (c == '+') { ++i_; x = ir_.rep(x, 1, -1); }
      else if (c == '?') { ++i_; x = ir_.rep(x, 0, 1); }
      else if (c == '{') {
        ++i_;
        const size_t close = p_.find('}', i_);
        if (close == std::string::npos) fail(CG_E_SYNTAX, "regex: unterminated {");
        const std::string body = p_.substr(i_, close - i_);
        i_ = close + 1;
        const size_t comma = body.find(',');
        auto num = [&](const std::string& t) {
          if (t.empty() || t.size() > 6) fail(CG_E_SYNTAX, "regex: bad {m,n}");
          int v = 0;
          for (char ch : t) {
            if (ch < '0' || ch > '9') fail(CG_E_SYNTAX, "regex: bad {m,n}");
            v = v * 10 + (ch - '0');
          }
          return v;
        };
        int lo, hi;
        if (comma == std::string::npos) { lo = hi = num(body); }
        else {
          if (body.find(',', comma + 1) != std::string::npos) fail(CG_E_SYNTAX, "regex: bad {m,n}");
          lo = num(body.substr(0, comma));
          const std::string h = body.substr(comma + 1);
          hi = h.empty() ? -1 : num(h);
          if (hi >= 0 && hi < lo) fail(CG_E_SYNTAX, "regex: bad {m,n}");
        }
        x = ir_.rep(x, lo, hi);
      } else {
        return x;
      }
    }
  }
  int atom() {
    const unsigned char c = next();
    if (c == '(') {
      if (more() && cur() == '?') fail(CG_E_UNSUPPORTED, "regex: group flags");
      int x = alternation();
      if (next() != ')') fail(CG_E_SYNTAX, "regex: unbalanced (");
      return x;
    }
    if (c == '[') return ir_.sym(cls());
    if (c == '.') { SymSet s; s.set_range(0, 255); SymSet t = s; return ir_.sym(without(t, 0x0A)); }
    if (c == '\\') {
      const unsigned char e = next();
      bool ok;
      SymSet s = class_escape(e, &ok);
      if (ok) return ir_.sym(s);
      const int ce = char_escape(e);
      if (ce >= 0) return ir_.byte(ce);
      if (is_special(e) || e == '-' || e == '/' || e == '"' || e == '\'') return ir_.byte(e);
      fail(CG_E_UNSUPPORTED, "regex: escape");
    }
    if (c == '^' || c == '$') fail(CG_E_UNSUPPORTED, "regex: anchors");
    if (c == ')' || c == '|' || c == '*' || c == '+' || c == '?' || c == '{' || c == '}' || c == ']')
      fail(CG_E_SYNTAX, "regex: unexpected operator");
    return ir_.byte(c);
  }
  static SymSet without(SymSet s, int b) {
    s.w[b >> 6] &= ~(uint64_t(1) << (b & 63));
    return s;
  }
  SymSet cls() {
    bool neg = false;
    if (more() && cur() == '^') { ++i_; neg = true; }
    SymSet s;
    bool first = true;
    for (;;) {
      unsigned char c = next();
      if (c == ']' && !first) break;
      first = false;
      int lo;
      if (c == '\\') {
        const unsigned char e = next();
        bool ok;
        SymSet esc = class_escape(e, &ok);
        if (ok) {
          for (int k = 0; k < 4; ++k) s.w[k] |= esc.w[k];
          continue;
        }
        const int ce = char_escape(e);
        lo = ce >= 0 ? ce : e;
      } else {
        lo = c;
      }
      if (lo >= 0x80) fail(CG_E_UNSUPPORTED, "regex: non-ASCII in a class");
      if (more() && cur() == '-' && i_ + 1 < p_.size() && p_[i_ + 1] != ']') {
        ++i_;
        int hi = next();
        if (hi == '\\') {
          const unsigned char e = next();
          const int ce = char_escape(e);
          hi = ce >= 0 ? ce : e;
        }
        if (hi >= 0x80 || hi < lo) fail(CG_E_SYNTAX, "regex: bad class range");
        s.set_range(lo, hi);
      } else {
        s.set(lo);
      }
    }
    if (neg) {
      SymSet all;
      all.set_range(0, 255);
      for (int k = 0; k < 4; ++k) all.w[k] &= ~s.w[k];
      return all;
    }
    return s;
  }
};

class StructTag {
 public:
  StructTag(IR& ir, uint32_t ws_max, uint32_t max_len, uint32_t max_items)
      : ir_(ir), ws_max_(ws_max), max_len_(max_len), max_items_(max_items) {}

  int lower(const JVal& e) {
    if (e.t != JVal::Obj) fail(CG_E_UNSUPPORTED, "structural tag: element must be an object");
    const JVal* ty = e.get("type");
    if (!ty || ty->t != JVal::Str) fail(CG_E_UNSUPPORTED, "structural tag: element without type");
    const std::string& t = ty->text;
    static const std::map<std::string, std::set<std::string>> keys = {
        {"literal", {"text"}}, {"regex", {"pattern"}}, {"json_schema", {"json_schema"}},
        {"sequence", {"elements"}}, {"or", {"elements"}}, {"tag", {"begin", "content", "end"}},
        {"evaluated_tag", {"begin", "content", "end", "evaluator", "result"}}};
    auto it = keys.find(t);
    if (it == keys.end()) fail(CG_E_UNSUPPORTED, "structural tag: unknown type " + t);
    std::set<std::string> have;
    for (auto& kv : e.obj)
      if (kv.first != "type") have.insert(kv.first);
    if (have != it->second) fail(CG_E_UNSUPPORTED, "structural tag: keys of " + t);
    if (t == "literal") return ir_.literal(str(e, "text"));
    if (t == "regex") {
      Regex r(ir_, str(e, "pattern"));
      const int x = r.parse();
      SymSet any;
      any.set_range(0, 255);
      return ir_.conj({x, ir_.rep(ir_.sym(any), 0, int(max_len_))});
    }
    if (t == "json_schema") return lower_json_schema_value(ir_, *e.get("json_schema"), ws_max_, max_len_, max_items_);
    if (t == "sequence" || t == "or") {
      const JVal* els = e.get("elements");
      if (els->t != JVal::Arr || (t == "or" && els->arr.empty()))
        fail(CG_E_UNSUPPORTED, "structural tag: elements of " + t);
      std::vector<int> kids;
      for (const JVal& x : els->arr) kids.push_back(lower(x));
      if (t == "or") return ir_.alt(kids);
      return kids.empty() ? ir_.eps() : ir_.cat(kids);
    }
    const int body = ir_.cat({ir_.literal(str(e, "begin")), lower(*e.get("content")), ir_.literal(str(e, "end"))});
    if (t == "tag") return body;
    const JVal* res = e.get("result");
    const JVal* rb = res->t == JVal::Obj ? res->get("begin") : nullptr;
    const JVal* re = res->t == JVal::Obj ? res->get("end") : nullptr;
    if (!rb || !re || res->obj.size() != 2 || rb->t != JVal::Str || re->t != JVal::Str || rb->text != "<result>" ||
        re->text != "</result>")
      fail(CG_E_UNSUPPORTED, "structural tag: result tags other than <result>");
    const std::string ev = str(e, "evaluator");
    int value;
    if (ev == "arithmetic") {
      value = ir_.cat({ir_.rep(ir_.byte('-'), 0, 1), ir_.rep(ir_.range('0', '9'), 1, 64)});
    } else if (ev == "string") {
      SymSet s;
      s.set_range(0, 255);
      s.w['<' >> 6] &= ~(uint64_t(1) << ('<' & 63));
      value = ir_.rep(ir_.sym(s), 0, 64);
    } else {
      fail(CG_E_UNSUPPORTED, "structural tag: unknown evaluator " + ev);
    }
    SymSet code;
    code.set_range('a', 'z');
    code.set('_');
    const int ok = ir_.cat({ir_.literal("<result>"), value, ir_.literal("</result>")});
    const int err = ir_.cat({ir_.literal("<result_error>"), ir_.rep(ir_.sym(code), 1, 32), ir_.literal("</result_error>")});
    return ir_.cat({body, ir_.injected(ir_.alt({ok, err}))});
  }

 private:
  IR& ir_;
  uint32_t ws_max_, max_len_, max_items_;

  static std::string str(const JVal& e, const char* k) {
    const JVal* v = e.get(k);
    if (!v || v->t != JVal::Str) fail(CG_E_UNSUPPORTED, std::string("structural tag: ") + k + " must be a string");
    return v->text;
  }
};

}  // namespace

int lower_structural_tag(IR& ir, const std::string& src, uint32_t ws_max, uint32_t max_len_default,
                         uint32_t max_items_default) {
  JsonReader r(src);
  const JVal doc = r.document();
  StructTag st(ir, ws_max, max_len_default, max_items_default);
  return st.lower(doc);
}

}  // namespace cg
