// JSON-schema subset front-end.
//
// Output language (WS = [ \t\n\r]{0,ws_max}, only between structural tokens;
// never before the root value nor after it, so a finished document leaves the
// automaton in a state without continuation):
//   object  "{" WS ( "\"k1\"" WS ":" WS v1 ( WS "," WS "\"k\"" WS ":" WS v )* )? WS "}"
//           properties in declared order; every property must be required and
//           additionalProperties false or absent (absent is read as false)
//   string  '"' CHAR{minLength,maxLength} '"'  (maxLength defaults to
//           max_len_default; "x-maxBytes" alone bounds the content in bytes)
//   integer -?(0|[1-9][0-9]{0,18});  number -?(0|[1-9][0-9]{0,15})(\.[0-9]{1,16})?([eE][+-]?[0-9]{1,3})?
//   boolean, null, enum / const (string, integer, boolean, null literals)
//   array   "[" WS ( "]" | v ( WS "," WS v ){0,max-1} WS "]" )      (minItems 0)
//           "[" WS v ( WS "," WS v ){min-1,max-1} WS "]"            (minItems >= 1)
//   anyOf / type lists: union
// CHAR: a well-formed UTF-8 scalar other than '"', '\\' and controls < 0x20,
// or one escape (\" \\ \/ \b \f \n \r \t \uXXXX), each counting as one
// character.  Every other keyword fails closed, as the compiler of dev.to "I
// found a runner bug..." refuses what it does not support; whitespace bounded per
// usetacet.com/docs/grammar "A valid call also has to end" and the pinned
// compact separators of the dev.to page).
#include <algorithm>
#include <cstring>
#include <set>

#include "../../../include/cg.h"
#include "ir.h"
#include "json.h"

namespace cg {
namespace {

[[noreturn]] void fail(int code, const std::string& m) { throw CompileError{code, m}; }

const std::set<std::string> kIgnored = {"title", "description", "$schema", "$id", "$comment", "default", "examples"};
const std::set<std::string> kKnown = {"type", "properties", "required", "additionalProperties", "enum", "const",
                                      "anyOf", "items", "minItems", "maxItems", "minLength", "maxLength",
                                      "x-maxBytes"};

std::string json_string_literal(const std::string& s) {
  static const char* hex = "0123456789abcdef";
  std::string o = "\"";
  for (unsigned char c : s) {
    if (c == '"') o += "\\\"";
    else if (c == '\\') o += "\\\\";
    else if (c < 0x20) { o += "\\u00"; o.push_back(hex[c >> 4]); o.push_back(hex[c & 15]); }
    else o.push_back(char(c));
  }
  return o + "\"";
}

class Lowering {
 public:
  Lowering(IR& ir, uint32_t ws_max, uint32_t max_len_default, uint32_t max_items_default)
      : ir_(ir), ws_max_(ws_max), max_len_(max_len_default), max_items_(max_items_default) {}

  int lower(const JVal& s) {
    if (s.t == JVal::Bool && s.b) fail(CG_E_UNSUPPORTED, "unconstrained value");
    if (s.t != JVal::Obj) fail(CG_E_UNSUPPORTED, "schema must be an object");
    if (s.obj.empty()) fail(CG_E_UNSUPPORTED, "unconstrained value");
    for (auto& kv : s.obj)
      if (!kKnown.count(kv.first) && !kIgnored.count(kv.first)) fail(CG_E_UNSUPPORTED, "keyword " + kv.first);

    if (const JVal* any = s.get("anyOf")) {
      for (auto& kv : s.obj)
        if (kv.first != "anyOf" && !kIgnored.count(kv.first)) fail(CG_E_UNSUPPORTED, "anyOf with sibling keywords");
      if (any->t != JVal::Arr || any->arr.empty()) fail(CG_E_UNSUPPORTED, "empty anyOf");
      std::vector<int> k;
      for (auto& b : any->arr) k.push_back(lower(b));
      return ir_.alt(k);
    }
    const JVal* ty = s.get("type");
    if (s.get("enum") || s.get("const")) {
      std::vector<const JVal*> vals;
      if (const JVal* e = s.get("enum")) {
        if (e->t != JVal::Arr) fail(CG_E_UNSUPPORTED, "enum must be a list");
        for (auto& v : e->arr) vals.push_back(&v);
      } else {
        vals.push_back(s.get("const"));
      }
      if (vals.empty()) fail(CG_E_UNSUPPORTED, "empty enum");
      std::vector<int> k;
      for (const JVal* v : vals) {
        if (v->t == JVal::Num && !v->is_int_num()) fail(CG_E_UNSUPPORTED, "non-integer number in enum");
        if (ty) {
          bool ok = false;
          if (ty->t == JVal::Str) {
            const std::string& tn = ty->text;
            ok = (tn == "string" && v->t == JVal::Str) || (tn == "integer" && v->t == JVal::Num) ||
                 (tn == "boolean" && v->t == JVal::Bool) || (tn == "null" && v->t == JVal::Null);
          }
          if (!ok) fail(CG_E_UNSUPPORTED, "enum value does not match type");
        }
        k.push_back(ir_.literal(value_literal(*v)));
      }
      return ir_.alt(k);
    }
    if (ty && ty->t == JVal::Arr) {
      if (ty->arr.empty()) fail(CG_E_UNSUPPORTED, "empty type list");
      std::vector<int> k;
      for (auto& t : ty->arr) {
        JVal copy = s;
        for (auto& kv : copy.obj) if (kv.first == "type") kv.second = t;
        k.push_back(lower(copy));
      }
      return ir_.alt(k);
    }
    std::string tn = (ty && ty->t == JVal::Str) ? ty->text : std::string();
    if (tn == "object") return object(s);
    if (tn == "string") return string(s);
    if (tn == "integer") {
      return ir_.cat({ir_.rep(ir_.byte('-'), 0, 1),
                      ir_.alt({ir_.byte('0'), ir_.cat({ir_.range('1', '9'), ir_.rep(ir_.range('0', '9'), 0, 18)})})});
    }
    if (tn == "number") {
      SymSet e; e.set('e'); e.set('E');
      SymSet pm; pm.set('+'); pm.set('-');
      int frac = ir_.rep(ir_.cat({ir_.byte('.'), ir_.rep(ir_.range('0', '9'), 1, 16)}), 0, 1);
      int expo = ir_.rep(ir_.cat({ir_.sym(e), ir_.rep(ir_.sym(pm), 0, 1), ir_.rep(ir_.range('0', '9'), 1, 3)}), 0, 1);
      return ir_.cat({ir_.rep(ir_.byte('-'), 0, 1),
                      ir_.alt({ir_.byte('0'), ir_.cat({ir_.range('1', '9'), ir_.rep(ir_.range('0', '9'), 0, 15)})}),
                      frac, expo});
    }
    if (tn == "boolean") return ir_.alt({ir_.literal("true"), ir_.literal("false")});
    if (tn == "null") return ir_.literal("null");
    if (tn == "array") return array(s);
    fail(CG_E_UNSUPPORTED, "type " + tn);
  }

 private:
  IR& ir_;
  uint32_t ws_max_, max_len_, max_items_;

  int ws() {
    SymSet s; s.set(' '); s.set('\t'); s.set('\n'); s.set('\r');
    return ir_.rep(ir_.sym(s), 0, int(ws_max_));
  }
  static long as_int(const JVal* v, const char* what) {
    if (!v || v->t != JVal::Num) fail(CG_E_UNSUPPORTED, std::string(what) + " must be a number");
    double d = std::stod(v->text);
    if (d < 0 || d > 1e7 || d != double(long(d))) fail(CG_E_UNSUPPORTED, std::string(what) + " out of range");
    return long(d);
  }
  static std::string value_literal(const JVal& v) {
    switch (v.t) {
      case JVal::Null: return "null";
      case JVal::Bool: return v.b ? "true" : "false";
      case JVal::Str: return json_string_literal(v.text);
      case JVal::Num: {
        std::string t = v.text;
        // canonical integer text: JSON already forbids leading zeros; -0 is 0
        if (t == "-0") t = "0";
        return t;
      }
      default: fail(CG_E_UNSUPPORTED, "enum/const value of this type");
    }
  }
  int char_() {
    SymSet plain;
    for (int b = 0x20; b < 0x80; ++b) if (b != '"' && b != '\\') plain.set(b);
    int cont = ir_.range(0x80, 0xBF);
    SymSet e1; e1.set_range(0xE1, 0xEC); e1.set(0xEE); e1.set(0xEF);
    int utf8 = ir_.alt({
        ir_.sym(plain),
        ir_.cat({ir_.range(0xC2, 0xDF), cont}),
        ir_.cat({ir_.byte(0xE0), ir_.range(0xA0, 0xBF), ir_.range(0x80, 0xBF)}),
        ir_.cat({ir_.sym(e1), ir_.range(0x80, 0xBF), ir_.range(0x80, 0xBF)}),
        ir_.cat({ir_.byte(0xED), ir_.range(0x80, 0x9F), ir_.range(0x80, 0xBF)}),
        ir_.cat({ir_.byte(0xF0), ir_.range(0x90, 0xBF), ir_.range(0x80, 0xBF), ir_.range(0x80, 0xBF)}),
        ir_.cat({ir_.range(0xF1, 0xF3), ir_.range(0x80, 0xBF), ir_.range(0x80, 0xBF), ir_.range(0x80, 0xBF)}),
        ir_.cat({ir_.byte(0xF4), ir_.range(0x80, 0x8F), ir_.range(0x80, 0xBF), ir_.range(0x80, 0xBF)}),
    });
    SymSet simple;
    for (char c : std::string("\"\\/bfnrt")) simple.set((unsigned char)c);
    SymSet hex;
    for (char c : std::string("0123456789abcdefABCDEF")) hex.set((unsigned char)c);
    int esc = ir_.cat({ir_.byte('\\'),
                       ir_.alt({ir_.sym(simple),
                                ir_.cat({ir_.byte('u'), ir_.sym(hex), ir_.sym(hex), ir_.sym(hex), ir_.sym(hex)})})});
    return ir_.alt({utf8, esc});
  }
  int string(const JVal& s) {
    long lo = s.get("minLength") ? as_int(s.get("minLength"), "minLength") : 0;
    int body;
    if (s.get("maxLength")) {
      long hi = as_int(s.get("maxLength"), "maxLength");
      if (hi < lo) fail(CG_E_UNSUPPORTED, "maxLength < minLength");
      body = ir_.rep(char_(), int(lo), int(hi));
    } else if (s.get("x-maxBytes")) {
      body = ir_.rep(char_(), int(lo), -1);
    } else {
      if (long(max_len_) < lo) fail(CG_E_UNSUPPORTED, "maxLength < minLength");
      body = ir_.rep(char_(), int(lo), int(max_len_));
    }
    if (s.get("x-maxBytes")) {
      long nb = as_int(s.get("x-maxBytes"), "x-maxBytes");
      body = ir_.conj({body, ir_.rep(ir_.range(0, 255), 0, int(nb))});
    }
    return ir_.cat({ir_.byte('"'), body, ir_.byte('"')});
  }
  int object(const JVal& s) {
    static const JVal empty_obj = [] { JVal v; v.t = JVal::Obj; return v; }();
    static const JVal empty_arr = [] { JVal v; v.t = JVal::Arr; return v; }();
    const JVal* props = s.get("properties");
    if (!props) props = &empty_obj;
    const JVal* req = s.get("required");
    if (!req) req = &empty_arr;
    if (props->t != JVal::Obj || req->t != JVal::Arr) fail(CG_E_UNSUPPORTED, "optional properties");
    std::vector<std::string> keys, reqs;
    for (auto& kv : props->obj) {
      if (std::find(keys.begin(), keys.end(), kv.first) == keys.end()) keys.push_back(kv.first);
    }
    for (auto& r : req->arr) {
      if (r.t != JVal::Str) fail(CG_E_UNSUPPORTED, "optional properties");
      reqs.push_back(r.text);
    }
    std::vector<std::string> a = keys, b = reqs;
    std::sort(a.begin(), a.end());
    std::sort(b.begin(), b.end());
    if (a != b || std::adjacent_find(b.begin(), b.end()) != b.end()) fail(CG_E_UNSUPPORTED, "optional properties");
    if (const JVal* ap = s.get("additionalProperties"))
      if (!(ap->t == JVal::Bool && !ap->b)) fail(CG_E_UNSUPPORTED, "additionalProperties");
    if (keys.empty()) return ir_.cat({ir_.byte('{'), ws(), ir_.byte('}')});
    std::vector<int> parts = {ir_.byte('{'), ws()};
    for (size_t i = 0; i < keys.size(); ++i) {
      if (i) { parts.push_back(ws()); parts.push_back(ir_.byte(',')); parts.push_back(ws()); }
      parts.push_back(ir_.literal(json_string_literal(keys[i])));
      parts.push_back(ws());
      parts.push_back(ir_.byte(':'));
      parts.push_back(ws());
      parts.push_back(lower(*props->get(keys[i])));
    }
    parts.push_back(ws());
    parts.push_back(ir_.byte('}'));
    return ir_.cat(parts);
  }
  int array(const JVal& s) {
    const JVal* items = s.get("items");
    if (!items) fail(CG_E_UNSUPPORTED, "array without items");
    long lo = s.get("minItems") ? as_int(s.get("minItems"), "minItems") : 0;
    long hi = s.get("maxItems") ? as_int(s.get("maxItems"), "maxItems") : long(max_items_);
    if (hi < lo) fail(CG_E_UNSUPPORTED, "maxItems < minItems");
    if (hi == 0) return ir_.cat({ir_.byte('['), ws(), ir_.byte(']')});
    int item = lower(*items);
    auto more = [&] { return ir_.cat({ws(), ir_.byte(','), ws(), lower(*items)}); };
    if (lo == 0)
      return ir_.cat({ir_.byte('['), ws(),
                      ir_.alt({ir_.byte(']'), ir_.cat({item, ir_.rep(more(), 0, int(hi - 1)), ws(), ir_.byte(']')})})});
    return ir_.cat({ir_.byte('['), ws(), item, ir_.rep(more(), int(lo - 1), int(hi - 1)), ws(), ir_.byte(']')});
  }
};

}  // namespace

int lower_json_schema(IR& ir, const std::string& src, uint32_t ws_max, uint32_t max_len_default,
                      uint32_t max_items_default) {
  JsonReader r(src);
  JVal doc = r.document();
  Lowering l(ir, ws_max, max_len_default, max_items_default);
  return l.lower(doc);
}

int lower_json_schema_value(IR& ir, const JVal& schema, uint32_t ws_max, uint32_t max_len_default,
                            uint32_t max_items_default) {
  Lowering l(ir, ws_max, max_len_default, max_items_default);
  return l.lower(schema);
}

}  // namespace cg
