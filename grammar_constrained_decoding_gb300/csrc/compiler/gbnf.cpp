// GBNF-style rule language front-end.
//
// Source form (one reading of the GBNF grammar shown in labs.miniml.ai
// "Evaluator aware decoding", "This is a grammar problem"):
//   NAME ::= expr     -- a rule starts at every NAME followed by ::=
//   expr: alternatives '|', intersections '&' (bind tighter), juxtaposition,
//         postfix ? * + {m} {m,} {m,n}; atoms "literal", [class], NAME,
//         ( expr ), @forced( expr ) for bytes the host injects.
//   Escapes \\ \" \] \[ \- \^ \n \r \t \xHH; '#' comments to end of line.
// Rules are expanded by inlining from "root"; one rule may be active at most
// depth_max times along an expansion path and a deeper reference is the empty
// language -- the bounded nesting that keeps the automaton finite
// (usetacet.com/docs/grammar, "The guarantee" / "A valid call also has to end").
#include <cctype>
#include <map>
#include <memory>

#include "../../../include/cg.h"
#include "ir.h"

namespace cg {

int IR::injected(int x) {
  const Node n = nodes[x];  // copy: add() may reallocate
  switch (n.kind) {
    case NodeKind::Sym: return sym(n.set.shifted_to_injected());
    case NodeKind::Cat:
    case NodeKind::Alt:
    case NodeKind::And: {
      std::vector<int> k;
      for (int c : n.kids) k.push_back(injected(c));
      Node m; m.kind = n.kind; m.kids = std::move(k);
      return add(std::move(m));
    }
    case NodeKind::Rep: return rep(injected(n.kids[0]), n.lo, n.hi);
    default: return x;
  }
}

namespace {

enum class Tok { Name, Def, Lit, Class, LParen, RParen, Bar, Amp, Quest, Star, Plus, Repeat, Forced, End };

struct Token {
  Tok kind;
  std::string text;   // Name, Lit
  SymSet set;         // Class
  int lo = 0, hi = 0; // Repeat (hi < 0 = open)
  size_t pos = 0;
};

[[noreturn]] void fail(int code, const std::string& m) { throw CompileError{code, m}; }

int hexdigit(int c) {
  if (c >= '0' && c <= '9') return c - '0';
  if (c >= 'a' && c <= 'f') return c - 'a' + 10;
  if (c >= 'A' && c <= 'F') return c - 'A' + 10;
  return -1;
}

// reads an escape starting at src[i] == '\\'; returns the byte, advances i
int read_escape(const std::string& src, size_t& i) {
  if (i + 1 >= src.size()) fail(CG_E_SYNTAX, "dangling backslash");
  unsigned char c = src[i + 1];
  if (c == 'x') {
    if (i + 3 >= src.size()) fail(CG_E_SYNTAX, "short \\x escape");
    int h = hexdigit((unsigned char)src[i + 2]), l = hexdigit((unsigned char)src[i + 3]);
    if (h < 0 || l < 0) fail(CG_E_SYNTAX, "bad \\x escape");
    i += 4;
    return h * 16 + l;
  }
  i += 2;
  if (c == 'n') return 0x0A;
  if (c == 'r') return 0x0D;
  if (c == 't') return 0x09;
  return c;
}

std::vector<Token> lex(const std::string& src) {
  std::vector<Token> out;
  size_t i = 0, n = src.size();
  while (i < n) {
    unsigned char c = src[i];
    Token t;
    t.pos = i;
    if (c == ' ' || c == '\t' || c == '\r' || c == '\n') { ++i; continue; }
    if (c == '#') { while (i < n && src[i] != '\n') ++i; continue; }
    if (c == '"') {
      ++i;
      std::string lit;
      for (;;) {
        if (i >= n) fail(CG_E_SYNTAX, "unterminated literal");
        if (src[i] == '"') { ++i; break; }
        if (src[i] == '\\') lit.push_back(char(read_escape(src, i)));
        else lit.push_back(src[i++]);
      }
      t.kind = Tok::Lit; t.text = lit; out.push_back(t); continue;
    }
    if (c == '[') {
      ++i;
      bool neg = false;
      if (i < n && src[i] == '^') { neg = true; ++i; }
      struct Item { int v; bool esc; };
      std::vector<Item> items;
      for (;;) {
        if (i >= n) fail(CG_E_SYNTAX, "unterminated class");
        if (src[i] == ']') { ++i; break; }
        if (src[i] == '\\') { int v = read_escape(src, i); items.push_back({v, true}); }
        else items.push_back({(unsigned char)src[i++], false});
      }
      SymSet s;
      for (size_t k = 0; k < items.size();) {
        bool range = k + 2 < items.size() && items[k + 1].v == '-' && !items[k + 1].esc;
        if (range) {
          if (items[k + 2].v < items[k].v) fail(CG_E_SYNTAX, "reversed class range");
          s.set_range(items[k].v, items[k + 2].v);
          k += 3;
        } else {
          s.set(items[k].v);
          k += 1;
        }
      }
      if (neg) {
        SymSet all; all.set_range(0, 255);
        for (int a = 0; a < 256; ++a) if (s.test(a)) all.w[a >> 6] &= ~(uint64_t(1) << (a & 63));
        s = all;
      }
      t.kind = Tok::Class; t.set = s; out.push_back(t); continue;
    }
    if (src.compare(i, 3, "::=") == 0) { t.kind = Tok::Def; i += 3; out.push_back(t); continue; }
    if (src.compare(i, 7, "@forced") == 0) { t.kind = Tok::Forced; i += 7; out.push_back(t); continue; }
    if (c == '(') { t.kind = Tok::LParen; ++i; out.push_back(t); continue; }
    if (c == ')') { t.kind = Tok::RParen; ++i; out.push_back(t); continue; }
    if (c == '|') { t.kind = Tok::Bar; ++i; out.push_back(t); continue; }
    if (c == '&') { t.kind = Tok::Amp; ++i; out.push_back(t); continue; }
    if (c == '?') { t.kind = Tok::Quest; ++i; out.push_back(t); continue; }
    if (c == '*') { t.kind = Tok::Star; ++i; out.push_back(t); continue; }
    if (c == '+') { t.kind = Tok::Plus; ++i; out.push_back(t); continue; }
    if (c == '{') {
      size_t j = src.find('}', i);
      if (j == std::string::npos) fail(CG_E_SYNTAX, "unterminated repetition");
      std::string body;
      for (size_t k = i + 1; k < j; ++k) if (src[k] != ' ') body.push_back(src[k]);
      size_t comma = body.find(',');
      auto num = [&](const std::string& s) -> long {
        if (s.empty() || s.size() > 7) fail(CG_E_SYNTAX, "bad repetition {" + body + "}");
        for (char ch : s) if (!isdigit((unsigned char)ch)) fail(CG_E_SYNTAX, "bad repetition {" + body + "}");
        return std::stol(s);
      };
      if (comma == std::string::npos) { t.lo = t.hi = int(num(body)); }
      else {
        if (body.find(',', comma + 1) != std::string::npos) fail(CG_E_SYNTAX, "bad repetition {" + body + "}");
        t.lo = int(num(body.substr(0, comma)));
        std::string h = body.substr(comma + 1);
        t.hi = h.empty() ? -1 : int(num(h));
        if (t.hi >= 0 && t.hi < t.lo) fail(CG_E_SYNTAX, "bad repetition bounds {" + body + "}");
      }
      t.kind = Tok::Repeat; i = j + 1; out.push_back(t); continue;
    }
    if (c == '_' || (c < 0x80 && isalpha(c))) {
      size_t j = i;
      while (j < n && ((unsigned char)src[j] < 0x80) &&
             (isalnum((unsigned char)src[j]) || src[j] == '_' || src[j] == '-')) ++j;
      t.kind = Tok::Name; t.text = src.substr(i, j - i); i = j; out.push_back(t); continue;
    }
    fail(CG_E_SYNTAX, "unexpected byte at offset " + std::to_string(i));
  }
  Token e; e.kind = Tok::End; e.pos = n; out.push_back(e);
  return out;
}

// Rule-body syntax tree before expansion.
struct Ast {
  enum K { Lit, Class, Ref, Cat, Alt, And, Rep, Forced, Eps } k;
  std::string text;
  SymSet set;
  std::vector<std::unique_ptr<Ast>> kids;
  int lo = 0, hi = 0;
};
using AstP = std::unique_ptr<Ast>;

class Parser {
 public:
  explicit Parser(std::vector<Token> t) : t_(std::move(t)) {}

  std::map<std::string, AstP> rules() {
    std::map<std::string, AstP> out;
    while (peek().kind != Tok::End) {
      if (!rule_start()) fail(CG_E_SYNTAX, "expected \"name ::=\"");
      std::string name = t_[i_].text;
      i_ += 2;
      if (out.count(name)) fail(CG_E_SYNTAX, "rule " + name + " defined twice");
      out[name] = alt();
    }
    return out;
  }

 private:
  std::vector<Token> t_;
  size_t i_ = 0;

  const Token& peek(size_t k = 0) const {
    size_t j = i_ + k;
    return j < t_.size() ? t_[j] : t_.back();
  }
  bool rule_start() const { return peek().kind == Tok::Name && peek(1).kind == Tok::Def; }

  AstP make(Ast::K k) { auto a = std::make_unique<Ast>(); a->k = k; return a; }

  AstP alt() {
    std::vector<AstP> xs;
    xs.push_back(conj());
    while (peek().kind == Tok::Bar) { ++i_; xs.push_back(conj()); }
    if (xs.size() == 1) return std::move(xs[0]);
    auto a = make(Ast::Alt); a->kids = std::move(xs); return a;
  }
  AstP conj() {
    std::vector<AstP> xs;
    xs.push_back(seq());
    while (peek().kind == Tok::Amp) { ++i_; xs.push_back(seq()); }
    if (xs.size() == 1) return std::move(xs[0]);
    auto a = make(Ast::And); a->kids = std::move(xs); return a;
  }
  AstP seq() {
    std::vector<AstP> xs;
    for (;;) {
      Tok k = peek().kind;
      if (k == Tok::Bar || k == Tok::Amp || k == Tok::RParen || k == Tok::End || rule_start()) break;
      xs.push_back(post());
    }
    if (xs.empty()) return make(Ast::Eps);
    if (xs.size() == 1) return std::move(xs[0]);
    auto a = make(Ast::Cat); a->kids = std::move(xs); return a;
  }
  AstP post() {
    AstP x = atom();
    for (;;) {
      const Token& t = peek();
      int lo, hi;
      if (t.kind == Tok::Quest) { lo = 0; hi = 1; }
      else if (t.kind == Tok::Star) { lo = 0; hi = -1; }
      else if (t.kind == Tok::Plus) { lo = 1; hi = -1; }
      else if (t.kind == Tok::Repeat) { lo = t.lo; hi = t.hi; }
      else return x;
      ++i_;
      auto r = make(Ast::Rep); r->lo = lo; r->hi = hi; r->kids.push_back(std::move(x));
      x = std::move(r);
    }
  }
  AstP atom() {
    const Token t = peek();
    ++i_;
    switch (t.kind) {
      case Tok::Lit: { auto a = make(Ast::Lit); a->text = t.text; return a; }
      case Tok::Class: { auto a = make(Ast::Class); a->set = t.set; return a; }
      case Tok::Name: { auto a = make(Ast::Ref); a->text = t.text; return a; }
      case Tok::LParen: {
        AstP x = alt();
        if (peek().kind != Tok::RParen) fail(CG_E_SYNTAX, "expected )");
        ++i_;
        return x;
      }
      case Tok::Forced: {
        if (peek().kind != Tok::LParen) fail(CG_E_SYNTAX, "expected ( after @forced");
        ++i_;
        AstP x = alt();
        if (peek().kind != Tok::RParen) fail(CG_E_SYNTAX, "expected )");
        ++i_;
        auto a = make(Ast::Forced); a->kids.push_back(std::move(x)); return a;
      }
      default: fail(CG_E_SYNTAX, "unexpected token at offset " + std::to_string(t.pos));
    }
  }
};

class Expander {
 public:
  Expander(IR& ir, const std::map<std::string, AstP>& rules, uint32_t depth_max)
      : ir_(ir), rules_(rules), depth_max_(depth_max) {}

  int ref(const std::string& name) {
    auto it = rules_.find(name);
    if (it == rules_.end()) fail(CG_E_UNDEFINED_RULE, name);
    uint32_t& d = active_[name];
    if (d >= depth_max_) return ir_.empty();
    ++d;
    int r = expand(*it->second);
    --active_[name];
    return r;
  }

 private:
  IR& ir_;
  const std::map<std::string, AstP>& rules_;
  uint32_t depth_max_;
  std::map<std::string, uint32_t> active_;

  int expand(const Ast& a) {
    switch (a.k) {
      case Ast::Eps: return ir_.eps();
      case Ast::Lit: return ir_.literal(a.text);
      case Ast::Class: return ir_.sym(a.set);
      case Ast::Ref: return ref(a.text);
      case Ast::Forced: return ir_.injected(expand(*a.kids[0]));
      case Ast::Rep: return ir_.rep(expand(*a.kids[0]), a.lo, a.hi);
      case Ast::Cat: case Ast::Alt: case Ast::And: {
        std::vector<int> k;
        for (auto& c : a.kids) k.push_back(expand(*c));
        if (a.k == Ast::Cat) return ir_.cat(std::move(k));
        if (a.k == Ast::Alt) return ir_.alt(std::move(k));
        return ir_.conj(std::move(k));
      }
    }
    return ir_.empty();
  }
};

// Rules that reach themselves through references (the rules on a cycle of
// the reference graph), by a search from each rule.
void collect_refs(const Ast& a, std::vector<std::string>& out) {
  if (a.k == Ast::Ref) out.push_back(a.text);
  for (auto& c : a.kids) collect_refs(*c, out);
}

std::map<std::string, int> recursive_rule_index(const std::map<std::string, AstP>& rules) {
  std::map<std::string, std::vector<std::string>> succ;
  for (auto& [name, body] : rules) {
    collect_refs(*body, succ[name]);
    for (auto& r : succ[name]) if (!rules.count(r)) fail(CG_E_UNDEFINED_RULE, r);
  }
  std::map<std::string, int> index;
  for (auto& [name, body] : rules) {
    std::map<std::string, bool> seen;
    std::vector<std::string> stack = succ[name];
    bool cyc = false;
    while (!stack.empty() && !cyc) {
      std::string r = stack.back();
      stack.pop_back();
      if (r == name) cyc = true;
      else if (!seen[r]) { seen[r] = true; for (auto& x : succ[r]) stack.push_back(x); }
    }
    if (cyc) {
      const int j = int(index.size());
      index[name] = j;
    }
  }
  if (index.size() > size_t(kNumCallSymbols)) fail(CG_E_LIMIT, "more than 64 recursive rules");
  return index;
}

// Lowers one rule body: other rules inline, recursive rule j becomes call
// symbol 512 + j.  A call inside @forced( ) or under '&' has no meaning for a
// deterministic pushdown automaton (its bytes would be injected, or matched
// against another language as a whole) and is refused.
class CallLowerer {
 public:
  CallLowerer(IR& ir, const std::map<std::string, AstP>& rules, const std::map<std::string, int>& rec)
      : ir_(ir), rules_(rules), rec_(rec) {}

  int lower(const Ast& a, bool in_forced, bool in_and) {
    switch (a.k) {
      case Ast::Eps: return ir_.eps();
      case Ast::Lit: return ir_.literal(a.text);
      case Ast::Class: return ir_.sym(a.set);
      case Ast::Ref: {
        auto r = rec_.find(a.text);
        if (r != rec_.end()) {
          if (in_forced || in_and)
            fail(CG_E_UNSUPPORTED, "recursive rule " + a.text + " referenced inside @forced( ) or '&'");
          SymSet s;
          s.set(kNumSymbols + r->second);
          return ir_.sym(s);
        }
        return lower(*rules_.at(a.text), in_forced, in_and);  // acyclic: terminates
      }
      case Ast::Forced: return ir_.injected(lower(*a.kids[0], true, in_and));
      case Ast::Rep: return ir_.rep(lower(*a.kids[0], in_forced, in_and), a.lo, a.hi);
      case Ast::Cat: case Ast::Alt: case Ast::And: {
        std::vector<int> k;
        for (auto& c : a.kids) k.push_back(lower(*c, in_forced, in_and || a.k == Ast::And));
        if (a.k == Ast::Cat) return ir_.cat(std::move(k));
        if (a.k == Ast::Alt) return ir_.alt(std::move(k));
        return ir_.conj(std::move(k));
      }
    }
    return ir_.empty();
  }

 private:
  IR& ir_;
  const std::map<std::string, AstP>& rules_;
  const std::map<std::string, int>& rec_;
};

}  // namespace

RuleSystem lower_gbnf_rules(IR& ir, const std::string& src) {
  Parser p(lex(src));
  auto rules = p.rules();
  if (!rules.count("root")) fail(CG_E_SYNTAX, "no root rule");
  const auto rec = recursive_rule_index(rules);
  RuleSystem out;
  out.names.assign(1 + rec.size(), "");
  out.automata.assign(1 + rec.size(), -1);
  CallLowerer low(ir, rules, rec);
  out.names[0] = "root";
  out.automata[0] = low.lower(*rules.at("root"), false, false);
  for (auto& [name, j] : rec) {
    out.names[1 + j] = name;
    out.automata[1 + j] = low.lower(*rules.at(name), false, false);
  }
  return out;
}

int parse_gbnf(IR& ir, const std::string& src, uint32_t depth_max) {
  Parser p(lex(src));
  auto rules = p.rules();
  if (!rules.count("root")) fail(CG_E_SYNTAX, "no root rule");
  Expander e(ir, rules, depth_max);
  return e.ref("root");
}

}  // namespace cg
