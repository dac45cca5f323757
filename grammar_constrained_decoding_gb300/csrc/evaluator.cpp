// Host side of evaluator-aware decoding: an exact arithmetic evaluator, a
// string-operation evaluator, the result formatting the host injects, and the
// per-row forced-token driver (labs.miniml.ai "Evaluator aware decoding": "The
// core idea" steps 1-4, "A concrete prototype on llama.cpp", "Not just
// arithmetic: string operations").
//
// Values are exact rationals num/den over arbitrary-precision integers; a
// span longer than 4096 bytes is refused as overflow (evaluators must stay
// time bounded, same page, "Where XGrammar-2 could take this").
#include <algorithm>
#include <cstring>
#include <string>
#include <vector>

#include "cg_internal.h"

namespace {

// ---------------------------------------------------------------- big integers
struct Big {
  bool neg = false;
  std::vector<uint32_t> m;  // little-endian base 2^32, no leading zero limbs

  bool zero() const { return m.empty(); }
  void trim() { while (!m.empty() && m.back() == 0) m.pop_back(); if (m.empty()) neg = false; }
};

int cmp_mag(const std::vector<uint32_t>& a, const std::vector<uint32_t>& b) {
  if (a.size() != b.size()) return a.size() < b.size() ? -1 : 1;
  for (size_t i = a.size(); i-- > 0;)
    if (a[i] != b[i]) return a[i] < b[i] ? -1 : 1;
  return 0;
}

std::vector<uint32_t> add_mag(const std::vector<uint32_t>& a, const std::vector<uint32_t>& b) {
  std::vector<uint32_t> r(std::max(a.size(), b.size()) + 1, 0);
  uint64_t carry = 0;
  for (size_t i = 0; i < r.size(); ++i) {
    uint64_t s = carry;
    if (i < a.size()) s += a[i];
    if (i < b.size()) s += b[i];
    r[i] = uint32_t(s);
    carry = s >> 32;
  }
  while (!r.empty() && r.back() == 0) r.pop_back();
  return r;
}

// a - b with |a| >= |b|
std::vector<uint32_t> sub_mag(const std::vector<uint32_t>& a, const std::vector<uint32_t>& b) {
  std::vector<uint32_t> r(a.size(), 0);
  int64_t borrow = 0;
  for (size_t i = 0; i < a.size(); ++i) {
    int64_t d = int64_t(a[i]) - borrow - (i < b.size() ? int64_t(b[i]) : 0);
    borrow = d < 0;
    r[i] = uint32_t(d + (borrow ? (int64_t(1) << 32) : 0));
  }
  while (!r.empty() && r.back() == 0) r.pop_back();
  return r;
}

Big add(const Big& a, const Big& b) {
  Big r;
  if (a.neg == b.neg) { r.m = add_mag(a.m, b.m); r.neg = a.neg; }
  else if (cmp_mag(a.m, b.m) >= 0) { r.m = sub_mag(a.m, b.m); r.neg = a.neg; }
  else { r.m = sub_mag(b.m, a.m); r.neg = b.neg; }
  r.trim();
  return r;
}

Big neg(Big a) { if (!a.zero()) a.neg = !a.neg; return a; }

Big mul(const Big& a, const Big& b) {
  Big r;
  if (a.zero() || b.zero()) return r;
  r.m.assign(a.m.size() + b.m.size(), 0);
  for (size_t i = 0; i < a.m.size(); ++i) {
    uint64_t carry = 0;
    for (size_t j = 0; j < b.m.size(); ++j) {
      uint64_t t = uint64_t(a.m[i]) * b.m[j] + r.m[i + j] + carry;
      r.m[i + j] = uint32_t(t);
      carry = t >> 32;
    }
    size_t k = i + b.m.size();
    while (carry) { uint64_t t = uint64_t(r.m[k]) + carry; r.m[k] = uint32_t(t); carry = t >> 32; ++k; }
  }
  r.neg = a.neg != b.neg;
  r.trim();
  return r;
}

// |a| = q*|b| + rem, bitwise long division (b nonzero)
void divmod_mag(const std::vector<uint32_t>& a, const std::vector<uint32_t>& b, std::vector<uint32_t>& q,
                std::vector<uint32_t>& rem) {
  q.assign(a.size(), 0);
  rem.clear();
  for (size_t bit = a.size() * 32; bit-- > 0;) {
    // rem = rem*2 + bit
    uint32_t carry = (a[bit / 32] >> (bit % 32)) & 1;
    for (auto& limb : rem) { uint32_t nc = limb >> 31; limb = (limb << 1) | carry; carry = nc; }
    if (carry) rem.push_back(carry);
    if (cmp_mag(rem, b) >= 0) { rem = sub_mag(rem, b); q[bit / 32] |= 1u << (bit % 32); }
  }
  while (!q.empty() && q.back() == 0) q.pop_back();
}

Big from_decimal(const std::string& digits) {
  Big r;
  Big ten; ten.m = {10};
  for (char c : digits) {
    r = mul(r, ten);
    Big d; if (c != '0') d.m = {uint32_t(c - '0')};
    r = add(r, d);
  }
  return r;
}

std::string to_decimal(const Big& a) {
  if (a.zero()) return "0";
  std::vector<uint32_t> cur = a.m, q, rem;
  std::vector<uint32_t> billion = {1000000000u};
  std::vector<uint32_t> chunks;
  while (!cur.empty()) {
    divmod_mag(cur, billion, q, rem);
    chunks.push_back(rem.empty() ? 0 : rem[0]);
    cur = q;
  }
  std::string s = std::to_string(chunks.back());
  for (size_t i = chunks.size() - 1; i-- > 0;) {
    std::string part = std::to_string(chunks[i]);
    s += std::string(9 - part.size(), '0') + part;
  }
  return a.neg ? "-" + s : s;
}

struct Rat {
  Big num, den;  // den > 0
};

Rat make_int(const Big& b) { Rat r; r.num = b; r.den.m = {1}; return r; }

struct EvalFail { const char* code; };

// Lexing runs over the whole span first, so a byte outside the language is a
// parse error whatever the arithmetic before it would have done.
struct Lexeme {
  char op;   // 0 for a number
  Rat value;
};

std::vector<Lexeme> lex(const std::string& s) {
  std::vector<Lexeme> out;
  size_t i = 0, n = s.size();
  while (i < n) {
    char c = s[i];
    if (c == ' ') { ++i; continue; }
    if (c == '+' || c == '-' || c == '*' || c == '/' || c == '(' || c == ')') {
      out.push_back({c, Rat{}});
      ++i;
      continue;
    }
    if ((c >= '0' && c <= '9') || c == '.') {
      std::string ip, fp;
      while (i < n && s[i] >= '0' && s[i] <= '9') ip.push_back(s[i++]);
      if (i < n && s[i] == '.') {
        ++i;
        while (i < n && s[i] >= '0' && s[i] <= '9') fp.push_back(s[i++]);
        if (ip.empty() && fp.empty()) throw EvalFail{"parse"};
      } else if (ip.empty()) {
        throw EvalFail{"parse"};
      }
      Rat r;
      r.num = from_decimal(ip + fp);
      r.den = from_decimal("1" + std::string(fp.size(), '0'));
      out.push_back({0, r});
      continue;
    }
    throw EvalFail{"parse"};
  }
  return out;
}

class Evaluator {
 public:
  explicit Evaluator(const std::string& s) : t_(lex(s)) {}

  Big run() {
    if (t_.empty()) throw EvalFail{"parse"};
    Rat v = expr();
    if (i_ != t_.size()) throw EvalFail{"parse"};
    std::vector<uint32_t> q, rem;
    divmod_mag(v.num.m, v.den.m, q, rem);
    if (!rem.empty()) throw EvalFail{"non_integer"};
    Big r; r.m = q; r.neg = v.num.neg; r.trim();
    std::string d = to_decimal(r);
    if (d.size() - (r.neg ? 1 : 0) > 64) throw EvalFail{"overflow"};
    return r;
  }

 private:
  std::vector<Lexeme> t_;
  size_t i_ = 0;

  char peek() const { return i_ < t_.size() ? (t_[i_].op ? t_[i_].op : '0') : 0; }

  Rat expr() {
    Rat v = term();
    for (;;) {
      char c = peek();
      if (c != '+' && c != '-') return v;
      ++i_;
      Rat w = term();
      if (c == '-') w.num = neg(w.num);
      v.num = add(mul(v.num, w.den), mul(w.num, v.den));
      v.den = mul(v.den, w.den);
    }
  }
  Rat term() {
    Rat v = unary();
    for (;;) {
      char c = peek();
      if (c != '*' && c != '/') return v;
      ++i_;
      Rat w = unary();
      if (c == '*') {
        v.num = mul(v.num, w.num);
        v.den = mul(v.den, w.den);
      } else {
        if (w.num.zero()) throw EvalFail{"div_zero"};
        Big n = mul(v.num, w.den), d = mul(v.den, w.num);
        n.neg = (n.neg != d.neg) && !n.zero();
        d.neg = false;
        v.num = n;
        v.den = d;
      }
    }
  }
  Rat unary() {
    if (peek() == '-') { ++i_; Rat v = unary(); v.num = neg(v.num); return v; }
    return primary();
  }
  Rat primary() {
    char c = peek();
    if (c == '0') return t_[i_++].value;
    if (c == '(') {
      ++i_;
      Rat v = expr();
      if (peek() != ')') throw EvalFail{"parse"};
      ++i_;
      return v;
    }
    throw EvalFail{"parse"};
  }
};

// ------------------------------------------------------------- string operations
// Span: NAME '(' ARG (',' ARG)* ')' with spaces around the pieces; ARG is a
// string literal "..." (escapes \" and \\ only) or an integer -?[0-9]{1,9}.
// count(s, sub) non-overlapping occurrences left to right (sub not empty),
// len(s) bytes, reverse(s), upper(s) (ASCII a-z), substr(s, i, j) the slice
// [i, j) with negative indices from the end, both clamped to [0, len].  Strings
// are bytes.  Results over 64 bytes are "overflow"; a result holding '<'
// (which would end the result tag) is "bad_char".
struct StrArg {
  bool is_str = false;
  std::string s;
  long long v = 0;
};

std::string eval_strop(const std::string& span) {
  if (span.size() > 4096) throw EvalFail{"overflow"};
  const size_t n = span.size();
  size_t i = 0;
  auto at = [&](size_t k) { return static_cast<unsigned char>(span[k]); };
  auto skip = [&]() { while (i < n && at(i) == ' ') ++i; };
  skip();
  const size_t name0 = i;
  while (i < n && at(i) >= 'a' && at(i) <= 'z') ++i;
  const std::string name = span.substr(name0, i - name0);
  if (name.empty()) throw EvalFail{"parse"};
  skip();
  if (i >= n || at(i) != '(') throw EvalFail{"parse"};
  ++i;
  std::vector<StrArg> args;
  for (;;) {
    skip();
    StrArg a;
    if (i < n && at(i) == '"') {
      a.is_str = true;
      ++i;
      for (;;) {
        if (i >= n) throw EvalFail{"parse"};
        const unsigned char ch = at(i);
        if (ch == '"') { ++i; break; }
        if (ch == '\\') {
          if (i + 1 >= n || (at(i + 1) != '"' && at(i + 1) != '\\')) throw EvalFail{"parse"};
          a.s.push_back(span[i + 1]);
          i += 2;
          continue;
        }
        a.s.push_back(span[i]);
        ++i;
      }
    } else {
      const bool neg = i < n && at(i) == '-';
      const size_t d0 = neg ? i + 1 : i;
      size_t d = d0;
      while (d < n && at(d) >= '0' && at(d) <= '9') ++d;
      if (d == d0 || d - d0 > 9) throw EvalFail{"parse"};
      long long v = 0;
      for (size_t k = d0; k < d; ++k) v = v * 10 + (at(k) - '0');
      a.v = neg ? -v : v;
      i = d;
    }
    args.push_back(std::move(a));
    skip();
    if (i < n && at(i) == ',') { ++i; continue; }
    if (i < n && at(i) == ')') { ++i; break; }
    throw EvalFail{"parse"};
  }
  skip();
  if (i != n) throw EvalFail{"parse"};
  auto kinds = [&](const char* k) {  // 's' string, 'i' integer, one letter per argument
    const size_t m = std::strlen(k);
    if (args.size() != m) return false;
    for (size_t q = 0; q < m; ++q)
      if (args[q].is_str != (k[q] == 's')) return false;
    return true;
  };
  std::string out;
  if (name == "count") {
    if (!kinds("ss")) throw EvalFail{"arity"};
    const std::string& h = args[0].s;
    const std::string& nd = args[1].s;
    if (nd.empty()) throw EvalFail{"empty"};
    size_t c = 0;
    for (size_t p = 0; p + nd.size() <= h.size();) {
      if (h.compare(p, nd.size(), nd) == 0) { ++c; p += nd.size(); } else { ++p; }
    }
    out = std::to_string(c);
  } else if (name == "len") {
    if (!kinds("s")) throw EvalFail{"arity"};
    out = std::to_string(args[0].s.size());
  } else if (name == "reverse") {
    if (!kinds("s")) throw EvalFail{"arity"};
    out.assign(args[0].s.rbegin(), args[0].s.rend());
  } else if (name == "upper") {
    if (!kinds("s")) throw EvalFail{"arity"};
    out = args[0].s;
    for (char& ch : out) {
      const unsigned char u = static_cast<unsigned char>(ch);
      if (u >= 'a' && u <= 'z') ch = char(u - 32);
    }
  } else if (name == "substr") {
    if (!kinds("sii")) throw EvalFail{"arity"};
    const long long L = static_cast<long long>(args[0].s.size());
    auto clamp = [&](long long x) { if (x < 0) x += L; return std::min(std::max(x, 0LL), L); };
    const long long a = clamp(args[1].v), b = clamp(args[2].v);
    if (a < b) out = args[0].s.substr(size_t(a), size_t(b - a));
  } else {
    throw EvalFail{"unknown_op"};
  }
  if (out.size() > 64) throw EvalFail{"overflow"};
  if (out.find('<') != std::string::npos) throw EvalFail{"bad_char"};
  return out;
}

bool put(uint8_t* out, size_t cap, size_t* out_len, const std::string& s) {
  *out_len = s.size();
  if (!out || s.size() > cap) return false;
  std::memcpy(out, s.data(), s.size());
  return true;
}

std::string format(const std::string& value, bool ok, int fmt) {
  if (fmt == CG_RESULT_CALC_TAG || fmt == CG_RESULT_STROP_TAG)
    return ok ? "<result>" + value + "</result>" : "<result_error>" + value + "</result_error>";
  return ok ? ", \"answer\": " + value + "}" : ", \"answer\": null, \"error\": \"" + value + "\"}";
}

std::string evaluate_and_format(const std::string& span, bool found, int fmt, bool* ok_out) {
  std::string value;
  bool ok = false;
  try {
    if (!found) throw EvalFail{"parse"};
    if (fmt == CG_RESULT_STROP_TAG) {
      value = eval_strop(span);
    } else {
      if (span.size() > 4096) throw EvalFail{"overflow"};
      value = to_decimal(Evaluator(span).run());
    }
    ok = true;
  } catch (const EvalFail& f) {
    value = f.code;
  }
  if (ok_out) *ok_out = ok;
  return format(value, ok, fmt);
}

}  // namespace

extern "C" {

int cg_eval_arith(const uint8_t* span, size_t n, int fmt, uint8_t* out, size_t cap, size_t* out_len, int* ok) {
  if ((!span && n) || !out_len) return CG_E_ARG;
  if (fmt != CG_RESULT_CALC_TAG && fmt != CG_RESULT_JSON_ANSWER) return CG_E_ARG;
  bool good = false;
  std::string s = evaluate_and_format(std::string(reinterpret_cast<const char*>(span), n), true, fmt, &good);
  if (ok) *ok = good ? 1 : 0;
  return put(out, cap, out_len, s) ? CG_OK : CG_E_LIMIT;
}

int cg_eval_strop(const uint8_t* span, size_t n, uint8_t* out, size_t cap, size_t* out_len, int* ok) {
  if ((!span && n) || !out_len) return CG_E_ARG;
  bool good = false;
  std::string s = evaluate_and_format(std::string(reinterpret_cast<const char*>(span), n), true, CG_RESULT_STROP_TAG,
                                      &good);
  if (ok) *ok = good ? 1 : 0;
  return put(out, cap, out_len, s) ? CG_OK : CG_E_LIMIT;
}

int cg_driver_create(const cg_vocab* v, uint32_t B, const uint16_t* h_gid, const cg_span_rule* rules,
                     uint32_t n_rules, cg_driver** out) {
  if (!v || !out || !rules || n_rules == 0) return CG_E_ARG;
  auto* d = new cg_driver;
  d->vocab = v;
  d->B = B;
  d->gid.assign(B, 0);
  for (uint32_t b = 0; b < B; ++b) {
    d->gid[b] = h_gid ? h_gid[b] : 0;
    if (d->gid[b] >= n_rules) { delete d; return CG_E_ARG; }
  }
  for (uint32_t r = 0; r < n_rules; ++r) {
    cg_driver::Rule rule;
    rule.open.assign(reinterpret_cast<const char*>(rules[r].span_open), rules[r].span_open_len);
    rule.close.assign(reinterpret_cast<const char*>(rules[r].span_close), rules[r].span_close_len);
    rule.fmt = rules[r].result_format;
    d->rules.push_back(rule);
  }
  d->text.assign(B, std::string());
  d->queue.assign(B, std::deque<uint32_t>());
  *out = d;
  return CG_OK;
}

void cg_driver_destroy(cg_driver* d) { delete d; }

int cg_driver_update(cg_driver* d, const uint32_t* h_toks, const uint8_t* h_flags, const int32_t* h_forced_used,
                     int32_t* h_forced_next, uint32_t* n_evals) {
  if (!d || !h_toks || !h_flags || !h_forced_next) return CG_E_ARG;
  const cg_vocab* v = d->vocab;
  uint32_t evals = 0;
  for (uint32_t b = 0; b < d->B; ++b) {
    uint32_t tok = h_toks[b];
    uint8_t fl = h_flags[b];
    auto& q = d->queue[b];
    auto& text = d->text[b];
    if (h_forced_used && h_forced_used[b] >= 0 && tok == uint32_t(h_forced_used[b]) && !q.empty()) q.pop_front();
    if (tok != CG_NO_TOKEN) {
      if (tok >= v->V) return CG_E_ARG;
      // only a row whose grammar evaluates spans needs its text
      if (d->rules[d->gid[b]].fmt >= 0)
        text.append(reinterpret_cast<const char*>(v->bytes.data() + v->off[tok]), v->off[tok + 1] - v->off[tok]);
    }
    if (fl & (CG_FLAG_DONE | CG_FLAG_CAPPED)) {
      text.clear();
      q.clear();
    } else if ((fl & CG_FLAG_FORCED_NEXT) && q.empty()) {
      const auto& rule = d->rules[d->gid[b]];
      if (rule.fmt < 0) return CG_E_ARG;
      if (text.size() < rule.close.size() ||
          text.compare(text.size() - rule.close.size(), rule.close.size(), rule.close) != 0)
        return CG_E_ARG;
      size_t end = text.size() - rule.close.size();
      size_t start = std::string::npos;
      if (end >= rule.open.size()) {
        // last occurrence of open that ends at or before `end`
        for (size_t p = end - rule.open.size() + 1; p-- > 0;) {
          if (text.compare(p, rule.open.size(), rule.open) == 0) { start = p; break; }
        }
      }
      bool found = start != std::string::npos;
      std::string span = found ? text.substr(start + rule.open.size(), end - start - rule.open.size()) : std::string();
      std::string inject = evaluate_and_format(span, found, rule.fmt, nullptr);
      size_t need = 0;
      std::vector<uint32_t> ids(inject.size() + 1);
      int rc = cg_tokenize_greedy(v, reinterpret_cast<const uint8_t*>(inject.data()), inject.size(), ids.data(),
                                  ids.size(), &need);
      if (rc != CG_OK) return rc;
      for (size_t k = 0; k < need; ++k) q.push_back(ids[k]);
      ++evals;
    }
    h_forced_next[b] = q.empty() ? -1 : int32_t(q.front());
  }
  if (n_evals) *n_evals = evals;
  return CG_OK;
}

}  // extern "C"
