// Pushdown compiler for recursive GBNF grammars.
//
// usetacet.com/docs/grammar, "The guarantee": the automaton that masks the
// logits at every step is a pushdown automaton.  Each rule that lies on a
// cycle of references keeps its own automaton; a reference to it is a call
// that pushes the caller's return state, and the end of its text pops it.
// The stack is bounded by `depth` frames, the same language the flattened
// grammar has when every reference to a recursive rule opens one frame and a
// reference past `depth` open frames is empty.
//
//  1. Rule automata: the start rule and every recursive rule, each a minimal
//     DFA over the 512 byte symbols plus one call symbol per recursive rule
//     (gbnf.cpp inlines the other rules).
//  2. Completion height h(q): the least number of levels above q's frame a
//     completion of q's rule needs; 0 where q may end its rule, through a call
//     max(1 + h(callee start), h(return state)).  A step is allowed only where
//     the frame's level + h of where it lands stays within `depth`, so every
//     configuration reached can still be completed (the trimmed language).
//  3. Determinism: every symbol has at most one action in every state.  The
//     consumed symbols of a state (its shifts and the first symbols of its
//     calls) must be disjoint; no recursive rule may match the empty string or
//     call itself before consuming a symbol; and where a state may end its
//     rule, no symbol it consumes may also follow the rule (else both popping
//     and consuming would be possible).  Grammars outside this class are
//     refused with CG_E_UNSUPPORTED.
//  4. Actions per (state, symbol): shift, a call chain (the calls that open
//     one after another before the symbol is consumed, with the headroom the
//     whole chain needs), or none (pop, when the rule may end here).
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <map>
#include <new>
#include <string>
#include <vector>

#include "../../../include/cg.h"
#include "../cg_internal.h"
#include "ir.h"

namespace cg {
namespace {

[[noreturn]] void fail(int code, const std::string& m) { throw CompileError{code, m}; }

constexpr int kInf = 1 << 20;

struct Bits {
  uint64_t w[8] = {};
  void set(int a) { w[a >> 6] |= uint64_t(1) << (a & 63); }
  bool test(int a) const { return (w[a >> 6] >> (a & 63)) & 1; }
  void merge(const Bits& o) { for (int i = 0; i < 8; ++i) w[i] |= o.w[i]; }
  int first_common(const Bits& o) const {
    for (int i = 0; i < 8; ++i)
      if (uint64_t x = w[i] & o.w[i]) return i * 64 + __builtin_ctzll(x);
    return -1;
  }
  bool operator==(const Bits& o) const { return std::memcmp(w, o.w, sizeof w) == 0; }
};

std::string sym_name(int c) {
  const int b = c & 255;
  std::string s = (c >= 256) ? "injected " : "";
  if (b >= 0x21 && b < 0x7F) return s + "'" + char(b) + "'";
  char buf[8];
  std::snprintf(buf, sizeof buf, "0x%02x", b);
  return s + buf;
}

cg_pda_grammar* compile(const std::string& src, uint32_t depth) {
  IR ir;
  RuleSystem rs = lower_gbnf_rules(ir, src);
  const int R = int(rs.automata.size()), K = R - 1, nsym = kNumSymbols + K;
  std::vector<Dfa> dfa(R);
  for (int r = 0; r < R; ++r) {
    try {
      dfa[r] = build_dfa(ir, rs.automata[r], nsym);
    } catch (const CompileError& e) {
      if (e.code == CG_E_EMPTY && r > 0) fail(CG_E_EMPTY, "rule " + rs.names[r] + " accepts no string");
      throw;
    }
  }
  std::vector<uint32_t> start(R);
  uint64_t S64 = 0;
  for (int r = 0; r < R; ++r) { start[r] = uint32_t(S64); S64 += dfa[r].n_states; }
  if (S64 >= (1u << 24)) fail(CG_E_LIMIT, "more than 2^24 states");
  const uint32_t S = uint32_t(S64);

  // 1. global tables: shifts over the 512 symbols, calls per recursive rule
  std::vector<int32_t> shift(size_t(S) * kNumSymbols, -1), call(size_t(S) * std::max(K, 1), -1);
  std::vector<uint32_t> rule_of(S);
  std::vector<uint8_t> acc(S);
  for (int r = 0; r < R; ++r) {
    const Dfa& d = dfa[r];
    for (uint32_t s = 0; s < d.n_states; ++s) {
      const uint32_t q = start[r] + s;
      rule_of[q] = uint32_t(r);
      acc[q] = d.accept[s];
      for (int c = 0; c < kNumSymbols; ++c) {
        const int32_t t = d.next[size_t(s) * nsym + c];
        if (t >= 0) shift[size_t(q) * kNumSymbols + c] = int32_t(start[r]) + t;
      }
      for (int j = 0; j < K; ++j) {
        const int32_t t = d.next[size_t(s) * nsym + kNumSymbols + j];
        if (t >= 0) call[size_t(q) * K + j] = int32_t(start[r]) + t;
      }
    }
  }

  // 2. completion heights (least fixpoint from "ends here" = 0)
  std::vector<int> h(S, kInf);
  for (uint32_t q = 0; q < S; ++q) if (acc[q]) h[q] = 0;
  for (bool changed = true; changed;) {
    changed = false;
    for (uint32_t q = 0; q < S; ++q) {
      int best = h[q];
      for (int c = 0; c < kNumSymbols; ++c) {
        const int32_t t = shift[size_t(q) * kNumSymbols + c];
        if (t >= 0) best = std::min(best, h[t]);
      }
      for (int j = 0; j < K; ++j) {
        const int32_t r = call[size_t(q) * K + j];
        if (r >= 0) best = std::min(best, std::max(std::min(1 + h[start[1 + j]], kInf), h[r]));
      }
      if (best < h[q]) { h[q] = best; changed = true; }
    }
  }
  if (h[0] >= kInf) fail(CG_E_EMPTY, "the grammar accepts no string");
  if (h[0] > int(depth)) fail(CG_E_EMPTY, "the grammar accepts no string within the stack bound");
  // edges into configurations that can never complete are no edges
  for (uint32_t q = 0; q < S; ++q) {
    for (int c = 0; c < kNumSymbols; ++c) {
      int32_t& t = shift[size_t(q) * kNumSymbols + c];
      if (t >= 0 && h[t] >= kInf) t = -1;
    }
    for (int j = 0; j < K; ++j) {
      int32_t& r = call[size_t(q) * K + j];
      if (r >= 0 && (h[r] >= kInf || h[start[1 + j]] >= kInf)) r = -1;
    }
  }

  // 3. determinism
  for (int j = 0; j < K; ++j)
    if (acc[start[1 + j]])
      fail(CG_E_UNSUPPORTED, "recursive rule " + rs.names[1 + j] + " matches the empty string");
  // first symbols of each recursive rule; calls made before any symbol must not cycle
  std::vector<Bits> first(K);
  std::vector<int> color(K, 0);  // 0 new, 1 on the path, 2 done
  std::vector<std::pair<int, int>> stack;
  auto first_of = [&](int j0) {
    stack.assign(1, {j0, 0});
    color[j0] = 1;
    while (!stack.empty()) {
      auto& [j, i] = stack.back();
      const uint32_t q = start[1 + j];
      if (i < K) {
        const int callee = i++;
        if (call[size_t(q) * K + callee] < 0) continue;
        if (color[callee] == 1) fail(CG_E_UNSUPPORTED, "left recursion through rule " + rs.names[1 + callee]);
        if (color[callee] == 0) { color[callee] = 1; stack.push_back({callee, 0}); }
        continue;
      }
      Bits f;
      for (int c = 0; c < kNumSymbols; ++c) if (shift[size_t(q) * kNumSymbols + c] >= 0) f.set(c);
      for (int callee = 0; callee < K; ++callee)
        if (call[size_t(q) * K + callee] >= 0) {
          const int clash = f.first_common(first[callee]);
          if (clash >= 0)
            fail(CG_E_UNSUPPORTED, "rule " + rs.names[1 + j] + " can start " + sym_name(clash) + " in two ways");
          f.merge(first[callee]);
        }
      first[j] = f;
      color[j] = 2;
      stack.pop_back();
    }
  };
  for (int j = 0; j < K; ++j) if (color[j] == 0) first_of(j);
  std::vector<Bits> cons(S);
  for (uint32_t q = 0; q < S; ++q) {
    Bits f;
    for (int c = 0; c < kNumSymbols; ++c) if (shift[size_t(q) * kNumSymbols + c] >= 0) f.set(c);
    for (int j = 0; j < K; ++j)
      if (call[size_t(q) * K + j] >= 0) {
        const int clash = f.first_common(first[j]);
        if (clash >= 0)
          fail(CG_E_UNSUPPORTED, "rule " + rs.names[rule_of[q]] + ": " + sym_name(clash) +
                                     " both continues and starts rule " + rs.names[1 + j]);
        f.merge(first[j]);
      }
    cons[q] = f;
  }
  std::vector<Bits> follow(K);
  for (bool changed = true; changed;) {
    changed = false;
    for (uint32_t p = 0; p < S; ++p)
      for (int j = 0; j < K; ++j) {
        const int32_t r = call[size_t(p) * K + j];
        if (r < 0) continue;
        Bits f = follow[j];
        f.merge(cons[r]);
        if (acc[r] && rule_of[r] > 0) f.merge(follow[rule_of[r] - 1]);
        if (!(f == follow[j])) { follow[j] = f; changed = true; }
      }
  }
  for (uint32_t q = 0; q < S; ++q) {
    if (!acc[q] || rule_of[q] == 0) continue;
    const int clash = cons[q].first_common(follow[rule_of[q] - 1]);
    if (clash >= 0)
      fail(CG_E_UNSUPPORTED, "rule " + rs.names[rule_of[q]] + " may end or continue on " + sym_name(clash));
  }

  // 4. actions per (state, symbol), call chains shared by content
  auto hv = [&](int x) { return std::min(x, int(kPdaInf)); };
  cg_pda_grammar* g = new cg_pda_grammar;
  g->depth = depth;
  g->n_states = S;
  g->rule_names = rs.names;
  g->rule_start = start;
  g->rule_of = rule_of;
  g->accept = acc;
  g->h.resize(S);
  for (uint32_t q = 0; q < S; ++q) g->h[q] = uint8_t(hv(h[q]));
  g->need_model.assign(S, kPdaInf);
  g->need_inj.assign(S, kPdaInf);
  std::vector<uint32_t> act_sym(size_t(S) * kNumSymbols, kPdaNone);
  std::map<std::vector<uint32_t>, uint32_t> chain_at;
  for (uint32_t q = 0; q < S; ++q)
    for (int c = 0; c < kNumSymbols; ++c) {
      std::vector<uint32_t> pushes;
      uint32_t cur = q;
      int target = -1;
      for (int guard = 0; guard <= K && target < 0; ++guard) {
        const int32_t t = shift[size_t(cur) * kNumSymbols + c];
        if (t >= 0) { target = t; break; }
        int via = -1;
        for (int j = 0; j < K && via < 0; ++j)
          if (call[size_t(cur) * K + j] >= 0 && first[j].test(c)) via = j;
        if (via < 0) break;
        pushes.push_back(uint32_t(call[size_t(cur) * K + via]));
        cur = start[1 + via];
      }
      if (target < 0) continue;
      int need;
      uint32_t a;
      if (pushes.empty()) {
        need = h[target];
        a = uint32_t(target);
      } else {
        need = int(pushes.size()) + h[target];
        for (size_t i = 0; i < pushes.size(); ++i) need = std::max(need, int(i) + h[pushes[i]]);
        need = hv(need);
        std::vector<uint32_t> key;
        key.push_back(uint32_t(pushes.size()) | (uint32_t(need) << 8));
        key.insert(key.end(), pushes.begin(), pushes.end());
        key.push_back(uint32_t(target));
        auto it = chain_at.find(key);
        if (it == chain_at.end()) {
          it = chain_at.emplace(key, uint32_t(g->chain.size())).first;
          g->chain.insert(g->chain.end(), key.begin(), key.end());
        }
        a = kPdaCall | it->second;
      }
      act_sym[size_t(q) * kNumSymbols + c] = a;
      uint8_t& nd = c < 256 ? g->need_model[q] : g->need_inj[q];
      nd = uint8_t(std::min<int>(nd, hv(need)));
    }
  // columns: symbols whose actions agree in every state share one
  std::map<std::vector<uint32_t>, uint16_t> col_at;
  g->col_of.assign(kNumSymbols, 0);
  std::vector<std::vector<uint32_t>> cols;
  for (int c = 0; c < kNumSymbols; ++c) {
    std::vector<uint32_t> colv(S);
    for (uint32_t q = 0; q < S; ++q) colv[q] = act_sym[size_t(q) * kNumSymbols + c];
    auto it = col_at.find(colv);
    if (it == col_at.end()) {
      it = col_at.emplace(colv, uint16_t(cols.size())).first;
      cols.push_back(colv);
    }
    g->col_of[c] = it->second;
  }
  g->n_cols = uint32_t(cols.size());
  g->returns_of.assign(R, {});
  for (uint32_t q = 0; q < S; ++q)
    for (int j = 0; j < K; ++j) {
      const int32_t r = call[size_t(q) * K + j];
      auto& v = g->returns_of[1 + j];
      if (r >= 0 && std::find(v.begin(), v.end(), uint32_t(r)) == v.end()) v.push_back(uint32_t(r));
    }
  g->act.assign(size_t(S) * g->n_cols, kPdaNone);
  for (uint32_t k = 0; k < g->n_cols; ++k)
    for (uint32_t q = 0; q < S; ++q) g->act[size_t(q) * g->n_cols + k] = cols[k][q];
  return g;
}

// One symbol from configuration (cur, stack): pops while the rule may end
// and the symbol has no action, then shifts or runs the call chain.  With
// depth >= 0 the headroom checks are enforced against it; with depth < 0
// (token walks relative to an unknown stack) `need` collects the largest
// level + requirement and a pop below `floor` returns kPdaTokPop.
uint32_t step_symbol(const cg_pda_grammar& g, uint32_t& cur, std::vector<uint32_t>& st, int c, long depth,
                     uint32_t& need) {
  for (;;) {
    const uint32_t a = g.act[size_t(cur) * g.n_cols + g.col_of[c]];
    const uint32_t lvl = uint32_t(st.size());
    if (a == kPdaNone) {
      if (!g.accept[cur]) return kPdaTokDead;
      if (st.empty()) return depth < 0 ? kPdaTokPop : kPdaTokDead;
      cur = st.back();
      st.pop_back();
      continue;
    }
    uint32_t req, target;
    if (a & kPdaCall) {
      const uint32_t o = a & ~kPdaCall, n = g.chain[o] & 0xFFu;
      req = g.chain[o] >> 8;
      if (depth >= 0 && lvl + req > uint32_t(depth)) return kPdaTokDead;
      for (uint32_t i = 0; i < n; ++i) st.push_back(g.chain[o + 1 + i]);
      target = g.chain[o + 1 + n];
    } else {
      req = g.h[a];
      if (depth >= 0 && lvl + req > uint32_t(depth)) return kPdaTokDead;
      target = a;
    }
    if (req >= kPdaInf) return kPdaTokDead;
    need = std::max(need, lvl + req);
    cur = target;
    return 0;
  }
}

}  // namespace

namespace {
// Can bytes[i..n) be walked from state q, its frame's caller being any of
// the return states the grammar pushes below q's rule (and so on below),
// with no bound on the stack?  `hops` counts pops taken at byte i without
// consuming it: more than the number of states means a cycle of pops.
bool survives_some_stack(const cg_pda_grammar& g, uint32_t q, const uint8_t* bytes, uint32_t i, uint32_t n,
                         uint32_t hops) {
  std::vector<uint32_t> st;
  uint32_t need = 0;
  for (; i < n; ++i, hops = 0) {
    const uint32_t r = step_symbol(g, q, st, bytes[i], -1, need);
    if (r == kPdaTokDead) return false;
    if (r == kPdaTokPop) {
      const uint32_t rule = g.rule_of[q];
      if (rule == 0 || hops > g.n_states) return false;
      for (uint32_t ret : g.returns_of[rule])
        if (survives_some_stack(g, ret, bytes, i, n, hops + 1)) return true;
      return false;
    }
  }
  return true;
}
}  // namespace

uint32_t pda_token_need(const cg_pda_grammar& g, uint32_t q, const uint8_t* bytes, uint32_t n) {
  std::vector<uint32_t> st;
  uint32_t cur = q, need = 0;
  for (uint32_t i = 0; i < n; ++i) {
    const uint32_t r = step_symbol(g, cur, st, bytes[i], -1, need);
    if (r == kPdaTokPop) {
      // the start rule is the base frame: nothing lies below it
      const uint32_t rule = g.rule_of[cur];
      if (rule == 0) return kPdaTokDead;
      for (uint32_t ret : g.returns_of[rule])
        if (survives_some_stack(g, ret, bytes, i, n, 1)) return kPdaTokPop;
      return kPdaTokDead;
    }
    if (r) return r;
  }
  return need;
}

}  // namespace cg

extern "C" {

int cg_pda_compile(const char* src, size_t src_len, uint32_t depth, cg_pda_grammar** out) {
  if (!src || !out || depth > CG_PDA_MAX_DEPTH) return CG_E_ARG;
  *out = nullptr;
  try {
    *out = cg::compile(std::string(src, src_len), depth);
    return CG_OK;
  } catch (const cg::CompileError& e) {
    return e.code;
  } catch (const std::bad_alloc&) {
    return CG_E_NOMEM;
  }
}

void cg_pda_grammar_destroy(cg_pda_grammar* g) { delete g; }

int cg_pda_grammar_info(const cg_pda_grammar* g, uint32_t* n_states, uint32_t* n_rules, uint32_t* n_cols,
                        uint32_t* depth) {
  if (!g) return CG_E_ARG;
  if (n_states) *n_states = g->n_states;
  if (n_rules) *n_rules = uint32_t(g->rule_names.size());
  if (n_cols) *n_cols = g->n_cols;
  if (depth) *depth = g->depth;
  return CG_OK;
}

int cg_pda_try_input(const cg_pda_grammar* g, const uint8_t* s, size_t n, const uint8_t* injected,
                     size_t* consumed, int* accepted, uint32_t* level) {
  if (!g || (!s && n) || !consumed || !accepted) return CG_E_ARG;
  try {
    std::vector<uint32_t> st;
    uint32_t cur = 0, need = 0;
    size_t i = 0;
    for (; i < n; ++i) {
      const int c = s[i] + ((injected && injected[i]) ? 256 : 0);
      if (cg::step_symbol(*g, cur, st, c, long(g->depth), need)) break;
    }
    *consumed = i;
    bool complete = i == n && g->accept[cur];
    for (size_t k = 0; complete && k < st.size(); ++k) complete = g->accept[st[k]];
    *accepted = complete ? 1 : 0;
    if (level) *level = uint32_t(st.size());
    return CG_OK;
  } catch (const std::bad_alloc&) {
    return CG_E_NOMEM;
  }
}

}  // extern "C"
