// Regular expression -> minimal trimmed DFA with canonical numbering.
//
//  1. Alphabet classes: the symbols (512, plus call symbols for the pushdown
//     compiler) are partitioned so that every symbol set of the IR is a union
//     of classes.
//  2. Thompson-style NFA over classes.  Bounded repetition x{m,n} is m copies
//     followed by n-m optional copies, each of which may exit to the end;
//     x{m,} loops.  An intersection is built as the product of its operands'
//     DFAs, minimised, and embedded as an NFA fragment.
//  3. Subset construction (epsilon closures keyed by their sorted member list).
//  4. Trimming: states that cannot reach acceptance are dropped (DEAD).
//  5. Hopcroft partition refinement on the completed automaton.
//  6. Canonical numbering: breadth-first from the start state, symbols in
//     order.  The minimal trimmed automaton is unique up to renaming, so
//     this numbering is unique.
#include <algorithm>
#include <cstring>
#include <functional>
#include <unordered_map>

#include "../../../include/cg.h"
#include "ir.h"

namespace cg {
namespace {

constexpr uint32_t kMaxStates = 1u << 24;

[[noreturn]] void fail(int code, const std::string& m) { throw CompileError{code, m}; }

struct VecHash {
  size_t operator()(const std::vector<int>& v) const {
    uint64_t h = 1469598103934665603ull;
    for (int x : v) { h ^= uint64_t(uint32_t(x)); h *= 1099511628211ull; h ^= h >> 29; }
    return size_t(h);
  }
};

// Partition of the alphabet induced by the IR's symbol sets.
struct Classes {
  int n = 0;
  std::vector<int> of_symbol;                       // [n_sym]
  std::vector<std::vector<uint16_t>> members_of_set;  // per distinct set: its classes
  std::unordered_map<int, int> set_index;           // IR node -> distinct set index
};

Classes make_classes(const IR& ir, int root, int n_sym) {
  std::vector<int> stack = {root};
  std::vector<char> seen(ir.nodes.size(), 0);
  std::vector<int> sym_nodes;
  while (!stack.empty()) {
    int x = stack.back();
    stack.pop_back();
    if (seen[x]) continue;
    seen[x] = 1;
    const Node& n = ir.nodes[x];
    if (n.kind == NodeKind::Sym) sym_nodes.push_back(x);
    for (int k : n.kids) stack.push_back(k);
  }
  Classes c;
  c.of_symbol.assign(n_sym, 0);
  c.n = 1;
  std::vector<SymSet> distinct;
  for (int x : sym_nodes) {
    const SymSet& s = ir.nodes[x].set;
    int idx = -1;
    for (size_t i = 0; i < distinct.size(); ++i) if (distinct[i] == s) { idx = int(i); break; }
    if (idx < 0) { idx = int(distinct.size()); distinct.push_back(s); }
    c.set_index[x] = idx;
  }
  for (const SymSet& s : distinct) {
    // split every class into (inside s) and (outside s)
    std::vector<int> remap_in(c.n, -1), remap_out(c.n, -1);
    int next_id = 0;
    std::vector<int> fresh(n_sym);
    for (int a = 0; a < n_sym; ++a) {
      int old = c.of_symbol[a];
      int& slot = s.test(a) ? remap_in[old] : remap_out[old];
      if (slot < 0) slot = next_id++;
      fresh[a] = slot;
    }
    c.of_symbol = fresh;
    c.n = next_id;
  }
  c.members_of_set.resize(distinct.size());
  for (size_t i = 0; i < distinct.size(); ++i) {
    std::vector<char> has(c.n, 0);
    for (int a = 0; a < n_sym; ++a) if (distinct[i].test(a)) has[c.of_symbol[a]] = 1;
    for (int k = 0; k < c.n; ++k) if (has[k]) c.members_of_set[i].push_back(uint16_t(k));
  }
  return c;
}

// Complete or partial DFA over classes.
struct ClassDfa {
  int n_cls = 0;
  int start = 0;
  std::vector<int> trans;     // [n * n_cls], -1 = none
  std::vector<uint8_t> acc;
  int size() const { return int(acc.size()); }
};

struct Nfa {
  std::vector<std::vector<int>> eps;
  // symbol edges: (list of classes, target)
  std::vector<std::vector<std::pair<const std::vector<uint16_t>*, int>>> edges;
  int add() {
    eps.emplace_back();
    edges.emplace_back();
    if (eps.size() > size_t(64) * kMaxStates) fail(CG_E_LIMIT, "NFA too large");
    return int(eps.size()) - 1;
  }
};

class Builder {
 public:
  Builder(const IR& ir, const Classes& cls) : ir_(ir), cls_(cls) {
    singles_.resize(cls.n);
    for (int k = 0; k < cls.n; ++k) singles_[k] = {uint16_t(k)};
  }

  ClassDfa dfa_of(int root) {
    Nfa nfa;
    auto [s, t] = build(nfa, root);
    return determinise(nfa, s, t);
  }

 private:
  const IR& ir_;
  const Classes& cls_;
  std::vector<std::vector<uint16_t>> singles_;
  std::unordered_map<int, ClassDfa> and_cache_;

  std::pair<int, int> build(Nfa& nfa, int x) {
    const Node& n = ir_.nodes[x];
    switch (n.kind) {
      case NodeKind::Empty: { int s = nfa.add(), t = nfa.add(); return {s, t}; }
      case NodeKind::Eps: { int s = nfa.add(), t = nfa.add(); nfa.eps[s].push_back(t); return {s, t}; }
      case NodeKind::Sym: {
        int s = nfa.add(), t = nfa.add();
        nfa.edges[s].push_back({&cls_.members_of_set[cls_.set_index.at(x)], t});
        return {s, t};
      }
      case NodeKind::Cat: {
        int s = nfa.add(), cur = s;
        for (int k : n.kids) {
          auto f = build(nfa, k);
          nfa.eps[cur].push_back(f.first);
          cur = f.second;
        }
        return {s, cur};
      }
      case NodeKind::Alt: {
        int s = nfa.add(), t = nfa.add();
        for (int k : n.kids) {
          auto f = build(nfa, k);
          nfa.eps[s].push_back(f.first);
          nfa.eps[f.second].push_back(t);
        }
        return {s, t};
      }
      case NodeKind::Rep: {
        int body = n.kids[0];
        int s = nfa.add(), cur = s;
        for (int i = 0; i < n.lo; ++i) {
          auto f = build(nfa, body);
          nfa.eps[cur].push_back(f.first);
          cur = f.second;
        }
        if (n.hi < 0) {
          int loop = nfa.add(), t = nfa.add();
          nfa.eps[cur].push_back(loop);
          auto f = build(nfa, body);
          nfa.eps[loop].push_back(f.first);
          nfa.eps[f.second].push_back(loop);
          nfa.eps[loop].push_back(t);
          return {s, t};
        }
        int t = nfa.add();
        nfa.eps[cur].push_back(t);
        for (int i = n.lo; i < n.hi; ++i) {
          auto f = build(nfa, body);
          nfa.eps[cur].push_back(f.first);
          cur = f.second;
          nfa.eps[cur].push_back(t);
        }
        return {s, t};
      }
      case NodeKind::And: {
        auto it = and_cache_.find(x);
        if (it == and_cache_.end()) it = and_cache_.emplace(x, intersection(n.kids)).first;
        const ClassDfa& d = it->second;
        std::vector<int> id(d.size());
        for (int q = 0; q < d.size(); ++q) id[q] = nfa.add();
        int t = nfa.add();
        for (int q = 0; q < d.size(); ++q) {
          for (int c = 0; c < d.n_cls; ++c) {
            int r = d.trans[size_t(q) * d.n_cls + c];
            if (r >= 0) nfa.edges[id[q]].push_back({&singles_[c], id[r]});
          }
          if (d.acc[q]) nfa.eps[id[q]].push_back(t);
        }
        if (d.size() == 0) { int s = nfa.add(); return {s, t}; }
        return {id[d.start], t};
      }
    }
    fail(CG_E_SYNTAX, "bad IR node");
  }

  ClassDfa intersection(const std::vector<int>& kids);

 public:
  ClassDfa determinise(const Nfa& nfa, int start, int final_state);
};

// epsilon closure restricted to "kernel" states (with symbol edges, or final)
void closure(const Nfa& nfa, std::vector<int>& set, int final_state, std::vector<int>& mark, int stamp,
             std::vector<int>& out) {
  out.clear();
  std::vector<int> stack(set.begin(), set.end());
  for (int s : set) mark[s] = stamp;
  while (!stack.empty()) {
    int s = stack.back();
    stack.pop_back();
    if (!nfa.edges[s].empty() || s == final_state) out.push_back(s);
    for (int t : nfa.eps[s]) if (mark[t] != stamp) { mark[t] = stamp; stack.push_back(t); }
  }
  std::sort(out.begin(), out.end());
}

ClassDfa Builder::determinise(const Nfa& nfa, int start, int final_state) {
  ClassDfa d;
  d.n_cls = cls_.n;
  std::unordered_map<std::vector<int>, int, VecHash> index;
  std::vector<std::vector<int>> sets;
  std::vector<int> mark(nfa.eps.size(), -1);
  int stamp = 0;
  std::vector<int> seed = {start}, cl;
  closure(nfa, seed, final_state, mark, stamp++, cl);
  index.emplace(cl, 0);
  sets.push_back(cl);
  std::vector<std::vector<int>> moves(cls_.n);
  std::vector<int> touched;
  for (size_t i = 0; i < sets.size(); ++i) {
    if (sets.size() > kMaxStates) fail(CG_E_LIMIT, "automaton too large");
    touched.clear();
    const std::vector<int> cur = sets[i];
    for (int s : cur) {
      for (auto& e : nfa.edges[s]) {
        for (uint16_t c : *e.first) {
          if (moves[c].empty()) touched.push_back(c);
          moves[c].push_back(e.second);
        }
      }
    }
    d.trans.resize((i + 1) * size_t(cls_.n), -1);
    for (int c : touched) {
      closure(nfa, moves[c], final_state, mark, stamp++, cl);
      moves[c].clear();
      if (cl.empty()) continue;
      auto it = index.find(cl);
      int id;
      if (it == index.end()) {
        id = int(sets.size());
        index.emplace(cl, id);
        sets.push_back(cl);
      } else {
        id = it->second;
      }
      d.trans[i * size_t(cls_.n) + c] = id;
    }
  }
  d.acc.resize(sets.size());
  for (size_t i = 0; i < sets.size(); ++i)
    d.acc[i] = std::binary_search(sets[i].begin(), sets[i].end(), final_state) ? 1 : 0;
  d.start = 0;
  return d;
}

// Drop states that cannot reach acceptance; returns the trimmed automaton
// (possibly empty: size() == 0).
ClassDfa trim(const ClassDfa& d) {
  int n = d.size(), C = d.n_cls;
  std::vector<std::vector<int>> preds(n);
  for (int s = 0; s < n; ++s)
    for (int c = 0; c < C; ++c) {
      int t = d.trans[size_t(s) * C + c];
      if (t >= 0) preds[t].push_back(s);
    }
  std::vector<char> live(n, 0);
  std::vector<int> stack;
  for (int s = 0; s < n; ++s) if (d.acc[s]) { live[s] = 1; stack.push_back(s); }
  while (!stack.empty()) {
    int s = stack.back();
    stack.pop_back();
    for (int p : preds[s]) if (!live[p]) { live[p] = 1; stack.push_back(p); }
  }
  ClassDfa r;
  r.n_cls = C;
  if (n == 0 || !live[d.start]) return r;
  std::vector<int> id(n, -1);
  int k = 0;
  for (int s = 0; s < n; ++s) if (live[s]) id[s] = k++;
  r.trans.assign(size_t(k) * C, -1);
  r.acc.resize(k);
  for (int s = 0; s < n; ++s) {
    if (!live[s]) continue;
    r.acc[id[s]] = d.acc[s];
    for (int c = 0; c < C; ++c) {
      int t = d.trans[size_t(s) * C + c];
      if (t >= 0 && live[t]) r.trans[size_t(id[s]) * C + c] = id[t];
    }
  }
  r.start = id[d.start];
  return r;
}

// Hopcroft minimisation of a trimmed automaton; missing transitions go to an
// implicit dead state, which is made explicit for the refinement.
ClassDfa minimise(const ClassDfa& d) {
  int n = d.size(), C = d.n_cls;
  if (n == 0) return d;
  int N = n + 1, dead = n;
  auto tr = [&](int s, int c) -> int {
    if (s == dead) return dead;
    int t = d.trans[size_t(s) * C + c];
    return t < 0 ? dead : t;
  };
  // predecessor lists per (class, target), CSR
  std::vector<int> cnt(size_t(C) * N + 1, 0);
  for (int s = 0; s < N; ++s)
    for (int c = 0; c < C; ++c) cnt[size_t(c) * N + tr(s, c) + 1]++;
  for (size_t i = 1; i < cnt.size(); ++i) cnt[i] += cnt[i - 1];
  std::vector<int> pred(cnt.back());
  {
    std::vector<int> fill(cnt.begin(), cnt.end() - 1);
    for (int s = 0; s < N; ++s)
      for (int c = 0; c < C; ++c) pred[fill[size_t(c) * N + tr(s, c)]++] = s;
  }
  // refinable partition
  std::vector<int> elems(N), loc(N), blk(N), first, end, marked;
  {
    int k = 0;
    for (int pass = 0; pass < 2; ++pass)
      for (int s = 0; s < N; ++s) {
        bool a = s < n && d.acc[s];
        if ((pass == 0) == a) { loc[s] = k; elems[k++] = s; }
      }
    int n_acc = 0;
    for (int s = 0; s < n; ++s) n_acc += d.acc[s] ? 1 : 0;
    if (n_acc > 0) { first.push_back(0); end.push_back(n_acc); }
    if (n_acc < N) { first.push_back(n_acc); end.push_back(N); }
    for (size_t b = 0; b < first.size(); ++b)
      for (int i = first[b]; i < end[b]; ++i) blk[elems[i]] = int(b);
    marked.assign(first.size(), 0);
  }
  std::vector<int> work;
  std::vector<char> in_work(first.size(), 0);
  for (size_t b = 0; b < first.size(); ++b) { work.push_back(int(b)); in_work[b] = 1; }
  std::vector<int> touched;
  std::vector<int> members;
  while (!work.empty()) {
    int A = work.back();
    work.pop_back();
    in_work[A] = 0;
    members.assign(elems.begin() + first[A], elems.begin() + end[A]);
    for (int c = 0; c < C; ++c) {
      touched.clear();
      for (int t : members) {
        size_t lo = cnt[size_t(c) * N + t], hi = cnt[size_t(c) * N + t + 1];
        for (size_t i = lo; i < hi; ++i) {
          int s = pred[i];
          int b = blk[s];
          int pos = first[b] + marked[b];
          if (loc[s] < pos) continue;  // already marked
          if (marked[b] == 0) touched.push_back(b);
          int other = elems[pos];
          std::swap(elems[pos], elems[loc[s]]);
          loc[other] = loc[s];
          loc[s] = pos;
          marked[b]++;
        }
      }
      for (int b : touched) {
        int m = marked[b];
        marked[b] = 0;
        int size = end[b] - first[b];
        if (m == size) continue;
        // marked part [first, first+m) becomes a new block
        int nb = int(first.size());
        first.push_back(first[b]);
        end.push_back(first[b] + m);
        first[b] += m;
        marked.push_back(0);
        in_work.push_back(0);
        for (int i = first[nb]; i < end[nb]; ++i) blk[elems[i]] = nb;
        if (in_work[b]) { work.push_back(nb); in_work[nb] = 1; }
        else {
          int smaller = (end[nb] - first[nb] <= end[b] - first[b]) ? nb : b;
          work.push_back(smaller);
          in_work[smaller] = 1;
        }
      }
    }
  }
  // quotient automaton without the dead block
  int dead_blk = blk[dead];
  std::vector<int> id(first.size(), -1);
  int k = 0;
  for (int s = 0; s < n; ++s) if (id[blk[s]] < 0 && blk[s] != dead_blk) id[blk[s]] = k++;
  ClassDfa r;
  r.n_cls = C;
  r.trans.assign(size_t(k) * C, -1);
  r.acc.assign(k, 0);
  for (int s = 0; s < n; ++s) {
    int b = id[blk[s]];
    if (b < 0) continue;
    r.acc[b] = d.acc[s];
    for (int c = 0; c < C; ++c) {
      int t = tr(s, c);
      r.trans[size_t(b) * C + c] = (t == dead || blk[t] == dead_blk) ? -1 : id[blk[t]];
    }
  }
  r.start = id[blk[d.start]];
  return r;
}

ClassDfa Builder::intersection(const std::vector<int>& kids) {
  std::vector<ClassDfa> parts;
  for (int k : kids) {
    ClassDfa p = minimise(trim(dfa_of(k)));
    if (p.size() == 0) { ClassDfa e; e.n_cls = cls_.n; return e; }
    parts.push_back(std::move(p));
  }
  int C = cls_.n;
  ClassDfa prod;
  prod.n_cls = C;
  std::unordered_map<std::vector<int>, int, VecHash> index;
  std::vector<std::vector<int>> tuples;
  std::vector<int> t0;
  for (auto& p : parts) t0.push_back(p.start);
  index.emplace(t0, 0);
  tuples.push_back(t0);
  std::vector<int> nt(parts.size());
  for (size_t i = 0; i < tuples.size(); ++i) {
    if (tuples.size() > kMaxStates) fail(CG_E_LIMIT, "intersection too large");
    prod.trans.resize((i + 1) * size_t(C), -1);
    for (int c = 0; c < C; ++c) {
      bool ok = true;
      for (size_t j = 0; j < parts.size() && ok; ++j) {
        nt[j] = parts[j].trans[size_t(tuples[i][j]) * C + c];
        ok = nt[j] >= 0;
      }
      if (!ok) continue;
      auto it = index.find(nt);
      int id;
      if (it == index.end()) {
        id = int(tuples.size());
        index.emplace(nt, id);
        tuples.push_back(nt);
      } else {
        id = it->second;
      }
      prod.trans[i * size_t(C) + c] = id;
    }
  }
  prod.acc.resize(tuples.size());
  for (size_t i = 0; i < tuples.size(); ++i) {
    bool a = true;
    for (size_t j = 0; j < parts.size(); ++j) a = a && parts[j].acc[tuples[i][j]];
    prod.acc[i] = a;
  }
  prod.start = 0;
  return minimise(trim(prod));
}

}  // namespace

Dfa build_dfa(IR& ir, int root, int n_sym) {
  if (n_sym < kNumSymbols || n_sym > kMaxSymbols) fail(CG_E_ARG, "alphabet size");
  Classes cls = make_classes(ir, root, n_sym);
  Builder b(ir, cls);
  ClassDfa d = minimise(trim(b.dfa_of(root)));
  if (d.size() == 0) fail(CG_E_EMPTY, "the grammar accepts no string");
  // canonical breadth-first numbering over the symbols in order
  int C = d.n_cls;
  std::vector<int> canon(d.size(), -1), order;
  canon[d.start] = 0;
  order.push_back(d.start);
  for (size_t q = 0; q < order.size(); ++q) {
    int s = order[q];
    for (int a = 0; a < n_sym; ++a) {
      int t = d.trans[size_t(s) * C + cls.of_symbol[a]];
      if (t >= 0 && canon[t] < 0) { canon[t] = int(order.size()); order.push_back(t); }
    }
  }
  Dfa out;
  out.n_states = uint32_t(order.size());
  out.n_sym = uint32_t(n_sym);
  out.next.assign(size_t(out.n_states) * n_sym, -1);
  out.accept.assign(out.n_states, 0);
  for (uint32_t i = 0; i < out.n_states; ++i) {
    int s = order[i];
    out.accept[i] = d.acc[s];
    for (int a = 0; a < n_sym; ++a) {
      int t = d.trans[size_t(s) * C + cls.of_symbol[a]];
      out.next[size_t(i) * n_sym + a] = t < 0 ? -1 : canon[t];
    }
  }
  return out;
}

}  // namespace cg
