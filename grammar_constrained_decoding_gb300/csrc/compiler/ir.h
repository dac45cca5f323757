// Regular-expression IR shared by the grammar front-ends and the automaton
// builder.  Symbols: 0..255 are bytes written by the model, 256..511 are the
// same bytes injected by the host (forced tokens), so the evaluator-aware rule
// that the model never writes the result block itself (labs.miniml.ai
// "Evaluator aware decoding", "A concrete prototype on llama.cpp") is
// automaton structure.
#pragma once

#include <cstdint>
#include <string>
#include <vector>

namespace cg {

constexpr int kNumSymbols = 512;
// The pushdown compiler (pda.cpp) extends the alphabet: symbol 512 + j stands
// for a reference to recursive rule j inside a rule body (a call).
constexpr int kNumCallSymbols = 64;
constexpr int kMaxSymbols = kNumSymbols + kNumCallSymbols;

struct SymSet {
  uint64_t w[kMaxSymbols / 64] = {};
  void set(int a) { w[a >> 6] |= uint64_t(1) << (a & 63); }
  bool test(int a) const { return (w[a >> 6] >> (a & 63)) & 1; }
  void set_range(int lo, int hi) { for (int a = lo; a <= hi; ++a) set(a); }
  bool empty() const {
    for (uint64_t x : w) if (x) return false;
    return true;
  }
  bool operator==(const SymSet& o) const {
    for (int i = 0; i < kMaxSymbols / 64; ++i) if (w[i] != o.w[i]) return false;
    return true;
  }
  SymSet shifted_to_injected() const {
    // model bytes move to the injected half; injected bytes stay (call
    // symbols never occur inside a forced region)
    SymSet r;
    for (int i = 0; i < 4; ++i) r.w[i + 4] = w[i] | w[i + 4];
    return r;
  }
};

enum class NodeKind : uint8_t { Empty, Eps, Sym, Cat, Alt, And, Rep };

struct Node {
  NodeKind kind = NodeKind::Empty;
  SymSet set;                // Sym
  std::vector<int> kids;     // Cat, Alt, And (Rep: kids[0])
  int lo = 0, hi = 0;        // Rep: hi < 0 means unbounded
};

class IR {
 public:
  std::vector<Node> nodes;
  int empty() { return add(Node{NodeKind::Empty}); }
  int eps() { return add(Node{NodeKind::Eps}); }
  int sym(const SymSet& s) {
    Node n; n.kind = NodeKind::Sym; n.set = s; return add(std::move(n));
  }
  int byte(int b) { SymSet s; s.set(b); return sym(s); }
  int range(int lo, int hi) { SymSet s; s.set_range(lo, hi); return sym(s); }
  int literal(const std::string& bytes) {
    if (bytes.empty()) return eps();
    std::vector<int> k;
    for (unsigned char c : bytes) k.push_back(byte(c));
    return cat(k);
  }
  int cat(std::vector<int> k) {
    if (k.size() == 1) return k[0];
    Node n; n.kind = NodeKind::Cat; n.kids = std::move(k); return add(std::move(n));
  }
  int alt(std::vector<int> k) {
    if (k.size() == 1) return k[0];
    Node n; n.kind = NodeKind::Alt; n.kids = std::move(k); return add(std::move(n));
  }
  int conj(std::vector<int> k) {
    if (k.size() == 1) return k[0];
    Node n; n.kind = NodeKind::And; n.kids = std::move(k); return add(std::move(n));
  }
  int rep(int x, int lo, int hi) {
    Node n; n.kind = NodeKind::Rep; n.kids = {x}; n.lo = lo; n.hi = hi; return add(std::move(n));
  }
  // copy of subtree x with every symbol set moved to the injected half
  int injected(int x);

 private:
  int add(Node n) { nodes.push_back(std::move(n)); return int(nodes.size()) - 1; }
};

// Error raised by front-ends and the builder; code is a CG_E_* value.
struct CompileError {
  int code;
  std::string msg;
};

// Front-ends (gbnf.cpp, schema.cpp, structtag.cpp): return the root node of the language.
int parse_gbnf(IR& ir, const std::string& src, uint32_t depth_max);
int lower_json_schema(IR& ir, const std::string& src, uint32_t ws_max, uint32_t max_len_default,
                      uint32_t max_items_default);
int lower_structural_tag(IR& ir, const std::string& src, uint32_t ws_max, uint32_t max_len_default,
                         uint32_t max_items_default);

// Minimal trimmed DFA over the first n_sym symbols (512, or more with call
// symbols) with canonical breadth-first numbering (automaton.cpp).
struct Dfa {
  uint32_t n_states = 0;
  uint32_t n_sym = kNumSymbols;
  std::vector<int32_t> next;   // [n_states * n_sym], -1 = DEAD
  std::vector<uint8_t> accept; // [n_states]
};
Dfa build_dfa(IR& ir, int root, int n_sym = kNumSymbols);

// Recursive GBNF rules for the pushdown compiler (gbnf.cpp).  automata[0] is
// the start rule's body, automata[1 + j] the body of recursive rule j (a rule
// on a cycle of the reference graph); in every body, references to other
// rules are inlined and a reference to recursive rule j is call symbol 512 + j.
struct RuleSystem {
  std::vector<std::string> names;  // [1 + n_rec]: "root", then the recursive rules
  std::vector<int> automata;       // IR roots, same order
  int n_rec() const { return int(names.size()) - 1; }
};
RuleSystem lower_gbnf_rules(IR& ir, const std::string& src);

}  // namespace cg
