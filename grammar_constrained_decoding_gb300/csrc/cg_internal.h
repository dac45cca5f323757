// Library-internal host structures behind the opaque C handles.
#pragma once

#include <cstdint>
#include <deque>
#include <string>
#include <string_view>
#include <unordered_map>
#include <vector>

#include "../../include/cg.h"
#include "compiler/ir.h"

struct cg_grammar {
  cg::Dfa dfa;                      // next[S*512] (-1 DEAD), accept[S]
  std::vector<uint8_t> flags;       // CG_STATE_* per state
  uint32_t n_cols = 0;              // distinct transition columns over the 512 symbols
  std::vector<uint16_t> col_of;     // [512] symbol -> column
  std::vector<uint32_t> table;      // [S * n_cols] next state, CG_DEAD for none
};

struct cg_vocab {
  uint32_t V = 0;
  uint32_t max_len = 0;
  std::vector<uint8_t> bytes;       // token t is bytes[off[t] .. off[t+1])
  std::vector<uint32_t> off;        // [V+1]
  // trie (lexicographic) order: sorted position i holds token perm[i]; lcp[i]
  // is the common prefix length of sorted tokens i-1 and i (lcp[0] = 0)
  std::vector<uint32_t> perm;
  std::vector<uint8_t> lcp;
  std::vector<uint8_t> sorted_bytes;
  std::vector<uint32_t> sorted_off;
  // token string (a view into `bytes`) -> lowest id with that string
  std::unordered_map<std::string_view, uint32_t> lowest_id;
  uint64_t len_mask[256] = {};      // bit L-1: some token of L bytes starts with this byte
};

struct cg_driver {
  const cg_vocab* vocab = nullptr;
  uint32_t B = 0;
  std::vector<uint16_t> gid;
  struct Rule { std::string open, close; int fmt; };
  std::vector<Rule> rules;
  std::vector<std::string> text;
  std::vector<std::deque<uint32_t>> queue;
};

// Pushdown automaton of a recursive GBNF grammar (compiler/pda.cpp).  States
// of all rule automata are numbered together, the start rule's first (state 0
// is the start).  A row's configuration is its state q and a stack of return
// states of level <= depth.  act[q * n_cols + col_of[symbol]] is the action of
// a symbol: kPdaNone (no edge: pop when q ends its rule and the stack is not
// empty, else refuse), a state (shift; allowed when level + h[target] <=
// depth), or kPdaCall | offset of a call chain in `chain`: chain[o] = n |
// req << 8, then the n return states to push (outermost first), then the
// state that consumes the symbol in the innermost rule; allowed when
// level + req <= depth.
constexpr uint32_t kPdaNone = 0xFFFFFFFFu;
constexpr uint32_t kPdaCall = 0x80000000u;
constexpr uint8_t kPdaInf = 0xFF;  // no completion / no continuation

struct cg_pda_grammar {
  uint32_t depth = 0;
  uint32_t n_states = 0;
  std::vector<std::string> rule_names;  // "root", then the recursive rules
  std::vector<uint32_t> rule_start;     // start state of each rule automaton
  std::vector<uint32_t> rule_of;        // [S] rule automaton of each state
  std::vector<uint8_t> accept;          // [S] the state may end its rule
  std::vector<uint8_t> h;               // [S] least extra levels needed to end the rule from here
  std::vector<uint8_t> need_model;      // [S] least headroom of a continuation by a model byte
  std::vector<uint8_t> need_inj;        // [S] same for an injected byte
  uint32_t n_cols = 0;
  std::vector<uint16_t> col_of;         // [512] symbol -> column
  std::vector<uint32_t> act;            // [S * n_cols]
  std::vector<uint32_t> chain;
  std::vector<std::vector<uint32_t>> returns_of;  // per rule: the return states its callers push
};

namespace cg {
// Result of walking one token from state q with an unknown stack below it
// (compiler/pda.cpp): kPdaTokDead (refused whatever the stack), kPdaTokPop
// (the walk pops below the start and survives under at least one stack the
// grammar can build: decided per row), or the least headroom depth - level at
// which the token is allowed.
constexpr uint32_t kPdaTokDead = 0xFFFFFFFFu;
constexpr uint32_t kPdaTokPop = 0xFFFFFFFEu;
uint32_t pda_token_need(const cg_pda_grammar& g, uint32_t q, const uint8_t* bytes, uint32_t n);

// Mask classes over several grammars at once (grammar.cpp): states, of any of
// the grammars, whose allowed-token sets agree for every token of at most
// max_len bytes share a class (one cached mask).  States are numbered grammar
// after grammar; rep_gid / rep_state give each class's representative
// (grammar, state).
uint32_t mask_classes_joint(const std::vector<const cg_grammar*>& gs, uint32_t max_len,
                            std::vector<uint32_t>& class_of, std::vector<uint32_t>& rep_gid,
                            std::vector<uint32_t>& rep_state);
}  // namespace cg
