// Library-internal host structures behind the opaque C handles.
#pragma once

#include <cstdint>
#include <deque>
#include <string>
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
  std::unordered_map<std::string, uint32_t> lowest_id;  // token string -> lowest id
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

namespace cg {
// Mask classes over several grammars at once (grammar.cpp): states, of any of
// the grammars, whose allowed-token sets agree for every token of at most
// max_len bytes share a class (one cached mask).  States are numbered grammar
// after grammar; rep_gid / rep_state give each class's representative
// (grammar, state).
uint32_t mask_classes_joint(const std::vector<const cg_grammar*>& gs, uint32_t max_len,
                            std::vector<uint32_t>& class_of, std::vector<uint32_t>& rep_gid,
                            std::vector<uint32_t>& rep_state);
}  // namespace cg
