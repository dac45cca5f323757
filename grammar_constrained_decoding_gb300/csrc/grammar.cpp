// Grammar and vocabulary entry points of the C ABI (host only).
#include <algorithm>
#include <cstring>
#include <new>
#include <numeric>

#include "cg_internal.h"

namespace {

void set_err(char* err, size_t errlen, const std::string& m) {
  if (!err || errlen == 0) return;
  size_t n = std::min(errlen - 1, m.size());
  std::memcpy(err, m.data(), n);
  err[n] = 0;
}

struct ColHash {
  size_t operator()(const std::vector<int32_t>& v) const {
    uint64_t h = 0x9E3779B97F4A7C15ull;
    for (int32_t x : v) { h ^= uint32_t(x); h *= 0xFF51AFD7ED558CCDull; h ^= h >> 31; }
    return size_t(h);
  }
};

void finish_grammar(cg_grammar* g) {
  const uint32_t S = g->dfa.n_states;
  g->flags.assign(S, 0);
  for (uint32_t s = 0; s < S; ++s) {
    const int32_t* row = &g->dfa.next[size_t(s) * cg::kNumSymbols];
    bool any = false, model = false, injected = false;
    for (int a = 0; a < cg::kNumSymbols; ++a) {
      if (row[a] >= 0) {
        any = true;
        (a < 256 ? model : injected) = true;
      }
    }
    uint8_t f = 0;
    if (g->dfa.accept[s]) f |= CG_STATE_ACCEPT;
    if (g->dfa.accept[s] && !any) f |= CG_STATE_SINK;
    if (!model && injected) f |= CG_STATE_FORCED_ONLY;
    g->flags[s] = f;
  }
  // distinct columns
  std::unordered_map<std::vector<int32_t>, uint16_t, ColHash> ids;
  g->col_of.assign(cg::kNumSymbols, 0);
  std::vector<int32_t> col(S);
  for (int a = 0; a < cg::kNumSymbols; ++a) {
    for (uint32_t s = 0; s < S; ++s) col[s] = g->dfa.next[size_t(s) * cg::kNumSymbols + a];
    auto it = ids.find(col);
    if (it == ids.end()) it = ids.emplace(col, uint16_t(ids.size())).first;
    g->col_of[a] = it->second;
  }
  g->n_cols = uint32_t(ids.size());
  g->table.assign(size_t(S) * g->n_cols, CG_DEAD);
  for (uint32_t s = 0; s < S; ++s)
    for (int a = 0; a < cg::kNumSymbols; ++a) {
      int32_t t = g->dfa.next[size_t(s) * cg::kNumSymbols + a];
      g->table[size_t(s) * g->n_cols + g->col_of[a]] = t < 0 ? CG_DEAD : uint32_t(t);
    }
}

}  // namespace

namespace cg {

uint32_t mask_classes_joint(const std::vector<const cg_grammar*>& gs, uint32_t max_len,
                            std::vector<uint32_t>& class_of, std::vector<uint32_t>& rep_gid,
                            std::vector<uint32_t>& rep_state) {
  // Model bytes that every grammar maps to one column each: one representative
  // byte per combination of columns carries all transitions.
  std::vector<int> rep_bytes;
  {
    std::unordered_map<std::vector<int32_t>, int, ColHash> seen;
    std::vector<int32_t> key(gs.size());
    for (int a = 0; a < 256; ++a) {
      for (size_t i = 0; i < gs.size(); ++i) key[i] = gs[i]->col_of[a];
      if (seen.emplace(key, a).second) rep_bytes.push_back(a);
    }
  }
  std::vector<uint32_t> off(gs.size() + 1, 0);
  for (size_t i = 0; i < gs.size(); ++i) off[i + 1] = off[i] + gs[i]->dfa.n_states;
  const uint32_t S = off.back();
  // Refine {all states of all grammars} by model-byte successors, as in
  // mask_classes: after k rounds two states share a class iff every model-byte
  // word of length <= k fails from both or from neither.
  std::vector<uint32_t> cls(S, 0), next_cls(S);
  uint32_t n = 1;
  std::unordered_map<std::vector<int32_t>, uint32_t, ColHash> ids;
  std::vector<int32_t> sig(rep_bytes.size() + 1);
  for (uint32_t round = 0; round < max_len; ++round) {
    ids.clear();
    for (size_t i = 0; i < gs.size(); ++i) {
      const cg_grammar& g = *gs[i];
      for (uint32_t s = 0; s < g.dfa.n_states; ++s) {
        sig[0] = int32_t(cls[off[i] + s]);
        for (size_t k = 0; k < rep_bytes.size(); ++k) {
          const uint32_t t = g.table[size_t(s) * g.n_cols + g.col_of[rep_bytes[k]]];
          sig[k + 1] = t == CG_DEAD ? -1 : int32_t(cls[off[i] + t]);
        }
        auto it = ids.find(sig);
        if (it == ids.end()) it = ids.emplace(sig, uint32_t(ids.size())).first;
        next_cls[off[i] + s] = it->second;
      }
    }
    const uint32_t m = uint32_t(ids.size());
    cls.swap(next_cls);
    if (m == n) break;
    n = m;
  }
  class_of = cls;
  rep_gid.assign(n, 0);
  rep_state.assign(n, 0);
  std::vector<char> seen(n, 0);
  for (size_t i = 0; i < gs.size(); ++i)
    for (uint32_t s = 0; s < gs[i]->dfa.n_states; ++s) {
      const uint32_t c = cls[off[i] + s];
      if (!seen[c]) { seen[c] = 1; rep_gid[c] = uint32_t(i); rep_state[c] = s; }
    }
  return n;
}

}  // namespace cg

extern "C" {

int cg_mask_classes(const cg_grammar* const* g, uint32_t n_g, uint32_t max_len, uint32_t* class_of, uint32_t cap,
                    uint32_t* n_states, uint32_t* n_classes) {
  if (!g || n_g == 0 || !n_states || !n_classes) return CG_E_ARG;
  std::vector<const cg_grammar*> gs;
  uint64_t S = 0;
  for (uint32_t i = 0; i < n_g; ++i) {
    if (!g[i]) return CG_E_ARG;
    gs.push_back(g[i]);
    S += g[i]->dfa.n_states;
  }
  try {
    std::vector<uint32_t> cls, rg, rs;
    *n_classes = cg::mask_classes_joint(gs, max_len, cls, rg, rs);
    *n_states = uint32_t(S);
    if (class_of) {
      if (cap < S) return CG_E_LIMIT;
      std::copy(cls.begin(), cls.end(), class_of);
    }
  } catch (const std::bad_alloc&) {
    return CG_E_NOMEM;
  }
  return CG_OK;
}


int cg_compile(const char* src, size_t src_len, int kind, const cg_bounds* bounds, cg_grammar** out,
               char* err, size_t errlen) {
  if (!src || !bounds || !out) return CG_E_ARG;
  if (kind != CG_GBNF && kind != CG_JSON_SCHEMA && kind != CG_STRUCTURAL_TAG) return CG_E_ARG;
  *out = nullptr;
  try {
    cg::IR ir;
    std::string text(src, src_len);
    int root = kind == CG_GBNF ? cg::parse_gbnf(ir, text, bounds->depth_max)
               : kind == CG_JSON_SCHEMA
                   ? cg::lower_json_schema(ir, text, bounds->ws_max, bounds->max_len_default, bounds->max_items_default)
                   : cg::lower_structural_tag(ir, text, bounds->ws_max, bounds->max_len_default,
                                              bounds->max_items_default);
    auto* g = new cg_grammar;
    g->dfa = cg::build_dfa(ir, root);
    finish_grammar(g);
    if (g->n_cols > 65535) { delete g; set_err(err, errlen, "too many columns"); return CG_E_LIMIT; }
    *out = g;
    set_err(err, errlen, "");
    return CG_OK;
  } catch (const cg::CompileError& e) {
    set_err(err, errlen, e.msg);
    return e.code;
  } catch (const std::bad_alloc&) {
    set_err(err, errlen, "out of memory");
    return CG_E_NOMEM;
  }
}

void cg_grammar_destroy(cg_grammar* g) { delete g; }

int cg_grammar_info(const cg_grammar* g, uint32_t* n_states, uint32_t* n_cols, uint32_t* start) {
  if (!g) return CG_E_ARG;
  if (n_states) *n_states = g->dfa.n_states;
  if (n_cols) *n_cols = g->n_cols;
  if (start) *start = 0;
  return CG_OK;
}

int cg_grammar_export(const cg_grammar* g, int32_t* next, uint8_t* flags) {
  if (!g || !next || !flags) return CG_E_ARG;
  std::memcpy(next, g->dfa.next.data(), g->dfa.next.size() * sizeof(int32_t));
  std::memcpy(flags, g->flags.data(), g->flags.size());
  return CG_OK;
}

int cg_try_input(const cg_grammar* g, const uint8_t* s, size_t n, const uint8_t* injected, size_t* refused_at,
                 uint32_t* end_state, int* accepted) {
  if (!g || (!s && n) || !refused_at) return CG_E_ARG;
  int32_t st = 0;
  size_t i = 0;
  for (; i < n; ++i) {
    int a = s[i] + ((injected && injected[i]) ? 256 : 0);
    int32_t t = g->dfa.next[size_t(st) * cg::kNumSymbols + a];
    if (t < 0) break;
    st = t;
  }
  *refused_at = i;
  if (end_state) *end_state = uint32_t(st);
  if (accepted) *accepted = (i == n && g->dfa.accept[st]) ? 1 : 0;
  return CG_OK;
}

int cg_live_states(const cg_grammar* g, uint32_t* out, uint32_t cap, uint32_t* n) {
  if (!g || !n) return CG_E_ARG;
  uint32_t k = 0;
  for (uint32_t s = 0; s < g->dfa.n_states; ++s) {
    if (g->flags[s] & (CG_STATE_SINK | CG_STATE_FORCED_ONLY)) continue;
    if (out) {
      if (k >= cap) return CG_E_LIMIT;
      out[k] = s;
    }
    ++k;
  }
  *n = k;
  return CG_OK;
}

int cg_vocab_create(const uint8_t* bytes, const uint32_t* off, uint32_t V, cg_vocab** out) {
  if (!off || !out || V == 0 || off[0] != 0) return CG_E_ARG;
  *out = nullptr;
  try {
    auto* v = new cg_vocab;
    v->V = V;
    v->off.assign(off, off + V + 1);
    for (uint32_t t = 0; t < V; ++t) {
      if (off[t + 1] <= off[t]) { delete v; return CG_E_ARG; }
      uint32_t len = off[t + 1] - off[t];
      if (len > 64) { delete v; return CG_E_LIMIT; }
      v->max_len = std::max(v->max_len, len);
    }
    if (!bytes) { delete v; return CG_E_ARG; }
    v->bytes.assign(bytes, bytes + off[V]);
    v->perm.resize(V);
    std::iota(v->perm.begin(), v->perm.end(), 0u);
    const uint8_t* base = v->bytes.data();
    std::sort(v->perm.begin(), v->perm.end(), [&](uint32_t a, uint32_t b) {
      uint32_t la = off[a + 1] - off[a], lb = off[b + 1] - off[b];
      int c = std::memcmp(base + off[a], base + off[b], std::min(la, lb));
      if (c != 0) return c < 0;
      if (la != lb) return la < lb;
      return a < b;
    });
    v->lcp.assign(V, 0);
    v->sorted_off.assign(V + 1, 0);
    for (uint32_t i = 0; i < V; ++i) {
      uint32_t t = v->perm[i];
      uint32_t len = off[t + 1] - off[t];
      v->sorted_off[i + 1] = v->sorted_off[i] + len;
      v->sorted_bytes.insert(v->sorted_bytes.end(), base + off[t], base + off[t] + len);
      if (i) {
        uint32_t p = v->perm[i - 1];
        uint32_t lp = off[p + 1] - off[p], k = 0;
        while (k < len && k < lp && base[off[t] + k] == base[off[p] + k]) ++k;
        v->lcp[i] = uint8_t(k);
      }
    }
    v->lowest_id.reserve(V);
    for (uint32_t t = 0; t < V; ++t) {
      const uint32_t len = off[t + 1] - off[t];
      v->lowest_id.emplace(std::string_view(reinterpret_cast<const char*>(base + off[t]), len), t);  // first = lowest id
      v->len_mask[base[off[t]]] |= uint64_t(1) << (len - 1);
    }
    *out = v;
    return CG_OK;
  } catch (const std::bad_alloc&) {
    return CG_E_NOMEM;
  }
}

void cg_vocab_destroy(cg_vocab* v) { delete v; }

int cg_tokenize_greedy(const cg_vocab* v, const uint8_t* text, size_t n, uint32_t* out, size_t cap,
                       size_t* n_out) {
  if (!v || (!text && n) || !n_out) return CG_E_ARG;
  size_t i = 0, k = 0;
  while (i < n) {
    // candidate lengths: those of the tokens that start with this byte, longest first
    uint64_t lens = v->len_mask[text[i]];
    if (n - i < 64) lens &= (uint64_t(1) << (n - i)) - 1u;
    bool found = false;
    while (lens) {
      const size_t L = 64 - size_t(__builtin_clzll(lens));
      lens &= ~(uint64_t(1) << (L - 1));
      auto it = v->lowest_id.find(std::string_view(reinterpret_cast<const char*>(text + i), L));
      if (it != v->lowest_id.end()) {
        if (out && k < cap) out[k] = it->second;
        ++k;
        i += L;
        found = true;
        break;
      }
    }
    if (!found) return CG_E_ARG;
  }
  *n_out = k;
  return (out && k > cap) ? CG_E_LIMIT : CG_OK;
}

}  // extern "C"
