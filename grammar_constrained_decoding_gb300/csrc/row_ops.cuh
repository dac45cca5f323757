// Per-row pieces shared by the step kernels: the bitmask source of a row (as
// cg_fill_bitmask defines it), the trie walk that computes a class mask, and
// the automaton advance of cg_accept.  The separate kernels and the fused step
// kernel call the same functions, so they agree bit for bit.
#pragma once

#include "device.cuh"

namespace cgk {

constexpr uint32_t kStateEmpty = 0, kStateBusy = 1, kStateReady = 2;

__device__ __forceinline__ uint32_t load_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void store_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Where row's mask comes from (usetacet.com/docs/grammar, "The guarantee": the
// mask holds exactly the tokens the grammar allows): 0 the state's mask class,
// 1 an all-zero row (bad grammar id, bad forced id, dead or out-of-range state,
// forced-only state without a forced token), 2 a one-hot row at the forced
// token.  *err receives the CG_DEV_* code to record (0 for none).
// The same decision from values already loaded: n_states of grammar g (when
// g < n_g) and the state's flags (when s < n_states).
__device__ __forceinline__ int row_mask_mode_of(uint32_t n_g, uint32_t V, uint32_t g, int32_t f, uint32_t s,
                                                uint32_t n_states, uint8_t sflags, uint32_t* err) {
  int mode = 0;
  if (g >= n_g) mode = 1;
  else if (f >= 0) mode = (uint32_t(f) < V) ? 2 : 1;
  else if (s == CG_DEAD || s >= n_states) mode = 1;
  else if (sflags & CG_STATE_FORCED_ONLY) mode = 1;
  uint32_t e = 0;
  if (g >= n_g) e = CG_DEV_BAD_GID;
  else if (f >= 0 && uint32_t(f) >= V) e = CG_DEV_BAD_FORCED;
  else if (f < 0 && s != CG_DEAD && s >= n_states) e = CG_DEV_BAD_STATE;
  else if (mode == 1 && f < 0 && s != CG_DEAD) e = CG_DEV_MISSING_FORCED;
  *err = e;
  return mode;
}

__device__ __forceinline__ int row_mask_mode(const Tables& t, uint32_t g, int32_t f, uint32_t s, uint32_t* err) {
  const uint32_t n_states = g < t.n_g ? t.grammars[g].n_states : 0u;
  const uint8_t sflags = (g < t.n_g && f < 0 && s != CG_DEAD && s < n_states)
                             ? t.state_flags[t.grammars[g].state_off + s]
                             : uint8_t(0);
  return row_mask_mode_of(t.n_g, t.V, g, f, s, n_states, sflags, err);
}

// Walk the tokens at positions [lo, hi) of the trie (lexicographic) order from
// state s of grammar g with threads tid = 0..nthreads-1; sets allowed bits in
// smask[W] (zeroed by the caller).  Each thread takes a contiguous run of
// positions and resumes each token's walk from the state reached after the
// prefix it shares with the previous token, so shared prefixes are walked
// once.  walk_tokens: the whole vocabulary.
__device__ inline void walk_tokens_range(const Tables& t, const DevGrammar& gd, const uint16_t* scol, uint32_t s,
                                         uint32_t* smask, uint32_t lo, uint32_t hi, uint32_t tid,
                                         uint32_t nthreads) {
  const uint32_t per = (hi - lo + nthreads - 1) / nthreads;
  const uint32_t i0 = lo + tid * per;
  const uint32_t i1 = min(hi, i0 + per);
  const uint32_t* table = t.table + gd.table_off;
  const uint32_t ncols = gd.n_cols;
  uint32_t stack[65];
  stack[0] = s;
  uint32_t valid = 0;  // stack[0..valid] hold the states after 0..valid bytes of the previous token
  for (uint32_t i = i0; i < i1; ++i) {
    const uint32_t b0 = t.sorted_off[i], len = t.sorted_off[i + 1] - b0;
    const uint32_t l = (i == i0) ? 0u : uint32_t(t.lcp[i]);
    bool ok = false;
    if (l <= valid) {
      uint32_t k = l, st = stack[l];
      ok = true;
      for (; k < len; ++k) {
        const uint32_t nx = __ldg(table + size_t(st) * ncols + scol[t.sorted_bytes[b0 + k]]);
        if (nx == CG_DEAD) { ok = false; break; }
        st = nx;
        stack[k + 1] = st;
      }
      valid = k;
    }
    // l > valid: the shared prefix already contains the byte that failed
    if (ok) {
      const uint32_t id = t.perm[i];
      atomicOr(smask + (id >> 5), 1u << (id & 31));
    }
  }
}

__device__ inline void walk_tokens(const Tables& t, const DevGrammar& gd, const uint16_t* scol, uint32_t s,
                                   uint32_t* smask, uint32_t tid, uint32_t nthreads) {
  walk_tokens_range(t, gd, scol, s, smask, 0u, t.V, tid, nthreads);
}

constexpr uint32_t kPrefetch = 16;  // token bytes whose columns are loaded up front

// Rows [lo, lo + rows) of a grammar's 16-bit transition table and the flags
// of those states, copied into shared memory: transitions from these states
// are read there instead of from global memory.
struct StateWindow {
  const uint16_t* next = nullptr;  // [rows][n_cols]
  const uint8_t* flags = nullptr;  // [rows]
  uint32_t lo = 0, rows = 0;
};

// Rows of the 16-bit table to copy for a window around state s: at most
// max_rows states and cap_bytes of shared memory (an aligned bulk copy may
// start up to 15 bytes early).  Fills lo/rows, the copy's 16-byte aligned
// source and size, and delta, the entries to skip at the start of the copy.
// rows == 0: no window (no 16-bit table, or nothing fits).
struct WindowCopy {
  uint32_t lo = 0, rows = 0, delta = 0, bytes = 0;
  const void* src = nullptr;
};
__device__ inline WindowCopy window_copy(const Tables& t, const DevGrammar& gd, uint32_t s, uint32_t cap_bytes,
                                         uint32_t max_rows) {
  WindowCopy w;
  if (!t.table16 || s >= gd.n_states || gd.n_cols == 0 || cap_bytes < 32) return w;
  const uint32_t cap = min(max_rows, (cap_bytes - 16) / (2 * gd.n_cols));
  if (cap == 0) return w;
  const uint32_t hi = min(gd.n_states, max(s, cap / 2) + (cap - cap / 2));
  w.lo = hi > cap ? hi - cap : 0u;
  w.rows = hi - w.lo;
  const uintptr_t src = reinterpret_cast<uintptr_t>(t.table16 + gd.table_off + size_t(w.lo) * gd.n_cols);
  const uintptr_t src0 = src & ~uintptr_t(15);
  w.src = reinterpret_cast<const void*>(src0);
  w.delta = uint32_t(src - src0) / 2;
  w.bytes = (uint32_t(src - src0) + w.rows * gd.n_cols * 2 + 15u) & ~15u;  // <= cap_bytes
  return w;
}

// Walks token tok's bytes from state st of grammar gd through the columns
// `cols` (the symbol -> column map, shifted by 256 for injected bytes); returns
// CG_DEAD when a byte has no transition.  win (optional): a window of the
// 16-bit table in shared memory, read instead of global memory for its states.
__device__ inline uint32_t walk_token(const Tables& t, const DevGrammar& gd, const uint16_t* cols, uint32_t st,
                                      uint32_t tok, const StateWindow& win, const uint4* rec = nullptr) {
  const uint32_t* table = t.table + gd.table_off;
  const uint32_t nc = gd.n_cols;
  auto step_from = [&](uint32_t s, uint32_t col) -> uint32_t {
    const uint32_t r = s - win.lo;
    if (r < win.rows) {
      const uint16_t nx = win.next[r * nc + col];
      return nx == kDead16 ? CG_DEAD : uint32_t(nx);
    }
    return table[size_t(s) * nc + col];
  };
  uint32_t len = kLongToken;
  uint4 r0 = make_uint4(0u, 0u, 0u, 0u), r1 = r0;
  if (rec || t.tok_rec) {
    // the token's bytes in one 32-byte record (rec: a copy already loaded)
    r0 = rec ? rec[0] : t.tok_rec[size_t(tok) * 2];
    r1 = rec ? rec[1] : t.tok_rec[size_t(tok) * 2 + 1];
    len = r0.x & 0xFFu;
  }
  if (len != kLongToken) {
    const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
    for (uint32_t k = 0; k < 31; ++k) {
      if (k >= len || st == CG_DEAD) break;
      const uint32_t byte = (w[(k + 1) >> 2] >> (8 * ((k + 1) & 3))) & 0xFFu;
      st = step_from(st, cols[byte]);
    }
    return st;
  }
  // the offset table; the token's columns first (independent loads), then the
  // chain of lookups
  const uint32_t i0 = t.tok_off[tok], n = t.tok_off[tok + 1] - i0;
  uint32_t col[kPrefetch];
#pragma unroll
  for (uint32_t k = 0; k < kPrefetch; ++k) col[k] = k < n ? cols[t.tok_bytes[i0 + k]] : 0u;
#pragma unroll
  for (uint32_t k = 0; k < kPrefetch; ++k)
    if (k < n && st != CG_DEAD) st = step_from(st, col[k]);
  for (uint32_t i = i0 + kPrefetch; i < i0 + n && st != CG_DEAD; ++i) st = step_from(st, cols[t.tok_bytes[i]]);
  return st;
}

// CG_FLAG_DONE / CG_FLAG_FORCED_NEXT of a live state from its CG_STATE_* bits.
__device__ __forceinline__ uint8_t state_result_flags(uint8_t sf) {
  uint8_t fl = 0;
  if (sf & CG_STATE_SINK) fl |= CG_FLAG_DONE;
  if (sf & CG_STATE_FORCED_ONLY) fl |= CG_FLAG_FORCED_NEXT;
  return fl;
}

// Advance one row by its token (labs.miniml.ai "Evaluator aware decoding":
// the automaton also moves forward over injected tokens; a forced token's
// bytes are walked as host-injected symbols).  With token counts, finished or capped
// rows restart from state 0 (usetacet.com/docs/grammar, "A valid call also has
// to end").  Writes out_states[b], out_flags[b] and counts[b].
// cols_g (optional) is a copy of grammar g's 512-entry symbol -> column map
// and win (optional) a window of its transition table, both in shared memory:
// they only shorten the chain of dependent loads.
__device__ inline void accept_row(const Tables& t, uint32_t b, uint32_t g, uint32_t s, uint32_t tok, int32_t f,
                                  uint32_t* counts, uint32_t max_tokens, uint32_t* out_states, uint8_t* out_flags,
                                  const uint16_t* cols_g = nullptr, const StateWindow& win = StateWindow()) {
  uint32_t ns = s;
  uint8_t fl = 0;
  const uint32_t n0 = counts ? counts[b] : 0u;  // independent of the walk: loaded first
  if (g >= t.n_g) {
    record_error(t.status, CG_DEV_BAD_GID);
    ns = CG_DEAD;
    fl = CG_FLAG_REJECTED;
  } else if (tok == CG_NO_TOKEN) {
    fl = CG_FLAG_NO_TOKEN;
  } else if (tok >= t.V) {
    record_error(t.status, CG_DEV_BAD_TOKEN);
    ns = CG_DEAD;
    fl = CG_FLAG_REJECTED;
  } else if (s == CG_DEAD) {
    fl = CG_FLAG_REJECTED;
  } else {
    const DevGrammar gd = t.grammars[g];
    if (s >= gd.n_states) {
      record_error(t.status, CG_DEV_BAD_STATE);
      ns = CG_DEAD;
      fl = CG_FLAG_REJECTED;
    } else if (f >= 0 && tok != uint32_t(f)) {
      record_error(t.status, CG_DEV_FORCED_MISMATCH);
      ns = CG_DEAD;
      fl = CG_FLAG_REJECTED;
    } else {
      const uint16_t* cols = (cols_g ? cols_g : t.colmap + size_t(g) * 512) + (f >= 0 ? 256u : 0u);
      const uint32_t st = walk_token(t, gd, cols, s, tok, win);
      ns = st;
      if (st == CG_DEAD) {
        record_error(t.status, CG_DEV_REJECTED);
        fl = CG_FLAG_REJECTED;
      } else {
        const uint32_t r = st - win.lo;
        fl = state_result_flags(r < win.rows ? win.flags[r] : t.state_flags[gd.state_off + st]);
      }
    }
  }
  if (counts) {
    uint32_t n = n0 + (tok != CG_NO_TOKEN ? 1u : 0u);
    if ((fl & CG_FLAG_DONE) || n >= max_tokens) {
      if (!(fl & CG_FLAG_DONE)) fl |= CG_FLAG_CAPPED;
      ns = 0u;
      n = 0u;
    }
    counts[b] = n;
  }
  out_states[b] = ns;
  out_flags[b] = fl;
}

// Speculative verification of row b's draft toks[0 .. n) (labs.miniml.ai
// "Evaluator aware decoding", "Where XGrammar-2 could take this": once a
// draft token ends an evaluated span the evaluator's result fixes the tokens
// after it, so checking them is a comparison of ids).  Accepts the longest prefix whose tokens
// the grammar allows one after another; a position with forced[j] >= 0 must
// carry exactly that id and is walked as injected bytes.  Stops at the first
// refused token (CG_FLAG_DRAFT_CUT, the state stays that of the prefix), after
// a token that ends the grammar, when the count reaches max_tokens, or after a
// token whose state continues only with injected bytes when the next position
// is not pinned.  With counts, a row ended or capped by its accepted tokens
// restarts from state 0 with count 0.  Writes out_n[b] (tokens accepted), out_states[b],
// out_flags[b] (CG_FLAG_DONE / CG_FLAG_FORCED_NEXT of the final state plus
// CG_FLAG_DRAFT_CUT / CG_FLAG_CAPPED; CG_FLAG_NO_TOKEN for an empty draft,
// CG_FLAG_REJECTED for a dead row), counts[b], and path[0 .. K] (optional):
// the state before each position up to out_n, CG_DEAD after.  recs (optional):
// the token records of positions 0 .. n_recs already copied into shared
// memory; win (optional): a window of the 16-bit table (only shorten loads).
__device__ inline void accept_many_row(const Tables& t, uint32_t b, uint32_t g, uint32_t s, const uint32_t* toks,
                                       uint32_t n, const int32_t* forced, uint32_t K, uint32_t* counts,
                                       uint32_t max_tokens, uint32_t* out_states, uint32_t* out_n,
                                       uint8_t* out_flags, uint32_t* path, const uint4* recs = nullptr,
                                       uint32_t n_recs = 0, const StateWindow& win = StateWindow()) {
  uint32_t c = counts ? counts[b] : 0u;
  uint32_t st = s, acc = 0;
  uint8_t fl = 0;
  if (n > K) {
    record_error(t.status, CG_DEV_BAD_LENGTH);
    n = K;
  }
  if (path) path[0] = s;
  if (n == 0) {
    fl = CG_FLAG_NO_TOKEN;
  } else if (g >= t.n_g) {
    record_error(t.status, CG_DEV_BAD_GID);
    st = CG_DEAD;
    fl = CG_FLAG_REJECTED;
  } else if (s == CG_DEAD) {
    fl = CG_FLAG_REJECTED;
  } else {
    const DevGrammar gd = t.grammars[g];
    if (s >= gd.n_states) {
      record_error(t.status, CG_DEV_BAD_STATE);
      st = CG_DEAD;
      fl = CG_FLAG_REJECTED;
    } else {
      const uint16_t* cols0 = t.colmap + size_t(g) * 512;
      uint8_t cut = 0, capped = 0;
      auto flags_of = [&](uint32_t x) -> uint8_t {
        const uint32_t r = x - win.lo;
        return state_result_flags(r < win.rows ? win.flags[r] : t.state_flags[gd.state_off + x]);
      };
      uint8_t sres = flags_of(st);
      int32_t f = forced ? forced[0] : -1;
      for (uint32_t j = 0; j < n; ++j) {
        const uint32_t tok = toks[j];
        const int32_t f_next = (forced && j + 1 < n) ? forced[j + 1] : -1;
        if (tok >= t.V) {
          record_error(t.status, CG_DEV_BAD_TOKEN);
          cut = CG_FLAG_DRAFT_CUT;
          break;
        }
        const uint32_t ns = (f >= 0 && tok != uint32_t(f))
                                ? CG_DEAD
                                : walk_token(t, gd, cols0 + (f >= 0 ? 256u : 0u), st, tok, win,
                                             j < n_recs ? recs + 2 * j : nullptr);
        if (ns == CG_DEAD) {
          cut = CG_FLAG_DRAFT_CUT;
          break;
        }
        st = ns;
        ++acc;
        ++c;
        if (path) path[acc] = st;
        sres = flags_of(st);
        if (sres & CG_FLAG_DONE) break;
        if (counts && c >= max_tokens) {
          capped = CG_FLAG_CAPPED;
          break;
        }
        if ((sres & CG_FLAG_FORCED_NEXT) && f_next < 0) break;
        f = f_next;
      }
      fl = sres | cut | capped;
      if (counts && acc > 0 && (fl & (CG_FLAG_DONE | CG_FLAG_CAPPED))) {
        st = 0u;
        c = 0u;
      }
    }
  }
  if (path)
    for (uint32_t j = acc + 1; j <= K; ++j) path[j] = CG_DEAD;
  if (counts) counts[b] = c;
  out_states[b] = st;
  out_n[b] = acc;
  out_flags[b] = fl;
}

}  // namespace cgk
