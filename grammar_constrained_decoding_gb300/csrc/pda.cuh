// Pushdown rows: the device view of a compiled pushdown automaton and the
// walks shared by the pushdown kernels (pda.cu) and the fused pushdown step
// (kernel_sample.cu).  usetacet.com/docs/grammar, "The guarantee": the
// automaton that masks the logits is a pushdown automaton; each row carries
// its state and a stack of return states.
#pragma once

#include <cstdint>

#include "cg_internal.h"
#include "device.cuh"

namespace cgk {

struct DevPda {
  // the walk tables, one 16-byte aligned block (`tabs`, tab_n16 uint4s):
  // colmap at offset 0, then sinfo, act and chain at their byte offsets
  const uint16_t* colmap;    // [512] symbol -> column
  const uint32_t* sinfo;     // [S] bit 0 may end its rule; bits 8..15 h; 16..23 need_model; 24..31 need_inj
  const uint32_t* act;       // [S * n_cols] actions (kPdaNone, a state, or kPdaCall | chain offset)
  const uint32_t* chain;     // call chains: n | req << 8, n return states, target
  const uint4* tabs;
  uint32_t tab_n16, off_sinfo, off_act, off_chain;
  bool tabs_in_smem;         // small enough to copy into each block's shared memory
  const uint32_t* key;       // [S] first key << 8 | largest headroom with its own key
  const uint32_t* mask_of;   // [n_keys] index of the cached mask
  const uint32_t* masks;     // [n_masks][W]
  const uint32_t* cand_off;  // [S + 1] per state, the tokens that pop below the row's frame
  const uint32_t* cand;
  uint32_t S, n_cols, depth, stride;
};

constexpr uint32_t kPdaSmemTables = 32 * 1024;  // walk tables up to this size live in shared memory

// Copies the walk tables into shared memory `sm` (all threads of the block
// take part; the caller synchronises) and returns a view reading them there.
__device__ __forceinline__ DevPda tables_to_smem(const DevPda& p, uint4* sm, uint32_t tid, uint32_t nthreads) {
  for (uint32_t i = tid; i < p.tab_n16; i += nthreads) sm[i] = p.tabs[i];
  DevPda v = p;
  const unsigned char* base = reinterpret_cast<const unsigned char*>(sm);
  v.colmap = reinterpret_cast<const uint16_t*>(base);
  v.sinfo = reinterpret_cast<const uint32_t*>(base + p.off_sinfo);
  v.act = reinterpret_cast<const uint32_t*>(base + p.off_act);
  v.chain = reinterpret_cast<const uint32_t*>(base + p.off_chain);
  return v;
}

// The row's own stack, read and written in place (accept).
struct RowStack {
  uint32_t* s;
  __device__ __forceinline__ uint32_t pop(uint32_t i) { return s[i]; }
  __device__ __forceinline__ uint32_t get(uint32_t i) const { return s[i]; }
  __device__ __forceinline__ void put(uint32_t i, uint32_t v) { s[i] = v; }
};

// A thread's view of a row's stack (fill): entries below `keep` are the
// row's, shared read-only in shared memory; entries pushed by this thread's
// walk live in its own array.  keep only falls (to the lowest level popped to).
struct OverlayStack {
  const uint32_t* base;
  uint32_t keep;
  uint32_t local[CG_PDA_MAX_DEPTH];
  __device__ __forceinline__ uint32_t pop(uint32_t i) {
    const uint32_t v = i < keep ? base[i] : local[i];
    keep = min(keep, i);
    return v;
  }
  __device__ __forceinline__ uint32_t get(uint32_t i) const { return i < keep ? base[i] : local[i]; }
  __device__ __forceinline__ void put(uint32_t i, uint32_t v) { local[i] = v; }
};

__device__ __forceinline__ uint32_t pda_h(uint32_t info) { return (info >> 8) & 0xFFu; }

// One symbol (column col) from (q, lvl): pops while q may end its rule and the
// symbol has no action here, then shifts or runs the call chain.  false: the
// symbol is refused (no action, nothing to pop, or the headroom is too small).
template <class Stack>
__device__ __forceinline__ bool pda_symbol(const DevPda& p, uint32_t col, uint32_t& q, uint32_t& lvl, Stack& st) {
  for (;;) {  // every pass returns or pops one level
    const uint32_t a = p.act[size_t(q) * p.n_cols + col];
    if (a == kPdaNone) {
      if (!(p.sinfo[q] & 1u) || lvl == 0) return false;
      --lvl;
      q = st.pop(lvl);
      continue;
    }
    if (a & kPdaCall) {
      const uint32_t o = a & ~kPdaCall, head = p.chain[o], n = head & 0xFFu, req = head >> 8;
      if (lvl + req > p.depth) return false;
      for (uint32_t i = 0; i < n; ++i) st.put(lvl + i, p.chain[o + 1 + i]);
      lvl += n;
      q = p.chain[o + 1 + n];
      return true;
    }
    if (lvl + pda_h(p.sinfo[a]) > p.depth) return false;
    q = a;
    return true;
  }
}

// Walks token tok's bytes (as injected bytes when sym_off is 256).
template <class Stack>
__device__ bool pda_walk(const DevPda& p, const Tables& t, uint32_t tok, uint32_t sym_off, uint32_t& q,
                         uint32_t& lvl, Stack& st) {
  const uint16_t* cols = p.colmap + sym_off;
  const uint4 r0 = t.tok_rec[size_t(tok) * 2];
  const uint32_t len = r0.x & 0xFFu;
  if (len != kLongToken) {
    const uint4 r1 = t.tok_rec[size_t(tok) * 2 + 1];
    const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
    for (uint32_t k = 0; k < len; ++k) {
      const uint32_t byte = (w[(k + 1) >> 2] >> (8 * ((k + 1) & 3))) & 0xFFu;
      if (!pda_symbol(p, cols[byte], q, lvl, st)) return false;
    }
    return true;
  }
  for (uint32_t i = t.tok_off[tok]; i < t.tok_off[tok + 1]; ++i)
    if (!pda_symbol(p, cols[t.tok_bytes[i]], q, lvl, st)) return false;
  return true;
}

// CG_FLAG_DONE / CG_FLAG_FORCED_NEXT of a configuration: a continuation exists
// in a frame when its state has one within the frame's headroom; the frame
// below is reached only through a state that may end its rule.
template <class Stack>
__device__ uint8_t pda_flags(const DevPda& p, uint32_t q, uint32_t lvl, const Stack& st) {
  bool model = false, inj = false, complete = false;
  uint32_t s = q, l = lvl;
  for (;;) {  // at most lvl + 1 frames
    const uint32_t info = p.sinfo[s], hr = p.depth - l;
    model = model || ((info >> 16) & 0xFFu) <= hr;
    inj = inj || (info >> 24) <= hr;
    if (!(info & 1u)) break;
    if (l == 0) {
      complete = true;
      break;
    }
    --l;
    s = st.get(l);
  }
  uint8_t fl = 0;
  if (complete && !model && !inj) fl |= CG_FLAG_DONE;
  if (!model && inj) fl |= CG_FLAG_FORCED_NEXT;
  return fl;
}

// Advances row b (configuration at `row`, updated in place) by token tok;
// returns the CG_FLAG_* bits and updates counts[b] when counts are kept.
__device__ inline uint8_t pda_accept_row(const DevPda& p, const DevPda& pv, const Tables& t, uint32_t* row,
                                         uint32_t b, uint32_t tok, int32_t f, uint32_t* counts, uint32_t max_tokens) {
  uint32_t q = row[0], lvl = row[1];
  const uint32_t n0 = counts ? counts[b] : 0u;
  uint8_t fl = 0;
  if (tok == CG_NO_TOKEN) {
    fl = CG_FLAG_NO_TOKEN;
  } else if (tok >= t.V) {
    record_error(t.status, CG_DEV_BAD_TOKEN);
    q = CG_DEAD;
    fl = CG_FLAG_REJECTED;
  } else if (q == CG_DEAD) {
    fl = CG_FLAG_REJECTED;
  } else if (q >= p.S || lvl > p.depth) {
    record_error(t.status, CG_DEV_BAD_STATE);
    q = CG_DEAD;
    fl = CG_FLAG_REJECTED;
  } else if (f >= 0 && tok != uint32_t(f)) {
    record_error(t.status, CG_DEV_FORCED_MISMATCH);
    q = CG_DEAD;
    fl = CG_FLAG_REJECTED;
  } else {
    RowStack st{row + 2};
    if (pda_walk(pv, t, tok, f >= 0 ? 256u : 0u, q, lvl, st)) {
      fl = pda_flags(pv, q, lvl, st);
    } else {
      record_error(t.status, CG_DEV_REJECTED);
      q = CG_DEAD;
      fl = CG_FLAG_REJECTED;
    }
  }
  if (q == CG_DEAD) lvl = 0;
  if (counts) {
    uint32_t n = n0 + (tok != CG_NO_TOKEN ? 1u : 0u);
    if ((fl & CG_FLAG_DONE) || n >= max_tokens) {
      if (!(fl & CG_FLAG_DONE)) fl |= CG_FLAG_CAPPED;
      q = 0u;
      lvl = 0u;
      n = 0u;
    }
    counts[b] = n;
  }
  row[0] = q;
  row[1] = lvl;
  return fl;
}

}  // namespace cgk
