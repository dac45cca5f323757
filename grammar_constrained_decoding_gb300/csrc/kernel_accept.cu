// Accept: advance each row's automaton by its token ("after injection the
// grammar state must be advanced ... so the forced tokens are legal",
// labs.miniml.ai "Evaluator aware decoding", "A concrete prototype on
// llama.cpp").  One thread per row; a forced token's bytes are walked as
// host-injected symbols.  With token counts the finished or capped rows are
// reset to the start state (usetacet.com/docs/grammar, "A valid call also has
// to end": generations are capped).
#include "device.cuh"

namespace cgk {

constexpr int kAcceptThreads = 128;
constexpr uint32_t kPrefetch = 16;  // token bytes whose columns are loaded up front

__global__ void __launch_bounds__(kAcceptThreads) accept_kernel(Tables t, const uint32_t* __restrict__ states,
                                                                const uint16_t* __restrict__ gid,
                                                                const uint32_t* __restrict__ toks,
                                                                const int32_t* __restrict__ forced, uint32_t B,
                                                                uint32_t* counts, uint32_t max_tokens,
                                                                uint32_t* out_states, uint8_t* out_flags) {
  griddep_launch_dependents();
  griddep_wait();  // the tokens come from the sampling kernel
  const uint32_t b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const uint32_t g = gid ? gid[b] : 0u;
  const uint32_t s = states[b];
  const uint32_t tok = toks[b];
  const int32_t f = forced ? forced[b] : -1;
  uint32_t ns = s;
  uint8_t fl = 0;
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
      const uint32_t shift = f >= 0 ? 256u : 0u;
      const uint16_t* cols = t.colmap + size_t(g) * 512 + shift;
      const uint32_t* table = t.table + gd.table_off;
      // the token's columns first (independent loads), then the chain of
      // table lookups
      const uint32_t i0 = t.tok_off[tok], len = t.tok_off[tok + 1] - i0;
      uint32_t col[kPrefetch];
#pragma unroll
      for (uint32_t k = 0; k < kPrefetch; ++k) col[k] = k < len ? cols[t.tok_bytes[i0 + k]] : 0u;
      uint32_t st = s;
#pragma unroll
      for (uint32_t k = 0; k < kPrefetch; ++k)
        if (k < len && st != CG_DEAD) st = table[size_t(st) * gd.n_cols + col[k]];
      for (uint32_t i = i0 + kPrefetch; i < i0 + len && st != CG_DEAD; ++i)
        st = table[size_t(st) * gd.n_cols + cols[t.tok_bytes[i]]];
      ns = st;
      if (st == CG_DEAD) {
        record_error(t.status, CG_DEV_REJECTED);
        fl = CG_FLAG_REJECTED;
      } else {
        const uint8_t sf = t.state_flags[gd.state_off + st];
        if (sf & CG_STATE_SINK) fl |= CG_FLAG_DONE;
        if (sf & CG_STATE_FORCED_ONLY) fl |= CG_FLAG_FORCED_NEXT;
      }
    }
  }
  if (counts) {
    uint32_t n = counts[b] + (tok != CG_NO_TOKEN ? 1u : 0u);
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

cudaError_t launch_accept(const Tables& t, const uint32_t* states, const uint16_t* gid, const uint32_t* toks,
                          const int32_t* forced, uint32_t B, uint32_t* counts, uint32_t max_tokens,
                          uint32_t* out_states, uint8_t* out_flags, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  return launch_dependent(accept_kernel, dim3((B + kAcceptThreads - 1) / kAcceptThreads), dim3(kAcceptThreads), 0,
                          stream, t, states, gid, toks, forced, B, counts, max_tokens, out_states, out_flags);
}

}  // namespace cgk
