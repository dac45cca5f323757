// Bitmask fill: which vocabulary tokens the grammar allows in each row's state
// (usetacet.com/docs/grammar, "The guarantee").  Masks are cached per mask
// class (states that allow the same tokens), which is what keeps grammar
// constraints cheap (labs.miniml.ai "Evaluator aware decoding", "Where
// XGrammar-2 could take this", on the token mask cache); a class is computed
// the first time a row needs it.
//
// One CTA per row.  A cache hit copies one W-word row (L2-resident cache).  A
// miss walks every token's bytes through the transition table in trie
// (lexicographic) order: each thread takes a contiguous run of the sorted
// vocabulary and resumes each token's walk from the state reached after the
// prefix it shares with the previous token, so shared prefixes are walked
// once.  Allowed tokens set their bit (token-id order) in a shared-memory mask.
#include <algorithm>

#include "row_ops.cuh"

namespace cgk {

constexpr int kFillThreads = 512;

__global__ void __launch_bounds__(kFillThreads) fill_bitmask_kernel(Tables t, const uint32_t* __restrict__ states,
                                                                      const uint16_t* __restrict__ gid,
                                                                      const int32_t* __restrict__ forced,
                                                                      uint32_t* __restrict__ bitmask,
                                                                      uint32_t cache_complete) {
  extern __shared__ uint32_t smem[];
  uint32_t* smask = smem;                                   // [W]
  uint16_t* scol = reinterpret_cast<uint16_t*>(smem + t.W); // [256] model-byte columns
  __shared__ uint32_t s_claim, s_ready;
  griddep_launch_dependents();
  griddep_wait();  // states (and forced tokens) come from the previous step
  const uint32_t b = blockIdx.x, W = t.W;
  uint32_t* out = bitmask + size_t(b) * W;
  const uint32_t g = gid ? gid[b] : 0u;
  const int32_t f = forced ? forced[b] : -1;
  const uint32_t s = states[b];

  // rows that do not read the cache: bad grammar, forced token, dead or bad state
  uint32_t err = 0;
  const int mode = row_mask_mode(t, g, f, s, &err);  // 0 lookup, 1 zero row, 2 one-hot row
  if (threadIdx.x == 0 && err) record_error(t.status, err);
  if (mode != 0) {
    for (uint32_t i = threadIdx.x; i < W; i += blockDim.x)
      out[i] = (mode == 2 && i == (uint32_t(f) >> 5)) ? (1u << (f & 31)) : 0u;
    return;
  }

  const DevGrammar gd = t.grammars[g];
  const uint32_t cls = t.class_of[gd.state_off + s];
  const uint32_t* crow = t.cache + size_t(cls) * t.Wc;
  // one thread reads the flag so that the whole block takes the same path;
  // after cg_ctx_prefill every class is ready and the flag is not read
  if (!cache_complete) {
    if (threadIdx.x == 0) s_ready = load_acquire(t.cache_state + cls) == kStateReady;
    __syncthreads();
  }
  if (cache_complete || s_ready) {
    if ((W & 3u) == 0) {
      const uint4* src = reinterpret_cast<const uint4*>(crow);
      uint4* dst = reinterpret_cast<uint4*>(out);
      for (uint32_t i = threadIdx.x; i < W / 4; i += blockDim.x) dst[i] = src[i];
    } else {
      for (uint32_t i = threadIdx.x; i < W; i += blockDim.x) out[i] = crow[i];
    }
    return;
  }

  // miss: compute the class mask from state s
  for (uint32_t i = threadIdx.x; i < W; i += blockDim.x) smask[i] = 0u;
  for (uint32_t i = threadIdx.x; i < 256; i += blockDim.x) scol[i] = t.colmap[size_t(g) * 512 + i];
  if (threadIdx.x == 0) s_claim = atomicCAS(t.cache_state + cls, kStateEmpty, kStateBusy) == kStateEmpty;
  __syncthreads();
  walk_tokens(t, gd, scol, s, smask, threadIdx.x, blockDim.x);
  __syncthreads();
  const bool claimed = s_claim != 0u;
  uint32_t* cw = t.cache + size_t(cls) * t.Wc;
  for (uint32_t i = threadIdx.x; i < W; i += blockDim.x) {
    const uint32_t w = smask[i];
    out[i] = w;
    if (claimed) cw[i] = w;
  }
  if (claimed) {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) store_release(t.cache_state + cls, kStateReady);
  }
}

// The miss pre-pass of the fused steps and of fill_bitmask (contexts without
// cg_ctx_prefill): every class mask the rows need is computed before the step,
// each by kMissSplits blocks that share its walk (a 1/kMissSplits share of the
// trie order each), so that a miss costs a short walk instead of one block
// walking the whole vocabulary.  Block (x, y) checks rows
// [y R, (y + 1) R), R = ceil(B / gridDim.y), one thread a row; for each row
// whose class is not ready it claims split x of the class (a bit in
// cache_claim: one block computes each split, whichever row asked), ORs the
// split's bits into the class's cache row (zero until then), and the block
// that finishes the last split marks the class ready.  stats[0] counts the
// rows that looked a class up, stats[1] the classes computed.
constexpr uint32_t kMissSplits = 32;
constexpr int kMissThreads = 256;
constexpr uint32_t kMissRowsMax = kMissThreads;  // rows a block checks (one thread each)

__global__ void __launch_bounds__(kMissThreads) cache_fill_kernel(Tables t, const uint32_t* __restrict__ states,
                                                                    const uint16_t* __restrict__ gid,
                                                                    const int32_t* __restrict__ forced, uint32_t B,
                                                                    unsigned long long* stats) {
  extern __shared__ uint32_t smem[];
  uint32_t* smask = smem;                                    // [W]
  uint16_t* scol = reinterpret_cast<uint16_t*>(smem + t.W);  // [256]
  __shared__ uint32_t s_n, s_cls[kMissRowsMax], s_st[kMissRowsMax], s_g[kMissRowsMax];
  griddep_launch_dependents();
  griddep_wait();  // states (and forced tokens) come from the previous step
  const uint32_t tid = threadIdx.x, split = blockIdx.x, W = t.W;
  const uint32_t R = (B + gridDim.y - 1) / gridDim.y, b0 = blockIdx.y * R;
  if (tid == 0) s_n = 0u;
  __syncthreads();
  if (tid < R && b0 + tid < B) {
    const uint32_t b = b0 + tid;
    const uint32_t g = gid ? gid[b] : 0u;
    const int32_t f = forced ? forced[b] : -1;
    const uint32_t s = states[b];
    uint32_t err = 0;
    if (row_mask_mode(t, g, f, s, &err) == 0) {  // errors are the step kernel's to record
      const uint32_t cls = t.class_of[t.grammars[g].state_off + s];
      if (split == 0) atomicAdd(stats, 1ull);
      const uint32_t bit = 1u << split;
      if (load_acquire(t.cache_state + cls) != kStateReady && !(atomicOr(t.cache_claim + cls, bit) & bit)) {
        const uint32_t k = atomicAdd(&s_n, 1u);
        s_cls[k] = cls;
        s_st[k] = s;
        s_g[k] = g;
      }
    }
  }
  __syncthreads();
  const uint32_t n = s_n, per = (t.V + kMissSplits - 1) / kMissSplits;
  const uint32_t lo = min(t.V, split * per), hi = min(t.V, lo + per);
  for (uint32_t k = 0; k < n; ++k) {
    const uint32_t cls = s_cls[k], g = s_g[k];
    for (uint32_t i = tid; i < W; i += blockDim.x) smask[i] = 0u;
    for (uint32_t i = tid; i < 256; i += blockDim.x) scol[i] = t.colmap[size_t(g) * 512 + i];
    __syncthreads();
    walk_tokens_range(t, t.grammars[g], scol, s_st[k], smask, lo, hi, tid, blockDim.x);
    __syncthreads();
    uint32_t* cw = t.cache + size_t(cls) * t.Wc;
    for (uint32_t i = tid; i < W; i += blockDim.x)
      if (smask[i]) atomicOr(cw + i, smask[i]);
    __threadfence();
    __syncthreads();
    if (tid == 0 && atomicAdd(t.cache_done + cls, 1u) == kMissSplits - 1) {
      __threadfence();
      store_release(t.cache_state + cls, kStateReady);
      atomicAdd(stats + 1, 1ull);
    }
  }
}

// One CTA per mask class: computes every class mask ahead of the decode steps.
__global__ void __launch_bounds__(kFillThreads) prefill_kernel(Tables t, const uint32_t* __restrict__ class_rep,
                                                                 const uint16_t* __restrict__ class_gid) {
  extern __shared__ uint32_t smem[];
  uint32_t* smask = smem;
  uint16_t* scol = reinterpret_cast<uint16_t*>(smem + t.W);
  const uint32_t cls = blockIdx.x, W = t.W;
  if (load_acquire(t.cache_state + cls) == kStateReady) return;  // uniform: no other writer runs meanwhile
  const uint32_t g = class_gid[cls];
  for (uint32_t i = threadIdx.x; i < W; i += blockDim.x) smask[i] = 0u;
  for (uint32_t i = threadIdx.x; i < 256; i += blockDim.x) scol[i] = t.colmap[size_t(g) * 512 + i];
  __syncthreads();
  walk_tokens(t, t.grammars[g], scol, class_rep[cls], smask, threadIdx.x, blockDim.x);
  __syncthreads();
  uint32_t* cw = t.cache + size_t(cls) * t.Wc;
  for (uint32_t i = threadIdx.x; i < W; i += blockDim.x) cw[i] = smask[i];
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) store_release(t.cache_state + cls, kStateReady);
}

cudaError_t launch_prefill(const Tables& t, const uint32_t* class_rep, const uint16_t* class_gid,
                           cudaStream_t stream) {
  if (t.n_classes == 0) return cudaSuccess;
  const size_t smem = size_t(t.W) * 4 + 256 * 2;
  prefill_kernel<<<t.n_classes, kFillThreads, smem, stream>>>(t, class_rep, class_gid);
  return cudaGetLastError();
}

cudaError_t launch_fill_bitmask(const Tables& t, const uint32_t* states, const uint16_t* gid, const int32_t* forced,
                                uint32_t B, uint32_t* bitmask, bool cache_complete, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  const size_t smem = size_t(t.W) * 4 + 256 * 2;
  return launch_dependent(fill_bitmask_kernel, dim3(B), dim3(kFillThreads), smem, stream, t, states, gid, forced,
                          bitmask, cache_complete ? 1u : 0u);
}

size_t fill_bitmask_smem(uint32_t W) { return size_t(W) * 4 + 256 * 2; }

cudaError_t launch_cache_fill(const Tables& t, const uint32_t* states, const uint16_t* gid, const int32_t* forced,
                              uint32_t B, unsigned long long* stats, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  const size_t smem = size_t(t.W) * 4 + 256 * 2;
  // about 8 rows a block (one thread each), every row group with all its splits
  const uint32_t groups = std::max((B + 7) / 8, (B + kMissRowsMax - 1) / kMissRowsMax);
  return launch_dependent(cache_fill_kernel, dim3(kMissSplits, groups), dim3(kMissThreads), smem, stream, t, states,
                          gid, forced, B, stats);
}

}  // namespace cgk
