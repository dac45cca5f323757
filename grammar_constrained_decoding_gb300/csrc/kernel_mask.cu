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

// The fused step's miss path: one CTA per row computes the mask of the row's
// class when it is not in the cache yet (claiming it first, so that one row
// computes each class); rows whose class is ready, or claimed by another row
// of the same launch, do nothing.  After this grid every class the rows need
// is ready.  stats[0] counts the rows that looked a class up, stats[1] the
// classes computed.
__global__ void __launch_bounds__(kFillThreads) cache_fill_kernel(Tables t, const uint32_t* __restrict__ states,
                                                                    const uint16_t* __restrict__ gid,
                                                                    const int32_t* __restrict__ forced,
                                                                    unsigned long long* stats) {
  extern __shared__ uint32_t smem[];
  uint32_t* smask = smem;
  uint16_t* scol = reinterpret_cast<uint16_t*>(smem + t.W);
  __shared__ uint32_t s_claim;
  griddep_launch_dependents();
  griddep_wait();  // states (and forced tokens) come from the previous step
  const uint32_t b = blockIdx.x, W = t.W;
  const uint32_t g = gid ? gid[b] : 0u;
  const int32_t f = forced ? forced[b] : -1;
  const uint32_t s = states[b];
  uint32_t err = 0;
  if (row_mask_mode(t, g, f, s, &err) != 0) return;  // errors are the step kernel's to record
  const DevGrammar gd = t.grammars[g];
  const uint32_t cls = t.class_of[gd.state_off + s];
  if (threadIdx.x == 0) {
    atomicAdd(stats, 1ull);
    s_claim = load_acquire(t.cache_state + cls) != kStateReady &&
              atomicCAS(t.cache_state + cls, kStateEmpty, kStateBusy) == kStateEmpty;
  }
  __syncthreads();
  if (!s_claim) return;
  for (uint32_t i = threadIdx.x; i < W; i += blockDim.x) smask[i] = 0u;
  for (uint32_t i = threadIdx.x; i < 256; i += blockDim.x) scol[i] = t.colmap[size_t(g) * 512 + i];
  __syncthreads();
  walk_tokens(t, gd, scol, s, smask, threadIdx.x, blockDim.x);
  __syncthreads();
  uint32_t* cw = t.cache + size_t(cls) * t.Wc;
  for (uint32_t i = threadIdx.x; i < W; i += blockDim.x) cw[i] = smask[i];
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    store_release(t.cache_state + cls, kStateReady);
    atomicAdd(stats + 1, 1ull);
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
  return launch_dependent(cache_fill_kernel, dim3(B), dim3(kFillThreads), smem, stream, t, states, gid, forced,
                          stats);
}

}  // namespace cgk
