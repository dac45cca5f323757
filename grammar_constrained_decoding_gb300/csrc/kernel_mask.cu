// Bitmask fill: which vocabulary tokens the grammar allows in each row's state
// (usetacet.com/docs/grammar, "The guarantee").  Masks are cached per mask
// class (states that allow the same tokens), "the token mask cache makes the
// surrounding constraints near-free" (labs.miniml.ai "Evaluator aware
// decoding", "Where XGrammar-2 could take this"); a class is computed the first
// time a row needs it.
//
// One CTA per row.  A cache hit copies one W-word row (L2-resident cache).  A
// miss walks every token's bytes through the transition table in trie
// (lexicographic) order: each thread takes a contiguous run of the sorted
// vocabulary and resumes each token's walk from the state reached after the
// prefix it shares with the previous token, so shared prefixes are walked
// once.  Allowed tokens set their bit (token-id order) in a shared-memory mask.
#include "device.cuh"

namespace cgk {

constexpr int kFillThreads = 512;
constexpr uint32_t kStateEmpty = 0, kStateBusy = 1, kStateReady = 2;

__device__ __forceinline__ uint32_t load_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void store_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Walk all tokens from state s of grammar g; sets allowed bits in smask[W].
__device__ void walk_tokens(const Tables& t, const DevGrammar& gd, const uint16_t* scol, uint32_t s,
                            uint32_t* smask) {
  const uint32_t V = t.V;
  const uint32_t per = (V + blockDim.x - 1) / blockDim.x;
  const uint32_t i0 = threadIdx.x * per;
  const uint32_t i1 = min(V, i0 + per);
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

__global__ void __launch_bounds__(kFillThreads) fill_bitmask_kernel(Tables t, const uint32_t* __restrict__ states,
                                                                      const uint16_t* __restrict__ gid,
                                                                      const int32_t* __restrict__ forced,
                                                                      uint32_t* __restrict__ bitmask) {
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
  int mode = 0;  // 0 lookup, 1 zero row, 2 one-hot row
  if (g >= t.n_g) mode = 1;
  else if (f >= 0) mode = (uint32_t(f) < t.V) ? 2 : 1;
  else if (s == CG_DEAD || s >= t.grammars[g].n_states) mode = 1;
  else if (t.state_flags[t.grammars[g].state_off + s] & CG_STATE_FORCED_ONLY) mode = 1;
  if (threadIdx.x == 0) {
    if (g >= t.n_g) record_error(t.status, CG_DEV_BAD_GID);
    else if (f >= 0 && uint32_t(f) >= t.V) record_error(t.status, CG_DEV_BAD_FORCED);
    else if (f < 0 && s != CG_DEAD && s >= t.grammars[g].n_states) record_error(t.status, CG_DEV_BAD_STATE);
    else if (mode == 1 && f < 0 && s != CG_DEAD) record_error(t.status, CG_DEV_MISSING_FORCED);
  }
  if (mode != 0) {
    for (uint32_t i = threadIdx.x; i < W; i += blockDim.x)
      out[i] = (mode == 2 && i == (uint32_t(f) >> 5)) ? (1u << (f & 31)) : 0u;
    return;
  }

  const DevGrammar gd = t.grammars[g];
  const uint32_t cls = t.class_of[gd.state_off + s];
  const uint32_t* crow = t.cache + size_t(cls) * W;
  // one thread reads the flag so that the whole block takes the same path
  if (threadIdx.x == 0) s_ready = load_acquire(t.cache_state + cls) == kStateReady;
  __syncthreads();
  if (s_ready) {
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
  walk_tokens(t, gd, scol, s, smask);
  __syncthreads();
  const bool claimed = s_claim != 0u;
  uint32_t* cw = t.cache + size_t(cls) * W;
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
  walk_tokens(t, t.grammars[g], scol, class_rep[cls], smask);
  __syncthreads();
  uint32_t* cw = t.cache + size_t(cls) * W;
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
                                uint32_t B, uint32_t* bitmask, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  const size_t smem = size_t(t.W) * 4 + 256 * 2;
  return launch_dependent(fill_bitmask_kernel, dim3(B), dim3(kFillThreads), smem, stream, t, states, gid, forced,
                          bitmask);
}

size_t fill_bitmask_smem(uint32_t W) { return size_t(W) * 4 + 256 * 2; }

}  // namespace cgk
