// Pushdown rows on the device (cg_pda_*): each row carries its state and a
// stack of return states (usetacet.com/docs/grammar, "The guarantee": the
// automaton that masks the logits is a pushdown automaton).
//
// Mask of a row in state q at level L (headroom depth - L):
//  * the cached part: tokens whose walk from q never pops below the row's own
//    frame.  Whether such a token is allowed depends only on q and on the
//    headroom (calls it opens must fit), so the host walks every token once
//    per state at creation, records the least headroom each needs, and keeps
//    one mask per (state, headroom up to the largest need), shared where equal;
//  * the per-row part: tokens whose walk pops below the row's frame (they end
//    the rule and continue in the caller).  Their fate depends on the stack,
//    so the fill kernel walks them against the row's own stack, in parallel
//    over the block's threads, and ORs the allowed ones into the cached mask.
// Accept walks the sampled token through the actions one thread per row,
// updating the row's state and stack in place.
#include <algorithm>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "pda.cuh"

namespace cgk {

constexpr uint32_t kPdaFillThreads = 256;
constexpr uint32_t kPdaVec = 8;  // uint4s of the row's mask a fill thread holds in registers

// Fills row b's mask for configuration (q, lvl) with the stack at row + 2;
// all threads of the block take part.  pv: the walk tables (in shared memory
// when tabs_in_smem, copied there by the caller and synchronised);
// bits / stk: shared scratch of W and depth words.
__device__ void pda_fill_row(const DevPda& p, const DevPda& pv, const Tables& t, uint32_t q, uint32_t lvl,
                             const uint32_t* row, int32_t f, uint32_t* __restrict__ out, uint32_t* bits,
                             uint32_t* stk) {
  const uint32_t W = t.W, tid = threadIdx.x;
  const bool ok = q < p.S && lvl <= p.depth;
  if (f >= 0 || !ok) {
    // forced row: exactly that token; failed or malformed row: nothing
    if (tid == 0) {
      if (f >= 0 && uint32_t(f) >= t.V) record_error(t.status, CG_DEV_BAD_FORCED);
      else if (f < 0 && q != CG_DEAD) record_error(t.status, CG_DEV_BAD_STATE);
    }
    const bool one = f >= 0 && uint32_t(f) < t.V;
    for (uint32_t w = tid; w < W; w += blockDim.x)
      out[w] = (one && w == uint32_t(f) >> 5) ? (1u << (uint32_t(f) & 31u)) : 0u;
    return;
  }
  const uint32_t kinfo = p.key[q], hr = p.depth - lvl;
  const uint32_t c0 = p.cand_off[q], c1 = p.cand_off[q + 1];
  const uint32_t* __restrict__ src = p.masks + size_t(p.mask_of[(kinfo >> 8) + min(hr, kinfo & 0xFFu)]) * W;
  // the cached mask: every load issued at once (into registers when the row
  // fits kPdaVec uint4s per thread), before the per-row walks
  const uint32_t W4 = W / 4;
  const bool vec = (W & 3u) == 0 && W4 <= kPdaVec * blockDim.x;
  uint4 v[kPdaVec];
  if (vec) {
    const uint4* __restrict__ s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (uint32_t k = 0; k < kPdaVec; ++k) {
      const uint32_t i = tid + k * blockDim.x;
      if (i < W4) v[k] = s4[i];
    }
  }
  uint4* o4 = reinterpret_cast<uint4*>(out);
  if (c0 == c1) {  // nothing decided per row: the cached mask as is
    if (vec) {
#pragma unroll
      for (uint32_t k = 0; k < kPdaVec; ++k) {
        const uint32_t i = tid + k * blockDim.x;
        if (i < W4) o4[i] = v[k];
      }
    } else {
      for (uint32_t w = tid; w < W; w += blockDim.x) out[w] = src[w];
    }
    return;
  }
  for (uint32_t w = tid; w < W; w += blockDim.x) bits[w] = 0u;
  for (uint32_t i = tid; i < lvl; i += blockDim.x) stk[i] = row[2 + i];
  __syncthreads();
  for (uint32_t i = c0 + tid; i < c1; i += blockDim.x) {
    const uint32_t tok = p.cand[i];
    uint32_t qq = q, ll = lvl;
    OverlayStack st;
    st.base = stk;
    st.keep = lvl;
    if (pda_walk(pv, t, tok, 0u, qq, ll, st)) atomicOr(&bits[tok >> 5], 1u << (tok & 31u));
  }
  __syncthreads();
  if (vec) {
    const uint4* b4 = reinterpret_cast<const uint4*>(bits);
#pragma unroll
    for (uint32_t k = 0; k < kPdaVec; ++k) {
      const uint32_t i = tid + k * blockDim.x;
      if (i < W4) {
        const uint4 x = b4[i];
        o4[i] = make_uint4(v[k].x | x.x, v[k].y | x.y, v[k].z | x.z, v[k].w | x.w);
      }
    }
  } else {
    for (uint32_t w = tid; w < W; w += blockDim.x) out[w] = src[w] | bits[w];
  }
}

// shared memory of a fill block: [tables (when they fit)] [W bits] [the row's stack]
__device__ __forceinline__ uint32_t* fill_bits(const DevPda& p, uint4* sm4) {
  return reinterpret_cast<uint32_t*>(sm4 + (p.tabs_in_smem ? p.tab_n16 : 0u));
}

__global__ void __launch_bounds__(kPdaFillThreads)
    pda_fill_kernel(DevPda p, Tables t, const uint32_t* __restrict__ cfg, const int32_t* __restrict__ forced,
                    uint32_t* __restrict__ bitmask) {
  extern __shared__ __align__(16) uint4 sm4[];
  griddep_launch_dependents();
  const DevPda pv = p.tabs_in_smem ? tables_to_smem(p, sm4, threadIdx.x, blockDim.x) : p;
  griddep_wait();  // configurations come from the previous accept
  const uint32_t b = blockIdx.x;
  const uint32_t* row = cfg + size_t(b) * p.stride;
  uint32_t* bits = fill_bits(p, sm4);
  pda_fill_row(p, pv, t, row[0], row[1], row, forced ? forced[b] : -1, bitmask + size_t(b) * t.W, bits,
               bits + t.W);
}

constexpr uint32_t kPdaAcceptThreads = 128;

__global__ void __launch_bounds__(kPdaAcceptThreads)
    pda_accept_kernel(DevPda p, Tables t, uint32_t* __restrict__ cfg, uint32_t B, const uint32_t* __restrict__ toks,
                      const int32_t* __restrict__ forced, uint32_t* counts, uint32_t max_tokens,
                      uint8_t* __restrict__ out_flags) {
  extern __shared__ __align__(16) uint4 sm4[];  // the walk tables, when they fit
  griddep_launch_dependents();
  const DevPda pv = p.tabs_in_smem ? tables_to_smem(p, sm4, threadIdx.x, blockDim.x) : p;
  if (p.tabs_in_smem) __syncthreads();
  griddep_wait();  // the tokens come from the sampling kernel
  const uint32_t b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  out_flags[b] = pda_accept_row(p, pv, t, cfg + size_t(b) * p.stride, b, toks[b], forced ? forced[b] : -1, counts,
                                max_tokens);
}

// Speculative verification of pushdown rows (cg_pda_accept_many), one thread
// per row: the draft's tokens are walked one after another, each on an
// overlay of the row's stack that is written back only when the token is
// accepted, so a refused token leaves the accepted prefix's configuration.
// The rules are those of cg_accept_many: stop at the first refused token
// (CG_FLAG_DRAFT_CUT), after a token that ends the grammar, at the token cap,
// or after a token whose configuration continues only with injected bytes when
// the next position is not pinned.
__global__ void __launch_bounds__(kPdaAcceptThreads)
    pda_accept_many_kernel(DevPda p, Tables t, uint32_t* __restrict__ cfg, uint32_t B,
                           const uint32_t* __restrict__ draft, const uint32_t* __restrict__ draft_len,
                           const int32_t* __restrict__ forced, uint32_t K, uint32_t* counts, uint32_t max_tokens,
                           uint32_t* __restrict__ out_n, uint8_t* __restrict__ out_flags) {
  extern __shared__ __align__(16) uint4 sm4[];  // the walk tables, when they fit
  griddep_launch_dependents();
  const DevPda pv = p.tabs_in_smem ? tables_to_smem(p, sm4, threadIdx.x, blockDim.x) : p;
  if (p.tabs_in_smem) __syncthreads();
  griddep_wait();  // drafts and configurations come from earlier work on the stream
  const uint32_t b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  uint32_t* row = cfg + size_t(b) * p.stride;
  const uint32_t* toks = draft + size_t(b) * K;
  const int32_t* fb = forced ? forced + size_t(b) * K : nullptr;
  uint32_t q = row[0], lvl = row[1], n = draft_len[b];
  uint32_t c = counts ? counts[b] : 0u, acc = 0;
  uint8_t fl = 0;
  if (n > K) {
    record_error(t.status, CG_DEV_BAD_LENGTH);
    n = K;
  }
  if (n == 0) {
    fl = CG_FLAG_NO_TOKEN;
  } else if (q == CG_DEAD) {
    fl = CG_FLAG_REJECTED;
  } else if (q >= p.S || lvl > p.depth) {
    record_error(t.status, CG_DEV_BAD_STATE);
    q = CG_DEAD;
    fl = CG_FLAG_REJECTED;
  } else {
    RowStack rs{row + 2};
    uint8_t cut = 0, capped = 0, sres = pda_flags(pv, q, lvl, rs);
    int32_t f = fb ? fb[0] : -1;
    for (uint32_t j = 0; j < n; ++j) {
      const uint32_t tok = toks[j];
      const int32_t f_next = (fb && j + 1 < n) ? fb[j + 1] : -1;
      if (tok >= t.V) {
        record_error(t.status, CG_DEV_BAD_TOKEN);
        cut = CG_FLAG_DRAFT_CUT;
        break;
      }
      OverlayStack st;
      st.base = row + 2;
      st.keep = lvl;
      uint32_t qq = q, ll = lvl;
      if ((f >= 0 && tok != uint32_t(f)) || !pda_walk(pv, t, tok, f >= 0 ? 256u : 0u, qq, ll, st)) {
        cut = CG_FLAG_DRAFT_CUT;
        break;
      }
      for (uint32_t i = st.keep; i < ll; ++i) row[2 + i] = st.local[i];  // the token's pushes
      q = qq;
      lvl = ll;
      ++acc;
      ++c;
      sres = pda_flags(pv, q, lvl, rs);
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
      q = 0u;
      lvl = 0u;
      c = 0u;
    }
  }
  if (q == CG_DEAD) lvl = 0;
  if (counts) counts[b] = c;
  row[0] = q;
  row[1] = lvl;
  out_n[b] = acc;
  out_flags[b] = fl;
}

// Accept of this step and fill of the next in one block per row: thread 0
// advances the row, the block then fills its next mask from the new
// configuration (the __syncthreads between them orders the row's global
// writes before the block's reads).
__global__ void __launch_bounds__(kPdaFillThreads)
    pda_accept_fill_kernel(DevPda p, Tables t, uint32_t* __restrict__ cfg, const uint32_t* __restrict__ toks,
                           const int32_t* __restrict__ forced, uint32_t* counts, uint32_t max_tokens,
                           uint8_t* __restrict__ out_flags, const int32_t* __restrict__ forced_next,
                           uint32_t* __restrict__ bitmask) {
  extern __shared__ __align__(16) uint4 sm4[];
  __shared__ uint32_t s_cfg[2];
  griddep_launch_dependents();
  const DevPda pv = p.tabs_in_smem ? tables_to_smem(p, sm4, threadIdx.x, blockDim.x) : p;
  if (p.tabs_in_smem) __syncthreads();
  griddep_wait();  // the tokens come from the sampling kernel
  const uint32_t b = blockIdx.x;
  uint32_t* row = cfg + size_t(b) * p.stride;
  if (threadIdx.x == 0) {
    out_flags[b] = pda_accept_row(p, pv, t, row, b, toks[b], forced ? forced[b] : -1, counts, max_tokens);
    s_cfg[0] = row[0];
    s_cfg[1] = row[1];
  }
  __syncthreads();
  uint32_t* bits = fill_bits(p, sm4);
  pda_fill_row(p, pv, t, s_cfg[0], s_cfg[1], row, forced_next ? forced_next[b] : -1, bitmask + size_t(b) * t.W,
               bits, bits + t.W);
}

}  // namespace cgk

struct cg_pda {
  cg_ctx* ctx = nullptr;
  cudaStream_t stream = nullptr;
  uint32_t* step_bitmask = nullptr;  // cg_pda_step's unfused path when the caller gives no bitmask
  size_t step_bitmask_bytes = 0;
  cgk::Tables t{};
  cgk::DevPda d{};
  std::vector<void*> allocations;
  uint32_t n_keys = 0, n_masks = 0, n_cand = 0;
  uint64_t cache_bytes = 0;
};

namespace cgk {
cudaError_t allow_smem(const void* kernel, size_t bytes);  // kernel_sample.cu
bool step_fusable(int dtype, uint32_t V, uint32_t W, float temp, float top_p, const void* logits);
size_t sample_scratch_bytes(uint32_t B, uint32_t V);
cudaError_t launch_pda_step(const Tables& t, const DevPda& pda, uint32_t* cfg, const int32_t* forced, uint32_t B,
                            void* logits, uint32_t V, float temp, float top_p, uint64_t seed, uint32_t step,
                            uint32_t* counts, uint32_t max_tokens, uint32_t* bitmask_out, uint32_t* out_tok,
                            uint8_t* out_flags, void* scratch, cudaStream_t stream);
}

namespace {

size_t pda_fill_smem(const cgk::DevPda& d, uint32_t W) {
  return (d.tabs_in_smem ? size_t(d.tab_n16) * 16 : 0) + (size_t(W) + d.depth) * 4;
}
size_t pda_accept_smem(const cgk::DevPda& d) { return d.tabs_in_smem ? size_t(d.tab_n16) * 16 : 0; }

void pda_release(cg_pda* p) {
  for (void* a : p->allocations) cudaFree(a);
  p->allocations.clear();
  if (p->step_bitmask) cudaFree(p->step_bitmask);
  p->step_bitmask = nullptr;
  p->step_bitmask_bytes = 0;
}

template <typename T>
cudaError_t pda_upload(cg_pda* p, const std::vector<T>& host, const T** dev) {
  void* d = nullptr;
  cudaError_t e = cudaMalloc(&d, std::max<size_t>(host.size() * sizeof(T), 16));
  if (e != cudaSuccess) return e;
  p->allocations.push_back(d);
  *dev = static_cast<const T*>(d);
  if (host.empty()) return cudaSuccess;
  return cudaMemcpyAsync(d, host.data(), host.size() * sizeof(T), cudaMemcpyHostToDevice, p->stream);
}

// Distinct masks of W words, by content.
struct MaskSet {
  uint32_t W;
  std::vector<uint32_t> words;
  std::unordered_multimap<uint64_t, uint32_t> at;
  uint32_t intern(const std::vector<uint32_t>& m) {
    uint64_t hsh = 1469598103934665603ull;
    for (uint32_t x : m) { hsh ^= x; hsh *= 1099511628211ull; }
    auto range = at.equal_range(hsh);
    for (auto it = range.first; it != range.second; ++it)
      if (std::memcmp(words.data() + size_t(it->second) * W, m.data(), size_t(W) * 4) == 0) return it->second;
    const uint32_t idx = uint32_t(words.size() / W);
    words.insert(words.end(), m.begin(), m.end());
    at.emplace(hsh, idx);
    return idx;
  }
};

}  // namespace

extern "C" {

int cg_pda_create(cg_ctx* c, const cg_vocab* v, const cg_pda_grammar* g, cg_pda** out) {
  if (!c || !v || !g || !out) return CG_E_ARG;
  *out = nullptr;
  cgk::DeviceGuard dg(cgk::ctx_device(c), "cg_pda_create");
  if (!dg.ok) return CG_E_CUDA;
  const cgk::CtxView view = cgk::ctx_view(c);
  if (v->V != view.t.V) return CG_E_ARG;
  const uint32_t V = v->V, W = view.t.W, S = g->n_states, D = g->depth;
  if ((size_t(W) + D) * 4 + cgk::kPdaSmemTables > 200 * 1024) return CG_E_LIMIT;
  cg_pda* p = new (std::nothrow) cg_pda;
  if (!p) return CG_E_NOMEM;
  p->ctx = c;
  p->stream = view.stream;
  p->t = view.t;
  std::vector<uint32_t> sinfo(S), key(S), mask_of, cand_off(S + 1, 0), cand;
  MaskSet ms{W, {}, {}};
  try {
    std::vector<uint32_t> need(V);
    std::vector<uint32_t> m(W);
    std::vector<std::vector<uint32_t>> by_need;
    for (uint32_t q = 0; q < S; ++q) {
      sinfo[q] = uint32_t(g->accept[q] ? 1u : 0u) | (uint32_t(g->h[q]) << 8) | (uint32_t(g->need_model[q]) << 16) |
                 (uint32_t(g->need_inj[q]) << 24);
      uint32_t cap = 0;
      for (uint32_t tk = 0; tk < V; ++tk) {
        const uint32_t r = cg::pda_token_need(*g, q, v->bytes.data() + v->off[tk], v->off[tk + 1] - v->off[tk]);
        need[tk] = r;
        if (r == cg::kPdaTokPop) cand.push_back(tk);
        else if (r != cg::kPdaTokDead) cap = std::max(cap, std::min(r, D));
      }
      cand_off[q + 1] = uint32_t(cand.size());
      // one key per headroom 0..cap (a larger headroom reads key cap)
      by_need.assign(cap + 1, {});
      for (uint32_t tk = 0; tk < V; ++tk)
        if (need[tk] <= cap) by_need[need[tk]].push_back(tk);
      if (mask_of.size() >= (1u << 24)) { delete p; return CG_E_LIMIT; }
      key[q] = (uint32_t(mask_of.size()) << 8) | cap;
      std::fill(m.begin(), m.end(), 0u);
      for (uint32_t hr = 0; hr <= cap; ++hr) {
        for (uint32_t tk : by_need[hr]) m[tk >> 5] |= 1u << (tk & 31u);
        mask_of.push_back(ms.intern(m));
      }
    }
  } catch (const std::bad_alloc&) {
    delete p;
    return CG_E_NOMEM;
  }
  p->n_keys = uint32_t(mask_of.size());
  p->n_masks = uint32_t(ms.words.size() / W);
  p->n_cand = uint32_t(cand.size());
  p->cache_bytes = uint64_t(ms.words.size()) * 4;
  cgk::DevPda& d = p->d;
  // the walk tables in one block: colmap, sinfo, act, chain, each 16-byte aligned
  std::vector<uint4> tabs;
  uint32_t off_sinfo = 0, off_act = 0, off_chain = 0;
  try {
    std::vector<unsigned char> blob;
    auto put = [&blob](const void* src, size_t bytes) {
      const uint32_t off = uint32_t(blob.size());
      blob.insert(blob.end(), static_cast<const unsigned char*>(src), static_cast<const unsigned char*>(src) + bytes);
      blob.resize((blob.size() + 15) & ~size_t(15), 0);
      return off;
    };
    put(g->col_of.data(), g->col_of.size() * 2);
    off_sinfo = put(sinfo.data(), sinfo.size() * 4);
    off_act = put(g->act.data(), g->act.size() * 4);
    off_chain = put(g->chain.data(), g->chain.size() * 4);
    tabs.resize(blob.size() / 16);
    std::memcpy(tabs.data(), blob.data(), blob.size());
  } catch (const std::bad_alloc&) {
    delete p;
    return CG_E_NOMEM;
  }
  cudaError_t e;
  if ((e = pda_upload(p, tabs, &d.tabs)) != cudaSuccess ||
      (e = pda_upload(p, key, &d.key)) != cudaSuccess || (e = pda_upload(p, mask_of, &d.mask_of)) != cudaSuccess ||
      (e = pda_upload(p, ms.words, &d.masks)) != cudaSuccess ||
      (e = pda_upload(p, cand_off, &d.cand_off)) != cudaSuccess || (e = pda_upload(p, cand, &d.cand)) != cudaSuccess ||
      (e = cudaStreamSynchronize(p->stream)) != cudaSuccess) {
    pda_release(p);
    delete p;
    return CG_E_CUDA;
  }
  const unsigned char* tb = reinterpret_cast<const unsigned char*>(d.tabs);
  d.colmap = reinterpret_cast<const uint16_t*>(tb);
  d.sinfo = reinterpret_cast<const uint32_t*>(tb + off_sinfo);
  d.act = reinterpret_cast<const uint32_t*>(tb + off_act);
  d.chain = reinterpret_cast<const uint32_t*>(tb + off_chain);
  d.tab_n16 = uint32_t(tabs.size());
  d.off_sinfo = off_sinfo;
  d.off_act = off_act;
  d.off_chain = off_chain;
  d.tabs_in_smem = size_t(d.tab_n16) * 16 <= cgk::kPdaSmemTables;
  d.S = S;
  d.n_cols = g->n_cols;
  d.depth = D;
  d.stride = D + 2;
  if (cgk::allow_smem(reinterpret_cast<const void*>(cgk::pda_fill_kernel), pda_fill_smem(d, W)) != cudaSuccess ||
      cgk::allow_smem(reinterpret_cast<const void*>(cgk::pda_accept_fill_kernel), pda_fill_smem(d, W)) !=
          cudaSuccess ||
      cgk::allow_smem(reinterpret_cast<const void*>(cgk::pda_accept_kernel), pda_accept_smem(d)) != cudaSuccess ||
      cgk::allow_smem(reinterpret_cast<const void*>(cgk::pda_accept_many_kernel), pda_accept_smem(d)) !=
          cudaSuccess) {
    pda_release(p);
    delete p;
    return CG_E_CUDA;
  }
  *out = p;
  return CG_OK;
}

void cg_pda_destroy(cg_pda* p) {
  if (!p) return;
  {
    cgk::DeviceGuard dg(cgk::ctx_device(p->ctx), "cg_pda_destroy");
    cudaStreamSynchronize(p->stream);
    pda_release(p);
  }
  delete p;
}

int cg_pda_info(const cg_pda* p, uint32_t* n_keys, uint32_t* n_masks, uint64_t* cache_bytes,
                uint32_t* n_candidates) {
  if (!p) return CG_E_ARG;
  if (n_keys) *n_keys = p->n_keys;
  if (n_masks) *n_masks = p->n_masks;
  if (cache_bytes) *cache_bytes = p->cache_bytes;
  if (n_candidates) *n_candidates = p->n_cand;
  return CG_OK;
}

int cg_pda_fill_bitmask(cg_pda* p, const uint32_t* d_cfg, uint32_t B, const int32_t* d_forced,
                        uint32_t* d_bitmask) {
  if (!p || (B && (!d_cfg || !d_bitmask))) return CG_E_ARG;
  if (B == 0) return CG_OK;
  cgk::DeviceGuard dg(cgk::ctx_device(p->ctx), "cg_pda_fill_bitmask");
  if (!dg.ok) return CG_E_CUDA;
  const size_t smem = pda_fill_smem(p->d, p->t.W);
  return cgk::launch_dependent(cgk::pda_fill_kernel, dim3(B), dim3(cgk::kPdaFillThreads), smem, p->stream, p->d,
                               p->t, d_cfg, d_forced, d_bitmask) == cudaSuccess
             ? CG_OK
             : CG_E_CUDA;
}

int cg_pda_accept(cg_pda* p, uint32_t* d_cfg, uint32_t B, const uint32_t* d_toks, const int32_t* d_forced,
                  uint32_t* d_counts, uint32_t max_tokens, uint8_t* d_out_flags) {
  if (!p || (B && (!d_cfg || !d_toks || !d_out_flags))) return CG_E_ARG;
  if (B == 0) return CG_OK;
  cgk::DeviceGuard dg(cgk::ctx_device(p->ctx), "cg_pda_accept");
  if (!dg.ok) return CG_E_CUDA;
  const uint32_t grid = (B + cgk::kPdaAcceptThreads - 1) / cgk::kPdaAcceptThreads;
  return cgk::launch_dependent(cgk::pda_accept_kernel, dim3(grid), dim3(cgk::kPdaAcceptThreads),
                               pda_accept_smem(p->d), p->stream,
                               p->d, p->t, d_cfg, B, d_toks, d_forced, d_counts, max_tokens, d_out_flags) ==
                 cudaSuccess
             ? CG_OK
             : CG_E_CUDA;
}

int cg_pda_accept_many(cg_pda* p, uint32_t* d_cfg, uint32_t B, const uint32_t* d_draft, const uint32_t* d_draft_len,
                       const int32_t* d_forced, uint32_t K, uint32_t* d_counts, uint32_t max_tokens,
                       uint32_t* d_out_n, uint8_t* d_out_flags) {
  if (!p || (B && (!d_cfg || !d_draft || !d_draft_len || !d_out_n || !d_out_flags || K == 0))) return CG_E_ARG;
  if (d_counts && max_tokens == 0) return CG_E_ARG;
  if (B == 0) return CG_OK;
  cgk::DeviceGuard dg(cgk::ctx_device(p->ctx), "cg_pda_accept_many");
  if (!dg.ok) return CG_E_CUDA;
  const uint32_t grid = (B + cgk::kPdaAcceptThreads - 1) / cgk::kPdaAcceptThreads;
  return cgk::launch_dependent(cgk::pda_accept_many_kernel, dim3(grid), dim3(cgk::kPdaAcceptThreads),
                               pda_accept_smem(p->d), p->stream, p->d, p->t, d_cfg, B, d_draft, d_draft_len, d_forced,
                               K, d_counts, max_tokens, d_out_n, d_out_flags) == cudaSuccess
             ? CG_OK
             : CG_E_CUDA;
}

int cg_pda_step(cg_pda* p, uint32_t* d_cfg, uint32_t B, void* d_logits, int dtype, uint32_t V, float temp,
                float top_p, uint64_t seed, uint32_t step, const int32_t* d_forced, uint32_t* d_counts,
                uint32_t max_tokens, uint32_t* d_bitmask, uint32_t* d_out_tok, uint8_t* d_out_flags) {
  if (!p || (B && (!d_cfg || !d_logits || !d_out_tok || !d_out_flags))) return CG_E_ARG;
  if (dtype != CG_F32 && dtype != CG_BF16) return CG_E_ARG;
  if (V != p->t.V || !(temp >= 0.f) || temp == INFINITY || !(top_p == top_p)) return CG_E_ARG;
  if (d_counts && max_tokens == 0) return CG_E_ARG;
  if (B == 0) return CG_OK;
  cgk::DeviceGuard dg(cgk::ctx_device(p->ctx), "cg_pda_step");
  if (!dg.ok) return CG_E_CUDA;
  void* scratch = nullptr;
  int rc = cgk::ctx_sample_scratch(p->ctx, cgk::sample_scratch_bytes(B, V), &scratch);
  if (rc != CG_OK) return rc;
  if (cgk::step_fusable(dtype, V, p->t.W, temp, top_p, d_logits))
    return cgk::launch_pda_step(p->t, p->d, d_cfg, d_forced, B, d_logits, V, temp, top_p, seed, step, d_counts,
                                max_tokens, d_bitmask, d_out_tok, d_out_flags, scratch, p->stream) == cudaSuccess
               ? CG_OK
               : CG_E_CUDA;
  // otherwise the three calls, through a bitmask of this object when the caller gives none
  uint32_t* bm = d_bitmask;
  if (!bm) {
    const size_t need = size_t(B) * p->t.W * 4;
    if (need > p->step_bitmask_bytes) {
      if (cudaStreamSynchronize(p->stream) != cudaSuccess) return CG_E_CUDA;
      if (p->step_bitmask) cudaFree(p->step_bitmask);
      p->step_bitmask = nullptr;
      p->step_bitmask_bytes = 0;
      if (cudaMalloc(reinterpret_cast<void**>(&p->step_bitmask), need) != cudaSuccess) return CG_E_NOMEM;
      p->step_bitmask_bytes = need;
    }
    bm = p->step_bitmask;
  }
  if ((rc = cg_pda_fill_bitmask(p, d_cfg, B, d_forced, bm)) != CG_OK) return rc;
  if ((rc = cg_mask_and_sample(p->ctx, d_logits, dtype, B, V, bm, temp, top_p, seed, step, d_out_tok, nullptr, 0)) !=
      CG_OK)
    return rc;
  return cg_pda_accept(p, d_cfg, B, d_out_tok, d_forced, d_counts, max_tokens, d_out_flags);
}

int cg_pda_accept_fill(cg_pda* p, uint32_t* d_cfg, uint32_t B, const uint32_t* d_toks, const int32_t* d_forced,
                       uint32_t* d_counts, uint32_t max_tokens, uint8_t* d_out_flags, const int32_t* d_forced_next,
                       uint32_t* d_bitmask) {
  if (!p || (B && (!d_cfg || !d_toks || !d_out_flags || !d_bitmask))) return CG_E_ARG;
  if (B == 0) return CG_OK;
  cgk::DeviceGuard dg(cgk::ctx_device(p->ctx), "cg_pda_accept_fill");
  if (!dg.ok) return CG_E_CUDA;
  return cgk::launch_dependent(cgk::pda_accept_fill_kernel, dim3(B), dim3(cgk::kPdaFillThreads),
                               pda_fill_smem(p->d, p->t.W), p->stream, p->d, p->t, d_cfg, d_toks, d_forced, d_counts,
                               max_tokens, d_out_flags, d_forced_next, d_bitmask) == cudaSuccess
             ? CG_OK
             : CG_E_CUDA;
}

}  // extern "C"
