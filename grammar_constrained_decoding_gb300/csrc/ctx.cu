// Device context: uploads grammars and vocabulary, owns the mask cache and the
// device status word, and launches the three step kernels on its stream.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "cg_internal.h"
#include "device.cuh"

namespace cgk {
cudaError_t launch_fill_bitmask(const Tables& t, const uint32_t* states, const uint16_t* gid, const int32_t* forced,
                                uint32_t B, uint32_t* bitmask, bool cache_complete, cudaStream_t stream);
size_t fill_bitmask_smem(uint32_t W);
cudaError_t launch_prefill(const Tables& t, const uint32_t* class_rep, const uint16_t* class_gid, cudaStream_t stream);
cudaError_t launch_mask_and_sample(void* logits, int dtype, uint32_t B, uint32_t V, uint32_t W,
                                   const uint32_t* bitmask, float temp, float top_p, uint64_t seed, uint32_t step,
                                   uint32_t* out_tok, float* probs, int inplace, void* scratch, uint32_t* status,
                                   cudaStream_t stream);
size_t sample_scratch_bytes(uint32_t B, uint32_t V);
cudaError_t launch_accept(const Tables& t, const uint32_t* states, const uint16_t* gid, const uint32_t* toks,
                          const int32_t* forced, uint32_t B, uint32_t* counts, uint32_t max_tokens,
                          uint32_t* out_states, uint8_t* out_flags, cudaStream_t stream);
cudaError_t launch_accept_many(const Tables& t, const uint32_t* states, const uint16_t* gid, const uint32_t* draft,
                               const uint32_t* draft_len, const int32_t* forced, uint32_t B, uint32_t K,
                               uint32_t* counts, uint32_t max_tokens, uint32_t* out_states, uint32_t* out_n,
                               uint8_t* out_flags, uint32_t* path, cudaStream_t stream);
cudaError_t launch_wait_timeout_self_test(uint32_t* status, cudaStream_t stream);
cudaError_t launch_cache_fill(const Tables& t, const uint32_t* states, const uint16_t* gid, const int32_t* forced,
                              uint32_t B, unsigned long long* stats, cudaStream_t stream);
bool step_fusable(int dtype, uint32_t V, uint32_t W, float temp, float top_p, const void* logits);
cudaError_t launch_step(const Tables& t, const uint32_t* states, const uint16_t* gid, const int32_t* forced,
                        uint32_t B, void* logits, uint32_t V, float temp, float top_p, uint64_t seed, uint32_t step,
                        uint32_t* counts, uint32_t max_tokens, uint32_t* bitmask_out, uint32_t* out_tok,
                        uint32_t* out_states, uint8_t* out_flags, void* scratch, const DevGrammar* host_grammars,
                        bool cache_complete, cudaStream_t stream);
size_t seg_scratch_bytes(uint32_t B);
bool seg_usable(int dtype, uint32_t V, const void* logits, float* probs, int inplace, float temp, float top_p);
bool seg_bitmask_ok(uint32_t W, const void* bitmask);
cudaError_t launch_seg_sample(const void* logits, uint32_t B, uint32_t V, uint32_t W, const uint32_t* bitmask,
                              float temp, float top_p, uint64_t seed, uint32_t step, uint32_t* out_tok,
                              void* scratch, uint32_t* status, cudaStream_t stream);
cudaError_t launch_seg_step(const Tables& t, const uint32_t* states, const uint16_t* gid, const int32_t* forced,
                            uint32_t B, const void* logits, uint32_t V, float temp, float top_p, uint64_t seed,
                            uint32_t step, uint32_t* counts, uint32_t max_tokens, uint32_t* bitmask_out,
                            uint32_t* out_tok, uint32_t* out_states, uint8_t* out_flags, void* scratch,
                            const DevGrammar* host_grammars, cudaStream_t stream);
}  // namespace cgk

struct cg_ctx {
  cudaStream_t stream = nullptr;
  int device = 0;
  cgk::Tables t{};
  std::vector<void*> allocations;
  uint64_t cache_bytes = 0;
  const uint32_t* class_rep = nullptr;   // representative state of each mask class
  const uint16_t* class_gid = nullptr;   // grammar of each mask class
  void* sample_scratch = nullptr;        // candidate lists of the per-row sampling kernels
  size_t sample_scratch_bytes = 0;
  void* seg_scratch = nullptr;           // the segmented sampler's counters, row accumulators and histograms
  size_t seg_scratch_bytes = 0;          // (zero when allocated; every launch leaves it at zero)
  unsigned long long* cache_stats = nullptr;  // [0] class lookups, [1] classes computed, by the fused step's miss path
  uint32_t* step_bitmask = nullptr;      // bitmask of cg_step's unfused path when the caller gives none
  size_t step_bitmask_bytes = 0;
  std::vector<cgk::DevGrammar> grammars; // host copy of t.grammars
  // cg_step_host: the copy stream, two logit buffers and their events
  cudaStream_t copy_stream = nullptr;
  void* host_in[2] = {nullptr, nullptr};
  size_t host_in_bytes[2] = {0, 0};
  cudaEvent_t copied[2] = {nullptr, nullptr};   // logits of buffer k on the device
  cudaEvent_t consumed[2] = {nullptr, nullptr}; // the step that read buffer k has finished
  uint32_t next_in = 0;
  uint32_t* host_tok = nullptr;                 // ids when the caller gives no device buffer
  size_t host_tok_bytes = 0;
  bool cache_complete = false;           // cg_ctx_prefill has filled every class mask (in stream order)
};

namespace cgk {
CtxView ctx_view(const cg_ctx* c) { return {c->stream, c->t}; }
}  // namespace cgk

namespace {

template <typename T>
cudaError_t upload(cg_ctx* c, const std::vector<T>& host, T** dev) {
  *dev = nullptr;
  size_t bytes = std::max<size_t>(host.size() * sizeof(T), 16);
  cudaError_t e = cudaMalloc(reinterpret_cast<void**>(dev), bytes);
  if (e != cudaSuccess) return e;
  c->allocations.push_back(*dev);
  if (!host.empty()) e = cudaMemcpyAsync(*dev, host.data(), host.size() * sizeof(T), cudaMemcpyHostToDevice, c->stream);
  return e;
}

void release(cg_ctx* c) {
  for (void* p : c->allocations) cudaFree(p);
  c->allocations.clear();
  if (c->sample_scratch) cudaFree(c->sample_scratch);
  c->sample_scratch = nullptr;
  c->sample_scratch_bytes = 0;
  if (c->seg_scratch) cudaFree(c->seg_scratch);
  c->seg_scratch = nullptr;
  c->seg_scratch_bytes = 0;
  if (c->step_bitmask) cudaFree(c->step_bitmask);
  c->step_bitmask = nullptr;
  c->step_bitmask_bytes = 0;
  for (int k = 0; k < 2; ++k) {
    if (c->host_in[k]) cudaFree(c->host_in[k]);
    c->host_in[k] = nullptr;
    c->host_in_bytes[k] = 0;
    if (c->copied[k]) cudaEventDestroy(c->copied[k]);
    if (c->consumed[k]) cudaEventDestroy(c->consumed[k]);
    c->copied[k] = c->consumed[k] = nullptr;
  }
  if (c->host_tok) cudaFree(c->host_tok);
  c->host_tok = nullptr;
  c->host_tok_bytes = 0;
  if (c->copy_stream) cudaStreamDestroy(c->copy_stream);
  c->copy_stream = nullptr;
}

// Grows a context-owned device buffer to at least `need` bytes (synchronising
// the stream first: kernels still queued may use the old buffer).
int grow(cg_ctx* c, void** buf, size_t* have, size_t need) {
  if (need <= *have) return CG_OK;
  if (cudaStreamSynchronize(c->stream) != cudaSuccess) return CG_E_CUDA;
  if (*buf) cudaFree(*buf);
  *buf = nullptr;
  *have = 0;
  if (cudaMalloc(buf, need) != cudaSuccess) return CG_E_NOMEM;
  *have = need;
  return CG_OK;
}

// grow() for the segmented sampler's scratch, which must start at zero
int grow_zeroed(cg_ctx* c, void** buf, size_t* have, size_t need) {
  if (need <= *have) return CG_OK;
  const int rc = grow(c, buf, have, need);
  if (rc != CG_OK) return rc;
  return cudaMemsetAsync(*buf, 0, need, c->stream) == cudaSuccess ? CG_OK : CG_E_CUDA;
}

}  // namespace

namespace cgk {
int ctx_device(const cg_ctx* c) { return c->device; }
int ctx_sample_scratch(cg_ctx* c, size_t bytes, void** out) {
  const int rc = grow(c, &c->sample_scratch, &c->sample_scratch_bytes, bytes);
  *out = c->sample_scratch;
  return rc;
}
}  // namespace cgk

// Scratch of cg_mask_and_sample_noalloc, fixed in the module so that the
// call never allocates: the per-row sampler's candidate lists of up to
// CG_NOALLOC_MAX_ROWS rows (u32 ids, then u16 keys), then the segmented
// sampler's counters and row blocks for as many rows.  Its callers are the
// ones that must not touch the allocator while decoding: cudaMalloc/cudaFree
// synchronise the device and can fail once a server has planned all of its
// memory at start-up.  Shared by every call on a device (calls that may
// overlap race on it).
constexpr size_t kNoAllocScratchBytes = cgk::kNoAllocListBytes + cgk::kNoAllocSegBytes;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
// device address of g_noalloc_scratch on the current device, looked up once
// per device (the caller makes the context's device current first)
void* noalloc_scratch(cudaError_t* err) {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

bool sample_args_ok(const cg_ctx* c, void* d_logits, int dtype, uint32_t B, uint32_t V, const uint32_t* d_bitmask,
                    float temp, float top_p, uint32_t* d_out_tok, uint32_t flags) {
  if (!c || (B && (!d_logits || !d_bitmask || !d_out_tok))) return false;
  if (dtype != CG_F32 && dtype != CG_BF16) return false;
  if (V != c->t.V || !(temp >= 0.f) || temp == INFINITY || !(top_p == top_p)) return false;
  return (flags & ~CG_SAMPLE_INPLACE) == 0;
}

// cg_mask_and_sample on the given scratch: the segmented sampler (needs
// `seg` zero) or the per-row kernels (`lists`)
int sample_on(cg_ctx* c, void* d_logits, int dtype, uint32_t B, uint32_t V, const uint32_t* d_bitmask, float temp,
              float top_p, uint64_t seed, uint32_t step, uint32_t* d_out_tok, float* d_probs, int inplace,
              bool seg_path, void* lists, void* seg) {
  const cudaError_t e =
      seg_path ? cgk::launch_seg_sample(d_logits, B, V, c->t.W, d_bitmask, temp, top_p, seed, step, d_out_tok, seg,
                                        c->t.status, c->stream)
               : cgk::launch_mask_and_sample(d_logits, dtype, B, V, c->t.W, d_bitmask, temp, top_p, seed, step,
                                             d_out_tok, d_probs, inplace, lists, c->t.status, c->stream);
  return e == cudaSuccess ? CG_OK : CG_E_CUDA;
}
}  // namespace

extern "C" {

int cg_ctx_create(const cg_grammar* const* g, uint32_t n_g, const cg_vocab* v, void* cuda_stream, cg_ctx** out) {
  if (!g || n_g == 0 || n_g > 65535 || !v || !out) return CG_E_ARG;
  for (uint32_t i = 0; i < n_g; ++i) if (!g[i]) return CG_E_ARG;
  *out = nullptr;
  cg_ctx* c = new (std::nothrow) cg_ctx;
  if (!c) return CG_E_NOMEM;
  c->stream = static_cast<cudaStream_t>(cuda_stream);
  cudaGetDevice(&c->device);
  const uint32_t V = v->V, W = (V + 31) / 32, Wc = (W + 3) & ~3u;

  std::vector<cgk::DevGrammar> gdesc(n_g);
  std::vector<uint32_t> table;
  std::vector<uint16_t> colmap(size_t(n_g) * 512);
  std::vector<uint8_t> flags;
  std::vector<uint32_t> class_of, class_rep;
  std::vector<uint16_t> class_gid;
  uint32_t n_classes = 0;
  uint64_t table_off = 0;
  uint32_t state_off = 0;
  try {
    // mask classes over all grammars at once: states of different grammars
    // with equal masks share one class and one cached mask
    std::vector<const cg_grammar*> gs(g, g + n_g);
    std::vector<uint32_t> rep_gid;
    n_classes = cg::mask_classes_joint(gs, v->max_len, class_of, rep_gid, class_rep);
    class_gid.assign(rep_gid.begin(), rep_gid.end());
    for (uint32_t i = 0; i < n_g; ++i) {
      const cg_grammar& gr = *g[i];
      gdesc[i] = {table_off, gr.dfa.n_states, gr.n_cols, state_off, 0};
      table.insert(table.end(), gr.table.begin(), gr.table.end());
      std::copy(gr.col_of.begin(), gr.col_of.end(), colmap.begin() + size_t(i) * 512);
      flags.insert(flags.end(), gr.flags.begin(), gr.flags.end());
      table_off += gr.table.size();
      state_off += gr.dfa.n_states;
    }
  } catch (const std::bad_alloc&) {
    delete c;
    return CG_E_NOMEM;
  }
  // the table in 16 bits when every state number fits (the fused step's
  // accept reads a window of it from shared memory), padded by 16 bytes for
  // that window's aligned bulk copy; 32-byte token records (length, bytes)
  std::vector<uint16_t> table16;
  std::vector<uint32_t> tok_rec;
  try {
    bool fits = true;
    for (uint32_t i = 0; i < n_g; ++i) fits = fits && gdesc[i].n_states < cgk::kDead16;
    if (fits) {
      table16.resize(table.size() + 8);
      for (size_t i = 0; i < table.size(); ++i)
        table16[i] = table[i] == CG_DEAD ? cgk::kDead16 : uint16_t(table[i]);
    }
    tok_rec.assign(size_t(V) * 8, 0u);
    for (uint32_t k = 0; k < V; ++k) {
      const uint32_t b0 = v->off[k], n = v->off[k + 1] - b0;
      uint8_t* rec = reinterpret_cast<uint8_t*>(tok_rec.data() + size_t(k) * 8);
      if (n >= 32) {
        rec[0] = uint8_t(cgk::kLongToken);
        continue;
      }
      rec[0] = uint8_t(n);
      for (uint32_t i = 0; i < n; ++i) rec[1 + i] = v->bytes[b0 + i];
    }
  } catch (const std::bad_alloc&) {
    delete c;
    return CG_E_NOMEM;
  }
  cgk::Tables& t = c->t;
  cudaError_t e = cudaSuccess;
  uint16_t* d_table16 = nullptr;
  uint32_t* d_rec = nullptr;
  uint32_t* d_table;
  cgk::DevGrammar* d_gd;
  uint16_t* d_col;
  uint8_t* d_flags;
  uint32_t* d_class;
  uint32_t *d_off, *d_soff, *d_perm, *d_rep;
  uint16_t* d_cgid;
  uint8_t *d_bytes, *d_sbytes, *d_lcp;
  if ((e = upload(c, table, &d_table)) != cudaSuccess || (e = upload(c, gdesc, &d_gd)) != cudaSuccess ||
      (e = upload(c, colmap, &d_col)) != cudaSuccess || (e = upload(c, flags, &d_flags)) != cudaSuccess ||
      (e = upload(c, class_of, &d_class)) != cudaSuccess || (e = upload(c, v->off, &d_off)) != cudaSuccess ||
      (e = upload(c, v->bytes, &d_bytes)) != cudaSuccess || (e = upload(c, v->sorted_off, &d_soff)) != cudaSuccess ||
      (e = upload(c, v->sorted_bytes, &d_sbytes)) != cudaSuccess || (e = upload(c, v->perm, &d_perm)) != cudaSuccess ||
      (e = upload(c, v->lcp, &d_lcp)) != cudaSuccess || (e = upload(c, class_rep, &d_rep)) != cudaSuccess ||
      (e = upload(c, class_gid, &d_cgid)) != cudaSuccess || (e = upload(c, tok_rec, &d_rec)) != cudaSuccess ||
      (!table16.empty() && (e = upload(c, table16, &d_table16)) != cudaSuccess)) {
    release(c);
    delete c;
    return CG_E_CUDA;
  }
  uint32_t *d_cache = nullptr, *d_cstate = nullptr, *d_status = nullptr;
  c->cache_bytes = uint64_t(n_classes) * Wc * 4;
  if ((e = cudaMalloc(&d_cache, std::max<uint64_t>(c->cache_bytes, 16))) != cudaSuccess) { release(c); delete c; return CG_E_CUDA; }
  c->allocations.push_back(d_cache);
  // per class: state, then the miss pre-pass's claimed and finished splits
  const size_t cls_words = size_t(n_classes) + 4;
  if ((e = cudaMalloc(&d_cstate, cls_words * 3 * 4)) != cudaSuccess) { release(c); delete c; return CG_E_CUDA; }
  c->allocations.push_back(d_cstate);
  if ((e = cudaMalloc(&d_status, 16)) != cudaSuccess) { release(c); delete c; return CG_E_CUDA; }
  c->allocations.push_back(d_status);
  unsigned long long* d_stats = nullptr;
  if ((e = cudaMalloc(&d_stats, 16)) != cudaSuccess) { release(c); delete c; return CG_E_CUDA; }
  c->allocations.push_back(d_stats);
  c->cache_stats = d_stats;
  e = cudaMemsetAsync(d_cstate, 0, cls_words * 3 * 4, c->stream);
  // the miss pre-pass ORs its splits' bits into class rows: they start at zero
  if (e == cudaSuccess) e = cudaMemsetAsync(d_cache, 0, std::max<uint64_t>(c->cache_bytes, 16), c->stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(d_status, 0, 16, c->stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(d_stats, 0, 16, c->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);
  if (e == cudaSuccess && cgk::fill_bitmask_smem(W) > 48 * 1024) e = cudaErrorInvalidValue;
  if (e != cudaSuccess) { release(c); delete c; return e == cudaErrorInvalidValue ? CG_E_LIMIT : CG_E_CUDA; }
  t.table = d_table;
  t.grammars = d_gd;
  t.n_g = n_g;
  t.colmap = d_col;
  t.state_flags = d_flags;
  t.class_of = d_class;
  t.cache = d_cache;
  t.cache_state = d_cstate;
  t.cache_claim = d_cstate + cls_words;
  t.cache_done = d_cstate + 2 * cls_words;
  t.n_classes = n_classes;
  t.V = V;
  t.W = W;
  t.Wc = Wc;
  t.max_len = v->max_len;
  t.tok_off = d_off;
  t.tok_bytes = d_bytes;
  t.sorted_off = d_soff;
  t.sorted_bytes = d_sbytes;
  t.perm = d_perm;
  t.lcp = d_lcp;
  t.status = d_status;
  t.table16 = d_table16;
  t.tok_rec = reinterpret_cast<const uint4*>(d_rec);
  c->class_rep = d_rep;
  c->class_gid = d_cgid;
  c->grammars = std::move(gdesc);
  *out = c;
  return CG_OK;
}

void cg_ctx_destroy(cg_ctx* c) {
  if (!c) return;
  {
    cgk::DeviceGuard dg(c->device, "cg_ctx_destroy");
    cudaStreamSynchronize(c->stream);
    if (c->copy_stream) cudaStreamSynchronize(c->copy_stream);
    release(c);
  }
  delete c;
}

int cg_ctx_info(const cg_ctx* c, uint32_t* n_classes, uint64_t* cache_bytes, uint32_t* V, uint32_t* W) {
  if (!c) return CG_E_ARG;
  if (n_classes) *n_classes = c->t.n_classes;
  if (cache_bytes) *cache_bytes = c->cache_bytes;
  if (V) *V = c->t.V;
  if (W) *W = c->t.W;
  return CG_OK;
}

int cg_ctx_status(cg_ctx* c, uint32_t* dev_code) {
  if (!c) return CG_E_ARG;
  cgk::DeviceGuard dg(c->device, "cg_ctx_status");
  if (!dg.ok) return CG_E_CUDA;
  uint32_t code = 0;
  if (cudaStreamSynchronize(c->stream) != cudaSuccess) return CG_E_CUDA;
  if (cudaMemcpy(&code, c->t.status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return CG_E_CUDA;
  if (code && cudaMemset(c->t.status, 0, 4) != cudaSuccess) return CG_E_CUDA;
  // a kernel that gave up on a bounded wait may have left the segmented
  // sampler's scratch (which every complete launch leaves at zero) dirty
  if (code == CG_DEV_TIMEOUT && c->seg_scratch && cudaMemset(c->seg_scratch, 0, c->seg_scratch_bytes) != cudaSuccess)
    return CG_E_CUDA;
  if (dev_code) *dev_code = code;
  return code ? CG_E_DEVICE : CG_OK;
}

int cg_ctx_cache_stats(cg_ctx* c, uint64_t* lookups, uint64_t* computed, uint32_t* ready) {
  if (!c) return CG_E_ARG;
  cgk::DeviceGuard dg(c->device, "cg_ctx_cache_stats");
  if (!dg.ok) return CG_E_CUDA;
  unsigned long long v[2] = {0ull, 0ull};
  if (cudaStreamSynchronize(c->stream) != cudaSuccess) return CG_E_CUDA;
  if (cudaMemcpy(v, c->cache_stats, 16, cudaMemcpyDeviceToHost) != cudaSuccess) return CG_E_CUDA;
  if (lookups) *lookups = v[0];
  if (computed) *computed = v[1];
  if (ready) {
    std::vector<uint32_t> st(c->t.n_classes);
    if (!st.empty() &&
        cudaMemcpy(st.data(), c->t.cache_state, st.size() * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
      return CG_E_CUDA;
    *ready = uint32_t(std::count(st.begin(), st.end(), 2u));  // kStateReady
  }
  return CG_OK;
}

int cg_ctx_prefill(cg_ctx* c) {
  if (!c) return CG_E_ARG;
  cgk::DeviceGuard dg(c->device, "cg_ctx_prefill");
  if (!dg.ok) return CG_E_CUDA;
  if (cgk::launch_prefill(c->t, c->class_rep, c->class_gid, c->stream) != cudaSuccess) return CG_E_CUDA;
  c->cache_complete = true;  // later kernels on the stream see every class ready
  return CG_OK;
}

int cg_fill_bitmask(cg_ctx* c, const uint32_t* d_states, const uint16_t* d_gid, const int32_t* d_forced, uint32_t B,
                    uint32_t* d_bitmask) {
  if (!c || (B && (!d_states || !d_bitmask))) return CG_E_ARG;
  cgk::DeviceGuard dg(c->device, "cg_fill_bitmask");
  if (!dg.ok) return CG_E_CUDA;
  // without prefill, the classes the rows miss first (each split over many blocks)
  if (!c->cache_complete &&
      cgk::launch_cache_fill(c->t, d_states, d_gid, d_forced, B, c->cache_stats, c->stream) != cudaSuccess)
    return CG_E_CUDA;
  return cgk::launch_fill_bitmask(c->t, d_states, d_gid, d_forced, B, d_bitmask, c->cache_complete, c->stream) ==
                 cudaSuccess
             ? CG_OK
             : CG_E_CUDA;
}

int cg_mask_and_sample(cg_ctx* c, void* d_logits, int dtype, uint32_t B, uint32_t V, const uint32_t* d_bitmask,
                       float temp, float top_p, uint64_t seed, uint32_t step, uint32_t* d_out_tok, float* d_probs,
                       uint32_t flags) {
  if (!sample_args_ok(c, d_logits, dtype, B, V, d_bitmask, temp, top_p, d_out_tok, flags)) return CG_E_ARG;
  if (B == 0) return CG_OK;
  cgk::DeviceGuard dg(c->device, "cg_mask_and_sample");
  if (!dg.ok) return CG_E_CUDA;
  const int inplace = (flags & CG_SAMPLE_INPLACE) ? 1 : 0;
  const bool seg_path =
      cgk::seg_usable(dtype, V, d_logits, d_probs, inplace, temp, top_p) && cgk::seg_bitmask_ok(c->t.W, d_bitmask);
  // grown once per larger batch (outside any stream capture)
  const int rc = seg_path ? grow_zeroed(c, &c->seg_scratch, &c->seg_scratch_bytes, cgk::seg_scratch_bytes(B))
                          : grow(c, &c->sample_scratch, &c->sample_scratch_bytes, cgk::sample_scratch_bytes(B, V));
  if (rc != CG_OK) return rc;
  return sample_on(c, d_logits, dtype, B, V, d_bitmask, temp, top_p, seed, step, d_out_tok, d_probs, inplace,
                   seg_path, c->sample_scratch, c->seg_scratch);
}

int cg_mask_and_sample_noalloc(cg_ctx* c, void* d_logits, int dtype, uint32_t B, uint32_t V,
                               const uint32_t* d_bitmask, float temp, float top_p, uint64_t seed, uint32_t step,
                               uint32_t* d_out_tok, float* d_probs, uint32_t flags) {
  if (!sample_args_ok(c, d_logits, dtype, B, V, d_bitmask, temp, top_p, d_out_tok, flags)) return CG_E_ARG;
  if (B > CG_NOALLOC_MAX_ROWS || cgk::sample_scratch_bytes(B, V) > cgk::kNoAllocListBytes ||
      cgk::seg_scratch_bytes(B) > cgk::kNoAllocSegBytes)
    return CG_E_LIMIT;
  if (B == 0) return CG_OK;
  cgk::DeviceGuard dg(c->device, "cg_mask_and_sample_noalloc");
  if (!dg.ok) return CG_E_CUDA;
  cudaError_t e = cudaSuccess;
  unsigned char* scratch = static_cast<unsigned char*>(noalloc_scratch(&e));
  if (!scratch) return CG_E_CUDA;
  const int inplace = (flags & CG_SAMPLE_INPLACE) ? 1 : 0;
  const bool seg_path =
      cgk::seg_usable(dtype, V, d_logits, d_probs, inplace, temp, top_p) && cgk::seg_bitmask_ok(c->t.W, d_bitmask);
  unsigned char* seg = scratch + cgk::kNoAllocListBytes;
  // the segmented sampler's part starts at zero: cleared here, whatever an
  // earlier call (or one that ran out of a bounded wait) left in it
  if (seg_path && cudaMemsetAsync(seg, 0, cgk::seg_scratch_bytes(B), c->stream) != cudaSuccess) return CG_E_CUDA;
  return sample_on(c, d_logits, dtype, B, V, d_bitmask, temp, top_p, seed, step, d_out_tok, d_probs, inplace,
                   seg_path, scratch, seg);
}

int cg_accept(cg_ctx* c, const uint32_t* d_states, const uint16_t* d_gid, const uint32_t* d_toks,
              const int32_t* d_forced, uint32_t B, uint32_t* d_counts, uint32_t max_tokens, uint32_t* d_out_states,
              uint8_t* d_out_flags) {
  if (!c || (B && (!d_states || !d_toks || !d_out_states || !d_out_flags))) return CG_E_ARG;
  if (d_counts && max_tokens == 0) return CG_E_ARG;
  cgk::DeviceGuard dg(c->device, "cg_accept");
  if (!dg.ok) return CG_E_CUDA;
  return cgk::launch_accept(c->t, d_states, d_gid, d_toks, d_forced, B, d_counts, max_tokens, d_out_states,
                            d_out_flags, c->stream) == cudaSuccess
             ? CG_OK
             : CG_E_CUDA;
}

int cg_step(cg_ctx* c, const uint32_t* d_states, const uint16_t* d_gid, const int32_t* d_forced, uint32_t B,
            void* d_logits, int dtype, uint32_t V, float temp, float top_p, uint64_t seed, uint32_t step,
            uint32_t* d_counts, uint32_t max_tokens, uint32_t* d_bitmask, uint32_t* d_out_tok,
            uint32_t* d_out_states, uint8_t* d_out_flags) {
  if (!c || (B && (!d_states || !d_logits || !d_out_tok || !d_out_states || !d_out_flags))) return CG_E_ARG;
  if (dtype != CG_F32 && dtype != CG_BF16) return CG_E_ARG;
  if (V != c->t.V || !(temp >= 0.f) || temp == INFINITY || !(top_p == top_p)) return CG_E_ARG;
  if (d_counts && max_tokens == 0) return CG_E_ARG;
  if (B == 0) return CG_OK;
  cgk::DeviceGuard dg(c->device, "cg_step");
  if (!dg.ok) return CG_E_CUDA;
  int rc;
  if (cgk::step_fusable(dtype, V, c->t.W, temp, top_p, d_logits)) {
    // top-p: one per-row kernel (mask, sample and accept in one launch), after
    // the classes the rows miss when the cache is not complete
    if ((rc = grow(c, &c->sample_scratch, &c->sample_scratch_bytes, cgk::sample_scratch_bytes(B, V))) != CG_OK)
      return rc;
    if (!c->cache_complete &&
        cgk::launch_cache_fill(c->t, d_states, d_gid, d_forced, B, c->cache_stats, c->stream) != cudaSuccess)
      return CG_E_CUDA;
    return cgk::launch_step(c->t, d_states, d_gid, d_forced, B, d_logits, V, temp, top_p, seed, step, d_counts,
                            max_tokens, d_bitmask, d_out_tok, d_out_states, d_out_flags, c->sample_scratch,
                            c->grammars.data(), c->cache_complete, c->stream) == cudaSuccess
               ? CG_OK
               : CG_E_CUDA;
  }
  if (cgk::seg_usable(dtype, V, d_logits, nullptr, 0, temp, top_p)) {
    // greedy / every allowed token: one segmented kernel (after the class
    // masks the rows miss, when the cache is not complete)
    if ((rc = grow_zeroed(c, &c->seg_scratch, &c->seg_scratch_bytes, cgk::seg_scratch_bytes(B))) != CG_OK) return rc;
    if (!c->cache_complete &&
        cgk::launch_cache_fill(c->t, d_states, d_gid, d_forced, B, c->cache_stats, c->stream) != cudaSuccess)
      return CG_E_CUDA;
    return cgk::launch_seg_step(c->t, d_states, d_gid, d_forced, B, d_logits, V, temp, top_p, seed, step, d_counts,
                                max_tokens, d_bitmask, d_out_tok, d_out_states, d_out_flags, c->seg_scratch,
                                c->grammars.data(), c->stream) == cudaSuccess
               ? CG_OK
               : CG_E_CUDA;
  }
  // otherwise the three calls, through a context bitmask when the caller gives none
  uint32_t* bm = d_bitmask;
  if (!bm) {
    rc = grow(c, reinterpret_cast<void**>(&c->step_bitmask), &c->step_bitmask_bytes, size_t(B) * c->t.W * 4);
    if (rc != CG_OK) return rc;
    bm = c->step_bitmask;
  }
  if ((rc = cg_fill_bitmask(c, d_states, d_gid, d_forced, B, bm)) != CG_OK) return rc;
  if ((rc = cg_mask_and_sample(c, d_logits, dtype, B, V, bm, temp, top_p, seed, step, d_out_tok, nullptr, 0)) !=
      CG_OK)
    return rc;
  return cg_accept(c, d_states, d_gid, d_out_tok, d_forced, B, d_counts, max_tokens, d_out_states, d_out_flags);
}

}  // extern "C"

int cg_ctx_sync(cg_ctx* c) {
  if (!c) return CG_E_ARG;
  cgk::DeviceGuard dg(c->device, "cg_ctx_sync");
  if (!dg.ok) return CG_E_CUDA;
  return cudaStreamSynchronize(c->stream) == cudaSuccess ? CG_OK : CG_E_CUDA;
}

int cg_step_host(cg_ctx* c, const uint32_t* d_states, const uint16_t* d_gid, const int32_t* d_forced, uint32_t B,
                 const void* h_logits, int dtype, uint32_t V, float temp, float top_p, uint64_t seed, uint32_t step,
                 uint32_t* d_counts, uint32_t max_tokens, uint32_t* h_out_tok, uint32_t* d_out_tok,
                 uint32_t* d_out_states, uint8_t* d_out_flags) {
  if (!c || (B && (!d_states || !h_logits || !h_out_tok || !d_out_states || !d_out_flags))) return CG_E_ARG;
  if (dtype != CG_F32 && dtype != CG_BF16) return CG_E_ARG;
  if (V != c->t.V || !(temp >= 0.f) || temp == INFINITY || !(top_p == top_p)) return CG_E_ARG;
  if (d_counts && max_tokens == 0) return CG_E_ARG;
  if (B == 0) return CG_OK;
  cgk::DeviceGuard dg(c->device, "cg_step_host");
  if (!dg.ok) return CG_E_CUDA;
  if (!c->copy_stream) {
    if (cudaStreamCreateWithFlags(&c->copy_stream, cudaStreamNonBlocking) != cudaSuccess) return CG_E_CUDA;
    for (int k = 0; k < 2; ++k)
      if (cudaEventCreateWithFlags(&c->copied[k], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&c->consumed[k], cudaEventDisableTiming) != cudaSuccess)
        return CG_E_CUDA;
  }
  const size_t bytes = size_t(B) * V * (dtype == CG_BF16 ? 2 : 4);
  const uint32_t k = c->next_in;
  if (bytes > c->host_in_bytes[k] && cudaStreamSynchronize(c->copy_stream) != cudaSuccess) return CG_E_CUDA;
  int rc = grow(c, &c->host_in[k], &c->host_in_bytes[k], bytes);
  if (rc != CG_OK) return rc;
  uint32_t* tok = d_out_tok;
  if (!tok) {
    rc = grow(c, reinterpret_cast<void**>(&c->host_tok), &c->host_tok_bytes, size_t(B) * 4);
    if (rc != CG_OK) return rc;
    tok = c->host_tok;
  }
  // buffer k is free once the step that last read it has finished (an event
  // never recorded is complete)
  if (cudaStreamWaitEvent(c->copy_stream, c->consumed[k], 0) != cudaSuccess ||
      cudaMemcpyAsync(c->host_in[k], h_logits, bytes, cudaMemcpyHostToDevice, c->copy_stream) != cudaSuccess ||
      cudaEventRecord(c->copied[k], c->copy_stream) != cudaSuccess ||
      cudaStreamWaitEvent(c->stream, c->copied[k], 0) != cudaSuccess)
    return CG_E_CUDA;
  c->next_in = k ^ 1u;
  rc = cg_step(c, d_states, d_gid, d_forced, B, c->host_in[k], dtype, V, temp, top_p, seed, step, d_counts,
               max_tokens, nullptr, tok, d_out_states, d_out_flags);
  if (rc != CG_OK) return rc;
  if (cudaEventRecord(c->consumed[k], c->stream) != cudaSuccess ||
      cudaMemcpyAsync(h_out_tok, tok, size_t(B) * 4, cudaMemcpyDeviceToHost, c->stream) != cudaSuccess)
    return CG_E_CUDA;
  return CG_OK;
}

int cg_accept_many(cg_ctx* c, const uint32_t* d_states, const uint16_t* d_gid, const uint32_t* d_draft,
                   const uint32_t* d_draft_len, const int32_t* d_forced, uint32_t B, uint32_t K, uint32_t* d_counts,
                   uint32_t max_tokens, uint32_t* d_out_states, uint32_t* d_out_n, uint8_t* d_out_flags,
                   uint32_t* d_out_path) {
  if (!c || (B && (!d_states || !d_draft || !d_draft_len || !d_out_states || !d_out_n || !d_out_flags))) return CG_E_ARG;
  if (B && K == 0) return CG_E_ARG;
  if (d_counts && max_tokens == 0) return CG_E_ARG;
  cgk::DeviceGuard dg(c->device, "cg_accept_many");
  if (!dg.ok) return CG_E_CUDA;
  return cgk::launch_accept_many(c->t, d_states, d_gid, d_draft, d_draft_len, d_forced, B, K, d_counts, max_tokens,
                                 d_out_states, d_out_n, d_out_flags, d_out_path, c->stream) == cudaSuccess
             ? CG_OK
             : CG_E_CUDA;
}

int cg_self_test_wait_timeout(cg_ctx* c) {
  if (!c) return CG_E_ARG;
  cgk::DeviceGuard dg(c->device, "cg_self_test_wait_timeout");
  if (!dg.ok) return CG_E_CUDA;
  return cgk::launch_wait_timeout_self_test(c->t.status, c->stream) == cudaSuccess ? CG_OK : CG_E_CUDA;
}
