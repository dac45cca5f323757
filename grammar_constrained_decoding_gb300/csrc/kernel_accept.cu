// Accept: advance each row's automaton by its token, one thread per row
// (accept_row in row_ops.cuh holds the rules).
#include "row_ops.cuh"

namespace cgk {

constexpr int kAcceptThreads = 128;

cudaError_t allow_smem(const void* kernel, size_t bytes);  // kernel_sample.cu

__global__ void __launch_bounds__(kAcceptThreads) accept_kernel(Tables t, const uint32_t* __restrict__ states,
                                                                const uint16_t* __restrict__ gid,
                                                                const uint32_t* __restrict__ toks,
                                                                const int32_t* __restrict__ forced, uint32_t B,
                                                                uint32_t* counts, uint32_t max_tokens,
                                                                uint32_t* out_states, uint8_t* out_flags) {
  // the column map in shared memory when every row uses one grammar (the
  // tables are static: copied before the wait for the sampled tokens)
  __shared__ uint16_t scol[512];
  griddep_launch_dependents();
  const bool staged = gid == nullptr || t.n_g == 1;
  if (staged)
    for (uint32_t i = threadIdx.x; i < 512; i += blockDim.x) scol[i] = t.colmap[i];
  __syncthreads();
  griddep_wait();  // the tokens come from the sampling kernel
  const uint32_t b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  accept_row(t, b, gid ? gid[b] : 0u, states[b], toks[b], forced ? forced[b] : -1, counts, max_tokens, out_states,
             out_flags, staged ? scol : nullptr);
}

cudaError_t launch_accept(const Tables& t, const uint32_t* states, const uint16_t* gid, const uint32_t* toks,
                          const int32_t* forced, uint32_t B, uint32_t* counts, uint32_t max_tokens,
                          uint32_t* out_states, uint8_t* out_flags, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  return launch_dependent(accept_kernel, dim3((B + kAcceptThreads - 1) / kAcceptThreads), dim3(kAcceptThreads), 0,
                          stream, t, states, gid, toks, forced, B, counts, max_tokens, out_states, out_flags);
}

// Speculative verification: one warp per row (accept_many_row in row_ops.cuh
// holds the rules).  Before the serial walk, the warp's lanes copy the draft's
// token records into shared memory (one load each, all in flight), and lane 0
// bulk-copies the 16-bit table rows of up to kManyWinRows states around the
// row's state, with their flags, so that most transitions of the walk are read
// on chip.
constexpr uint32_t kManyRows = 4;                   // rows (warps) per block
constexpr uint32_t kManyRecs = 64;                  // draft positions whose records are staged
constexpr uint32_t kManyWinRows = 1024;             // states in a row's table window
constexpr uint32_t kManyWinBytes = 40 * 1024;       // shared memory for that window
constexpr uint32_t kManyRowBytes = kManyRecs * 32 + kManyWinRows + kManyWinBytes;

__global__ void __launch_bounds__(kManyRows * 32)
    accept_many_kernel(Tables t, const uint32_t* __restrict__ states, const uint16_t* __restrict__ gid,
                       const uint32_t* __restrict__ draft, const uint32_t* __restrict__ draft_len,
                       const int32_t* __restrict__ forced, uint32_t B, uint32_t K, uint32_t* counts,
                       uint32_t max_tokens, uint32_t* out_states, uint32_t* out_n, uint8_t* out_flags,
                       uint32_t* path) {
  extern __shared__ __align__(16) unsigned char dsm[];
  __shared__ __align__(8) uint64_t mbar[kManyRows];
  const uint32_t lane = threadIdx.x & 31, w = threadIdx.x >> 5, b = blockIdx.x * kManyRows + w;
  uint4* recs = reinterpret_cast<uint4*>(dsm + size_t(w) * kManyRowBytes);       // [kManyRecs][2]
  uint8_t* wflags = dsm + size_t(w) * kManyRowBytes + kManyRecs * 32;             // [kManyWinRows]
  uint16_t* win = reinterpret_cast<uint16_t*>(wflags + kManyWinRows);             // [kManyWinBytes / 2]
  griddep_launch_dependents();
  if (lane == 0) {
    mbar_init(&mbar[w], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  griddep_wait();  // the drafts and states come from earlier work on the stream
  if (b >= B) return;
  const uint32_t s = states[b], g = gid ? gid[b] : 0u;
  const uint32_t n = min(draft_len[b], K);
  const uint32_t* row_draft = draft + size_t(b) * K;
  const uint32_t n_recs = t.tok_rec ? min(n, kManyRecs) : 0u;
  for (uint32_t j = lane; j < n_recs; j += 32) {
    const uint32_t tok = row_draft[j];
    if (tok < t.V) {
      recs[2 * j] = t.tok_rec[size_t(tok) * 2];
      recs[2 * j + 1] = t.tok_rec[size_t(tok) * 2 + 1];
    }
  }
  WindowCopy wc;
  DevGrammar gd{};
  if (g < t.n_g && s != CG_DEAD) {
    gd = t.grammars[g];
    wc = window_copy(t, gd, s, kManyWinBytes, kManyWinRows);
  }
  if (lane == 0 && wc.rows) {
    mbar_expect_tx(&mbar[w], wc.bytes);
    bulk_g2s(win, wc.src, wc.bytes, &mbar[w]);
  }
  for (uint32_t i = lane; i < wc.rows; i += 32) wflags[i] = t.state_flags[gd.state_off + wc.lo + i];
  __syncwarp();
  if (lane != 0) return;
  StateWindow sw;
  if (wc.rows) {
    if (mbar_wait(&mbar[w], 0)) {
      sw.next = win + wc.delta;
      sw.flags = wflags;
      sw.lo = wc.lo;
      sw.rows = wc.rows;
    } else {
      record_error(t.status, CG_DEV_TIMEOUT);
      mbar_wait(&mbar[w], 0);  // let the copy land before the block exits (bounded again)
    }
  }
  accept_many_row(t, b, g, s, row_draft, draft_len[b], forced ? forced + size_t(b) * K : nullptr, K, counts,
                  max_tokens, out_states, out_n, out_flags, path ? path + size_t(b) * (K + 1) : nullptr, recs,
                  n_recs, sw);
}

cudaError_t launch_accept_many(const Tables& t, const uint32_t* states, const uint16_t* gid, const uint32_t* draft,
                               const uint32_t* draft_len, const int32_t* forced, uint32_t B, uint32_t K,
                               uint32_t* counts, uint32_t max_tokens, uint32_t* out_states, uint32_t* out_n,
                               uint8_t* out_flags, uint32_t* path, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  const size_t smem = size_t(kManyRows) * kManyRowBytes;
  cudaError_t e = allow_smem(reinterpret_cast<const void*>(accept_many_kernel), smem);
  if (e != cudaSuccess) return e;
  return launch_dependent(accept_many_kernel, dim3((B + kManyRows - 1) / kManyRows), dim3(kManyRows * 32), smem,
                          stream, t, states, gid, draft, draft_len, forced, B, K, counts, max_tokens, out_states,
                          out_n, out_flags, path);
}

// Self-test of the bounded waits every kernel here uses: one block arms a
// barrier for bytes no copy will deliver, waits with mbar_wait (the same
// polling limit as the sampling and accept kernels), and records
// CG_DEV_TIMEOUT when the limit runs out.  Nothing is in flight, so the block
// simply returns: the context stays usable.
__global__ void wait_timeout_self_test_kernel(uint32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  mbar_expect_tx(&bar, 16);  // arrives, but the 16 bytes never come: the phase stays open
  if (!mbar_wait(&bar, 0)) record_error(status, CG_DEV_TIMEOUT);
}

cudaError_t launch_wait_timeout_self_test(uint32_t* status, cudaStream_t stream) {
  wait_timeout_self_test_kernel<<<1, 32, 0, stream>>>(status);
  return cudaGetLastError();
}

}  // namespace cgk
