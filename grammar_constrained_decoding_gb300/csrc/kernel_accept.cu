// Accept: advance each row's automaton by its token, one thread per row
// (accept_row in row_ops.cuh holds the rules).
#include "row_ops.cuh"

namespace cgk {

constexpr int kAcceptThreads = 128;

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
  accept_row(t, b, gid ? gid[b] : 0u, states[b], toks[b], forced ? forced[b] : -1, counts, max_tokens, out_states,
             out_flags);
}

cudaError_t launch_accept(const Tables& t, const uint32_t* states, const uint16_t* gid, const uint32_t* toks,
                          const int32_t* forced, uint32_t B, uint32_t* counts, uint32_t max_tokens,
                          uint32_t* out_states, uint8_t* out_flags, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  return launch_dependent(accept_kernel, dim3((B + kAcceptThreads - 1) / kAcceptThreads), dim3(kAcceptThreads), 0,
                          stream, t, states, gid, toks, forced, B, counts, max_tokens, out_states, out_flags);
}

// Speculative verification: one thread per row walks its draft (accept_many_row
// in row_ops.cuh holds the rules).
__global__ void __launch_bounds__(kAcceptThreads)
    accept_many_kernel(Tables t, const uint32_t* __restrict__ states, const uint16_t* __restrict__ gid,
                       const uint32_t* __restrict__ draft, const uint32_t* __restrict__ draft_len,
                       const int32_t* __restrict__ forced, uint32_t B, uint32_t K, uint32_t* counts,
                       uint32_t max_tokens, uint32_t* out_states, uint32_t* out_n, uint8_t* out_flags,
                       uint32_t* path) {
  griddep_launch_dependents();
  griddep_wait();  // the drafts and states come from earlier work on the stream
  const uint32_t b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  accept_many_row(t, b, gid ? gid[b] : 0u, states[b], draft + size_t(b) * K, draft_len[b],
                  forced ? forced + size_t(b) * K : nullptr, K, counts, max_tokens, out_states, out_n, out_flags,
                  path ? path + size_t(b) * (K + 1) : nullptr);
}

cudaError_t launch_accept_many(const Tables& t, const uint32_t* states, const uint16_t* gid, const uint32_t* draft,
                               const uint32_t* draft_len, const int32_t* forced, uint32_t B, uint32_t K,
                               uint32_t* counts, uint32_t max_tokens, uint32_t* out_states, uint32_t* out_n,
                               uint8_t* out_flags, uint32_t* path, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  return launch_dependent(accept_many_kernel, dim3((B + kAcceptThreads - 1) / kAcceptThreads), dim3(kAcceptThreads),
                          0, stream, t, states, gid, draft, draft_len, forced, B, K, counts, max_tokens, out_states,
                          out_n, out_flags, path);
}

}  // namespace cgk
