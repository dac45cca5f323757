// Device-side views and helpers shared by the step kernels.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "../../include/cg.h"

namespace cgk {

// Programmatic dependent launch: the step's kernels (fill_bitmask ->
// mask_and_sample -> accept -> next fill_bitmask) are launched so that each
// may start while its predecessor finishes.  A kernel lets its dependents be
// scheduled as soon as it starts (launch_dependents) and waits for its
// predecessor's completion and memory (griddep_wait) before it reads anything
// the predecessor wrote.  Both are no-ops for a normally launched kernel.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct DevGrammar {
  uint64_t table_off;   // first element of this grammar's [n_states x n_cols] table
  uint32_t n_states;
  uint32_t n_cols;
  uint32_t state_off;   // first element of this grammar's per-state arrays
  uint32_t pad;
};

// Everything the step kernels read, by value (a few pointers and sizes).
struct Tables {
  const uint32_t* table;       // next state per (state, column), CG_DEAD for none
  const DevGrammar* grammars;
  uint32_t n_g;
  const uint16_t* colmap;      // [n_g][512] symbol -> column
  const uint8_t* state_flags;  // CG_STATE_* per state (all grammars)
  const uint32_t* class_of;    // mask class per state (all grammars, global ids)
  uint32_t* cache;             // [n_classes][Wc] allowed-token bitmask per class (words W..Wc unused)
  uint32_t* cache_state;       // per class: 0 empty, 1 being filled, 2 ready
  uint32_t* cache_claim;       // per class: the miss pre-pass's splits claimed (bit per split)
  uint32_t* cache_done;        // per class: the miss pre-pass's splits finished
  uint32_t n_classes;
  uint32_t V, W, max_len;
  uint32_t Wc;                 // row stride of the mask cache: W rounded up to 4 words (16-byte aligned rows)
  const uint32_t* tok_off;     // [V+1] token bytes in id order
  const uint8_t* tok_bytes;
  const uint32_t* sorted_off;  // [V+1] token bytes in trie (lexicographic) order
  const uint8_t* sorted_bytes;
  const uint32_t* perm;        // trie position -> token id
  const uint8_t* lcp;          // common prefix with the previous trie position
  uint32_t* status;            // first CG_DEV_* error
  const uint16_t* table16;     // `table` in 16 bits (kDead16 for CG_DEAD); null when a grammar has too many states
  const uint4* tok_rec;        // [V][2] 32-byte token records: byte 0 the length, bytes 1..31 the token's bytes;
                               // length kLongToken: 32 bytes or more, read through tok_off
};

// A context's stream and device tables, for the pushdown rows (pda.cu) that
// run on a context without being part of it (ctx.cu).
struct CtxView {
  cudaStream_t stream;
  Tables t;
};
CtxView ctx_view(const cg_ctx* c);
// The context's candidate-list scratch of the sampling kernels, grown to at
// least `bytes` (CG_OK or a CG_E_* code).
int ctx_sample_scratch(cg_ctx* c, size_t bytes, void** out);
// The device a context was created on.
int ctx_device(const cg_ctx* c);

// The fixed scratch of cg_mask_and_sample_noalloc (ctx.cu): the per-row
// sampler's candidate lists (kSampleListEntries u32 ids and u16 keys a row),
// then the segmented sampler's counters and row blocks, for
// CG_NOALLOC_MAX_ROWS rows.  Each sampler static_asserts that its layout for
// that many rows fits.
constexpr uint32_t kSampleListEntries = 8192;
constexpr size_t kNoAllocListBytes = size_t(CG_NOALLOC_MAX_ROWS) * kSampleListEntries * 6;
constexpr size_t kNoAllocSegBytes = size_t(64) << 10;

// Makes a device current for the duration of a call and puts the caller's
// back: every launch, allocation and symbol lookup of a library call then
// happens on the device its context's tables live on.  The call is also an
// NVTX range named after the entry point (free unless a profiler is
// attached), so that a timeline attributes host time to library calls.
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev, const char* call) {
    nvtxRangePushA(call);
    int cur = 0;
    if (cudaGetDevice(&cur) != cudaSuccess) {
      ok = false;
      return;
    }
    if (cur != dev) {
      if (cudaSetDevice(dev) != cudaSuccess) {
        ok = false;
        return;
      }
      prev = cur;
    }
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
    nvtxRangePop();
  }
  DeviceGuard(const DeviceGuard&) = delete;
  DeviceGuard& operator=(const DeviceGuard&) = delete;
};

constexpr uint16_t kDead16 = 0xFFFFu;      // CG_DEAD in table16
constexpr uint32_t kLongToken = 0xFFu;     // token record length of a token read through tok_off

// ---- mbarrier waits and bulk (TMA) copies into shared memory ----------------------

constexpr uint32_t kWaitLimit = 1u << 18;  // polls of a bounded mbarrier wait (about a second: a poll
                                           // suspends for a few microseconds when the phase is open)

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// A bulk copy wants both addresses 16-byte aligned and a size that is a
// multiple of 16: one that breaks the rule is not issued (the waiter's bounded
// wait then runs out and records CG_DEV_TIMEOUT) instead of faulting the GPU.
__device__ __forceinline__ bool bulk_ok(const void* dst, const void* src, uint32_t bytes) {
  return ((smem_addr(dst) | static_cast<uint32_t>(reinterpret_cast<uintptr_t>(src)) | bytes) & 15u) == 0;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  if (!bulk_ok(dst, src, bytes)) return;
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
// L2 policy for data read once per step (the logits): evicted first, so the
// stream does not push the mask cache and the tables out of L2
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// bulk_g2s with an L2 cache hint (a policy from evict_first_policy)
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t pol) {
  if (!bulk_ok(dst, src, bytes)) return;
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// bounded wait on a phase; false when the limit ran out (the caller records
// CG_DEV_TIMEOUT and drains its copies)
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

__device__ __forceinline__ void record_error(uint32_t* status, uint32_t code) {
  atomicCAS(status, 0u, code);
}

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of
// (c0,c1,c2,c3) -> (hi(M1 c2)^c1^k0, lo(M1 c2), hi(M0 c0)^c3^k1, lo(M0 c0))
// with the key bumped by the Weyl constants between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

__device__ __forceinline__ uint32_t philox_word(uint4 blk, uint32_t lane) {
  return lane == 0 ? blk.x : lane == 1 ? blk.y : lane == 2 ? blk.z : blk.w;
}

// u = (2 * (r >> 9) + 1) * 2^-24 (exact in binary32); g = -log(-log u)
__device__ __forceinline__ float gumbel_from_word(uint32_t r) {
  const float u = float(2u * (r >> 9) + 1u) * 5.9604644775390625e-08f;
  return -logf(-logf(u));
}

// Monotone 32-bit key of a float (larger float <=> larger key); -0 and +0,
// which compare equal, share the key of +0.
__device__ __forceinline__ uint32_t fkey(float x) {
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float fkey_inv(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// (value, id) packed so that the unsigned maximum picks the larger value and,
// among equal values, the lower id.
__device__ __forceinline__ unsigned long long pack_best(float v, uint32_t id) {
  return (static_cast<unsigned long long>(fkey(v)) << 32) | static_cast<unsigned long long>(~id);
}
__device__ __forceinline__ uint32_t best_id(unsigned long long p) { return ~static_cast<uint32_t>(p); }

struct MaxOp {
  template <typename T> __device__ __forceinline__ T operator()(T a, T b) const { return a > b ? a : b; }
};
struct SumOp {
  template <typename T> __device__ __forceinline__ T operator()(T a, T b) const { return a + b; }
};

// ---- block reductions (blockDim.x a multiple of 32, <= 1024) ----------------
template <typename T, typename Op>
__device__ __forceinline__ T warp_reduce(T v, Op op) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// Result is returned to every thread.  `scratch` holds >= 33 elements of T;
// `identity` is the neutral element of op.
template <typename T, typename Op>
__device__ T block_reduce(T v, Op op, T identity, T* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_reduce(v, op);
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  if (warp == 0) {
    T w = lane < nw ? scratch[lane] : identity;
    w = warp_reduce(w, op);
    if (lane == 0) scratch[32] = w;
  }
  __syncthreads();
  return scratch[32];
}

}  // namespace cgk
