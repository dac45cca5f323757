// Mask-apply + temperature + softmax + top-p + sampling, one CTA per row
// (the sampler sees only masked logits, whatever the sampling strategy:
// usetacet.com/docs/grammar, "The guarantee").
//
// Per row b, over the tokens t the bitmask allows, with x_t the logit:
//   temp == 0 : argmax x_t, ties to the lowest id.
//   temp  > 0 : z_t = x_t / temp; m = max z; S = sum exp(z - m);
//               nucleus = {t : z_t >= tau}, tau the largest value whose
//               upper set carries at least top_p of the probability mass
//               (top_p >= 1: every allowed token); token = argmax over the
//               nucleus of z_t + g_t, g_t = -log(-log u_t), u_t from
//               Philox4x32-10 word t&3 of counter (t>>2, b, step, 0), key seed.
// Pass A streams the row once (max, sum of exponentials, greedy argmax; with
// top_p >= 1 also every Gumbel score).  For 0 < top_p < 1 the threshold comes
// from a per-key count histogram of the keys just below the maximum (bf16:
// all tokens with one key share one probability, so the upper-set mass is
// count x exp, exactly order-independent), falling back to a bisection over
// the key space when the nucleus reaches below that window; a last pass draws
// the Gumbel scores of the nucleus only.  Exponentials use exp2 with the
// temperature folded into one scale c = log2(e) / temp.
#include <cuda_bf16.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <utility>

#include "bf16_ops.cuh"
#include "pda.cuh"
#include "row_ops.cuh"

namespace cgk {

constexpr int kSampleThreads = 512;
constexpr int kWindow = 4096;     // keys kept below the row maximum (bf16 path)
constexpr int kAcc = 8;           // independent partial sums per thread
constexpr uint32_t kNotFound = 0xFFFFFFFFu;

enum SampleMode { kGreedy = 0, kTopP = 1, kFull = 2 };

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Calls f(t, x) for every allowed token t of the row.
template <bool BF16, bool VEC, typename F>
__device__ __forceinline__ void for_allowed(const void* row, uint32_t V, const uint32_t* smask, F& f) {
  if (VEC) {
    constexpr uint32_t CH = BF16 ? 8 : 4;
    const uint4* p = reinterpret_cast<const uint4*>(row);
    const uint32_t n = V / CH;
    for (uint32_t i = threadIdx.x; i < n; i += blockDim.x) {
      const uint4 v = ld_stream(p + i);
      const uint32_t t0 = i * CH;
      const uint32_t bits = (smask[t0 >> 5] >> (t0 & 31)) & ((1u << CH) - 1u);
      if (!bits) continue;
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (uint32_t j = 0; j < CH; ++j) {
        if ((bits >> j) & 1u) {
          const float x = BF16 ? bf16_bits_to_float((w[j >> 1] >> (16 * (j & 1))) & 0xFFFFu)
                               : __uint_as_float(w[j]);
          f(t0 + j, x);
        }
      }
    }
  } else {
    for (uint32_t t = threadIdx.x; t < V; t += blockDim.x) {
      if (!((smask[t >> 5] >> (t & 31)) & 1u)) continue;
      const float x = BF16 ? bf16_bits_to_float(reinterpret_cast<const uint16_t*>(row)[t])
                           : reinterpret_cast<const float*>(row)[t];
      f(t, x);
    }
  }
}

// Gumbel score of token t: z_t + g_t (Philox block cached across neighbours)
struct Gumbel {
  uint32_t row, step, k0, k1;
  float temp;
  uint32_t cached = 0xFFFFFFFFu;
  uint4 blk;
  __device__ __forceinline__ float score(uint32_t t, float x) {
    const uint32_t q = t >> 2;
    if (q != cached) {
      blk = philox4x32_10(make_uint4(q, row, step, 0u), k0, k1);
      cached = q;
    }
    return __fdiv_rn(x, temp) + gumbel_from_word(philox_word(blk, t & 3u));
  }
};

// The whole step for one row from the row in global memory (any dtype, any
// V, any mode): pass A streams max / sum / greedy or full Gumbel; the top-p
// threshold comes from the per-key window or, failing that, bisection; a last
// pass samples the nucleus.  `smask` holds the row's bitmask; `cnt` is
// kWindow words of shared scratch.  Returns the token; M and S through refs.
template <bool BF16, bool VEC, int MODE>
__device__ uint32_t general_row(char* row, uint32_t V, const uint32_t* smask, uint32_t* cnt, float temp,
                                float top_p, uint32_t b, uint32_t k0, uint32_t k1, uint32_t step, float& M_out,
                                double& S_out) {
  __shared__ unsigned long long red_u64[33];
  __shared__ float red_f[33];
  __shared__ double red_d[33];
  __shared__ uint32_t s_tau;

  const float c = (MODE == kGreedy) ? 0.f : 1.4426950408889634f / temp;
  unsigned long long best = 0ull;  // packed (value, id); 0 = none
  float m = -INFINITY;
  float sum = 0.f, comp = 0.f;  // compensated (Kahan) sum of exp2((x - m) c)
  Gumbel gum{b, step, k0, k1, temp};
  auto pass_a = [&](uint32_t t, float x) {
    if (MODE == kGreedy) {
      best = max(best, pack_best(x, t));
      return;
    }
    if (x > m) {
      const float r = exp2f((m - x) * c);
      sum *= r;
      comp *= r;
      m = x;
    }
    const float y = exp2f((x - m) * c) - comp;
    const float nt = sum + y;
    comp = (nt - sum) - y;
    sum = nt;
    if (MODE == kFull) best = max(best, pack_best(gum.score(t, x), t));
  };
  for_allowed<BF16, VEC>(row, V, smask, pass_a);

  float M = -INFINITY;
  double S = 0.0;
  if (MODE == kGreedy) {
    best = block_reduce(best, MaxOp(), 0ull, red_u64);
  } else {
    M = block_reduce(m, MaxOp(), -INFINITY, red_f);
    double part = 0.0;
    if (m > -INFINITY) part = (double(sum) - double(comp)) * double(exp2f((m - M) * c));
    S = block_reduce(part, SumOp(), 0.0, red_d);
    if (MODE == kFull) best = block_reduce(best, MaxOp(), 0ull, red_u64);
  }

  if (MODE == kTopP && M > -INFINITY) {
    const double target = double(top_p) * S;
    uint32_t tau = kNotFound;  // bf16: 16-bit key; f32: 32-bit key
    if (BF16) {
      const uint32_t km = fkey(M) >> 16;
      const uint32_t lo = km >= uint32_t(kWindow - 1) ? km - uint32_t(kWindow - 1) : 0u;
      for (uint32_t i = threadIdx.x; i < kWindow; i += blockDim.x) cnt[i] = 0u;
      __syncthreads();
      auto pass_b = [&](uint32_t, float x) {
        const uint32_t k = fkey(x) >> 16;
        if (k >= lo) atomicAdd(cnt + (km - k), 1u);
      };
      for_allowed<BF16, VEC>(row, V, smask, pass_b);
      __syncthreads();
      if (threadIdx.x < 32) {
        const uint32_t lane = threadIdx.x;
        double cum = 0.0;
        uint32_t found = kNotFound;
        for (uint32_t base = 0; base <= km - lo && found == kNotFound; base += 32) {
          const uint32_t j = base + lane;
          double mass = 0.0;
          if (j <= km - lo && cnt[j]) mass = double(cnt[j]) * double(exp2f((bf16key_to_float(km - j) - M) * c));
          double incl = mass;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= uint32_t(o)) incl += y;
          }
          const unsigned hit = __ballot_sync(0xFFFFFFFFu, cum + incl >= target);
          if (hit) found = base + uint32_t(__ffs(hit) - 1);
          cum += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (lane == 0) s_tau = (found == kNotFound) ? kNotFound : km - found;
      }
      __syncthreads();
      tau = s_tau;
    }
    if (tau == kNotFound) {
      // bisection: largest key kappa whose upper set carries >= target
      uint32_t lo = 0, hi = BF16 ? (fkey(M) >> 16) : fkey(M);
      while (lo < hi) {
        const uint32_t mid = lo + (hi - lo + 1) / 2;
        float part = 0.f;
        auto pass_s = [&](uint32_t, float x) {
          const uint32_t k = BF16 ? (fkey(x) >> 16) : fkey(x);
          if (k >= mid) part += exp2f((x - M) * c);
        };
        for_allowed<BF16, VEC>(row, V, smask, pass_s);
        const double mass = block_reduce(double(part), SumOp(), 0.0, red_d);
        if (mass >= target) lo = mid; else hi = mid - 1;
      }
      tau = lo;
    }
    auto pass_c = [&](uint32_t t, float x) {
      const uint32_t k = BF16 ? (fkey(x) >> 16) : fkey(x);
      if (k >= tau) best = max(best, pack_best(gum.score(t, x), t));
    };
    for_allowed<BF16, VEC>(row, V, smask, pass_c);
    best = block_reduce(best, MaxOp(), 0ull, red_u64);
  }
  M_out = M;
  S_out = S;
  return best ? best_id(best) : CG_NO_TOKEN;
}

// Optional outputs: softmax over allowed tokens (greedy: 1 at the token) and
// -inf written into masked logits.
template <bool BF16, int MODE>
__device__ void write_outputs(char* row, uint32_t V, const uint32_t* smask, uint32_t tok, float M, double S,
                              float temp, float* probs, int inplace, uint32_t b) {
  const float c = (MODE == kGreedy) ? 0.f : 1.4426950408889634f / temp;
  if (probs) {
    float* prow = probs + size_t(b) * V;
    const float invS = (MODE == kGreedy || S <= 0.0) ? 0.f : float(1.0 / S);
    for (uint32_t t = threadIdx.x; t < V; t += blockDim.x) {
      float p = 0.f;
      if ((smask[t >> 5] >> (t & 31)) & 1u) {
        if (MODE == kGreedy) {
          p = (t == tok) ? 1.f : 0.f;
        } else {
          const float x = BF16 ? bf16_bits_to_float(reinterpret_cast<const uint16_t*>(row)[t])
                               : reinterpret_cast<const float*>(row)[t];
          p = exp2f((x - M) * c) * invS;
        }
      }
      prow[t] = p;
    }
  }
  if (inplace) {
    __syncthreads();  // every read of the row is done
    for (uint32_t t = threadIdx.x; t < V; t += blockDim.x) {
      if ((smask[t >> 5] >> (t & 31)) & 1u) continue;
      if (BF16) reinterpret_cast<uint16_t*>(row)[t] = 0xFF80u;
      else reinterpret_cast<float*>(row)[t] = -INFINITY;
    }
  }
}

template <bool BF16, bool VEC, int MODE>
__global__ void __launch_bounds__(kSampleThreads) sample_kernel(void* logits, uint32_t V,
                                                                 uint32_t W, const uint32_t* __restrict__ bitmask,
                                                                 float temp, float top_p, uint32_t k0, uint32_t k1,
                                                                 uint32_t step, uint32_t* __restrict__ out_tok,
                                                                 float* __restrict__ probs, int inplace) {
  extern __shared__ uint32_t smem[];
  uint32_t* smask = smem;             // [W]
  uint32_t* cnt = smem + W;           // [kWindow] (top-p, bf16)
  griddep_launch_dependents();
  griddep_wait();  // the bitmask comes from fill_bitmask
  const uint32_t b = blockIdx.x;
  const size_t esz = BF16 ? 2 : 4;
  char* row = reinterpret_cast<char*>(logits) + size_t(b) * V * esz;
  const uint32_t* mrow = bitmask + size_t(b) * W;
  for (uint32_t i = threadIdx.x; i < W; i += blockDim.x) smask[i] = mrow[i];
  __syncthreads();
  float M;
  double S;
  const uint32_t tok = general_row<BF16, VEC, MODE>(row, V, smask, cnt, temp, top_p, b, k0, k1, step, M, S);
  if (threadIdx.x == 0) out_tok[b] = tok;
  write_outputs<BF16, MODE>(row, V, smask, tok, M, S, temp, probs, inplace, b);
}

// ============================================================================
// Top-p kernel for bf16 rows (the path of the throughput metric): each logit is
// read from HBM once.
//
// One CTA of 512 threads per row.  Warp 15 fills a kStages-slot shared-memory
// ring with bulk asynchronous copies (cp.async.bulk completing on "full"
// mbarriers; slots come back through "empty" mbarriers).  Warps 0..14 take each
// chunk 16 logits per thread (two 8-logit groups): the bitmask is applied
// through a 256-entry table of pair masks indexed by the group's mask byte, the
// group maximum comes from packed bf16 max, and exp2((x - m) c) is summed into
// 8 partial sums against the thread's own running maximum m (so that S does
// not depend on warp timing).  The block's running maximum is published per
// chunk (warp max-reduction and a shared atomicMax); a group whose maximum
// reaches it minus kMarginZ nats is copied, masked, into its warp's staging
// area in shared memory (positions from a warp ballot); whenever 32 groups are staged the warp turns them into
// candidates -- allowed logits at or above the block's running maximum minus
// the margin -- one group per lane, and appends them (id, 16-bit key) to the
// row's candidate list in global memory.  The running maximum never exceeds
// the final maximum M, so every allowed logit within kMarginZ nats of M
// becomes a candidate; which others do depends on timing, but only candidates
// at or above M - margin count afterwards.
//
// After the stream: M and S = sum exp2((x - M) c) come from the block; the
// nucleus threshold tau is the largest key whose upper set carries top_p * S
// (per-key counts over the candidates, by keys or by coarse bins then keys);
// the nucleus entries are packed into shared memory and Gumbel scores drawn
// for them only.  Rows whose nucleus reaches below the margin, or whose list
// overflows, run general_row instead.
// ============================================================================
namespace fast {

constexpr int kThreads = 512;
constexpr uint32_t kConsumerWarps = 15;
constexpr uint32_t kConsumers = kConsumerWarps * 32;            // 480
constexpr int kStages = 4;
constexpr uint32_t kChunkElems = kConsumers * 16;               // 7680 logits per slot
constexpr uint32_t kChunkBytes = kChunkElems * 2;               // 15 KiB
constexpr uint32_t kGroupsPerChunk = kChunkElems / 8;           // 960
constexpr uint32_t kRing = kStages * kChunkBytes;               // 60 KiB
constexpr uint32_t kStage = 64;                                 // staged groups per warp
constexpr uint32_t kBins = 512;                                 // bins per histogram
constexpr uint32_t kHists = 4;                                  // histogram copies
static_assert(kBins == kThreads, "one histogram bin per thread in the scans");
// after the stream the ring holds the histograms, then the packed nucleus
constexpr uint32_t kHistBytes = kHists * kBins * 8;
constexpr uint32_t kNucCap = (kRing - kHistBytes) / 6;          // packed nucleus entries (u32 id + u16 key)
// nats below the maximum kept as candidates: a row whose top-p boundary lies
// deeper takes the general path (same result, one more pass over the row).
// Where a few percent of the tokens carry most of the mass the boundary lies
// within about 7.2 nats of the maximum; flat rows (Gaussian logits over tens
// of thousands of tokens, no dominant ones) can reach past 9.
constexpr float kMarginZ = 8.5f;
constexpr float kNoRef = -1e30f;                                // finite reference before any allowed logit
constexpr uint32_t kWinRowsMax = 512;                           // states in the accept's table window
constexpr uint32_t kWinBytesMax = 16384;                        // shared memory for that window
constexpr uint32_t kSlots = 16;                                 // list entries per thread after the stream
constexpr uint32_t kCandPerRow = kThreads * kSlots;             // candidate list entries per row (8192)
static_assert(kCandPerRow == kSampleListEntries, "the no-allocation scratch holds the rows' lists");
constexpr uint32_t kBatchIds = 4;                               // nucleus id loads in flight per thread

// Prefix sums over bins 0..kBins-1 (bin = thread; q = this thread's bin mass),
// starting from `base`: returns the first bin whose inclusive sum reaches
// target (or kNotFound) and, through `above`, the sum before that bin.
// `s_first` must hold kNotFound on entry.  Ends with the block in step.
__device__ uint32_t scan_bins(unsigned long long q, unsigned long long target, unsigned long long base,
                              unsigned long long* red, uint32_t* s_first, unsigned long long& above) {
  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned long long qi = q;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, qi, o);
    if (lane >= uint32_t(o)) qi += y;
  }
  if (lane == 31) red[warp] = qi;
  __syncthreads();
  unsigned long long before = base;
  for (uint32_t wi = 0; wi < warp; ++wi) before += red[wi];
  if (before + qi >= target) atomicMin(s_first, tid);
  __syncthreads();
  const uint32_t j = *s_first;
  if (j != kNotFound && tid == j) red[32] = before + qi - q;
  __syncthreads();
  above = j != kNotFound ? red[32] : 0ull;
  return j;
}

__device__ __forceinline__ void issue_chunk(unsigned char* ring, uint64_t* full, const char* row, uint32_t V,
                                            uint32_t k) {
  const uint32_t slot = k % kStages;
  const uint32_t bytes = min(kChunkElems, V - k * kChunkElems) * 2;
  mbar_expect_tx(full + slot, bytes);
  // the logits are read once: evict them first, keep the mask cache in L2
  bulk_g2s_hint(ring + size_t(slot) * kChunkBytes, row + size_t(k) * kChunkBytes, bytes, full + slot,
                evict_first_policy());
}

// One warp turns staged groups [top - n, top) into candidates: lane l takes
// group top - n + l, keeps its allowed logits >= thr, and the warp appends them
// to the row's list (one shared atomic per call).
__device__ __forceinline__ void drain_stage(const uint4* stg, const uint16_t* sgid, uint32_t top, uint32_t n,
                                            float thr, uint32_t* s_count, uint32_t* gid_out, uint16_t* gkey_out,
                                            uint32_t gcap) {
  const uint32_t lane = threadIdx.x & 31;
  uint32_t hits = 0, g = 0;
  uint4 d = make_uint4(0u, 0u, 0u, 0u);
  if (lane < n) {
    d = stg[top - n + lane];
    g = sgid[top - n + lane];
    // x >= thr for a bf16 x exactly when x >= the least bf16 not below thr
    const __nv_bfloat162 t2 = __bfloat162bfloat162(__float2bfloat16_ru(thr));
    const uint32_t wv[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t m = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&wv[q]), t2);
      hits |= ((m & 1u) | ((m >> 15) & 2u)) << (2 * q);
    }
  }
  const uint32_t nh = __popc(hits);
  uint32_t inc = nh;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
    if (lane >= uint32_t(o)) inc += y;
  }
  uint32_t wb = 0;
  if (lane == 31 && inc) wb = atomicAdd(s_count, inc);
  uint32_t pos = __shfl_sync(0xFFFFFFFFu, wb, 31) + inc - nh;
  while (hits) {
    const uint32_t e = __ffs(hits) - 1;
    hits &= hits - 1;
    if (pos < gcap) {
      gid_out[pos] = g * 8 + e;
      gkey_out[pos] = bf16_key(group_bits(d, e));
    }
    ++pos;
  }
}

// Inputs and outputs of the fused step (cg_step): the row's bitmask is built
// in shared memory as cg_fill_bitmask would write it, and the sampled token is
// accepted as cg_accept would.
constexpr uint32_t kParamGrammars = 8;  // grammar descriptors passed by value

struct StepArgs {
  Tables t;
  const uint32_t* states;
  const uint16_t* gid;      // may be null
  const int32_t* forced;    // may be null
  uint32_t* counts;         // may be null
  uint32_t max_tokens;
  uint32_t* out_states;
  uint8_t* out_flags;
  uint32_t* bitmask_out;    // may be null: the mask then never leaves the chip
  DevGrammar pg[kParamGrammars];  // copies of t.grammars[0 .. n_pg): one dependent load fewer
  uint32_t n_pg;
  uint32_t cache_complete;  // every class mask is in the cache (cg_ctx_prefill ran): skip the ready check
  uint32_t win_bytes;       // shared memory for the accept's table window (0: none)
  DevPda pda;               // pushdown step: the automaton (its tables read from global memory)
  uint32_t* pda_cfg;        // pushdown step: row configurations [B][depth + 2], updated in place
};

// Grammar g's descriptor from the kernel parameters when they hold it (an
// unrolled select keeps the reads in the parameter space), else from memory.
__device__ __forceinline__ DevGrammar step_grammar(const StepArgs& sa, uint32_t g) {
  if (g >= sa.n_pg) return sa.t.grammars[g];
  DevGrammar gd = sa.pg[0];
#pragma unroll
  for (uint32_t i = 1; i < kParamGrammars; ++i)
    if (g == i) gd = sa.pg[i];
  return gd;
}

// The row's mask in shared memory, as cg_fill_bitmask defines it.  All threads
// of the block take part.  Thread 0 loads the row's grammar, forced token and
// state, then the state's flags and mask class together; a cached class mask
// arrives as one bulk copy completing on *mbar_mask (the caller waits on it,
// parity 0, when *s_copied is set).  scol is 512 bytes of free shared memory
// for the miss path.
__device__ void step_row_mask(const StepArgs& sa, uint32_t b, uint32_t W, uint32_t* smask, uint16_t* scol,
                              uint64_t* mbar_mask, uint32_t& s_copied, uint32_t& s_mode,
                              uint32_t& s_cls, uint32_t& s_ready, uint32_t& s_claim, uint32_t& s_g, uint32_t& s_s,
                              int32_t& s_f) {
  const Tables& t = sa.t;
  const uint32_t tid = threadIdx.x;
  if (tid == 0) {
    const uint32_t g = sa.gid ? sa.gid[b] : 0u;
    const int32_t f = sa.forced ? sa.forced[b] : -1;
    const uint32_t s = sa.states[b];
    DevGrammar gd{};
    if (g < t.n_g) gd = step_grammar(sa, g);
    const bool in_range = g < t.n_g && s != CG_DEAD && s < gd.n_states;
    uint8_t sflags = 0;
    uint32_t cls = 0;
    if (in_range && f < 0) {
      sflags = t.state_flags[gd.state_off + s];
      cls = t.class_of[gd.state_off + s];
    }
    uint32_t err = 0;
    const int mode = row_mask_mode_of(t.n_g, t.V, g, f, s, gd.n_states, sflags, &err);
    if (err) record_error(t.status, err);
    uint32_t copied = 0, ready = 0;
    if (mode == 0) {
      ready = sa.cache_complete ? 1u : (load_acquire(t.cache_state + cls) == kStateReady);
      if (ready && (W & 3u) == 0) {
        mbar_expect_tx(mbar_mask, W * 4);
        bulk_g2s(smask, t.cache + size_t(cls) * t.Wc, W * 4, mbar_mask);
        copied = 1;
      }
    }
    s_copied = copied;
    s_mode = uint32_t(mode);
    s_cls = cls;
    s_ready = ready;
    s_g = g;
    s_s = s;
    s_f = f;
  }
  __syncthreads();
  const uint32_t mode = s_mode;
  if (mode == 1) {
    for (uint32_t i = tid; i < W; i += blockDim.x) smask[i] = 0u;
  } else if (mode == 2) {
    const uint32_t f = uint32_t(s_f);
    for (uint32_t i = tid; i < W; i += blockDim.x) smask[i] = (i == (f >> 5)) ? (1u << (f & 31)) : 0u;
  } else if (s_ready) {
    if (!s_copied) {
      const uint32_t* crow = t.cache + size_t(s_cls) * t.Wc;
      for (uint32_t i = tid; i < W; i += blockDim.x) smask[i] = crow[i];
    }
  } else {
    // miss: compute the class mask from the row's state, publish it if this
    // block claims the class (as cg_fill_bitmask does)
    const uint32_t g = s_g, cls = s_cls;
    for (uint32_t i = tid; i < W; i += blockDim.x) smask[i] = 0u;
    for (uint32_t i = tid; i < 256; i += blockDim.x) scol[i] = t.colmap[size_t(g) * 512 + i];
    if (tid == 0) s_claim = atomicCAS(t.cache_state + cls, kStateEmpty, kStateBusy) == kStateEmpty;
    __syncthreads();
    walk_tokens(t, t.grammars[g], scol, s_s, smask, tid, blockDim.x);
    __syncthreads();
    if (s_claim) {
      uint32_t* cw = t.cache + size_t(cls) * t.Wc;
      for (uint32_t i = tid; i < W; i += blockDim.x) cw[i] = smask[i];
      __threadfence();
      __syncthreads();
      if (tid == 0) store_release(t.cache_state + cls, kStateReady);
    }
  }
}

// The accept's tables, staged by the producer warp while the row streams:
// grammar g's symbol -> column map, and (lane 0, one bulk copy completing on
// *mbar_win) the rows of the states around s in the 16-bit table, with their
// flags.  *s_wlo / *s_wrows / *s_wdelta describe the window (rows 0: none).
__device__ void stage_accept_tables(const StepArgs& sa, uint32_t g, uint32_t s, uint16_t* scols, uint16_t* win,
                                    uint8_t* wflags, uint64_t* mbar_win, uint32_t* s_wlo, uint32_t* s_wrows,
                                    uint32_t* s_wdelta, uint32_t lane) {
  const Tables& t = sa.t;
  if (g >= t.n_g) return;
  for (uint32_t i = lane; i < 512; i += 32) scols[i] = t.colmap[size_t(g) * 512 + i];
  const DevGrammar gd = step_grammar(sa, g);
  const WindowCopy wc = window_copy(t, gd, s, sa.win_bytes, kWinRowsMax);
  if (wc.rows == 0) return;
  if (lane == 0) {
    mbar_expect_tx(mbar_win, wc.bytes);
    bulk_g2s(win, wc.src, wc.bytes, mbar_win);
    *s_wlo = wc.lo;
    *s_wdelta = wc.delta;
    *s_wrows = wc.rows;
  }
  const uint32_t lo = wc.lo, rows = wc.rows;
  for (uint32_t i = lane; i < rows; i += 32) wflags[i] = t.state_flags[gd.state_off + lo + i];
}

// The mask of a pushdown row (cg_pda_step), as cg_pda_fill_bitmask defines
// it.  All threads of the block take part.  Thread 0 reads the row's
// configuration and forced token and starts the bulk copy of the cached mask
// of (state, headroom), completing on *mbar_mask (parity 0); meanwhile the
// threads walk the state's listed tokens against the row's stack (tables read
// from global memory) and collect the allowed ones in `list` (list_cap words
// of free shared memory); once the copy has landed they are ORed into the
// mask.  A longer list than list_cap is ORed in directly after the copy.
__device__ void pda_row_mask(const StepArgs& sa, uint32_t b, uint32_t W, uint32_t* smask, uint32_t* list,
                             uint32_t list_cap, uint64_t* mbar_mask, uint32_t& s_copied, uint32_t& s_mode,
                             uint32_t& s_mi, uint32_t& s_c0, uint32_t& s_c1, uint32_t& s_n, int32_t& s_f,
                             uint32_t& s_flag) {
  const Tables& t = sa.t;
  const DevPda& p = sa.pda;
  const uint32_t tid = threadIdx.x;
  const uint32_t* row = sa.pda_cfg + size_t(b) * p.stride;
  if (tid == 0) {
    const uint32_t q = row[0], lvl = row[1];
    const int32_t f = sa.forced ? sa.forced[b] : -1;
    uint32_t mode = 0, copied = 0, mi = 0, c0 = 0, c1 = 0;
    if (f >= 0) {
      mode = uint32_t(f) < t.V ? 2u : 1u;
      if (mode == 1) record_error(t.status, CG_DEV_BAD_FORCED);
    } else if (q >= p.S || lvl > p.depth) {
      mode = 1;
      if (q != CG_DEAD) record_error(t.status, CG_DEV_BAD_STATE);
    } else {
      const uint32_t kinfo = p.key[q];
      mi = p.mask_of[(kinfo >> 8) + min(p.depth - lvl, kinfo & 0xFFu)];
      c0 = p.cand_off[q];
      c1 = p.cand_off[q + 1];
      if ((W & 3u) == 0) {
        mbar_expect_tx(mbar_mask, W * 4);
        bulk_g2s(smask, p.masks + size_t(mi) * W, W * 4, mbar_mask);
        copied = 1;
      }
    }
    s_mode = mode;
    s_f = f;
    s_copied = copied;
    s_mi = mi;
    s_c0 = c0;
    s_c1 = c1;
    s_n = 0;
  }
  __syncthreads();
  const uint32_t mode = s_mode;
  if (mode == 1) {
    for (uint32_t i = tid; i < W; i += blockDim.x) smask[i] = 0u;
    return;
  }
  if (mode == 2) {
    const uint32_t f = uint32_t(s_f);
    for (uint32_t i = tid; i < W; i += blockDim.x) smask[i] = (i == (f >> 5)) ? (1u << (f & 31)) : 0u;
    return;
  }
  const bool copied = s_copied != 0;
  if (!copied) {
    const uint32_t* crow = p.masks + size_t(s_mi) * W;
    for (uint32_t i = tid; i < W; i += blockDim.x) smask[i] = crow[i];
  }
  const uint32_t c0 = s_c0, c1 = s_c1, q = row[0], lvl = row[1];
  const bool listed = c1 - c0 <= list_cap;
  if (!listed) {
    if (copied && !mbar_wait(mbar_mask, 0)) atomicOr(&s_flag, 1u);
    __syncthreads();
  }
  for (uint32_t i = c0 + tid; i < c1; i += blockDim.x) {
    const uint32_t tok = p.cand[i];
    uint32_t qq = q, ll = lvl;
    OverlayStack st;
    st.base = row + 2;
    st.keep = lvl;
    if (pda_walk(p, t, tok, 0u, qq, ll, st)) {
      if (listed) list[atomicAdd(&s_n, 1u)] = tok;
      else atomicOr(&smask[tok >> 5], 1u << (tok & 31u));
    }
  }
  if (listed) {
    if (copied && !mbar_wait(mbar_mask, 0)) atomicOr(&s_flag, 1u);
    __syncthreads();
    for (uint32_t i = tid; i < s_n; i += blockDim.x) atomicOr(&smask[list[i] >> 5], 1u << (list[i] & 31u));
  }
}

// STEP: 0 sampling from a bitmask (cg_mask_and_sample); 1 the fused step of
// automaton rows (cg_step); 2 the fused step of pushdown rows (cg_pda_step).
template <int STEP>
__global__ void __launch_bounds__(kThreads, 2)
    stream_topp_kernel(void* logits, uint32_t V, uint32_t W, const uint32_t* __restrict__ bitmask, float temp,
                       float top_p, uint32_t k0, uint32_t k1, uint32_t step, uint32_t* __restrict__ out_tok,
                       float* __restrict__ probs, int inplace, uint32_t* cand_id, uint16_t* cand_key,
                       uint32_t gcap, uint32_t* status, const StepArgs sa) {
  extern __shared__ __align__(128) unsigned char dsm[];
  unsigned char* ring = dsm;                                                // kStages slots
  uint4* lut = reinterpret_cast<uint4*>(dsm + kRing);                       // [256]
  uint4* stg_all = lut + 256;                                               // [kConsumerWarps][kStage]
  uint16_t* sgid_all = reinterpret_cast<uint16_t*>(stg_all + kConsumerWarps * kStage);
  uint32_t* smask = reinterpret_cast<uint32_t*>(sgid_all + kConsumerWarps * kStage);  // [W]
  uint16_t* scols = reinterpret_cast<uint16_t*>(smask + ((W + 3) & ~3u));          // [512] (fused step)
  uint8_t* wflags = reinterpret_cast<uint8_t*>(scols + 512);                        // [kWinRowsMax] (fused step)
  uint16_t* win = reinterpret_cast<uint16_t*>(wflags + kWinRowsMax);                // [win_bytes / 2] (fused step)
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages], mbar_mask, mbar_win;
  __shared__ uint32_t s_copied, s_wlo, s_wrows, s_wdelta;
  __shared__ float red_f[33];
  __shared__ unsigned long long red_u64[33];
  __shared__ uint32_t s_maxkey, s_flag, s_count, s_tau;
  __shared__ uint32_t s_mode, s_cls, s_ready, s_claim, s_g, s_s;
  __shared__ int32_t s_f;

  griddep_launch_dependents();
  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, b = blockIdx.x;
  char* row = reinterpret_cast<char*>(logits) + size_t(b) * V * 2;
  const uint32_t nchunks = (V + kChunkElems - 1) / kChunkElems;
  uint32_t* gid_row = cand_id + size_t(b) * gcap;
  uint16_t* gkey_row = cand_key + size_t(b) * gcap;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, kConsumerWarps);
    }
    mbar_init(&mbar_mask, 1);
    mbar_init(&mbar_win, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_maxkey = fkey(-INFINITY);
    s_flag = 0;  // bit 0: a wait ran out
    s_count = 0;
    s_copied = 0;
    s_wrows = 0;
  }
  for (uint32_t i = tid; i < 256; i += kThreads) lut[i] = pair_mask_entry(i);
  __syncthreads();  // barriers initialised
  griddep_wait();   // the bitmask (or, fused, the states) come from the previous kernel
  if (STEP == 0) {
    const uint32_t* mrow = bitmask + size_t(b) * W;
    for (uint32_t i = tid; i < W; i += kThreads) smask[i] = mrow[i];
  } else {
    // the logits do not depend on the mask: start the first copies now
    if (warp == kConsumerWarps && lane == 0)
      for (uint32_t k = 0; k < nchunks && k < uint32_t(kStages); ++k) issue_chunk(ring, full, row, V, k);
    if (STEP == 1)
      step_row_mask(sa, b, W, smask, reinterpret_cast<uint16_t*>(stg_all), &mbar_mask, s_copied, s_mode, s_cls,
                    s_ready, s_claim, s_g, s_s, s_f);
    else
      pda_row_mask(sa, b, W, smask, reinterpret_cast<uint32_t*>(stg_all), kConsumerWarps * kStage * 4, &mbar_mask,
                   s_copied, s_mode, s_cls, s_g, s_s, s_ready, s_f, s_flag);
  }
  __syncthreads();

  const float c = 1.4426950408889634f / temp;
  const float margin = kMarginZ * temp;  // z = x / temp: kMarginZ nats are kMarginZ * temp logit units
  const uint8_t* smask8 = reinterpret_cast<const uint8_t*>(smask);
  float mt = kNoRef;  // reference of this thread's sums: its running maximum
  float2 acc[kAcc / 2];
#pragma unroll
  for (int j = 0; j < kAcc / 2; ++j) acc[j] = make_float2(0.f, 0.f);

  if (warp == kConsumerWarps) {
    // ---- producer warp --------------------------------------------------------------
    if (STEP == 1) stage_accept_tables(sa, s_g, s_s, scols, win, wflags, &mbar_win, &s_wlo, &s_wrows, &s_wdelta, lane);
    if (lane == 0) {
      bool ok = true;
      for (uint32_t k = STEP != 0 ? min(nchunks, uint32_t(kStages)) : 0u; k < nchunks; ++k) {
        if (k >= uint32_t(kStages) && !mbar_wait(empty + k % kStages, ((k / kStages) - 1) & 1u)) {
          ok = false;
          break;
        }
        issue_chunk(ring, full, row, V, k);
      }
      if (!ok) atomicOr(&s_flag, 1u);
    }
  } else {
    // ---- consumers ----------------------------------------------------------------
    uint4* stg = stg_all + warp * kStage;
    uint16_t* sgid = sgid_all + warp * kStage;
    uint32_t sc = 0;  // staged groups of this warp (warp-uniform)
    const uint32_t lt = (1u << lane) - 1u;
    // the row's mask (fused step: a bulk copy from the mask cache)
    if (STEP != 0 && s_copied && !mbar_wait(&mbar_mask, 0)) atomicOr(&s_flag, 1u);
    // chunk 0's maximum seeds the reference, so the first chunk does not flag
    // every group
    if (!mbar_wait(full + 0, 0)) atomicOr(&s_flag, 1u);
    {
      const uint4* r4 = reinterpret_cast<const uint4*>(ring);
      float lm = -INFINITY;
#pragma unroll
      for (uint32_t g = 0; g < 2; ++g) {
        const uint32_t gi = tid + kConsumers * g;
        if (gi * 8 < V) lm = fmaxf(lm, group_max(apply_mask(r4[gi], lut[smask8[gi]])));
      }
      const uint32_t wk = __reduce_max_sync(0xFFFFFFFFu, fkey(lm));
      if (lane == 0) atomicMax(&s_maxkey, wk);
      asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");  // consumer warps only
    }
    bool ok = true;
    // two slots per pass: the threshold, the warp's maximum and the hand-back
    // are paid once for four groups per thread
    for (uint32_t k = 0; k < nchunks; k += 2) {
      const bool two = k + 1 < nchunks;
      // flag threshold for these chunks: the block's running maximum minus the
      // margin (never above M - margin; finite, so masked groups never flag)
      const float thr = fmaxf(fkey_inv(*reinterpret_cast<volatile uint32_t*>(&s_maxkey)), kNoRef) - margin;
      if (!mbar_wait(full + k % kStages, (k / kStages) & 1u) ||
          (two && !mbar_wait(full + (k + 1) % kStages, ((k + 1) / kStages) & 1u))) {
        atomicOr(&s_flag, 1u);
        ok = false;
        break;
      }
      uint4 v[4];
      uint32_t gg[4];  // row group index of each of the thread's groups
#pragma unroll
      for (uint32_t h = 0; h < 2; ++h) {
        const uint32_t kk = k + h;
        const uint4* r4 = reinterpret_cast<const uint4*>(ring + size_t(kk % kStages) * kChunkBytes);
        const uint32_t gbase = kk * kGroupsPerChunk;  // row group index of the chunk's group 0
        const uint32_t ngroups = (h == 0 || two) ? min(kGroupsPerChunk, V / 8 - gbase) : 0u;
#pragma unroll
        for (uint32_t q = 0; q < 2; ++q) {
          const uint32_t gi = tid + kConsumers * q;
          v[2 * h + q] = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
          if (gi < ngroups) v[2 * h + q] = apply_mask(r4[gi], lut[smask8[gbase + gi]]);
          gg[2 * h + q] = gbase + gi;
        }
      }
      // the slots' data are in registers: hand the slots back
      float gq[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) gq[q] = group_max(v[q]);
      const float gm = fmaxf(fmaxf(gq[0], gq[1]), fmaxf(gq[2], gq[3]));
      const uint32_t wk = __reduce_max_sync(0xFFFFFFFFu, fkey(gm));
      __syncwarp();
      if (lane == 0) {
        atomicMax(&s_maxkey, wk);
        mbar_arrive(empty + k % kStages);
        if (two) mbar_arrive(empty + (k + 1) % kStages);
      }
      if (gm > mt) {
        // the sums' reference is this thread's own running maximum, so that
        // they do not depend on the other warps' timing (S is reproducible)
        const float r = ex2((mt - gm) * c);
#pragma unroll
        for (int j = 0; j < kAcc / 2; ++j) acc[j] = __fmul2_rn(acc[j], make_float2(r, r));
        mt = gm;
      }
      const float mc = mt * c;
#pragma unroll
      for (int q = 0; q < 4; ++q) add_exps(acc, v[q], make_float2(c, c), make_float2(-mc, -mc));
      // stage the flagged groups (fewer than 32 are staged before each group
      // is added, at most 63 after); turn staged groups into candidates 32 at a
      // time
#pragma unroll
      for (uint32_t q = 0; q < 4; ++q) {
        const bool f = gq[q] >= thr;
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, f);
        if (bal) {
          if (f) {
            const uint32_t p = sc + __popc(bal & lt);
            stg[p] = v[q];
            sgid[p] = uint16_t(gg[q]);
          }
          sc += __popc(bal);
          if (sc >= 32) {
            __syncwarp();
            const float thr_now = fmaxf(fkey_inv(*reinterpret_cast<volatile uint32_t*>(&s_maxkey)), kNoRef) - margin;
            drain_stage(stg, sgid, sc, 32, thr_now, &s_count, gid_row, gkey_row, gcap);
            sc -= 32;
            __syncwarp();
          }
        }
      }
    }
    if (ok && sc) {
      __syncwarp();
      const float thr_now = fmaxf(fkey_inv(*reinterpret_cast<volatile uint32_t*>(&s_maxkey)), kNoRef) - margin;
      drain_stage(stg, sgid, sc, sc, thr_now, &s_count, gid_row, gkey_row, gcap);
    }
  }
  __syncthreads();

  // ---- row statistics -----------------------------------------------------------
  if ((s_flag & 1u) && tid == 0) {
    // a wait ran out: let copies still in flight land before the shared memory
    // is reused or released (again with a bounded wait)
    for (uint32_t sl = 0; sl < uint32_t(kStages) && sl < nchunks; ++sl) {
      const uint32_t issued = (nchunks - sl + kStages - 1) / kStages;
      mbar_wait(full + sl, (issued - 1) & 1u);
    }
    if (STEP != 0 && s_copied) mbar_wait(&mbar_mask, 0);
    if (STEP == 1 && s_wrows) mbar_wait(&mbar_win, 0);
  }
  const float M = fkey_inv(s_maxkey);  // -inf when no logit is allowed
  // S: per-thread partial sums, warp sums and the 16 warp sums, all in float
  // (relative error near 1e-7; double arithmetic is slow on this part)
  {
    float part = 0.f;
    if (M > -INFINITY) {
      float a = 0.f;
#pragma unroll
      for (int jj = 0; jj < kAcc / 2; ++jj) a = (a + acc[jj].x) + acc[jj].y;
      if (a > 0.f) part = a * ex2((mt - M) * c);
    }
    part = warp_reduce(part, SumOp());
    if (lane == 0) red_f[warp] = part;
  }
  const bool stats_ok = !(s_flag & 1u) && M > -1e29f && M < 1e29f;
  const float thrF = M - margin;     // every allowed logit >= thrF is a candidate
  const uint32_t km = fkey(M) >> 16;
  uint32_t kthr = fkey(thrF) >> 16;  // smallest key whose value is >= thrF
  if (stats_ok && bf16key_to_float(kthr) < thrF) ++kthr;
  // histogram bin j: keys km - j (coarse: keys (km - (j+1) 2^sh, km - j 2^sh])
  const uint32_t span = stats_ok ? km - kthr : 0u;
  uint32_t sh = 0;
  while ((span >> sh) >= kBins) ++sh;
  unsigned long long* hq = reinterpret_cast<unsigned long long*>(ring);  // [kHists][kBins]
  uint32_t* hc = reinterpret_cast<uint32_t*>(ring);                      // [kHists][kBins] (counts)
  __syncthreads();  // red_f complete; the ring is free
  const uint32_t n_all = s_count;
  if (tid == 0) s_tau = kNotFound;
  // counts (keys) need kHists x kBins words, masses (coarse bins) twice that
  for (uint32_t i = tid; i < kHists * kBins * (sh ? 2 : 1); i += kThreads) hc[i] = 0u;
  float Sf = 0.f;
#pragma unroll
  for (uint32_t wi = 0; wi < kThreads / 32; ++wi) Sf += red_f[wi];
  const double S = Sf;
  __syncthreads();
  uint32_t tok = CG_NO_TOKEN;
  bool general = false;
  if (s_flag & 1u) {
    if (tid == 0) record_error(status, CG_DEV_TIMEOUT);
  } else if (!stats_ok) {
    general = M > -INFINITY;  // huge or infinite logits: the plain path copes with them
  } else if (n_all > gcap) {
    general = true;
  } else {
    const unsigned long long target_q =
        static_cast<unsigned long long>(top_p * Sf * 1099511627776.0f);  // top_p of the mass, 2^-40 units
    const uint32_t n = n_all;
    const uint32_t nslots = (n + kThreads - 1) / kThreads;  // slots any thread uses
    // the keys of this thread's list entries tid + 512 j, all loads in flight
    // at once; keys below kthr (and empty slots) read as 0, under every
    // threshold (ids are read later, for nucleus entries only)
    static_assert(kCandPerRow == kThreads * kSlots, "list entries per thread");
    uint32_t kk[kSlots / 2];
#pragma unroll
    for (uint32_t j = 0; j < kSlots; ++j) {
      const uint32_t i = tid + kThreads * j;
      uint32_t key = (j < nslots && i < n) ? gkey_row[i] : 0u;
      if (key < kthr) key = 0;
      if (j & 1) kk[j / 2] |= key << 16; else kk[j / 2] = key;
    }
    auto key_at = [&](uint32_t j) { return (kk[j / 2] >> ((j & 1) * 16)) & 0xFFFFu; };
    // ---- nucleus threshold: per-key counts (or per-bin masses when the keys
    // span more than kBins), scanned from the top
    unsigned long long above = 0;
    uint32_t J;
    if (sh == 0) {
      uint32_t* hmine = hc + (warp % kHists) * kBins;
#pragma unroll
      for (uint32_t j = 0; j < kSlots; ++j) {
        if (j >= nslots) break;
        const uint32_t key = key_at(j);
        if (key) atomicAdd(hmine + (km - key), 1u);
      }
      __syncthreads();
      uint32_t cnt = 0;
#pragma unroll
      for (uint32_t h = 0; h < kHists; ++h) cnt += hc[h * kBins + tid];
      const unsigned long long q =
          (tid <= span && cnt) ? (unsigned long long)cnt * mass_q(bf16key_to_float(km - tid), M, c) : 0ull;
      J = scan_bins(q, target_q, 0ull, red_u64, &s_tau, above);
      if (J != kNotFound) J = km - J;
    } else {
      unsigned long long* hmine = hq + (warp % kHists) * kBins;
#pragma unroll
      for (uint32_t j = 0; j < kSlots; ++j) {
        if (j >= nslots) break;
        const uint32_t key = key_at(j);
        if (key) atomicAdd(hmine + ((km - key) >> sh), mass_q(bf16key_to_float(key), M, c));
      }
      __syncthreads();
      unsigned long long q = 0;
#pragma unroll
      for (uint32_t h = 0; h < kHists; ++h) q += hq[h * kBins + tid];
      const uint32_t Jc = scan_bins(q, target_q, 0ull, red_u64, &s_tau, above);
      J = kNotFound;
      if (Jc != kNotFound) {
        // refine inside coarse bin Jc: keys top - i, i in [0, 2^sh)
        for (uint32_t i = tid; i < kHists * kBins; i += kThreads) hq[i] = 0ull;
        if (tid == 0) s_tau = kNotFound;
        __syncthreads();
        const uint32_t top = km - (Jc << sh);
#pragma unroll
        for (uint32_t j = 0; j < kSlots; ++j) {
          if (j >= nslots) break;
          const uint32_t key = key_at(j);
          if (key && key <= top && top - key < (1u << sh))
            atomicAdd(hmine + (top - key), mass_q(bf16key_to_float(key), M, c));
        }
        __syncthreads();
        unsigned long long q2 = 0;
#pragma unroll
        for (uint32_t h = 0; h < kHists; ++h) q2 += hq[h * kBins + tid];
        unsigned long long above2;
        const uint32_t j2 = scan_bins(q2, target_q, above, red_u64, &s_tau, above2);
        if (j2 != kNotFound) J = top - j2;
      }
    }
    const uint32_t tau = J;  // a 16-bit key
    general = tau == kNotFound || tau < kthr;
    if (!general) {
      // ---- nucleus entries packed into shared memory, then Gumbel-max over them
      uint32_t* nid = reinterpret_cast<uint32_t*>(ring + kHistBytes);
      uint16_t* nkey = reinterpret_cast<uint16_t*>(nid + kNucCap);
      if (tid == 0) s_count = 0;
      __syncthreads();
      unsigned long long best = 0ull;
      // ids of this thread's nucleus entries, kBatchIds slots at a time with
      // the loads in flight together
#pragma unroll
      for (uint32_t j0 = 0; j0 < kSlots; j0 += kBatchIds) {
        if (j0 >= nslots) break;
        uint32_t idb[kBatchIds];
#pragma unroll
        for (uint32_t u = 0; u < kBatchIds; ++u) {
          idb[u] = 0;
          if (key_at(j0 + u) >= tau) idb[u] = gid_row[tid + kThreads * (j0 + u)];  // tau > 0: empty slots stay out
        }
#pragma unroll
        for (uint32_t u = 0; u < kBatchIds; ++u) {
          const uint32_t key = key_at(j0 + u);
          const bool in = key >= tau;
          const unsigned bal = __ballot_sync(0xFFFFFFFFu, in);
          if (!bal) continue;
          uint32_t wb = 0;
          if (lane == 0) wb = atomicAdd(&s_count, __popc(bal));
          const uint32_t pos = __shfl_sync(0xFFFFFFFFu, wb, 0) + __popc(bal & ((1u << lane) - 1u));
          if (in) {
            const uint32_t id = idb[u];
            if (pos < kNucCap) {
              nid[pos] = id;
              nkey[pos] = uint16_t(key);
            } else {
              const uint4 blk = philox4x32_10(make_uint4(id >> 2, b, step, 0u), k0, k1);
              const float score = __fdiv_rn(bf16key_to_float(key), temp) + gumbel_from_word(philox_word(blk, id & 3u));
              best = max(best, pack_best(score, id));
            }
          }
        }
      }
      __syncthreads();
      const uint32_t nn = min(s_count, kNucCap);
      for (uint32_t j = tid; j < nn; j += kThreads) {
        const uint32_t id = nid[j];
        const uint4 blk = philox4x32_10(make_uint4(id >> 2, b, step, 0u), k0, k1);
        const float score = __fdiv_rn(bf16key_to_float(nkey[j]), temp) + gumbel_from_word(philox_word(blk, id & 3u));
        best = max(best, pack_best(score, id));
      }
      best = block_reduce(best, MaxOp(), 0ull, red_u64);
      tok = best ? best_id(best) : CG_NO_TOKEN;
    }
  }
  if (general) {
    __syncthreads();
    float M2;
    double S2;
    tok = general_row<true, true, kTopP>(row, V, smask, reinterpret_cast<uint32_t*>(ring), temp, top_p, b, k0, k1,
                                         step, M2, S2);
  }
  if (tid == 0) {
    out_tok[b] = tok;
    if (STEP == 2) {
      sa.out_flags[b] = pda_accept_row(sa.pda, sa.pda, sa.t, sa.pda_cfg + size_t(b) * sa.pda.stride, b, tok, s_f,
                                       sa.counts, sa.max_tokens);
    } else if (STEP == 1) {
      StateWindow w;
      if (s_wrows) {
        if (mbar_wait(&mbar_win, 0)) {
          w.next = win + s_wdelta;
          w.flags = wflags;
          w.lo = s_wlo;
          w.rows = s_wrows;
        } else {
          record_error(status, CG_DEV_TIMEOUT);
        }
      }
      accept_row(sa.t, b, s_g, s_s, tok, s_f, sa.counts, sa.max_tokens, sa.out_states, sa.out_flags,
                 s_g < sa.t.n_g ? scols : nullptr, w);
    }
  }
  if (STEP != 0 && sa.bitmask_out) {
    uint32_t* out = sa.bitmask_out + size_t(b) * W;
    for (uint32_t i = tid; i < W; i += kThreads) out[i] = smask[i];
  }
  if (probs || inplace) write_outputs<true, kTopP>(row, V, smask, tok, M, S, temp, probs, inplace, b);
}

// ============================================================================
// Greedy and full-softmax rows (bf16): the same bulk-copy ring, one CTA per
// row; the consumers keep the best (value, id) of their groups.  Greedy: the
// largest allowed logit, lowest id among equal ones.  Full: Gumbel-max over
// every allowed logit, z_t + g_t with z = x / temp and g from the row's
// Philox stream (two 4-word blocks per 8-logit group); fully masked groups
// draw nothing.  With probabilities requested, the full mode also sums
// exp2((x - m) c) for S.
// ============================================================================
template <int MODE, bool WANT_S>
__global__ void __launch_bounds__(kThreads, 2)
    stream_pick_kernel(void* logits, uint32_t V, uint32_t W, const uint32_t* __restrict__ bitmask, float temp,
                       uint32_t k0, uint32_t k1, uint32_t step, uint32_t* __restrict__ out_tok,
                       float* __restrict__ probs, int inplace, uint32_t* status) {
  extern __shared__ __align__(128) unsigned char dsm[];
  unsigned char* ring = dsm;                                  // kStages slots
  uint4* lut = reinterpret_cast<uint4*>(dsm + kRing);         // [256]
  uint32_t* smask = reinterpret_cast<uint32_t*>(lut + 256);   // [W]
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages];
  __shared__ float red_f[33];
  __shared__ unsigned long long red_u64[33];
  __shared__ uint32_t s_flag;

  griddep_launch_dependents();
  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, b = blockIdx.x;
  char* row = reinterpret_cast<char*>(logits) + size_t(b) * V * 2;
  const uint32_t nchunks = (V + kChunkElems - 1) / kChunkElems;
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, kConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_flag = 0;
  }
  for (uint32_t i = tid; i < 256; i += kThreads) lut[i] = pair_mask_entry(i);
  __syncthreads();
  griddep_wait();  // the bitmask comes from fill_bitmask
  const uint32_t* mrow = bitmask + size_t(b) * W;
  for (uint32_t i = tid; i < W; i += kThreads) smask[i] = mrow[i];
  __syncthreads();

  const float c = (MODE == kGreedy) ? 0.f : 1.4426950408889634f / temp;
  const uint8_t* smask8 = reinterpret_cast<const uint8_t*>(smask);
  unsigned long long best = 0ull;  // packed (value or score, id); 0 = none
  float bestv = -INFINITY;         // greedy: this thread's best value
  float lm = -INFINITY;            // this thread's largest allowed logit
  float mt = kNoRef;               // reference of this thread's sums (WANT_S)
  float2 acc[kAcc / 2];
#pragma unroll
  for (int j = 0; j < kAcc / 2; ++j) acc[j] = make_float2(0.f, 0.f);

  if (warp == kConsumerWarps) {
    if (lane == 0) {
      bool ok = true;
      for (uint32_t k = 0; k < nchunks; ++k) {
        if (k >= uint32_t(kStages) && !mbar_wait(empty + k % kStages, ((k / kStages) - 1) & 1u)) {
          ok = false;
          break;
        }
        issue_chunk(ring, full, row, V, k);
      }
      if (!ok) atomicOr(&s_flag, 1u);
    }
  } else {
    for (uint32_t k = 0; k < nchunks; ++k) {
      const uint32_t slot = k % kStages;
      if (!mbar_wait(full + slot, (k / kStages) & 1u)) {
        atomicOr(&s_flag, 1u);
        break;
      }
      const uint4* r4 = reinterpret_cast<const uint4*>(ring + size_t(slot) * kChunkBytes);
      const uint32_t gbase = k * kGroupsPerChunk;
      const uint32_t ngroups = min(kGroupsPerChunk, V / 8 - gbase);
      uint4 v[2];
      uint32_t mb[2];
#pragma unroll
      for (uint32_t g = 0; g < 2; ++g) {
        const uint32_t gi = tid + kConsumers * g;
        v[g] = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
        mb[g] = 0;
        if (gi < ngroups) {
          mb[g] = smask8[gbase + gi];
          v[g] = apply_mask(r4[gi], lut[mb[g]]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + slot);  // the slot's data are in registers
#pragma unroll
      for (uint32_t g = 0; g < 2; ++g) {
        const uint32_t t0 = (gbase + tid + kConsumers * g) * 8;  // id of the group's first logit
        const float gm = group_max(v[g]);
        lm = fmaxf(lm, gm);
        if (MODE == kGreedy) {
          if (gm > bestv) {  // strictly: this thread sees ids in increasing order
            uint32_t e = 0;
            while (e < 7 && bf16_bits_to_float(group_bits(v[g], e)) != gm) ++e;
            best = pack_best(gm, t0 + e);
            bestv = gm;
          }
        } else if (mb[g]) {
          const uint4 p0 = philox4x32_10(make_uint4(t0 >> 2, b, step, 0u), k0, k1);
          const uint4 p1 = philox4x32_10(make_uint4((t0 >> 2) + 1u, b, step, 0u), k0, k1);
#pragma unroll
          for (uint32_t e = 0; e < 8; ++e) {
            if ((mb[g] >> e) & 1u) {
              const float x = bf16_bits_to_float(group_bits(v[g], e));
              const uint32_t w = philox_word(e < 4 ? p0 : p1, e & 3u);
              best = max(best, pack_best(__fdiv_rn(x, temp) + gumbel_from_word(w), t0 + e));
            }
          }
        }
      }
      if (WANT_S) {
        const float gm = fmaxf(group_max(v[0]), group_max(v[1]));
        if (gm > mt) {
          const float r = ex2((mt - gm) * c);
#pragma unroll
          for (int j = 0; j < kAcc / 2; ++j) acc[j] = __fmul2_rn(acc[j], make_float2(r, r));
          mt = gm;
        }
        const float mc = mt * c;
        add_exps(acc, v[0], make_float2(c, c), make_float2(-mc, -mc));
        add_exps(acc, v[1], make_float2(c, c), make_float2(-mc, -mc));
      }
    }
  }
  __syncthreads();
  if ((s_flag & 1u) && tid == 0) {
    for (uint32_t sl = 0; sl < uint32_t(kStages) && sl < nchunks; ++sl) {
      const uint32_t issued = (nchunks - sl + kStages - 1) / kStages;
      mbar_wait(full + sl, (issued - 1) & 1u);
    }
  }
  best = block_reduce(best, MaxOp(), 0ull, red_u64);
  const float M = block_reduce(lm, MaxOp(), -INFINITY, red_f);
  double S = 0.0;
  if (WANT_S) {
    float part = 0.f;
    if (M > -INFINITY) {
      float a = 0.f;
#pragma unroll
      for (int jj = 0; jj < kAcc / 2; ++jj) a = (a + acc[jj].x) + acc[jj].y;
      if (a > 0.f) part = a * ex2((mt - M) * c);
    }
    S = double(block_reduce(part, SumOp(), 0.f, red_f));
  }
  uint32_t tok = best ? best_id(best) : CG_NO_TOKEN;
  if (s_flag & 1u) {
    tok = CG_NO_TOKEN;
    if (tid == 0) record_error(status, CG_DEV_TIMEOUT);
  }
  if (tid == 0) out_tok[b] = tok;
  if (probs || inplace) write_outputs<true, MODE>(row, V, smask, tok, M, S, temp, probs, inplace, b);
}

size_t pick_smem(uint32_t W) { return size_t(kRing) + 4096 + size_t((W + 3) & ~3u) * 4; }

// Dynamic shared memory of the top-p kernel; the fused step adds win_bytes for
// the accept's table window.
size_t stream_smem(uint32_t W, uint32_t win_bytes = 0) {
  return size_t(kRing) + 4096 + size_t(kConsumerWarps) * kStage * 18 + size_t((W + 3) & ~3u) * 4 + 512 * 2 +
         kWinRowsMax + win_bytes;
}

// Dynamic shared memory per CTA that still lets two CTAs share an SM: 228 KB
// per SM, less 1 KB reserved and up to 2 KB of static shared memory per CTA.
constexpr size_t kTwoCtaSmem = 111 * 1024;

}  // namespace fast

// Raises a kernel's dynamic shared memory limit once per device (the setting
// is per function and device; repeating it costs a driver call per launch).
cudaError_t allow_smem(const void* kernel, size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, size_t> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  size_t& have = done[{kernel, dev}];
  if (bytes <= have) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
  if (e == cudaSuccess) have = bytes;
  return e;
}

template <bool BF16, bool VEC, int MODE>
cudaError_t launch_variant(void* logits, uint32_t B, uint32_t V, uint32_t W, const uint32_t* bitmask,
                           float temp, float top_p, uint64_t seed, uint32_t step, uint32_t* out_tok, float* probs,
                           int inplace, cudaStream_t stream) {
  const size_t smem = size_t(W) * 4 + ((MODE == kTopP && BF16) ? size_t(kWindow) * 4 : 0);
  auto* k = sample_kernel<BF16, VEC, MODE>;
  cudaError_t e = allow_smem(reinterpret_cast<const void*>(k), smem);
  if (e != cudaSuccess) return e;
  return launch_dependent(k, dim3(B), dim3(kSampleThreads), smem, stream, logits, V, W, bitmask, temp, top_p,
                          uint32_t(seed), uint32_t(seed >> 32), step, out_tok, probs, inplace);
}

template <bool BF16, bool VEC>
cudaError_t launch_mode(int mode, void* logits, uint32_t B, uint32_t V, uint32_t W, const uint32_t* bitmask,
                        float temp, float top_p, uint64_t seed, uint32_t step, uint32_t* out_tok, float* probs,
                        int inplace, cudaStream_t stream) {
  if (mode == kGreedy)
    return launch_variant<BF16, VEC, kGreedy>(logits, B, V, W, bitmask, temp, top_p, seed, step, out_tok, probs,
                                              inplace, stream);
  if (mode == kTopP)
    return launch_variant<BF16, VEC, kTopP>(logits, B, V, W, bitmask, temp, top_p, seed, step, out_tok, probs,
                                            inplace, stream);
  return launch_variant<BF16, VEC, kFull>(logits, B, V, W, bitmask, temp, top_p, seed, step, out_tok, probs,
                                          inplace, stream);
}

// Device scratch the sampling kernels need for B rows of V logits: the top-p
// path's per-row candidate lists (u32 ids, then u16 keys).
size_t sample_scratch_bytes(uint32_t B, uint32_t V) {
  (void)V;
  return size_t(B) * fast::kCandPerRow * 6;
}

cudaError_t launch_mask_and_sample(void* logits, int dtype, uint32_t B, uint32_t V, uint32_t W,
                                   const uint32_t* bitmask, float temp, float top_p, uint64_t seed, uint32_t step,
                                   uint32_t* out_tok, float* probs, int inplace, void* scratch, uint32_t* status,
                                   cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  const int mode = (temp == 0.f) ? kGreedy : (top_p >= 1.f ? kFull : kTopP);
  const bool bf16 = dtype == CG_BF16;
  const uint32_t ch = bf16 ? 8u : 4u;
  const bool vec = (V % ch == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15u) == 0);
  const size_t s1 = fast::stream_smem(W);
  if (bf16 && vec && mode == kTopP && s1 <= 112 * 1024) {
    cudaError_t e = allow_smem(reinterpret_cast<const void*>(fast::stream_topp_kernel<0>), s1);
    if (e != cudaSuccess) return e;
    uint32_t* cand_id = static_cast<uint32_t*>(scratch);
    uint16_t* cand_key = reinterpret_cast<uint16_t*>(cand_id + size_t(B) * fast::kCandPerRow);
    return launch_dependent(fast::stream_topp_kernel<0>, dim3(B), dim3(fast::kThreads), s1, stream, logits, V,
                            W, bitmask, temp, top_p, uint32_t(seed), uint32_t(seed >> 32), step, out_tok, probs,
                            inplace, cand_id, cand_key, fast::kCandPerRow, status, fast::StepArgs{});
  }
  if (bf16 && vec && mode != kTopP && fast::pick_smem(W) <= 112 * 1024) {
    const size_t sm = fast::pick_smem(W);
    auto k = mode == kGreedy ? fast::stream_pick_kernel<kGreedy, false>
                             : (probs ? fast::stream_pick_kernel<kFull, true> : fast::stream_pick_kernel<kFull, false>);
    cudaError_t e = allow_smem(reinterpret_cast<const void*>(k), sm);
    if (e != cudaSuccess) return e;
    return launch_dependent(k, dim3(B), dim3(fast::kThreads), sm, stream, logits, V, W, bitmask, temp,
                            uint32_t(seed), uint32_t(seed >> 32), step, out_tok, probs, inplace, status);
  }
  if (bf16)
    return vec ? launch_mode<true, true>(mode, logits, B, V, W, bitmask, temp, top_p, seed, step, out_tok, probs,
                                         inplace, stream)
               : launch_mode<true, false>(mode, logits, B, V, W, bitmask, temp, top_p, seed, step, out_tok, probs,
                                          inplace, stream);
  return vec ? launch_mode<false, true>(mode, logits, B, V, W, bitmask, temp, top_p, seed, step, out_tok, probs,
                                        inplace, stream)
             : launch_mode<false, false>(mode, logits, B, V, W, bitmask, temp, top_p, seed, step, out_tok, probs,
                                         inplace, stream);
}

// The fused step (fill + sample + accept) runs as one kernel when the sampling
// takes the top-p bf16 path; returns false (nothing launched) otherwise.
bool step_fusable(int dtype, uint32_t V, uint32_t W, float temp, float top_p, const void* logits) {
  return dtype == CG_BF16 && temp > 0.f && top_p < 1.f && V % 8 == 0 &&
         (reinterpret_cast<uintptr_t>(logits) & 15u) == 0 && fast::stream_smem(W) <= 112 * 1024;
}

cudaError_t launch_step(const Tables& t, const uint32_t* states, const uint16_t* gid, const int32_t* forced,
                        uint32_t B, void* logits, uint32_t V, float temp, float top_p, uint64_t seed, uint32_t step,
                        uint32_t* counts, uint32_t max_tokens, uint32_t* bitmask_out, uint32_t* out_tok,
                        uint32_t* out_states, uint8_t* out_flags, void* scratch, const DevGrammar* host_grammars,
                        bool cache_complete, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  const uint32_t W = t.W;
  const size_t base = fast::stream_smem(W);
  const uint32_t win_bytes =
      base + 1024 <= fast::kTwoCtaSmem
          ? uint32_t(std::min<size_t>(fast::kWinBytesMax, fast::kTwoCtaSmem - base) & ~size_t(15))
          : 0u;
  const size_t s1 = base + win_bytes;
  cudaError_t e = allow_smem(reinterpret_cast<const void*>(fast::stream_topp_kernel<1>), s1);
  if (e != cudaSuccess) return e;
  uint32_t* cand_id = static_cast<uint32_t*>(scratch);
  uint16_t* cand_key = reinterpret_cast<uint16_t*>(cand_id + size_t(B) * fast::kCandPerRow);
  fast::StepArgs sa{t, states, gid, forced, counts, max_tokens, out_states, out_flags, bitmask_out, {}, 0u, 0u, 0u};
  if (host_grammars && t.n_g <= fast::kParamGrammars) {
    for (uint32_t i = 0; i < t.n_g; ++i) sa.pg[i] = host_grammars[i];
    sa.n_pg = t.n_g;
  }
  sa.cache_complete = cache_complete ? 1u : 0u;
  sa.win_bytes = win_bytes;
  return launch_dependent(fast::stream_topp_kernel<1>, dim3(B), dim3(fast::kThreads), s1, stream, logits, V, W,
                          static_cast<const uint32_t*>(nullptr), temp, top_p, uint32_t(seed), uint32_t(seed >> 32),
                          step, out_tok, static_cast<float*>(nullptr), 0, cand_id, cand_key, fast::kCandPerRow,
                          t.status, sa);
}

// The fused step of pushdown rows (cg_pda_step): the row's mask from the
// (state, headroom) cache and its listed tokens, the masked top-p sampling of
// cg_mask_and_sample, and the accept into the row's configuration, in one
// kernel per row.
cudaError_t launch_pda_step(const Tables& t, const DevPda& pda, uint32_t* cfg, const int32_t* forced, uint32_t B,
                            void* logits, uint32_t V, float temp, float top_p, uint64_t seed, uint32_t step,
                            uint32_t* counts, uint32_t max_tokens, uint32_t* bitmask_out, uint32_t* out_tok,
                            uint8_t* out_flags, void* scratch, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  const uint32_t W = t.W;
  const size_t s1 = fast::stream_smem(W);
  cudaError_t e = allow_smem(reinterpret_cast<const void*>(fast::stream_topp_kernel<2>), s1);
  if (e != cudaSuccess) return e;
  uint32_t* cand_id = static_cast<uint32_t*>(scratch);
  uint16_t* cand_key = reinterpret_cast<uint16_t*>(cand_id + size_t(B) * fast::kCandPerRow);
  fast::StepArgs sa{t,  nullptr, nullptr, forced, counts, max_tokens, nullptr, out_flags, bitmask_out,
                    {}, 0u,      0u,      0u,     pda,    cfg};
  return launch_dependent(fast::stream_topp_kernel<2>, dim3(B), dim3(fast::kThreads), s1, stream, logits, V, W,
                          static_cast<const uint32_t*>(nullptr), temp, top_p, uint32_t(seed), uint32_t(seed >> 32),
                          step, out_tok, static_cast<float*>(nullptr), 0, cand_id, cand_key, fast::kCandPerRow,
                          t.status, sa);
}

}  // namespace cgk
