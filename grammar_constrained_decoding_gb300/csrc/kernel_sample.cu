// Mask-apply + temperature + softmax + top-p + sampling, one CTA per row
// ("Sampling runs after masking, so no sampling strategy can escape it",
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

#include "device.cuh"

namespace cgk {

constexpr int kSampleThreads = 512;
constexpr int kWindow = 4096;     // keys kept below the row maximum (bf16 path)
constexpr int kAcc = 8;           // independent partial sums per thread
constexpr uint32_t kNotFound = 0xFFFFFFFFu;

enum SampleMode { kGreedy = 0, kTopP = 1, kFull = 2 };

__device__ __forceinline__ float bf16_bits_to_float(uint32_t h) { return __uint_as_float(h << 16); }

// inverse of the 16-bit monotone bf16 key (fkey(x) >> 16)
__device__ __forceinline__ float bf16key_to_float(uint32_t k16) {
  const uint32_t h = (k16 & 0x8000u) ? (k16 & 0x7FFFu) : (~k16 & 0xFFFFu);
  return bf16_bits_to_float(h);
}

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
// Top-p kernel for bf16 rows (the path of the throughput metric).  Each logit
// is read from HBM once; the few groups that can hold nucleus candidates are
// read a second time from L2.
//
// One CTA of 512 threads per row.  Warp 15 fills a kStages-slot shared-memory
// ring with bulk asynchronous copies (cp.async.bulk, completing on "full"
// mbarriers; the copies carry an L2 evict_last hint so that the row stays in
// L2 for the second look).  Warps 0..14 take each chunk from the ring 16 logits
// per thread (two 8-logit groups): the bitmask is applied through a 256-entry
// table of pair masks indexed by the group's mask byte, the group maximum is
// taken with packed bf16 max, and exp2((x - m) c) is summed into 8 partial sums
// against a reference m that follows the block's running maximum (published
// per chunk with a warp max-reduction and a shared atomicMax).  A group whose
// maximum reaches the reference minus kMarginZ nats sets its bit in a per-row
// flag bitmap (one warp ballot per 32 groups).  The reference never exceeds the
// final maximum M, so every allowed logit within kMarginZ nats of M lies in a
// flagged group.
//
// After the stream: M and S = sum exp2((x - M) c) come from the block; the
// flagged groups are re-read (L2) and their allowed logits >= M - margin become
// the candidates; the nucleus threshold is the largest key whose upper
// set carries top_p * S (per-key counts of the candidates, or bisection), and
// Gumbel scores are drawn for the nucleus entries only.  Rows whose nucleus
// reaches below the margin, or whose lists overflow, run general_row instead.
// ============================================================================
namespace fast {

constexpr int kThreads = 512;
constexpr uint32_t kConsumerWarps = 15;
constexpr uint32_t kConsumers = kConsumerWarps * 32;            // 480
constexpr int kStages = 5;
constexpr uint32_t kChunkElems = kConsumers * 16;               // 7680 logits per slot
constexpr uint32_t kChunkBytes = kChunkElems * 2;               // 15 KiB
constexpr uint32_t kGroupsPerChunk = kChunkElems / 8;           // 960
constexpr uint32_t kWordsPerChunk = kGroupsPerChunk / 32;       // 30 flag words
constexpr uint32_t kRing = kStages * kChunkBytes;               // 75 KiB
// after the stream the ring holds the candidate list, then the key histograms
// (later the packed nucleus entries)
constexpr uint32_t kCap = 10000;                                // candidates (u32 id + u16 key)
constexpr uint32_t kBins = 512;                                 // keys per histogram
constexpr uint32_t kHists = 8;                                  // histogram copies
constexpr uint32_t kHistOff = (kCap * 6 + 127) / 128 * 128;
constexpr uint32_t kNucCap = kHists * kBins * 2;                // packed nucleus entries (u16)
static_assert(kHistOff + kHists * kBins * 4 <= kRing, "histograms must fit the ring");
constexpr int kBatch = 8;                                       // flagged groups loaded per round
constexpr float kMarginZ = 9.5f;                                // nats below the maximum kept as candidates
constexpr float kRefJump = 60.f;                                // logit/temp units a reference may lag
constexpr float kNoRef = -1e30f;                                // finite reference before any allowed logit
constexpr uint32_t kWaitLimit = 1u << 22;

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
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_addr(dst)),
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
// bounded wait on a phase; false when the limit ran out
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
// 2^x with the multi-function unit (relative error about 2^-22; results
// below 2^-126 flush to zero, far below any mass that matters here)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&a), y = *reinterpret_cast<__nv_bfloat162*>(&b);
  __nv_bfloat162 r = __hmax2(x, y);
  return *reinterpret_cast<uint32_t*>(&r);
}
// masked logits become -inf (bf16 0xFF80)
__device__ __forceinline__ uint4 apply_mask(uint4 v, uint4 pm) {
  v.x = (v.x & pm.x) | (~pm.x & 0xFF80FF80u);
  v.y = (v.y & pm.y) | (~pm.y & 0xFF80FF80u);
  v.z = (v.z & pm.z) | (~pm.z & 0xFF80FF80u);
  v.w = (v.w & pm.w) | (~pm.w & 0xFF80FF80u);
  return v;
}
__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float group_max(const uint4& v) {
  const uint32_t mx = bmax2(bmax2(v.x, v.y), bmax2(v.z, v.w));
  return fmaxf(lo_f(mx), hi_f(mx));
}
__device__ __forceinline__ void add_exps(float* acc, const uint4& v, float c, float mc) {
  acc[0] += ex2(fmaf(lo_f(v.x), c, -mc));
  acc[1] += ex2(fmaf(hi_f(v.x), c, -mc));
  acc[2] += ex2(fmaf(lo_f(v.y), c, -mc));
  acc[3] += ex2(fmaf(hi_f(v.y), c, -mc));
  acc[4] += ex2(fmaf(lo_f(v.z), c, -mc));
  acc[5] += ex2(fmaf(hi_f(v.z), c, -mc));
  acc[6] += ex2(fmaf(lo_f(v.w), c, -mc));
  acc[7] += ex2(fmaf(hi_f(v.w), c, -mc));
}

__device__ __forceinline__ void issue_chunk(unsigned char* ring, uint64_t* full, const char* row, uint32_t V,
                                            uint32_t k, uint64_t pol) {
  const uint32_t slot = k % kStages;
  const uint32_t bytes = min(kChunkElems, V - k * kChunkElems) * 2;
  mbar_expect_tx(full + slot, bytes);
  bulk_g2s(ring + size_t(slot) * kChunkBytes, row + size_t(k) * kChunkBytes, bytes, full + slot, pol);
}

__global__ void __launch_bounds__(kThreads, 2)
    stream_topp_kernel(void* logits, uint32_t V, uint32_t W, const uint32_t* __restrict__ bitmask, float temp,
                       float top_p, uint32_t k0, uint32_t k1, uint32_t step, uint32_t* __restrict__ out_tok,
                       float* __restrict__ probs, int inplace, uint32_t* status) {
  extern __shared__ __align__(128) unsigned char dsm[];
  unsigned char* ring = dsm;                                                // kStages slots
  uint4* lut = reinterpret_cast<uint4*>(dsm + kRing);                       // [256]
  uint32_t* smask = reinterpret_cast<uint32_t*>(lut + 256);                 // [W]
  const uint32_t nchunks = (V + kChunkElems - 1) / kChunkElems;
  const uint32_t nfw = nchunks * kWordsPerChunk;
  uint32_t* fbits = smask + ((W + 3) & ~3u);                                // [nfw] flag bitmap
  // after the stream
  uint32_t* cid = reinterpret_cast<uint32_t*>(ring);                        // [kCap]
  uint16_t* ckey = reinterpret_cast<uint16_t*>(ring + kCap * 4);            // [kCap]
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages];
  __shared__ float red_f[33];
  __shared__ double red_d[33];
  __shared__ unsigned long long red_u64[33];
  __shared__ uint32_t s_maxkey, s_flag, s_count, s_tau;

  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, b = blockIdx.x;
  char* row = reinterpret_cast<char*>(logits) + size_t(b) * V * 2;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, kConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_maxkey = fkey(-INFINITY);
    s_flag = 0;  // bit 0: a wait ran out
    s_count = 0;
  }
  for (uint32_t i = tid; i < 256; i += kThreads) {
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      w[q] = (((i >> (2 * q)) & 1u) ? 0x0000FFFFu : 0u) | (((i >> (2 * q + 1)) & 1u) ? 0xFFFF0000u : 0u);
    lut[i] = make_uint4(w[0], w[1], w[2], w[3]);
  }
  const uint32_t* mrow = bitmask + size_t(b) * W;
  for (uint32_t i = tid; i < W; i += kThreads) smask[i] = mrow[i];
  __syncthreads();

  const float c = 1.4426950408889634f / temp;
  const float margin = kMarginZ * temp;  // z = x / temp: kMarginZ nats are kMarginZ * temp logit units
  const uint8_t* smask8 = reinterpret_cast<const uint8_t*>(smask);
  float mt = kNoRef;  // this thread's reference (never above the row maximum)
  float acc[kAcc];
#pragma unroll
  for (int j = 0; j < kAcc; ++j) acc[j] = 0.f;

  if (warp == kConsumerWarps) {
    // ---- producer warp --------------------------------------------------------------
    if (lane == 0) {
      const uint64_t pol = l2_evict_last_policy();
      bool ok = true;
      for (uint32_t k = 0; k < nchunks; ++k) {
        if (k >= uint32_t(kStages) && !mbar_wait(empty + k % kStages, ((k / kStages) - 1) & 1u)) {
          ok = false;
          break;
        }
        issue_chunk(ring, full, row, V, k, pol);
      }
      if (!ok) atomicOr(&s_flag, 1u);
    }
  } else {
    // ---- consumers ----------------------------------------------------------------
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
    for (uint32_t k = 0; k < nchunks; ++k) {
      const uint32_t slot = k % kStages;
      // reference for this chunk: the block's running maximum
      const float mref = fkey_inv(*reinterpret_cast<volatile uint32_t*>(&s_maxkey));
      if (mref > mt) {
        const float r = ex2((mt - mref) * c);
#pragma unroll
        for (int j = 0; j < kAcc; ++j) acc[j] *= r;
        mt = mref;
      }
      const float thr = mt - margin;
      if (!mbar_wait(full + slot, (k / kStages) & 1u)) {
        atomicOr(&s_flag, 1u);
        break;
      }
      const uint4* r4 = reinterpret_cast<const uint4*>(ring + size_t(slot) * kChunkBytes);
      const uint32_t gbase = k * kGroupsPerChunk;  // row group index of the chunk's group 0
      const uint32_t gi0 = tid, gi1 = tid + kConsumers;
      const uint32_t ngroups = min(kGroupsPerChunk, V / 8 - gbase);
      uint4 v0 = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u), v1 = v0;
      if (gi0 < ngroups) v0 = apply_mask(r4[gi0], lut[smask8[gbase + gi0]]);
      if (gi1 < ngroups) v1 = apply_mask(r4[gi1], lut[smask8[gbase + gi1]]);
      const float g0 = group_max(v0), g1 = group_max(v1);
      const float gm = fmaxf(g0, g1);
      if (gm > mt + kRefJump * temp) {
        // far above the reference (or the first allowed logits): move this
        // thread's reference before the sums can overflow
        const float r = ex2((mt - gm) * c);
#pragma unroll
        for (int j = 0; j < kAcc; ++j) acc[j] *= r;
        mt = gm;
      }
      const float mc = mt * c;
      add_exps(acc, v0, c, mc);
      add_exps(acc, v1, c, mc);
      // chunk-local group of this lane = 480 g + tid = 32 * (15 g + warp) + lane
      const unsigned b0 = __ballot_sync(0xFFFFFFFFu, g0 >= thr);
      const unsigned b1 = __ballot_sync(0xFFFFFFFFu, g1 >= thr);
      const uint32_t wk = __reduce_max_sync(0xFFFFFFFFu, fkey(gm));
      __syncwarp();
      if (lane == 0) {
        fbits[k * kWordsPerChunk + warp] = b0;
        fbits[k * kWordsPerChunk + kConsumerWarps + warp] = b1;
        atomicMax(&s_maxkey, wk);
        mbar_arrive(empty + slot);
      }
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
  }
  const float M = fkey_inv(s_maxkey);  // -inf when no logit is allowed
  // S: per-thread partial sums in float (each already a float sum), warp sums
  // in float, the 16 warp sums in double
  {
    float part = 0.f;
    if (M > -INFINITY) {
      float a = 0.f;
#pragma unroll
      for (int jj = 0; jj < kAcc; ++jj) a += acc[jj];
      if (a > 0.f) part = a * ex2((mt - M) * c);
    }
    part = warp_reduce(part, SumOp());
    if (lane == 0) red_f[warp] = part;
  }
  __syncthreads();
  double S = 0.0;
  for (uint32_t wi = 0; wi < kThreads / 32; ++wi) S += double(red_f[wi]);
  uint32_t tok = CG_NO_TOKEN;
  bool general = false;
  if (s_flag & 1u) {
    if (tid == 0) record_error(status, CG_DEV_TIMEOUT);
  } else if (!(M > -1e29f && M < 1e29f)) {
    general = M > -INFINITY;  // huge or infinite logits: the plain path copes with them
  } else {
    // ---- candidates: allowed logits >= M - margin, read again (from L2) in the
    // flagged groups.  Thread t takes flag words t, t + 512, ...; per round it
    // loads up to kBatch of its flagged groups, then the warp reserves room for
    // all their hits with one shared atomic.
    const float thrF = M - margin;
    const uint4* g4 = reinterpret_cast<const uint4*>(row);
    for (uint32_t w0 = 0; w0 < nfw; w0 += kThreads) {
      const uint32_t w = w0 + tid;
      uint32_t bits = w < nfw ? fbits[w] : 0u;
      while (__any_sync(0xFFFFFFFFu, bits != 0u)) {
        uint4 v[kBatch];
        uint32_t gsel[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          gsel[u] = kNotFound;
          if (bits) {
            gsel[u] = w * 32 + (__ffs(bits) - 1);
            bits &= bits - 1;
            v[u] = ld_stream(g4 + gsel[u]);
          }
        }
        uint32_t hits[kBatch];
        uint32_t nh = 0;
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          hits[u] = 0;
          if (gsel[u] != kNotFound) {
            v[u] = apply_mask(v[u], lut[smask8[gsel[u]]]);
            const uint32_t wv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              hits[u] |= uint32_t(lo_f(wv[q]) >= thrF) << (2 * q);
              hits[u] |= uint32_t(hi_f(wv[q]) >= thrF) << (2 * q + 1);
            }
            nh += __popc(hits[u]);
          }
        }
        uint32_t inc = nh;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
          if (lane >= uint32_t(o)) inc += y;
        }
        uint32_t wb = 0;
        if (lane == 31 && inc) wb = atomicAdd(&s_count, inc);
        uint32_t pos = __shfl_sync(0xFFFFFFFFu, wb, 31) + inc - nh;
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          uint32_t h = hits[u];
          while (h) {
            const uint32_t e = __ffs(h) - 1;
            h &= h - 1;
            if (pos < kCap) {
              const uint32_t wd = e < 4 ? (e < 2 ? v[u].x : v[u].y) : (e < 6 ? v[u].z : v[u].w);
              cid[pos] = gsel[u] * 8 + e;
              ckey[pos] = uint16_t(fkey((e & 1u) ? hi_f(wd) : lo_f(wd)) >> 16);
            }
            ++pos;
          }
        }
      }
    }
    __syncthreads();
    const uint32_t n_all = s_count;
    const uint32_t n = min(n_all, kCap);
    const double target = double(top_p) * S;
    uint32_t kthr = fkey(thrF) >> 16;  // every allowed logit with key >= kthr is a candidate
    if (bf16key_to_float(kthr) < thrF) ++kthr;
    const uint32_t km = fkey(M) >> 16;
    const double fx = 1099511627776.0;  // masses in 2^-40 units: exact sums, no rounding order
    const unsigned long long target_q = (unsigned long long)(target * fx);
    uint32_t tau = kNotFound;
    uint32_t* hb = reinterpret_cast<uint32_t*>(ring + kHistOff);
    if (n_all > kCap) {
      general = true;
    } else if (km - kthr < kBins) {
      // per-key counts (kHists histograms, warp w counts into histogram
      // w % kHists), mass from the top (bin j is key km - j), block-wide prefix
      // sum, first bin where the upper set reaches the target
      for (uint32_t i = tid; i < kHists * kBins; i += kThreads) hb[i] = 0u;
      __syncthreads();
      uint32_t* mine = hb + (warp % kHists) * kBins;
      for (uint32_t i = tid; i < n; i += kThreads) atomicAdd(mine + (km - ckey[i]), 1u);
      __syncthreads();
      const uint32_t L = km - kthr + 1;
      unsigned long long q = 0;
      if (tid < L) {
        uint32_t cnt = 0;
#pragma unroll
        for (uint32_t hw = 0; hw < kHists; ++hw) cnt += hb[hw * kBins + tid];
        if (cnt) q = (unsigned long long)(double(cnt) * double(ex2((bf16key_to_float(km - tid) - M) * c)) * fx);
      }
      unsigned long long qi = q;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, qi, o);
        if (lane >= uint32_t(o)) qi += y;
      }
      if (lane == 31) red_u64[warp] = qi;
      if (tid == 0) s_tau = kNotFound;
      __syncthreads();
      unsigned long long before = 0;
      for (uint32_t wi = 0; wi < warp; ++wi) before += red_u64[wi];
      if (tid < L && before + qi >= target_q) atomicMin(&s_tau, tid);
      __syncthreads();
      tau = s_tau == kNotFound ? kNotFound : km - s_tau;
      general = tau == kNotFound;
    } else {
      // bisection over the list: largest key whose upper set carries >= target
      auto mass_at = [&](uint32_t kappa) {
        unsigned long long p = 0;
        for (uint32_t i = tid; i < n; i += kThreads) {
          const uint32_t key = ckey[i];
          if (key >= kappa) p += (unsigned long long)(double(ex2((bf16key_to_float(key) - M) * c)) * fx);
        }
        return block_reduce(p, SumOp(), 0ull, red_u64);
      };
      if (mass_at(kthr) < target_q) {
        general = true;
      } else {
        uint32_t lo = kthr, hi = km;
        while (lo < hi) {
          const uint32_t mid = lo + (hi - lo + 1) / 2;
          if (mass_at(mid) >= target_q) lo = mid; else hi = mid - 1;
        }
        tau = lo;
      }
    }
    if (!general) {
      // nucleus entries (candidate indices) packed densely, so that the Philox
      // draws spread over all threads; entries past kNucCap are scored in place
      uint16_t* nuc = reinterpret_cast<uint16_t*>(ring + kHistOff);
      if (tid == 0) s_count = 0;
      __syncthreads();
      unsigned long long best = 0ull;
      for (uint32_t i0 = 0; i0 < n; i0 += kThreads) {
        const uint32_t i = i0 + tid;
        const bool in = i < n && ckey[i] >= tau;
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, in);
        uint32_t wb = 0;
        if (lane == 0 && bal) wb = atomicAdd(&s_count, __popc(bal));
        const uint32_t pos = __shfl_sync(0xFFFFFFFFu, wb, 0) + __popc(bal & ((1u << lane) - 1u));
        if (in) {
          if (pos < kNucCap) {
            nuc[pos] = uint16_t(i);
          } else {
            const uint32_t id = cid[i];
            const uint4 blk = philox4x32_10(make_uint4(id >> 2, b, step, 0u), k0, k1);
            const float score = __fdiv_rn(bf16key_to_float(ckey[i]), temp) + gumbel_from_word(philox_word(blk, id & 3u));
            best = max(best, pack_best(score, id));
          }
        }
      }
      __syncthreads();
      const uint32_t nn = min(s_count, kNucCap);
      for (uint32_t j = tid; j < nn; j += kThreads) {
        const uint32_t i = nuc[j];
        const uint32_t id = cid[i];
        const uint4 blk = philox4x32_10(make_uint4(id >> 2, b, step, 0u), k0, k1);
        const float score = __fdiv_rn(bf16key_to_float(ckey[i]), temp) + gumbel_from_word(philox_word(blk, id & 3u));
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
  if (tid == 0) out_tok[b] = tok;
  if (probs || inplace) write_outputs<true, kTopP>(row, V, smask, tok, M, S, temp, probs, inplace, b);
}

size_t stream_smem(uint32_t V, uint32_t W) {
  const uint32_t nchunks = (V + kChunkElems - 1) / kChunkElems;
  return size_t(kRing) + 4096 + size_t((W + 3) & ~3u) * 4 + size_t(nchunks) * kWordsPerChunk * 4;
}

}  // namespace fast

template <bool BF16, bool VEC, int MODE>
cudaError_t launch_variant(void* logits, uint32_t B, uint32_t V, uint32_t W, const uint32_t* bitmask,
                           float temp, float top_p, uint64_t seed, uint32_t step, uint32_t* out_tok, float* probs,
                           int inplace, cudaStream_t stream) {
  const size_t smem = size_t(W) * 4 + ((MODE == kTopP && BF16) ? size_t(kWindow) * 4 : 0);
  auto* k = sample_kernel<BF16, VEC, MODE>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  k<<<B, kSampleThreads, smem, stream>>>(logits, V, W, bitmask, temp, top_p, uint32_t(seed), uint32_t(seed >> 32),
                                          step, out_tok, probs, inplace);
  return cudaGetLastError();
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

cudaError_t launch_mask_and_sample(void* logits, int dtype, uint32_t B, uint32_t V, uint32_t W,
                                   const uint32_t* bitmask, float temp, float top_p, uint64_t seed, uint32_t step,
                                   uint32_t* out_tok, float* probs, int inplace, uint32_t* status,
                                   cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  const int mode = (temp == 0.f) ? kGreedy : (top_p >= 1.f ? kFull : kTopP);
  const bool bf16 = dtype == CG_BF16;
  const uint32_t ch = bf16 ? 8u : 4u;
  const bool vec = (V % ch == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15u) == 0);
  const size_t s1 = fast::stream_smem(V, W);
  if (bf16 && vec && mode == kTopP && s1 <= 112 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(fast::stream_topp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(s1));
    if (e != cudaSuccess) return e;
    fast::stream_topp_kernel<<<B, fast::kThreads, s1, stream>>>(logits, V, W, bitmask, temp, top_p, uint32_t(seed),
                                                               uint32_t(seed >> 32), step, out_tok, probs, inplace,
                                                               status);
    return cudaGetLastError();
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

}  // namespace cgk
