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

template <bool BF16, bool VEC, int MODE>
__global__ void __launch_bounds__(kSampleThreads) sample_kernel(void* logits, uint32_t V,
                                                                 uint32_t W, const uint32_t* __restrict__ bitmask,
                                                                 float temp, float top_p, uint32_t k0, uint32_t k1,
                                                                 uint32_t step, uint32_t* __restrict__ out_tok,
                                                                 float* __restrict__ probs, int inplace) {
  extern __shared__ uint32_t smem[];
  uint32_t* smask = smem;             // [W]
  uint32_t* cnt = smem + W;           // [kWindow] (top-p, bf16)
  __shared__ unsigned long long red_u64[33];
  __shared__ float red_f[33];
  __shared__ double red_d[33];
  __shared__ uint32_t s_tau;

  const uint32_t b = blockIdx.x;
  const size_t esz = BF16 ? 2 : 4;
  char* row = reinterpret_cast<char*>(logits) + size_t(b) * V * esz;
  const uint32_t* mrow = bitmask + size_t(b) * W;
  for (uint32_t i = threadIdx.x; i < W; i += blockDim.x) smask[i] = mrow[i];
  __syncthreads();

  // ---- pass A --------------------------------------------------------------
  const float c = (MODE == kGreedy) ? 0.f : 1.4426950408889634f / temp;
  unsigned long long best = 0ull;  // packed (value, id); 0 = none
  float m = -INFINITY;
  float acc[kAcc];
#pragma unroll
  for (int j = 0; j < kAcc; ++j) acc[j] = 0.f;
  Gumbel gum{b, step, k0, k1, temp};
  auto pass_a = [&](uint32_t t, float x) {
    if (MODE == kGreedy) {
      best = max(best, pack_best(x, t));
      return;
    }
    if (x > m) {
      const float r = exp2f((m - x) * c);
#pragma unroll
      for (int j = 0; j < kAcc; ++j) acc[j] *= r;
      m = x;
    }
    acc[t & (kAcc - 1)] += exp2f((x - m) * c);
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
    if (m > -INFINITY) {
      const float r = exp2f((m - M) * c);
#pragma unroll
      for (int j = 0; j < kAcc; ++j) part += double(acc[j]) * double(r);
    }
    S = block_reduce(part, SumOp(), 0.0, red_d);
    if (MODE == kFull) best = block_reduce(best, MaxOp(), 0ull, red_u64);
  }

  // ---- top-p threshold and nucleus sample ------------------------------------
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
        for (uint32_t base = 0; base < uint32_t(kWindow) && base <= km - lo && found == kNotFound; base += 32) {
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

  const uint32_t tok = best ? best_id(best) : CG_NO_TOKEN;
  if (threadIdx.x == 0) out_tok[b] = tok;

  // ---- optional outputs -------------------------------------------------------
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
    for (uint32_t t = threadIdx.x; t < V; t += blockDim.x) {
      if ((smask[t >> 5] >> (t & 31)) & 1u) continue;
      if (BF16) reinterpret_cast<uint16_t*>(row)[t] = 0xFF80u;
      else reinterpret_cast<float*>(row)[t] = -INFINITY;
    }
  }
}

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
                                   uint32_t* out_tok, float* probs, int inplace, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  const int mode = (temp == 0.f) ? kGreedy : (top_p >= 1.f ? kFull : kTopP);
  const bool bf16 = dtype == CG_BF16;
  const uint32_t ch = bf16 ? 8u : 4u;
  const bool vec = (V % ch == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15u) == 0);
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
