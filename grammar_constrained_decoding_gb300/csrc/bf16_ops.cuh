// Arithmetic on packed bf16 logits shared by the streaming sampling kernels:
// unpacking, masking through a pair-mask table, packed maxima, exponential
// sums and the 16-bit monotone key of a bf16 value.
#pragma once

#include <cuda_bf16.h>

#include "device.cuh"

namespace cgk {

__device__ __forceinline__ float bf16_bits_to_float(uint32_t h) { return __uint_as_float(h << 16); }

// inverse of the 16-bit monotone bf16 key (fkey(x) >> 16)
__device__ __forceinline__ float bf16key_to_float(uint32_t k16) {
  const uint32_t h = (k16 & 0x8000u) ? (k16 & 0x7FFFu) : (~k16 & 0xFFFFu);
  return bf16_bits_to_float(h);
}

// monotone 16-bit key of a bf16 (the high half of fkey of its float)
__device__ __forceinline__ uint16_t bf16_key(uint32_t h) {
  if (h == 0x8000u) h = 0u;
  return uint16_t((h & 0x8000u) ? (~h & 0xFFFFu) : (h | 0x8000u));
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

// masked logits become -inf (bf16 0xFF80); pm holds 0xFFFF for every allowed half
__device__ __forceinline__ uint4 apply_mask(uint4 v, uint4 pm) {
  v.x = (v.x & pm.x) | (~pm.x & 0xFF80FF80u);
  v.y = (v.y & pm.y) | (~pm.y & 0xFF80FF80u);
  v.z = (v.z & pm.z) | (~pm.z & 0xFF80FF80u);
  v.w = (v.w & pm.w) | (~pm.w & 0xFF80FF80u);
  return v;
}

// the 256-entry table of pair masks, indexed by an 8-logit group's mask byte
__device__ __forceinline__ uint4 pair_mask_entry(uint32_t i) {
  uint32_t w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q)
    w[q] = (((i >> (2 * q)) & 1u) ? 0x0000FFFFu : 0u) | (((i >> (2 * q + 1)) & 1u) ? 0xFFFF0000u : 0u);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// The same four pair masks computed from the byte itself: multiplying its low
// (high) nibble by 0x10204080 (0x01020408) puts mask bit i of the nibble on
// the top bit of byte i of the product (the sixteen shifted copies land on
// distinct bits, so nothing carries), and prmt's sign mode (selector nibble
// 8 + byte) spreads each top bit over a byte.
__device__ __forceinline__ uint32_t prmt_sign(uint32_t x, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(r) : "r"(x), "r"(sel));
  return r;
}
__device__ __forceinline__ uint4 pair_mask_of(uint32_t mb) {
  const uint32_t r0 = (mb & 0x0Fu) * 0x10204080u, r1 = (mb & 0xF0u) * 0x01020408u;
  return make_uint4(prmt_sign(r0, 0x9988u), prmt_sign(r0, 0xBBAAu), prmt_sign(r1, 0x9988u), prmt_sign(r1, 0xBBAAu));
}

__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// packed (bf16x2) maximum of an 8-logit group
__device__ __forceinline__ uint32_t group_pmax(const uint4& v) { return bmax2(bmax2(v.x, v.y), bmax2(v.z, v.w)); }
__device__ __forceinline__ float pmax_f(uint32_t p) { return fmaxf(lo_f(p), hi_f(p)); }
__device__ __forceinline__ float group_max(const uint4& v) { return pmax_f(group_pmax(v)); }

// acc[j] += exp2(x_j c - mc) for the group's logits, sums j and j + 1 paired in
// one float2 (the packed fp32 multiply-add and add round each lane as the
// scalar instructions do, so the sums are those of scalar code)
__device__ __forceinline__ float2 ex2_pair(float2 z) { return make_float2(ex2(z.x), ex2(z.y)); }
__device__ __forceinline__ void add_exps(float2* acc, const uint4& v, float2 c2, float2 nmc2) {
  acc[0] = __fadd2_rn(acc[0], ex2_pair(__ffma2_rn(make_float2(lo_f(v.x), hi_f(v.x)), c2, nmc2)));
  acc[1] = __fadd2_rn(acc[1], ex2_pair(__ffma2_rn(make_float2(lo_f(v.y), hi_f(v.y)), c2, nmc2)));
  acc[2] = __fadd2_rn(acc[2], ex2_pair(__ffma2_rn(make_float2(lo_f(v.z), hi_f(v.z)), c2, nmc2)));
  acc[3] = __fadd2_rn(acc[3], ex2_pair(__ffma2_rn(make_float2(lo_f(v.w), hi_f(v.w)), c2, nmc2)));
}

// logit e (0..7) of an 8-logit group
__device__ __forceinline__ float group_at(const uint4& v, uint32_t e) {
  const uint32_t wd = e < 4 ? (e < 2 ? v.x : v.y) : (e < 6 ? v.z : v.w);
  return (e & 1u) ? hi_f(wd) : lo_f(wd);
}
// bf16 bits of logit e (0..7) of an 8-logit group
__device__ __forceinline__ uint32_t group_bits(const uint4& v, uint32_t e) {
  const uint32_t wd = e < 4 ? (e < 2 ? v.x : v.y) : (e < 6 ? v.z : v.w);
  return (e & 1u) ? (wd >> 16) : (wd & 0xFFFFu);
}

// mass of logit x in 2^-40 units of exp2((M - M) c) = 1: fixed point, so that
// sums do not depend on their order
__device__ __forceinline__ unsigned long long mass_q(float x, float M, float c) {
  return static_cast<unsigned long long>(ex2((x - M) * c) * 1099511627776.0f);
}

// bit e (0..7) set when logit e of the group is >= the bf16 threshold t2
// (t2: the threshold's bf16 bits in both halves)
__device__ __forceinline__ uint32_t group_ge_bits(const uint4& v, uint32_t t2) {
  const __nv_bfloat162 t = *reinterpret_cast<const __nv_bfloat162*>(&t2);
  const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
  uint32_t bits = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t m = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&wv[q]), t);
    bits |= ((m & 1u) | ((m >> 15) & 2u)) << (2 * q);
  }
  return bits;
}

}  // namespace cgk
