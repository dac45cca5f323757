// Segmented streaming sampler for greedy rows and for Gumbel-max over every
// allowed token (top_p >= 1), with every SM carrying the same share of the
// logits whatever the batch size (the sampler sees only masked logits:
// usetacet.com/docs/grammar, "The guarantee").  Top-p rows take the per-row
// kernels of kernel_sample.cu.
//
// What is computed per row b is what kernel_sample.cu's header states: with
// z_t = x_t / temp over the allowed tokens, the token argmax of z_t + g_t,
// g_t = -log(-log u_t), u_t from Philox4x32-10 word t&3 of counter
// (t>>2, b, step, 0); greedy (temp = 0) the allowed token of largest logit,
// lowest id on ties.
//
// Work decomposition.  Each row is cut into segments of up to four 4096-logit
// chunks; a persistent grid (three CTAs per SM) takes segments from a work
// counter in segment-major order (segment s of every row before segment
// s + 1, so that a row's best score so far is mostly known before its later
// segments are read), and the bytes each SM streams differ by at most a
// segment.  A CTA has three roles.  The producer warp resolves each segment's
// mask source (the caller's bitmask, or in the fused step the row's mask class
// in the mask cache) ahead of time and streams the segment's logits and mask
// words into a 6-slot shared-memory ring with bulk asynchronous copies.
// Eight consumer warps take each chunk 16 logits per thread (two 8-logit
// groups).  The service warp counts each row's finished segments (a fence and
// an atomic per segment, off the consumers' path).  Once the stream is done,
// the consumers finish the rows their CTA owns (b = blockIdx.x + k gridDim.x),
// each as soon as every segment of it is counted.
//
// Greedy keeps each thread's best (x, lowest id).  Gumbel-max over every
// allowed token draws the Philox block of each group of four tokens with an
// allowed one and tests a cheap upper bound of each token's score (the noise
// g(u) = -ln(-ln u) is at most -ln(1 - u)) against the best score found so
// far (the row's best from its earlier segments included); the few tokens
// that pass are queued per warp and scored exactly 32 at a time.  Both publish
// a packed (value, id) maximum per row; the finisher takes the row's.
//
// The fused step (cg_step) also builds each row's mask from the mask-class
// cache (rows with a forced token or without allowed tokens stream nothing:
// the token is the forced one, or none), writes the bitmask when asked, and
// accepts the token when the row finishes.
//
// Device scratch (the context's, zero before the first launch): a work counter
// pair and a (segments counted, best) pair per row.  Every launch leaves them
// at zero again (the last CTA to stop taking work resets the counters; each
// row's finisher its pair).
#include <algorithm>
#include <map>
#include <mutex>
#include <utility>

#include "bf16_ops.cuh"
#include "row_ops.cuh"

namespace cgk {

cudaError_t allow_smem(const void* kernel, size_t bytes);  // kernel_sample.cu

namespace seg {

constexpr uint32_t kConsWarps = 8;
constexpr uint32_t kCons = kConsWarps * 32;                // 256 consumer threads
constexpr uint32_t kProdWarp = kConsWarps;                 // the producer warp
constexpr uint32_t kSvcWarp = kConsWarps + 1;              // the service warp
constexpr uint32_t kThreads = kCons + 64;
constexpr uint32_t kChunk = 4096;                          // logits per ring slot
constexpr uint32_t kChunkBytes = kChunk * 2;               // 8 KiB
constexpr uint32_t kChunkWords = kChunk / 32;              // mask words per slot
constexpr uint32_t kGroups = kChunk / 8;                   // 8-logit groups per slot
constexpr uint32_t kMaxSegChunks = 4;
constexpr uint32_t kSlots = 6;                             // a segment and a half of four chunks in flight
constexpr uint32_t kMaxNS = 64;                            // segments per row
constexpr uint32_t kSQ = 16;                               // records queued for the service warp (> kSlots)
constexpr uint32_t kQ = 160;                               // queued exact scores per consumer warp (full)
constexpr uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;   // Philox4x32 multipliers
static_assert(kGroups == 2 * kCons, "two groups per consumer thread and slot");

// dynamic shared memory
constexpr uint32_t kOffRing = 0;
constexpr uint32_t kOffMask = kOffRing + kSlots * kChunkBytes;
constexpr uint32_t kOffPool = kOffMask + kSlots * kChunkWords * 4;
constexpr uint32_t kPoolBytes = kConsWarps * kQ * 10;      // exact-score queues (full)
constexpr uint32_t kOffDesc = kOffPool + kPoolBytes;
constexpr uint32_t kSmem = kOffDesc + kSlots * 16;
static_assert(kSmem <= 74 * 1024, "three CTAs a multiprocessor");

enum Mode { kModeGreedy = 0, kModeFull = 2 };
// kinds of ring descriptors and service records
constexpr uint32_t kStream = 0, kEmptyRow = 1, kForcedRow = 2, kNone = 3, kEnd = 4, kSkipPending = 5;

struct RowAcc {
  uint32_t done;              // segments counted
  uint32_t pad;
  unsigned long long best;    // packed (value, id) maximum over the row's segments
};

// Per-row accumulators in the scratch, after a work-counter pair.  Every
// launch leaves them at zero (the last CTA to stop taking work resets the
// counters, each row's finisher its accumulators).
constexpr uint32_t kRowStride = 16;
constexpr uint32_t kCtlBytes = 256;
static_assert(sizeof(RowAcc) == kRowStride, "one accumulator block a row");
static_assert(kCtlBytes + size_t(CG_NOALLOC_MAX_ROWS) * kRowStride <= kNoAllocSegBytes,
              "the no-allocation scratch holds the segmented sampler's rows");

struct Scratch {
  unsigned char* base;        // [kCtlBytes] counters, then [B] row blocks of kRowStride bytes
  __device__ uint32_t* ctl() const { return reinterpret_cast<uint32_t*>(base); }  // [0] next segment, [1] CTAs done
  __device__ RowAcc* row(uint32_t b) const {
    return reinterpret_cast<RowAcc*>(base + kCtlBytes + size_t(b) * kRowStride);
  }
};

struct Fused {
  Tables t;
  const uint32_t* states;
  const uint16_t* gid;        // may be null
  const int32_t* forced;      // may be null
  uint32_t* counts;           // may be null
  uint32_t max_tokens;
  uint32_t* out_states;
  uint8_t* out_flags;
  uint32_t* bitmask_out;      // may be null
  DevGrammar pg[8];           // grammar descriptors by value (one dependent load fewer)
  uint32_t n_pg;
};

struct Params {
  const uint16_t* logits;     // [B][V] bf16 bits, 16-byte aligned rows (V % 8 == 0)
  uint32_t V, W, B, NS, segc, nchunks, N;
  const uint32_t* bitmask;    // sampling from a bitmask: [B][W], W % 4 == 0, 16-byte aligned
  float temp, top_p;
  uint32_t step;
  uint32_t rk[20];            // Philox round keys: rk[2r] = seed lo + r W0, rk[2r + 1] = seed hi + r W1
  uint32_t ph_lo1, ph_hi1;    // M1 x step, the step's term of the first Philox round
  uint32_t* out_tok;
  uint32_t* status;
  Scratch sc;
  Fused f;
};

struct Src {
  uint32_t b, s, kind, aux;
  const uint32_t* mask;
};

// shared memory views and scalars
struct Smem {
  uint4* ring4;
  uint32_t* mask32;
  uint32_t* pool;              // per consumer warp: the exact-score queue (full)
  uint4* desc;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* sq_full;           // [kSQ] consumers -> service: a record is ready (kCons arrivals)
  uint64_t* sq_empty;          // [kSQ] service -> consumers: the record slot is free again
  uint4* sq_rec;               // [kSQ]
  uint32_t* words;             // [32] scalars
};
enum {
  kWAbort = 0,  // a bounded wait ran out
  kWIssued,     // ring slots the producer used
  kWRowOk,      // the finishing row's segments are all counted
  kWKind,       // the finishing row's kind and forced token
  kWAux,
};

__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, %0;" ::"n"(kCons) : "memory"); }
// consumer barrier that also returns whether any consumer thread passed true
// (bounded waits can run out in some threads only; what follows must be uniform)
__device__ __forceinline__ void red_add_u32(uint32_t* p, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_max_u32(uint32_t* p, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_max_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_relaxed64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_volatile_s(const uint32_t* p) { return *reinterpret_cast<const volatile uint32_t*>(p); }

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long y = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = y > v ? y : v;
  }
  return v;
}

__device__ __forceinline__ DevGrammar grammar_of(const Fused& f, uint32_t g) {
  if (g >= f.n_pg) return f.t.grammars[g];
  DevGrammar gd = f.pg[0];
#pragma unroll
  for (uint32_t i = 1; i < 8; ++i)
    if (g == i) gd = f.pg[i];
  return gd;
}

// ---- Philox4x32-10 with the row's constant terms hoisted ---------------------------
// The counter of token t is (t >> 2, b, step, 0): in round one the product
// M1 x step is the same for every block of the launch, and the first word
// after round one depends on the row only, so round two's M0 product is the
// row's too.  philox_q(row, q) equals philox4x32_10((q, b, step, 0), seed).
__device__ __forceinline__ void mul_wide(uint32_t a, uint32_t b, uint32_t& lo, uint32_t& hi) {
  unsigned long long r;
  asm("mul.wide.u32 %0, %1, %2;" : "=l"(r) : "r"(a), "r"(b));
  lo = static_cast<uint32_t>(r);
  hi = static_cast<uint32_t>(r >> 32);
}
struct PhRow {
  uint32_t a1, l2, h2;  // word 0 after round one; M0 x a1 (lo, hi)
};
__device__ __forceinline__ PhRow philox_row(const Params& p, uint32_t b) {
  PhRow r;
  r.a1 = p.ph_hi1 ^ b ^ p.rk[0];
  mul_wide(kM0, r.a1, r.l2, r.h2);
  return r;
}
__device__ __forceinline__ uint4 philox_q(const Params& p, const PhRow& r, uint32_t q) {
  uint32_t lo0, hi0, lo1, hi1;
  mul_wide(kM0, q, lo0, hi0);
  // after round one: (a1, lo(M1 step), hi0 ^ k1, lo0); round two
  const uint32_t c2 = hi0 ^ p.rk[1];
  mul_wide(kM1, c2, lo1, hi1);
  uint32_t c0 = hi1 ^ p.ph_lo1 ^ p.rk[2], c1 = lo1, c3 = r.l2;
  uint32_t cz = r.h2 ^ lo0 ^ p.rk[3];
#pragma unroll
  for (int rr = 2; rr < 10; ++rr) {
    uint32_t l0, h0, l1, h1;
    mul_wide(kM0, c0, l0, h0);
    mul_wide(kM1, cz, l1, h1);
    const uint32_t n0 = h1 ^ c1 ^ p.rk[2 * rr], n2 = h0 ^ c3 ^ p.rk[2 * rr + 1];
    c0 = n0;
    c1 = l1;
    cz = n2;
    c3 = l0;
  }
  return make_uint4(c0, c1, cz, c3);
}

// Gumbel score of token id with logit bits xb: z + g, g = -log(-log u)
__device__ __forceinline__ float gumbel_score(float x, float temp, uint32_t w) {
  return __fdiv_rn(x, temp) + gumbel_from_word(w);
}

// Where segment idx's mask comes from, in two stages so that the producer can
// have the loads of both in flight while it streams: stage1 loads the row's
// grammar, forced token and state; stage2 the state's flags and mask class.
// Fused: the row's mask class in the cache, or -- for a row with a forced
// token or without allowed tokens -- no stream at all (kSkipPending: the
// producer counts the row's segments and the row's owner finishes it once all
// have been counted, so that nothing writes the row's state before every
// segment has read it).
struct Stage1 {
  uint32_t idx, g, st;
  int32_t fo;
};
template <int FUSED>
__device__ __forceinline__ Stage1 stage1(const Params& p, uint32_t idx) {
  Stage1 r{idx, 0u, 0u, -1};
  if (!FUSED || idx >= p.N) return r;
  const Fused& f = p.f;
  const uint32_t b = idx % p.B;
  r.g = f.gid ? f.gid[b] : 0u;
  r.fo = f.forced ? f.forced[b] : -1;
  r.st = f.states[b];
  return r;
}
template <int FUSED>
__device__ __forceinline__ Src stage2(const Params& p, const Stage1& a, bool record = true) {
  Src r;
  r.s = a.idx / p.B;  // segment-major: segment s of every row before segment s + 1
  r.b = a.idx - r.s * p.B;
  r.kind = kStream;
  r.aux = 0;
  r.mask = nullptr;
  if (!FUSED) {
    r.mask = p.bitmask + size_t(r.b) * p.W;
    return r;
  }
  const Fused& f = p.f;
  const Tables& t = f.t;
  DevGrammar gd{};
  if (a.g < t.n_g) gd = grammar_of(f, a.g);
  uint8_t sflags = 0;
  uint32_t cls = 0;
  if (a.g < t.n_g && a.fo < 0 && a.st != CG_DEAD && a.st < gd.n_states) {
    sflags = t.state_flags[gd.state_off + a.st];
    cls = t.class_of[gd.state_off + a.st];
  }
  uint32_t err = 0;
  const int mode = row_mask_mode_of(t.n_g, t.V, a.g, a.fo, a.st, gd.n_states, sflags, &err);
  if (mode == 0) {
    r.mask = t.cache + size_t(cls) * t.Wc;
    return r;
  }
  if (record && err && r.s == 0) record_error(t.status, err);
  r.kind = kSkipPending;
  r.aux = (mode == 2) ? (uint32_t(a.fo) | 0x80000000u) : 0u;
  return r;
}

// The producer warp's lane 0: takes segments from the work counter and
// streams their chunks (logits with an evict-first L2 hint, then the chunk's
// mask words) into the ring.  The next item's mask source and the row of the
// one after are loaded while the current item's chunks are issued.  Returns
// the slots used.
template <int FUSED>
__device__ uint32_t produce(const Params& p, unsigned char* dsm, uint64_t* full, uint64_t* empty, uint4* desc,
                            uint32_t* s_abort) {
  const uint32_t N = p.N;
  const uint64_t pol = evict_first_policy();
  uint32_t q = 0;
  bool ok = true;
  uint32_t i0 = atomicAdd(p.sc.ctl(), 1u);
  uint32_t i1 = i0 < N ? atomicAdd(p.sc.ctl(), 1u) : N;
  uint32_t i2 = i1 < N ? atomicAdd(p.sc.ctl(), 1u) : N;
  Src cur{};
  if (i0 < N) cur = stage2<FUSED>(p, stage1<FUSED>(p, i0));
  Stage1 s1 = stage1<FUSED>(p, i1);
  auto take_slot = [&](uint32_t& sl) -> bool {
    sl = q % kSlots;
    return q < kSlots || mbar_wait(empty + sl, ((q / kSlots) - 1u) & 1u);
  };
  while (i0 < N) {
    // loads for the items ahead, in flight while this one streams
    Src nxt{};
    if (i1 < N) nxt = stage2<FUSED>(p, s1);
    const Stage1 s2 = stage1<FUSED>(p, i2);
    const uint32_t i3 = i2 < N ? atomicAdd(p.sc.ctl(), 1u) : N;
    uint32_t kind = cur.kind;
    if (FUSED && kind == kSkipPending) {
      // a row without a stream: its segments only count, and the row's owner
      // finishes it once every segment has read the row's state
      red_release_add(&p.sc.row(cur.b)->done, 1u);
      kind = kNone;
    }
    if (kind != kNone) {
      const uint32_t nch = kind == kStream ? min(p.segc, p.nchunks - cur.s * p.segc) : 1u;
      for (uint32_t k = 0; k < nch; ++k, ++q) {
        uint32_t sl;
        if (!take_slot(sl)) {
          ok = false;
          break;
        }
        desc[sl] = make_uint4(cur.b, cur.s, kind | (nch << 8), cur.aux & 0x7FFFFFFFu);
        if (kind == kStream) {
          const uint32_t ck = cur.s * p.segc + k;
          const uint32_t n = min(kChunk, p.V - ck * kChunk);
          const uint32_t mw = (((n + 31u) >> 5) + 3u) & ~3u;
          mbar_expect_tx(full + sl, n * 2 + mw * 4);
          bulk_g2s_hint(dsm + kOffRing + sl * kChunkBytes, p.logits + size_t(cur.b) * p.V + size_t(ck) * kChunk,
                        n * 2, full + sl, pol);
          bulk_g2s(dsm + kOffMask + sl * (kChunkWords * 4), cur.mask + size_t(ck) * kChunkWords, mw * 4, full + sl);
        } else {
          mbar_arrive(full + sl);  // the descriptor is the whole message
        }
      }
      if (!ok) break;
    }
    cur = nxt;
    s1 = s2;
    i0 = i1;
    i1 = i2;
    i2 = i3;
  }
  if (ok) {
    uint32_t sl;
    if (take_slot(sl)) {
      desc[sl] = make_uint4(0u, 0u, kEnd, 0u);
      mbar_arrive(full + sl);
      ++q;
    } else {
      ok = false;
    }
  }
  if (!ok) {
    record_error(p.status, CG_DEV_TIMEOUT);
    atomicExch(s_abort, 1u);
  }
  // this CTA takes no more segments: the last one to stop resets the counters
  // for the next launch
  __threadfence();
  if (atomicAdd(p.sc.ctl() + 1, 1u) == gridDim.x - 1) {
    p.sc.ctl()[0] = 0u;
    p.sc.ctl()[1] = 0u;
  }
  return q;
}

// Outputs of a finished row: the token, and in the fused step the accept.
template <int FUSED>
__device__ __noinline__ void emit(const Params& p, uint32_t b, uint32_t tok) {
  p.out_tok[b] = tok;
  if (FUSED) {
    const Fused& f = p.f;
    const uint32_t g = f.gid ? f.gid[b] : 0u;
    const int32_t fo = f.forced ? f.forced[b] : -1;
    accept_row(f.t, b, g, f.states[b], tok, fo, f.counts, f.max_tokens, f.out_states, f.out_flags);
  }
}

// ---- the service warp ------------------------------------------------------------------

// Counts the rows' finished segments: takes the consumers' records in order
// (one per segment, then the end record) and, per stream record, fences and
// adds one to the row's count.  The consumers go on streaming meanwhile: the
// fence is off their path.
__device__ void service(const Params& p, const Smem& sm) {
  const uint32_t lane = threadIdx.x & 31;
  for (uint32_t k = 0;; ++k) {
    bool ok = true;
    if (lane == 0) ok = mbar_wait(sm.sq_full + k % kSQ, (k / kSQ) & 1u);
    if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) {
      if (lane == 0) {
        record_error(p.status, CG_DEV_TIMEOUT);
        atomicExch(&sm.words[kWAbort], 1u);
      }
      return;
    }
    const uint4 r = sm.sq_rec[k % kSQ];
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(sm.sq_empty + k % kSQ);
      if (r.z == kStream) {
        // every consumer thread's writes for the segment precede its arrival
        // on the record's barrier; the fence orders them before the count
        __threadfence();
        red_add_u32(&p.sc.row(r.x)->done, 1u);
      }
    }
    if (r.z == kEnd) return;
  }
}

// ---- finishing a row (the consumer threads of the row's CTA, together) ------------------

// A row without a stream (fused step): a forced token or no allowed token.
template <int FUSED>
__device__ void finish_skip(const Params& p, uint32_t b, uint32_t kind, uint32_t f) {
  if (FUSED && p.f.bitmask_out) {
    uint32_t* out = p.f.bitmask_out + size_t(b) * p.W;
    for (uint32_t i = threadIdx.x; i < p.W; i += kCons)
      out[i] = (kind == kForcedRow && i == (f >> 5)) ? (1u << (f & 31u)) : 0u;
  }
  if (threadIdx.x == 0) {
    p.sc.row(b)->done = 0u;
    emit<FUSED>(p, b, kind == kForcedRow ? f : CG_NO_TOKEN);
  }
}

// Finishes row b once every segment of it is counted: its token (and the
// accept in the fused step), then its accumulators back to zero.
template <int MODE, int FUSED>
__device__ void finish_row(const Params& p, uint32_t b, const Smem& sm) {
  const uint32_t tid = threadIdx.x;
  RowAcc* ra = p.sc.row(b);
  if (FUSED) {
    if (tid == 0) {
      const Src r = stage2<FUSED>(p, stage1<FUSED>(p, b), false);
      sm.words[kWKind] = r.kind == kSkipPending ? ((r.aux & 0x80000000u) ? kForcedRow : kEmptyRow) : kStream;
      sm.words[kWAux] = r.aux & 0x7FFFFFFFu;
    }
    cbar();
    const uint32_t kind = sm.words[kWKind], aux = sm.words[kWAux];
    cbar();
    if (kind != kStream) {
      finish_skip<FUSED>(p, b, kind, aux);
      return;
    }
  }
  const unsigned long long v = __ldcg(&ra->best);
  const uint32_t tok = v ? best_id(v) : CG_NO_TOKEN;
  if (tid == 0) {
    ra->done = 0u;
    ra->best = 0ull;
    emit<FUSED>(p, b, tok);
  }
}

// ---- the consumer warps ------------------------------------------------------------------

// Full mode: score the warp's queued tokens [base, base + n) exactly, one per
// lane, and raise the lanes' bests and the warp's bound reference.
__device__ __noinline__ void drain_queue(const uint32_t* qid, const uint32_t* qw, const uint16_t* qx,
                                            uint32_t base, uint32_t n, float temp, unsigned long long& best,
                                            float& bestv, float& offB) {
  const uint32_t lane = threadIdx.x & 31;
  if (lane < n) {
    const uint32_t i = base + lane;
    const float sc = gumbel_score(bf16_bits_to_float(qx[i]), temp, qw[i]);
    const unsigned long long pk = pack_best(sc, qid[i]);
    if (pk > best) best = pk;
  }
  // the warp's best score is the bound reference of all its lanes
  const uint32_t wk = __reduce_max_sync(0xFFFFFFFFu, best ? static_cast<uint32_t>(best >> 32) : 0u);
  if (wk) {
    const float wb = fkey_inv(wk);
    if (wb > bestv) {
      bestv = wb;
      offB = 23.f - wb * 1.4426950408889634f;
    }
  }
}

// Each consumer warp works on its own share of every chunk (64 groups of 8
// logits) and ends each segment on its own: no consumer-wide barrier on the
// stream's path.  Per segment a warp raises the row's packed best with its
// own and arrives on the service record.
template <int MODE, int FUSED>
__device__ void consume(const Params& p, const Smem& sm) {
  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float temp = p.temp;
  const float c = (MODE == kModeGreedy) ? 0.f : 1.4426950408889634f / temp;
  const uint32_t g0 = warp * 64 + lane, g1 = g0 + 32;
  const uint4 kNeg4 = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
  uint32_t q = 0;     // ring slots taken
  uint32_t nrec = 0;  // records sent to the service warp
  bool ok = true;
  // One record for the service warp: thread 0 writes it once its slot is
  // free; every consumer thread arrives once its own writes for it are done.
  auto post = [&](uint32_t b, uint32_t s, uint32_t kind, uint32_t aux) {
    const uint32_t k = nrec % kSQ;
    if (tid == 0) {
      if (nrec >= kSQ && !mbar_wait(sm.sq_empty + k, ((nrec / kSQ) - 1u) & 1u)) {
        record_error(p.status, CG_DEV_TIMEOUT);
        atomicExch(&sm.words[kWAbort], 1u);
      }
      sm.sq_rec[k] = make_uint4(b, s, kind, aux);
    }
    mbar_arrive(sm.sq_full + k);
    ++nrec;
  };
  // per warp: the exact-score queue (full)
  uint32_t* qid = sm.pool + warp * kQ;
  uint32_t* qw = sm.pool + kConsWarps * kQ + warp * kQ;
  uint16_t* qx = reinterpret_cast<uint16_t*>(sm.pool + 2 * kConsWarps * kQ) + warp * kQ;
  for (;;) {
    const uint32_t sl0 = q % kSlots;
    if (!mbar_wait(sm.full + sl0, (q / kSlots) & 1u)) {
      ok = false;
      break;
    }
    const uint4 d = sm.desc[sl0];
    const uint32_t kind = d.z & 0xFFu;
    if (kind == kEnd) break;
    const uint32_t b = d.x, s = d.y, nch = (d.z >> 8) & 0xFFu;
    RowAcc* ra = p.sc.row(b);
    if (kind != kStream) {
      // fused step: a row with a forced token or without allowed tokens, for the service warp
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.empty + sl0);
      post(b, s, kind, d.w);
      ++q;
      continue;
    }
    // ---- greedy / full: the segment's chunks one by one ------------------------------
    unsigned long long best = 0ull;    // greedy / full: packed (value, id)
    float bestv = -INFINITY;           // greedy: value of best; full: the bound's reference score
    float offB = INFINITY;             // full: 23 - bestv log2(e)
    uint32_t qn = 0;                   // full: this warp's queued exact scores
    PhRow phr{};
    unsigned long long seed_best = 0ull;
    if (MODE == kModeFull) {
      phr = philox_row(p, b);
      if (lane == 0) seed_best = ld_relaxed64(&ra->best);  // the row's best so far (other segments)
    }
#pragma unroll 1
    for (uint32_t k = 0; k < nch; ++k) {
      const uint32_t qk = q + k, sl = qk % kSlots;
      if (k > 0 && !mbar_wait(sm.full + sl, (qk / kSlots) & 1u)) {
        ok = false;
        break;
      }
      const uint32_t ck = s * p.segc + k;
      const uint32_t ng = min(kGroups, (p.V - ck * kChunk) >> 3);
      const uint4* r4 = sm.ring4 + sl * kGroups;
      const uint8_t* m8 = reinterpret_cast<const uint8_t*>(sm.mask32 + sl * kChunkWords);
      uint4 v0 = kNeg4, v1 = kNeg4;
      uint32_t mb0 = 0, mb1 = 0;
      if (g0 < ng) {
        mb0 = m8[g0];
        v0 = apply_mask(r4[g0], pair_mask_of(mb0));
      }
      if (g1 < ng) {
        mb1 = m8[g1];
        v1 = apply_mask(r4[g1], pair_mask_of(mb1));
      }
      if (FUSED && p.f.bitmask_out && lane < 16) {
        const uint32_t wi = ck * kChunkWords + warp * 16 + lane;
        if (wi < p.W) p.f.bitmask_out[size_t(b) * p.W + wi] = sm.mask32[sl * kChunkWords + warp * 16 + lane];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.empty + sl);
      if (MODE == kModeGreedy) {
        const uint32_t a0 = group_pmax(v0), a1 = group_pmax(v1);
#pragma unroll
        for (uint32_t h = 0; h < 2; ++h) {
          const uint4& v = h ? v1 : v0;
          const float gm = pmax_f(h ? a1 : a0);
          if (gm > bestv) {  // strictly: this thread sees ids in increasing order
            uint32_t e = 0;
            while (e < 7 && group_at(v, e) != gm) ++e;
            best = pack_best(gm, ck * kChunk + (h ? g1 : g0) * 8 + e);
            bestv = gm;
          }
        }
      } else {
        if (k == 1) {
          // the bound's first outside reference: the row's best score from its other segments
          const unsigned long long sb = __shfl_sync(0xFFFFFFFFu, seed_best, 0);
          if (sb) {
            const float v = fkey_inv(static_cast<uint32_t>(sb >> 32));
            if (v > bestv) {
              bestv = v;
              offB = 23.f - v * 1.4426950408889634f;
            }
          }
        }
#pragma unroll 1
        for (uint32_t h = 0; h < 2; ++h) {
          const uint4 v = h ? v1 : v0;
          const uint32_t mb = h ? mb1 : mb0;
          const uint32_t t0 = ck * kChunk + (h ? g1 : g0) * 8;
#pragma unroll
          for (uint32_t half = 0; half < 2; ++half) {
            const uint32_t nib = (mb >> (4 * half)) & 15u;
            if (!__any_sync(0xFFFFFFFFu, nib != 0u)) continue;  // four tokens a lane, masked out for the whole warp
            const uint4 blk = philox_q(p, phr, (t0 >> 2) + half);
            const uint32_t wa = half ? v.z : v.x, wb = half ? v.w : v.y;
            // the token's score can beat bestv only if 2^23 exp(z - bestv)
            // (slightly enlarged) exceeds 2^23 - 1 - (w >> 9), i.e. the bound
            // -ln(1 - u) of its noise reaches bestv - z: one bit a token
            uint32_t pm = 0;
#pragma unroll
            for (uint32_t e = 0; e < 4; ++e) {
              const uint32_t wd = e < 2 ? wa : wb;
              const float x = (e & 1u) ? hi_f(wd) : lo_f(wd);
              const uint32_t w = e == 0 ? blk.x : e == 1 ? blk.y : e == 2 ? blk.z : blk.w;
              const float tq = ex2(fmaf(x, c, offB)) * 1.0001f;
              const float vv = __uint_as_float((w >> 9) ^ 0x4B7FFFFFu) - 8388608.0f;
              if (((nib >> e) & 1u) && vv < tq) pm |= 1u << e;
            }
            if (__any_sync(0xFFFFFFFFu, pm != 0u)) {
              // queue the passing tokens (at most 4 a lane: qn stays below kQ)
              const uint32_t n = __popc(pm);
              uint32_t inc = n;
#pragma unroll
              for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
                if (lane >= uint32_t(o)) inc += y;
              }
              uint32_t pos = qn + inc - n;
#pragma unroll
              for (uint32_t e = 0; e < 4; ++e) {
                if ((pm >> e) & 1u) {
                  const uint32_t wd = e < 2 ? wa : wb;
                  qid[pos] = t0 + 4 * half + e;
                  qw[pos] = e == 0 ? blk.x : e == 1 ? blk.y : e == 2 ? blk.z : blk.w;
                  qx[pos] = uint16_t((e & 1u) ? (wd >> 16) : (wd & 0xFFFFu));
                  ++pos;
                }
              }
              qn += __shfl_sync(0xFFFFFFFFu, inc, 31);
              while (qn >= 32) {
                __syncwarp();
                drain_queue(qid, qw, qx, qn - 32, 32, temp, best, bestv, offB);
                qn -= 32;
                __syncwarp();
              }
            }
          }
        }
      }
    }
    if (!__all_sync(0xFFFFFFFFu, ok)) {
      ok = false;
      break;
    }

    // ---- segment end (this warp's slice) ------------------------------------------------
    {
      // greedy / full: the slice's packed maximum into the row's
      if (MODE == kModeFull && qn) {
        __syncwarp();
        drain_queue(qid, qw, qx, 0, qn, temp, best, bestv, offB);
      }
      const unsigned long long v = warp_max_u64(best);
      if (lane == 0 && v) red_max_u64(&ra->best, v);
    }
    post(b, s, kStream, 0u);
    q += nch;
  }
  if (!ok) {
    record_error(p.status, CG_DEV_TIMEOUT);
    atomicExch(&sm.words[kWAbort], 1u);
  }
  post(0u, 0u, kEnd, 0u);
  // together now: the rows this CTA owns (b = blockIdx.x + k gridDim.x), each
  // once the service warps have counted all its segments
  for (uint32_t own = blockIdx.x; own < p.B; own += gridDim.x) {
    if (tid == 0) {
      bool ready = false;
      for (uint32_t i = 0; i < kWaitLimit && !ready; ++i) {
        if (ld_acquire_gpu(&p.sc.row(own)->done) >= p.NS) {
          ready = true;
        } else {
          if (ld_volatile_s(&sm.words[kWAbort])) break;
          __nanosleep(64);
        }
      }
      if (!ready) {
        record_error(p.status, CG_DEV_TIMEOUT);
        atomicExch(&sm.words[kWAbort], 1u);
      }
      // (after an abort copies may still be in flight into the ring: no finishing)
      sm.words[kWRowOk] = (ready && !ld_volatile_s(&sm.words[kWAbort])) ? 1u : 0u;
    }
    cbar();
    if (!sm.words[kWRowOk]) break;
    finish_row<MODE, FUSED>(p, own, sm);
    cbar();  // before the next row reuses the shared memory
  }
}

template <int MODE, int FUSED>
__global__ void __launch_bounds__(kThreads, 3) seg_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ __align__(8) uint64_t full[kSlots], empty[kSlots], sq_full[kSQ], sq_empty[kSQ];
  __shared__ uint4 sq_rec[kSQ];
  __shared__ uint32_t words[32];
  Smem sm;
  sm.ring4 = reinterpret_cast<uint4*>(dsm + kOffRing);
  sm.mask32 = reinterpret_cast<uint32_t*>(dsm + kOffMask);
  sm.pool = reinterpret_cast<uint32_t*>(dsm + kOffPool);
  sm.desc = reinterpret_cast<uint4*>(dsm + kOffDesc);
  sm.full = full;
  sm.empty = empty;
  sm.sq_full = sq_full;
  sm.sq_empty = sq_empty;
  sm.sq_rec = sq_rec;
  sm.words = words;

  griddep_launch_dependents();
  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (uint32_t i = 0; i < kSlots; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, kConsWarps);
    }
    for (uint32_t i = 0; i < kSQ; ++i) {
      mbar_init(sq_full + i, kCons);
      mbar_init(sq_empty + i, 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    for (uint32_t i = 0; i < 32; ++i) words[i] = 0u;
  }
  __syncthreads();
  griddep_wait();  // the logits, the bitmask or the rows' states come from earlier work on the stream

  if (warp == kProdWarp) {
    if (lane == 0) words[kWIssued] = produce<FUSED>(p, dsm, full, empty, sm.desc, &words[kWAbort]);
  } else if (warp == kSvcWarp) {
    service(p, sm);
  } else {
    consume<MODE, FUSED>(p, sm);
  }
  __syncthreads();
  if (tid == 0 && words[kWAbort]) {
    // a wait ran out: let the copies still in flight land before the shared
    // memory is released (again with bounded waits)
    const uint32_t used = words[kWIssued];
    for (uint32_t sl = 0; sl < kSlots && sl < used; ++sl) {
      const uint32_t last = used - 1 - ((used - 1 - sl) % kSlots);  // last sequence index of slot sl
      mbar_wait(full + sl, (last / kSlots) & 1u);
    }
  }
}

// ---- host side ---------------------------------------------------------------------------

// Chunks per segment: the largest of 4, 2, 1 that still gives the grid a few
// segments per CTA, among those that keep a row within kMaxNS segments.
uint32_t segs_for(uint32_t B, uint32_t nchunks, uint32_t grid) {
  uint32_t pick = 0;
  for (uint32_t sc = 1; sc <= kMaxSegChunks; sc *= 2) {
    const uint32_t ns = (nchunks + sc - 1) / sc;
    if (ns > kMaxNS) continue;
    if (pick == 0 || uint64_t(B) * ns >= uint64_t(4) * grid) pick = sc;
  }
  return pick;  // seg_usable() guarantees that sc = kMaxSegChunks fits
}

struct Occ {
  int sms = 0, per_sm = 0;
};
template <int MODE, int FUSED>
cudaError_t occupancy(Occ* o) {
  static std::mutex mu;
  static std::map<int, Occ> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  auto it = done.find(dev);
  if (it != done.end()) {
    *o = it->second;
    return cudaSuccess;
  }
  auto* k = seg_kernel<MODE, FUSED>;
  if ((e = allow_smem(reinterpret_cast<const void*>(k), kSmem)) != cudaSuccess) return e;
  Occ r;
  if ((e = cudaDeviceGetAttribute(&r.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r.per_sm, k, kThreads, kSmem)) != cudaSuccess) return e;
  if (r.per_sm < 1) return cudaErrorInvalidConfiguration;
  done[dev] = r;
  *o = r;
  return cudaSuccess;
}

template <int MODE, int FUSED>
cudaError_t launch(Params& p, void* scratch, uint32_t B, uint32_t V, cudaStream_t stream) {
  Occ o;
  cudaError_t e = occupancy<MODE, FUSED>(&o);
  if (e != cudaSuccess) return e;
  const uint32_t grid_max = uint32_t(o.sms) * uint32_t(o.per_sm);
  p.nchunks = (V + kChunk - 1) / kChunk;
  p.segc = segs_for(B, p.nchunks, grid_max);
  p.NS = (p.nchunks + p.segc - 1) / p.segc;
  p.N = B * p.NS;
  p.sc.base = static_cast<unsigned char*>(scratch);
  const uint32_t grid = std::min<uint32_t>(grid_max, p.N);
  return launch_dependent(seg_kernel<MODE, FUSED>, dim3(grid), dim3(kThreads), size_t(kSmem), stream, p);
}

// Philox round keys of the seed and the step's first-round product.
void set_philox(Params& p, uint64_t seed, uint32_t step) {
  uint32_t k0 = uint32_t(seed), k1 = uint32_t(seed >> 32);
  for (int r = 0; r < 10; ++r) {
    p.rk[2 * r] = k0;
    p.rk[2 * r + 1] = k1;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  const uint64_t m = uint64_t(kM1) * step;
  p.ph_lo1 = uint32_t(m);
  p.ph_hi1 = uint32_t(m >> 32);
  p.step = step;
}

template <int FUSED>
cudaError_t launch_mode(Params& p, void* scratch, uint32_t B, uint32_t V, cudaStream_t stream) {
  if (p.temp == 0.f) return launch<kModeGreedy, FUSED>(p, scratch, B, V, stream);
  if (p.top_p >= 1.f) return launch<kModeFull, FUSED>(p, scratch, B, V, stream);
  return cudaErrorInvalidValue;  // top-p rows take the per-row kernels (seg_usable)
}

}  // namespace seg

// Scratch bytes of the segmented sampler for B rows (zero before the first
// launch; every launch leaves it at zero).
size_t seg_scratch_bytes(uint32_t B) { return seg::kCtlBytes + size_t(B) * seg::kRowStride; }

// The segmented sampler takes greedy rows and Gumbel-max over every allowed
// token (top_p >= 1): bf16 rows of V % 8 == 0 logits at 16-byte aligned
// addresses, up to kMaxNS x 4 chunks, without the optional outputs.  Top-p
// rows (0 < top_p < 1) take the per-row kernels of kernel_sample.cu, measured
// faster at every batch size tried (16 to 512 rows of 32000 to 151936 logits).
bool seg_usable(int dtype, uint32_t V, const void* logits, float* probs, int inplace, float temp, float top_p) {
  const uint32_t nchunks = (V + seg::kChunk - 1) / seg::kChunk;
  return dtype == CG_BF16 && V % 8 == 0 && V > 0 && nchunks <= seg::kMaxNS * seg::kMaxSegChunks &&
         (reinterpret_cast<uintptr_t>(logits) & 15u) == 0 && probs == nullptr && inplace == 0 &&
         (temp == 0.f || top_p >= 1.f);
}

// cg_mask_and_sample through the segmented sampler (the bitmask must have
// W % 4 == 0 words per row at a 16-byte aligned address).
bool seg_bitmask_ok(uint32_t W, const void* bitmask) {
  return W % 4 == 0 && (reinterpret_cast<uintptr_t>(bitmask) & 15u) == 0;
}

cudaError_t launch_seg_sample(const void* logits, uint32_t B, uint32_t V, uint32_t W, const uint32_t* bitmask,
                              float temp, float top_p, uint64_t seed, uint32_t step, uint32_t* out_tok,
                              void* scratch, uint32_t* status, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  seg::Params p{};
  p.logits = static_cast<const uint16_t*>(logits);
  p.V = V;
  p.W = W;
  p.B = B;
  p.bitmask = bitmask;
  p.temp = temp;
  p.top_p = top_p;
  seg::set_philox(p, seed, step);
  p.out_tok = out_tok;
  p.status = status;
  return seg::launch_mode<0>(p, scratch, B, V, stream);
}

cudaError_t launch_seg_step(const Tables& t, const uint32_t* states, const uint16_t* gid, const int32_t* forced,
                            uint32_t B, const void* logits, uint32_t V, float temp, float top_p, uint64_t seed,
                            uint32_t step, uint32_t* counts, uint32_t max_tokens, uint32_t* bitmask_out,
                            uint32_t* out_tok, uint32_t* out_states, uint8_t* out_flags, void* scratch,
                            const DevGrammar* host_grammars, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  seg::Params p{};
  p.logits = static_cast<const uint16_t*>(logits);
  p.V = V;
  p.W = t.W;
  p.B = B;
  p.temp = temp;
  p.top_p = top_p;
  seg::set_philox(p, seed, step);
  p.out_tok = out_tok;
  p.status = t.status;
  seg::Fused& f = p.f;
  f.t = t;
  f.states = states;
  f.gid = gid;
  f.forced = forced;
  f.counts = counts;
  f.max_tokens = max_tokens;
  f.out_states = out_states;
  f.out_flags = out_flags;
  f.bitmask_out = bitmask_out;
  f.n_pg = 0;
  if (host_grammars && t.n_g <= 8) {
    for (uint32_t i = 0; i < t.n_g; ++i) f.pg[i] = host_grammars[i];
    f.n_pg = t.n_g;
  }
  return seg::launch_mode<1>(p, scratch, B, V, stream);
}

}  // namespace cgk
