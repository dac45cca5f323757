/*
 * cg.h -- C ABI of the grammar-constrained decoding library (libcg.so).
 *
 * The shape follows the constraint contract of usetacet.com/docs/grammar,
 * "The guarantee is not tied to this engine": three calls over logits and
 * u32 token ids that name no model, tokenizer, device or file --
 *     cg_fill_bitmask    which tokens the grammar allows in each row's state,
 *     cg_mask_and_sample mask the logits and sample after masking,
 *     cg_accept          advance each row's automaton by its token --
 * plus grammar compilation, vocabulary upload, the host-side evaluator of
 * labs.miniml.ai "Evaluator aware decoding" and a host driver for forced
 * tokens.
 *
 * Conventions
 *  - Return codes: CG_OK (0) or a negative CG_E_* code; a failing call leaves
 *    its outputs unspecified and changes no library state.  Argument errors are
 *    detected on the host before anything is launched.
 *  - Ownership: pointers named d_* are device pointers owned by the caller;
 *    h_* and plain pointers are host memory owned by the caller.  Opaque
 *    objects (cg_grammar, cg_vocab, cg_ctx, cg_driver, cg_pda_grammar, cg_pda)
 *    are owned by the library and released by their *_destroy call.
 *  - Asynchrony: the three step calls only enqueue kernels on the context's
 *    CUDA stream and return; results are ready after the stream is
 *    synchronised.  Errors that only the device can see (a state or token id
 *    out of range, a forced token the automaton does not allow, ...) are
 *    recorded in a device status word read by cg_ctx_status().
 *  - States: each grammar's states are numbered 0..n_states-1 breadth-first
 *    from the start state 0 (bytes visited in order 0..255 as written by the
 *    model, then the same bytes as injected by the host).  CG_DEAD marks a
 *    row whose automaton has failed.
 *  - Bitmask layout: row-major u32 [B][W], W = ceil(V / 32); token t is bit
 *    (t & 31) of word (t >> 5); pad bits beyond V are zero.
 *  - Device: a context belongs to the device current at cg_ctx_create.  Every
 *    call on a context (or on a cg_pda built on it) makes that device current
 *    for its duration and puts the caller's back, so its allocations, launches
 *    and symbol lookups happen there whatever device the calling thread has
 *    current; device pointers passed in must live on that device.  Each such
 *    call is also an NVTX range named after the call (nothing is recorded
 *    unless a profiler is attached).
 */
#ifndef CG_H
#define CG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes -------------------------------------------------------- */
#define CG_OK                0
#define CG_E_ARG            -1  /* null pointer, size out of range, mismatched sizes */
#define CG_E_SYNTAX         -2  /* grammar source does not parse */
#define CG_E_UNSUPPORTED    -3  /* schema feature outside the supported subset: fail closed
                                   (dev.to "I found a runner bug...", "What exists beyond
                                   the experiment") */
#define CG_E_EMPTY          -4  /* the grammar accepts no string */
#define CG_E_UNDEFINED_RULE -5  /* a GBNF rule reference has no definition */
#define CG_E_LIMIT          -6  /* automaton, table or token length beyond a library limit */
#define CG_E_CUDA           -7  /* a CUDA runtime call failed */
#define CG_E_DEVICE         -8  /* cg_ctx_status: the device recorded an error */
#define CG_E_NOMEM          -9  /* host allocation failed */

/* ---- enumerations ---------------------------------------------------------- */
#define CG_GBNF        0        /* GBNF-style rule text, start rule "root" */
#define CG_JSON_SCHEMA 1        /* JSON-schema subset */
#define CG_STRUCTURAL_TAG 2     /* structural tag: nested literal / regex / json_schema / sequence / or /
                                   tag / evaluated_tag elements (labs.miniml.ai "Evaluator aware
                                   decoding", "Where XGrammar-2 could take this") */

#define CG_F32  0               /* logits as IEEE binary32 */
#define CG_BF16 1               /* logits as bfloat16 */

#define CG_DEAD     0xFFFFFFFFu /* failed automaton */
#define CG_NO_TOKEN 0xFFFFFFFFu /* the row had no allowed token */

/* per-row flags written by cg_accept */
#define CG_FLAG_DONE        1u  /* new state accepts and has no continuation */
#define CG_FLAG_FORCED_NEXT 2u  /* new state continues only with host-injected bytes */
#define CG_FLAG_REJECTED    4u  /* the token was not allowed: state is CG_DEAD */
#define CG_FLAG_NO_TOKEN    8u  /* the row had no token this step */
#define CG_FLAG_CAPPED     16u  /* the row hit max_tokens and was reset */
#define CG_FLAG_DRAFT_CUT  32u  /* accept_many: a draft token was refused; the state is the accepted prefix's */

/* state flags exported by cg_grammar_export */
#define CG_STATE_ACCEPT      1u
#define CG_STATE_SINK        2u  /* accepting, no outgoing transition */
#define CG_STATE_FORCED_ONLY 4u  /* only host-injected bytes continue */

/* device status codes reported through cg_ctx_status (first one wins) */
#define CG_DEV_OK              0
#define CG_DEV_BAD_STATE       1  /* a state id >= n_states (and not CG_DEAD) */
#define CG_DEV_BAD_TOKEN       2  /* a token id >= V (and not CG_NO_TOKEN) */
#define CG_DEV_BAD_FORCED      3  /* a forced token id >= V */
#define CG_DEV_FORCED_MISMATCH 4  /* accept: the token differs from the forced token */
#define CG_DEV_MISSING_FORCED  5  /* fill: a forced-only state without a forced token */
#define CG_DEV_BAD_GID         6  /* a grammar index >= n_grammars */
#define CG_DEV_REJECTED        7  /* accept: the token walks the automaton to CG_DEAD */
#define CG_DEV_TIMEOUT         8  /* sample: a bounded wait for an asynchronous copy ran out;
                                     the row gets CG_NO_TOKEN */
#define CG_DEV_BAD_LENGTH      9  /* accept_many: a draft length > K (clamped to K) */

/* mask_and_sample flags */
#define CG_SAMPLE_INPLACE 1u     /* also write -inf into masked logits (the "&mut [f32]" form) */

typedef struct cg_grammar cg_grammar;
typedef struct cg_vocab   cg_vocab;
typedef struct cg_ctx     cg_ctx;
typedef struct cg_driver  cg_driver;

/* Termination bounds, usetacet.com/docs/grammar "A valid call also has to
 * end": whitespace runs and open fields are bounded and a generation is
 * capped at max_tokens. */
typedef struct {
    uint32_t ws_max;             /* longest whitespace run in one JSON slot */
    uint32_t max_len_default;    /* maxLength of a JSON string that states none */
    uint32_t depth_max;          /* simultaneous activations of one GBNF rule */
    uint32_t max_items_default;  /* maxItems of a JSON array that states none */
    uint32_t max_tokens;         /* host cap on one generation (cg_accept with counts) */
} cg_bounds;

/* ---- grammar ---------------------------------------------------------------- */

/* Compile a grammar to its minimal byte-level automaton (usetacet.com/docs/grammar,
 * "The guarantee": the automaton masks the logits at every step; nesting is
 * bounded so the automaton is finite).
 *  src, src_len : grammar text (GBNF rules, a JSON schema or a structural tag), not NUL-terminated
 *  kind         : CG_GBNF, CG_JSON_SCHEMA or CG_STRUCTURAL_TAG
 *  bounds       : termination bounds (not retained)
 *  out          : receives the grammar on CG_OK
 *  err, errlen  : optional buffer for a NUL-terminated message (may be NULL/0)
 * Errors: CG_E_ARG, CG_E_SYNTAX, CG_E_UNSUPPORTED, CG_E_EMPTY,
 * CG_E_UNDEFINED_RULE, CG_E_LIMIT (more than 2^24 states), CG_E_NOMEM. */
int cg_compile(const char* src, size_t src_len, int kind, const cg_bounds* bounds,
               cg_grammar** out, char* err, size_t errlen);

void cg_grammar_destroy(cg_grammar* g);

/* n_states: states of the minimal trimmed automaton; n_cols: distinct
 * transition columns over the 512 symbols; start is always 0.  Any output
 * pointer may be NULL. */
int cg_grammar_info(const cg_grammar* g, uint32_t* n_states, uint32_t* n_cols, uint32_t* start);

/* Export the automaton: next[s*512 + a] for symbol a (0..255 model bytes,
 * 256..511 the same bytes injected by the host), -1 for DEAD; flags[s] is a
 * CG_STATE_* mask.  Buffers hold n_states*512 int32 and n_states bytes. */
int cg_grammar_export(const cg_grammar* g, int32_t* next, uint8_t* flags);

/* --try-input (usetacet.com/docs/grammar, "Reading the grammar for a tool"):
 * run a candidate string from the start state and report where it is refused.
 *  s, n        : candidate bytes
 *  injected    : optional per-byte marks (nonzero = byte injected by the host)
 *  refused_at  : receives the offset of the first refused byte, or n
 *  end_state   : receives the state after the accepted prefix (may be NULL)
 *  accepted    : receives 1 if all n bytes are consumed and the state accepts */
int cg_try_input(const cg_grammar* g, const uint8_t* s, size_t n, const uint8_t* injected,
                 size_t* refused_at, uint32_t* end_state, int* accepted);

/* States that are neither finished nor forced-only, increasing; a random
 * start state is live[r mod n].  out may be NULL to query n. */
int cg_live_states(const cg_grammar* g, uint32_t* out, uint32_t cap, uint32_t* n);

/* Mask classes of grammars used together in one context: a mask depends on the
 * automaton state alone, so states with equal masks can share one cached row,
 * across grammars too (labs.miniml.ai "Evaluator aware decoding", "Where
 * XGrammar-2 could take this", on caching across grammars).  States
 * of all n_g grammars, numbered grammar after grammar, share a class when every
 * model-byte word of at most max_len bytes fails from both or from neither, so
 * their token masks for tokens of at most max_len bytes agree; a context keeps
 * one cached mask per class.
 *  class_of : u32 [sum of the grammars' states] or NULL (cap entries available)
 *  n_states : receives the total number of states; n_classes the classes
 * Errors: CG_E_ARG, CG_E_LIMIT (cap too small), CG_E_NOMEM. */
int cg_mask_classes(const cg_grammar* const* g, uint32_t n_g, uint32_t max_len, uint32_t* class_of, uint32_t cap,
                    uint32_t* n_states, uint32_t* n_classes);

/* ---- vocabulary --------------------------------------------------------------- */

/* Token t is bytes[off[t] .. off[t+1]); V >= 1, every token 1..64 bytes.
 * The library copies the data.  Errors: CG_E_ARG, CG_E_LIMIT. */
int cg_vocab_create(const uint8_t* bytes, const uint32_t* off, uint32_t V, cg_vocab** out);
void cg_vocab_destroy(cg_vocab* v);

/* Greedy longest-match tokenisation of text (lowest id among equal strings),
 * the forced-token encoding of labs.miniml.ai "Evaluator aware decoding", "The
 * core idea" step 3.  Writes up to cap ids, n_out receives the count needed;
 * CG_E_LIMIT if cap is too small, CG_E_ARG if a byte has no token. */
int cg_tokenize_greedy(const cg_vocab* v, const uint8_t* text, size_t n, uint32_t* out,
                       size_t cap, size_t* n_out);

/* ---- device context ------------------------------------------------------------ */

/* Upload n_g grammars and one vocabulary to the current CUDA device and bind
 * the context to cuda_stream (a cudaStream_t; NULL = legacy default stream).
 * Allocates the transition tables, the trie-ordered vocabulary and the
 * per-mask-class cache of allowed-token bitmasks (token mask cache,
 * labs.miniml.ai "Where XGrammar-2 could take this").  Grammars and vocab may
 * be destroyed afterwards.  Errors: CG_E_ARG, CG_E_CUDA, CG_E_LIMIT, CG_E_NOMEM. */
int cg_ctx_create(const cg_grammar* const* g, uint32_t n_g, const cg_vocab* v,
                  void* cuda_stream, cg_ctx** out);
void cg_ctx_destroy(cg_ctx* c);

/* n_classes: total mask classes (states with identical masks share one);
 * cache_bytes: device bytes of the mask cache; V, W of the vocabulary. */
int cg_ctx_info(const cg_ctx* c, uint32_t* n_classes, uint64_t* cache_bytes, uint32_t* V, uint32_t* W);

/* Synchronise the context's stream, return CG_OK or CG_E_DEVICE, and move the
 * first recorded CG_DEV_* code into *dev_code (may be NULL), clearing it.
 * CG_DEV_TIMEOUT from a sampling or step call (not from
 * cg_self_test_wait_timeout, which has no copy in flight) means a block gave
 * up on a bounded wait; its own last wait for the copies it had issued is
 * bounded too, so a copy may still have landed in shared memory after the
 * block exited.  The rows it served got CG_NO_TOKEN; destroy the context and
 * create a new one before trusting further results. */
int cg_ctx_status(cg_ctx* c, uint32_t* dev_code);

/* Compute the bitmask of every mask class now (one CTA per class) instead of
 * on first use, so that later steps never walk the vocabulary.  Asynchronous
 * on the context's stream.  The pages exclude such one-time grammar work from
 * timing by discarding warm-up calls (seedpath.ai "Guided Decoding &
 * Structured-Output Reliability", "What we measured": fairness controls).
 * Errors: CG_E_ARG, CG_E_CUDA. */
int cg_ctx_prefill(cg_ctx* c);

/* Mask-cache behaviour on a context without cg_ctx_prefill (labs.miniml.ai
 * "Evaluator aware decoding", "Where XGrammar-2 could take this", on the token
 * mask cache).  On such a context cg_fill_bitmask and cg_step first run a
 * miss pre-pass: every class mask a row needs and the cache lacks is computed
 * by 32 blocks sharing its walk, so the step that follows finds it ready.
 *  lookups  : rows that looked their class up in the pre-pass (hits + misses)
 *  computed : class masks the pre-pass computed because a row missed them
 *  ready    : class masks in the cache now, by any path (of n_classes)
 * Counted since the context was created; synchronises the context's stream.
 * Any output may be NULL.  Errors: CG_E_ARG, CG_E_CUDA. */
int cg_ctx_cache_stats(cg_ctx* c, uint64_t* lookups, uint64_t* computed, uint32_t* ready);

/* Step 1 -- which tokens may follow each row's state (usetacet.com/docs/grammar,
 * "The guarantee"; a mask depends on the automaton state alone and is known
 * before the step, labs.miniml.ai "Why isn't this in production APIs yet?").
 *  d_states  : u32 [B] automaton state of each row (CG_DEAD -> empty mask)
 *  d_gid     : u16 [B] grammar index of each row, or NULL for grammar 0
 *  d_forced  : i32 [B] token the host forces on the row, -1 for none, or NULL;
 *              a forced row gets exactly that token
 *  d_bitmask : u32 [B][W] output
 * Token t is allowed iff walking its bytes from the state never fails.  Masks
 * are served from the per-class cache, computed on first use. */
int cg_fill_bitmask(cg_ctx* c, const uint32_t* d_states, const uint16_t* d_gid,
                    const int32_t* d_forced, uint32_t B, uint32_t* d_bitmask);

/* Step 2 -- mask, temperature, softmax, top-p, sample ("Sampling runs after
 * masking", usetacet.com/docs/grammar).
 *  d_logits  : [B][V] CG_F32 or CG_BF16 (dtype), row-major, V = the vocab size
 *  d_bitmask : u32 [B][W] from cg_fill_bitmask
 *  temp      : 0 -> greedy argmax (ties to the lowest id); > 0 -> z = x / temp
 *  top_p     : nucleus mass; >= 1 keeps every allowed token
 *  seed,step : Philox4x32-10 stream; token t of row b uses word t&3 of
 *              Philox((t>>2, b, step, 0), (seed lo, seed hi))
 *  d_out_tok : u32 [B] sampled id, CG_NO_TOKEN for a row without allowed tokens
 *  d_probs   : optional f32 [B][V] softmax over allowed tokens (0 elsewhere;
 *              greedy rows get 1 at the chosen token), or NULL
 *  flags     : CG_SAMPLE_INPLACE to also store -inf into masked logits
 * Sampling is Gumbel-max over the nucleus: argmax z_t + g_t, g = -log(-log u).
 * The context keeps a device scratch for per-row candidate lists (6 bytes x
 * 8192 per row); the first call with a larger B than before synchronises the
 * stream and grows it with cudaMalloc, so make that first call before any
 * stream capture.  Returns CG_E_NOMEM when the scratch cannot be allocated. */
int cg_mask_and_sample(cg_ctx* c, void* d_logits, int dtype, uint32_t B, uint32_t V,
                       const uint32_t* d_bitmask, float temp, float top_p, uint64_t seed,
                       uint32_t step, uint32_t* d_out_tok, float* d_probs, uint32_t flags);

/* One decode step in one call: cg_fill_bitmask, cg_mask_and_sample (no probs,
 * no in-place write) and cg_accept with the same arguments, giving the same
 * tokens, states, flags and counts bit for bit.  When the sampling takes the
 * top-p bf16 path (dtype CG_BF16, temp > 0, top_p < 1, V a multiple of 8,
 * 16-byte aligned logits) the three run as one kernel per row: the row's mask
 * is built on chip from the mask-class cache, the logits are streamed once, and
 * the token is accepted at the end of the row's block.  Otherwise the three
 * calls run in turn.
 *  d_bitmask : u32 [B][W] or NULL; when given it receives the masks exactly as
 *              cg_fill_bitmask writes them.  With NULL on the unfused path the
 *              context keeps the masks in a buffer of its own (grown like the
 *              sampling scratch: the first call with a larger B synchronises
 *              the stream and allocates).
 *  d_out_states may equal d_states (each row reads its state before writing it).
 * Errors: as the three calls. */
int cg_step(cg_ctx* c, const uint32_t* d_states, const uint16_t* d_gid, const int32_t* d_forced, uint32_t B,
            void* d_logits, int dtype, uint32_t V, float temp, float top_p, uint64_t seed, uint32_t step,
            uint32_t* d_counts, uint32_t max_tokens, uint32_t* d_bitmask, uint32_t* d_out_tok,
            uint32_t* d_out_states, uint8_t* d_out_flags);

/* cg_step with the logits in HOST memory and the sampled ids returned to host
 * memory: the end-to-end form of the step for a caller whose logits are not on
 * the device.  The pages have no counterpart: it only moves the inputs and
 * outputs of the step (usetacet.com/docs/grammar, "Constrained decoding").
 *  h_logits  : [B][V] of dtype in host memory, page-locked (cudaHostAlloc or
 *              cudaHostRegister) for the copy to run asynchronously; pageable
 *              memory works but the copy then blocks the calling thread
 *  h_out_tok : u32 [B] host memory (page-locked for an asynchronous copy)
 *  d_out_tok : u32 [B] device memory that also receives the ids, or NULL
 *  the rest  : as cg_step (states, forced ids, counts and flags stay on the device)
 * The logits are copied on a stream of the context's own into one of two
 * context-owned device buffers (grown like the sampling scratch), the step
 * waits for that copy on the context stream, and the ids are copied back on
 * the context stream.  The buffers alternate from call to call, so the copy of
 * one step's logits overlaps the previous step's kernels.
 * Asynchronous: the call returns once all of this is queued.  h_logits must
 * stay unchanged and h_out_tok unread until cg_ctx_sync (or cg_ctx_status)
 * has returned.  Not for stream capture.
 * Errors: as cg_step; CG_E_CUDA when a copy, stream or event call fails. */
int cg_step_host(cg_ctx* c, const uint32_t* d_states, const uint16_t* d_gid, const int32_t* d_forced, uint32_t B,
                 const void* h_logits, int dtype, uint32_t V, float temp, float top_p, uint64_t seed, uint32_t step,
                 uint32_t* d_counts, uint32_t max_tokens, uint32_t* h_out_tok, uint32_t* d_out_tok,
                 uint32_t* d_out_states, uint8_t* d_out_flags);

/* Waits until everything queued on the context has finished (the context
 * stream, and through it the copies of cg_step_host).  CG_E_CUDA on a CUDA
 * error. */
int cg_ctx_sync(cg_ctx* c);

/* Variant of cg_mask_and_sample that never allocates device memory.  The pages
 * have no counterpart: it is a deployment variant of step 2, not a step of the
 * method.  Arguments, results and error codes are those of cg_mask_and_sample,
 * except where this block says otherwise.
 *  - It is for callers that must not allocate device memory while decoding:
 *    cudaMalloc/cudaFree synchronise the device and can fail once a server has
 *    planned all of HBM (e.g. for its KV cache) at start-up.
 *  - Scratch: a fixed array inside the library, one per device: the per-row
 *    kernels' candidate lists (CG_NOALLOC_MAX_ROWS x 8192 x 6 bytes, 3 MiB),
 *    then the segmented kernel's counters and per-row pairs (64 KiB; the
 *    greedy and top_p >= 1 calls without probabilities take that kernel).
 *    B > CG_NOALLOC_MAX_ROWS returns CG_E_LIMIT without launching anything.
 *  - The list part need not start at zero (every entry is written before it is
 *    read); the segmented part is cleared on the context's stream before each
 *    launch that uses it.
 *  - Every call on a device uses the same array, so calls that may overlap on
 *    the device (other streams, other contexts, other host threads) race on it;
 *    the caller must serialise them (one stream at a time).
 *  - The context's device is made current for the call (as for every entry
 *    point), so the array is the one on the context's device.  The first call
 *    on a device looks up its address (cudaGetSymbolAddress; CG_E_CUDA if that
 *    fails) and keeps it; make that first call before capturing any stream, and
 *    do not call it again on a device after cudaDeviceReset (the kept address
 *    is then stale). */
#define CG_NOALLOC_MAX_ROWS 64u
int cg_mask_and_sample_noalloc(cg_ctx* c, void* d_logits, int dtype, uint32_t B, uint32_t V,
                               const uint32_t* d_bitmask, float temp, float top_p, uint64_t seed,
                               uint32_t step, uint32_t* d_out_tok, float* d_probs, uint32_t flags);

/* Step 3 -- advance each row's automaton by its token (labs.miniml.ai "Evaluator
 * aware decoding", "A concrete prototype on llama.cpp": the automaton also moves
 * forward over injected tokens).
 *  d_states, d_gid : as in cg_fill_bitmask (d_gid may be NULL)
 *  d_toks          : u32 [B] tokens from cg_mask_and_sample
 *  d_forced        : i32 [B] or NULL; a row with d_forced >= 0 must carry that
 *                    token, and its bytes are walked as host-injected bytes
 *  d_counts        : u32 [B] or NULL; when given, each row's token count is
 *                    advanced and a row that finishes (CG_FLAG_DONE) or reaches
 *                    max_tokens is reset to state 0 with count 0
 *  max_tokens      : the cap used with d_counts (usetacet.com/docs/grammar)
 *  d_out_states    : u32 [B] new states (may alias d_states)
 *  d_out_flags     : u8 [B] CG_FLAG_* bits */
int cg_accept(cg_ctx* c, const uint32_t* d_states, const uint16_t* d_gid, const uint32_t* d_toks,
              const int32_t* d_forced, uint32_t B, uint32_t* d_counts, uint32_t max_tokens,
              uint32_t* d_out_states, uint8_t* d_out_flags);

/* Speculative verification of drafts against the grammar (labs.miniml.ai
 * "Evaluator aware decoding", "Where XGrammar-2 could take this": once a draft
 * token ends an evaluated span, the evaluator's result fixes the tokens after
 * it, so checking them is a comparison of ids).  Per row, the longest prefix of the
 * draft whose tokens the grammar allows one after another is accepted, as
 * cg_accept would accept them one per step.
 *  d_states, d_gid : as in cg_accept (d_gid may be NULL)
 *  d_draft         : u32 [B][K] draft token ids, row-major; d_draft_len u32 [B]
 *                    the number of them per row (at most K; a longer length is
 *                    clamped to K and recorded as CG_DEV_BAD_LENGTH)
 *  d_forced        : i32 [B][K] or NULL; forced[b][j] >= 0 pins position j: the
 *                    draft token there must equal it and is walked as
 *                    host-injected bytes (the result tokens the host computed)
 *  d_counts, max_tokens : as in cg_accept; each accepted token counts
 *  d_out_states    : u32 [B] the state after the accepted prefix (may alias d_states)
 *  d_out_n         : u32 [B] draft tokens accepted
 *  d_out_flags     : u8 [B] CG_FLAG_DONE / CG_FLAG_FORCED_NEXT of that state, plus
 *                    CG_FLAG_DRAFT_CUT (a token was refused: not an error, the
 *                    state is the accepted prefix's), CG_FLAG_CAPPED,
 *                    CG_FLAG_NO_TOKEN (empty draft), CG_FLAG_REJECTED (dead row)
 *  d_out_path      : u32 [B][K + 1] or NULL: the state before each position
 *                    0..out_n (the caller masks the next position's logits from
 *                    it), CG_DEAD after out_n
 * Verification of a row stops at the first refused token, after a token that
 * ends the grammar, when the count reaches max_tokens, and after a token whose
 * state continues only with injected bytes when the next position is not
 * pinned (the host evaluates the span, then pins its result).  With d_counts a
 * row ended or capped by its accepted tokens restarts from state 0 with count
 * 0.  Device errors as cg_accept (a refused token is not one).
 * Errors: CG_E_ARG for a NULL required pointer, K == 0 with B > 0, or d_counts
 * with max_tokens == 0. */
int cg_accept_many(cg_ctx* c, const uint32_t* d_states, const uint16_t* d_gid, const uint32_t* d_draft,
                   const uint32_t* d_draft_len, const int32_t* d_forced, uint32_t B, uint32_t K, uint32_t* d_counts,
                   uint32_t max_tokens, uint32_t* d_out_states, uint32_t* d_out_n, uint8_t* d_out_flags,
                   uint32_t* d_out_path);

/* Self-test of the device's failure detection: every wait of the library's
 * kernels (bulk copies into shared memory, the mask-cache claim) is bounded
 * and, when its limit runs out, records CG_DEV_TIMEOUT in the status word
 * and returns instead of hanging.  This call launches one block whose
 * bounded wait on a barrier that no copy completes runs out; afterwards
 * cg_ctx_status reports CG_DEV_TIMEOUT and the context stays usable.
 * Asynchronous on the context stream; the wait polls for well under a second.
 * Errors: CG_E_ARG, CG_E_CUDA. */
int cg_self_test_wait_timeout(cg_ctx* c);

/* ---- pushdown automaton for recursive grammars ---------------------------------- */

/* usetacet.com/docs/grammar, "The guarantee": the automaton that masks the
 * logits is a pushdown automaton.  cg_compile flattens nesting into a DFA
 * (each rule active at most depth_max times), whose size grows with the
 * bound; these calls keep one automaton per recursive rule and a stack per
 * row instead.
 *
 * Language: GBNF as in cg_compile.  Every reference to a recursive rule (one
 * on a cycle of references) opens a frame; other rules are inlined; the start
 * rule is the base frame and opens none.  At most `depth` frames are open at
 * once; a reference past that matches nothing.  Prefixes that can no longer
 * be completed within the bound are refused.
 *
 * Grammar class (CG_E_UNSUPPORTED otherwise): deterministic with one symbol
 * of lookahead -- in every state the bytes that continue the rule and the
 * first bytes of each rule it may call are disjoint; no recursive rule
 * matches the empty string or calls itself before its first byte; where a
 * state may end its rule, none of the bytes it consumes can follow the rule.
 * Recursive rules may not be referenced inside @forced( ) or under '&'.
 *
 * Row configuration, u32 [B][depth + 2] on the device, updated in place by
 * cg_pda_accept: word 0 the state (CG_DEAD for a failed row), word 1 the stack
 * level L (0..depth), words 2..2+L-1 the return states bottom to top (words
 * past L are unused).  A fresh row is {0, 0}. */
#define CG_PDA_MAX_DEPTH 64

typedef struct cg_pda_grammar cg_pda_grammar;
typedef struct cg_pda cg_pda;

/* Compile a recursive GBNF grammar with a stack bound depth <= CG_PDA_MAX_DEPTH.
 * Errors: CG_E_ARG, CG_E_SYNTAX, CG_E_UNDEFINED_RULE, CG_E_UNSUPPORTED (the
 * grammar class above), CG_E_EMPTY, CG_E_LIMIT (more than 64 recursive rules
 * or 2^24 states), CG_E_NOMEM. */
int cg_pda_compile(const char* src, size_t src_len, uint32_t depth, cg_pda_grammar** out);
void cg_pda_grammar_destroy(cg_pda_grammar* g);

/* Sizes: states of all rule automata, rules (the start rule and the recursive
 * ones), transition columns, stack bound.  Any output may be NULL. */
int cg_pda_grammar_info(const cg_pda_grammar* g, uint32_t* n_states, uint32_t* n_rules, uint32_t* n_cols,
                        uint32_t* depth);

/* Walk bytes s[0..n) from a fresh row (injected[i] != 0: byte i is host-injected;
 * injected may be NULL).  consumed receives the number of bytes walked before
 * the first refused one (n when none is refused), accepted 1 when all were
 * walked and the text may end there, level (optional) the stack level after
 * the walk.  Host only. */
int cg_pda_try_input(const cg_pda_grammar* g, const uint8_t* s, size_t n, const uint8_t* injected,
                     size_t* consumed, int* accepted, uint32_t* level);

/* Device pushdown object on context c, for the vocabulary v the context was
 * created with (same V).  Precomputes, per state and stack headroom, the mask
 * of the tokens whose walk never pops below the row's level (one cached mask
 * per distinct set), and per state the list of tokens that do (decided per row
 * against its stack).  Uses c's stream and status word; destroy it before c.
 * Errors: CG_E_ARG, CG_E_CUDA, CG_E_NOMEM. */
int cg_pda_create(cg_ctx* c, const cg_vocab* v, const cg_pda_grammar* g, cg_pda** out);
void cg_pda_destroy(cg_pda* p);

/* Sizes of the precomputation: (state, headroom) keys, distinct cached masks,
 * their bytes, tokens on the per-state lists.  Any output may be NULL. */
int cg_pda_info(const cg_pda* p, uint32_t* n_keys, uint32_t* n_masks, uint64_t* cache_bytes,
                uint32_t* n_candidates);

/* Step 1 for pushdown rows: d_cfg u32 [B][depth + 2] as above; d_forced as in
 * cg_fill_bitmask (NULL for none); d_bitmask u32 [B][W].  A failed row gets an
 * empty mask; a row whose state or level is out of range records
 * CG_DEV_BAD_STATE and gets an empty mask.  Sampling is cg_mask_and_sample on
 * the same context. */
int cg_pda_fill_bitmask(cg_pda* p, const uint32_t* d_cfg, uint32_t B, const int32_t* d_forced,
                        uint32_t* d_bitmask);

/* Step 3 for pushdown rows: advance each row's configuration in place by its
 * token (as injected bytes where d_forced >= 0, which must match the token).
 * d_counts / max_tokens and the flags as in cg_accept: CG_FLAG_DONE when the
 * text is complete and nothing may follow, CG_FLAG_FORCED_NEXT when only
 * injected bytes may follow; a finished or capped row restarts at {0, 0} when
 * counts are kept. */
int cg_pda_accept(cg_pda* p, uint32_t* d_cfg, uint32_t B, const uint32_t* d_toks, const int32_t* d_forced,
                  uint32_t* d_counts, uint32_t max_tokens, uint8_t* d_out_flags);

/* Speculative verification for pushdown rows, as cg_accept_many is for
 * automaton rows (same draft, pin, count and stopping rules and the same
 * flags): d_cfg u32 [B][depth + 2] is updated in place to the configuration
 * after the accepted prefix (a refused token leaves it unchanged); d_draft
 * u32 [B][K], d_draft_len u32 [B], d_forced i32 [B][K] or NULL, d_out_n u32 [B]
 * tokens accepted, d_out_flags u8 [B].  No path output: a pushdown
 * configuration is a stack, not one word.  Errors: CG_E_ARG for a NULL required
 * pointer, K == 0 with B > 0, or d_counts with max_tokens == 0. */
int cg_pda_accept_many(cg_pda* p, uint32_t* d_cfg, uint32_t B, const uint32_t* d_draft, const uint32_t* d_draft_len,
                       const int32_t* d_forced, uint32_t K, uint32_t* d_counts, uint32_t max_tokens,
                       uint32_t* d_out_n, uint8_t* d_out_flags);

/* The whole step for pushdown rows, as cg_step is for automaton rows: the
 * mask of each row (as cg_pda_fill_bitmask, into d_bitmask too when it is not
 * NULL), masked sampling (as cg_mask_and_sample, same arguments) and the
 * accept into d_cfg (as cg_pda_accept with d_forced, d_counts, max_tokens).
 * On the bf16 top-p path it is one kernel per row; otherwise the three calls.
 * Results are identical to the three calls.  Errors: as those calls. */
int cg_pda_step(cg_pda* p, uint32_t* d_cfg, uint32_t B, void* d_logits, int dtype, uint32_t V, float temp,
                float top_p, uint64_t seed, uint32_t step, const int32_t* d_forced, uint32_t* d_counts,
                uint32_t max_tokens, uint32_t* d_bitmask, uint32_t* d_out_tok, uint8_t* d_out_flags);

/* Step 3 of one step and step 1 of the next in one launch: cg_pda_accept with
 * these arguments, then cg_pda_fill_bitmask of the updated configurations with
 * d_forced_next (NULL for none) into d_bitmask.  Results are identical to the
 * two calls in sequence. */
int cg_pda_accept_fill(cg_pda* p, uint32_t* d_cfg, uint32_t B, const uint32_t* d_toks, const int32_t* d_forced,
                       uint32_t* d_counts, uint32_t max_tokens, uint8_t* d_out_flags, const int32_t* d_forced_next,
                       uint32_t* d_bitmask);

/* ---- evaluator-aware host side --------------------------------------------------- */

#define CG_RESULT_CALC_TAG    0  /* <result>V</result> | <result_error>code</result_error> */
#define CG_RESULT_JSON_ANSWER 1  /* , "answer": V}     | , "answer": null, "error": "code"} */
#define CG_RESULT_STROP_TAG   2  /* string operation: <result>V</result> | <result_error>code</result_error> */

/* Evaluate an arithmetic span exactly over the rationals (labs.miniml.ai
 * "Evaluator aware decoding": "17 * 23 + 91 = 482") and format the bytes the
 * host forces.  Grammar: expr := term (('+'|'-') term)*, term := unary
 * (('*'|'/') unary)*, unary := '-' unary | primary, primary := NUMBER |
 * '(' expr ')', NUMBER := [0-9]+('.'[0-9]*)? | '.'[0-9]+, spaces skipped.
 * Failures format an error code: parse, div_zero, non_integer, overflow (more
 * than 64 digits).  Writes up to cap bytes; out_len receives the length
 * (CG_E_LIMIT if cap is too small).  *ok receives 1 for a numeric result. */
int cg_eval_arith(const uint8_t* span, size_t n, int fmt, uint8_t* out, size_t cap,
                  size_t* out_len, int* ok);

/* Evaluate a string operation (labs.miniml.ai "Evaluator aware decoding", "Not
 * just arithmetic: string operations": count("strawberry", "r") = 3) and format
 * the bytes the host forces as CG_RESULT_STROP_TAG.  Span: NAME(ARG, ...) with
 * spaces around the pieces; ARG a string literal "..." (escapes \" and \\
 * only) or an integer -?[0-9]{1,9}.  count(s, sub) counts non-overlapping
 * occurrences left to right; len(s) counts bytes; reverse(s); upper(s) raises
 * ASCII a-z; substr(s, i, j) is the slice [i, j) with negative indices counted
 * from the end and both ends clamped.  Strings are bytes.  Failures format an
 * error code: parse, unknown_op, arity, empty (count of ""), overflow (a result
 * over 64 bytes or a span over 4096), bad_char (a result holding '<').
 * Writes up to cap bytes; out_len receives the length (CG_E_LIMIT if cap is
 * too small).  *ok receives 1 for a result, 0 for an error code. */
int cg_eval_strop(const uint8_t* span, size_t n, uint8_t* out, size_t cap, size_t* out_len, int* ok);

/* Host driver of forced tokens for B rows (labs.miniml.ai "Evaluator aware
 * decoding", "The core idea" steps 1-4).  Row b uses grammar rules[gid[b]]:
 * when a step leaves the row in a forced-only state with nothing queued, the
 * text between the last span_open and the trailing span_close is evaluated and
 * its formatted result is tokenised into the row's queue. */
typedef struct {
    const uint8_t* span_open;  size_t span_open_len;
    const uint8_t* span_close; size_t span_close_len;
    int result_format;         /* CG_RESULT_* (the evaluator follows from it), or -1 for a grammar
                                  without evaluator */
} cg_span_rule;

int cg_driver_create(const cg_vocab* v, uint32_t B, const uint16_t* h_gid,
                     const cg_span_rule* rules, uint32_t n_rules, cg_driver** out);
void cg_driver_destroy(cg_driver* d);

/* Apply one step's results on the host, in this order per row: a used forced
 * token leaves the queue; a real token extends the row's text; a row flagged
 * CG_FLAG_DONE or CG_FLAG_CAPPED forgets its text and queue; otherwise a row
 * flagged CG_FLAG_FORCED_NEXT with an empty queue is evaluated.  Then writes
 * the next step's forced token per row (-1 for none) into h_forced_next.
 *  h_toks, h_flags, h_forced_used : this step's tokens, flags and forced ids
 *  n_evals : optional, receives the number of evaluations this call made */
int cg_driver_update(cg_driver* d, const uint32_t* h_toks, const uint8_t* h_flags,
                     const int32_t* h_forced_used, int32_t* h_forced_next, uint32_t* n_evals);

#ifdef __cplusplus
}
#endif
#endif /* CG_H */
