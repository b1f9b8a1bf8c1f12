/*
 * s2.h -- C ABI of the GB300 Dual-AR frame-decode library (libs2.so).
 *
 * What it computes: the Dual-AR generation stage of the Fish Audio S2
 * text-to-speech model ("SGLang Day-0 Support for FishAudio S2", Architecture,
 * Stage 2; "Fish Audio Abre Codigo do S2", Por Dentro do Modelo: Arquitetura
 * Dual-AR).  Each frame is one Slow AR decode step (a GQA transformer over a
 * paged KV cache) whose head, restricted to the semantic ids, picks code 0,
 * followed by the Fast AR depth loop (a small transformer seeded by the slow
 * hidden state) that greedily emits codes 1..9 ("s2pro-native", What happens
 * to a sentence: ten residual codes, nine greedy steps deep).  VQ codebook
 * embeddings are summed into the input embedding at masked prompt positions
 * and for every decoded frame fed back; prompts share KV through a radix
 * prefix cache ("SGLang Day-0 ...", Optimizations with SGLang Omni: paged KV
 * cache, radix prefix caching).
 *
 * Conventions for every call:
 *   - Return 0 (S2_OK) or a negative S2_E* status; nothing throws across the
 *     ABI.  s2_strerror() names a status.
 *   - Buffers belong to the caller.  Pointer arguments may be host or device
 *     memory; the library tells them apart with cudaPointerGetAttributes.
 *   - Work is enqueued on the stream given at creation.  Results written to
 *     device buffers are valid once that stream has synchronised; results
 *     written to host buffers are valid when the call returns.
 *   - A context is not thread-safe; use one context per host thread.
 */
#ifndef S2_H_
#define S2_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define S2_OK 0
#define S2_EINVAL (-1)    /* bad id, length, pointer or code value */
#define S2_ENOMEM (-2)    /* KV page pool or device memory short; no state changed */
#define S2_ECUDA (-3)     /* a CUDA call failed */
#define S2_ETIMEOUT (-4)  /* a bounded device-side wait gave up */
#define S2_EBADFILE (-5)  /* weight file missing or malformed */
#define S2_ESTATE (-6)    /* sequence in the wrong state for this call */

/* s2_opts.flags */
#define S2_FLAG_NO_GRAPH 1  /* launch kernels directly instead of replaying CUDA graphs */
#define S2_FLAG_NO_TC 2     /* never use the tcgen05 tensor-core GEMM (CUDA-core GEMV only) */
#define S2_FLAG_NO_PDL 4    /* no programmatic dependent launch between kernels */
#define S2_FLAG_NO_RADIX 8  /* never share prompt pages through the radix cache */
#define S2_FLAG_INT8 16     /* per-output-channel INT8 weights for every streamed matrix
                               (layer projections, semantic head slice, Fast AR heads);
                               all projections then run on the CUDA-core GEMV */
#define S2_FLAG_KV_BF16 64  /* store the Slow AR KV cache in bf16 (half the KV bytes; the
                               default keeps it in fp32, which the logit tolerance needs) */
#define S2_FLAG_PERSIST 128 /* run the full frames of a decode call in one persistent
                               cooperative kernel (grid barriers between operations) instead
                               of replaying the per-frame CUDA graph; same kernel code and work
                               split, bit-identical codes; measured slower than the graphs on
                               GB300, kept as an option */
#define S2_FLAG_NO_PREFIX_TC 512 /* decode batches whose rows share radix prompt pages attend
                               to them with the CUDA-core decode attention like any other key
                               (by default the shared prefix goes to the tcgen05 prefix
                               attention, read once per kv head for the whole batch) */
#define S2_FLAG_STREAM 256  /* run the full frames of a decode call at batch 1-2 in the
                               streaming kernel: one persistent launch whose per-SM producer
                               warp streams the weights through a shared-memory ring of bulk
                               copies while 16 consumer warps run the operations (grid
                               barriers between them); results agree with the per-frame CUDA
                               graphs to rounding (the GEMV sums in another order); frames it
                               cannot run (INT8, bf16 KV cache, larger batches, debug sinks,
                               select-kernel heads) replay the graphs */

typedef struct s2_ctx s2_ctx;

typedef struct {
  int32_t max_seqs;        /* sequence ids are 0 .. max_seqs-1 */
  int32_t max_batch;       /* largest decode batch */
  int32_t kv_pool_pages;   /* 16-token pages in the Slow AR KV pool */
  int32_t page_size;       /* must be 16 */
  int32_t max_ctx;         /* longest sequence (prompt + frames), positions */
  int32_t max_prompt;      /* longest prefill */
  uint64_t page_perm_seed; /* 0: free pages handed out in ascending order;
                              otherwise in a seeded random order (scattered pages) */
  void* cuda_stream;       /* cudaStream_t to enqueue on; NULL = a blocking stream the
                              context creates (synchronises with the default stream) */
  int32_t flags;           /* S2_FLAG_* */
  int32_t prefill_rows;    /* uncached prompt rows one s2_prefill_batch pass may hold
                              (0: max_prompt; at least max_prompt) */
  int32_t reserved[6];
} s2_opts;

typedef struct {
  int64_t prefill_tokens;   /* positions computed by prefills */
  int64_t cached_tokens;    /* prompt positions served from the radix cache */
  int64_t frames_decoded;   /* frames emitted, summed over sequences */
  int32_t pages_used;       /* pages referenced by sequences or the radix tree */
  int32_t pages_total;
  int32_t radix_pages;      /* pages held by the radix tree */
  int32_t last_error;       /* last non-zero status, 0 if none */
  int32_t device_error;     /* device-side error flag (1 = a bounded wait expired) */
  int32_t num_sms;
  int64_t weight_bytes;     /* bytes of weights resident on the device */
  int64_t kernel_launches;  /* library kernels launched, graph replays included */
  int64_t evicted_pages;    /* radix pages dropped (least recently used) to make room */
  int64_t reserved[4];
} s2_stats_t;

/* Load a weight file (format of s2_inputs/weights.py) onto the current CUDA
 * device and allocate the KV pool and work buffers.  ``opts`` may be NULL for
 * defaults (64 sequences, batch 64, pool for 64 x 2048 positions).  On
 * success *out owns all device memory until s2_destroy. */
int s2_create(const char* weights_path, const s2_opts* opts, s2_ctx** out);

/* Free everything owned by the context (synchronises its stream). */
void s2_destroy(s2_ctx* ctx);

/* Prefill sequence ``seq`` (which must be free) with a prompt of T positions
 * ("SGLang Day-0 Support for FishAudio S2", Architecture: the prompt's VQ
 * codebook embeddings are summed into the input embedding at masked
 * positions; Optimizations with SGLang Omni: paged KV cache and radix prefix
 * caching, so a prompt sharing a cached prefix computes only its suffix).
 * Pages: as for decoding, unused radix pages are evicted (LRU) if the pool
 * is short, and none are when that could not make enough room (S2_ENOMEM,
 * nothing changed).
 *   tokens   int32 [T], ids in [0, vocab)
 *   vq_codes int32 [n_codebooks, T] (row-major); column t is read iff
 *            vq_mask[t] != 0, and each read code must lie in [0, codebook_size)
 *   vq_mask  uint8 [T] or NULL (no VQ positions)
 * The longest page-aligned prefix already in the radix cache (keys: token,
 * mask and, at masked positions, all codes) is reused, at most T-1 positions;
 * its count is written to *cached_len_out when non-NULL.  Afterwards the
 * sequence is primed: its first decoded frame reads the prompt's last hidden
 * state.  The prompt's full pages enter the radix cache. */
int s2_prefill(s2_ctx* ctx, int32_t seq, const int32_t* tokens, int32_t T,
               const int32_t* vq_codes, const uint8_t* vq_mask, int32_t* cached_len_out);

/* Prefill n free sequences in one call, with the same result as calling
 * s2_prefill for seqs[0], seqs[1], ... in that order: each prompt reuses the
 * longest cached prefix, including pages that an earlier prompt of the same
 * call inserts.  The uncached rows of many prompts share each pass over the
 * Slow AR weights (one pass per group of at most max_batch prompts and
 * prefill_rows rows; a prompt that would reuse pages of a prompt still
 * pending in the group starts the next group).
 *   seqs      int32 [n], distinct free sequence ids
 *   lengths   int32 [n], each in [1, max_prompt]
 *   tokens    int32 [sum of lengths], the prompts one after another
 *   vq_codes  int32, prompt i's [n_codebooks, lengths[i]] block after those
 *             of prompts 0..i-1; read as in s2_prefill (NULL if no mask)
 *   vq_mask   uint8 [sum of lengths] or NULL
 *   cached_out int32 [n] or NULL: each prompt's cached positions (-1 for a
 *             prompt not prefilled because the call failed)
 * Arguments are validated before anything is computed (S2_EINVAL /
 * S2_ESTATE, nothing changed).  S2_ENOMEM when the page pool cannot admit a
 * prompt even after eviction: the prompts before it are prefilled (as by
 * separate calls), it and the rest are not.  Floating-point results may
 * differ from separate calls in the last bits (the kernels' tiling depends on
 * the number of rows per pass). */
int s2_prefill_batch(s2_ctx* ctx, int32_t n, const int32_t* seqs, const int32_t* tokens,
                     const int32_t* lengths, const int32_t* vq_codes, const uint8_t* vq_mask,
                     int32_t* cached_out);

/* Decode ``n`` greedy frames for each of ``batch`` live sequences.  A frame
 * is one Slow AR step over the paged KV cache whose head, restricted to the
 * semantic ids, gives code 0 ("SGLang Day-0 Support for FishAudio S2",
 * Background and Motivation: constrained decoding), then the Fast AR depth
 * loop seeded by the slow hidden state that emits codes 1..9 ("s2pro-native",
 * What happens to a sentence: ten residual codes, nine greedy steps deep);
 * the frame re-enters the Slow AR as its semantic token's embedding plus its
 * VQ codebook embeddings (same page, Background and Motivation).  A batch
 * may mix freshly prefilled sequences (their first frame reads the prompt's
 * last hidden state) with continuing ones (their first frame runs a slow step
 * on the previous frame): sequences join and leave between calls.
 * out_codes int32 [batch, n, 10] in the order of ``seqs``: code 0 is the
 * semantic code (token - sem_begin), codes 1..9 the Fast AR's.  Pages for all
 * n frames are reserved before any launch; when the pool is short, radix
 * pages no sequence uses are evicted least-recently-used first, and if even
 * evicting all of them would not be enough, nothing is evicted and S2_ENOMEM
 * leaves every sequence and the radix cache unchanged.  A later call
 * continues each sequence.  (Debug sinks, when set, see mixed batches in the
 * internal order: continuing sequences first.) */
int s2_decode_frames(s2_ctx* ctx, const int32_t* seqs, int32_t batch, int32_t n,
                     int32_t* out_codes);

/* Drop the sequence; its private pages return to the pool, shared radix
 * pages stay cached. */
int s2_release(s2_ctx* ctx, int32_t seq);

/* Empty the radix prefix cache: the tree drops its page references; pages no
 * live sequence holds return to the pool.  Live sequences are unaffected. */
int s2_radix_clear(s2_ctx* ctx);

/* Counters and the sticky device error flag (reading it synchronises). */
int s2_stats(s2_ctx* ctx, s2_stats_t* out);

/* Human-readable name of a status code (static storage). */
const char* s2_strerror(int status);

/* Test hooks.  While set, decode runs kernel by kernel (no graphs) and
 * writes, per sequence b and frame f of each later s2_decode_frames call:
 *   logits  float [batch][max_frames][10][codebook_size]: head logits of
 *           code k (k = 0: semantic slice of the tied embedding);
 *   hidden  float [batch][max_frames][d]: the slow hidden (after the final
 *           RMSNorm) that seeds the frame's Fast AR;
 *   layers  float [max_frames][n_slow][batch][d]: the residual stream after
 *           each Slow AR layer of the frame's slow step (frames with a step).
 * Any pointer may be NULL.  Device buffers are written by the kernels
 * directly; host buffers are filled from device copies the library allocates
 * here (sized for max_batch rows) when each decode call returns (the call
 * then synchronises).  Returns S2_ENOMEM when such a copy cannot be
 * allocated (no sink is then set).  Pass all NULL to switch the hooks off. */
int s2_set_debug_sinks(s2_ctx* ctx, float* logits, float* hidden, float* layers,
                       int32_t max_frames);

/* Sampling instead of greedy picks for later decode calls.  Code k of a frame
 * is argmax_i(logit_i / T + G_i) -- a draw from softmax(logits / T) by the
 * Gumbel-max rule -- with T = temperature_slow for code 0 (over the semantic
 * ids) and temperature_fast for codes 1..9; T = 0 keeps the greedy pick.
 * G_i = -ln(-ln U_i), U_i from Philox4x32-10 with key = seed and counter =
 * (i / 4, k, position of the slow step that produced the frame, sequence id),
 * word i % 4, as an odd multiple of 2^-24 -- so every draw is reproducible.
 * The pages name no sampling parameters (the SGLang page's appendix mentions
 * early-EOS divergence only), so this is a reading; see also s2_set_top_p and
 * s2_set_stop. */
int s2_set_sampling(s2_ctx* ctx, float temperature_slow, float temperature_fast, uint64_t seed);

/* Nucleus (top-p) filtering of the sampled draws (temperature > 0): with
 * v = logits / T and p = softmax(v), the kept candidates are those whose v is
 * at least the k-th largest, k the first rank at which the cumulative p of the
 * sorted candidates reaches top_p (ties at the cut all kept); the Gumbel-max
 * draw above is taken over them.  top_p in (0, 1]; 1 (the default) keeps
 * every candidate.  A reading, like the sampling itself: the pages give no
 * sampling parameters.  Returns S2_EINVAL outside (0, 1]. */
int s2_set_top_p(s2_ctx* ctx, float top_p_slow, float top_p_fast);

/* Stopping on an end-of-speech token ("SGLang Day-0 Support for FishAudio
 * S2", Engineering Appendix: decoding ends when the model emits EOS, which
 * the wrong attention backend made happen early).  With eos_token >= 0 the
 * Slow head's constrained set gains that token's row of the tied embedding
 * after the semantic ids (ties go to the semantic ids).  A sequence whose
 * frame picks it emits S2_CODE_EOS for all codebooks of that frame and of
 * every later frame of the call, and is finished: decoding it again returns
 * S2_ESTATE; release it.  eos_token must be a text token (below the semantic
 * range), else S2_EINVAL; eos_token < 0 (the default) turns stopping off. */
#define S2_CODE_EOS (-1)
int s2_set_stop(s2_ctx* ctx, int32_t eos_token);

/* Model dimensions of a loaded context: d, n_heads, n_kv, head_dim, ffn,
 * n_slow, n_fast, vocab, sem_begin, n_codebooks, codebook_size, weight dtype
 * (0 f32, 1 bf16) -- 12 ints. */
int s2_model_dims(s2_ctx* ctx, int32_t* dims12);

#ifdef __cplusplus
}
#endif
#endif /* S2_H_ */
