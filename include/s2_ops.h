/*
 * s2_ops.h -- per-kernel C ABI of libs2.so, for kernel-level parity tests
 * and for callers that drive the Dual-AR layers themselves.
 *
 * Every pointer argument is DEVICE memory owned by the caller; nothing is
 * allocated.  Work is enqueued on ``stream`` (a cudaStream_t, NULL = legacy
 * default stream).  Returns S2_OK (0) or a negative S2_E* status from s2.h:
 * S2_EINVAL for shapes the kernels do not support (stated per call), S2_ECUDA
 * when the launch fails.  Matrices are row-major; "ld" is a row pitch in
 * elements.
 */
#ifndef S2_OPS_H_
#define S2_OPS_H_

#include <stddef.h>
#include <stdint.h>

#include "s2.h"

#ifdef __cplusplus
extern "C" {
#endif

/* K1 -- weight-streaming GEMV on CUDA cores.
 *   Y[b, n] (op)= sum_k W[n, k] * a[b, k],  b < B (1..8), n < N
 * with a = RMSNorm(X[b]) * gain (eps) when gain != NULL, else a = X[b]
 * ("s2pro-native", Where it stands: at batch 1 a frame is bound by reading
 * every weight once; "SGLang Day-0 ...", Architecture: Qwen3-style blocks,
 * whose projections are preceded by RMSNorm).
 *   W: [N, K] bf16 (w_bf16 = 1) or fp32; K % 8 == 0, rows 16-byte aligned.
 *   X: fp32 [B, ldx]; Y: fp32.
 *   mode 0: Y[b, n] = y;  1: Y[b, n] += y (residual);
 *   mode 2: rows (2i, 2i+1) hold (gate_i, up_i): Y[b, i] = silu(gate) * up
 *   (SwiGLU MLP), N even.
 *   grid_ctas: CTAs to launch (0 = one per SM). */
int s2op_gemv(const void* W, int w_bf16, int N, int K, const float* X, int ldx, int B,
              const float* gain, float eps, float* Y, int ldy, int mode, int grid_ctas,
              void* stream);

/* K6 -- constrained greedy head: codes[b] = argmax_n sum_k W[n, k] a[b, k]
 * (a as in s2op_gemv), ties to the lowest n ("SGLang Day-0 ...",
 * Background: constrained decoding restricts the head to the legal ids; the
 * caller passes only those rows).  logits (optional, fp32 [B, N]) receives
 * the scores.  workspace: at least s2op_argmax_workspace_bytes(B) bytes of
 * zero-initialised device memory; it is left zeroed again on exit. */
size_t s2op_argmax_workspace_bytes(int B);
int s2op_gemv_argmax(const void* W, int w_bf16, int N, int K, const float* X, int ldx, int B,
                     const float* gain, float eps, int32_t* codes, float* logits,
                     void* workspace, void* stream);

/* K2 -- tcgen05 tensor-core GEMM (bf16 in, fp32 accumulate):
 *   Y[t, n] (op)= sum_k A[n, k] * Bm[t, k],  t < T, n < N
 *   A: bf16 [N, K] (weights), Bm: bf16 [T, ldb] (activations), both
 *   16-byte aligned; N % 128 == 0, K % 64 == 0, ldb % 8 == 0.
 *   epi 0: Y = y;  1: Y += y;  2: SwiGLU of interleaved (gate, up) rows into
 *   bf16 Y16[t, n/2] (the MLP of the S2 blocks).
 *   split_k: 0 = automatic; otherwise the number of K splits (at most K/64;
 *   split s covers 64-wide k-tiles [s*kt/S, (s+1)*kt/S) of the kt = K/64,
 *   summed in split order).  With more than one split, workspace (fp32, at least
 *   s2op_tc_gemm_workspace_bytes) and tickets (zeroed, at least
 *   s2op_tc_gemm_tickets) are required; tickets are zero again on exit. */
size_t s2op_tc_gemm_workspace_bytes(int N, int K, int T, int split_k);
size_t s2op_tc_gemm_tickets(int N, int T);
int s2op_tc_gemm(const void* A, int N, int K, const void* Bm, int T, int ldb, float* Y, int ldy,
                 void* Y16, int ldy16, int epi, int split_k, float* workspace, uint32_t* tickets,
                 void* stream);

/* K2, two-plane operand: as s2op_tc_gemm but the activations arrive as a bf16
 * pair (Bhi, Blo) with x ~= Bhi + Blo (Blo = bf16(x - Bhi)), and the kernel
 * accumulates A*Bhi + A*Blo -- ~16 mantissa bits of the activations at twice
 * the tensor work and the same weight traffic.  For epi 2 the bf16 output is
 * written the same way: Y16 (hi) and, when non-NULL, Y16lo (remainder).
 * Token tiles are at most 128 wide in this mode; workspace and tickets as
 * given by the *_2 size queries. */
size_t s2op_tc_gemm2_workspace_bytes(int N, int K, int T, int split_k);
size_t s2op_tc_gemm2_tickets(int N, int T);
int s2op_tc_gemm2(const void* A, int N, int K, const void* Bhi, const void* Blo, int T, int ldb,
                  float* Y, int ldy, void* Y16, void* Y16lo, int ldy16, int epi, int split_k,
                  float* workspace, uint32_t* tickets, void* stream);

/* K2 phase trace (diagnostics): every later K2 launch of the process has
 * each CTA c write six globaltimer stamps (ns, uint64) to buf[6c .. 6c+5]:
 * kernel entry, setup done (barriers, tensor memory, programmatic-launch
 * wait), first operand stage landed, last MMA issued, accumulator complete,
 * epilogue done.  buf: device memory of max_ctas * 48 bytes; CTAs with a
 * linear index >= max_ctas write nothing.  max_ctas = 0 turns it off.
 * S2_EINVAL for a NULL buf with max_ctas > 0. */
int s2op_tc_set_trace(void* buf, int max_ctas);

/* K3 + K4 -- decode attention over a paged KV cache for B sequences with m
 * (1 or 2) new rows each ("SGLang Day-0 ...", Optimizations: paged KV cache;
 * Engineering Appendix: bf16-rounded RoPE table).  For row i of sequence b at
 * position p = pos[b] + i:
 *   q_h, k, v from qkv[(b*m + i), :] = [q (H*hd) | k (Hkv*hd) | v (Hkv*hd)];
 *   q_h, k <- RMSNorm per head (gains q_gain, k_gain [hd]) then rotate-half
 *   RoPE with rope_cos/rope_sin [positions][hd/2];
 *   k, v are written to slot p % 16 of page table[b*table_ld + p/16];
 *   o[b*m+i, h] = softmax_j(q_h . k_j / sqrt(hd)) v_j over keys j <= p of kv
 *   head h / (H/Hkv).
 * kv: one layer's pool, pages of [2][Hkv][16][hd] (kv_bf16 = 1: bf16, else
 * fp32).  Supported: (hd, H/Hkv) = (128, 4) or (64, 2).  nsplit >= 1 splits
 * the keys across CTAs (32-key chunks); the splits are merged in fixed order.
 * A sequence with at most 64 keys (p + 1 for its last row) is attended by one
 * split whatever nsplit is, so its rows round as with nsplit = 1.  workspace:
 * s2op_attn_decode_workspace_bytes(...) bytes, zero-initialised (zero again
 * on exit); may be NULL when nsplit == 1.  o: fp32 [B*m, o_ld]. */
size_t s2op_attn_decode_workspace_bytes(int B, int m, int H, int Hkv, int hd, int nsplit);
/* The key-split count the model path takes for B sequences on this device:
 * within one wave of resident CTAs, enough CTAs for twice the SMs and up to
 * as many as the wave holds; past one wave, the fewest splits (at most 16)
 * whose waves are at least 90% full.  A negative status for bad sizes. */
int s2op_attn_decode_pick_split(int B, int H, int Hkv, int hd, int kv_bf16);
int s2op_attn_decode(const float* qkv, int qkv_ld, int B, int m, int H, int Hkv, int hd,
                     const float* q_gain, const float* k_gain, float eps, const float* rope_cos,
                     const float* rope_sin, const int32_t* pos, void* kv, int kv_bf16,
                     const int32_t* table, int table_ld, float* o, int o_ld, int nsplit,
                     void* workspace, void* stream);

/* K11 + K3/K4 -- decode attention (m = 1 new row per sequence) for B
 * sequences whose page tables share their first ``shared_len`` keys (whole
 * 16-token pages: one radix-cached prompt prefix, "SGLang Day-0 ...",
 * Optimizations with SGLang Omni: radix prefix caching).  The same result as
 * s2op_attn_decode: the keys from shared_len on (each sequence's own, with
 * the appended new key) by the split-KV decode attention, which leaves its
 * partials; the keys below shared_len on the tcgen05 tensor cores, once per
 * kv head for all B x 4 query rows (128-row tiles; products of bf16 hi/lo
 * operand planes, fp32 accumulation), in thread-block clusters of 8 CTAs
 * that merge their partials with the split-KV ones (in key order) into o.
 * Supported: hd 128, H = 4 Hkv.  max_keys bounds every context (sizes the
 * workspace); shared_len a multiple of 16, at most max_keys.
 *
 * workspace: s2op_attn_decode_prefix_workspace_bytes zero-initialised bytes
 * (its tickets are zero again on exit).  Its first part holds the shared
 * keys as the MMAs' operand images: s2op_attn_prefix_planes writes them
 * from the pages (table row 0 must hold the shared pages), and
 * s2op_attn_decode_shared_prefix reads them, so call s2op_attn_prefix_planes
 * (same kv, kv_bf16, table, Hkv, hd, shared_len, max_keys, workspace) first,
 * and again whenever those pages change.  s2op_attn_decode_shared_prefix
 * synchronises ``stream`` once (it uploads shared_len).  S2_EINVAL for
 * unsupported shapes or a shared_len that is not a multiple of 16 (below 16
 * for s2op_attn_prefix_planes). */
size_t s2op_attn_decode_prefix_workspace_bytes(int B, int H, int Hkv, int hd, int nsplit, int max_keys);
int s2op_attn_prefix_planes(const void* kv, int kv_bf16, const int32_t* table, int Hkv, int hd, int shared_len,
                            int max_keys, void* workspace, void* stream);
int s2op_attn_decode_shared_prefix(const float* qkv, int qkv_ld, int B, int H, int Hkv, int hd,
                                   const float* q_gain, const float* k_gain, float eps,
                                   const float* rope_cos, const float* rope_sin, const int32_t* pos,
                                   void* kv, int kv_bf16, const int32_t* table, int table_ld,
                                   int shared_len, int max_keys, float* o, int o_ld, int nsplit,
                                   void* workspace, void* stream);

/* Phase trace of the shared-prefix tensor-core kernel (measurement only):
 * while on, each launch's CTA i < max_ctas (i = (tile * Hkv + kv head) * 8 +
 * cluster rank) writes 16 uint64 globaltimer stamps (ns) to device memory
 * ``buf`` + 16 i: entry, after setup, after the wait on the previous launch,
 * after issuing the query tile's copy, operands of its first chunk landed,
 * after S = Q K^T, after the softmax, after O = P V, after its last chunk,
 * after the first cluster barrier, after the merge, at exit (slots 12-15
 * unused; stamps of phases a CTA skips stay as they were).  max_ctas 0 turns
 * it off.  S2_EINVAL for max_ctas < 0 or a NULL buf with max_ctas > 0. */
int s2op_attn_prefix_set_trace(void* buf, int max_ctas);

/* K9 -- prefill attention for T new rows of one sequence at positions
 * pos0 .. pos0+T-1 whose q/k/v are in qkv (layout as above): q/k norm +
 * RoPE, K/V appended to the sequence's pages, then causal attention over all
 * keys 0 .. pos0+T-1 (keys before pos0 come from cached -- e.g. radix-shared
 * -- pages and are not recomputed).  q_scratch: fp32 [T, H*hd].  o: fp32
 * [T, o_ld]. */
int s2op_attn_prefill(const float* qkv, int qkv_ld, int T, int pos0, int H, int Hkv, int hd,
                      const float* q_gain, const float* k_gain, float eps, const float* rope_cos,
                      const float* rope_sin, void* kv, int kv_bf16, const int32_t* table,
                      float* q_scratch, float* o, int o_ld, void* stream);

/* RoPE table of the S2 blocks: cos/sin of p * theta^(-2i/hd) for p < n_pos,
 * i < hd/2, rounded to float then to bf16 (ties to even), stored as fp32
 * ("SGLang Day-0 ...", Engineering Appendix: BF16 RoPE Precision Mismatch).
 * Host buffers of n_pos*hd/2 floats each. */
int s2op_rope_table(int n_pos, int hd, float theta, float* cos_out, float* sin_out);

/* HBM read-bandwidth calibration: streams n_ops device buffers (bufs[i],
 * bytes[i] bytes, 16-byte aligned, bytes % 16 == 0; bufs and bytes are HOST
 * arrays of n_ops entries, read during the call) reps times over and
 * discards the data ("s2pro-native", Where it stands: a decode frame is
 * bound by how fast the weights can be read, so this is the stream to
 * compare the weight-streaming kernels against).
 *   mode 0: one launch per buffer, each thread eight 16-byte loads in flight;
 *   mode 1: one persistent launch (one CTA per SM): a producer thread copies
 *     the CTA's contiguous share of each buffer into a ring of ``stages``
 *     shared-memory chunks of ``chunk_bytes`` (bulk copies by the TMA engine,
 *     chunk_bytes * stages <= 200 KB), consumer warps read and release them;
 *     barrier != 0 puts a grid barrier before each buffer on the consumer
 *     side only (a dependent chain of operations), the producer streams on.
 * scratch: device memory of s2op_stream_read_scratch_bytes(n_ops) bytes,
 * owned by the caller.  err_out (host, may be NULL): receives the kernel's
 * error word (0 = ok, nonzero = a bounded wait gave up); reading it
 * synchronises the stream.  Returns S2_EINVAL for bad sizes, S2_ECUDA when a
 * launch fails. */
size_t s2op_stream_read_scratch_bytes(int n_ops);
int s2op_stream_read(const void* const* bufs, const unsigned long long* bytes, int n_ops, int reps,
                     int mode, int chunk_bytes, int stages, int barrier, void* scratch,
                     int* err_out, void* stream);

/* Decode attention without any allocation -- no counterpart on the pages;
 * an addition of this library.  Same arguments and results as
 * s2op_attn_decode, minus the workspace.  It is meant for callers that
 * cannot allocate device memory themselves: a real-time audio thread, where
 * cudaMalloc/cudaFree may block on the driver or synchronise the device in
 * the middle of a frame, or a host whose device memory is owned by another
 * allocator (a framework's caching pool, a fixed per-plugin budget).
 *   Scratch: the split-KV partials and tickets live in a file-scope device
 *   array of S2_NOALLOC_SCRATCH_BYTES (8 MiB) that every GPU loading the
 *   library holds until the process exits.  A call needing more --
 *   B*m*H*nsplit*(hd+2)*4 bytes of partials plus B*Hkv*4 bytes of tickets,
 *   the tickets on a 256-byte boundary -- returns S2_EINVAL
 *   (s2op_attn_decode_noalloc_max_bytes() reports the limit).
 *   Set-up: the first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current); make that first call
 *   before any stream capture.  The address is kept per device index and is
 *   valid only within the device's current primary context: after
 *   cudaDeviceReset (or anything else that destroys that context) the kept
 *   address is stale, so do not call this entry point again in that process.
 *   Sharing: every call uses the same array, which keeps the previous
 *   call's contents; each call clears its tickets itself (a memset on
 *   ``stream``).  Calls whose work overlaps on the GPU -- e.g. on two
 *   streams -- race on the array and must be serialised by the caller.
 *   No cudaMalloc, cudaFree or allocating library routine is called. */
#define S2_NOALLOC_SCRATCH_BYTES (8u << 20)
size_t s2op_attn_decode_noalloc_max_bytes(void);
int s2op_attn_decode_noalloc(const float* qkv, int qkv_ld, int B, int m, int H, int Hkv, int hd,
                             const float* q_gain, const float* k_gain, float eps,
                             const float* rope_cos, const float* rope_sin, const int32_t* pos,
                             void* kv, int kv_bf16, const int32_t* table, int table_ld, float* o,
                             int o_ld, int nsplit, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* S2_OPS_H_ */
