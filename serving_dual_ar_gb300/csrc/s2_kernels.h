// Internal declarations of the sm_103a kernels and their host launchers.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <vector>

namespace s2 {

// Kernels launched by this library on the calling thread (for launch accounting).
extern thread_local long long g_launch_count;

// cudaLaunchKernelEx that counts successful launches.
template <typename... K, typename... A>
inline cudaError_t s2_launch(const cudaLaunchConfig_t* cfg, void (*k)(K...), A&&... args) {
  cudaError_t e = cudaLaunchKernelEx(cfg, k, static_cast<A&&>(args)...);
  if (e == cudaSuccess) ++g_launch_count;
  return e;
}

// Frame timeline: CTAs per launch whose stamps are kept.
constexpr int kFrameTraceCtas = 160;
// Decode attention: a key range of at most this many keys (no shared-prefix
// slots) is attended by one split whatever the launch's split count.
constexpr int kAttnOneSplitKeys = 64;
// ------------------------------------------------------------------ K1 GEMV
enum GemvMode { GEMV_STORE = 0, GEMV_ADD = 1, GEMV_SWIGLU = 2, GEMV_ARGMAX = 3 };

struct GemvArgs {
  const void* W = nullptr;  // [N, K] row-major weights
  int w_is_bf16 = 1;
  int w_int8 = 0;               // int8 weights with per-row scales (overrides w_is_bf16)
  const float* wscale = nullptr;
  int N = 0, K = 0;
  int unit = 1;             // rows kept together on one CTA (2 for gate/up pairs)
  const float* X = nullptr; // [B, ldx] activations (fp32)
  int ldx = 0;
  int B = 1;                // batch rows, 1..8
  const float* gain = nullptr;  // RMSNorm gain [K]; null = no norm prologue
  float eps = 1e-6f;
  float* normed_out = nullptr;  // CTA 0 writes the normalised x rows here
  int normed_ld = 0;
  float* Y = nullptr;       // output rows (ldy)
  int ldy = 0;
  int mode = GEMV_STORE;
  // arg-max mode
  float* part_val = nullptr;   // [B][grid]
  int* part_idx = nullptr;
  unsigned* ticket = nullptr;  // zero on entry, reset to zero on exit
  float* logits = nullptr;     // optional sink [B][logits_ld]
  int logits_ld = 0;
  int* codes = nullptr;        // codes[b*codes_ld + frame*codes_per_frame + code_slot]
  int codes_ld = 0, codes_per_frame = 10, code_slot = 0;
  const int* frame = nullptr;  // device frame counter (null = 0)
  int* last_codes = nullptr;   // [B][codes_per_frame]
  int* frame_inc = nullptr;    // incremented once by the last CTA
  int tail_d = 0;              // row length for the tail copies
  const float* copy_src = nullptr; int copy_src_ld = 0;
  float* copy_dst = nullptr; int copy_dst_ld = 0;
  const void* emb_next = nullptr; int emb_is_bf16 = 1;  // [C][tail_d] table
  float* emb_dst = nullptr; int emb_dst_ld = 0;
  int* err = nullptr;
  // frame timeline (measurement): thread 0 of CTA c < kFrameTraceCtas stamps
  // the global timer into trace[4 c .. 4 c + 3] (entry, after the wait on the
  // previous kernel, after the prologue, exit); null = off
  unsigned long long* trace = nullptr;
  // temperature sampling of the arg-max (0: greedy): pick argmax(y / T + Gumbel)
  float temperature = 0.f;
  unsigned long long seed = 0;
  const int* samp_seq = nullptr;       // [B] sequence ids
  const int* samp_pos = nullptr;       // [B] position base; + *frame
};

// Streaming layout of one GEMV launch (host-computed, passed to the kernel).
struct GemvLayout {
  int KS, NSEG, slot_bytes, spw, rows_max, smem, warps, hint;
  int ring_off, xs_off, res_off, part_off, bar_off;
  int xstage;  // activations staged in shared memory (always with the RMSNorm prologue)
  int kp;      // row stride of the staged activations (floats, multiple of 256)
};

int gemv_grid(const GemvArgs& a, int num_sms);
int gemv_max_grid(int num_sms);  // upper bound of gemv_grid over all arguments
cudaError_t launch_gemv(const GemvArgs& a, cudaStream_t st, bool pdl, int grid);

// ------------------------------------------------------------------ K3+K4 decode attention
struct AttnDecodeArgs {
  const float* qkv = nullptr; int qkv_ld = 0;  // rows b*m + i: [q | k | v]
  int B = 1, m = 1;         // sequences, new rows per sequence (1 or 2)
  int H = 0, Hkv = 0, hd = 0;
  const float* q_gain = nullptr; const float* k_gain = nullptr; float eps = 1e-6f;
  const float* rope_cos = nullptr; const float* rope_sin = nullptr;  // [pos][hd/2]
  const int* pos_base = nullptr;   // first new position = pos_base[b] + *frame + pos_off
  const int* frame = nullptr;
  int pos_off = 0;
  void* kv = nullptr;       // this layer's page pool base
  int kv_bf16 = 1;
  long long page_elems = 0; // elements per page (2 * Hkv * 16 * hd)
  const int* table = nullptr; int table_ld = 0;  // page table (null: page = b)
  float* o = nullptr; int o_ld = 0;              // fp32 output rows (optional)
  __nv_bfloat16* o16 = nullptr; int o16_ld = 0;  // bf16 output rows (optional)
  __nv_bfloat16* o16lo = nullptr;                // bf16 remainder rows (optional, same ld)
  int nsplit = 1;
  float* part = nullptr;       // [B*m][H][part_base + nsplit][hd+2]
  unsigned* tickets = nullptr; // [B][Hkv], zero on entry
  int* err = nullptr;
  // shared prefix: keys below *key_begin (device word; null = 0) are not
  // this launch's: the splits cover keys key_begin.., after part_base slots
  // filled by another launch, and the merge adds all part_base + nsplit
  // slots in slot order
  const int* key_begin = nullptr;
  int part_base = 0;
  // 1: the splits only write their partial slots (no ticket, no merge; even
  // with one split); a later launch merges them (launch_attn_prefix_cl)
  int merge_later = 0;
  unsigned long long* trace = nullptr;   // frame timeline, as GemvArgs::trace
  // m = 1, hd 128, 4 heads per kv head: split 0 of (b, g) also writes the
  // 4 query rows b*4 .. b*4+3 of kv head g (normalised, rotated, scaled by
  // 1/sqrt(hd)) as the shared-prefix attention's query operand: per (g,
  // 128-row tile t) 64 KB = [hi, lo][k-block][128 rows][128 B], 128-byte
  // swizzled, at q_img + (g * tiles + t) * 64 KB (tiles = ceil(4 B / 128))
  uint8_t* q_img = nullptr;
};
// Bytes of the query images for B sequences and Hkv kv heads.
size_t attn_prefix_qimg_bytes(int B, int Hkv);
cudaError_t launch_attn_decode(const AttnDecodeArgs& a, cudaStream_t st, bool pdl);
// Decode-attention CTAs that fit one SM (occupancy of the stand-alone kernel).
int attn_decode_ctas_per_sm(int hd, int group, bool kv_bf16);
// Key splits per (sequence, kv head): within one wave of resident CTAs,
// enough CTAs for twice the SMs and up to as many as the wave holds; beyond
// one wave, the fewest splits whose waves are at least 90% full (at most
// max_split).
int attn_pick_split(int B, int Hkv, int num_sms, int ctas_per_sm, int max_split);
size_t attn_decode_scratch_floats(int B, int m, int H, int hd, int nsplit);
// K11, tensor-core attention over a batch's shared prefix (k_attn_prefix.cu).
// The prefix keys 0 .. P-1 of every (layer, kv head), converted once per
// decode call into the operand images the MMAs read: bf16 hi / lo planes in
// the 128-byte swizzled K-major layout (keys; values transposed), ``stride``
// keys per (layer, kv head) (a multiple of 128), 8 * hd bytes per key; keys
// P .. round_up(P, 128) - 1 are written as zeros.
struct PrefixPlanesArgs {
  const void* kv = nullptr;     // page pool of layer 0
  long long layer_bytes = 0;    // bytes from one layer's pool to the next
  int kv_bf16 = 0;
  long long page_elems = 0;     // elements per page (2 * Hkv * 16 * hd)
  const int* table = nullptr;   // the shared pages (any row holding them)
  int Hkv = 0, hd = 0, layers = 1;
  int P = 0;                    // shared keys (a multiple of 16, <= stride)
  int stride = 0;               // keys per (layer, kv head) in the images
  void* planes = nullptr;       // layers x Hkv images
};
size_t attn_prefix_plane_bytes(int Hkv, int hd, int stride, int layers);
int attn_prefix_plane_stride(int max_keys);
cudaError_t launch_attn_prefix_planes(const PrefixPlanesArgs& p, cudaStream_t st);
// The attention of a.B sequences (m = 1, hd 128, 4 heads per kv head) over
// the shared keys 0 .. *a.key_begin - 1 from one layer's images (planes,
// stride), merged with the a.nsplit partial slots a split-KV decode launch
// (key_begin, part_base 0, merge_later) left for the later keys: writes the
// normalised rows to a.o and / or a.o16 + a.o16lo.  Grid (8, Hkv, query
// tiles of 128 rows) in clusters of 8 CTAs.
cudaError_t launch_attn_prefix_cl(const AttnDecodeArgs& a, const void* planes, int stride, cudaStream_t st,
                                  bool pdl);
// Phase trace of launch_attn_prefix_cl's kernel: 16 globaltimer slots per
// CTA (CTA index (z * Hkv + g) * 8 + rank) into device ``buf`` for the first
// ``max_ctas`` CTAs of the launches that follow; max_ctas 0 turns it off.
void attn_prefix_set_trace(unsigned long long* buf, int max_ctas);

// ------------------------------------------------------------------ prefill: q/k norm, RoPE, KV append
// Several sequences' prefill rows concatenated (batched prefill): segment i
// = info[5i .. 5i+4] = {first row, rows, position of its first row, offset of
// its page table in ``tables``, first 32-token query tile}; row_seg[row] and
// tile_seg[tile] name the segment of a row / query tile.  info == null: one
// sequence (the arguments' own T, pos0, table).
struct PrefillSegs {
  const int* info = nullptr;
  const int* row_seg = nullptr;
  const int* tile_seg = nullptr;
  const int* tables = nullptr;
  int n_tiles = 0;
};

struct QkRopeArgs {
  const float* qkv = nullptr; int qkv_ld = 0;  // T rows
  int T = 0, pos0 = 0;      // row t sits at position pos0 + t
  int H = 0, Hkv = 0, hd = 0;
  const float* q_gain = nullptr; const float* k_gain = nullptr; float eps = 1e-6f;
  const float* rope_cos = nullptr; const float* rope_sin = nullptr;
  void* kv = nullptr; int kv_bf16 = 1; long long page_elems = 0;
  const int* table = nullptr;  // this sequence's page table
  float* q_out = nullptr;      // [T][H*hd] fp32, pre-scaled by 1/sqrt(hd)
  PrefillSegs segs;            // batched: T = all rows, per-row position and table
};
cudaError_t launch_qk_rope_append(const QkRopeArgs& a, cudaStream_t st, bool pdl);

// ------------------------------------------------------------------ K9 prefill attention
struct AttnPrefillArgs {
  const float* q = nullptr;  // [T][H*hd] pre-scaled
  int T = 0, pos0 = 0;       // query t at position pos0 + t; keys 0..pos0+T-1 in pages
  int H = 0, Hkv = 0, hd = 0;
  const void* kv = nullptr; int kv_bf16 = 1; long long page_elems = 0;
  const int* table = nullptr;
  float* o = nullptr; int o_ld = 0;
  __nv_bfloat16* o16 = nullptr; int o16_ld = 0;
  __nv_bfloat16* o16lo = nullptr;
  // key split (short queries over a long context): ksplit CTAs per (query
  // tile, head) each take a contiguous range of 64-key tiles; the last one
  // merges the partials in split order.  part: attn_prefill_part_floats()
  // floats; tickets: [query tiles][H], zero on entry, zero again on exit.
  int ksplit = 1;
  float* part = nullptr;
  unsigned* tickets = nullptr;
  int* err = nullptr;        // device error word (tensor-core kernel's bounded waits)
  int tc = 1;                // take the tcgen05 kernel where it applies
  PrefillSegs segs;          // batched (tcgen05 kernel only): T = all rows, q / o rows global
};
cudaError_t launch_attn_prefill(const AttnPrefillArgs& a, cudaStream_t st, bool pdl);
// The same attention on tcgen05 (hd 128, 4 heads per kv head): 32-token x 4
// head query tiles, 64-key chunks, online softmax (k_attn_tc.cu).
bool attn_prefill_tc_supported(const AttnPrefillArgs& a);
// Batched prefill attention on tcgen05 (a.segs set): one launch over every
// segment's query tiles.  cudaErrorNotSupported when the tcgen05 kernel does
// not apply (the caller then launches segment by segment).
cudaError_t launch_attn_prefill_segs(const AttnPrefillArgs& a, cudaStream_t st, bool pdl);
cudaError_t launch_attn_prefill_tc(const AttnPrefillArgs& a, cudaStream_t st, bool pdl);
size_t attn_prefill_part_floats(int T, int H, int hd, int ksplit);

// ------------------------------------------------------------------ K8 embedding
struct EmbedArgs {
  const void* tok_emb = nullptr; const void* vq_emb = nullptr; int w_bf16 = 1;
  int d = 0, n_codebooks = 10, codebook_size = 0, sem_begin = 0;
  int rows = 0;
  // prompt mode: tokens[r], codes[k*codes_ld + r], mask[r]
  const int* tokens = nullptr; const int* codes = nullptr; int codes_ld = 0;
  const uint8_t* mask = nullptr;
  // feedback mode (tokens == null): frame codes fb[r*n_codebooks + k], token sem_begin + fb[r*nc]
  const int* fb = nullptr;
  float* out = nullptr; int out_ld = 0;
};
cudaError_t launch_embed(const EmbedArgs& a, cudaStream_t st, bool pdl);

// ------------------------------------------------------------------ K6 arg-max over logit rows
// (batched heads: logits come from the tensor-core GEMM)
struct ArgmaxRowsArgs {
  const float* logits = nullptr; int ld = 0; int rows = 0; int C = 0;
  float* sink = nullptr; int sink_ld = 0;           // optional copy of the logits
  int* codes = nullptr; int codes_ld = 0, codes_per_frame = 10, code_slot = 0;
  const int* frame = nullptr;
  int* last_codes = nullptr;
  int* frame_inc = nullptr;
  unsigned* ticket = nullptr;                       // needed with frame_inc
  int d = 0;
  const float* copy_src = nullptr; int copy_src_ld = 0;
  float* copy_dst = nullptr; int copy_dst_ld = 0;
  const void* emb_next = nullptr; int emb_is_bf16 = 1;
  float* emb_dst = nullptr; int emb_dst_ld = 0;
  float temperature = 0.f;
  unsigned long long seed = 0;
  const int* samp_seq = nullptr;
  const int* samp_pos = nullptr;
  float top_p = 1.f;                 // nucleus filter of the sampled draw (1: off)
  // end of speech: with eos_row set, candidate C is that embedding row's
  // logit against the normalised hidden rows h; a row that picks it (or whose
  // done flag is already set) writes code -1, feeds back code 0, sets done
  const void* eos_row = nullptr; int eos_bf16 = 1;
  const float* h = nullptr; int h_ld = 0;
  int* done = nullptr;               // [rows] finished flags (read with or without eos_row)
};
cudaError_t launch_argmax_rows(const ArgmaxRowsArgs& a, cudaStream_t st, bool pdl);

// ------------------------------------------------------------------ INT8 row quantisation
// q[n,k] = rint(w[n,k] / s_n), s_n = max_k |w[n,k]| / 127 (1 for a zero row)
cudaError_t launch_quantize_rows(const void* W, int w_bf16, int N, int K, int8_t* Q, float* S,
                                 cudaStream_t st);

// ------------------------------------------------------------------ RMSNorm rows
struct RmsRowsArgs {
  const float* x = nullptr; int ldx = 0; int rows = 0, d = 0;
  const float* gain = nullptr; float eps = 1e-6f;
  float* out = nullptr; int out_ld = 0;               // optional fp32
  __nv_bfloat16* out16 = nullptr; int out16_ld = 0;  // optional bf16
  __nv_bfloat16* out16lo = nullptr;                  // optional bf16 remainder (same ld)
  unsigned long long* trace = nullptr;               // frame timeline, as GemvArgs::trace
};
cudaError_t launch_rms_rows(const RmsRowsArgs& a, cudaStream_t st, bool pdl);

// Row copy/gather of fp32 rows: dst[i] = src[idx[i]] (idx null: identity).
cudaError_t launch_gather_rows(float* dst, int dst_ld, const float* src, int src_ld,
                               const int* idx, int rows, int d, cudaStream_t st, bool pdl);
cudaError_t launch_gather_rows_i32(int* dst, int dst_ld, const int* src, int src_ld,
                                   const int* idx, int rows, int d, cudaStream_t st, bool pdl);
cudaError_t launch_scatter_rows_i32(int* dst, int dst_ld, const int* src, int src_ld,
                                    const int* idx, int rows, int d, cudaStream_t st, bool pdl);
cudaError_t launch_scatter_rows(float* dst, int dst_ld, const float* src, int src_ld,
                                const int* idx, int rows, int d, cudaStream_t st, bool pdl);

// ------------------------------------------------------------------ K2 tcgen05 GEMM
// Y[t, n] (+)= sum_k A[n, k] * Bm[t, k];  A = weights [N, K] bf16, Bm = activations
// [T, K] bf16 (both K-major), fp32 accumulation in tensor memory.
enum TcEpi { TC_STORE = 0, TC_ADD = 1, TC_SWIGLU_BF16 = 2 };
struct TcGemmArgs {
  const __nv_bfloat16* A = nullptr; int N = 0, K = 0;
  const __nv_bfloat16* Bm = nullptr; int T = 0; int ldb = 0;
  const __nv_bfloat16* Blo = nullptr;            // remainder plane of Bm (same ldb): D = A (Bm + Blo)
  float* Y = nullptr; int ldy = 0;               // fp32 output (STORE/ADD)
  __nv_bfloat16* Y16 = nullptr; int ldy16 = 0;   // bf16 output (SWIGLU)
  __nv_bfloat16* Y16lo = nullptr;                // bf16 remainder of Y16 (same ld)
  int epi = TC_STORE;
  int split_k = 1;
  float* ws = nullptr;          // split-K partials [split_k][T_pad][N]
  size_t ws_floats = 0;         // capacity of ws (0: unchecked)
  unsigned* tickets = nullptr;  // [N/128 * T tiles], zero on entry
  size_t n_tickets = 0;         // capacity of tickets (0: unchecked)
  int* err = nullptr;
  // frame timeline, as GemvArgs::trace; the four stamps here are entry, after
  // the wait on the previous kernel, accumulator complete, exit
  unsigned long long* trace = nullptr;
};
cudaError_t launch_tc_gemm(const TcGemmArgs& a, cudaStream_t st, bool pdl, int num_sms);
// Phase trace of every K2 launch that follows (null / 0: off): CTA c writes 6
// globaltimer stamps (ns) to buf[c*6..]: entry, setup done (barriers, tensor
// memory, PDL wait), first stage landed, last MMA issued, accumulator
// complete, epilogue done.  CTAs beyond max_ctas write nothing.
void tc_set_trace(unsigned long long* buf, int max_ctas);
int tc_gemm_pick_tn(int T, bool two_plane = false);
void tc_gemm_plan(int N, int K, int T, int num_sms, int* tn, int* split_k, bool two_plane = false);
size_t tc_gemm_ws_floats(int N, int T, int split_k, bool two_plane = false);
size_t tc_gemm_tickets(int N, int T, bool two_plane = false);

// ------------------------------------------------------------------ persistent decode
// One cooperative launch runs whole decode frames: the same sequence of GEMV,
// attention and embedding operations the per-frame CUDA graph launches, with a
// grid barrier between consecutive operations instead of a kernel boundary.
// Each GEMV starts loading its weights before it waits at the barrier, so the
// weight stream runs on through the dependency on the previous operation.
constexpr int kPersistThreads = 512;  // one CTA of 16 warps per SM
constexpr int kPersistVmax = 8;       // 16-byte weight vectors per lane per segment
constexpr int kPersistAttnUnits = kPersistThreads / 128;  // attention units side by side per CTA
// Segments in flight per warp in the persistent GEMV (a cp.async ring in
// shared memory; it shares the CTA's shared memory with the normalised
// activations, which take 4 * maxb * d bytes).
constexpr int persist_adepth(int maxb) { return maxb <= 2 ? 3 : 2; }

enum PersistKind { PK_GEMV = 1, PK_ATTN = 2, PK_EMBED = 3 };
struct alignas(16) PersistOp {
  int kind = 0;
  int grid = 0;     // GEMV: CTAs of the stand-alone launch (<= the persistent grid)
  int maxb = 0;     // GEMV: batch instance (1, 2, 4 or 8)
  int pad = 0;
  GemvArgs g;
  GemvLayout L;
  AttnDecodeArgs at;
  EmbedArgs e;
};

// While installed on the calling thread, launch_gemv, launch_attn_decode and
// launch_embed append their launch here instead of launching; ``ok`` turns
// false when one of them has no persistent counterpart.
struct OpRecorder {
  std::vector<PersistOp> ops;
  int max_grid = 0;   // CTAs of the persistent grid
  bool ok = true;
};
extern thread_local OpRecorder* g_recorder;

// The persistent kernel runs every GEMV with one batch instance MAXB (the
// largest of the program, 1, 2, 4 or 8); a row's arithmetic does not depend
// on MAXB.  gemv_persist_layout re-plans a recorded GEMV for that instance.
bool gemv_persist_layout(PersistOp& op, int maxb);
// Dynamic shared memory the persistent kernel needs for these operations.
size_t persist_smem_bytes(const std::vector<PersistOp>& ops);
// CTAs of the persistent grid that fit on this device (one per SM when the
// kernel fits there, else 0).
int persist_grid(int num_sms, int maxb, size_t smem);
// Run ``n_frames`` passes over ops[0 .. n_ops) (device array).  ``bar`` and
// ``abort_flag``: zeroed device words (the barrier counter, and the flag a CTA
// sets when a barrier wait gives up); ``err``: the sticky device error flag
// (set to 2 on such a timeout).
// ``trace`` (optional, [n_ops][3]): CTA 0's globaltimer (ns) at the start
// of each operation of one frame, when it passed the operation's barrier, and
// at its end.
// ``fault_op`` >= 0 (fault injection): at the barrier before operation
// fault_op of the first frame CTA 0 does not arrive, so every CTA's wait runs
// out; ``budget_ns``: the barrier waits' time budget (0: 2 s).
cudaError_t launch_persist(const PersistOp* ops, int n_ops, int n_frames, int maxb, unsigned* bar,
                           int* abort_flag, int* err, int grid, size_t smem, cudaStream_t st,
                           unsigned long long* trace = nullptr, int fault_op = -1,
                           unsigned long long budget_ns = 0);

// ------------------------------------------------------------------ streaming decode
// One persistent launch over whole decode frames (batch 1-2): a producer warp
// per CTA streams every GEMV's weight rows through a shared-memory ring of
// bulk copies, independent of the grid barriers between operations; 16
// consumer warps run the recorded operations (see k_stream.cu).
struct StreamPlan {        // per recorded operation (GEMV: W set)
  const void* W = nullptr;
  int rowbytes = 0, N = 0, unit = 1;
  int rc = 0;              // weight rows per ring slot
  int parts = 0;           // K-parts per row (one consumer warp each)
  int stage = 0;           // activations staged in shared memory
  int pad = 0;
};
struct StreamLayout {      // consumer work area (bytes, after the ring)
  int res_off = 0, yold_off = 0, part_off = 0, ssq_off = 0, xs_off = 0, work_bytes = 0;
};
bool stream_plan(const std::vector<PersistOp>& ops, int grid, std::vector<StreamPlan>& plan,
                 StreamLayout& L, int& maxb);
size_t stream_smem_bytes(const StreamLayout& L);
bool stream_fits(int maxb, size_t smem);
// n_frames passes over ops; bar / abort_flag zeroed words, err the sticky
// device error word (2 on a wait that gave up); trace as for launch_persist.
cudaError_t launch_stream(const PersistOp* ops, const StreamPlan* plan, int n_ops, int n_frames, int maxb,
                          const StreamLayout& L, unsigned* bar, int* abort_flag, int* err, int grid,
                          cudaStream_t st, unsigned long long* trace = nullptr);

// RoPE table (host): cos/sin of p * theta^(-2i/hd), rounded to float and then
// to bf16 with ties to even ("SGLang Day-0 Support for FishAudio S2",
// Engineering Appendix: BF16 RoPE Precision Mismatch).
void rope_fill(int n_pos, int hd, float theta, float* cs, float* sn);

}  // namespace s2
