// K1: weight-streaming GEMV / skinny GEMM on CUDA cores,  y[b, n] = W[n, :] . x[b, :]
//
// Decode at batch 1 reads every weight once per frame ("s2pro-native", Where
// it stands: the frame is bound by the bandwidth of reading ~7.75 G weight
// parameters, not by arithmetic).  So this kernel is a pure HBM stream:
//   * one CTA of 16 warps per SM owns a contiguous block of output rows.  Its
//     slice of W is cut into K-segments of up to 4 KB; the flattened (row,
//     segment) list is split into equal contiguous ranges, one per warp;
//   * bf16 and int8 weights: each lane copies its own 16-byte vectors of a
//     segment into the warp's ring of three segment slots in shared memory
//     (cp.async, L2 evict-first) and reads back only what it copied, so no
//     lane waits for another and no registers hold data in flight; fp32
//     weights stream through a per-warp ring filled by the TMA engine
//     (cp.async.bulk, completion on an mbarrier);
//   * the first segments are issued before griddepcontrol.wait: with
//     programmatic dependent launch the weight stream starts while the
//     previous kernel (whose output x is) finishes;
//   * the activations sit in shared memory (RMSNorm-ed by the prologue, or
//     copied) in an order that makes every warp's 16-byte loads contiguous;
//     fp32 accumulation, split-K across lanes and segments, a warp-shuffle
//     reduction closes each row; rows split between two warps are merged once
//     at the end, in warp order (deterministic);
//   * epilogues: store, residual add, SwiGLU on interleaved gate/up rows, or
//     arg-max over the rows (the constrained heads) with a last-CTA final
//     reduction that also writes the code and gathers the next embedding.
// The per-CTA body is in gemv_body.cuh (shared with the persistent decode
// kernel); this file holds the launch planning and the stand-alone kernel.
#include "gemv_body.cuh"

#include <type_traits>

namespace s2 {

// Streaming shape.  bf16 weights take the direct path: each lane copies its
// own 16-byte weight vectors of a segment into a per-warp ring of three
// segment slots in shared memory (cp.async, L2 evict-first) and reads back
// only what it copied, so no lane waits for another; fp32 and int8 weights
// stream through the per-warp TMA ring.  Measured on the S2 batch-1 frame
// (stand-alone launches in a CUDA graph with PDL): cp.async ring, 16 warps x
// 1 CTA per SM, 4 KB segments: 210 frames/s; the same with the two segments
// in flight held in registers: 175; registers, 8 warps x 4 CTAs per SM, 2 KB
// segments: 183; ring with 2 KB segments and two CTAs per SM (so the next
// kernel's CTA can start under PDL): 148; TMA ring: 106.  The 16-warp shape
// is also the one the persistent decode kernel runs, so both paths split
// every projection the same way.
struct GemvTune {
  int warps = 8;                // ring path
  int direct_warps = 16;        // direct path
  int ring_bytes = 96 * 1024;   // all warps' slots (ring path)
  int seg_bytes = 4096;         // largest K-segment per copy (ring path)
  int direct_seg_bytes = 4096;  // largest K-segment per load round (direct path)
  int hint = 1;                 // L2 evict-first hint on the weight copies
  int direct = 1;               // bf16: lanes load weights straight into registers
  int ctas_per_sm = 1;          // ring path: grid = SMs x this
  int direct_ctas_per_sm = 1;   // direct path: grid = SMs x this
  int vmax = 0;                 // direct: 16-byte vectors per lane per segment (4 or 8; 0 = by segment)
  int adepth = 3;               // direct: cp.async ring depth (0: register double buffer)
  int nc = 0;                   // direct: activations via the read-only path (1) or coherent loads
};

template <typename WT>
static GemvLayout gemv_layout(int K, int B, bool norm, int rows_max, int maxb, const GemvTune& t,
                              int seg_bytes, int warps) {
  GemvLayout L{};
  const int esz = sizeof(WT);
  int best = 0;
  for (int ks = 8; ks <= K; ks += 8)
    if (K % ks == 0 && (ks * esz) % 16 == 0 && ks * esz <= seg_bytes) best = ks;
  L.warps = warps;
  L.hint = t.hint;
  L.KS = best;
  L.NSEG = best ? K / best : 0;
  L.slot_bytes = best * esz;
  L.spw = best ? t.ring_bytes / (L.warps * L.slot_bytes) : 0;
  if (L.spw > kGemvMaxSlots) L.spw = kGemvMaxSlots;
  L.rows_max = rows_max;
  auto al = [](int x) { return (x + 127) / 128 * 128; };
  L.kp = (K + 255) / 256 * 256;
  L.xstage = norm ? 1 : 0;
  L.ring_off = 0;
  L.xs_off = al(L.warps * L.spw * L.slot_bytes);
  L.res_off = L.xs_off + al(norm ? B * L.kp * 4 : 0);
  L.part_off = L.res_off + al(2 * rows_max * maxb * 4);  // results, old residual
  L.bar_off = L.part_off + al(L.warps * 2 * (maxb + 1) * 4);
  L.smem = L.bar_off + L.warps * kGemvMaxSlots * 8;
  return L;
}

// The measured shape (see the struct); fixed at compile time.
static const GemvTune& gemv_tune() {
  static const GemvTune t;
  return t;
}

// Whether a launch with these arguments takes the direct path (bf16 or int8
// weights; fp32 weights stream through the TMA ring).
static bool gemv_direct(const GemvArgs& a) {
  return (a.w_int8 || a.w_is_bf16) && gemv_tune().direct;
}

template <typename WT, int MAXB, bool DIRECT, int VMAX, int MAXT, int MINB, int ADEPTH, bool NC>
__global__ void __launch_bounds__(MAXT, MINB)
gemv_kernel(GemvArgs a, GemvLayout L) {
  extern __shared__ __align__(128) uint8_t smem[];
  gemv_body<WT, MAXB, DIRECT, VMAX, NC, ADEPTH>(a, L, blockIdx.x, gridDim.x, smem, PdlSync{});
}

// Layout of one launch over ``grid`` CTAs with batch instance ``maxb``.
template <typename WT, bool DIRECT>
static GemvLayout plan_layout(const GemvArgs& a, int grid, int maxb, int adepth = 0) {
  const int n_units = a.N / a.unit;
  const int rows_max = ((n_units + grid - 1) / grid) * a.unit;
  const GemvTune tune = gemv_tune();
  GemvLayout L = gemv_layout<WT>(a.K, a.B, a.gain != nullptr, rows_max, maxb, tune,
                                 DIRECT ? tune.direct_seg_bytes : tune.seg_bytes,
                                 DIRECT ? tune.direct_warps : tune.warps);
  if (DIRECT) {  // no ring, or (adepth > 0) a cp.async ring of adepth slots per warp
    auto al = [](int x) { return (x + 127) / 128 * 128; };
    const int ve = 16 / (int)sizeof(WT);  // weights per 16-byte vector
    L.kp = (a.K + 32 * ve - 1) / (32 * ve) * (32 * ve);
    L.spw = adepth;
    L.xs_off = al(L.warps * adepth * L.slot_bytes);
    const int tail = al(rows_max * maxb * 4) + al(L.warps * 2 * (maxb + 1) * 4);
    // without a norm prologue the activations are staged too when they fit
    // (2 KB stay free for the persistent kernel's descriptor slots)
    const int xs_bytes = al(a.B * L.kp * 4);
    L.xstage = (a.gain || L.xs_off + xs_bytes + tail <= 225 * 1024) ? 1 : 0;
    L.res_off = L.xs_off + (L.xstage ? xs_bytes : 0);
    L.part_off = L.res_off + al(2 * rows_max * maxb * 4);  // results, old residual
    L.bar_off = L.part_off + al(L.warps * 2 * (maxb + 1) * 4);
    L.smem = L.bar_off;
  }
  return L;
}

bool gemv_persist_layout(PersistOp& op, int maxb) {
  if (op.kind != PK_GEMV || maxb < op.g.B) return false;
  op.L = plan_layout<__nv_bfloat16, true>(op.g, op.grid, maxb, persist_adepth(maxb));
  op.maxb = maxb;
  return op.L.smem <= 227 * 1024 && op.L.KS > 0 && op.L.KS / 8 <= 32 * kPersistVmax;
}

template <typename WT, int MAXB, bool DIRECT, int VMAX, int MAXT, int MINB, int ADEPTH = 0, bool NC = true>
static cudaError_t launch_d(const GemvArgs& a, cudaStream_t st, bool pdl, int grid) {
  const GemvLayout L = plan_layout<WT, DIRECT>(a, grid, MAXB, ADEPTH);
  if (DIRECT && L.KS / (16 / (int)sizeof(WT)) > 32 * VMAX) return cudaErrorInvalidValue;
  if (L.warps * 32 > MAXT) return cudaErrorInvalidValue;
  if (L.KS == 0 || (!DIRECT && L.spw < 2)) return cudaErrorInvalidValue;
  if (L.smem > 227 * 1024) return cudaErrorInvalidValue;
  if (g_recorder) {
    // persistent decode: it runs the bf16 direct body with 512 threads, 8
    // vectors per lane, one CTA per SM
    if (!std::is_same<WT, __nv_bfloat16>::value || !DIRECT || L.warps * 32 != kPersistThreads ||
        L.KS / 8 > 32 * kPersistVmax || grid > g_recorder->max_grid) {
      g_recorder->ok = false;
      return cudaSuccess;
    }
    PersistOp op;
    op.kind = PK_GEMV;
    op.grid = grid;
    op.maxb = MAXB;
    op.g = a;
    op.L = L;
    g_recorder->ops.push_back(op);
    return cudaSuccess;
  }
  auto kern = gemv_kernel<WT, MAXB, DIRECT, VMAX, MAXT, MINB, ADEPTH, NC>;
  static int attr_bytes = 0;  // grows to the largest dynamic size a launch has asked for
  if (L.smem > attr_bytes) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L.smem);
    if (e != cudaSuccess) return e;
    attr_bytes = L.smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(L.warps * 32);
  cfg.dynamicSmemBytes = L.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return s2_launch(&cfg, kern, a, L);
}

template <typename WT, int MAXB>
static cudaError_t launch_t(const GemvArgs& a, cudaStream_t st, bool pdl, int grid) {
  if constexpr (std::is_same<WT, __nv_bfloat16>::value || std::is_same<WT, int8_t>::value) {
    const GemvTune& t = gemv_tune();
    if (gemv_direct(a)) {
      // cp.async ring of three segments (GemvTune::adepth); the register
      // double buffer with read-only or coherent activation loads, and the
      // 4-vector register instance (<= 64 registers), are the measured
      // alternatives the tune's other settings select
      if (t.adepth > 0) return launch_d<WT, MAXB, true, 8, 512, 1, 3, false>(a, st, pdl, grid);
      if constexpr (std::is_same<WT, __nv_bfloat16>::value) {
        const int vmax = t.vmax ? t.vmax : (t.direct_seg_bytes <= 2048 ? 4 : 8);
        if (vmax <= 4) return launch_d<WT, MAXB, true, 4, 512, 2>(a, st, pdl, grid);
        if (t.nc) return launch_d<WT, MAXB, true, 8, 512, 1, 0, true>(a, st, pdl, grid);
        return launch_d<WT, MAXB, true, 8, 512, 1, 0, false>(a, st, pdl, grid);
      }
    }
  }
  return launch_d<WT, MAXB, false, 1, kGemvMaxWarps * 32, 1>(a, st, pdl, grid);
}

int gemv_grid(const GemvArgs& a, int num_sms) {
  const int n_units = a.N / a.unit;
  const int want = num_sms * (gemv_direct(a) ? gemv_tune().direct_ctas_per_sm : gemv_tune().ctas_per_sm);
  return n_units < want ? n_units : want;
}

int gemv_max_grid(int num_sms) {
  const GemvTune& t = gemv_tune();
  return num_sms * (t.ctas_per_sm > t.direct_ctas_per_sm ? t.ctas_per_sm : t.direct_ctas_per_sm);
}

cudaError_t launch_gemv(const GemvArgs& a_in, cudaStream_t st, bool pdl, int grid) {
  GemvArgs a = a_in;
  if (a.B < 1 || a.B > 8 || a.N % a.unit || (a.K % 8) || grid < 1) return cudaErrorInvalidValue;
  if (a.mode == GEMV_SWIGLU && (a.unit != 2)) return cudaErrorInvalidValue;
  if (a.w_int8) {
    if (!a.wscale || (a.K % 16)) return cudaErrorInvalidValue;
    if (a.B <= 1) return launch_t<int8_t, 1>(a, st, pdl, grid);
    if (a.B <= 2) return launch_t<int8_t, 2>(a, st, pdl, grid);
    if (a.B <= 4) return launch_t<int8_t, 4>(a, st, pdl, grid);
    return launch_t<int8_t, 8>(a, st, pdl, grid);
  }
  if (a.w_is_bf16) {
    if (a.B <= 1) return launch_t<__nv_bfloat16, 1>(a, st, pdl, grid);
    if (a.B <= 2) return launch_t<__nv_bfloat16, 2>(a, st, pdl, grid);
    if (a.B <= 4) return launch_t<__nv_bfloat16, 4>(a, st, pdl, grid);
    return launch_t<__nv_bfloat16, 8>(a, st, pdl, grid);
  }
  if (a.B <= 1) return launch_t<float, 1>(a, st, pdl, grid);
  if (a.B <= 2) return launch_t<float, 2>(a, st, pdl, grid);
  if (a.B <= 4) return launch_t<float, 4>(a, st, pdl, grid);
  return launch_t<float, 8>(a, st, pdl, grid);
}

}  // namespace s2
