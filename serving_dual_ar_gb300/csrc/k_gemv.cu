// K1: weight-streaming GEMV / skinny GEMM on CUDA cores,  y[b, n] = W[n, :] . x[b, :]
//
// Decode at batch 1 reads every weight once per frame ("s2pro-native", Where
// it stands: the frame is bound by the bandwidth of reading ~7.75 G weight
// parameters, not by arithmetic).  So this kernel is a pure HBM stream:
//   * one CTA per SM owns a contiguous block of output rows.  Its slice of W
//     is cut into K-segments of 1-4 KB; the flattened (row, segment) list is
//     split into equal contiguous ranges, one per warp;
//   * each warp streams its own range through a private ring of shared-memory
//     slots filled by the TMA engine (cp.async.bulk, one copy per segment,
//     completion on an mbarrier).  Lane 0 re-issues into a slot as soon as
//     the warp has consumed it, so there is no CTA-wide synchronisation while
//     streaming;
//   * the first copies are issued before griddepcontrol.wait: with
//     programmatic dependent launch the weight stream starts while the
//     previous kernel (whose output x is) is still running;
//   * lanes read the slot with 128-bit shared loads and accumulate in fp32
//     (split-K across lanes and segments), then a warp-shuffle reduction
//     closes each row.  Rows split between two warps are merged once at the
//     end, in warp order (deterministic);
//   * epilogues: store, residual add, SwiGLU on interleaved gate/up rows, or
//     arg-max over the rows (the constrained heads) with a last-CTA final
//     reduction that also writes the code and gathers the next embedding.
// An optional RMSNorm prologue normalises x (per batch row) into shared
// memory, so the norm before each projection costs no extra kernel.
#include "s2_kernels.h"
#include "s2_common.cuh"

#include <cstdlib>
#include <type_traits>

namespace s2 {

constexpr int kGemvMaxWarps = 16;
constexpr int kGemvMaxSlots = 16;           // per warp

// Streaming shape.  bf16 weights take the direct path (lanes load 16-byte
// vectors straight into registers, two segments in flight); fp32 and int8
// weights stream through the per-warp TMA ring.  On the S2 decode frame the
// direct path with 4 CTAs of 8 warps per SM and 2 KB segments measured 179
// frames/s against 106 for the ring (1 CTA per SM, 4 KB segments).  The
// S2_GEMV_* environment variables override the shape for tuning.
struct GemvTune {
  int warps = 8;
  int ring_bytes = 96 * 1024;   // all warps' slots (ring path)
  int seg_bytes = 4096;         // largest K-segment per copy (ring path)
  int direct_seg_bytes = 2048;  // largest K-segment per load round (direct path)
  int hint = 1;                 // L2 evict-first hint on the weight copies
  int direct = 1;               // bf16: lanes load weights straight into registers
  int ctas_per_sm = 1;          // ring path: grid = SMs x this
  int direct_ctas_per_sm = 4;   // direct path: grid = SMs x this
  int vmax = 0;                 // direct: 16-byte vectors per lane per segment (4 or 8; 0 = by segment)
  long long pf_limit = 0;       // default bytes of next-weight L2 prefetch per launch
};

struct GemvLayout {
  int KS, NSEG, slot_bytes, spw, rows_max, smem, warps, hint;
  int ring_off, xs_off, res_off, part_off, bar_off;
};

// 8 int8 weights (8 bytes) as floats.
S2_DEV void load8(const int8_t* p, float (&v)[8]) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[i] = (float)((int)(u.x << (24 - 8 * i)) >> 24);
    v[4 + i] = (float)((int)(u.y << (24 - 8 * i)) >> 24);
  }
}

template <typename WT>
static GemvLayout gemv_layout(int K, int B, bool norm, int rows_max, int maxb, const GemvTune& t,
                              int seg_bytes) {
  GemvLayout L{};
  const int esz = sizeof(WT);
  int best = 0;
  for (int ks = 8; ks <= K; ks += 8)
    if (K % ks == 0 && (ks * esz) % 16 == 0 && ks * esz <= seg_bytes) best = ks;
  L.warps = t.warps;
  L.hint = t.hint;
  L.KS = best;
  L.NSEG = best ? K / best : 0;
  L.slot_bytes = best * esz;
  L.spw = best ? t.ring_bytes / (L.warps * L.slot_bytes) : 0;
  if (L.spw > kGemvMaxSlots) L.spw = kGemvMaxSlots;
  L.rows_max = rows_max;
  auto al = [](int x) { return (x + 127) / 128 * 128; };
  L.ring_off = 0;
  L.xs_off = al(L.warps * L.spw * L.slot_bytes);
  L.res_off = L.xs_off + al(norm ? B * K * 4 : 0);
  L.part_off = L.res_off + al(rows_max * maxb * 4);
  L.bar_off = L.part_off + al(L.warps * 2 * (maxb + 1) * 4);
  L.smem = L.bar_off + L.warps * kGemvMaxSlots * 8;
  return L;
}

static GemvTune gemv_tune() {
  static GemvTune t = [] {
    GemvTune v;
    auto env = [](const char* n, int& dst, int scale = 1) {
      if (const char* e = std::getenv(n)) dst = std::atoi(e) * scale;
    };
    env("S2_GEMV_WARPS", v.warps);
    env("S2_GEMV_RING_KB", v.ring_bytes, 1024);
    env("S2_GEMV_HINT", v.hint);
    env("S2_GEMV_DIRECT", v.direct);
    env("S2_GEMV_VMAX", v.vmax);
    if (const char* e = std::getenv("S2_GEMV_PF_MB")) v.pf_limit = (long long)(std::atof(e) * 1048576.0);
    if (const char* e = std::getenv("S2_GEMV_SEG_KB")) v.seg_bytes = v.direct_seg_bytes = std::atoi(e) * 1024;
    if (const char* e = std::getenv("S2_GEMV_CTAS_PER_SM")) v.ctas_per_sm = v.direct_ctas_per_sm = std::atoi(e);
    if (v.ctas_per_sm < 1 || v.ctas_per_sm > 16) v.ctas_per_sm = 1;
    if (v.direct_ctas_per_sm < 1 || v.direct_ctas_per_sm > 16) v.direct_ctas_per_sm = 4;
    if (v.warps < 1 || v.warps > kGemvMaxWarps) v.warps = 8;
    if (v.ring_bytes < 16384) v.ring_bytes = 96 * 1024;
    if (v.seg_bytes < 512) v.seg_bytes = 4096;
    if (v.direct_seg_bytes < 512) v.direct_seg_bytes = 2048;
    return v;
  }();
  return t;
}

// Whether a launch with these arguments takes the direct (register) path.
static bool gemv_direct(const GemvArgs& a) {
  return a.w_is_bf16 && !a.w_int8 && gemv_tune().direct;
}

// DIRECT: VMAX 16-byte vectors per lane per segment, two segments in flight.
template <typename WT, int MAXB, bool DIRECT, int VMAX, int MAXT, int MINB>
__global__ void __launch_bounds__(MAXT, MINB)
gemv_kernel(GemvArgs a, GemvLayout L) {
  constexpr int kDirectVmax = VMAX;
  const int kGemvWarps = L.warps;
  const int kGemvThreads = kGemvWarps * 32;
  extern __shared__ __align__(128) uint8_t smem[];
  const int B = a.B, K = a.K;
  const bool norm = a.gain != nullptr;
  float* xs = reinterpret_cast<float*>(smem + L.xs_off);
  float* res = reinterpret_cast<float*>(smem + L.res_off);           // [row][MAXB]
  float* part = reinterpret_cast<float*>(smem + L.part_off);         // [warp][2][MAXB]
  int* prow = reinterpret_cast<int*>(part + kGemvWarps * 2 * MAXB);  // [warp][2]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_off);    // [warp][kGemvMaxSlots]
  (void)kGemvThreads;
  __shared__ float s_inv[MAXB];
  __shared__ int s_last;
  __shared__ int s_code[MAXB];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  const int unit = a.unit;
  const int n_units = a.N / unit;
  const int u0 = (int)((long long)n_units * blockIdx.x / gridDim.x);
  const int u1 = (int)((long long)n_units * (blockIdx.x + 1) / gridDim.x);
  const int r0 = u0 * unit, nrows = (u1 - u0) * unit;
  const int NSEG = L.NSEG, KS = L.KS, spw = L.spw;
  const int Q = nrows * NSEG;
  const int q0 = (int)((long long)Q * warp / kGemvWarps);
  const int q1 = (int)((long long)Q * (warp + 1) / kGemvWarps);
  const int cnt = q1 - q0;
  uint8_t* ring = smem + L.ring_off + (size_t)warp * spw * L.slot_bytes;
  uint64_t* bars = full + warp * kGemvMaxSlots;
  const WT* W = reinterpret_cast<const WT*>(a.W);

  auto seg_src = [&](int q) {
    const int row = r0 + q / NSEG, seg = q % NSEG;
    return W + (size_t)row * K + (size_t)seg * KS;
  };
  uint64_t pol = 0;
  auto issue = [&](int slot, int q) {
    mbar_arrive_expect_tx(&bars[slot], L.slot_bytes);
    if (L.hint)
      bulk_g2s_evict_first(ring + (size_t)slot * L.slot_bytes, seg_src(q), L.slot_bytes, &bars[slot], pol);
    else
      bulk_g2s(ring + (size_t)slot * L.slot_bytes, seg_src(q), L.slot_bytes, &bars[slot]);
  };
  // DIRECT: each lane's 16-byte weight vectors of a segment, one segment ahead
  uint4 bufA[DIRECT ? kDirectVmax : 1], bufB[DIRECT ? kDirectVmax : 1];
  auto load_seg = [&](int q, uint4* buf) {
    const uint4* src = reinterpret_cast<const uint4*>(seg_src(q));
#pragma unroll
    for (int j = 0; j < (DIRECT ? kDirectVmax : 1); ++j) {
      const int v = lane + 32 * j;
      if (v < KS / 8) buf[j] = __ldcs(src + v);
    }
  };
  if (DIRECT) {
    if (cnt > 0) load_seg(q0, bufA);
    if (cnt > 1) load_seg(q0 + 1, bufB);
  } else if (lane == 0) {
    for (int s = 0; s < spw; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
    pol = policy_evict_first();
    // weights do not depend on the previous kernel: start streaming now
    for (int i = 0; i < spw && i < cnt; ++i) issue(i, q0 + i);
    if (!DIRECT && a.l2_prefetch > 0 && cnt > spw) {
      // warm L2 with the next part of this warp's range as well
      const int pf = min(cnt - spw, a.l2_prefetch / L.slot_bytes);
      for (int i = 0; i < pf; ++i) bulk_prefetch_l2(seg_src(q0 + spw + i), L.slot_bytes);
    }
  }
  __syncwarp();
  pdl_launch_next();
  pdl_wait();

  if (norm) {
    // RMSNorm prologue: xs[b] = x[b] * rsqrt(mean(x^2) + eps) * g
    for (int b = warp; b < B; b += kGemvWarps) {
      const float* xr = a.X + (size_t)b * a.ldx;
      float ss = 0.f;
      for (int k = lane * 4; k < K; k += 128) {
        float4 v = *reinterpret_cast<const float4*>(xr + k);
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
      }
      ss = warp_sum(ss);
      if (lane == 0) s_inv[b] = rsqrtf(ss / (float)K + a.eps);
    }
    __syncthreads();
    for (int i = tid * 4; i < B * K; i += kGemvThreads * 4) {
      const int b = i / K, k = i % K;
      float4 v = *reinterpret_cast<const float4*>(a.X + (size_t)b * a.ldx + k);
      float4 g = *reinterpret_cast<const float4*>(a.gain + k);
      const float s = s_inv[b];
      float4 o = make_float4(v.x * s * g.x, v.y * s * g.y, v.z * s * g.z, v.w * s * g.w);
      *reinterpret_cast<float4*>(xs + i) = o;
      if (a.normed_out && blockIdx.x == 0)
        *reinterpret_cast<float4*>(a.normed_out + (size_t)b * a.normed_ld + k) = o;
    }
    __syncthreads();
  }
  if (lane < 2) prow[warp * 2 + lane] = -1;

  // ---------------- stream this warp's range
  float acc[MAXB];
#pragma unroll
  for (int b = 0; b < MAXB; ++b) acc[b] = 0.f;
  bool ok = true;
  // accumulate one 8-element weight vector at K offset col
  auto fma8 = [&](const float (&w)[8], int col) {
#pragma unroll
    for (int b = 0; b < MAXB; ++b) {
      if (b < B) {
        float xv[8];
        if (norm) load8(xs + b * K + col, xv);
        else ldg8(a.X + (size_t)b * a.ldx + col, xv);
        float t = acc[b];
#pragma unroll
        for (int e = 0; e < 8; ++e) t = fmaf(w[e], xv[e], t);
        acc[b] = t;
      }
    }
  };
  // close a row at its last segment or at the end of the range
  auto close_row = [&](int i, int q, int seg) {
    if (seg == NSEG - 1 || i == cnt - 1) {
      const int row = q / NSEG;
      const bool starts_here = row * NSEG >= q0;
      const bool whole = starts_here && seg == NSEG - 1;
      const int side = starts_here ? 1 : 0;
#pragma unroll
      for (int b = 0; b < MAXB; ++b) {
        const float t = warp_sum(acc[b]);
        acc[b] = 0.f;
        if (lane == 0 && b < B) {
          if (whole) res[row * MAXB + b] = t;
          else part[(warp * 2 + side) * MAXB + b] = t;
        }
      }
      if (lane == 0 && !whole) prow[warp * 2 + side] = row;
    }
  };
  if (DIRECT) {
    auto consume = [&](int i, uint4* buf) {
      const int q = q0 + i, seg = q % NSEG;
#pragma unroll
      for (int j = 0; j < (DIRECT ? kDirectVmax : 1); ++j) {
        const int v = lane + 32 * j;
        if (v < KS / 8) {
          float w[8];
          const uint4 u = buf[j];
          w[0] = bf16lo(u.x); w[1] = bf16hi(u.x); w[2] = bf16lo(u.y); w[3] = bf16hi(u.y);
          w[4] = bf16lo(u.z); w[5] = bf16hi(u.z); w[6] = bf16lo(u.w); w[7] = bf16hi(u.w);
          fma8(w, seg * KS + v * 8);
        }
      }
      close_row(i, q, seg);
      if (i + 2 < cnt) load_seg(q + 2, buf);
    };
    for (int i = 0; i < cnt; i += 2) {
      consume(i, bufA);
      if (i + 1 < cnt) consume(i + 1, bufB);
    }
  } else {
    for (int i = 0; i < cnt; ++i) {
      const int q = q0 + i;
      const int slot = i % spw;
      if (ok && !mbar_wait(&bars[slot], (i / spw) & 1, a.err)) ok = false;
      const WT* st = reinterpret_cast<const WT*>(ring + (size_t)slot * L.slot_bytes);
      const int seg = q % NSEG;
      if (ok) {
        for (int v = lane; v < KS / 8; v += 32) {
          float w[8];
          load8(st + v * 8, w);
          fma8(w, seg * KS + v * 8);
        }
      }
      __syncwarp();
      if (lane == 0 && ok && i + spw < cnt) {
        fence_proxy_async();  // the generic reads of this slot precede the async refill
        issue(slot, q + spw);
      }
      close_row(i, q, seg);
    }
  }
  if (a.pf_next && a.pf_limit > 0 && lane == 0) {
    // this warp is done streaming: warm L2 with the head of its slice of the
    // next weights (bulk prefetch, no completion to wait for)
    const long long nsl = (long long)gridDim.x * kGemvWarps;
    const long long sl = (long long)blockIdx.x * kGemvWarps + warp;
    const long long slice = a.pf_next_bytes / nsl;
    const long long beg = (sl * slice) & ~15LL;
    long long len = (slice < a.pf_limit / nsl ? slice : a.pf_limit / nsl) & ~15LL;
    if (beg + len > a.pf_next_bytes) len = (a.pf_next_bytes - beg) & ~15LL;
    const char* p = static_cast<const char*>(a.pf_next) + beg;
    while (len > 0) {
      const uint32_t n = (uint32_t)(len < 65536 ? len : 65536);
      bulk_prefetch_l2(p, n);
      p += n;
      len -= n;
    }
  }
  __syncthreads();
  // rows shared by neighbouring warps: sum the partials in warp order
  if (tid < kGemvWarps * 2) {
    const int R = prow[tid];
    bool first = R >= 0;
    for (int e = 0; e < tid && first; ++e) first = prow[e] != R;
    if (first)
      for (int b = 0; b < B; ++b) {
        float t = 0.f;
        for (int e = tid; e < kGemvWarps * 2; ++e)
          if (prow[e] == R) t += part[e * MAXB + b];
        res[R * MAXB + b] = t;
      }
  }
  __syncthreads();

  // ---------------- epilogue over the CTA's rows
  if (a.mode == GEMV_STORE || a.mode == GEMV_ADD) {
    for (int i = tid; i < nrows * B; i += kGemvThreads) {
      const int b = i / nrows, row = i % nrows;
      float t = res[row * MAXB + b];
      if (a.wscale) t *= a.wscale[r0 + row];
      float* y = a.Y + (size_t)b * a.ldy + r0 + row;
      if (a.mode == GEMV_ADD) *y += t; else *y = t;
    }
    return;
  }
  if (a.mode == GEMV_SWIGLU) {
    // rows (2i, 2i+1) = (gate_i, up_i) -> y[i] = silu(gate) * up
    const int np = nrows / 2;
    for (int i = tid; i < np * B; i += kGemvThreads) {
      const int b = i / np, pr = i % np;
      float g = res[(2 * pr) * MAXB + b], u = res[(2 * pr + 1) * MAXB + b];
      if (a.wscale) {
        g *= a.wscale[r0 + 2 * pr];
        u *= a.wscale[r0 + 2 * pr + 1];
      }
      a.Y[(size_t)b * a.ldy + (r0 >> 1) + pr] = g / (1.f + __expf(-g)) * u;
    }
    return;
  }

  // ---------------- arg-max: per-CTA best, last CTA reduces
  if (warp < B) {
    const int b = warp;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    const bool samp = a.temperature > 0.f;
    const int sseq = samp ? a.samp_seq[b] : 0;
    const int spos = samp ? a.samp_pos[b] + (a.frame ? *a.frame : 0) : 0;
    for (int row = lane; row < nrows; row += 32) {
      float t = res[row * MAXB + b];
      if (a.wscale) t *= a.wscale[r0 + row];
      if (a.logits) a.logits[(size_t)b * a.logits_ld + r0 + row] = t;
      if (samp) t = t / a.temperature + gumbel_noise(a.seed, sseq, spos, a.code_slot, r0 + row);
      if (better(t, r0 + row, bv, bi)) { bv = t; bi = r0 + row; }
    }
    warp_argmax(bv, bi);
    if (lane == 0) {
      a.part_val[b * gridDim.x + blockIdx.x] = bv;
      a.part_idx[b * gridDim.x + blockIdx.x] = bi;
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned prev = atomicAdd(a.ticket, 1u);
    s_last = (prev == gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int b = warp; b < B; b += kGemvWarps) {
    float v = -INFINITY;
    int i = 0x7fffffff;
    for (int c = lane; c < (int)gridDim.x; c += 32) {
      const float cv = __ldcg(a.part_val + b * gridDim.x + c);
      const int ci = __ldcg(a.part_idx + b * gridDim.x + c);
      if (better(cv, ci, v, i)) { v = cv; i = ci; }
    }
    warp_argmax(v, i);
    if (lane == 0) {
      s_code[b] = i;
      const int frame = a.frame ? *a.frame : 0;
      if (a.codes) a.codes[(size_t)b * a.codes_ld + frame * a.codes_per_frame + a.code_slot] = i;
      if (a.last_codes) a.last_codes[b * a.codes_per_frame + a.code_slot] = i;
    }
  }
  __syncthreads();
  // tail: copy rows and gather the next input embedding
  const int d = a.tail_d;
  for (int b = 0; b < B; ++b) {
    if (a.copy_src)
      for (int k = tid; k < d; k += kGemvThreads)
        a.copy_dst[(size_t)b * a.copy_dst_ld + k] = __ldcg(a.copy_src + (size_t)b * a.copy_src_ld + k);
    if (a.emb_next) {
      const size_t base = (size_t)s_code[b] * d;
      if (a.emb_is_bf16) {
        const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(a.emb_next) + base;
        for (int k = tid; k < d; k += kGemvThreads)
          a.emb_dst[(size_t)b * a.emb_dst_ld + k] = __bfloat162float(e[k]);
      } else {
        const float* e = reinterpret_cast<const float*>(a.emb_next) + base;
        for (int k = tid; k < d; k += kGemvThreads) a.emb_dst[(size_t)b * a.emb_dst_ld + k] = e[k];
      }
    }
  }
  if (tid == 0) {
    *a.ticket = 0u;
    if (a.frame_inc) *a.frame_inc += 1;
  }
}

template <typename WT, int MAXB, bool DIRECT, int VMAX, int MAXT, int MINB>
static cudaError_t launch_d(const GemvArgs& a, cudaStream_t st, bool pdl, int grid) {
  const int n_units = a.N / a.unit;
  const int rows_max = ((n_units + grid - 1) / grid) * a.unit;
  const GemvTune tune = gemv_tune();
  GemvLayout L = gemv_layout<WT>(a.K, a.B, a.gain != nullptr, rows_max, MAXB, tune,
                                 DIRECT ? tune.direct_seg_bytes : tune.seg_bytes);
  if (DIRECT) {  // no ring
    L.spw = 0;
    L.xs_off = 0;
    L.res_off = L.xs_off + (a.gain ? (a.B * a.K * 4 + 127) / 128 * 128 : 0);
    L.part_off = L.res_off + (rows_max * MAXB * 4 + 127) / 128 * 128;
    L.bar_off = L.part_off + (L.warps * 2 * (MAXB + 1) * 4 + 127) / 128 * 128;
    L.smem = L.bar_off;
    if (L.KS / 8 > 32 * VMAX) return cudaErrorInvalidValue;
  }
  if (L.warps * 32 > MAXT) return cudaErrorInvalidValue;
  if (L.KS == 0 || (!DIRECT && L.spw < 2)) return cudaErrorInvalidValue;
  if (L.smem > 227 * 1024) return cudaErrorInvalidValue;
  auto kern = gemv_kernel<WT, MAXB, DIRECT, VMAX, MAXT, MINB>;
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
  if constexpr (std::is_same<WT, __nv_bfloat16>::value) {
    const GemvTune& t = gemv_tune();
    if (gemv_direct(a)) {
      // vectors per lane per segment: 4 keeps a thread at <= 64 registers
      const int vmax = t.vmax ? t.vmax : (t.direct_seg_bytes <= 2048 ? 4 : 8);
      if (vmax <= 4) return launch_d<WT, MAXB, true, 4, 512, 2>(a, st, pdl, grid);
      return launch_d<WT, MAXB, true, 8, 512, 1>(a, st, pdl, grid);
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

static int default_l2_prefetch() {
  static int v = [] {
    const char* e = std::getenv("S2_GEMV_L2_PREFETCH");
    return e ? std::atoi(e) : 0;
  }();
  return v;
}

cudaError_t launch_gemv(const GemvArgs& a_in, cudaStream_t st, bool pdl, int grid) {
  GemvArgs a = a_in;
  if (a.l2_prefetch < 0) a.l2_prefetch = default_l2_prefetch();
  if (a.l2_prefetch < 0) a.l2_prefetch = 0;
  if (a.pf_limit < 0) a.pf_limit = gemv_tune().pf_limit;
  if (a.pf_next && ((reinterpret_cast<uintptr_t>(a.pf_next) & 15) || a.pf_next_bytes < 0))
    return cudaErrorInvalidValue;
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
