// K1: weight-streaming GEMV / skinny GEMM on CUDA cores,  y[b, n] = W[n, :] . x[b, :]
//
// Decode at batch 1 reads every weight once per frame ("s2pro-native", Where
// it stands: the frame is bound by the bandwidth of reading ~7.75 G weight
// parameters, not by arithmetic).  So this kernel is a pure HBM stream:
//   * one CTA per SM owns a contiguous block of output rows; its slice of W
//     is streamed by the TMA engine (cp.async.bulk, one copy per row slice)
//     into an S-stage shared-memory ring guarded by mbarriers;
//   * the weight copies are issued before griddepcontrol.wait, so with
//     programmatic dependent launch the ring fills while the previous kernel
//     is still finishing (weights never depend on it);
//   * 8 consumer warps read the ring with 128-bit shared loads, each thread
//     accumulating a K-slice of a row group of RG rows for up to MAXB batch
//     rows (split-K inside the CTA), then warp-shuffle and cross-warp
//     reductions give the dot products;
//   * epilogues: store, residual add, SwiGLU on interleaved gate/up rows, or
//     arg-max over the rows (the constrained heads) with a last-CTA final
//     reduction that also writes the code and gathers the next embedding.
// An optional RMSNorm prologue normalises x (per batch row) into shared
// memory first, so the norm before each projection costs no extra kernel.
#include "s2_kernels.h"
#include "s2_common.cuh"

#include <cstdlib>

namespace s2 {

constexpr int kGemvConsumerWarps = 8;
constexpr int kGemvThreads = (kGemvConsumerWarps + 1) * 32;
constexpr int kGemvStages = 6;
constexpr int kGemvRG = 4;              // rows per row group
constexpr int kGemvStageBytes = 12288;  // ring stage payload (max)

struct GemvLayout {
  int KS, NKS, stage_bytes, xs_floats, smem;
};

template <typename WT>
static GemvLayout gemv_layout(int K, int B, bool norm) {
  GemvLayout L;
  const int esz = sizeof(WT);
  int best = 0;
  for (int ks = 8; ks <= K; ks += 8)
    if (K % ks == 0 && (ks * esz) % 16 == 0 && kGemvRG * ks * esz <= kGemvStageBytes) best = ks;
  L.KS = best;
  L.NKS = best ? K / best : 0;
  L.stage_bytes = kGemvRG * best * esz;
  L.xs_floats = norm ? B * K : 0;
  L.smem = kGemvStages * L.stage_bytes + L.xs_floats * 4 + 2 * kGemvStages * 8 +
           kGemvConsumerWarps * kGemvRG * 8 * 4 + 256;
  return L;
}

// 8 int8 weights (8 bytes) as floats.
S2_DEV void load8(const int8_t* p, float (&v)[8]) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[i] = (float)((int)(u.x << (24 - 8 * i)) >> 24);
    v[4 + i] = (float)((int)(u.y << (24 - 8 * i)) >> 24);
  }
}

template <typename WT, int MAXB>
__global__ void __launch_bounds__(kGemvThreads, 1)
gemv_kernel(GemvArgs a, int KS, int NKS, int stage_bytes) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  float* xs = reinterpret_cast<float*>(smem + kGemvStages * stage_bytes);
  const int B = a.B, K = a.K;
  const bool norm = a.gain != nullptr;
  uint64_t* full = reinterpret_cast<uint64_t*>(
      reinterpret_cast<uint8_t*>(xs) + (norm ? B * K * 4 : 0));
  uint64_t* empty = full + kGemvStages;
  float* red = reinterpret_cast<float*>(empty + kGemvStages);  // [warps][RG][MAXB]
  __shared__ float s_inv[MAXB];
  __shared__ int s_abort;
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = a.unit;
  const int n_units = a.N / unit;
  const int u0 = (int)((long long)n_units * blockIdx.x / gridDim.x);
  const int u1 = (int)((long long)n_units * (blockIdx.x + 1) / gridDim.x);
  const int r0 = u0 * unit, r1 = u1 * unit;
  const int n_rg = (r1 - r0 + kGemvRG - 1) / kGemvRG;
  const int n_stages = n_rg * NKS;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGemvStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kGemvConsumerWarps);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_next();

  if (warp == kGemvConsumerWarps) {
    // ---------------- producer: stream this CTA's weight rows
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const WT* W = reinterpret_cast<const WT*>(a.W);
      if (a.l2_prefetch > 0) {
        // Warm L2 with the part of this CTA's slice just past what the ring
        // requests first, so the stream keeps flowing while the kernel
        // before this one (on whose output it waits) is still running.
        const char* base = reinterpret_cast<const char*>(W + (size_t)r0 * K);
        const size_t total = (size_t)(r1 - r0) * K * sizeof(WT);
        const size_t beg = min(total, (size_t)kGemvStages * stage_bytes);
        const size_t end = min(total, beg + (size_t)a.l2_prefetch);
        for (size_t off = beg; off < end; off += 32768)
          bulk_prefetch_l2(base + off, (uint32_t)min((size_t)32768, end - off));
      }
      for (int s = 0; s < n_stages; ++s) {
        const int slot = s % kGemvStages;
        if (s >= kGemvStages) {
          if (!mbar_wait(&empty[slot], ((s / kGemvStages) + 1) & 1, a.err)) { s_abort = 1; break; }
        }
        const int rg = s / NKS, ks = s % NKS;
        const int row = r0 + rg * kGemvRG;
        const int nr = min(kGemvRG, r1 - row);
        const uint32_t slice = (uint32_t)(KS * sizeof(WT));
        mbar_arrive_expect_tx(&full[slot], slice * nr);
        for (int r = 0; r < nr; ++r)
          bulk_g2s_evict_first(ring + slot * stage_bytes + r * slice,
                               W + (size_t)(row + r) * K + (size_t)ks * KS, slice,
                               &full[slot], pol);
      }
    }
    return;
  }

  // ---------------- consumers
  pdl_wait();
  const int tid = threadIdx.x;  // 0..255
  if (norm) {
    // RMSNorm prologue: xs[b] = x[b] * rsqrt(mean(x^2) + eps) * g
    for (int b = warp; b < B; b += kGemvConsumerWarps) {
      const float* xr = a.X + (size_t)b * a.ldx;
      float ss = 0.f;
      for (int k = lane * 4; k < K; k += 128) {
        float4 v = *reinterpret_cast<const float4*>(xr + k);
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
      }
      ss = warp_sum(ss);
      if (lane == 0) s_inv[b] = rsqrtf(ss / (float)K + a.eps);
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    for (int i = tid * 4; i < B * K; i += 256 * 4) {
      const int b = i / K, k = i % K;
      float4 v = *reinterpret_cast<const float4*>(a.X + (size_t)b * a.ldx + k);
      float4 g = *reinterpret_cast<const float4*>(a.gain + k);
      const float s = s_inv[b];
      float4 o = make_float4(v.x * s * g.x, v.y * s * g.y, v.z * s * g.z, v.w * s * g.w);
      *reinterpret_cast<float4*>(xs + i) = o;
      if (a.normed_out && blockIdx.x == 0)
        *reinterpret_cast<float4*>(a.normed_out + (size_t)b * a.normed_ld + k) = o;
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
  }

  float best_v = -INFINITY;  // arg-max state, thread b < B
  int best_i = 0x7fffffff;

  int s = 0;
  for (int rg = 0; rg < n_rg; ++rg) {
    const int row = r0 + rg * kGemvRG;
    const int nr = min(kGemvRG, r1 - row);
    float acc[kGemvRG][MAXB];
#pragma unroll
    for (int r = 0; r < kGemvRG; ++r)
#pragma unroll
      for (int b = 0; b < MAXB; ++b) acc[r][b] = 0.f;

    for (int ks = 0; ks < NKS; ++ks, ++s) {
      const int slot = s % kGemvStages;
      if (!s_abort && !mbar_wait(&full[slot], (s / kGemvStages) & 1, a.err)) s_abort = 1;
      const WT* st = reinterpret_cast<const WT*>(ring + slot * stage_bytes);
      if (!s_abort) {
        for (int v = tid; v < KS / 8; v += 256) {
          const int col = ks * KS + v * 8;
          float xv[MAXB][8];
#pragma unroll
          for (int b = 0; b < MAXB; ++b) {
            if (b < B) {
              if (norm) load8(xs + b * K + col, xv[b]);
              else ldg8(a.X + (size_t)b * a.ldx + col, xv[b]);
            }
          }
#pragma unroll
          for (int r = 0; r < kGemvRG; ++r) {
            if (r < nr) {
              float w[8];
              load8(st + r * KS + v * 8, w);
#pragma unroll
              for (int b = 0; b < MAXB; ++b) {
                if (b < B) {
                  float t = acc[r][b];
#pragma unroll
                  for (int e = 0; e < 8; ++e) t = fmaf(w[e], xv[b][e], t);
                  acc[r][b] = t;
                }
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }

    // reduce the row group across lanes, then across warps
#pragma unroll
    for (int r = 0; r < kGemvRG; ++r)
#pragma unroll
      for (int b = 0; b < MAXB; ++b) {
        float t = warp_sum(acc[r][b]);
        if (lane == 0) red[(warp * kGemvRG + r) * MAXB + b] = t;
      }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (a.mode == GEMV_ARGMAX) {
      if (tid < B) {
        for (int r = 0; r < nr; ++r) {
          float t = 0.f;
          for (int w = 0; w < kGemvConsumerWarps; ++w) t += red[(w * kGemvRG + r) * MAXB + tid];
          if (a.wscale) t *= a.wscale[row + r];
          if (a.logits) a.logits[(size_t)tid * a.logits_ld + row + r] = t;
          if (better(t, row + r, best_v, best_i)) { best_v = t; best_i = row + r; }
        }
      }
    } else if (a.mode == GEMV_SWIGLU) {
      // rows (2i, 2i+1) = (gate_i, up_i) -> y[i] = silu(gate) * up
      const int np = nr / 2;
      if (tid < np * B) {
        const int pr = tid / B, b = tid % B;
        float g = 0.f, u = 0.f;
        for (int w = 0; w < kGemvConsumerWarps; ++w) {
          g += red[(w * kGemvRG + 2 * pr) * MAXB + b];
          u += red[(w * kGemvRG + 2 * pr + 1) * MAXB + b];
        }
        if (a.wscale) {
          g *= a.wscale[row + 2 * pr];
          u *= a.wscale[row + 2 * pr + 1];
        }
        const float sg = g / (1.f + __expf(-g));
        a.Y[(size_t)b * a.ldy + (row >> 1) + pr] = sg * u;
      }
    } else {
      if (tid < nr * B) {
        const int r = tid / B, b = tid % B;
        float t = 0.f;
        for (int w = 0; w < kGemvConsumerWarps; ++w) t += red[(w * kGemvRG + r) * MAXB + b];
        if (a.wscale) t *= a.wscale[row + r];
        float* y = a.Y + (size_t)b * a.ldy + row + r;
        if (a.mode == GEMV_ADD) *y += t; else *y = t;
      }
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
  }

  if (a.mode != GEMV_ARGMAX) return;

  // ---------------- arg-max: per-CTA partials, last CTA reduces
  if (tid < B) {
    a.part_val[tid * gridDim.x + blockIdx.x] = best_v;
    a.part_idx[tid * gridDim.x + blockIdx.x] = best_i;
  }
  __threadfence();
  asm volatile("bar.sync 1, 256;" ::: "memory");
  if (tid == 0) {
    const unsigned prev = atomicAdd(a.ticket, 1u);
    s_last = (prev == gridDim.x - 1);
  }
  asm volatile("bar.sync 1, 256;" ::: "memory");
  if (!s_last) return;
  __threadfence();
  __shared__ int s_code[MAXB];
  for (int b = warp; b < B; b += kGemvConsumerWarps) {
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
  asm volatile("bar.sync 1, 256;" ::: "memory");
  // tail: copy rows and gather the next input embedding
  const int d = a.tail_d;
  for (int b = 0; b < B; ++b) {
    if (a.copy_src)
      for (int k = tid; k < d; k += 256)
        a.copy_dst[(size_t)b * a.copy_dst_ld + k] = __ldcg(a.copy_src + (size_t)b * a.copy_src_ld + k);
    if (a.emb_next) {
      const size_t base = (size_t)s_code[b] * d;
      if (a.emb_is_bf16) {
        const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(a.emb_next) + base;
        for (int k = tid; k < d; k += 256)
          a.emb_dst[(size_t)b * a.emb_dst_ld + k] = __bfloat162float(e[k]);
      } else {
        const float* e = reinterpret_cast<const float*>(a.emb_next) + base;
        for (int k = tid; k < d; k += 256) a.emb_dst[(size_t)b * a.emb_dst_ld + k] = e[k];
      }
    }
  }
  if (tid == 0) {
    *a.ticket = 0u;
    if (a.frame_inc) *a.frame_inc += 1;
  }
}

template <typename WT, int MAXB>
static cudaError_t launch_t(const GemvArgs& a, cudaStream_t st, bool pdl, int grid) {
  GemvLayout L = gemv_layout<WT>(a.K, a.B, a.gain != nullptr);
  if (L.KS == 0) return cudaErrorInvalidValue;
  auto kern = gemv_kernel<WT, MAXB>;
  static int attr_bytes = 0;  // grows to the largest dynamic size a launch has asked for
  if (L.smem > attr_bytes) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L.smem);
    if (e != cudaSuccess) return e;
    attr_bytes = L.smem;
  }
  if (L.smem > 227 * 1024) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGemvThreads);
  cfg.dynamicSmemBytes = L.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return s2_launch(&cfg, kern, a, L.KS, L.NKS, L.stage_bytes);
}

int gemv_grid(const GemvArgs& a, int num_sms) {
  const int n_units = a.N / a.unit;
  return n_units < num_sms ? n_units : num_sms;
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
  if (a.l2_prefetch < 0 || a.l2_prefetch % 16) a.l2_prefetch = 0;
  if (a.B < 1 || a.B > 8 || a.N % a.unit || (a.K % 8)) return cudaErrorInvalidValue;
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
