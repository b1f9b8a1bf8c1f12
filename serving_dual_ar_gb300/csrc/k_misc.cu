// K8 input embedding with the VQ codebook sum, RMSNorm of rows (for the
// tensor-core path's bf16 operands and the prefill's last hidden), and small
// row gather/scatter helpers for per-sequence state.
#include "embed_body.cuh"

namespace s2 {

static cudaLaunchConfig_t make_cfg(dim3 grid, dim3 block, cudaStream_t st, bool pdl,
                                   cudaLaunchAttribute* attr, size_t smem = 0) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cfg;
}

template <typename WT>
__global__ void __launch_bounds__(256) embed_kernel(EmbedArgs a) {
  embed_body<WT>(a, blockIdx.x, blockIdx.y * blockDim.x, gridDim.y * blockDim.x, threadIdx.x, [] {
    pdl_launch_next();
    pdl_wait();
  });
}

cudaError_t launch_embed(const EmbedArgs& a, cudaStream_t st, bool pdl) {
  if (a.rows <= 0) return cudaSuccess;
  if (a.n_codebooks > 16) return cudaErrorInvalidValue;
  if (g_recorder) {  // persistent decode: bf16 tables only
    if (!a.w_bf16) {
      g_recorder->ok = false;
      return cudaSuccess;
    }
    PersistOp op;
    op.kind = PK_EMBED;
    op.e = a;
    g_recorder->ops.push_back(op);
    return cudaSuccess;
  }
  cudaLaunchAttribute attr[1];
  // one CTA per (row, 256 columns)
  cudaLaunchConfig_t cfg = make_cfg(dim3(a.rows, (a.d + 255) / 256), dim3(256), st, pdl, attr);
  return a.w_bf16 ? s2_launch(&cfg, embed_kernel<__nv_bfloat16>, a)
                  : s2_launch(&cfg, embed_kernel<float>, a);
}

// Order-preserving map of a float to an unsigned key (larger float, larger key).
S2_DEV unsigned order_key(float v) {
  const unsigned u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Sum over the block (256 threads); every thread gets the result.
S2_DEV float block_sum256(float v, float* red) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) t += red[w];
  return t;
}
S2_DEV float block_max256(float v, float* red) {
  v = warp_max(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = -INFINITY;
#pragma unroll
  for (int w = 0; w < 8; ++w) t = fmaxf(t, red[w]);
  return t;
}

// Pick per row of a logit matrix, then the same tail as the CUDA-core head:
// write the code, keep it for feedback, copy the slow hidden / gather the
// next Fast AR input row.  Greedy (ties -> lowest index) at temperature 0,
// else Gumbel-max over the candidates, restricted with top_p < 1 to the
// nucleus: the candidates whose scaled logit is at least the largest cut at
// which the kept softmax mass reaches top_p (found by bisection over the
// order-preserving integer image of the scaled logits).  With an EOS row the
// candidates are the C logits and then the EOS logit.  Dynamic shared
// memory: 2 * (C + 1) floats.
__global__ void __launch_bounds__(256) argmax_rows_kernel(ArgmaxRowsArgs a) {
  extern __shared__ __align__(16) float cand[];   // [C + 1] scores, then [C + 1] weights
  __shared__ float sv[8];
  __shared__ int si[8];
  __shared__ float red[8];
  __shared__ int s_code;
  const int r = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_next();
  pdl_wait();
  const float* lg = a.logits + (size_t)r * a.ld;
  const bool was_done = a.done && __ldcg(a.done + r) != 0;
  const int n = a.C + (a.eos_row ? 1 : 0);
  float* ew = cand + n;
  for (int c = threadIdx.x; c < a.C; c += 256) {
    const float v = lg[c];
    if (a.sink) a.sink[(size_t)r * a.sink_ld + c] = v;
    cand[c] = v;
  }
  if (a.eos_row) {
    // EOS logit: the row against the normalised hidden, fixed summation order
    float t = 0.f;
    const float* hr = a.h + (size_t)r * a.h_ld;
    for (int k = threadIdx.x; k < a.d; k += 256) {
      const float e = a.eos_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.eos_row)[k])
                                 : reinterpret_cast<const float*>(a.eos_row)[k];
      t = fmaf(e, hr[k], t);
    }
    t = block_sum256(t, red);
    if (threadIdx.x == 0) cand[a.C] = t;
  }
  __syncthreads();
  const bool samp = a.temperature > 0.f;
  const int sseq = samp ? a.samp_seq[r] : 0;
  const int spos = samp ? a.samp_pos[r] + (a.frame ? __ldcg(a.frame) : 0) : 0;
  unsigned cut = 0;  // candidates with order_key(score) >= cut are kept
  if (samp) {
    for (int c = threadIdx.x; c < n; c += 256) cand[c] = cand[c] / a.temperature;
    __syncthreads();
    if (a.top_p < 1.f) {
      float m = -INFINITY;
      for (int c = threadIdx.x; c < n; c += 256) m = fmaxf(m, cand[c]);
      m = block_max256(m, red);
      float z = 0.f;
      for (int c = threadIdx.x; c < n; c += 256) {
        ew[c] = expf(cand[c] - m);
        z += ew[c];
      }
      const float target = a.top_p * block_sum256(z, red);
      // largest cut whose kept mass still reaches the target (cut 0 keeps all)
      unsigned long long lo = 0, hi = 1ull << 32;
      while (hi - lo > 1) {
        const unsigned mid = (unsigned)((lo + hi) >> 1);
        float t = 0.f;
        for (int c = threadIdx.x; c < n; c += 256)
          if (order_key(cand[c]) >= mid) t += ew[c];
        if (block_sum256(t, red) >= target) lo = mid; else hi = mid;
      }
      cut = (unsigned)lo;
    }
  }
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int c = threadIdx.x; c < n; c += 256) {
    float v = cand[c];
    if (samp) {
      if (order_key(v) < cut) continue;
      v += gumbel_noise(a.seed, sseq, spos, a.code_slot, c);
    }
    if (better(v, c, bv, bi)) { bv = v; bi = c; }
  }
  warp_argmax(bv, bi);
  if (lane == 0) { sv[warp] = bv; si[warp] = bi; }
  __syncthreads();
  if (warp == 0) {
    bv = lane < 8 ? sv[lane] : -INFINITY;
    bi = lane < 8 ? si[lane] : 0x7fffffff;
    warp_argmax(bv, bi);
    if (lane == 0) {
      const bool stop = was_done || (a.eos_row && bi == a.C);
      if (stop && a.done && !was_done) a.done[r] = 1;
      const int code = stop ? 0 : bi;   // what the next input is gathered with
      s_code = code;
      const int frame = a.frame ? __ldcg(a.frame) : 0;
      if (a.codes) a.codes[(size_t)r * a.codes_ld + frame * a.codes_per_frame + a.code_slot] = stop ? -1 : bi;
      if (a.last_codes) a.last_codes[r * a.codes_per_frame + a.code_slot] = code;
    }
  }
  __syncthreads();
  if (a.copy_src)
    for (int k = threadIdx.x; k < a.d; k += 256)
      a.copy_dst[(size_t)r * a.copy_dst_ld + k] = a.copy_src[(size_t)r * a.copy_src_ld + k];
  if (a.emb_next) {
    const size_t base = (size_t)s_code * a.d;
    if (a.emb_is_bf16) {
      const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(a.emb_next) + base;
      for (int k = threadIdx.x; k < a.d; k += 256) a.emb_dst[(size_t)r * a.emb_dst_ld + k] = __bfloat162float(e[k]);
    } else {
      const float* e = reinterpret_cast<const float*>(a.emb_next) + base;
      for (int k = threadIdx.x; k < a.d; k += 256) a.emb_dst[(size_t)r * a.emb_dst_ld + k] = e[k];
    }
  }
  if (a.frame_inc) {
    // the frame counter advances once every row has read it
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0 && atomicAdd(a.ticket, 1u) == gridDim.x - 1) {
      *a.frame_inc += 1;
      *a.ticket = 0u;
    }
  }
}

cudaError_t launch_argmax_rows(const ArgmaxRowsArgs& a, cudaStream_t st, bool pdl) {
  if (g_recorder) {  // no persistent counterpart
    g_recorder->ok = false;
    return cudaSuccess;
  }
  if (a.rows <= 0) return cudaSuccess;
  if (a.frame_inc && !a.ticket) return cudaErrorInvalidValue;
  if (a.eos_row && !a.h) return cudaErrorInvalidValue;
  const size_t smem = (size_t)2 * (a.C + 1) * sizeof(float);
  if (smem > 48 * 1024) return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(a.rows), dim3(256), st, pdl, attr, smem);
  return s2_launch(&cfg, argmax_rows_kernel, a);
}

// Per-row symmetric INT8 quantisation ("s2pro-native", The gate that says
// no: INT8 with per-channel weight scales).  IEEE division and
// round-half-even, so the result is bit-identical to any other correct
// implementation of the same definition.
template <typename WT>
__global__ void __launch_bounds__(256) quantize_rows_kernel(const WT* W, int K, int8_t* Q, float* S) {
  __shared__ float red[8];
  const size_t row = blockIdx.x;
  const WT* w = W + row * K;
  float m = 0.f;
  for (int k = threadIdx.x; k < K; k += 256) m = fmaxf(m, fabsf(to_f(w[k])));
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = threadIdx.x < 8 ? red[threadIdx.x] : 0.f;
    t = warp_max(t);
    if (threadIdx.x == 0) red[0] = t;
  }
  __syncthreads();
  float scale = red[0] / 127.0f;
  if (scale == 0.f) scale = 1.0f;
  for (int k = threadIdx.x; k < K; k += 256) {
    int q = __float2int_rn(to_f(w[k]) / scale);
    q = max(-127, min(127, q));
    Q[row * K + k] = (int8_t)q;
  }
  if (threadIdx.x == 0) S[row] = scale;
}

cudaError_t launch_quantize_rows(const void* W, int w_bf16, int N, int K, int8_t* Q, float* S,
                                 cudaStream_t st) {
  if (N <= 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(N), dim3(256), st, false, attr);
  return w_bf16 ? s2_launch(&cfg, quantize_rows_kernel<__nv_bfloat16>, static_cast<const __nv_bfloat16*>(W), K, Q, S)
                : s2_launch(&cfg, quantize_rows_kernel<float>, static_cast<const float*>(W), K, Q, S);
}

// RMSNorm of rows: out = x * rsqrt(mean(x^2) + eps) * g (fp32 and/or bf16).
// One CTA per row; each thread holds up to kRmsVec float4s of the row in
// registers across both passes (one round of loads), the bf16 planes are
// written two values per store.  Rows longer than 256 * 4 * kRmsVec take the
// scalar path.
constexpr int kRmsVec = 4;
__global__ void __launch_bounds__(256) rms_rows_kernel(RmsRowsArgs a) {
  __shared__ float red[8];
  const int r = blockIdx.x;
  frame_stamp(a.trace, r, 0);
  const bool vec = (a.d % 4 == 0) && a.d <= 256 * 4 * kRmsVec && (a.ldx % 4 == 0) &&
                   !(reinterpret_cast<uintptr_t>(a.x) & 15) && !(reinterpret_cast<uintptr_t>(a.gain) & 15) &&
                   (!a.out || ((a.out_ld % 4 == 0) && !(reinterpret_cast<uintptr_t>(a.out) & 15))) &&
                   (!a.out16 || ((a.out16_ld % 2 == 0) && !(reinterpret_cast<uintptr_t>(a.out16) & 3) &&
                                 !(reinterpret_cast<uintptr_t>(a.out16lo) & 3)));
  // the gain is a weight: read before the wait on the previous kernel
  float4 gv[kRmsVec];
  if (vec) {
#pragma unroll
    for (int j = 0; j < kRmsVec; ++j) {
      const int i = (threadIdx.x + 256 * j) * 4;
      if (i < a.d) gv[j] = *reinterpret_cast<const float4*>(a.gain + i);
    }
  }
  pdl_launch_next();
  pdl_wait();
  frame_stamp(a.trace, r, 1);
  const float* x = a.x + (size_t)r * a.ldx;
  float4 v[kRmsVec];
  float ss = 0.f;
  if (vec) {
#pragma unroll
    for (int j = 0; j < kRmsVec; ++j) {
      const int i = (threadIdx.x + 256 * j) * 4;
      v[j] = i < a.d ? *reinterpret_cast<const float4*>(x + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < kRmsVec; ++j) ss += v[j].x * v[j].x + v[j].y * v[j].y + v[j].z * v[j].z + v[j].w * v[j].w;
  } else {
    for (int i = threadIdx.x; i < a.d; i += 256) ss += x[i] * x[i];
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = threadIdx.x < 8 ? red[threadIdx.x] : 0.f;
    t = warp_sum(t);
    if (threadIdx.x == 0) red[0] = t;
  }
  __syncthreads();
  frame_stamp(a.trace, r, 2);
  const float inv = rsqrtf(red[0] / (float)a.d + a.eps);
  if (vec) {
#pragma unroll
    for (int j = 0; j < kRmsVec; ++j) {
      const int i = (threadIdx.x + 256 * j) * 4;
      if (i >= a.d) break;
      const float4 g = gv[j];
      const float o[4] = {v[j].x * inv * g.x, v[j].y * inv * g.y, v[j].z * inv * g.z, v[j].w * inv * g.w};
      if (a.out) *reinterpret_cast<float4*>(a.out + (size_t)r * a.out_ld + i) = make_float4(o[0], o[1], o[2], o[3]);
      if (a.out16) {
        __nv_bfloat16 h[4], l[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          h[e] = __float2bfloat16_rn(o[e]);
          l[e] = __float2bfloat16_rn(o[e] - __bfloat162float(h[e]));
        }
        __nv_bfloat162* dh = reinterpret_cast<__nv_bfloat162*>(a.out16 + (size_t)r * a.out16_ld + i);
        dh[0] = __halves2bfloat162(h[0], h[1]);
        dh[1] = __halves2bfloat162(h[2], h[3]);
        if (a.out16lo) {
          __nv_bfloat162* dl = reinterpret_cast<__nv_bfloat162*>(a.out16lo + (size_t)r * a.out16_ld + i);
          dl[0] = __halves2bfloat162(l[0], l[1]);
          dl[1] = __halves2bfloat162(l[2], l[3]);
        }
      }
    }
  } else {
    for (int i = threadIdx.x; i < a.d; i += 256) {
      const float w = x[i] * inv * a.gain[i];
      if (a.out) a.out[(size_t)r * a.out_ld + i] = w;
      if (a.out16) st_bf16_split(a.out16, a.out16lo, (size_t)r * a.out16_ld + i, w);
    }
  }
  frame_stamp(a.trace, r, 3);
}

cudaError_t launch_rms_rows(const RmsRowsArgs& a, cudaStream_t st, bool pdl) {
  if (g_recorder) {  // no persistent counterpart
    g_recorder->ok = false;
    return cudaSuccess;
  }
  if (a.rows <= 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(a.rows), dim3(256), st, pdl, attr);
  return s2_launch(&cfg, rms_rows_kernel, a);
}

template <typename T, bool SCATTER>
__global__ void __launch_bounds__(256) rows_kernel(T* dst, int dst_ld, const T* src, int src_ld,
                                                   const int* idx, int d) {
  const int r = blockIdx.x;
  pdl_launch_next();
  pdl_wait();
  const int j = idx ? idx[r] : r;
  const T* s = src + (size_t)(SCATTER ? r : j) * src_ld;
  T* o = dst + (size_t)(SCATTER ? j : r) * dst_ld;
  for (int i = threadIdx.x; i < d; i += 256) o[i] = s[i];
}

template <typename T, bool SCATTER>
static cudaError_t launch_rows(T* dst, int dst_ld, const T* src, int src_ld, const int* idx,
                               int rows, int d, cudaStream_t st, bool pdl) {
  if (rows <= 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(rows), dim3(256), st, pdl, attr);
  return s2_launch(&cfg, rows_kernel<T, SCATTER>, dst, dst_ld, src, src_ld, idx, d);
}

cudaError_t launch_gather_rows(float* dst, int dst_ld, const float* src, int src_ld,
                               const int* idx, int rows, int d, cudaStream_t st, bool pdl) {
  return launch_rows<float, false>(dst, dst_ld, src, src_ld, idx, rows, d, st, pdl);
}
cudaError_t launch_scatter_rows(float* dst, int dst_ld, const float* src, int src_ld,
                                const int* idx, int rows, int d, cudaStream_t st, bool pdl) {
  return launch_rows<float, true>(dst, dst_ld, src, src_ld, idx, rows, d, st, pdl);
}
cudaError_t launch_gather_rows_i32(int* dst, int dst_ld, const int* src, int src_ld,
                                   const int* idx, int rows, int d, cudaStream_t st, bool pdl) {
  return launch_rows<int, false>(dst, dst_ld, src, src_ld, idx, rows, d, st, pdl);
}
cudaError_t launch_scatter_rows_i32(int* dst, int dst_ld, const int* src, int src_ld,
                                    const int* idx, int rows, int d, cudaStream_t st, bool pdl) {
  return launch_rows<int, true>(dst, dst_ld, src, src_ld, idx, rows, d, st, pdl);
}

}  // namespace s2
