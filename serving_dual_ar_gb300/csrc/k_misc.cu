// K8 input embedding with the VQ codebook sum, RMSNorm of rows (for the
// tensor-core path's bf16 operands and the prefill's last hidden), and small
// row gather/scatter helpers for per-sequence state.
#include "s2_kernels.h"
#include "s2_common.cuh"

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

// e = E_tok[tok] + mask * sum_k E_vq[k, code_k]  ("SGLang Day-0 Support for
// FishAudio S2", Architecture: VQ embeddings are injected into the input
// embedding at masked positions; decoded frames re-enter the stream the same
// way, with the token being the frame's semantic id).  Summed in codebook
// order, fp32.
template <typename WT>
__global__ void __launch_bounds__(256) embed_kernel(EmbedArgs a) {
  const int r = blockIdx.x;
  pdl_launch_next();
  pdl_wait();
  int tok, masked;
  int code[16];
  const int nc = a.n_codebooks;
  if (a.tokens) {
    tok = a.tokens[r];
    masked = a.mask ? a.mask[r] : 0;
    for (int k = 0; k < nc; ++k) code[k] = masked ? a.codes[(size_t)k * a.codes_ld + r] : 0;
  } else {
    for (int k = 0; k < nc; ++k) code[k] = a.fb[(size_t)r * nc + k];
    tok = a.sem_begin + code[0];
    masked = 1;
  }
  const WT* te = reinterpret_cast<const WT*>(a.tok_emb) + (size_t)tok * a.d;
  const WT* ve = reinterpret_cast<const WT*>(a.vq_emb);
  for (int i = threadIdx.x; i < a.d; i += blockDim.x) {
    float e = to_f(te[i]);
    if (masked)
      for (int k = 0; k < nc; ++k)
        e += to_f(ve[((size_t)k * a.codebook_size + code[k]) * a.d + i]);
    a.out[(size_t)r * a.out_ld + i] = e;
  }
}

cudaError_t launch_embed(const EmbedArgs& a, cudaStream_t st, bool pdl) {
  if (a.rows <= 0) return cudaSuccess;
  if (a.n_codebooks > 16) return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(a.rows), dim3(256), st, pdl, attr);
  return a.w_bf16 ? s2_launch(&cfg, embed_kernel<__nv_bfloat16>, a)
                  : s2_launch(&cfg, embed_kernel<float>, a);
}

// RMSNorm of rows: out = x * rsqrt(mean(x^2) + eps) * g (fp32 and/or bf16).
__global__ void __launch_bounds__(256) rms_rows_kernel(RmsRowsArgs a) {
  __shared__ float red[8];
  const int r = blockIdx.x;
  pdl_launch_next();
  pdl_wait();
  const float* x = a.x + (size_t)r * a.ldx;
  float ss = 0.f;
  for (int i = threadIdx.x; i < a.d; i += 256) ss += x[i] * x[i];
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = threadIdx.x < 8 ? red[threadIdx.x] : 0.f;
    t = warp_sum(t);
    if (threadIdx.x == 0) red[0] = t;
  }
  __syncthreads();
  const float inv = rsqrtf(red[0] / (float)a.d + a.eps);
  for (int i = threadIdx.x; i < a.d; i += 256) {
    const float v = x[i] * inv * a.gain[i];
    if (a.out) a.out[(size_t)r * a.out_ld + i] = v;
    if (a.out16) a.out16[(size_t)r * a.out16_ld + i] = __float2bfloat16_rn(v);
  }
}

cudaError_t launch_rms_rows(const RmsRowsArgs& a, cudaStream_t st, bool pdl) {
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
