// K3 + K4: decode attention over the paged KV cache, and K9: prefill attention.
//
// Layer arithmetic (Qwen3-style block of the S2 Slow and Fast AR): per-head
// RMSNorm of q and k (gains shared across heads), rotate-half RoPE at the
// token's absolute position with the bf16-rounded cos/sin table ("SGLang
// Day-0 Support for FishAudio S2", Engineering Appendix: BF16 RoPE Precision
// Mismatch), causal softmax attention with scale 1/sqrt(hd), q head h reading
// kv head h / (H / Hkv).  KV lives in 16-token pages ("Optimizations with
// SGLang Omni": paged KV cache; radix-shared prefixes are just pages several
// sequences' tables point to).  Page layout: [2 (K,V)][Hkv][16][hd].
// Softmax and accumulation are fp32 (the page's attention-backend note asks
// for training-time numerics, which were fp32-accumulated FlashAttention).
#include "s2_kernels.h"
#include "s2_common.cuh"

namespace s2 {

constexpr int kPage = 16;

template <typename KT> S2_DEV void load_kv8(const KT* p, float* dst);
template <> S2_DEV void load_kv8<float>(const float* p, float* dst) {
  float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
  dst[0] = a.x; dst[1] = a.y; dst[2] = a.z; dst[3] = a.w;
  dst[4] = b.x; dst[5] = b.y; dst[6] = b.z; dst[7] = b.w;
}
template <> S2_DEV void load_kv8<__nv_bfloat16>(const __nv_bfloat16* p, float* dst) {
  float v[8];
  load8(p, v);
#pragma unroll
  for (int i = 0; i < 8; ++i) dst[i] = v[i];
}

// RMSNorm + gain + RoPE of one head vector held as HD/32 values per lane
// (lane owns dims lane + 32 t).  Rotate-half pairs dims i and i + HD/2, which
// sit in the same lane at t and t + HD/64.
template <int HD>
S2_DEV void norm_rope_lane(float (&v)[HD / 32], const float* gain, float eps, int pos,
                           const float* cosT, const float* sinT, int lane) {
  constexpr int NT = HD / 32;
  float ss = 0.f;
#pragma unroll
  for (int t = 0; t < NT; ++t) ss += v[t] * v[t];
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / (float)HD + eps);
#pragma unroll
  for (int t = 0; t < NT; ++t) v[t] = v[t] * inv * gain[lane + 32 * t];
  const float* cr = cosT + (size_t)pos * (HD / 2);
  const float* sr = sinT + (size_t)pos * (HD / 2);
#pragma unroll
  for (int t = 0; t < NT / 2; ++t) {
    const int i = lane + 32 * t;  // i < HD/2
    const float c = cr[i], s = sr[i];
    const float x1 = v[t], x2 = v[t + NT / 2];
    v[t] = x1 * c - x2 * s;
    v[t + NT / 2] = x2 * c + x1 * s;
  }
}

// --------------------------------------------------------------------------
// Decode attention: grid (B, Hkv, nsplit), 128 threads.
template <typename KT, int HD, int GROUP>
__global__ void __launch_bounds__(128)
attn_decode_kernel(AttnDecodeArgs a) {
  constexpr int NT = HD / 32;
  constexpr int KST = HD + 4;                 // padded K row (floats)
  constexpr int MAXP = (GROUP * 2 + 3) / 4;   // (head,row) pairs per warp
  __shared__ __align__(16) float Ks[32][KST];
  __shared__ __align__(16) float Vs[32][HD];
  __shared__ __align__(16) float qs[GROUP * 2][HD];
  __shared__ __align__(16) float knew[2][HD];
  __shared__ __align__(16) float vnew[2][HD];
  __shared__ int s_last;

  const int b = blockIdx.x, g = blockIdx.y, split = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = a.m;
  pdl_launch_next();
  pdl_wait();
  const int fr = a.frame ? *a.frame : 0;
  const int p0 = (a.pos_base ? a.pos_base[b] + fr : 0) + a.pos_off;
  const int ctx = p0 + m;
  KT* kv = reinterpret_cast<KT*>(a.kv);
  const int qd = a.H * HD, kvd = a.Hkv * HD;

  // new keys/values of kv head g
  for (int i = warp; i < m; i += 4) {
    const float* row = a.qkv + (size_t)(b * m + i) * a.qkv_ld;
    float kr[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) kr[t] = row[qd + g * HD + lane + 32 * t];
    norm_rope_lane<HD>(kr, a.k_gain, a.eps, p0 + i, a.rope_cos, a.rope_sin, lane);
    const int pos = p0 + i;
    const int page = a.table ? a.table[(size_t)b * a.table_ld + pos / kPage] : b;
    KT* kd = kv + (size_t)page * a.page_elems + ((size_t)g * kPage + pos % kPage) * HD;
    KT* vd = kd + (size_t)a.Hkv * kPage * HD;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float vv = row[qd + kvd + g * HD + lane + 32 * t];
      knew[i][lane + 32 * t] = kr[t];
      vnew[i][lane + 32 * t] = vv;
      if (split == 0) {
        kd[lane + 32 * t] = from_f<KT>(kr[t]);
        vd[lane + 32 * t] = from_f<KT>(vv);
      }
    }
  }
  // queries of the GROUP heads of this kv head (pre-scaled by 1/sqrt(hd))
  const float scale = rsqrtf((float)HD);
  for (int pr = warp; pr < GROUP * m; pr += 4) {
    const int hh = pr % GROUP, i = pr / GROUP;
    const float* row = a.qkv + (size_t)(b * m + i) * a.qkv_ld + (g * GROUP + hh) * HD;
    float qr[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) qr[t] = row[lane + 32 * t];
    norm_rope_lane<HD>(qr, a.q_gain, a.eps, p0 + i, a.rope_cos, a.rope_sin, lane);
#pragma unroll
    for (int t = 0; t < NT; ++t) qs[pr][lane + 32 * t] = qr[t] * scale;
  }
  __syncthreads();

  // key range of this split (chunks of 32 keys)
  const int per = (ctx + a.nsplit - 1) / a.nsplit;
  const int kps = (per + 31) / 32 * 32;
  const int s0 = split * kps;
  const int s1 = min(ctx, s0 + kps);

  float m_run[MAXP], l_run[MAXP], o[MAXP][NT];
#pragma unroll
  for (int p = 0; p < MAXP; ++p) {
    m_run[p] = -INFINITY; l_run[p] = 0.f;
#pragma unroll
    for (int t = 0; t < NT; ++t) o[p][t] = 0.f;
  }

  // Each thread moves LPT (key, 8-dim) slices of K and V per 32-key chunk.
  // Chunk c+1 is loaded into registers while chunk c is being computed.
  constexpr int LPT = 32 * (HD / 8) / 128;
  uint4 kreg[LPT], vreg[LPT];   // raw 16-byte slices (8 bf16 or 4 fp32 + 4 fp32 in two halves)
  float4 kf32[LPT], vf32[LPT];  // second halves for fp32 pools
  auto fetch = [&](int c0) {
#pragma unroll
    for (int j = 0; j < LPT; ++j) {
      const int idx = threadIdx.x + j * 128;
      const int key = idx / (HD / 8), dv = (idx % (HD / 8)) * 8;
      const int kp = c0 + key;
      if (kp < s1 && kp < p0) {
        const int page = a.table ? a.table[(size_t)b * a.table_ld + kp / kPage] : b;
        const KT* ks = kv + (size_t)page * a.page_elems + ((size_t)g * kPage + kp % kPage) * HD + dv;
        const KT* vs = ks + (size_t)a.Hkv * kPage * HD;
        kreg[j] = *reinterpret_cast<const uint4*>(ks);
        vreg[j] = *reinterpret_cast<const uint4*>(vs);
        if (sizeof(KT) == 4) {
          kf32[j] = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(ks) + 4);
          vf32[j] = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(vs) + 4);
        }
      }
    }
  };
  auto stage = [&](int c0) {
#pragma unroll
    for (int j = 0; j < LPT; ++j) {
      const int idx = threadIdx.x + j * 128;
      const int key = idx / (HD / 8), dv = (idx % (HD / 8)) * 8;
      const int kp = c0 + key;
      float kf[8], vf[8];
      if (kp < s1 && kp < p0) {
        if (sizeof(KT) == 2) {
          const uint4 u = kreg[j], w = vreg[j];
          kf[0] = bf16lo(u.x); kf[1] = bf16hi(u.x); kf[2] = bf16lo(u.y); kf[3] = bf16hi(u.y);
          kf[4] = bf16lo(u.z); kf[5] = bf16hi(u.z); kf[6] = bf16lo(u.w); kf[7] = bf16hi(u.w);
          vf[0] = bf16lo(w.x); vf[1] = bf16hi(w.x); vf[2] = bf16lo(w.y); vf[3] = bf16hi(w.y);
          vf[4] = bf16lo(w.z); vf[5] = bf16hi(w.z); vf[6] = bf16lo(w.w); vf[7] = bf16hi(w.w);
        } else {
          kf[0] = __uint_as_float(kreg[j].x); kf[1] = __uint_as_float(kreg[j].y);
          kf[2] = __uint_as_float(kreg[j].z); kf[3] = __uint_as_float(kreg[j].w);
          kf[4] = kf32[j].x; kf[5] = kf32[j].y; kf[6] = kf32[j].z; kf[7] = kf32[j].w;
          vf[0] = __uint_as_float(vreg[j].x); vf[1] = __uint_as_float(vreg[j].y);
          vf[2] = __uint_as_float(vreg[j].z); vf[3] = __uint_as_float(vreg[j].w);
          vf[4] = vf32[j].x; vf[5] = vf32[j].y; vf[6] = vf32[j].z; vf[7] = vf32[j].w;
        }
      } else if (kp < s1) {
#pragma unroll
        for (int e = 0; e < 8; ++e) { kf[e] = knew[kp - p0][dv + e]; vf[e] = vnew[kp - p0][dv + e]; }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) { kf[e] = 0.f; vf[e] = 0.f; }
      }
      *reinterpret_cast<float4*>(&Ks[key][dv]) = make_float4(kf[0], kf[1], kf[2], kf[3]);
      *reinterpret_cast<float4*>(&Ks[key][dv + 4]) = make_float4(kf[4], kf[5], kf[6], kf[7]);
      *reinterpret_cast<float4*>(&Vs[key][dv]) = make_float4(vf[0], vf[1], vf[2], vf[3]);
      *reinterpret_cast<float4*>(&Vs[key][dv + 4]) = make_float4(vf[4], vf[5], vf[6], vf[7]);
    }
  };

  if (s0 < s1) fetch(s0);
  for (int c0 = s0; c0 < s1; c0 += 32) {
    stage(c0);
    __syncthreads();
    if (c0 + 32 < s1) fetch(c0 + 32);
#pragma unroll
    for (int p = 0; p < MAXP; ++p) {
      const int pr = warp + 4 * p;
      if (pr >= GROUP * m) break;
      const int i = pr / GROUP;
      const int qpos = p0 + i;
      const int kp = c0 + lane;
      const bool valid = kp < s1 && kp <= qpos;
      float sc = -INFINITY;
      if (valid) {
        float acc = 0.f;
#pragma unroll 8
        for (int dd = 0; dd < HD; dd += 4) {
          const float4 q4 = *reinterpret_cast<const float4*>(&qs[pr][dd]);
          const float4 k4 = *reinterpret_cast<const float4*>(&Ks[lane][dd]);
          acc = fmaf(q4.x, k4.x, acc); acc = fmaf(q4.y, k4.y, acc);
          acc = fmaf(q4.z, k4.z, acc); acc = fmaf(q4.w, k4.w, acc);
        }
        sc = acc;
      }
      const float mx = warp_max(sc);
      if (mx == -INFINITY) continue;
      const float m_new = fmaxf(m_run[p], mx);
      const float corr = __expf(m_run[p] - m_new);
      const float pj = valid ? __expf(sc - m_new) : 0.f;
      l_run[p] = l_run[p] * corr + warp_sum(pj);
#pragma unroll
      for (int t = 0; t < NT; ++t) o[p][t] *= corr;
      const int nk = min(32, s1 - c0);
      for (int j = 0; j < nk; ++j) {
        const float pb = __shfl_sync(0xffffffffu, pj, j);
#pragma unroll
        for (int t = 0; t < NT; ++t) o[p][t] = fmaf(pb, Vs[j][lane + 32 * t], o[p][t]);
      }
      m_run[p] = m_new;
    }
    __syncthreads();
  }

  if (a.nsplit == 1) {
#pragma unroll
    for (int p = 0; p < MAXP; ++p) {
      const int pr = warp + 4 * p;
      if (pr >= GROUP * m) break;
      const int hh = pr % GROUP, i = pr / GROUP;
      const int h = g * GROUP + hh;
      const float inv = 1.f / l_run[p];
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const float v = o[p][t] * inv;
        if (a.o) a.o[(size_t)(b * m + i) * a.o_ld + h * HD + lane + 32 * t] = v;
        if (a.o16) st_bf16_split(a.o16, a.o16lo, (size_t)(b * m + i) * a.o16_ld + h * HD + lane + 32 * t, v);
      }
    }
    return;
  }

  // split-KV: write partial (m, l, o) and let the last split combine
  const int ns = a.nsplit;
#pragma unroll
  for (int p = 0; p < MAXP; ++p) {
    const int pr = warp + 4 * p;
    if (pr >= GROUP * m) break;
    const int hh = pr % GROUP, i = pr / GROUP;
    const int h = g * GROUP + hh;
    float* dst = a.part + (((size_t)(b * m + i) * a.H + h) * ns + split) * (HD + 2);
    if (lane == 0) { dst[0] = m_run[p]; dst[1] = l_run[p]; }
#pragma unroll
    for (int t = 0; t < NT; ++t) dst[2 + lane + 32 * t] = o[p][t];
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(a.tickets + b * a.Hkv + g, 1u);
    s_last = (prev == (unsigned)ns - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int pr = warp; pr < GROUP * m; pr += 4) {
    const int hh = pr % GROUP, i = pr / GROUP;
    const int h = g * GROUP + hh;
    const float* src = a.part + ((size_t)(b * m + i) * a.H + h) * ns * (HD + 2);
    float M = -INFINITY;
    for (int s = 0; s < ns; ++s) M = fmaxf(M, __ldcg(src + s * (HD + 2)));
    float L = 0.f, acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = 0.f;
    for (int s = 0; s < ns; ++s) {
      const float ms = __ldcg(src + s * (HD + 2));
      if (ms == -INFINITY) continue;
      const float w = __expf(ms - M);
      L += w * __ldcg(src + s * (HD + 2) + 1);
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[t] += w * __ldcg(src + s * (HD + 2) + 2 + lane + 32 * t);
    }
    const float inv = 1.f / L;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float v = acc[t] * inv;
      if (a.o) a.o[(size_t)(b * m + i) * a.o_ld + h * HD + lane + 32 * t] = v;
      if (a.o16) st_bf16_split(a.o16, a.o16lo, (size_t)(b * m + i) * a.o16_ld + h * HD + lane + 32 * t, v);
    }
  }
  if (threadIdx.x == 0) a.tickets[b * a.Hkv + g] = 0u;
}

size_t attn_decode_scratch_floats(int B, int m, int H, int hd, int nsplit) {
  return (size_t)B * m * H * nsplit * (hd + 2);
}

template <typename KT, int HD, int GROUP>
static cudaError_t launch_dec(const AttnDecodeArgs& a, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B, a.Hkv, a.nsplit);
  cfg.blockDim = dim3(128);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return s2_launch(&cfg, attn_decode_kernel<KT, HD, GROUP>, a);
}

cudaError_t launch_attn_decode(const AttnDecodeArgs& a, cudaStream_t st, bool pdl) {
  if (a.m < 1 || a.m > 2 || a.nsplit < 1 || a.B < 1) return cudaErrorInvalidValue;
  if (a.nsplit > 1 && (!a.part || !a.tickets)) return cudaErrorInvalidValue;
  const int group = a.H / a.Hkv;
  if (a.hd == 128 && group == 4)
    return a.kv_bf16 ? launch_dec<__nv_bfloat16, 128, 4>(a, st, pdl) : launch_dec<float, 128, 4>(a, st, pdl);
  if (a.hd == 64 && group == 2)
    return a.kv_bf16 ? launch_dec<__nv_bfloat16, 64, 2>(a, st, pdl) : launch_dec<float, 64, 2>(a, st, pdl);
  return cudaErrorInvalidValue;
}

// --------------------------------------------------------------------------
// Prefill: q/k RMSNorm + RoPE, K/V written to pages; grid T rows, 128 threads.
template <typename KT, int HD>
__global__ void __launch_bounds__(128) qk_rope_append_kernel(QkRopeArgs a) {
  constexpr int NT = HD / 32;
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_next();
  pdl_wait();
  const int pos = a.pos0 + t;
  const float* row = a.qkv + (size_t)t * a.qkv_ld;
  const int qd = a.H * HD, kvd = a.Hkv * HD;
  const float scale = rsqrtf((float)HD);
  for (int h = warp; h < a.H; h += 4) {
    float v[NT];
#pragma unroll
    for (int i = 0; i < NT; ++i) v[i] = row[h * HD + lane + 32 * i];
    norm_rope_lane<HD>(v, a.q_gain, a.eps, pos, a.rope_cos, a.rope_sin, lane);
#pragma unroll
    for (int i = 0; i < NT; ++i) a.q_out[(size_t)t * qd + h * HD + lane + 32 * i] = v[i] * scale;
  }
  KT* kv = reinterpret_cast<KT*>(a.kv);
  const int page = a.table[pos / kPage];
  for (int g = warp; g < a.Hkv; g += 4) {
    float v[NT];
#pragma unroll
    for (int i = 0; i < NT; ++i) v[i] = row[qd + g * HD + lane + 32 * i];
    norm_rope_lane<HD>(v, a.k_gain, a.eps, pos, a.rope_cos, a.rope_sin, lane);
    KT* kd = kv + (size_t)page * a.page_elems + ((size_t)g * kPage + pos % kPage) * HD;
    KT* vd = kd + (size_t)a.Hkv * kPage * HD;
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      kd[lane + 32 * i] = from_f<KT>(v[i]);
      vd[lane + 32 * i] = from_f<KT>(row[qd + kvd + g * HD + lane + 32 * i]);
    }
  }
}

cudaError_t launch_qk_rope_append(const QkRopeArgs& a, cudaStream_t st, bool pdl) {
  if (a.T <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.T);
  cfg.blockDim = dim3(128);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (a.hd == 128)
    return a.kv_bf16 ? s2_launch(&cfg, qk_rope_append_kernel<__nv_bfloat16, 128>, a)
                     : s2_launch(&cfg, qk_rope_append_kernel<float, 128>, a);
  if (a.hd == 64)
    return a.kv_bf16 ? s2_launch(&cfg, qk_rope_append_kernel<__nv_bfloat16, 64>, a)
                     : s2_launch(&cfg, qk_rope_append_kernel<float, 64>, a);
  return cudaErrorInvalidValue;
}

// --------------------------------------------------------------------------
// Prefill attention (causal, fp32 CUDA cores): grid (ceil(T/64), H), 256
// threads.  Thread (ty, tx) = (tid / 16, tid % 16) owns query rows ty + 16 r
// (r < 4) and, for S, key columns tx + 16 c (c < 4); for O, head dims
// tx + 16 c (c < HD/16).  Keys before pos0 come from cached (possibly
// radix-shared) pages: no work is repeated for them.
template <typename KT, int HD>
__global__ void __launch_bounds__(256) attn_prefill_kernel(AttnPrefillArgs a) {
  constexpr int BQ = 64, BK = 64, ST = HD + 4, NO = HD / 16;
  extern __shared__ __align__(16) float sm[];
  float* Qs = sm;                  // [BQ][ST]
  float* Ks = Qs + BQ * ST;        // [BK][ST]
  float* Vs = Ks + BK * ST;        // [BK][HD]
  float* Ps = Vs + BK * HD;        // [BQ][BK + 4]
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int q0 = blockIdx.x * BQ;
  const int h = blockIdx.y;
  const int g = h / (a.H / a.Hkv);
  pdl_launch_next();
  pdl_wait();
  const int qd = a.H * HD;
  for (int i = tid; i < BQ * HD / 4; i += 256) {
    const int r = i / (HD / 4), c = (i % (HD / 4)) * 4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (q0 + r < a.T) v = *reinterpret_cast<const float4*>(a.q + (size_t)(q0 + r) * qd + h * HD + c);
    *reinterpret_cast<float4*>(Qs + r * ST + c) = v;
  }
  float mrow[4], lrow[4], acc[4][NO];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    mrow[r] = -INFINITY; lrow[r] = 0.f;
#pragma unroll
    for (int c = 0; c < NO; ++c) acc[r][c] = 0.f;
  }
  const int qlast = a.pos0 + min(a.T, q0 + BQ) - 1;   // last query position of the tile
  const KT* kv = reinterpret_cast<const KT*>(a.kv);
  for (int k0 = 0; k0 <= qlast; k0 += BK) {
    __syncthreads();
    for (int i = tid; i < BK * HD / 8; i += 256) {
      const int r = i / (HD / 8), c = (i % (HD / 8)) * 8;
      const int kp = k0 + r;
      float kf[8], vf[8];
      if (kp <= qlast) {
        const KT* ks = kv + (size_t)a.table[kp / kPage] * a.page_elems +
                       ((size_t)g * kPage + kp % kPage) * HD + c;
        load_kv8<KT>(ks, kf);
        load_kv8<KT>(ks + (size_t)a.Hkv * kPage * HD, vf);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) { kf[e] = 0.f; vf[e] = 0.f; }
      }
      *reinterpret_cast<float4*>(Ks + r * ST + c) = make_float4(kf[0], kf[1], kf[2], kf[3]);
      *reinterpret_cast<float4*>(Ks + r * ST + c + 4) = make_float4(kf[4], kf[5], kf[6], kf[7]);
      *reinterpret_cast<float4*>(Vs + r * HD + c) = make_float4(vf[0], vf[1], vf[2], vf[3]);
      *reinterpret_cast<float4*>(Vs + r * HD + c + 4) = make_float4(vf[4], vf[5], vf[6], vf[7]);
    }
    __syncthreads();
    float s[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) s[r][c] = 0.f;
    for (int dd = 0; dd < HD; dd += 4) {
      float4 q4[4], k4[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) q4[r] = *reinterpret_cast<const float4*>(Qs + (ty + 16 * r) * ST + dd);
#pragma unroll
      for (int c = 0; c < 4; ++c) k4[c] = *reinterpret_cast<const float4*>(Ks + (tx + 16 * c) * ST + dd);
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          s[r][c] = fmaf(q4[r].x, k4[c].x, s[r][c]);
          s[r][c] = fmaf(q4[r].y, k4[c].y, s[r][c]);
          s[r][c] = fmaf(q4[r].z, k4[c].z, s[r][c]);
          s[r][c] = fmaf(q4[r].w, k4[c].w, s[r][c]);
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int qpos = a.pos0 + q0 + ty + 16 * r;
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int kp = k0 + tx + 16 * c;
        if (kp > qpos) s[r][c] = -INFINITY;
        mx = fmaxf(mx, s[r][c]);
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_new = fmaxf(mrow[r], mx);
      float psum = 0.f;
      const bool live = m_new != -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float p = live ? __expf(s[r][c] - m_new) : 0.f;
        Ps[(ty + 16 * r) * (BK + 4) + tx + 16 * c] = p;
        psum += p;
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
      const float corr = live ? __expf(mrow[r] - m_new) : 1.f;
      lrow[r] = lrow[r] * corr + psum;
#pragma unroll
      for (int c = 0; c < NO; ++c) acc[r][c] *= corr;
      mrow[r] = m_new;
    }
    __syncthreads();
    for (int j = 0; j < BK; ++j) {
      float v[NO];
#pragma unroll
      for (int c = 0; c < NO; ++c) v[c] = Vs[j * HD + tx + 16 * c];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float p = Ps[(ty + 16 * r) * (BK + 4) + j];
#pragma unroll
        for (int c = 0; c < NO; ++c) acc[r][c] = fmaf(p, v[c], acc[r][c]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int t = q0 + ty + 16 * r;
    if (t >= a.T) continue;
    const float inv = 1.f / lrow[r];
#pragma unroll
    for (int c = 0; c < NO; ++c) {
      const float v = acc[r][c] * inv;
      if (a.o) a.o[(size_t)t * a.o_ld + h * HD + tx + 16 * c] = v;
      if (a.o16) st_bf16_split(a.o16, a.o16lo, (size_t)t * a.o16_ld + h * HD + tx + 16 * c, v);
    }
  }
}

cudaError_t launch_attn_prefill(const AttnPrefillArgs& a, cudaStream_t st, bool pdl) {
  if (a.T <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.T + 63) / 64, a.H);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  auto smem = [](int hd) { return (size_t)(64 * (hd + 4) * 2 + 64 * hd + 64 * 68) * 4; };
  cfg.dynamicSmemBytes = smem(a.hd);
  auto k = a.hd == 128 ? (a.kv_bf16 ? attn_prefill_kernel<__nv_bfloat16, 128> : attn_prefill_kernel<float, 128>)
                       : (a.kv_bf16 ? attn_prefill_kernel<__nv_bfloat16, 64> : attn_prefill_kernel<float, 64>);
  if (a.hd != 128 && a.hd != 64) return cudaErrorInvalidValue;
  static bool attr_set[4] = {false, false, false, false};
  const int which = (a.hd == 128 ? 2 : 0) + (a.kv_bf16 ? 1 : 0);
  if (!attr_set[which]) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cfg.dynamicSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[which] = true;
  }
  return s2_launch(&cfg, k, a);
}

}  // namespace s2
