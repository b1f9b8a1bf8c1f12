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
#include "attn_body.cuh"

#include <algorithm>

namespace s2 {

// MAXM = 1 (one new row per sequence, every launch but the Fast AR's first
// pass) keeps the unit within 36 KB of shared memory and 80 registers, so
// six CTAs share an SM.
template <typename KT, int HD, int GROUP, bool PF, int MAXM>
__global__ void __launch_bounds__(128, MAXM == 1 ? 6 : 5)
attn_decode_kernel(AttnDecodeArgs a) {
  __shared__ __align__(16) AttnSmem<HD, GROUP, MAXM> S;
  attn_body<KT, HD, GROUP, PF, !PF && sizeof(KT) == 4>(a, blockIdx.x, blockIdx.y, blockIdx.z, threadIdx.x, 0,
                                                       S, [] {
    pdl_launch_next();
    pdl_wait();
  });
}

size_t attn_decode_scratch_floats(int B, int m, int H, int hd, int nsplit) {
  return (size_t)B * m * H * nsplit * (hd + 2);
}

// The key chunks are staged chunk by chunk (fp32 pages: by cp.async) rather
// than prefetched into registers one chunk ahead: the prefetch hides one load
// latency per chunk, but its registers (125 a thread for fp32 pages against
// 92) leave room for 4 CTAs per SM instead of 5.  Measured on the S2 heads
// (32 sequences x 1,090 keys: 102.7 against 86.0 us; one sequence x 100 keys,
// 16 splits: 11.1 against 10.3 us).
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
  if (a.m == 1) return s2_launch(&cfg, attn_decode_kernel<KT, HD, GROUP, false, 1>, a);
  return s2_launch(&cfg, attn_decode_kernel<KT, HD, GROUP, false, 2>, a);
}

int attn_decode_ctas_per_sm(int hd, int group, bool kv_bf16) {
  static int cache[2][2] = {{-1, -1}, {-1, -1}};   // [hd 128?][bf16?]
  const int i = hd == 128 ? 1 : 0, j = kv_bf16 ? 1 : 0;
  if (cache[i][j] < 0) {
    int n = 0;
    cudaError_t e = cudaErrorInvalidValue;
    if (hd == 128 && group == 4)
      e = kv_bf16 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_decode_kernel<__nv_bfloat16, 128, 4, false, 1>, 128, 0)
                  : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_decode_kernel<float, 128, 4, false, 1>, 128, 0);
    else if (hd == 64 && group == 2)
      e = kv_bf16 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_decode_kernel<__nv_bfloat16, 64, 2, false, 1>, 128, 0)
                  : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_decode_kernel<float, 64, 2, false, 1>, 128, 0);
    if (e != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = 1;
    }
    cache[i][j] = n;
  }
  return cache[i][j];
}

int attn_pick_split(int B, int Hkv, int num_sms, int ctas_per_sm, int max_split) {
  const int base = B * Hkv, cap = num_sms * ctas_per_sm;
  // enough CTAs for twice the SMs (latency hiding at small batches), and up
  // to as many as one wave of resident CTAs holds
  int ns = std::max(1, std::min(max_split, (2 * num_sms + base - 1) / base));
  if (base * ns <= cap) return std::max(ns, std::min(max_split, cap / base));   // one wave
  // more than one wave: the fewest splits whose last wave is at least 90%
  // full, so the CTAs of the last wave do not run alone on a few SMs
  for (int k = ns; k <= max_split; ++k) {
    const long long ctas = (long long)base * k;
    const long long waves = (ctas + cap - 1) / cap;
    if (ctas * 10 >= waves * cap * 9) return k;
  }
  return ns;
}

cudaError_t launch_attn_decode(const AttnDecodeArgs& a, cudaStream_t st, bool pdl) {
  if (a.m < 1 || a.m > 2 || a.nsplit < 1 || a.B < 1) return cudaErrorInvalidValue;
  if (a.nsplit > 1 && (!a.part || !a.tickets)) return cudaErrorInvalidValue;
  const int group = a.H / a.Hkv;
  if (g_recorder) {  // persistent decode: (hd, group) = (128, 4) only
    if (a.hd != 128 || group != 4) {
      g_recorder->ok = false;
      return cudaSuccess;
    }
    PersistOp op;
    op.kind = PK_ATTN;
    op.at = a;
    g_recorder->ops.push_back(op);
    return cudaSuccess;
  }
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
  int pos = a.pos0 + t;
  const int* table = a.table;
  if (a.segs.info) {   // batched: this row's sequence
    const int* si = a.segs.info + 5 * a.segs.row_seg[t];
    pos = si[2] + (t - si[0]);
    table = a.segs.tables + si[3];
  }
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
  const int page = table[pos / kPage];
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
  const int split = blockIdx.z, ns = gridDim.z;
  __shared__ int s_last;
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
  // this split's key tiles [kt0, kt1) of the tile's kt_n
  const int kt_n = qlast / BK + 1;
  const int kt0 = (int)((long long)split * kt_n / ns), kt1 = (int)((long long)(split + 1) * kt_n / ns);
  for (int k0 = kt0 * BK; k0 < kt1 * BK; k0 += BK) {
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
  auto store = [&](int t, int c, float v) {
    if (a.o) a.o[(size_t)t * a.o_ld + h * HD + tx + 16 * c] = v;
    if (a.o16) st_bf16_split(a.o16, a.o16lo, (size_t)t * a.o16_ld + h * HD + tx + 16 * c, v);
  };
  if (ns == 1) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int t = q0 + ty + 16 * r;
      if (t >= a.T) continue;
      const float inv = 1.f / lrow[r];
#pragma unroll
      for (int c = 0; c < NO; ++c) store(t, c, acc[r][c] * inv);
    }
    return;
  }
  // key split: partial rows (m, l, acc[HD]) of this split, then the last
  // split of the (query tile, head) merges them in split order
  const int tile = blockIdx.x * a.H + h;
  constexpr int RS = HD + 2;
  float* mine = a.part + ((size_t)tile * ns + split) * BQ * RS;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    float* row = mine + (size_t)(ty + 16 * r) * RS;
    if (tx == 0) { row[0] = mrow[r]; row[1] = lrow[r]; }
#pragma unroll
    for (int c = 0; c < NO; ++c) row[2 + tx + 16 * c] = acc[r][c];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(a.tickets + tile, 1u) == (unsigned)ns - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const float* all = a.part + (size_t)tile * ns * BQ * RS;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int t = q0 + ty + 16 * r;
    if (t >= a.T) continue;
    const size_t ro = (size_t)(ty + 16 * r) * RS;
    float M = -INFINITY;
    for (int sp = 0; sp < ns; ++sp) M = fmaxf(M, __ldcg(all + (size_t)sp * BQ * RS + ro));
    float L = 0.f, o[NO];
#pragma unroll
    for (int c = 0; c < NO; ++c) o[c] = 0.f;
    for (int sp = 0; sp < ns; ++sp) {
      const float* row = all + (size_t)sp * BQ * RS + ro;
      const float ms = __ldcg(row);
      if (ms == -INFINITY) continue;
      const float w = __expf(ms - M);
      L += w * __ldcg(row + 1);
#pragma unroll
      for (int c = 0; c < NO; ++c) o[c] += w * __ldcg(row + 2 + tx + 16 * c);
    }
    const float inv = 1.f / L;
#pragma unroll
    for (int c = 0; c < NO; ++c) store(t, c, o[c] * inv);
  }
  if (tid == 0) a.tickets[tile] = 0u;
}

size_t attn_prefill_part_floats(int T, int H, int hd, int ksplit) {
  return ksplit > 1 ? (size_t)((T + 63) / 64) * H * ksplit * 64 * (hd + 2) : 0;
}

cudaError_t launch_attn_prefill(const AttnPrefillArgs& a, cudaStream_t st, bool pdl) {
  if (a.T <= 0) return cudaSuccess;
  // the tensor-core kernel takes a whole (kv head, 32-token tile) per CTA and
  // does not split keys: it pays off once the tiles cover the SMs (long
  // prompts); short ones -- a 41-token prompt, a 44-row suffix after a radix
  // hit -- keep the CUDA-core kernel and its key split (measured: 41 tokens
  // 4.6 against 5.8 ms of prefill, 32 radix suffixes 254 against 388 ms)
  if (a.tc && attn_prefill_tc_supported(a) && a.Hkv * ((a.T + 31) / 32) >= 128)
    return launch_attn_prefill_tc(a, st, pdl);
  if (a.ksplit < 1 || (a.ksplit > 1 && (!a.part || !a.tickets))) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.T + 63) / 64, a.H, a.ksplit);
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
