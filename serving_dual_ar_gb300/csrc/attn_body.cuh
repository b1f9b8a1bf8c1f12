// K3 + K4 decode attention: the per-unit body shared by the stand-alone
// kernel (k_attn.cu) and the persistent decode kernel (k_persist.cu), with
// the q/k RMSNorm + RoPE helper also used by prefill.  See k_attn.cu for the
// layer arithmetic.
#pragma once

#include "s2_kernels.h"
#include "s2_common.cuh"
#include "tc_common.cuh"
#include "attn_tc_util.cuh"

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
  // the table loads go out first, to overlap the norm's reduction
  const float* cr = cosT + (size_t)pos * (HD / 2);
  const float* sr = sinT + (size_t)pos * (HD / 2);
  float cs[NT / 2], sn[NT / 2], gn[NT];
#pragma unroll
  for (int t = 0; t < NT / 2; ++t) {
    cs[t] = cr[lane + 32 * t];
    sn[t] = sr[lane + 32 * t];
  }
#pragma unroll
  for (int t = 0; t < NT; ++t) gn[t] = gain[lane + 32 * t];
  float ss = 0.f;
#pragma unroll
  for (int t = 0; t < NT; ++t) ss += v[t] * v[t];
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / (float)HD + eps);
#pragma unroll
  for (int t = 0; t < NT; ++t) v[t] = v[t] * inv * gn[t];
#pragma unroll
  for (int t = 0; t < NT / 2; ++t) {
    const float c = cs[t], s = sn[t];
    const float x1 = v[t], x2 = v[t + NT / 2];
    v[t] = x1 * c - x2 * s;
    v[t + NT / 2] = x2 * c + x1 * s;
  }
}

// --------------------------------------------------------------------------
// Decode attention: one unit of 128 threads per (sequence b, kv head g, key
// split).  Stand-alone: grid (B, Hkv, nsplit), one unit per CTA.  The
// persistent decode kernel runs several units side by side in one CTA, each
// on its own named barrier ``bar`` and its own AttnSmem.
// MAXM: new rows per sequence the unit handles (1 or 2).  Key rows are
// stored with their 16-byte units permuted (ksw), so the QK loop's loads,
// one row per lane, spread over all banks without padding.
template <int HD, int GROUP, int MAXM = 2>
struct alignas(16) AttnSmem {
  float Ks[32][HD];
  float Vs[32][HD];
  float qs[GROUP * MAXM][HD];
  float knew[MAXM][HD];
  float vnew[MAXM][HD];
  int s_last;
};

// Position of dim d of key row ``key`` in its shared-memory row: the 16-byte
// unit index XORed with the row's low three bits (a permutation within each
// eight units).
S2_DEV int ksw(int key, int d) { return ((((d >> 2) ^ (key & 7))) << 2) | (d & 3); }

// N consecutive floats from 16-byte-aligned (N = 4) or 8-byte-aligned (N = 2)
// shared memory in one load.
template <int N> S2_DEV void lds_vec(const float* p, float (&v)[N]);
template <> S2_DEV void lds_vec<4>(const float* p, float (&v)[4]) {
  const float4 x = *reinterpret_cast<const float4*>(p);
  v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
}
template <> S2_DEV void lds_vec<2>(const float* p, float (&v)[2]) {
  const float2 x = *reinterpret_cast<const float2*>(p);
  v[0] = x.x; v[1] = x.y;
}

// Barrier over the ``n`` threads of named barrier ``id`` (id 0 with the whole
// block is __syncthreads()).
S2_DEV void unit_bar(int id, int n) { asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(n) : "memory"); }

// PF: load chunk c+1 into registers while chunk c is computed (the
// stand-alone kernel's alternative route); without PF each chunk is loaded
// just before it is staged, which keeps the unit's registers low inside the
// persistent kernel.  ASYNC (fp32 pages, without PF; the stand-alone
// kernel's default): the cached keys of a chunk are copied from global memory
// straight into the tiles with cp.async, so no registers hold them and more
// CTAs fit on an SM.  The staging route does not change the arithmetic.
template <int HD, int GROUP>
S2_DEV void attn_merge_rows(const AttnDecodeArgs& a, int b, int g, int ns, int used, int warp, int lane);

template <typename KT, int HD, int GROUP, bool PF = true, bool ASYNC = false, int MAXM = 2, class Wait>
S2_DEV void attn_body(const AttnDecodeArgs& a, const int b, const int g, const int split,
                      const int tid, const int bar, AttnSmem<HD, GROUP, MAXM>& S, Wait&& wait) {
  constexpr int NT = HD / 32;
  constexpr int MAXP = (GROUP * MAXM + 3) / 4;   // (head,row) pairs per warp
  auto& Ks = S.Ks;
  auto& Vs = S.Vs;
  auto& qs = S.qs;
  auto& knew = S.knew;
  auto& vnew = S.vnew;
  const int warp = tid >> 5, lane = tid & 31;
  const int m = a.m;
  // frame timeline: unit (b, g, split) = grid position of the stand-alone kernel
  const int unit_id = (split * a.Hkv + g) * a.B + b;
  auto stamp = [&](int i) {
    if (a.trace && tid == 0 && unit_id < kFrameTraceCtas) {
      unsigned long long t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      a.trace[unit_id * 4 + i] = t;
    }
  };
  stamp(0);
  wait();
  stamp(1);
  const int fr = a.frame ? __ldcg(a.frame) : 0;
  const int p0 = (a.pos_base ? a.pos_base[b] + fr : 0) + a.pos_off;
  const int ctx = p0 + m;
  KT* kv = reinterpret_cast<KT*>(a.kv);
  const int qd = a.H * HD, kvd = a.Hkv * HD;

  // key range of this split (chunks of 32 keys) within keys kb.. (keys below
  // kb: the shared prefix, whose partials fill slots 0 .. part_base-1)
  const int kb = a.key_begin ? __ldcg(a.key_begin) : 0;
  // A short range (at most kAttnOneSplitKeys keys, no prefix slots to fill)
  // is attended by split 0 alone, which writes the output rows itself: the
  // partial slots, the arrival ticket and the merge would cost more than the
  // two chunks they spread.  The rule reads only ctx and kb, so every split
  // of a (sequence, kv head) takes the same branch; the others leave after
  // the prologue (leaving before it measured slower).
  const bool one = a.nsplit > 1 && a.part_base == 0 && !a.merge_later && ctx - kb <= kAttnOneSplitKeys;
  const int nsplit = one ? 1 : a.nsplit;
  const int per = (ctx - kb + nsplit - 1) / nsplit;
  const int kps = (per + 31) / 32 * 32;
  const int s0 = kb + split * kps;
  const int s1 = min(ctx, s0 + kps);

  // o[p][t]: output dimension NT * lane + t of the warp's p-th (head, row) pair
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
      const int idx = tid + j * 128;
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
      const int idx = tid + j * 128;
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
      *reinterpret_cast<float4*>(&Ks[key][ksw(key, dv)]) = make_float4(kf[0], kf[1], kf[2], kf[3]);
      *reinterpret_cast<float4*>(&Ks[key][ksw(key, dv + 4)]) = make_float4(kf[4], kf[5], kf[6], kf[7]);
      *reinterpret_cast<float4*>(&Vs[key][dv]) = make_float4(vf[0], vf[1], vf[2], vf[3]);
      *reinterpret_cast<float4*>(&Vs[key][dv + 4]) = make_float4(vf[4], vf[5], vf[6], vf[7]);
    }
  };

  static_assert(!ASYNC || (!PF && sizeof(KT) == 4), "cp.async staging is for fp32 pages without PF");
  auto stage_async = [&](int c0) {
#pragma unroll
    for (int j = 0; j < LPT; ++j) {
      const int idx = tid + j * 128;
      const int key = idx / (HD / 8), dv = (idx % (HD / 8)) * 8;
      const int kp = c0 + key;
      if (kp < s1 && kp < p0) {
        const int page = a.table ? a.table[(size_t)b * a.table_ld + kp / kPage] : b;
        const KT* ks = kv + (size_t)page * a.page_elems + ((size_t)g * kPage + kp % kPage) * HD + dv;
        const KT* vs = ks + (size_t)a.Hkv * kPage * HD;
        cp_async16(&Ks[key][ksw(key, dv)], ks);
        cp_async16(&Ks[key][ksw(key, dv + 4)], ks + 4);
        cp_async16(&Vs[key][dv], vs);
        cp_async16(&Vs[key][dv + 4], vs + 4);
      } else if (kp < s1) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          Ks[key][ksw(key, dv + e)] = knew[kp - p0][dv + e];
          Vs[key][dv + e] = vnew[kp - p0][dv + e];
        }
      }
      // keys at or past s1 are never read: masked in the scores, outside the PV range
    }
    cp_async_commit();
    cp_async_wait_all();
  };

  // the first chunk of cached keys depends only on positions and pages:
  // start loading it before the new key's and the queries' work
  if (PF && s0 < s1) fetch(s0);

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
  unit_bar(bar, 128);
  stamp(2);
  if (one && split > 0) {
    stamp(3);
    return;
  }
  if constexpr (HD == 128 && GROUP == 4) {
    // the query operand of the shared-prefix attention: thread (row pr, k-block
    // kb, 16-byte unit c) of the first 64 threads, hi and lo planes
    if (a.q_img && split == 0 && m == 1 && tid < 64) {
      const int pr = tid >> 4, kb = (tid >> 3) & 1, c = tid & 7;
      const int r = b * GROUP + pr, tiles = (a.B * GROUP + 127) / 128;
      uint8_t* tile = a.q_img + ((size_t)g * tiles + (r >> 7)) * 65536;
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = qs[pr][kb * 64 + c * 8 + e];
      uint4 hi, lo;
      split8(x, hi, lo);
      const uint32_t off = kb * 16384 + sw128_offset(r & 127, c);
      *reinterpret_cast<uint4*>(tile + off) = hi;
      *reinterpret_cast<uint4*>(tile + 32768 + off) = lo;
    }
  }

  for (int c0 = s0; c0 < s1; c0 += 32) {
    if constexpr (ASYNC) {
      stage_async(c0);
    } else {
      if (!PF) fetch(c0);
      stage(c0);
    }
    unit_bar(bar, 128);
    if (PF && c0 + 32 < s1) fetch(c0 + 32);
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
        // four partial sums (dims 4i + c), so the FMAs form four short chains
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 8
        for (int dd = 0; dd < HD; dd += 4) {
          const float4 q4 = *reinterpret_cast<const float4*>(&qs[pr][dd]);
          const float4 k4 = *reinterpret_cast<const float4*>(&Ks[lane][ksw(lane, dd)]);
          a0 = fmaf(q4.x, k4.x, a0); a1 = fmaf(q4.y, k4.y, a1);
          a2 = fmaf(q4.z, k4.z, a2); a3 = fmaf(q4.w, k4.w, a3);
        }
        sc = (a0 + a1) + (a2 + a3);
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
      auto pv_key = [&](int j) {
        const float pb = __shfl_sync(0xffffffffu, pj, j);
        float vj[NT];
        lds_vec<NT>(&Vs[j][NT * lane], vj);
#pragma unroll
        for (int t = 0; t < NT; ++t) o[p][t] = fmaf(pb, vj[t], o[p][t]);
      };
      if (nk == 32) {   // full chunk: unrolled, so the shuffles and loads run ahead
#pragma unroll
        for (int j = 0; j < 32; ++j) pv_key(j);
      } else {
        for (int j = 0; j < nk; ++j) pv_key(j);
      }
      m_run[p] = m_new;
    }
    unit_bar(bar, 128);
  }

  if (nsplit == 1 && a.part_base == 0 && !a.merge_later) {
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
        if (a.o) a.o[(size_t)(b * m + i) * a.o_ld + h * HD + NT * lane + t] = v;
        if (a.o16) st_bf16_split(a.o16, a.o16lo, (size_t)(b * m + i) * a.o16_ld + h * HD + NT * lane + t, v);
      }
    }
    stamp(3);
    return;
  }

  // split-KV: write partial (m, l, o) and let the last split combine
  const int ns = a.part_base + a.nsplit;   // slots of a row
  const int slot = a.part_base + split;
#pragma unroll
  for (int p = 0; p < MAXP; ++p) {
    const int pr = warp + 4 * p;
    if (pr >= GROUP * m) break;
    const int hh = pr % GROUP, i = pr / GROUP;
    const int h = g * GROUP + hh;
    float* dst = a.part + (((size_t)(b * m + i) * a.H + h) * ns + slot) * (HD + 2);
    if (lane == 0) { dst[0] = m_run[p]; dst[1] = l_run[p]; }
#pragma unroll
    for (int t = 0; t < NT; ++t) dst[2 + NT * lane + t] = o[p][t];
  }
  if (a.merge_later) {   // a later launch merges
    stamp(3);
    return;
  }
  __threadfence();
  unit_bar(bar, 128);
  if (tid == 0) {
    const unsigned prev = atomicAdd(a.tickets + b * a.Hkv + g, 1u);
    S.s_last = (prev == (unsigned)a.nsplit - 1);
  }
  unit_bar(bar, 128);
  if (!S.s_last) {
    stamp(3);
    return;
  }
  __threadfence();
  // slots past the last split that held keys carry no terms: read none of them
  const int used = a.part_base + min(a.nsplit, (ctx - kb + kps - 1) / kps);
  attn_merge_rows<HD, GROUP>(a, b, g, ns, used, warp, lane);
  if (tid == 0) a.tickets[b * a.Hkv + g] = 0u;
  stamp(3);
}

// The last arrival's merge of sequence b, kv head g: for each of its
// GROUP * m (head, row) pairs (warp-strided; lane = NT output dimensions) the
// first ``used`` of the row's ns partial slots (m, l, O) combined in slot order
// into softmax-normalised output rows (fp32 and / or bf16 hi + lo planes).
template <int HD, int GROUP>
S2_DEV void attn_merge_rows(const AttnDecodeArgs& a, int b, int g, int ns, int used, int warp, int lane) {
  constexpr int NT = HD / 32;
  const int m = a.m;
  for (int pr = warp; pr < GROUP * m; pr += 4) {
    const int hh = pr % GROUP, i = pr / GROUP;
    const int h = g * GROUP + hh;
    const float* src = a.part + ((size_t)(b * m + i) * a.H + h) * ns * (HD + 2);
    // eight slots' values are requested before any is used (one round trip
    // per eight slots), and the running max, sum and output are rescaled
    // when a later batch of eight raises the max (the terms still add in
    // slot order; with eight or fewer slots this is the plain two-pass merge)
    constexpr int SB = 8;
    float M = -INFINITY, L = 0.f, acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = 0.f;
    for (int s0 = 0; s0 < used; s0 += SB) {
      float mv[SB], lv[SB], ov[SB][NT];
#pragma unroll
      for (int j = 0; j < SB; ++j) {
        const float* sp = src + (s0 + j) * (HD + 2);
        const bool in = s0 + j < used;
        mv[j] = in ? __ldcg(sp) : -INFINITY;
        lv[j] = in ? __ldcg(sp + 1) : 0.f;
#pragma unroll
        for (int t = 0; t < NT; ++t) ov[j][t] = in ? __ldcg(sp + 2 + NT * lane + t) : 0.f;
      }
      float Mb = M;
#pragma unroll
      for (int j = 0; j < SB; ++j) Mb = fmaxf(Mb, mv[j]);
      if (Mb == -INFINITY) continue;
      if (Mb != M) {   // rescale what was summed against the old max
        const float r = __expf(M - Mb);
        L *= r;
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[t] *= r;
        M = Mb;
      }
#pragma unroll
      for (int j = 0; j < SB; ++j) {
        if (mv[j] == -INFINITY) continue;
        const float w = __expf(mv[j] - M);
        L += w * lv[j];
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[t] += w * ov[j][t];
      }
    }
    const float inv = 1.f / L;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float v = acc[t] * inv;
      if (a.o) a.o[(size_t)(b * m + i) * a.o_ld + h * HD + NT * lane + t] = v;
      if (a.o16) st_bf16_split(a.o16, a.o16lo, (size_t)(b * m + i) * a.o16_ld + h * HD + NT * lane + t, v);
    }
  }
}

}  // namespace s2
