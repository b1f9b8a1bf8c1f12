// K1 weight-streaming GEMV: the per-CTA body shared by the stand-alone
// kernel (k_gemv.cu) and the persistent decode kernel (k_persist.cu).  See
// k_gemv.cu for the design.
#pragma once

#include "s2_kernels.h"
#include "s2_common.cuh"

namespace s2 {

constexpr int kGemvMaxWarps = 16;
constexpr int kGemvMaxSlots = 16;           // per warp


// 8 int8 weights (8 bytes) as floats.
S2_DEV void load8(const int8_t* p, float (&v)[8]) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[i] = (float)((int)(u.x << (24 - 8 * i)) >> 24);
    v[4 + i] = (float)((int)(u.y << (24 - 8 * i)) >> 24);
  }
}

// The GEMV of one CTA ``cta`` of ``ncta`` (the whole block takes part).
// DIRECT: VMAX 16-byte vectors per lane per segment, two segments in flight.
// NC: activations not written by this grid may use the read-only cache path.
// ``sync.arrive()`` runs first, ``sync.wait()`` after the weight stream has
// been started and before the first read of anything an earlier kernel or
// phase writes (see PdlSync).
// Staged activations are stored so that a warp's 16-byte loads of them are
// contiguous (conflict-free).  With VE weights per 16-byte vector (8 bf16,
// 16 int8), element k (k % 4 == 0) of vector vv = k / VE sits at
// 32*VE * (vv / 32) + 128 * ((k % VE) / 4) + 4 * (vv % 32): the 4-element
// quarters of a vector are 128 floats apart.
template <int VE>
S2_DEV int xperm(int k) {
  const unsigned u = (unsigned)k, vv = u / VE;   // unsigned: shifts and masks only
  return (int)(vv / 32 * (32 * VE) + ((u % VE) >> 2) * 128 + (vv % 32) * 4);
}

// The weights of one 16-byte vector as floats.
S2_DEV void unpack16(const uint4& u, float (&w)[8]) {   // 8 bf16
  w[0] = bf16lo(u.x); w[1] = bf16hi(u.x); w[2] = bf16lo(u.y); w[3] = bf16hi(u.y);
  w[4] = bf16lo(u.z); w[5] = bf16hi(u.z); w[6] = bf16lo(u.w); w[7] = bf16hi(u.w);
}
// 16 int8 weights: each byte, flipped to offset binary (b + 128), becomes
// the low mantissa byte of 2^23, and 2^23 + 128 is subtracted -- exact, with
// full-rate byte permutes and adds instead of integer-to-float conversions.
S2_DEV void unpack16(const uint4& u, float (&w)[16]) {
  const uint32_t x[4] = {u.x ^ 0x80808080u, u.y ^ 0x80808080u, u.z ^ 0x80808080u, u.w ^ 0x80808080u};
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[4 * q + i] = __uint_as_float(__byte_perm(x[q], 0x4B000000u, 0x7440u + i)) - 8388736.0f;
}

// The epilogue over a CTA's rows [r0, r0 + nrows) once res[row * MAXB + b]
// holds their dot products: store, residual add (old values in yold[row *
// MAXB + b]), SwiGLU of interleaved (gate, up) rows, or the arg-max heads
// (per-CTA best, the last CTA to finish reduces, writes the code and runs
// the tail copies and the next-embedding gather).  Threads tid < nthreads
// take part; bar() synchronises exactly them.
template <int MAXB, class Bar>
S2_DEV void gemv_epilogue(const GemvArgs& a, const float* res, const float* yold, const int r0,
                          const int nrows, const int cta, const int ncta, const int tid,
                          const int nthreads, const Bar& bar) {
  __shared__ int s_last;
  __shared__ int s_code[MAXB];
  const int B = a.B;
  const int warp = tid >> 5, lane = tid & 31, nwarps = nthreads >> 5;
  if (a.mode == GEMV_STORE || a.mode == GEMV_ADD) {
    for (int i = tid; i < nrows * B; i += nthreads) {
      const int b = i / nrows, row = i % nrows;
      float t = res[row * MAXB + b];
      if (a.wscale) t *= a.wscale[r0 + row];
      float* y = a.Y + (size_t)b * a.ldy + r0 + row;
      *y = a.mode == GEMV_ADD ? yold[row * MAXB + b] + t : t;
    }
    return;
  }
  if (a.mode == GEMV_SWIGLU) {
    // rows (2i, 2i+1) = (gate_i, up_i) -> y[i] = silu(gate) * up
    const int np = nrows / 2;
    for (int i = tid; i < np * B; i += nthreads) {
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
    const int spos = samp ? a.samp_pos[b] + (a.frame ? __ldcg(a.frame) : 0) : 0;
    for (int row = lane; row < nrows; row += 32) {
      float t = res[row * MAXB + b];
      if (a.wscale) t *= a.wscale[r0 + row];
      if (a.logits) a.logits[(size_t)b * a.logits_ld + r0 + row] = t;
      if (samp) t = t / a.temperature + gumbel_noise(a.seed, sseq, spos, a.code_slot, r0 + row);
      if (better(t, r0 + row, bv, bi)) { bv = t; bi = r0 + row; }
    }
    warp_argmax(bv, bi);
    if (lane == 0) {
      a.part_val[b * ncta + cta] = bv;
      a.part_idx[b * ncta + cta] = bi;
    }
  }
  __threadfence();
  bar();
  if (tid == 0) {
    const unsigned prev = atomicAdd(a.ticket, 1u);
    s_last = (prev == (unsigned)ncta - 1);
  }
  bar();
  if (!s_last) return;
  __threadfence();
  for (int b = warp; b < B; b += nwarps) {
    float v = -INFINITY;
    int i = 0x7fffffff;
    for (int c = lane; c < ncta; c += 32) {
      const float cv = __ldcg(a.part_val + b * ncta + c);
      const int ci = __ldcg(a.part_idx + b * ncta + c);
      if (better(cv, ci, v, i)) { v = cv; i = ci; }
    }
    warp_argmax(v, i);
    if (lane == 0) {
      s_code[b] = i;
      const int frame = a.frame ? __ldcg(a.frame) : 0;
      if (a.codes) a.codes[(size_t)b * a.codes_ld + frame * a.codes_per_frame + a.code_slot] = i;
      if (a.last_codes) a.last_codes[b * a.codes_per_frame + a.code_slot] = i;
    }
  }
  bar();
  // tail: copy rows and gather the next input embedding
  const int d = a.tail_d;
  for (int b = 0; b < B; ++b) {
    if (a.copy_src)
      for (int k = tid; k < d; k += nthreads)
        a.copy_dst[(size_t)b * a.copy_dst_ld + k] = __ldcg(a.copy_src + (size_t)b * a.copy_src_ld + k);
    if (a.emb_next) {
      const size_t base = (size_t)s_code[b] * d;
      if (a.emb_is_bf16) {
        const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(a.emb_next) + base;
        for (int k = tid; k < d; k += nthreads)
          a.emb_dst[(size_t)b * a.emb_dst_ld + k] = __bfloat162float(e[k]);
      } else {
        const float* e = reinterpret_cast<const float*>(a.emb_next) + base;
        for (int k = tid; k < d; k += nthreads) a.emb_dst[(size_t)b * a.emb_dst_ld + k] = e[k];
      }
    }
  }
  if (tid == 0) {
    *a.ticket = 0u;
    if (a.frame_inc) *a.frame_inc += 1;
  }
}

// ADEPTH > 0 (with DIRECT): instead of registers, each lane lands its
// vectors in a per-warp ring of ADEPTH segment slots in shared memory with
// cp.async and reads back only what it copied itself (no synchronisation
// between lanes); ADEPTH segments are in flight and no registers are held.
template <typename WT, int MAXB, bool DIRECT, int VMAX, bool NC, int ADEPTH = 0, class Sync>
S2_DEV void gemv_body(const GemvArgs& a, const GemvLayout& L, const int cta, const int ncta,
                      uint8_t* smem, const Sync& sync) {
  frame_stamp(a.trace, cta, 0);
  sync.arrive();
  constexpr int kDirectVmax = VMAX;
  constexpr bool ASYNC = DIRECT && ADEPTH > 0;
  constexpr int kDepth = ASYNC ? ADEPTH : 1;
  constexpr int kRegBufs = (DIRECT && !ASYNC) ? kDirectVmax : 1;
  // weights per 16-byte vector on the direct path (8 bf16, 16 int8); the TMA
  // ring path reads 8-weight vectors
  constexpr int VE = DIRECT ? 16 / (int)sizeof(WT) : 8;
  const int kGemvWarps = L.warps;
  const int kGemvThreads = kGemvWarps * 32;
  const int B = a.B, K = a.K;
  const bool norm = a.gain != nullptr;
  const bool staged = L.xstage != 0;  // activations read from xs (norm implies staged)
  const int KP = L.kp;
  const float* const Xg = a.X;
  const int ldx = a.ldx;
  float* xs = reinterpret_cast<float*>(smem + L.xs_off);
  float* res = reinterpret_cast<float*>(smem + L.res_off);           // [row][MAXB]
  float* part = reinterpret_cast<float*>(smem + L.part_off);         // [warp][2][MAXB]
  int* prow = reinterpret_cast<int*>(part + kGemvWarps * 2 * MAXB);  // [warp][2]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_off);    // [warp][kGemvMaxSlots]
  (void)kGemvThreads;
  __shared__ float s_inv[MAXB];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  const int unit = a.unit;
  const int n_units = a.N / unit;
  const int u0 = (int)((long long)n_units * cta / ncta);
  const int u1 = (int)((long long)n_units * (cta + 1) / ncta);
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
  uint4 bufA[kRegBufs], bufB[kRegBufs];
  auto load_seg = [&](int q, uint4* buf) {
    const uint4* src = reinterpret_cast<const uint4*>(seg_src(q));
#pragma unroll
    for (int j = 0; j < kRegBufs; ++j) {
      const int v = lane + 32 * j;
      if (v < KS / VE) buf[j] = __ldcs(src + v);
    }
  };
  // ASYNC: this lane's vectors of segment q into ring slot ``slot``
  uint8_t* aring = smem + L.ring_off + (size_t)warp * (ASYNC ? kDepth : 0) * L.slot_bytes;
  auto issue_async = [&](int q, int slot) {
    const uint4* src = reinterpret_cast<const uint4*>(seg_src(q));
    uint4* dst = reinterpret_cast<uint4*>(aring + (size_t)slot * L.slot_bytes);
#pragma unroll
    for (int j = 0; j < kDirectVmax; ++j) {
      const int v = lane + 32 * j;
      if (v < KS / VE) cp_async16_hint(dst + v, src + v, pol);
    }
  };
  if (ASYNC) {
    pol = policy_evict_first();
    for (int i = 0; i < kDepth; ++i) {
      if (i < cnt) issue_async(q0 + i, i);
      cp_async_commit();  // one group per segment (empty past the range)
    }
  } else if (DIRECT) {
    if (cnt > 0) load_seg(q0, bufA);
    if (cnt > 1) load_seg(q0 + 1, bufB);
  } else if (lane == 0) {
    for (int s = 0; s < spw; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
    pol = policy_evict_first();
    // weights do not depend on the previous kernel: start streaming now
    for (int i = 0; i < spw && i < cnt; ++i) issue(i, q0 + i);
  }
  // RMSNorm gain: a weight, so this thread's slices (k = 4 (tid + j T)) are
  // loaded before the wait on the previous kernel
  constexpr int kGainVecs = 2;   // covers K <= 8 T floats (K = d in the model)
  float4 gv[kGainVecs];
  if (norm) {
#pragma unroll
    for (int j = 0; j < kGainVecs; ++j) {
      const int k = (tid + j * kGemvThreads) * 4;
      if (k < K) gv[j] = *reinterpret_cast<const float4*>(a.gain + k);
    }
  }
  __syncwarp();
  sync.wait();
  frame_stamp(a.trace, cta, 1);

  if (norm) {
    // RMSNorm prologue: xs[b] = x[b] * rsqrt(mean(x^2) + eps) * g.  Every
    // thread loads its slices k = 4 (tid + j T) of every row once (one round
    // of loads), stores them raw and adds their squares; the partial sums
    // meet in shared memory, summed in warp order; then each thread scales
    // its own staged slices in place.
    float* ssp = part;  // [warp][MAXB], free until the stream's partial rows
#pragma unroll
    for (int b = 0; b < MAXB; ++b) {
      if (b < B) {
        const float* xr = a.X + (size_t)b * a.ldx;
        float ss = 0.f;
        for (int k = tid * 4; k < K; k += kGemvThreads * 4) {
          const float4 v = *reinterpret_cast<const float4*>(xr + k);
          ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
          *reinterpret_cast<float4*>(xs + (size_t)b * KP + xperm<VE>(k)) = v;
        }
        ss = warp_sum(ss);
        if (lane == 0) ssp[warp * MAXB + b] = ss;
      }
    }
    __syncthreads();
    if (tid < B) {
      float ss = 0.f;
      for (int w = 0; w < kGemvWarps; ++w) ss += ssp[w * MAXB + tid];
      s_inv[tid] = rsqrtf(ss / (float)K + a.eps);
    }
    __syncthreads();
    auto scale4 = [&](int b, int k, float s, const float4& g) {
      float4* xp = reinterpret_cast<float4*>(xs + (size_t)b * KP + xperm<VE>(k));
      const float4 v = *xp;
      const float4 o = make_float4(v.x * s * g.x, v.y * s * g.y, v.z * s * g.z, v.w * s * g.w);
      *xp = o;
      if (a.normed_out && cta == 0)
        *reinterpret_cast<float4*>(a.normed_out + (size_t)b * a.normed_ld + k) = o;
    };
#pragma unroll
    for (int b = 0; b < MAXB; ++b) {
      if (b < B) {
        const float s = s_inv[b];
#pragma unroll
        for (int j = 0; j < kGainVecs; ++j) {
          const int k = (tid + j * kGemvThreads) * 4;
          if (k < K) scale4(b, k, s, gv[j]);
        }
        for (int k = (tid + kGainVecs * kGemvThreads) * 4; k < K; k += kGemvThreads * 4)
          scale4(b, k, s, *reinterpret_cast<const float4*>(a.gain + k));
      }
    }
    __syncthreads();
  } else if (staged) {
    // per row, two of a thread's vectors loaded before either is stored (half
    // the serial round trips of one at a time)
    for (int b = 0; b < B; ++b) {
      const float* xr = a.X + (size_t)b * a.ldx;
      float* xd = xs + (size_t)b * KP;
      for (int k = tid * 4; k < K; k += 2 * kGemvThreads * 4) {
        const int k2 = k + kGemvThreads * 4;
        const float4 v0 = *reinterpret_cast<const float4*>(xr + k);
        float4 v1;
        if (k2 < K) v1 = *reinterpret_cast<const float4*>(xr + k2);
        *reinterpret_cast<float4*>(xd + xperm<VE>(k)) = v0;
        if (k2 < K) *reinterpret_cast<float4*>(xd + xperm<VE>(k2)) = v1;
      }
    }
    __syncthreads();
  }
  // residual epilogue: fetch the old values now, off the kernel's tail
  float* yold = res + L.rows_max * MAXB;  // [row][MAXB]
  if (a.mode == GEMV_ADD)
    for (int i = tid; i < nrows * B; i += kGemvThreads) {
      const int b = i / nrows, row = i % nrows;
      yold[row * MAXB + b] = a.Y[(size_t)b * a.ldy + r0 + row];
    }
  if (lane < 2) prow[warp * 2 + lane] = -1;
  frame_stamp(a.trace, cta, 2);

  // ---------------- stream this warp's range
  float acc[MAXB];
#pragma unroll
  for (int b = 0; b < MAXB; ++b) acc[b] = 0.f;
  bool ok = true;
  // accumulate one VE-element weight vector at K offset col
  auto fmav = [&](const float (&w)[VE], int col) {
#pragma unroll
    for (int b = 0; b < MAXB; ++b) {
      if (b < B) {
        float xv[VE];
        if (staged) {
          const float* p = xs + b * KP + xperm<VE>(col);
#pragma unroll
          for (int q = 0; q < VE / 4; ++q) {
            const float4 f = *reinterpret_cast<const float4*>(p + 128 * q);
            xv[4 * q] = f.x; xv[4 * q + 1] = f.y; xv[4 * q + 2] = f.z; xv[4 * q + 3] = f.w;
          }
        } else {
#pragma unroll
          for (int h = 0; h < VE / 8; ++h) {
            float x8[8];
            if (NC) ldg8(Xg + (size_t)b * ldx + col + 8 * h, x8);
            else load8(Xg + (size_t)b * ldx + col + 8 * h, x8);
#pragma unroll
            for (int e = 0; e < 8; ++e) xv[8 * h + e] = x8[e];
          }
        }
        float t = acc[b];
#pragma unroll
        for (int e = 0; e < VE; ++e) t = fmaf(w[e], xv[e], t);
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
  if constexpr (ASYNC) {
    for (int i = 0; i < cnt; ++i) {
      cp_async_wait_group<kDepth - 1>();  // segment i has landed
      const int q = q0 + i, seg = q % NSEG, slot = i % kDepth;
      const uint4* st = reinterpret_cast<const uint4*>(aring + (size_t)slot * L.slot_bytes);
#pragma unroll
      for (int j = 0; j < kDirectVmax; ++j) {
        const int v = lane + 32 * j;
        if (v < KS / VE) {
          float w[VE];
          unpack16(st[v], w);
          fmav(w, seg * KS + v * VE);
        }
      }
      close_row(i, q, seg);
      if (i + kDepth < cnt) issue_async(q + kDepth, slot);
      cp_async_commit();
    }
  } else if constexpr (DIRECT) {
    auto consume = [&](int i, uint4* buf) {
      const int q = q0 + i, seg = q % NSEG;
#pragma unroll
      for (int j = 0; j < kRegBufs; ++j) {
        const int v = lane + 32 * j;
        if (v < KS / VE) {
          float w[VE];
          unpack16(buf[j], w);
          fmav(w, seg * KS + v * VE);
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
    int issued = cnt < spw ? cnt : spw;  // segments lane 0 has issued
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
          fmav(w, seg * KS + v * 8);
        }
      }
      __syncwarp();
      if (lane == 0 && ok && i + spw < cnt) {
        fence_proxy_async();  // the generic reads of this slot precede the async refill
        issue(slot, q + spw);
        issued = i + spw + 1;
      }
      close_row(i, q, seg);
    }
    // after a wait that gave up, copies this warp issued may still be in
    // flight: each slot's last issue must land before the CTA may exit
    // (bounded; in the normal path every one was consumed already)
    if (lane == 0 && !ok)
      for (int j = issued > spw ? issued - spw : 0; j < issued; ++j)
        mbar_wait(&bars[j % spw], (j / spw) & 1, nullptr);
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

  gemv_epilogue<MAXB>(a, res, yold, r0, nrows, cta, ncta, tid, kGemvThreads, [] { __syncthreads(); });
  frame_stamp(a.trace, cta, 3);
}

}  // namespace s2
