// Streaming decode kernel: whole Dual-AR decode frames at small batch in one
// persistent launch whose weight stream never waits for the dependency chain.
//
// At batch 1 a frame reads every weight once ("s2pro-native", Where it
// stands: bandwidth, not arithmetic) in ~370 dependent operations of 3-15 us
// of streaming each.  As separate launches every operation pays a ramp and a
// tail; a grid barrier per operation, with each CTA prefetching only after it
// arrives, pays the barrier's latency.  Here the weight stream is a thread of
// its own:
//   * one CTA per SM, 16 consumer warps + 1 producer warp;
//   * the producer walks the recorded operation list frame after frame and,
//     for every GEMV, copies this CTA's contiguous share of the weight rows
//     into a ring of 4 x 40 KB shared-memory slots with bulk copies (TMA
//     engine, one mbarrier per slot).  A slot holds whole rows (8 rows of
//     K = 2560, 4 of 4096, 2 of 9728).  The producer waits only for a free
//     slot, never for the barrier between operations, so while the consumers
//     wait for an operation's inputs the next weights are already landing;
//   * the consumers run the operations in order with a grid barrier between
//     consecutive ones.  A GEMV stages its activations (RMSNorm-ed when the
//     projection is normalised) in shared memory, then takes the slots in
//     order: each row of a slot is split into 16 / rows K-parts, one warp per
//     (row, part); the part sums meet in shared memory and are added in part
//     order; the epilogue (store, residual, SwiGLU, arg-max heads with their
//     tails) is the stand-alone GEMV's own (gemv_epilogue).  Attention and
//     the embedding run the stand-alone kernels' bodies (one attention unit
//     of 128 threads per CTA, fp32 pages staged by cp.async).
// Results agree with the per-frame CUDA graph to rounding: the GEMV's
// dot products are summed in a different order.  Every wait is bounded (2 s
// or a poll limit); a wait that gives up sets the device error word and an
// abort flag every CTA checks; the producer stops issuing and waits (bounded)
// for the copies it has in flight before its CTA exits.
#include "gemv_body.cuh"
#include "attn_body.cuh"
#include "embed_body.cuh"

#include <algorithm>

namespace s2 {

namespace {

constexpr int kSCWarps = 16;                   // consumer warps
constexpr int kSConsumers = 32 * kSCWarps;     // 512
constexpr int kSThreads = kSConsumers + 32;    // + the producer warp
constexpr int kSSlotBytes = 40 * 1024;
constexpr int kSStages = 4;
constexpr int kSRingBytes = kSSlotBytes * kSStages;
constexpr uint32_t kSPollLimit = 1u << 22;
constexpr unsigned long long kSTimeoutNs = 2000000000ull;  // 2 s
constexpr int kSBarConsumers = 1;              // named barrier ids (0 = __syncthreads)
constexpr int kSBarAttn = 2;
constexpr int kSMaxSmem = 227 * 1024;
constexpr int kSGroup = 4;                     // slots whose reductions a consumer warp batches
// trace words per operation: start, barrier passed, prologue done, first and
// last slot ready (GEMV), end
constexpr int kSTraceWords = 6;
// Chunks the producer's L2 prefetch runs ahead of the ring (0: none).
constexpr int kStreamPrefetchAhead = 0;

using AttnS = AttnSmem<128, 4>;

S2_DEV unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
S2_DEV unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
S2_DEV void consumer_bar() {
  asm volatile("bar.sync %0, %1;" :: "n"(kSBarConsumers), "n"(kSConsumers) : "memory");
}

struct StreamState {
  unsigned target;   // barrier arrivals awaited next (consumer thread 0)
  int abort;         // set when any wait of this CTA gave up (or another CTA's did)
  int stop;          // consumers' snapshot of abort, taken before a barrier (uniform)
};

// Bounded wait on an mbarrier phase that also gives up once the CTA aborts.
S2_DEV bool sw_wait(uint64_t* bar, uint32_t parity, StreamState* st, int* err) {
  const unsigned long long t0 = now_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 63u) {
      if (*reinterpret_cast<volatile int*>(&st->abort)) return false;
      if (i > kSPollLimit || now_ns() - t0 > kSTimeoutNs) {
        if (err) atomicExch(err, 2);
        *reinterpret_cast<volatile int*>(&st->abort) = 1;
        return false;
      }
    }
  }
}

// Rows [r0, r0 + nrows) of the CTA in a GEMV over N rows in units of ``unit``
// (the stand-alone kernel's partition over ncta CTAs).
S2_DEV void cta_rows(int N, int unit, int cta, int ncta, int& r0, int& nrows) {
  const int n_units = N / unit;
  const int u0 = (int)((long long)n_units * cta / ncta);
  const int u1 = (int)((long long)n_units * (cta + 1) / ncta);
  r0 = u0 * unit;
  nrows = (u1 - u0) * unit;
}

// ------------------------------------------------------------ the producer

// The producer's walk over this CTA's weight chunks: every GEMV operation of
// every frame in order, ``rc`` rows (one ring slot) at a time.
struct ChunkCursor {
  int t = -1, c = 0, nrows = 0, rc = 0, rowbytes = 0;
  const uint8_t* src = nullptr;
  // advance to the next chunk; false past the last one
  S2_DEV bool next(const StreamPlan* plan, int n_ops, int total) {
    c += rc;
    while (c >= nrows) {
      if (++t >= total) return false;
      const StreamPlan sp = plan[t % n_ops];
      if (!sp.W) { nrows = 0; c = 0; rc = 1; continue; }
      int r0;
      cta_rows(sp.N, sp.unit, blockIdx.x, gridDim.x, r0, nrows);
      rc = sp.rc;
      rowbytes = sp.rowbytes;
      src = static_cast<const uint8_t*>(sp.W) + (size_t)r0 * sp.rowbytes;
      c = 0;
    }
    return true;
  }
  S2_DEV const uint8_t* ptr() const { return src + (size_t)c * rowbytes; }
  S2_DEV uint32_t bytes() const { return (uint32_t)(min(rc, nrows - c) * rowbytes); }
};

S2_DEV void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p), "r"(bytes) : "memory");
}

// ``pf_ahead`` > 0: a second cursor runs that many chunks ahead of the ring
// and asks the L2 for them (no shared memory, nothing to wait for), so HBM
// keeps streaming while the ring is full and the consumers wait at a barrier.
S2_DEV void producer(const PersistOp* __restrict__ ops, const StreamPlan* __restrict__ plan, int n_ops,
                     int n_frames, int pf_ahead, uint8_t* ring, uint64_t* full, uint64_t* empty,
                     StreamState* st, int* err) {
  (void)ops;
  const uint64_t pol = policy_evict_first();
  long long k = 0;  // chunks issued
  bool ok = true;
  const int total = n_ops * n_frames;
  ChunkCursor cur, pf;
  bool pf_live = pf_ahead > 0;
  for (int i = 0; i < pf_ahead && pf_live; ++i)
    if ((pf_live = pf.next(plan, n_ops, total))) prefetch_l2(pf.ptr(), pf.bytes());
  while (ok && cur.next(plan, n_ops, total)) {
    const int slot = (int)(k % kSStages);
    if (k >= kSStages && !sw_wait(&empty[slot], (uint32_t)((k / kSStages - 1) & 1), st, err)) {
      ok = false;
      break;
    }
    const uint32_t bytes = cur.bytes();
    mbar_arrive_expect_tx(&full[slot], bytes);
    bulk_g2s_evict_first(ring + (size_t)slot * kSSlotBytes, cur.ptr(), bytes, &full[slot], pol);
    ++k;
    if (pf_live && (pf_live = pf.next(plan, n_ops, total))) prefetch_l2(pf.ptr(), pf.bytes());
  }
  // every copy issued must have landed before this CTA may exit
  for (long long j = k > kSStages ? k - kSStages : 0; j < k; ++j) {
    const int slot = (int)(j % kSStages);
    const uint32_t par = (uint32_t)((j / kSStages) & 1);
    const unsigned long long t0 = now_ns();
    for (uint32_t i = 0; !mbar_try_wait(&full[slot], par); ++i)
      if (i > kSPollLimit || now_ns() - t0 > kSTimeoutNs) {
        if (err) atomicExch(err, 2);
        break;
      }
  }
}

// ------------------------------------------------------------ the consumers

// Grid barrier between operations (consumer threads only): all consumers of
// this CTA done with the previous operation, then thread 0 arrives (release)
// and polls (acquire) until every CTA has; bounded, abort-aware.
S2_DEV void grid_sync(unsigned* bar, int* abort_g, StreamState* st, int* err, int ctid) {
  consumer_bar();
  if (ctid == 0) {
    st->target += gridDim.x;
    if (!st->abort) {
      asm volatile("red.release.gpu.global.add.u32 [%0], 1;" :: "l"(bar) : "memory");
      const unsigned long long t0 = now_ns();
      for (uint32_t it = 0; ld_acquire_u32(bar) < st->target; ++it) {
        if ((it & 255u) == 255u) {
          if (*reinterpret_cast<volatile int*>(abort_g)) { st->abort = 1; break; }
          if (it > (1u << 26) || now_ns() - t0 > kSTimeoutNs) {
            atomicExch(abort_g, 1);
            if (err) atomicExch(err, 2);
            st->abort = 1;
            break;
          }
        }
      }
    }
    st->stop = *reinterpret_cast<volatile int*>(&st->abort);
  }
  consumer_bar();
}

template <int MAXB>
S2_DEV void consume_gemv(const GemvArgs& a, const StreamPlan& sp, const StreamLayout& L, uint8_t* ring,
                         uint8_t* work, uint64_t* full, uint64_t* empty, long long& kc, StreamState* st,
                         int* err, const int ctid, unsigned long long* tr) {
  const int cw = ctid >> 5, lane = ctid & 31;
  const int B = a.B, K = a.K;
  const int cta = blockIdx.x, ncta = gridDim.x;
  int r0, nrows;
  cta_rows(a.N, a.unit, cta, ncta, r0, nrows);
  const int rc = sp.rc, P = sp.parts;
  const int V = K / 8;                       // 16-byte weight vectors per row
  const int jr = cw / P, p = cw % P;         // this warp's row of a slot and K-part
  const int vb = (int)((long long)V * p / P), ve = (int)((long long)V * (p + 1) / P);
  const bool busy = cw < rc * P;
  const int KP = (K + 255) / 256 * 256;
  const bool staged = sp.stage != 0;
  float* xs = reinterpret_cast<float*>(work + L.xs_off);
  float* res = reinterpret_cast<float*>(work + L.res_off);
  float* yold = reinterpret_cast<float*>(work + L.yold_off);
  float* part = reinterpret_cast<float*>(work + L.part_off);
  float* ssq = reinterpret_cast<float*>(work + L.ssq_off);   // [16][MAXB], then inv[MAXB]

  // prologue: activations into shared memory (RMSNorm-ed for normalised
  // projections: the sum of squares in the stand-alone kernel's order)
  if (a.gain) {
#pragma unroll
    for (int b = 0; b < MAXB; ++b) {
      if (b < B) {
        const float* xr = a.X + (size_t)b * a.ldx;
        float s = 0.f;
        for (int k = ctid * 4; k < K; k += kSConsumers * 4) {
          const float4 v = *reinterpret_cast<const float4*>(xr + k);
          s += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
        s = warp_sum(s);
        if (lane == 0) ssq[cw * MAXB + b] = s;
      }
    }
    consumer_bar();
    // every thread adds the warps' sums itself (same order for all: no
    // second barrier)
    float inv[MAXB];
#pragma unroll
    for (int b = 0; b < MAXB; ++b) {
      float s = 0.f;
      if (b < B)
        for (int w = 0; w < kSCWarps; ++w) s += ssq[w * MAXB + b];
      inv[b] = rsqrtf(s / (float)K + a.eps);
    }
    for (int i = ctid * 4; i < B * K; i += kSConsumers * 4) {
      const int b = i / K, k = i % K;
      const float4 v = *reinterpret_cast<const float4*>(a.X + (size_t)b * a.ldx + k);
      const float4 g = *reinterpret_cast<const float4*>(a.gain + k);
      float s = inv[0];
#pragma unroll
      for (int bb = 1; bb < MAXB; ++bb)
        if (b == bb) s = inv[bb];
      const float4 o = make_float4(v.x * s * g.x, v.y * s * g.y, v.z * s * g.z, v.w * s * g.w);
      *reinterpret_cast<float4*>(xs + (size_t)b * KP + xperm<8>(k)) = o;
      if (a.normed_out && cta == 0)
        *reinterpret_cast<float4*>(a.normed_out + (size_t)b * a.normed_ld + k) = o;
    }
  } else if (staged) {
    for (int i = ctid * 4; i < B * K; i += kSConsumers * 4) {
      const int b = i / K, k = i % K;
      *reinterpret_cast<float4*>(xs + (size_t)b * KP + xperm<8>(k)) =
          *reinterpret_cast<const float4*>(a.X + (size_t)b * a.ldx + k);
    }
  }
  if (a.mode == GEMV_ADD)
    for (int i = ctid; i < nrows * B; i += kSConsumers) {
      const int b = i / nrows, row = i % nrows;
      yold[row * MAXB + b] = a.Y[(size_t)b * a.ldy + r0 + row];
    }
  consumer_bar();
  if (tr) tr[2] = now_ns();   // prologue done

  // the CTA's rows, slot by slot, in the order the producer issued them.
  // A warp's dot products of four slots accumulate in registers (two
  // independent FMA chains each); each slot is released as soon as its
  // multiply-adds are done, and the four slots' warp reductions run
  // together afterwards, off the slots' critical path.
  const int nch = (nrows + rc - 1) / rc;
  for (int c0 = 0; c0 < nch; c0 += kSGroup) {
    float acc[kSGroup][MAXB];
#pragma unroll
    for (int u = 0; u < kSGroup; ++u)
#pragma unroll
      for (int b = 0; b < MAXB; ++b) acc[u][b] = 0.f;
#pragma unroll
    for (int u = 0; u < kSGroup; ++u) {
      const int ci = c0 + u;
      if (ci < nch) {   // uniform across the CTA
        const int c = ci * rc;
        const int slot = (int)(kc % kSStages);
        const bool ok = sw_wait(&full[slot], (uint32_t)((kc / kSStages) & 1), st, err);
        if (tr) {   // when the first and the last slot of the operation were ready
          if (ci == 0) tr[3] = now_ns();
          if (ci == nch - 1) tr[4] = now_ns();
        }
        if (ok && busy && jr < min(rc, nrows - c)) {
          const uint4* wr =
              reinterpret_cast<const uint4*>(ring + (size_t)slot * kSSlotBytes + (size_t)jr * K * 2);
          float e0[MAXB], e1[MAXB];
#pragma unroll
          for (int b = 0; b < MAXB; ++b) e0[b] = e1[b] = 0.f;
          for (int v = vb + lane; v < ve; v += 32) {
            float w[8];
            unpack16(wr[v], w);
#pragma unroll
            for (int b = 0; b < MAXB; ++b) {
              if (b < B) {
                float xv[8];
                if (staged) {
                  const float* px = xs + (size_t)b * KP + xperm<8>(v * 8);
                  const float4 f0 = *reinterpret_cast<const float4*>(px);
                  const float4 f1 = *reinterpret_cast<const float4*>(px + 128);
                  xv[0] = f0.x; xv[1] = f0.y; xv[2] = f0.z; xv[3] = f0.w;
                  xv[4] = f1.x; xv[5] = f1.y; xv[6] = f1.z; xv[7] = f1.w;
                } else {
                  load8(a.X + (size_t)b * a.ldx + v * 8, xv);
                }
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                  e0[b] = fmaf(w[e], xv[e], e0[b]);
                  e1[b] = fmaf(w[e + 1], xv[e + 1], e1[b]);
                }
              }
            }
          }
#pragma unroll
          for (int b = 0; b < MAXB; ++b) acc[u][b] = e0[b] + e1[b];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        ++kc;
      }
    }
#pragma unroll
    for (int u = 0; u < kSGroup; ++u) {
      const int c = (c0 + u) * rc;
      if (c0 + u < nch && busy && jr < min(rc, nrows - c)) {   // uniform across the warp
#pragma unroll
        for (int b = 0; b < MAXB; ++b) {
          if (b < B) {
            const float t = warp_sum(acc[u][b]);
            if (lane == 0) part[((c + jr) * P + p) * MAXB + b] = t;
          }
        }
      }
    }
  }
  consumer_bar();
  // each row's K-parts, added in part order.  Store, residual and SwiGLU
  // finish right here; the arg-max heads go through the shared epilogue.
  // (After an abort the results are void -- the error word says so -- but
  // every consumer thread still reaches the same barriers.)
  auto row_sum = [&](int row, int b) {
    float t = 0.f;
    for (int q = 0; q < P; ++q) t += part[(row * P + q) * MAXB + b];
    return t;
  };
  if (a.mode == GEMV_STORE || a.mode == GEMV_ADD) {
    for (int i = ctid; i < nrows * B; i += kSConsumers) {
      const int b = i / nrows, row = i % nrows;
      const float t = row_sum(row, b);
      a.Y[(size_t)b * a.ldy + r0 + row] = a.mode == GEMV_ADD ? yold[row * MAXB + b] + t : t;
    }
    return;
  }
  if (a.mode == GEMV_SWIGLU) {   // rows (2i, 2i+1) = (gate_i, up_i)
    const int np = nrows / 2;
    for (int i = ctid; i < np * B; i += kSConsumers) {
      const int b = i / np, pr = i % np;
      const float g = row_sum(2 * pr, b), u = row_sum(2 * pr + 1, b);
      a.Y[(size_t)b * a.ldy + (r0 >> 1) + pr] = g / (1.f + __expf(-g)) * u;
    }
    return;
  }
  for (int i = ctid; i < nrows * B; i += kSConsumers) {
    const int row = i / B, b = i % B;
    res[row * MAXB + b] = row_sum(row, b);
  }
  consumer_bar();
  gemv_epilogue<MAXB>(a, res, yold, r0, nrows, cta, ncta, ctid, kSConsumers, [] { consumer_bar(); });
}

template <int MAXB>
__global__ void __launch_bounds__(kSThreads, 1)
stream_decode_kernel(const PersistOp* __restrict__ ops, const StreamPlan* __restrict__ plan, int n_ops,
                     int n_frames, int pf_ahead, StreamLayout L, unsigned* bar, int* abort_g, int* err,
                     unsigned long long* trace) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kSStages], empty[kSStages];
  __shared__ StreamState st;
  uint8_t* ring = smem;
  uint8_t* work = smem + kSRingBytes;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kSCWarps);
    }
    st.target = 0;
    st.abort = 0;
    st.stop = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x >= kSConsumers) {   // the producer warp (lane 0 issues)
    if (threadIdx.x == kSConsumers)
      producer(ops, plan, n_ops, n_frames, pf_ahead, ring, full, empty, &st, err);
    return;
  }
  const int ctid = threadIdx.x;
  const int total = n_ops * n_frames;
  const int trace_frame = n_frames > 1 ? 1 : 0;
  const bool tracer = trace && blockIdx.x == 0 && ctid == 0;
  long long kc = 0;   // slots consumed
  for (int t = 0; t < total; ++t) {
    const int i = t % n_ops;
    const bool traced = tracer && t / n_ops == trace_frame;
    unsigned long long* tr = traced ? trace + (size_t)i * kSTraceWords : nullptr;
    if (tr) tr[0] = now_ns();
    if (t > 0) grid_sync(bar, abort_g, &st, err, ctid);
    if (st.stop) break;   // written by thread 0 before grid_sync's last barrier: uniform
    if (tr) tr[1] = now_ns();
    const PersistOp& op = ops[i];
    if (op.kind == PK_GEMV) {
      consume_gemv<MAXB>(op.g, plan[i], L, ring, work, full, empty, kc, &st, err, ctid, tr);
    } else if (op.kind == PK_ATTN) {
      const AttnDecodeArgs& a = op.at;
      if (ctid < 128) {
        AttnS& S = *reinterpret_cast<AttnS*>(work);
        const int units = a.B * a.Hkv * a.nsplit;
        auto none = [] {};
        for (int u = blockIdx.x; u < units; u += gridDim.x) {
          const int b = u % a.B, g = (u / a.B) % a.Hkv, split = u / (a.B * a.Hkv);
          attn_body<float, 128, 4, false, true>(a, b, g, split, ctid, kSBarAttn, S, none);
        }
      }
    } else if (op.kind == PK_EMBED) {
      const int nb = (op.e.d + kSConsumers - 1) / kSConsumers;
      for (int u = blockIdx.x; u < op.e.rows * nb; u += gridDim.x)
        embed_body<__nv_bfloat16>(op.e, u / nb, (u % nb) * kSConsumers, op.e.d, ctid, [] {});
    }
    if (tr) tr[5] = now_ns();
  }
}

using StreamKernel = void (*)(const PersistOp*, const StreamPlan*, int, int, int, StreamLayout, unsigned*,
                              int*, int*, unsigned long long*);

StreamKernel stream_kernel_for(int maxb) {
  switch (maxb) {
    case 1: return stream_decode_kernel<1>;
    case 2: return stream_decode_kernel<2>;
    case 4: return stream_decode_kernel<4>;
    default: return nullptr;
  }
}

}  // namespace

// Plan of a recorded frame for the streaming kernel; false when an operation
// has no streaming counterpart or the shared memory does not fit.
bool stream_plan(const std::vector<PersistOp>& ops, int grid, std::vector<StreamPlan>& plan,
                 StreamLayout& L, int& maxb) {
  plan.assign(ops.size(), StreamPlan{});
  int rows = 1;
  for (const PersistOp& op : ops) {
    if (op.kind == PK_GEMV) rows = std::max(rows, op.g.B);
    // attention: the S2 head shape with fp32 pages (keys staged by cp.async;
    // a bf16 cache stays on the per-frame graphs)
    if (op.kind == PK_ATTN && (op.at.hd != 128 || op.at.H != 4 * op.at.Hkv || op.at.kv_bf16)) return false;
    if (op.kind == PK_EMBED && !op.e.w_bf16) return false;
  }
  maxb = rows <= 1 ? 1 : rows <= 2 ? 2 : rows <= 4 ? 4 : 0;
  if (!maxb) return false;
  auto al = [](size_t x) { return (x + 127) / 128 * 128; };
  size_t rows_max = 0, part_max = 0;
  for (size_t i = 0; i < ops.size(); ++i) {
    const PersistOp& op = ops[i];
    if (op.kind != PK_GEMV) continue;
    const GemvArgs& a = op.g;
    if (!a.w_is_bf16 || a.w_int8 || a.K % 8 || a.N % a.unit || a.B < 1 || a.B > maxb) return false;
    if (a.mode == GEMV_ARGMAX && (!a.part_val || !a.part_idx || !a.ticket)) return false;
    const int rowbytes = a.K * 2;
    int rc = 1;
    while (rc * 2 <= kSCWarps && rc * 2 * rowbytes <= kSSlotBytes) rc *= 2;
    if (rowbytes > kSSlotBytes) return false;
    StreamPlan& sp = plan[i];
    sp.W = a.W;
    sp.rowbytes = rowbytes;
    sp.N = a.N;
    sp.unit = a.unit;
    sp.rc = rc;
    sp.parts = kSCWarps / rc;
    const size_t nr = ((size_t)(a.N / a.unit) + grid - 1) / grid * a.unit;
    rows_max = std::max(rows_max, nr);
    part_max = std::max(part_max, nr * sp.parts);
  }
  L.res_off = 0;
  L.yold_off = (int)al(rows_max * maxb * 4);
  L.part_off = L.yold_off + (int)al(rows_max * maxb * 4);
  L.ssq_off = L.part_off + (int)al(part_max * maxb * 4);
  L.xs_off = L.ssq_off + (int)al((kSCWarps + 1) * maxb * 4);
  // static shared memory of the kernel (barriers, the epilogue's words, the
  // state) stays below 1 KB
  const size_t cap = kSMaxSmem - 1024 - kSRingBytes;
  if ((size_t)L.xs_off > cap) return false;
  size_t xs_max = 0;
  for (size_t i = 0; i < ops.size(); ++i) {
    const PersistOp& op = ops[i];
    if (op.kind != PK_GEMV) continue;
    const size_t xs = (size_t)op.g.B * ((op.g.K + 255) / 256 * 256) * 4;
    if (L.xs_off + xs <= cap) {
      plan[i].stage = 1;
      xs_max = std::max(xs_max, xs);
    } else if (op.g.gain) {
      return false;   // the RMSNorm prologue needs the staged activations
    }
  }
  L.work_bytes = (int)std::max(L.xs_off + al(xs_max), al(sizeof(AttnS)));
  if ((size_t)L.work_bytes > cap) return false;
  return true;
}

size_t stream_smem_bytes(const StreamLayout& L) { return (size_t)kSRingBytes + L.work_bytes; }

bool stream_fits(int maxb, size_t smem) {
  StreamKernel k = stream_kernel_for(maxb);
  if (!k || smem > (size_t)kSMaxSmem) return false;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kSThreads, smem) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return per_sm >= 1;
}

cudaError_t launch_stream(const PersistOp* ops, const StreamPlan* plan, int n_ops, int n_frames, int maxb,
                          const StreamLayout& L, unsigned* bar, int* abort_flag, int* err, int grid,
                          cudaStream_t st, unsigned long long* trace) {
  StreamKernel k = stream_kernel_for(maxb);
  if (!k || !ops || !plan || n_ops < 1 || n_frames < 1 || !bar || !abort_flag || grid < 1)
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kSThreads);
  cfg.dynamicSmemBytes = stream_smem_bytes(L);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs co-resident: the barrier cannot deadlock
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return s2_launch(&cfg, k, ops, plan, n_ops, n_frames, kStreamPrefetchAhead, L, bar, abort_flag, err,
                   trace);
}

}  // namespace s2
