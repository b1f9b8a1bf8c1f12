// K9 on tcgen05: causal prefill attention (single prompt, or every prompt
// of a batched prefill through a segment table), S = Q K^T and O = P V on the
// tensor cores with split-bf16 operands (hi = bf16(x), lo = bf16(x - hi):
// three products hi hi + hi lo + lo hi, ~16 mantissa bits of both operands),
// the softmax state per row in registers and the running output in tensor
// memory; cached radix keys come from their pages.
#include "s2_kernels.h"
#include "s2_common.cuh"
#include "tc_common.cuh"
#include "attn_tc_util.cuh"

namespace s2 {

namespace {

constexpr int kPxHD = 128;
constexpr int kPxKeys = 64;
constexpr int kPxRows = 128;
constexpr int kPxGroup = 4;
constexpr int kPxPage = 16;      // tokens per KV page
// shared memory: two bf16 planes each of Q [128 rows x 128 dims] (two
// 64-dim k-blocks), K [64 keys x 128 dims] (two k-blocks), V^T [128 dims x 64
// keys], P [128 rows x 64 keys]; every tile on a 1,024-byte boundary
constexpr int kPxQPlane = kPxRows * kPxHD * 2;     // 32 KB
constexpr int kPxKPlane = kPxKeys * kPxHD * 2;     // 16 KB
constexpr int kPxVPlane = kPxHD * kPxKeys * 2;     // 16 KB
constexpr int kPxPPlane = kPxRows * kPxKeys * 2;   // 16 KB
constexpr int kPxOffQ = 0;
constexpr int kPxOffK = kPxOffQ + 2 * kPxQPlane;
constexpr int kPxOffV = kPxOffK + 2 * kPxKPlane;
constexpr int kPxOffP = kPxOffV + 2 * kPxVPlane;
constexpr int kPxSmem = kPxOffP + 2 * kPxPPlane + 1024;   // + alignment slack
constexpr int kPxTmemCols = 256;   // S: columns 0..63, O: columns 128..255

// Keys [k0, k0 + nk) of kv head g (pages from ``table``) into the K planes
// (K-major) and the V^T planes (hd rows x 64 keys); keys past nk are zero.
// Thread tid moves key tid / 2, dims 64 * (tid % 2) .. + 64.
template <typename KT>
S2_DEV void stage_kv_chunk(uint8_t* sm, const void* kv_base, const int* table, long long page_elems, int Hkv,
                           int g, int k0, int nk, int tid) {
  uint8_t* k_hi = sm + kPxOffK;
  uint8_t* k_lo = k_hi + kPxKPlane;
  uint8_t* v_hi = sm + kPxOffV;
  uint8_t* v_lo = v_hi + kPxVPlane;
  const int kk = tid >> 1, half = tid & 1;
  const KT* kv = reinterpret_cast<const KT*>(kv_base);
  const bool key_ok = kk < nk;
  const KT* ks = nullptr;
  if (key_ok) {
    const int kp = k0 + kk;
    const int page = table[kp / kPxPage];
    ks = kv + (size_t)page * page_elems + ((size_t)g * kPxPage + kp % kPxPage) * kPxHD + half * 64;
  }
  const KT* vs = key_ok ? ks + (size_t)Hkv * kPxPage * kPxHD : nullptr;
  // four 8-dim units of keys and values loaded before any is converted: two
  // rounds of load latency per chunk instead of eight
#pragma unroll
  for (int c0 = 0; c0 < 8; c0 += 4) {
    float x[4][8], y[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (key_ok) {
        load8kv<KT>(ks + (c0 + u) * 8, x[u]);
        load8kv<KT>(vs + (c0 + u) * 8, y[u]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[u][e] = y[u][e] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + u;
      uint4 hi, lo;
      split8(x[u], hi, lo);
      st_shared16(k_hi + half * (kPxKPlane / 2), sw128_offset(kk, c), hi);
      st_shared16(k_lo + half * (kPxKPlane / 2), sw128_offset(kk, c), lo);
#pragma unroll
      for (int e = 0; e < 8; ++e) {   // V^T[dim][key]
        const int dim = half * 64 + c * 8 + e;
        const float vh = __bfloat162float(__float2bfloat16_rn(y[u][e]));
        const uint32_t off = sw128_offset(dim, kk >> 3) + (kk & 7) * 2;
        st_shared_bf16(v_hi, off, vh);
        st_shared_bf16(v_lo, off, y[u][e] - vh);
      }
    }
  }
}

// One thread: S = Q K^T (M 128 rows, N 64 keys, K 128 dims) into t_s as the
// three plane products, then a commit to ``bar``.
S2_DEV void issue_qk(uint8_t* sm, uint32_t t_s, uint64_t* bar) {
  constexpr uint32_t idesc = idesc_bf16(kPxRows, kPxKeys);
  uint8_t* q_hi = sm + kPxOffQ;
  uint8_t* q_lo = q_hi + kPxQPlane;
  uint8_t* k_hi = sm + kPxOffK;
  uint8_t* k_lo = k_hi + kPxKPlane;
  const uint8_t* qa[3] = {q_hi, q_hi, q_lo};
  const uint8_t* kb_[3] = {k_hi, k_lo, k_hi};
  uint32_t acc = 0;
  for (int pr = 0; pr < 3; ++pr)
    for (int kb = 0; kb < 2; ++kb)
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const uint32_t aa = smem_u32(qa[pr] + kb * (kPxQPlane / 2)) + ks * 32;
        const uint32_t ba = smem_u32(kb_[pr] + kb * (kPxKPlane / 2)) + ks * 32;
        umma_bf16(t_s, smem_desc_sw128(aa), smem_desc_sw128(ba), idesc, acc);
        acc = 1;
      }
  umma_commit(bar);
}

// One thread: O (+)= P V (M 128 rows, N 128 dims, K 64 keys) into t_o, the
// first product accumulating iff acc0, then a commit to ``bar``.
S2_DEV void issue_pv(uint8_t* sm, uint32_t t_o, uint32_t acc0, uint64_t* bar) {
  constexpr uint32_t idesc = idesc_bf16(kPxRows, kPxHD);
  uint8_t* p_hi = sm + kPxOffP;
  uint8_t* p_lo = p_hi + kPxPPlane;
  uint8_t* v_hi = sm + kPxOffV;
  uint8_t* v_lo = v_hi + kPxVPlane;
  const uint8_t* pa[3] = {p_hi, p_hi, p_lo};
  const uint8_t* vb[3] = {v_hi, v_lo, v_hi};
  uint32_t acc = acc0;
  for (int pr = 0; pr < 3; ++pr)
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      umma_bf16(t_o, smem_desc_sw128(smem_u32(pa[pr]) + ks * 32), smem_desc_sw128(smem_u32(vb[pr]) + ks * 32),
                idesc, acc);
      acc = 1;
    }
  umma_commit(bar);
}

// K9 on tcgen05: causal prefill attention of one sequence.  Grid (kv head g,
// query tile of 32 tokens x the 4 heads of g); 128 threads, thread = query
// row.  The queries arrive normalised, rotated and pre-scaled (fp32); keys
// 0 .. pos0 + T - 1 (cached pages first, then the new rows' appended keys)
// are taken in 64-key chunks: S = Q K^T on the tensor cores, the row's
// softmax state (max m, sum l) updated in registers, the running output in
// tensor memory scaled by exp(m_old - m_new) before O += P V.  Rows stop at
// their own position (causal); the output is O / l.
template <typename KT>
__global__ void __launch_bounds__(128, 1)
attn_prefill_tc_kernel(AttnPrefillArgs a) {
  extern __shared__ __align__(1024) uint8_t px_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(px_raw) + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t bar_s, bar_o;
  __shared__ uint32_t tmem_base;
  const int g = blockIdx.x, qt = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5;
  constexpr int kTok = kPxRows / kPxGroup;   // 32 tokens per tile

  pdl_launch_next();
  pdl_wait();
  // this tile's sequence: its rows, first position, page table (batched
  // prefill: from the segment table; rows of q and the output are global)
  int T = a.T, pos0 = a.pos0, row0 = 0, tl = qt;
  const int* table = a.table;
  if (a.segs.info) {
    const int* si = a.segs.info + 5 * a.segs.tile_seg[qt];
    row0 = si[0];
    T = si[1];
    pos0 = si[2];
    table = a.segs.tables + si[3];
    tl = qt - si[4];
  }
  const int t0 = tl * kTok;
  const int t = t0 + tid / kPxGroup, h = g * kPxGroup + tid % kPxGroup;
  const bool row_ok = t < T;
  const int kend = pos0 + min(T, t0 + kTok);   // keys the tile needs
  const int kmax = pos0 + t;                   // this row's last key
  const int nch = (kend + kPxKeys - 1) / kPxKeys;
  const int qd = a.H * kPxHD;
  if (tid == 0) {
    mbar_init(&bar_s, 1);
    mbar_init(&bar_o, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(&tmem_base)), "n"(kPxTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // the query row (already normalised, rotated and scaled) as two planes
  uint8_t* q_hi = sm + kPxOffQ;
  uint8_t* q_lo = q_hi + kPxQPlane;
  const float* q = a.q + (size_t)(row0 + t) * qd + (size_t)h * kPxHD;
  for (int c = 0; c < 16; ++c) {
    float x[8];
    if (row_ok) {
      const float4 u = *reinterpret_cast<const float4*>(q + c * 8);
      const float4 w = *reinterpret_cast<const float4*>(q + c * 8 + 4);
      x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w; x[4] = w.x; x[5] = w.y; x[6] = w.z; x[7] = w.w;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = 0.f;
    }
    uint4 hi, lo;
    split8(x, hi, lo);
    const int kb = c / 8;
    st_shared16(q_hi + kb * (kPxQPlane / 2), sw128_offset(tid, c % 8), hi);
    st_shared16(q_lo + kb * (kPxQPlane / 2), sw128_offset(tid, c % 8), lo);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  const uint32_t t_s = tmem, t_o = tmem + 128;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  uint8_t* p_hi = sm + kPxOffP;
  uint8_t* p_lo = p_hi + kPxPPlane;
  float m_run = -INFINITY, l_run = 0.f;
  bool ok = true;
  for (int j = 0; j < nch; ++j) {
    const int k0 = j * kPxKeys;
    const int nk = min(kPxKeys, kend - k0);
    // the previous chunk's P V has read P and V: their planes are free
    if (j > 0) ok = mbar_wait(&bar_o, (uint32_t)((j - 1) & 1), a.err) && ok;
    stage_kv_chunk<KT>(sm, a.kv, table, a.page_elems, a.Hkv, g, k0, nk, tid);
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) issue_qk(sm, t_s, &bar_s);
    __syncwarp();
    ok = mbar_wait(&bar_s, (uint32_t)(j & 1), a.err) && ok;
    tc_fence_after();
    float s[kPxKeys];
#pragma unroll
    for (int c = 0; c < kPxKeys; c += 8) {
      float v[8];
      tmem_ld8(t_s + lane_base + c, v);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int key = k0 + c + e;
        s[c + e] = (c + e < nk && key <= kmax) ? v[e] : -INFINITY;
      }
    }
    float mc = -INFINITY;
#pragma unroll
    for (int e = 0; e < kPxKeys; ++e) mc = fmaxf(mc, s[e]);
    const float m_new = fmaxf(m_run, mc);
    const float corr = (m_new == -INFINITY || m_run == -INFINITY) ? 0.f : __expf(m_run - m_new);
    float lc = 0.f;
#pragma unroll
    for (int c = 0; c < kPxKeys; c += 8) {
      float pv[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        pv[e] = s[c + e] == -INFINITY ? 0.f : __expf(s[c + e] - m_new);
        lc += pv[e];
      }
      uint4 hi, lo;
      split8(pv, hi, lo);
      st_shared16(p_hi, sw128_offset(tid, c / 8), hi);
      st_shared16(p_lo, sw128_offset(tid, c / 8), lo);
    }
    l_run = l_run * corr + lc;
    if (j > 0) {
      // the running output (complete: the previous P V was awaited above)
      // scaled to the new maximum, in tensor memory
#pragma unroll 1
      for (int c = 0; c < kPxHD; c += 8) {
        float v[8];
        tmem_ld8(t_o + lane_base + c, v);
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] *= corr;
        tmem_st8(t_o + lane_base + c, v);
      }
    }
    m_run = m_new;
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) issue_pv(sm, t_o, j > 0 ? 1u : 0u, &bar_o);
    __syncwarp();
  }
  if (nch > 0) ok = mbar_wait(&bar_o, (uint32_t)((nch - 1) & 1), a.err) && ok;
  tc_fence_after();
  const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll 1
  for (int c = 0; c < kPxHD; c += 8) {
    float v[8];
    tmem_ld8(t_o + lane_base + c, v);
    if (row_ok) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float y = ok ? v[e] * inv : 0.f;
        const size_t col = (size_t)h * kPxHD + c + e;
        if (a.o) a.o[(size_t)(row0 + t) * a.o_ld + col] = y;
        if (a.o16) st_bf16_split(a.o16, a.o16lo, (size_t)(row0 + t) * a.o16_ld + col, y);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "n"(kPxTmemCols)
                 : "memory");
  }
}

}  // namespace

bool attn_prefill_tc_supported(const AttnPrefillArgs& a) {
  // 16-byte loads of the query rows and the pages
  return a.hd == kPxHD && a.H == kPxGroup * a.Hkv && a.T > 0 && a.table && a.q &&
         !(reinterpret_cast<uintptr_t>(a.q) & 15) && !(reinterpret_cast<uintptr_t>(a.kv) & 15);
}

static cudaError_t launch_prefill_tc_grid(const AttnPrefillArgs& a, int q_tiles, cudaStream_t st, bool pdl);

cudaError_t launch_attn_prefill_tc(const AttnPrefillArgs& a, cudaStream_t st, bool pdl) {
  if (!attn_prefill_tc_supported(a)) return cudaErrorInvalidValue;
  return launch_prefill_tc_grid(a, (a.T + kPxRows / kPxGroup - 1) / (kPxRows / kPxGroup), st, pdl);
}

cudaError_t launch_attn_prefill_segs(const AttnPrefillArgs& a, cudaStream_t st, bool pdl) {
  if (!a.segs.info || !a.segs.tile_seg || !a.segs.tables || a.segs.n_tiles < 1 || a.T < 1 || !a.q)
    return cudaErrorInvalidValue;
  if (!a.tc || a.hd != kPxHD || a.H != kPxGroup * a.Hkv || (reinterpret_cast<uintptr_t>(a.q) & 15) ||
      (reinterpret_cast<uintptr_t>(a.kv) & 15))
    return cudaErrorNotSupported;
  return launch_prefill_tc_grid(a, a.segs.n_tiles, st, pdl);
}

static cudaError_t launch_prefill_tc_grid(const AttnPrefillArgs& a, int q_tiles, cudaStream_t st, bool pdl) {
  auto k = a.kv_bf16 ? attn_prefill_tc_kernel<__nv_bfloat16> : attn_prefill_tc_kernel<float>;
  static bool attr[2] = {false, false};
  if (!attr[a.kv_bf16 ? 1 : 0]) {
    const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kPxSmem);
    if (e != cudaSuccess) return e;
    attr[a.kv_bf16 ? 1 : 0] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.Hkv, q_tiles);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = kPxSmem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return s2_launch(&cfg, k, a);
}

}  // namespace s2
