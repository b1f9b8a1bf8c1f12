// K11: decode attention over a radix-shared prefix on the tensor cores.
//
// When the sequences of a decode batch share their first P cached keys (one
// set of radix-cached prompt pages: "SGLang Day-0 Support for FishAudio S2",
// Optimizations with SGLang Omni -- paged KV with radix prefix reuse; the
// batch-32 workload shares a 900-position VQ prompt), the attention over
// those keys is one dense contraction per kv head: the batch's B sequences x
// 4 query heads form a 128-row query tile that meets the same keys.
//
// Two launches:
//   * attn_prefix_planes_kernel, once per decode call: the prefix keys and
//     values of every layer, read from their pages, written once as the
//     tensor-core operand images the MMAs consume -- two bf16 planes (hi =
//     bf16(x), lo = bf16(x - hi)) in the 128-byte swizzled K-major layout,
//     keys K-major and values transposed.  The pages of a shared prefix do
//     not change while it is shared, so each frame's prefix attention only
//     copies these images (bulk copies) instead of converting fp32 rows.
//   * attn_prefix_cl_kernel, once per layer per frame, after the split-KV
//     decode attention has left its partials (m, l, O) for the private keys
//     (keys P.., merge_later): one thread-block cluster of 8 CTAs per (kv
//     head, 128-row query tile).  CTA rank c takes the 128-key chunks c, c +
//     8, ...: bulk copies of the chunk's images (issued before the wait on
//     the previous launch: the images do not depend on it), and of the
//     query tile the split-KV launch wrote (its normalised, rotated, scaled
//     query rows as two bf16 planes in the same layout), S = Q K^T and O =
//     P V each as three tcgen05 MMAs (hi hi + hi lo + lo hi) into tensor
//     memory, the softmax in registers; chunks of one CTA are combined in
//     registers.  The 8 partials are then merged through distributed shared
//     memory (rank order), together with the private-key partial slots
//     (split order), into the softmax-normalised output rows (fp32 and / or
//     the bf16 hi + lo planes of the O projection's input).
//
// Every wait is bounded; after a wait that gave up the error word is set,
// the CTA's partial is left out (void results, reported by the error word)
// and the issuing thread waits once more (bounded) for what it issued before
// the CTA exits.
#include "s2_kernels.h"
#include "s2_common.cuh"
#include "tc_common.cuh"
#include "attn_tc_util.cuh"

namespace s2 {

namespace {

constexpr int kPcHD = 128;
constexpr int kPcRows = 128;      // query rows of a tile: 32 sequences x 4 heads
constexpr int kPcGroup = 4;       // query heads per kv head
constexpr int kPcChunk = 128;     // keys per chunk
constexpr int kPcCluster = 8;     // CTAs per (kv head, query tile)
constexpr int kPcPage = 16;       // tokens per KV page
constexpr int kPcThreads = 256;
constexpr int kPcKeyBytes = 8 * kPcHD;   // image bytes per key: K hi, K lo, V hi, V lo (bf16)
// shared memory: six [128 x 128] bf16 planes (each two 64-column k-blocks of
// 16 KB), every tile on a 1,024-byte boundary
constexpr int kPcPlane = kPcRows * kPcHD * 2;   // 32 KB
constexpr int kPcKb = kPcPlane / 2;             // 16 KB: one k-block of a plane
constexpr int kPcOffQ = 0;                      // Q hi, Q lo
constexpr int kPcOffK = 2 * kPcPlane;           // K hi, K lo; then P hi, P lo
constexpr int kPcOffV = 4 * kPcPlane;           // V^T hi, V^T lo
constexpr int kPcSmem = 6 * kPcPlane + 1024;    // + alignment slack
constexpr int kPcOst = kPcHD + 4;               // row stride (floats) of the staged partial O
constexpr int kPcTmemCols = 256;                // S: columns 0..127, O: 128..255
static_assert(kPcRows * kPcOst * 4 <= 4 * kPcPlane, "the staged O fits the Q and K regions");

// Byte offsets inside the image of one (layer, kv head) of `stride` keys:
//   K hi  [k-block kb][key][128 B]              at kb * stride * 128
//   K lo  the same                              at 2 * stride * 128
//   V hi  [64-key block j][dim][128 B]          at 4 * stride * 128 + j * 16 KB
//   V lo  the same                              at 6 * stride * 128
// Rows are in the 128-byte swizzled layout of their 8-row atom, so a chunk
// of 128 keys (a multiple of 8 rows) lands in shared memory as it is.
S2_DEV size_t img_k(int stride, int lo) { return (size_t)lo * 2 * stride * 128; }
S2_DEV size_t img_v(int stride, int lo) { return (size_t)(4 + 2 * lo) * stride * 128; }

// One 64-key block j of kv head g in layer l: keys 64 j .. 64 j + 63 (zero
// past P).  Thread t reads key t / 4, dims 32 (t % 4) .. + 31 of K and V;
// the values go through shared memory to be transposed.
template <typename KT>
__global__ void __launch_bounds__(256) attn_prefix_planes_kernel(PrefixPlanesArgs p) {
  __shared__ __align__(16) float vs[64][kPcHD + 4];
  const int j = blockIdx.x, g = blockIdx.y, l = blockIdx.z;
  const int tid = threadIdx.x;
  const int kk = tid >> 2, qd = tid & 3;
  const int k = j * 64 + kk;
  const KT* kv = reinterpret_cast<const KT*>(static_cast<const char*>(p.kv) + (size_t)l * p.layer_bytes);
  uint8_t* img = static_cast<uint8_t*>(p.planes) + ((size_t)l * p.Hkv + g) * (size_t)p.stride * kPcKeyBytes;
  float x[4][8], y[4][8];
  if (k < p.P) {
    const int page = p.table[k / kPcPage];
    const KT* ks = kv + (size_t)page * p.page_elems + ((size_t)g * kPcPage + k % kPcPage) * kPcHD + 32 * qd;
    const KT* vsrc = ks + (size_t)p.Hkv * kPcPage * kPcHD;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      load8kv<KT>(ks + 8 * u, x[u]);
      load8kv<KT>(vsrc + 8 * u, y[u]);
    }
  } else {
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int e = 0; e < 8; ++e) x[u][e] = y[u][e] = 0.f;
  }
  // keys: units 4 (qd % 2) .. + 3 of k-block qd / 2, row k
  const int kb = qd >> 1;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    uint4 hi, lo;
    split8(x[u], hi, lo);
    const size_t off = (size_t)kb * p.stride * 128 + sw128_offset(k, 4 * (qd & 1) + u);
    *reinterpret_cast<uint4*>(img + img_k(p.stride, 0) + off) = hi;
    *reinterpret_cast<uint4*>(img + img_k(p.stride, 1) + off) = lo;
  }
  // values: V^T rows (one dim, 8 keys per 16-byte unit) from shared memory
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    *reinterpret_cast<float4*>(&vs[kk][32 * qd + 8 * u]) = make_float4(y[u][0], y[u][1], y[u][2], y[u][3]);
    *reinterpret_cast<float4*>(&vs[kk][32 * qd + 8 * u + 4]) = make_float4(y[u][4], y[u][5], y[u][6], y[u][7]);
  }
  __syncthreads();
  const int d = tid >> 1, kh = tid & 1;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = vs[32 * kh + 8 * u + e][d];
    uint4 hi, lo;
    split8(v, hi, lo);
    const size_t off = (size_t)j * kPcKb + sw128_offset(d, 4 * kh + u);
    *reinterpret_cast<uint4*>(img + img_v(p.stride, 0) + off) = hi;
    *reinterpret_cast<uint4*>(img + img_v(p.stride, 1) + off) = lo;
  }
}

// One thread: S = Q K^T (M 128 rows, N n16 keys, K 128 dims) into t_s as the
// three plane products, then a commit to ``bar``.
S2_DEV void pc_issue_qk(uint8_t* sm, uint32_t t_s, int n16, uint64_t* bar) {
  const uint32_t idesc = idesc_bf16(kPcRows, n16);
  const uint8_t* qa[3] = {sm + kPcOffQ, sm + kPcOffQ, sm + kPcOffQ + kPcPlane};
  const uint8_t* kb_[3] = {sm + kPcOffK, sm + kPcOffK + kPcPlane, sm + kPcOffK};
  uint32_t acc = 0;
  for (int pr = 0; pr < 3; ++pr)
    for (int kb = 0; kb < 2; ++kb)
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const uint32_t aa = smem_u32(qa[pr] + kb * kPcKb) + ks * 32;
        const uint32_t ba = smem_u32(kb_[pr] + kb * kPcKb) + ks * 32;
        umma_bf16(t_s, smem_desc_sw128(aa), smem_desc_sw128(ba), idesc, acc);
        acc = 1;
      }
  umma_commit(bar);
}

// One thread: O = P V (M 128 rows, N 128 dims, K n16 keys) into t_o, then a
// commit to ``bar``.  P sits in the K region, V^T in the V region.
S2_DEV void pc_issue_pv(uint8_t* sm, uint32_t t_o, int n16, uint64_t* bar) {
  constexpr uint32_t idesc = idesc_bf16(kPcRows, kPcHD);
  const uint8_t* pa[3] = {sm + kPcOffK, sm + kPcOffK, sm + kPcOffK + kPcPlane};
  const uint8_t* vb[3] = {sm + kPcOffV, sm + kPcOffV + kPcPlane, sm + kPcOffV};
  uint32_t acc = 0;
  for (int pr = 0; pr < 3; ++pr)
    for (int st = 0; st < n16 / 16; ++st) {
      const int kb = st >> 2, ks = st & 3;
      const uint32_t aa = smem_u32(pa[pr] + kb * kPcKb) + ks * 32;
      const uint32_t ba = smem_u32(vb[pr] + kb * kPcKb) + ks * 32;
      umma_bf16(t_o, smem_desc_sw128(aa), smem_desc_sw128(ba), idesc, acc);
      acc = 1;
    }
  umma_commit(bar);
}

// Phase trace (attn_prefix_set_trace): per CTA, thread 0 stamps the global
// timer at entry, after setup, after the dependency wait, after the query
// tile's copy is issued, when its first chunk's operands have landed, after
// S, after the softmax, after P V (first chunk), after the last chunk, after
// the first cluster barrier, after the merge and at exit (12 of 16 slots).
constexpr int kPcTraceSlots = 16;
unsigned long long* g_pc_trace = nullptr;
int g_pc_trace_ctas = 0;

__global__ void __launch_bounds__(kPcThreads, 1)
attn_prefix_cl_kernel(AttnDecodeArgs a, const uint8_t* __restrict__ planes, int stride,
                      unsigned long long* trace, int trace_ctas) {
  extern __shared__ __align__(1024) uint8_t pc_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(pc_raw) + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t bar_ld, bar_q, bar_s, bar_o;
  __shared__ uint32_t tmem_base;
  __shared__ float s_mx[2][kPcRows], s_sum[2][kPcRows];   // softmax exchange of a row's two halves
  __shared__ float s_m[kPcRows], s_l[kPcRows];             // this CTA's partial (m, l) per row
  const int rank = (int)cluster_rank();
  const int g = blockIdx.y, qt = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rows_total = a.B * kPcGroup;
  const int cta = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
  auto stamp = [&](int i) {
    if (trace && tid == 0 && cta < trace_ctas) {
      unsigned long long t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      trace[(size_t)cta * kPcTraceSlots + i] = t;
    }
  };
  stamp(0);

  if (tid == 0) {
    mbar_init(&bar_ld, 1);
    mbar_init(&bar_q, 1);
    mbar_init(&bar_s, 1);
    mbar_init(&bar_o, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(&tmem_base)), "n"(kPcTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  const uint32_t t_s = tmem, t_o = tmem + 128;
  stamp(1);

  // the prefix length (set before the decode call) and the images (written
  // by the per-call conversion) do not depend on the previous launch
  const int P = __ldcg(a.key_begin);
  const int nchunks = (P + kPcChunk - 1) / kPcChunk;
  const uint8_t* img = planes + (size_t)g * stride * kPcKeyBytes;
  // tid 0's account of what it issued and has not seen complete (so that a
  // wait that gave up is followed by one more before the CTA exits)
  uint32_t ld_phase = 0, mma_phase = 0;
  bool ld_pending = false, s_pending = false, o_pending = false;
  auto issue_chunk = [&](int j) {
    mbar_arrive_expect_tx(&bar_ld, 4 * kPcKb + 2 * kPcPlane);
#pragma unroll
    for (int lo = 0; lo < 2; ++lo) {
#pragma unroll
      for (int kb = 0; kb < 2; ++kb)
        bulk_g2s(sm + kPcOffK + lo * kPcPlane + kb * kPcKb,
                 img + img_k(stride, lo) + (size_t)kb * stride * 128 + (size_t)j * kPcChunk * 128, kPcKb, &bar_ld);
      bulk_g2s(sm + kPcOffV + lo * kPcPlane, img + img_v(stride, lo) + (size_t)j * 2 * kPcKb, kPcPlane, &bar_ld);
    }
    ld_pending = true;
  };
  if (tid == 0 && rank < nchunks) issue_chunk(rank);

  pdl_launch_next();
  pdl_wait();
  stamp(2);
  // ---- the query tile: written by the split-KV attention just before
  // (normalised, rotated, scaled, as two bf16 planes in the swizzled layout)
  bool q_pending = false;
  if (tid == 0 && rank < nchunks) {
    const int tiles = (rows_total + kPcRows - 1) / kPcRows;
    mbar_arrive_expect_tx(&bar_q, 2 * kPcPlane);
    bulk_g2s(sm + kPcOffQ, a.q_img + ((size_t)g * tiles + qt) * (2 * kPcPlane), 2 * kPcPlane, &bar_q);
    q_pending = true;
  }
  stamp(3);

  // thread = (row = tensor-memory lane of its warp's quarter, half hf of
  // the key / output columns)
  const int lrow = (warp & 3) * 32 + lane, hf = warp >> 2;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  float m_run = -INFINITY, l_run = 0.f, o_run[64];
#pragma unroll
  for (int e = 0; e < 64; ++e) o_run[e] = 0.f;
  bool ok = true;
  for (int j = rank; j < nchunks; j += kPcCluster) {
    const int nk = min(kPcChunk, P - j * kPcChunk);
    const int n16 = (nk + 15) & ~15;
    if (tid == 0) {
      bool got = true;
      if (q_pending) {
        got = mbar_wait(&bar_q, 0, a.err);
        if (got) q_pending = false;
      }
      got = got && mbar_wait(&bar_ld, ld_phase, a.err);
      ok = got && ok;
      if (got) { ld_pending = false; ld_phase ^= 1; }
      if (j == rank) stamp(4);
      tc_fence_after();
      if (got) {
        pc_issue_qk(sm, t_s, n16, &bar_s);
        s_pending = true;
      }
    }
    __syncwarp();
    {
      const bool got = mbar_wait(&bar_s, mma_phase, a.err);
      ok = got && ok;
      if (tid == 0 && got) s_pending = false;
    }
    tc_fence_after();
    if (j == rank) stamp(5);

    // ---- softmax over the chunk's keys: this thread's 64 columns
    float s[64];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float v[32];
      if (64 * hf + 32 * c < nk) {   // warp-uniform
        tmem_ld32(t_s + lane_base + 64 * hf + 32 * c, v);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = -INFINITY;
      }
#pragma unroll
      for (int e = 0; e < 32; ++e) s[32 * c + e] = (64 * hf + 32 * c + e < nk) ? v[e] : -INFINITY;
    }
    float mx = -INFINITY;
#pragma unroll
    for (int e = 0; e < 64; ++e) mx = fmaxf(mx, s[e]);
    s_mx[hf][lrow] = mx;
    __syncthreads();
    const float m_c = fmaxf(s_mx[0][lrow], s_mx[1][lrow]);
    float lsum = 0.f;
    uint8_t* p_hi = sm + kPcOffK + hf * kPcKb;   // P: k-block hf = keys 64 hf ..
    uint8_t* p_lo = p_hi + kPcPlane;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      float pv[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        pv[e] = (64 * hf + 8 * u + e < nk) ? __expf(s[8 * u + e] - m_c) : 0.f;
        lsum += pv[e];
      }
      uint4 hi, lo;
      split8(pv, hi, lo);
      st_shared16(p_hi, sw128_offset(lrow, u), hi);
      st_shared16(p_lo, sw128_offset(lrow, u), lo);
    }
    s_sum[hf][lrow] = lsum;
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const float l_c = s_sum[0][lrow] + s_sum[1][lrow];
    if (j == rank) stamp(6);

    // ---- O = P V
    if (tid == 0 && !s_pending) {
      pc_issue_pv(sm, t_o, n16, &bar_o);
      o_pending = true;
    }
    __syncwarp();
    {
      const bool got = mbar_wait(&bar_o, mma_phase, a.err);
      ok = got && ok;
      if (tid == 0 && got) o_pending = false;
    }
    tc_fence_after();
    if (j == rank) stamp(7);
    mma_phase ^= 1;
    // P and V are read: the next chunk's images may land (tid 0 only issues
    // when everything it issued before has completed)
    if (tid == 0 && j + kPcCluster < nchunks && !ld_pending && !s_pending && !o_pending)
      issue_chunk(j + kPcCluster);

    // ---- the chunk's O into the running partial (thread: 64 output dims)
    const float m_new = fmaxf(m_run, m_c);
    const float wa = __expf(m_run - m_new), wb = __expf(m_c - m_new);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float v[32];
      tmem_ld32(t_o + lane_base + 64 * hf + 32 * c, v);
#pragma unroll
      for (int e = 0; e < 32; ++e) o_run[32 * c + e] = o_run[32 * c + e] * wa + v[e] * wb;
    }
    l_run = l_run * wa + l_c * wb;
    m_run = m_new;
    if (!__syncthreads_and(ok ? 1 : 0)) break;   // uniform: a CTA whose wait gave up stops
  }
  ok = __syncthreads_and(ok ? 1 : 0) != 0;
  stamp(8);

  // ---- the CTA's partial into shared memory for the cluster (the Q and K
  // regions are free: every MMA that read them has completed)
  float* ost = reinterpret_cast<float*>(sm + kPcOffQ);
  const bool has = rank < nchunks && ok;
  if (has) {
#pragma unroll
    for (int e = 0; e < 64; e += 4)
      *reinterpret_cast<float4*>(ost + lrow * kPcOst + 64 * hf + e) =
          make_float4(o_run[e], o_run[e + 1], o_run[e + 2], o_run[e + 3]);
  }
  if (hf == 0) {
    s_m[lrow] = has ? m_run : -INFINITY;
    s_l[lrow] = has ? l_run : 0.f;
  }
  // ---- merge: rank c finalises rows 16 c .. 16 c + 15 (warp w: rows 16 c +
  // 2 w and + 1; lane = 4 output dims): the 8 partials in rank order, then
  // the private-key slots in split order.  The first kPre slots of each row
  // are requested before the cluster barrier (the split-KV launch has
  // completed), the partners' partials right after it, both rows at once.
  constexpr int kPre = 4;
  const int ns = a.nsplit;
  bool rv[2];
  int rb[2], rh[2];
  float pm[2][kPre], pl[2][kPre];
  float2 pa[2][kPre], pb[2][kPre];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = qt * kPcRows + rank * (kPcRows / kPcCluster) + warp * 2 + i;
    rv[i] = r < rows_total;
    rb[i] = r / kPcGroup;
    rh[i] = g * kPcGroup + r % kPcGroup;
    const float* src = a.part + ((size_t)rb[i] * a.H + rh[i]) * ns * (kPcHD + 2);
#pragma unroll
    for (int s = 0; s < kPre; ++s) {
      const bool in = rv[i] && s < ns;
      const float* sp = src + s * (kPcHD + 2);
      pm[i][s] = in ? __ldcg(sp) : -INFINITY;
      pl[i][s] = in ? __ldcg(sp + 1) : 0.f;
      // a slot is hd + 2 floats: its O starts 8-byte aligned
      pa[i][s] = in ? __ldcg(reinterpret_cast<const float2*>(sp + 2 + 4 * lane)) : make_float2(0.f, 0.f);
      pb[i][s] = in ? __ldcg(reinterpret_cast<const float2*>(sp + 4 + 4 * lane)) : make_float2(0.f, 0.f);
    }
  }
  cluster_sync_all();
  stamp(9);
  float mq[2][kPcCluster], lq[2][kPcCluster];
  float4 oq[2][kPcCluster];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int row = rank * (kPcRows / kPcCluster) + warp * 2 + i;
#pragma unroll
    for (int q = 0; q < kPcCluster; ++q) {   // ranks past the chunks hold no partial
      const bool in = rv[i] && q < nchunks;
      mq[i][q] = in ? ld_dsmem_f32(s_m + row, (uint32_t)q) : -INFINITY;
      lq[i][q] = in ? ld_dsmem_f32(s_l + row, (uint32_t)q) : 0.f;
      oq[i][q] = in ? ld_dsmem_f32x4(ost + row * kPcOst + 4 * lane, (uint32_t)q) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (!rv[i]) continue;   // warp-uniform
    const float* src = a.part + ((size_t)rb[i] * a.H + rh[i]) * ns * (kPcHD + 2);
    float M = -INFINITY;
#pragma unroll
    for (int q = 0; q < kPcCluster; ++q) M = fmaxf(M, mq[i][q]);
#pragma unroll
    for (int s = 0; s < kPre; ++s) M = fmaxf(M, pm[i][s]);
    for (int s = kPre; s < ns; ++s) M = fmaxf(M, __ldcg(src + s * (kPcHD + 2)));
    float L = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int q = 0; q < kPcCluster; ++q) {
      if (mq[i][q] == -INFINITY) continue;
      const float w = __expf(mq[i][q] - M);
      L += w * lq[i][q];
      acc[0] += w * oq[i][q].x; acc[1] += w * oq[i][q].y; acc[2] += w * oq[i][q].z; acc[3] += w * oq[i][q].w;
    }
#pragma unroll
    for (int s = 0; s < kPre; ++s) {
      if (pm[i][s] == -INFINITY) continue;
      const float w = __expf(pm[i][s] - M);
      L += w * pl[i][s];
      acc[0] += w * pa[i][s].x; acc[1] += w * pa[i][s].y; acc[2] += w * pb[i][s].x; acc[3] += w * pb[i][s].y;
    }
    for (int s = kPre; s < ns; ++s) {
      const float* sp = src + s * (kPcHD + 2);
      const float mv = __ldcg(sp);
      if (mv == -INFINITY) continue;
      const float w = __expf(mv - M);
      L += w * __ldcg(sp + 1);
      const float2 o01 = __ldcg(reinterpret_cast<const float2*>(sp + 2 + 4 * lane));
      const float2 o23 = __ldcg(reinterpret_cast<const float2*>(sp + 4 + 4 * lane));
      acc[0] += w * o01.x; acc[1] += w * o01.y; acc[2] += w * o23.x; acc[3] += w * o23.y;
    }
    const float inv = 1.f / L;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float v = acc[t] * inv;
      const size_t col = (size_t)rh[i] * kPcHD + 4 * lane + t;
      if (a.o) a.o[(size_t)rb[i] * a.o_ld + col] = v;
      if (a.o16) st_bf16_split(a.o16, a.o16lo, (size_t)rb[i] * a.o16_ld + col, v);
    }
  }

  stamp(10);
  // what tid 0 issued and did not see complete: one more bounded wait each
  // (a failed MMA wait is followed by the phase flip of its chunk, and the
  // loop stops after that chunk; ld_phase only flips on completion)
  if (tid == 0) {
    if (q_pending) mbar_wait(&bar_q, 0, nullptr);
    if (ld_pending) mbar_wait(&bar_ld, ld_phase, nullptr);
    if (s_pending) mbar_wait(&bar_s, mma_phase ^ 1u, nullptr);
    if (o_pending) mbar_wait(&bar_o, mma_phase ^ 1u, nullptr);
  }
  tc_fence_before();
  cluster_sync_all();   // the partners have read this CTA's shared memory
  stamp(11);
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "n"(kPcTmemCols)
                 : "memory");
  }
}

}  // namespace

size_t attn_prefix_qimg_bytes(int B, int Hkv) {
  return (size_t)Hkv * ((B * kPcGroup + kPcRows - 1) / kPcRows) * (2 * kPcPlane);
}

size_t attn_prefix_plane_bytes(int Hkv, int hd, int stride, int layers) {
  return (size_t)layers * Hkv * stride * 8 * hd;
}

int attn_prefix_plane_stride(int max_keys) {
  return (max_keys + kPcChunk - 1) / kPcChunk * kPcChunk;
}

cudaError_t launch_attn_prefix_planes(const PrefixPlanesArgs& p, cudaStream_t st) {
  if (p.hd != kPcHD || p.Hkv < 1 || p.layers < 1 || p.P < 1 || p.P % kPcPage || p.stride % kPcChunk ||
      p.P > p.stride || !p.kv || !p.table || !p.planes || p.page_elems < 1)
    return cudaErrorInvalidValue;
  // 16-byte loads of the pages, 16-byte stores of the images
  if ((reinterpret_cast<uintptr_t>(p.kv) & 15) || (reinterpret_cast<uintptr_t>(p.planes) & 15) ||
      (p.layer_bytes & 15))
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.P + kPcChunk - 1) / kPcChunk * 2, p.Hkv, p.layers);   // 64-key blocks, zero past P
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  if (p.kv_bf16) return s2_launch(&cfg, attn_prefix_planes_kernel<__nv_bfloat16>, p);
  return s2_launch(&cfg, attn_prefix_planes_kernel<float>, p);
}

cudaError_t launch_attn_prefix_cl(const AttnDecodeArgs& a, const void* planes, int stride, cudaStream_t st,
                                  bool pdl) {
  if (g_recorder) {
    g_recorder->ok = false;
    return cudaSuccess;
  }
  if (a.hd != kPcHD || a.H != kPcGroup * a.Hkv || a.m != 1 || !a.key_begin || !a.part || a.nsplit < 1 ||
      a.B < 1 || !planes || stride < kPcChunk || stride % kPcChunk || (!a.o && !a.o16) || !a.q_img)
    return cudaErrorInvalidValue;
  // 8-byte loads of the partial slots; 16-byte bulk copies of the images
  // and the query tiles
  if ((reinterpret_cast<uintptr_t>(a.qkv) & 15) || (a.qkv_ld & 3) || (reinterpret_cast<uintptr_t>(a.part) & 7) ||
      (reinterpret_cast<uintptr_t>(a.q_gain) & 15) || (reinterpret_cast<uintptr_t>(a.rope_cos) & 15) ||
      (reinterpret_cast<uintptr_t>(a.rope_sin) & 15) || (reinterpret_cast<uintptr_t>(planes) & 15) ||
      (reinterpret_cast<uintptr_t>(a.q_img) & 15))
    return cudaErrorInvalidValue;
  static bool attr = false;
  if (!attr) {
    const cudaError_t e =
        cudaFuncSetAttribute(attn_prefix_cl_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPcSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kPcCluster, a.Hkv, (a.B * kPcGroup + kPcRows - 1) / kPcRows);
  cfg.blockDim = dim3(kPcThreads);
  cfg.dynamicSmemBytes = kPcSmem;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kPcCluster;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 2 : 1;
  return s2_launch(&cfg, attn_prefix_cl_kernel, a, static_cast<const uint8_t*>(planes), stride, g_pc_trace,
                   g_pc_trace_ctas);
}

void attn_prefix_set_trace(unsigned long long* buf, int max_ctas) {
  g_pc_trace = max_ctas > 0 ? buf : nullptr;
  g_pc_trace_ctas = max_ctas > 0 ? max_ctas : 0;
}

}  // namespace s2
