// K2: tcgen05 tensor-core GEMM for the batched regime (prefill rows, decode
// batches of many sequences):  Y[t, n] (+)= sum_k A[n, k] * B[t, k].
//
// "Swap-AB": the weight matrix A [N, K] (row-major, K contiguous) is the
// M = 128 operand, the activations B [T, K] the N = TN operand (32..256), so
// a decode batch of 32 still fills the 128-row MMA.  Both operands are
// K-major; tiles of 128 x 64 (A) and TN x 64 (B) bf16 are brought into shared
// memory by TMA (cp.async.bulk.tensor, 128-byte swizzle) through a multi-stage
// mbarrier ring; one thread issues tcgen05.mma (kind::f16, fp32 accumulate)
// into a TN-column tensor-memory accumulator; tcgen05.commit releases each
// stage back to the producer.  The four warps then read the accumulator with
// tcgen05.ld (warp w owns TMEM lanes 32w..32w+31 = output features) and
// apply the epilogue: store, residual add, or SwiGLU of interleaved gate/up
// features into bf16.  When the tile grid is too small to cover the SMs, K
// is split across CTAs; partials go to a workspace and the last CTA of a tile
// (atomic ticket) sums them in split order -- deterministic -- before the
// epilogue.  Weight tiles are requested before griddepcontrol.wait, so with
// programmatic dependent launch the weight stream starts while the previous
// kernel drains.
#include "s2_kernels.h"
#include "s2_common.cuh"
#include "tc_common.cuh"
#include "tma_map.h"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

namespace s2 {

constexpr int kTcBM = 128;
constexpr int kTcBK = 64;
// Threads of a CTA: warp 0's thread 0 issues the copies, warp 1's the MMAs;
// all warps drain the accumulator, kTcParts per tensor-memory lane quarter
// (warp w serves quarter w % 4 and takes every kTcParts-th 8-column group /
// column, starting at part w / 4).
constexpr int kTcThreads = 512;
constexpr int kTcParts = kTcThreads / 128;

S2_DEV unsigned long long tc_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

struct TcParams {
  int N, K, T, ldy, ldy16, epi, split_k, k_tiles, tn;  // k_tiles: K / 64, shared out over the splits
  // optional phase trace (s2op_tc_set_trace): per CTA 6 globaltimer stamps
  unsigned long long* trace;
  int trace_ctas;
  unsigned long long* ftrace;   // frame timeline (4 stamps per CTA), null = off
  float* Y;
  __nv_bfloat16* Y16;
  __nv_bfloat16* Y16lo;
  float* ws;
  unsigned* tickets;
  int* err;
};

// PLANES = 2: the activation operand comes as two bf16 planes (hi, lo) and
// every k-step issues two MMAs into the same accumulator, D += A hi + A lo.
// CL: the K-splits of a tile form one thread-block cluster (split s = cluster
// rank s) and sum their partials through distributed shared memory instead of
// a global workspace.
template <int TN, int STAGES, int PLANES, bool CL = false>
__global__ void __launch_bounds__(kTcThreads, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
               const __grid_constant__ CUtensorMap mapBlo, TcParams p) {
  constexpr int A_BYTES = kTcBM * kTcBK * 2;
  constexpr int B_BYTES = TN * kTcBK * 2;
  constexpr int STAGE = A_BYTES + PLANES * B_BYTES;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t full[STAGES], empty[STAGES], done;
  __shared__ uint32_t tmem_base;
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tile = blockIdx.x, t_tile = blockIdx.y, split = blockIdx.z;
  const int cta_lin = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
  unsigned long long* tr = (p.trace && cta_lin < p.trace_ctas) ? p.trace + (size_t)cta_lin * 6 : nullptr;
  if (tr && threadIdx.x == 0) tr[0] = tc_now();   // entry
  frame_stamp(p.ftrace, cta_lin, 0);
  const int n0 = n_tile * kTcBM, t0 = t_tile * TN;
  // split s takes k-tiles [s*kt/S, (s+1)*kt/S): any split count, sizes within one
  const int kt0 = (int)((long long)split * p.k_tiles / p.split_k);
  const int nk = (int)((long long)(split + 1) * p.k_tiles / p.split_k) - kt0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&done, 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_next();

  // Producer: the weight tiles of the first stages do not depend on the
  // previous kernel; issue them before waiting on it.
  const int pre = nk < STAGES ? nk : STAGES;
  if (threadIdx.x == 0) {
    const uint64_t pol = policy_evict_first();
    for (int s = 0; s < pre; ++s) {
      mbar_arrive_expect_tx(&full[s], STAGE);
      tma_load_2d_hint(smem + s * STAGE, &mapA, (kt0 + s) * kTcBK, n0, &full[s], pol);
    }
  }
  pdl_wait();
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(&tmem_base)), "r"(TN) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  if (tr && threadIdx.x == 0) tr[1] = tc_now();   // barriers, TMEM, PDL wait done
  frame_stamp(p.ftrace, cta_lin, 1);

  int issued = pre;  // k-tiles whose copies thread 0 has issued
  if (threadIdx.x == 0) {
    const uint64_t pol = policy_evict_first();
    for (int s = 0; s < pre; ++s) {
      tma_load_2d(smem + s * STAGE + A_BYTES, &mapB, (kt0 + s) * kTcBK, t0, &full[s]);
      if (PLANES == 2)
        tma_load_2d(smem + s * STAGE + A_BYTES + B_BYTES, &mapBlo, (kt0 + s) * kTcBK, t0, &full[s]);
    }
    for (int s = STAGES; s < nk; ++s) {
      const int slot = s % STAGES;
      if (!mbar_wait(&empty[slot], ((s / STAGES) + 1) & 1, p.err)) break;
      mbar_arrive_expect_tx(&full[slot], STAGE);
      tma_load_2d_hint(smem + slot * STAGE, &mapA, (kt0 + s) * kTcBK, n0, &full[slot], pol);
      tma_load_2d(smem + slot * STAGE + A_BYTES, &mapB, (kt0 + s) * kTcBK, t0, &full[slot]);
      if (PLANES == 2)
        tma_load_2d(smem + slot * STAGE + A_BYTES + B_BYTES, &mapBlo, (kt0 + s) * kTcBK, t0, &full[slot]);
      issued = s + 1;
    }
  } else if (threadIdx.x == 32) {
    // MMA issuer
    constexpr uint32_t idesc = idesc_bf16(kTcBM, TN);
    for (int s = 0; s < nk; ++s) {
      const int slot = s % STAGES;
      if (!mbar_wait(&full[slot], (s / STAGES) & 1, p.err)) break;
      if (tr && s == 0) tr[2] = tc_now();   // first stage landed
      tc_fence_after();
      const uint32_t a_addr = smem_u32(smem + slot * STAGE);
      const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
      for (int kk = 0; kk < kTcBK / 16; ++kk) {
        umma_bf16(tmem, smem_desc_sw128(a_addr + kk * 32), smem_desc_sw128(b_addr + kk * 32), idesc,
                  (s > 0 || kk > 0) ? 1u : 0u);
        if (PLANES == 2)
          umma_bf16(tmem, smem_desc_sw128(a_addr + kk * 32), smem_desc_sw128(b_addr + B_BYTES + kk * 32),
                    idesc, 1u);
      }
      umma_commit(&empty[slot]);
    }
    umma_commit(&done);
    if (tr) tr[3] = tc_now();   // last MMA issued
  }
  __syncwarp();

  // ---------------- epilogue: all warps, warp w = TMEM lanes 32 (w % 4) ..
  // + 31 (features), column part w / 4
  const bool ok = mbar_wait(&done, 0, p.err);
  if (tr && threadIdx.x == 0) tr[4] = tc_now();   // accumulator complete
  frame_stamp(p.ftrace, cta_lin, 2);
  tc_fence_after();
  const int quarter = warp & 3, part_i = warp >> 2;
  const int feat = n0 + quarter * 32 + lane;
  const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16);
  const int t_lim = min(TN, p.T - t0);

  if (CL) {
    // Every split leaves its fp32 partial (TN columns x 128 features) in its
    // own shared memory (the pipeline stages are all consumed by now); after
    // a cluster barrier, CTA s finalises columns s, s + S, ...: each thread
    // adds its feature's S partials, read from the partners' shared memory,
    // in split order 0, 1, ... (the workspace path's order) and applies the
    // epilogue.  A second barrier keeps every partial alive until read.
    float* red = reinterpret_cast<float*>(smem);
    const int f = quarter * 32 + lane;
    const int S = p.split_k;
    // this CTA's columns split, s + S, s + 2S, ... go in turn to the parts:
    // part h takes split + (kTcParts k + h) S, four at a time
    const int CS = kTcParts * S;
    const int cfirst = split + part_i * S;
    // the residual the first four of this part's columns add to (independent
    // of the reduction: requested before the cluster barrier)
    const bool add = p.epi == TC_ADD;
    float yv[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = cfirst + j * CS;
      yv[j] = (add && c < t_lim) ? p.Y[(size_t)(t0 + c) * p.ldy + feat] : 0.f;
    }
    for (int c = part_i * 8; c < TN; c += 8 * kTcParts) {
      float v[8];
      tmem_ld8(taddr + c, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) red[(c + i) * kTcBM + f] = ok ? v[i] : 0.f;
    }
    tc_fence_before();
    cluster_sync_all();
    const bool ranks_ok = (int)cluster_rank() == split;   // split s is rank s
    if (!ranks_ok && threadIdx.x == 0 && p.err) atomicExch(p.err, 3);
    // four of this CTA's columns at a time: all their partials (up to 4 x 8
    // distributed-shared-memory loads) are requested before any is added, then
    // each column sums its S partials in split order
    for (int c0 = cfirst; c0 < t_lim; c0 += 4 * CS) {   // uniform across the warp
      float ynext[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = c0 + (4 + j) * CS;
        ynext[j] = (add && c < t_lim) ? p.Y[(size_t)(t0 + c) * p.ldy + feat] : 0.f;
      }
      float part[4][8];
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int c = c0 + j * CS;
          part[j][q] = (q < S && c < t_lim) ? ld_dsmem_f32(red + c * kTcBM + f, (uint32_t)q) : 0.f;
        }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = c0 + j * CS;
        if (c >= t_lim) break;   // uniform across the warp
        float acc = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (q < S) acc += part[j][q];
        const int t = t0 + c;
        if (p.epi == TC_SWIGLU_BF16) {
          const float u = __shfl_xor_sync(0xffffffffu, acc, 1);
          if (!(lane & 1) && ranks_ok)
            st_bf16_split(p.Y16, p.Y16lo, (size_t)t * p.ldy16 + (feat >> 1), acc / (1.f + __expf(-acc)) * u);
        } else if (ranks_ok) {
          p.Y[(size_t)t * p.ldy + feat] = add ? yv[j] + acc : acc;
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) yv[j] = ynext[j];
    }
    cluster_sync_all();
  } else if (p.split_k > 1) {
    const int tiles_mn = gridDim.x * gridDim.y;
    const int tile = t_tile * gridDim.x + n_tile;
    float* wsp = p.ws + ((size_t)split * tiles_mn + tile) * (size_t)TN * kTcBM;
    for (int c = part_i * 8; c < TN; c += 8 * kTcParts) {
      float v[8];
      tmem_ld8(taddr + c, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) wsp[(size_t)(c + i) * kTcBM + quarter * 32 + lane] = ok ? v[i] : 0.f;
    }
    __threadfence();
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(p.tickets + tile, 1u) == (unsigned)p.split_k - 1;
    __syncthreads();
    if (s_last) {
      __threadfence();
      // 8 token columns at a time with up to 8 splits' partials loaded
      // together (64 loads in flight), then summed in split order 0, 1, ...
      const float* base = p.ws + (size_t)tile * TN * kTcBM + quarter * 32 + lane;
      const size_t split_stride = (size_t)tiles_mn * TN * kTcBM;
      for (int cb = part_i * 8; cb < t_lim; cb += 8 * kTcParts) {
        float accs[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) accs[j] = 0.f;
        for (int s0 = 0; s0 < p.split_k; s0 += 8) {
          float v[8][8];
#pragma unroll
          for (int ss = 0; ss < 8; ++ss)
#pragma unroll
            for (int j = 0; j < 8; ++j)
              v[ss][j] = (s0 + ss < p.split_k && cb + j < t_lim)
                             ? __ldcg(base + (size_t)(s0 + ss) * split_stride + (size_t)(cb + j) * kTcBM)
                             : 0.f;
#pragma unroll
          for (int ss = 0; ss < 8; ++ss)
            if (s0 + ss < p.split_k)
#pragma unroll
              for (int j = 0; j < 8; ++j) accs[j] += v[ss][j];
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (cb + j >= t_lim) break;   // uniform across the warp
          const float acc = accs[j];
          const int t = t0 + cb + j;
          if (p.epi == TC_SWIGLU_BF16) {
            const float u = __shfl_xor_sync(0xffffffffu, acc, 1);
            if (!(lane & 1)) {
              const float g = acc;
              st_bf16_split(p.Y16, p.Y16lo, (size_t)t * p.ldy16 + (feat >> 1), g / (1.f + __expf(-g)) * u);
            }
          } else if (p.epi == TC_ADD) {
            p.Y[(size_t)t * p.ldy + feat] += acc;
          } else {
            p.Y[(size_t)t * p.ldy + feat] = acc;
          }
        }
      }
      if (threadIdx.x == 0) p.tickets[tile] = 0u;
    }
  } else {
    for (int c = part_i * 8; c < TN; c += 8 * kTcParts) {
      float v[8];
      tmem_ld8(taddr + c, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int cc = c + i;
        const float acc = ok ? v[i] : 0.f;
        if (p.epi == TC_SWIGLU_BF16) {
          const float u = __shfl_xor_sync(0xffffffffu, acc, 1);
          if (cc < t_lim && !(lane & 1))
            st_bf16_split(p.Y16, p.Y16lo, (size_t)(t0 + cc) * p.ldy16 + (feat >> 1),
                          acc / (1.f + __expf(-acc)) * u);
        } else if (cc < t_lim) {
          float* y = p.Y + (size_t)(t0 + cc) * p.ldy + feat;
          if (p.epi == TC_ADD) *y += acc; else *y = acc;
        }
      }
    }
    tc_fence_before();
    __syncthreads();
  }
  if (tr && threadIdx.x == 0) tr[5] = tc_now();   // epilogue (and reduction) done
  frame_stamp(p.ftrace, cta_lin, 3);
  if (warp == 0) {
    // Before the CTA may exit, every tile copy thread 0 issued must have
    // landed: after a wait that gave up, the MMA thread may have stopped
    // consuming while up to STAGES copies were still in flight.  Each slot's
    // last issue is awaited (bounded); in the normal path all of them
    // completed long ago.
    if (threadIdx.x == 0)
      for (int j = issued > STAGES ? issued - STAGES : 0; j < issued; ++j)
        mbar_wait(&full[j % STAGES], (j / STAGES) & 1, p.err);
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(TN) : "memory");
  }
}

// ---------------------------------------------------------------- host side

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;

static bool get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// 2-D bf16 map over [rows, cols] (cols contiguous, row pitch ld elements)
// with a box of box_rows x 64 and 128-byte swizzle; rows past the end read 0.
static bool make_map(CUtensorMap* m, const void* base, int rows, int cols, int ld, int box_rows) {
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)kTcBK, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                        box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool tma_map_bf16_2d(CUtensorMap* m, const void* base, long long rows, int cols, int ld, int box_rows) {
  if (!get_encode() || rows <= 0 || cols <= 0 || box_rows <= 0 || box_rows > 256) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)kTcBK, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int tc_gemm_pick_tn(int T, bool two_plane) {
  if (T <= 32) return 32;
  if (T <= 64) return 64;
  if (T <= 128 || two_plane) return 128;
  return 256;
}

void tc_gemm_plan(int N, int K, int T, int num_sms, int* tn, int* split_k, bool two_plane) {
  *tn = tc_gemm_pick_tn(T, two_plane);
  const int tiles = (N / kTcBM) * ((T + *tn - 1) / *tn);
  const int kt = K / kTcBK;
  // the most K splits that still fit one wave of CTAs (one per SM), keeping
  // at least 4 k-tiles per split; splits need not divide the k-tile count
  int best = 1;
  for (int s = 2; s <= kt / 4 && tiles * s <= num_sms; ++s) best = s;
  *split_k = best;
}

size_t tc_gemm_ws_floats(int N, int T, int split_k, bool two_plane) {
  if (split_k <= 1) return 0;
  const int tn = tc_gemm_pick_tn(T, two_plane);
  return (size_t)split_k * (N / kTcBM) * ((T + tn - 1) / tn) * tn * kTcBM;
}

size_t tc_gemm_tickets(int N, int T, bool two_plane) {
  const int tn = tc_gemm_pick_tn(T, two_plane);
  return (size_t)(N / kTcBM) * ((T + tn - 1) / tn);
}

template <int TN, int STAGES, int PLANES, bool CL>
static cudaError_t launch_tn(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mbl,
                             const TcParams& p, dim3 grid, cudaStream_t st, bool pdl) {
  constexpr int STAGE = kTcBM * kTcBK * 2 + PLANES * TN * kTcBK * 2;
  static_assert(!CL || TN * kTcBM * 4 <= STAGES * STAGE, "the partial tile must fit the stages");
  const int smem = STAGES * STAGE + 1024;
  auto k = tc_gemm_kernel<TN, STAGES, PLANES, CL>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (CL) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 1;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = grid.z;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return s2_launch(&cfg, k, ma, mb, mbl, p);
}

// Clusters of S CTAs (one K-split each) of this kernel that can be resident
// at once on the device (0 when a cluster of S does not fit), cached.
template <int TN, int STAGES, int PLANES>
static int tc_cluster_capacity(int S) {
  static int cap[9] = {-1, -1, -1, -1, -1, -1, -1, -1, -1};
  if (S < 2 || S > 8) return 0;
  if (cap[S] >= 0) return cap[S];
  constexpr int STAGE = kTcBM * kTcBK * 2 + PLANES * TN * kTcBK * 2;
  const int smem = STAGES * STAGE + 1024;
  auto k = tc_gemm_kernel<TN, STAGES, PLANES, true>;
  int n = 0;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, S);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = S;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  cap[S] = n;
  return n;
}

// Launch with the K-splits of each tile in one cluster when the plan has 2..8
// splits and the clusters fit one wave with at least 4/5 of the planned
// splits (splits reduced until they fit); otherwise through the global
// workspace with the planned splits (or unsplit).  Measured at 32 rows
// (ncu): O and down with 6 clustered splits 18.2 / 22.8 us against 34.1 /
// 38.4 us through the workspace with 7; QKV with 2 clustered splits 18.6 us
// against 17.1 us with 3 through the workspace.
template <int TN, int STAGES, int PLANES>
static cudaError_t launch_plan(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mbl,
                               TcParams p, dim3 grid, cudaStream_t st, bool pdl, bool explicit_split) {
  const int tiles = (int)(grid.x * grid.y);
  if (grid.z > 1 && grid.z <= 8 && !explicit_split) {
    int S = (int)grid.z;
    while (S >= 2 && tiles > tc_cluster_capacity<TN, STAGES, PLANES>(S)) --S;
    if (S >= 2 && 5 * S >= 4 * (int)grid.z) {
      p.split_k = S;
      return launch_tn<TN, STAGES, PLANES, true>(ma, mb, mbl, p, dim3(grid.x, grid.y, S), st, pdl);
    }
  }
  return launch_tn<TN, STAGES, PLANES, false>(ma, mb, mbl, p, grid, st, pdl);
}

static unsigned long long* g_tc_trace = nullptr;
static int g_tc_trace_ctas = 0;

void tc_set_trace(unsigned long long* buf, int max_ctas) {
  g_tc_trace = max_ctas > 0 ? buf : nullptr;
  g_tc_trace_ctas = g_tc_trace ? max_ctas : 0;
}

cudaError_t launch_tc_gemm(const TcGemmArgs& a, cudaStream_t st, bool pdl, int num_sms) {
  if (g_recorder) {  // no persistent counterpart
    g_recorder->ok = false;
    return cudaSuccess;
  }
  if (a.T <= 0) return cudaSuccess;
  if (a.N % kTcBM || a.K % kTcBK || a.ldb % 8 || !a.A || !a.Bm) return cudaErrorInvalidValue;
  if ((reinterpret_cast<uintptr_t>(a.A) | reinterpret_cast<uintptr_t>(a.Bm)) & 15) return cudaErrorInvalidValue;
  if (a.epi == TC_SWIGLU_BF16 ? !a.Y16 : !a.Y) return cudaErrorInvalidValue;
  if (!get_encode()) return cudaErrorNotSupported;
  const bool two = a.Blo != nullptr;
  if (two && (reinterpret_cast<uintptr_t>(a.Blo) & 15)) return cudaErrorInvalidValue;
  int tn, sk;
  tc_gemm_plan(a.N, a.K, a.T, num_sms, &tn, &sk, two);
  if (a.split_k > 0) sk = a.split_k;  // explicit choice
  if (sk > a.K / kTcBK) return cudaErrorInvalidValue;
  // automatic splits shrink to what the workspace holds
  while (a.split_k <= 0 && sk > 1 && a.ws_floats && tc_gemm_ws_floats(a.N, a.T, sk, two) > a.ws_floats)
    --sk;
  if (sk > 1 && a.ws_floats && tc_gemm_ws_floats(a.N, a.T, sk, two) > a.ws_floats) return cudaErrorInvalidValue;
  if (sk > 1 && a.n_tickets && tc_gemm_tickets(a.N, a.T, two) > a.n_tickets) return cudaErrorInvalidValue;
  if (sk > 1 && (!a.ws || !a.tickets)) return cudaErrorInvalidValue;
  CUtensorMap ma, mb, mbl;
  if (!make_map(&ma, a.A, a.N, a.K, a.K, kTcBM)) return cudaErrorInvalidValue;
  if (!make_map(&mb, a.Bm, a.T, a.K, a.ldb, tn)) return cudaErrorInvalidValue;
  if (!make_map(&mbl, two ? a.Blo : a.Bm, a.T, a.K, a.ldb, tn)) return cudaErrorInvalidValue;
  TcParams p;
  p.N = a.N; p.K = a.K; p.T = a.T; p.ldy = a.ldy; p.ldy16 = a.ldy16; p.epi = a.epi;
  p.split_k = sk; p.k_tiles = a.K / kTcBK; p.tn = tn;
  p.Y = a.Y; p.Y16 = a.Y16; p.Y16lo = a.Y16lo; p.ws = a.ws; p.tickets = a.tickets; p.err = a.err;
  p.trace = g_tc_trace;
  p.trace_ctas = g_tc_trace_ctas;
  p.ftrace = a.trace;
  dim3 grid(a.N / kTcBM, (a.T + tn - 1) / tn, sk);
  const bool ex = a.split_k > 0;
  if (two) {
    switch (tn) {
      case 32: return launch_plan<32, 6, 2>(ma, mb, mbl, p, grid, st, pdl, ex);
      case 64: return launch_plan<64, 6, 2>(ma, mb, mbl, p, grid, st, pdl, ex);
      default: return launch_plan<128, 4, 2>(ma, mb, mbl, p, grid, st, pdl, ex);
    }
  }
  switch (tn) {
    case 32: return launch_plan<32, 6, 1>(ma, mb, mbl, p, grid, st, pdl, ex);
    case 64: return launch_plan<64, 6, 1>(ma, mb, mbl, p, grid, st, pdl, ex);
    case 128: return launch_plan<128, 4, 1>(ma, mb, mbl, p, grid, st, pdl, ex);
    default: return launch_tn<256, 4, 1, false>(ma, mb, mbl, p, grid, st, pdl);
  }
}

}  // namespace s2
