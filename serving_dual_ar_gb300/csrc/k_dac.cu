// DAC vocoder decode kernels: residual codebook lookup, the convolutions as
// tcgen05 implicit GEMMs, halo clearing and the one-channel output stage.
//
// The codec stage of "SGLang Day-0 Support for FishAudio S2" (Architecture,
// Stage 3) at 2,048 samples per frame ("s2pro-native", What happens to a
// sentence); the decoder layers follow the published DAC decoder (Kumar et
// al. 2023): per-codebook lookup + 1x1 projection summed, k=7 conv,
// upsampling blocks (Snake, transposed conv 2s / s, residual units with
// dilations 1, 3, 9), Snake, k=7 conv to one channel, tanh.
//
// Convolution as a GEMM.  Time rows are the MMA's M = 128 side, output
// channels its N side (64..256), and K runs over (tap, 64-channel chunk):
// for tap j the A tile is the 128 input rows shifted by the tap's offset,
// loaded by TMA from the bf16 planes of the input (the offset can be any
// row: the per-sequence zero halo supplies the convolution's padding, and
// rows past the buffer read 0).  The fp32 activation is carried as two bf16
// planes hi + lo; every k-step issues two MMAs into one fp32 accumulator in
// tensor memory (weights are bf16 values exactly), so the product is as
// exact as with fp32 activations to ~2^-17.  The epilogue (four warps, one
// time row per thread, eight channels per tcgen05.ld) adds the bias and the
// residual, stores the fp32 value when it is needed later (the residual
// stream), and stores Snake(value) -- the next convolution's input -- as
// the two bf16 planes.  A transposed convolution of stride s runs polyphase
// (two 2-tap groups of output phases), its epilogue scattering phase r of
// input row q to output row q*s + r.
#include "dac.h"
#include "s2_kernels.h"
#include "s2_common.cuh"
#include "tc_common.cuh"

#include <algorithm>

namespace s2 {

constexpr int kDacBM = 128;   // time rows per tile (MMA M)
constexpr int kDacBK = 64;    // input channels per k-chunk (128-byte rows)

// sin(x): additive range reduction to [-pi, pi] with 2 pi split in two
// floats (Cody and Waite, "Software Manual for the Elementary Functions",
// 1980), then the hardware sine approximation, whose absolute error on that
// interval is below 2^-21.  Snake only needs sin^2 / alpha to well below the
// 2^-17 relative precision of the bf16 hi + lo planes it is stored in.
S2_DEV float dac_sin(float x) {
  constexpr float kInv2Pi = 0.15915494309189535f;
  constexpr float k2PiHi = 6.28318548202514648f;     // float nearest 2 pi
  constexpr float k2PiLo = -1.7484556000744883e-7f;  // 2 pi - k2PiHi
  const float k = rintf(x * kInv2Pi);
  const float r = fmaf(-k, k2PiLo, fmaf(-k, k2PiHi, x));
  return __sinf(r);
}

struct DacConvLaunch {
  DacConvParams p;
  int n_tiles;                // column tiles of NT
  int total_tiles;            // sequences x time tiles x column tiles
};

template <int NT>
constexpr int dac_stages() {
  return NT <= 64 ? 5 : NT <= 128 ? 4 : 3;
}

constexpr int kDacEpiWarps = 8;                       // two teams of four (one per TMEM lane quarter)
constexpr int kDacThreads = 32 * (2 + kDacEpiWarps);  // producer, MMA, epilogue

// Persistent, warp-specialised: warp 0 streams the tiles' operands through
// the shared-memory ring (continuously across tiles), warp 1 issues the MMAs
// into tensor-memory accumulators in rotation (4 of them up to 128 columns, 2
// above), warps 2..9 drain finished ones in two teams (epilogues of two tiles
// overlap each other and the MMAs of the next).  Tile i of
// the CTA is grid tile blockIdx.x + i * gridDim.x; column tiles of one time
// tile are adjacent, so concurrently running CTAs share A tiles in L2.
template <int NT>
__global__ void __launch_bounds__(kDacThreads, 1)
dac_conv_kernel(const __grid_constant__ CUtensorMap mapXh, const __grid_constant__ CUtensorMap mapXl,
                const __grid_constant__ CUtensorMap mapW, const __grid_constant__ DacConvLaunch L) {
  constexpr int STAGES = dac_stages<NT>();
  constexpr int A_BYTES = kDacBM * kDacBK * 2;
  constexpr int W_BYTES = NT * kDacBK * 2;
  constexpr int STAGE = 2 * A_BYTES + W_BYTES;
  constexpr int ACC_COLS = NT <= 64 ? 64 : NT <= 128 ? 128 : 256;
  constexpr int ACC = NT <= 128 ? 4 : 2;        // tensor-memory accumulators
  constexpr int TMEM_COLS = ACC * ACC_COLS;     // 256 or 512
  constexpr int NG = NT / 32;                   // 32-column groups per tile row
  static_assert(W_BYTES % 1024 == 0, "stages stay 1024-byte aligned");
  static_assert(NT % 32 == 0, "epilogue groups of 32 columns");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t full[STAGES], empty[STAGES], acc_full[ACC], acc_empty[ACC];
  __shared__ uint32_t tmem_base;
  __shared__ volatile int abort_flag;
  // per epilogue team, double-buffered by tile: bias, alpha, 1 / (alpha + 1e-9) of the tile's columns
  __shared__ float s_prm[2][2][3 * NT];
  const DacConvParams& p = L.p;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nit = p.taps * p.kchunks;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < ACC; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 4);   // the four warps of the team that drains it
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(&tmem_base)), "r"(TMEM_COLS) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  // grid tile -> (sequence b, first time row t0, phase group g, column in group nl0)
  auto decode = [&](int tile, int& b, int& t0, int& g, int& nl0) {
    const int n_idx = tile % L.n_tiles, tt = tile / L.n_tiles;
    b = tt / p.tiles_per_seq;
    t0 = (tt - b * p.tiles_per_seq) * kDacBM;
    const int n0 = n_idx * NT;
    g = n0 / p.n_group;
    nl0 = n0 - g * p.n_group;
  };

  int issued = 0;   // producer: k-iterations whose copies it issued (across tiles)
  if (warp == 0) {
    if (lane == 0) {
      for (int tile = blockIdx.x; tile < L.total_tiles && !abort_flag; tile += gridDim.x) {
        int b, t0, g, nl0;
        decode(tile, b, t0, g, nl0);
        const int row_in = b * p.S_in + kDacHalo + t0;
        for (int it = 0; it < nit; ++it) {
          const int slot = issued % STAGES;
          if (issued >= STAGES && !mbar_wait(&empty[slot], ((issued / STAGES) + 1) & 1, p.err)) {
            abort_flag = 1;
            break;
          }
          const int tap = it / p.kchunks, kc = it - tap * p.kchunks;
          uint8_t* stg = smem + slot * STAGE;
          const int y = row_in + p.tap_off[g][tap];
          mbar_arrive_expect_tx(&full[slot], STAGE);
          tma_load_2d(stg, &mapXh, kc * kDacBK, y, &full[slot]);
          tma_load_2d(stg + A_BYTES, &mapXl, kc * kDacBK, y, &full[slot]);
          tma_load_2d(stg + 2 * A_BYTES, &mapW, kc * kDacBK, (g * p.taps + tap) * p.n_group + nl0, &full[slot]);
          ++issued;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kDacBM, NT);
      int used = 0, lt = 0;   // k-iterations consumed, tiles done
      for (int tile = blockIdx.x; tile < L.total_tiles && !abort_flag; tile += gridDim.x, ++lt) {
        const int acc = lt % ACC, u = lt / ACC;
        if (u > 0 && !mbar_wait(&acc_empty[acc], (u - 1) & 1, p.err)) {
          abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + acc * ACC_COLS;
        bool ok = true;
        for (int it = 0; it < nit; ++it, ++used) {
          const int slot = used % STAGES;
          if (!mbar_wait(&full[slot], (used / STAGES) & 1, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = smem_u32(smem + slot * STAGE);
          const uint32_t w = a + 2 * A_BYTES;
#pragma unroll
          for (int kk = 0; kk < kDacBK / 16; ++kk) {
            umma_bf16(d, smem_desc_sw128(a + kk * 32), smem_desc_sw128(w + kk * 32), idesc,
                      (it > 0 || kk > 0) ? 1u : 0u);
            umma_bf16(d, smem_desc_sw128(a + A_BYTES + kk * 32), smem_desc_sw128(w + kk * 32), idesc, 1u);
          }
          umma_commit(&empty[slot]);
        }
        umma_commit(&acc_full[acc]);
        if (!ok) {
          abort_flag = 1;
          break;
        }
      }
    }
  } else {
    // epilogue: two teams of four warps; team k drains the CTA's tiles k, k + 2,
    // ... (all columns), so two tiles' epilogues are in flight.  Warp w reads
    // TMEM lanes 32 (w % 4) .. + 31 (time rows).  The tile's bias and Snake
    // parameters are staged in shared memory (double-buffered per team: one
    // barrier of the team per tile, which also ANDs the team's wait results).
    const int quarter = warp & 3, team = (warp - 2) >> 2;
    const int tt_idx = threadIdx.x - 64 - team * 128;   // 0..127 within the team
    int lt = team;
    for (int tile = blockIdx.x + team * gridDim.x; tile < L.total_tiles; tile += 2 * gridDim.x, lt += 2) {
      const int acc = lt % ACC, u = lt / ACC;
      int b, t0, g, nl0;
      decode(tile, b, t0, g, nl0);
      float* prm = s_prm[team][(lt >> 1) & 1];
      for (int c = tt_idx; c < NT; c += 128) {
        const int nl = nl0 + c, co = nl - (nl / p.cphase) * p.cphase;
        prm[c] = p.bias[co];
        prm[NT + c] = p.alpha ? p.alpha[co] : 0.f;
        prm[2 * NT + c] = p.alpha ? p.inv_alpha[co] : 0.f;
      }
      const int t = t0 + quarter * 32 + lane;
      const bool in_seq = t < p.T_in;
      // output element offset of column c of this thread's row
      auto out_off = [&](int c) {
        const int nl = nl0 + c;
        const int ph = nl / p.cphase;
        return ((size_t)b * p.S_out + kDacHalo + (size_t)t * p.up + g * p.phases + ph) * p.cphase +
               (nl - ph * p.cphase);
      };
      // the residual of the first group is independent of the MMAs: load it
      // before waiting for the accumulator
      float4 rv[8];
      if (p.resid && in_seq) {
        const float* rp = p.resid + out_off(0);
#pragma unroll
        for (int i = 0; i < 8; ++i) rv[i] = *reinterpret_cast<const float4*>(rp + 4 * i);
      }
      const bool mine = !abort_flag && mbar_wait(&acc_full[acc], u & 1, p.err);
      uint32_t all_ok;
      asm volatile(
          "{\n\t.reg .pred pa, pb;\n\tsetp.ne.u32 pa, %1, 0;\n\t"
          "barrier.cta.red.and.pred pb, %2, 128, pa;\n\tselp.u32 %0, 1, 0, pb;\n\t}"
          : "=r"(all_ok) : "r"((uint32_t)mine), "r"(1 + team) : "memory");
      const bool ok = all_ok != 0;
      if (!ok) abort_flag = 1;
      tc_fence_after();
      const uint32_t taddr = tmem + acc * ACC_COLS + ((uint32_t)(quarter * 32) << 16);
      if (ok) {
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
          const int c = gi * 32;
          float v[32];
          tmem_ld32(taddr + c, v);
          if (in_seq) {
            const size_t o = out_off(c);
            float4 rn[8];
            if (p.resid && gi + 1 < NG) {   // next group's residual while this one computes
              const float* rp = p.resid + out_off(c + 32);
#pragma unroll
              for (int i = 0; i < 8; ++i) rn[i] = *reinterpret_cast<const float4*>(rp + 4 * i);
            }
            if (p.resid) {
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                v[4 * i] = rv[i].x + (v[4 * i] + prm[c + 4 * i]);
                v[4 * i + 1] = rv[i].y + (v[4 * i + 1] + prm[c + 4 * i + 1]);
                v[4 * i + 2] = rv[i].z + (v[4 * i + 2] + prm[c + 4 * i + 2]);
                v[4 * i + 3] = rv[i].w + (v[4 * i + 3] + prm[c + 4 * i + 3]);
              }
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] += prm[c + i];
            }
            if (p.out_f32) {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                *reinterpret_cast<float4*>(p.out_f32 + o + 4 * i) =
                    make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
            }
            if (p.alpha) {
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const float s = dac_sin(prm[NT + c + i] * v[i]);
                v[i] = v[i] + s * s * prm[2 * NT + c + i];
              }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t hw[4], lw[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float x0 = v[8 * q + 2 * i], x1 = v[8 * q + 2 * i + 1];
                const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
                const __nv_bfloat16 l0 = __float2bfloat16_rn(x0 - __bfloat162float(h0));
                const __nv_bfloat16 l1 = __float2bfloat16_rn(x1 - __bfloat162float(h1));
                hw[i] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
                lw[i] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
              }
              *reinterpret_cast<uint4*>(p.out_hi + o + 8 * q) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
              *reinterpret_cast<uint4*>(p.out_lo + o + 8 * q) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
            if (p.resid && gi + 1 < NG) {
#pragma unroll
              for (int i = 0; i < 8; ++i) rv[i] = rn[i];
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
      if (!ok) break;
    }
  }
  __syncwarp();
  // every copy the producer issued must have landed before the CTA exits
  // (after a wait that gave up, the MMA thread may have stopped consuming)
  if (threadIdx.x == 0)
    for (int j = issued > STAGES ? issued - STAGES : 0; j < issued; ++j)
      mbar_wait(&full[j % STAGES], (j / STAGES) & 1, p.err);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

int dac_conv_smem_bytes(int nt) {
  const int stage = 2 * kDacBM * kDacBK * 2 + nt * kDacBK * 2;
  const int stages = nt <= 64 ? 5 : nt <= 128 ? 4 : 3;
  return stages * stage + 1024;
}

static int dac_num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 1;
    cudaGetLastError();
  }
  return n;
}

template <int NT>
static cudaError_t launch_nt(const CUtensorMap& mxh, const CUtensorMap& mxl, const CUtensorMap& mw,
                             const DacConvLaunch& L, cudaStream_t st) {
  auto k = dac_conv_kernel<NT>;
  const int smem = dac_conv_smem_bytes(NT);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::min(L.total_tiles, dac_num_sms()));
  cfg.blockDim = dim3(kDacThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  return s2_launch(&cfg, k, mxh, mxl, mw, L);
}

cudaError_t launch_dac_conv(const CUtensorMap& mapXh, const CUtensorMap& mapXl, const CUtensorMap& mapW,
                            const DacConvParams& p, int groups, int nt, int batch, cudaStream_t st) {
  if (p.taps < 1 || p.taps > kDacMaxTaps || groups < 1 || groups > 2 || p.kchunks < 1 || p.n_group % nt ||
      p.cphase % 8 || p.phases * p.cphase != p.n_group || !p.bias || !p.out_hi || !p.out_lo ||
      (p.alpha && !p.inv_alpha) || p.T_in <= 0 || batch <= 0)
    return cudaErrorInvalidValue;
  DacConvLaunch L;
  L.p = p;
  L.n_tiles = groups * p.n_group / nt;
  const long long tiles = (long long)batch * p.tiles_per_seq * L.n_tiles;
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
  L.total_tiles = (int)tiles;
  switch (nt) {
    case 64: return launch_nt<64>(mapXh, mapXl, mapW, L, st);
    case 128: return launch_nt<128>(mapXh, mapXl, mapW, L, st);
    case 192: return launch_nt<192>(mapXh, mapXl, mapW, L, st);
    case 256: return launch_nt<256>(mapXh, mapXl, mapW, L, st);
    default: return cudaErrorInvalidValue;
  }
}

// ---------------------------------------------------------------- codebook lookup

constexpr int kDacMaxCb = 16;

// Projected tables: E[k][i][c] = (sum_j proj_w[k][c][j] * codebook[k][i][j]) + proj_b[k][c],
// one codebook entry's contribution to the latent, computed once per vocoder.
__global__ void __launch_bounds__(256) dac_project_kernel(int ncb, int csize, int cbd, int latent,
                                                          const float* __restrict__ cb, const float* __restrict__ pw,
                                                          const float* __restrict__ pb, float* __restrict__ E) {
  const long long total = (long long)ncb * csize * latent;
  for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < total;
       x += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(x % latent);
    const long long ki = x / latent;   // k * csize + i
    const int k = (int)(ki / csize);
    const float* w = pw + ((size_t)k * latent + c) * cbd;
    const float* e = cb + (size_t)ki * cbd;
    float s = 0.f;
    for (int j = 0; j < cbd; ++j) s += w[j] * e[j];
    E[x] = s + pb[(size_t)k * latent + c];
  }
}

cudaError_t launch_dac_project(int ncb, int csize, int cbd, int latent, const float* codebook, const float* proj_w,
                               const float* proj_b, float* tables, cudaStream_t st) {
  if (ncb < 1 || ncb > kDacMaxCb || cbd < 1 || cbd > kDacMaxCb || latent < 1 || csize < 1)
    return cudaErrorInvalidValue;
  dac_project_kernel<<<152 * 8, 256, 0, st>>>(ncb, csize, cbd, latent, codebook, proj_w, proj_b, tables);
  ++g_launch_count;
  return cudaGetLastError();
}

// z[b, t, :] = sum_k E[k][codes[b, t, k]] in codebook order; one block per
// time step, four latent channels per thread.
__global__ void __launch_bounds__(256) dac_rvq_kernel(const int32_t* __restrict__ codes, int n, int ncb, int csize,
                                                      int latent, const float* __restrict__ E, float* zf,
                                                      __nv_bfloat16* zh, __nv_bfloat16* zl, int ld, int S, int* err) {
  __shared__ int cs[kDacMaxCb];
  const int row = blockIdx.x, b = row / n, t = row - b * n;
  if (threadIdx.x < ncb) {
    int c = codes[(size_t)row * ncb + threadIdx.x];
    if (c < 0 || c >= csize) {
      if (err) atomicExch(err, 4);
      c = 0;
    }
    cs[threadIdx.x] = c;
  }
  __syncthreads();
  const size_t o = ((size_t)b * S + kDacHalo + t) * ld;
  for (int c = threadIdx.x * 4; c < latent; c += blockDim.x * 4) {
    float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < ncb; ++k) {
      const float4 e = __ldg(reinterpret_cast<const float4*>(E + ((size_t)k * csize + cs[k]) * latent + c));
      z.x += e.x; z.y += e.y; z.z += e.z; z.w += e.w;
    }
    *reinterpret_cast<float4*>(zf + o + c) = z;
    st_bf16_split(zh, zl, o + c, z.x);
    st_bf16_split(zh, zl, o + c + 1, z.y);
    st_bf16_split(zh, zl, o + c + 2, z.z);
    st_bf16_split(zh, zl, o + c + 3, z.w);
  }
}

cudaError_t launch_dac_rvq(const int32_t* codes, int batch, int n, int ncb, int csize, int latent,
                           const float* tables, float* z_f32, __nv_bfloat16* z_hi, __nv_bfloat16* z_lo, int ld, int S,
                           int* err, cudaStream_t st) {
  if (ncb < 1 || ncb > kDacMaxCb || latent > ld || latent % 4 || batch <= 0 || n <= 0) return cudaErrorInvalidValue;
  dac_rvq_kernel<<<batch * n, 256, 0, st>>>(codes, n, ncb, csize, latent, tables, z_f32, z_hi, z_lo, ld, S, err);
  ++g_launch_count;
  return cudaGetLastError();
}

// ---------------------------------------------------------------- halos

__global__ void __launch_bounds__(128) dac_zero_halos_kernel(const __grid_constant__ DacHaloJobs jobs) {
  const DacHaloJob& j = jobs.job[blockIdx.y];
  const int b = blockIdx.x / (2 * kDacHalo), i = blockIdx.x - b * 2 * kDacHalo;
  const size_t row = i < kDacHalo ? (size_t)b * j.S + i : (size_t)b * j.S + kDacHalo + j.T + (i - kDacHalo);
  uint4* hi = reinterpret_cast<uint4*>(j.hi + row * j.ld);
  uint4* lo = reinterpret_cast<uint4*>(j.lo + row * j.ld);
  for (int c = threadIdx.x; c < j.ld / 8; c += blockDim.x) {
    hi[c] = make_uint4(0, 0, 0, 0);
    lo[c] = make_uint4(0, 0, 0, 0);
  }
}

cudaError_t launch_dac_zero_halos(const DacHaloJobs& jobs, int batch, cudaStream_t st) {
  if (jobs.n <= 0 || jobs.n > 16 || batch <= 0) return cudaErrorInvalidValue;
  for (int i = 0; i < jobs.n; ++i)
    if (jobs.job[i].ld % 8 || jobs.job[i].S != jobs.job[i].T + 2 * kDacHalo) return cudaErrorInvalidValue;
  dac_zero_halos_kernel<<<dim3(batch * 2 * kDacHalo, jobs.n), 128, 0, st>>>(jobs);
  ++g_launch_count;
  return cudaGetLastError();
}

// ---------------------------------------------------------------- output stage

constexpr int kDacOutT = 512;            // samples per block (4 per thread)
constexpr int kDacOutL = kDacOutT + 12;  // row length of the channel-major tile

// One block per 512 samples of one sequence.  The 518 input rows (hi + lo,
// 16-byte loads) go to shared memory channel-major as fp32, so a thread's
// four consecutive samples and their 6 neighbours are three 16-byte loads
// per channel (conflict-free); then
// audio[t] = tanh(bias + sum_c sum_j w[j][c] x[t + j - 3][c]).
__global__ void __launch_bounds__(128) dac_out_kernel(const __nv_bfloat16* __restrict__ xh,
                                                      const __nv_bfloat16* __restrict__ xl, int ld, int C,
                                                      const float* __restrict__ w, const float* __restrict__ bias,
                                                      int T, int S, int tiles_per_seq, float* audio) {
  extern __shared__ __align__(16) float xs[];   // [C][kDacOutL], then w [7][C]
  float* ws = xs + C * kDacOutL;
  const int b = blockIdx.x / tiles_per_seq, t0 = (blockIdx.x - b * tiles_per_seq) * kDacOutT;
  const size_t r0 = (size_t)b * S + kDacHalo + t0 - 3;
  const int c8 = C / 8;
  for (int e = threadIdx.x; e < kDacOutL * c8; e += blockDim.x) {
    const int i = e / c8, c = (e - i * c8) * 8;
    float h[8], l[8];
    if (i < kDacOutT + 6) {
      const size_t o = (r0 + i) * ld + c;
      load8(xh + o, h);
      load8(xl + o, l);
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q) h[q] = l[q] = 0.f;
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) xs[(c + q) * kDacOutL + i] = h[q] + l[q];
  }
  for (int e = threadIdx.x; e < 7 * C; e += blockDim.x) ws[e] = w[e];
  __syncthreads();
  const int k = threadIdx.x * 4;   // first of the thread's four samples
  float acc[4];
  const float b0 = bias[0];
#pragma unroll
  for (int q = 0; q < 4; ++q) acc[q] = b0;
  for (int c = 0; c < C; ++c) {
    const float4* row = reinterpret_cast<const float4*>(xs + c * kDacOutL + k);
    const float4 x0 = row[0], x1 = row[1], x2 = row[2];
    const float x[12] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w, x2.x, x2.y, x2.z, x2.w};
#pragma unroll
    for (int j = 0; j < 7; ++j) {
      const float wj = ws[j * C + c];
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[q] = fmaf(wj, x[q + j], acc[q]);
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int t = t0 + k + q;
    if (t < T) audio[(size_t)b * T + t] = tanhf(acc[q]);
  }
}

cudaError_t launch_dac_out(const __nv_bfloat16* x_hi, const __nv_bfloat16* x_lo, int ld, int C, const float* w,
                           const float* bias, int batch, int T, int S, float* audio, cudaStream_t st) {
  if (C < 8 || C % 8 || C > ld || C > 96 || batch <= 0 || T <= 0) return cudaErrorInvalidValue;
  const int tiles = (T + kDacOutT - 1) / kDacOutT;
  const size_t smem = (size_t)(C * kDacOutL + 7 * C) * sizeof(float);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(dac_out_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         96 * (kDacOutL + 7) * (int)sizeof(float));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dac_out_kernel<<<batch * tiles, 128, smem, st>>>(x_hi, x_lo, ld, C, w, bias, T, S, tiles, audio);
  ++g_launch_count;
  return cudaGetLastError();
}

}  // namespace s2
