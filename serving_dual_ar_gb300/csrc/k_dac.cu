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

namespace s2 {

constexpr int kDacBM = 128;   // time rows per tile (MMA M)
constexpr int kDacBK = 64;    // input channels per k-chunk (128-byte rows)

struct DacConvLaunch {
  DacConvParams p;
  int n_tiles;                // column tiles of NT
};

template <int NT>
constexpr int dac_stages() {
  return NT <= 64 ? 5 : NT <= 128 ? 4 : 3;
}

template <int NT>
__global__ void __launch_bounds__(128, 1)
dac_conv_kernel(const __grid_constant__ CUtensorMap mapXh, const __grid_constant__ CUtensorMap mapXl,
                const __grid_constant__ CUtensorMap mapW, const __grid_constant__ DacConvLaunch L) {
  constexpr int STAGES = dac_stages<NT>();
  constexpr int A_BYTES = kDacBM * kDacBK * 2;
  constexpr int W_BYTES = NT * kDacBK * 2;
  constexpr int STAGE = 2 * A_BYTES + W_BYTES;
  constexpr int TMEM_COLS = NT <= 64 ? 64 : NT <= 128 ? 128 : 256;
  static_assert(W_BYTES % 1024 == 0, "stages stay 1024-byte aligned");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t full[STAGES], empty[STAGES], done;
  __shared__ uint32_t tmem_base;
  const DacConvParams& p = L.p;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_idx = blockIdx.x % L.n_tiles;   // column tiles of one time tile are adjacent:
  const int tt = blockIdx.x / L.n_tiles;      // they share the A tiles in L2
  const int b = tt / p.tiles_per_seq, t0 = (tt - b * p.tiles_per_seq) * kDacBM;
  const int n0 = n_idx * NT;
  const int g = n0 / p.n_group, nl0 = n0 - g * p.n_group;
  const int row_in = b * p.S_in + kDacHalo + t0;
  const int nit = p.taps * p.kchunks;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&done, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(&tmem_base)), "r"(TMEM_COLS) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  int issued = 0;   // k-iterations whose copies thread 0 has issued
  if (threadIdx.x == 0) {
    for (int it = 0; it < nit; ++it) {
      const int slot = it % STAGES;
      if (it >= STAGES && !mbar_wait(&empty[slot], ((it / STAGES) + 1) & 1, p.err)) break;
      const int tap = it / p.kchunks, kc = it - tap * p.kchunks;
      uint8_t* stg = smem + slot * STAGE;
      const int y = row_in + p.tap_off[g][tap];
      mbar_arrive_expect_tx(&full[slot], STAGE);
      tma_load_2d(stg, &mapXh, kc * kDacBK, y, &full[slot]);
      tma_load_2d(stg + A_BYTES, &mapXl, kc * kDacBK, y, &full[slot]);
      tma_load_2d(stg + 2 * A_BYTES, &mapW, kc * kDacBK, (g * p.taps + tap) * p.n_group + nl0, &full[slot]);
      issued = it + 1;
    }
  } else if (threadIdx.x == 32) {
    constexpr uint32_t idesc = idesc_bf16(kDacBM, NT);
    for (int it = 0; it < nit; ++it) {
      const int slot = it % STAGES;
      if (!mbar_wait(&full[slot], (it / STAGES) & 1, p.err)) break;
      tc_fence_after();
      const uint32_t a = smem_u32(smem + slot * STAGE);
      const uint32_t w = a + 2 * A_BYTES;
#pragma unroll
      for (int kk = 0; kk < kDacBK / 16; ++kk) {
        umma_bf16(tmem, smem_desc_sw128(a + kk * 32), smem_desc_sw128(w + kk * 32), idesc,
                  (it > 0 || kk > 0) ? 1u : 0u);
        umma_bf16(tmem, smem_desc_sw128(a + A_BYTES + kk * 32), smem_desc_sw128(w + kk * 32), idesc, 1u);
      }
      umma_commit(&empty[slot]);
    }
    umma_commit(&done);
  }
  __syncwarp();

  // ---------------- epilogue: warp w reads TMEM lanes 32w..32w+31 = time rows
  const bool ok = mbar_wait(&done, 0, p.err);
  tc_fence_after();
  const int t = t0 + warp * 32 + lane;
  const bool valid = ok && t < p.T_in;
  const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
  for (int c = 0; c < NT; c += 8) {
    float v[8];
    tmem_ld8(taddr + c, v);
    if (valid) {
      const int nl = nl0 + c;
      const int ph = nl / p.cphase;
      const int co = nl - ph * p.cphase;
      const size_t o = ((size_t)b * p.S_out + kDacHalo + (size_t)t * p.up + g * p.phases + ph) * p.cphase + co;
      float bv[8];
      load8(p.bias + co, bv);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] += bv[i];
      if (p.resid) {
        float rv[8];
        load8(p.resid + o, rv);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = rv[i] + v[i];
      }
      if (p.out_f32) {
        *reinterpret_cast<float4*>(p.out_f32 + o) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4*>(p.out_f32 + o + 4) = make_float4(v[4], v[5], v[6], v[7]);
      }
      if (p.alpha) {
        float av[8], iv[8];
        load8(p.alpha + co, av);
        load8(p.inv_alpha + co, iv);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float s = sinf(av[i] * v[i]);
          v[i] = v[i] + s * s * iv[i];
        }
      }
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat16 h0 = __float2bfloat16_rn(v[2 * i]), h1 = __float2bfloat16_rn(v[2 * i + 1]);
        const __nv_bfloat16 l0 = __float2bfloat16_rn(v[2 * i] - __bfloat162float(h0));
        const __nv_bfloat16 l1 = __float2bfloat16_rn(v[2 * i + 1] - __bfloat162float(h1));
        hw[i] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
        lw[i] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
      }
      *reinterpret_cast<uint4*>(p.out_hi + o) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4*>(p.out_lo + o) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    // every copy thread 0 issued must have landed before the CTA exits (after
    // a wait that gave up, the MMA thread may have stopped consuming)
    if (threadIdx.x == 0)
      for (int j = issued > STAGES ? issued - STAGES : 0; j < issued; ++j)
        mbar_wait(&full[j % STAGES], (j / STAGES) & 1, p.err);
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

int dac_conv_smem_bytes(int nt) {
  const int stage = 2 * kDacBM * kDacBK * 2 + nt * kDacBK * 2;
  const int stages = nt <= 64 ? 5 : nt <= 128 ? 4 : 3;
  return stages * stage + 1024;
}

template <int NT>
static cudaError_t launch_nt(const CUtensorMap& mxh, const CUtensorMap& mxl, const CUtensorMap& mw,
                             const DacConvLaunch& L, int tiles, cudaStream_t st) {
  auto k = dac_conv_kernel<NT>;
  const int smem = dac_conv_smem_bytes(NT);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)tiles);
  cfg.blockDim = dim3(128);
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
  switch (nt) {
    case 64: return launch_nt<64>(mapXh, mapXl, mapW, L, (int)tiles, st);
    case 128: return launch_nt<128>(mapXh, mapXl, mapW, L, (int)tiles, st);
    case 192: return launch_nt<192>(mapXh, mapXl, mapW, L, (int)tiles, st);
    case 256: return launch_nt<256>(mapXh, mapXl, mapW, L, (int)tiles, st);
    default: return cudaErrorInvalidValue;
  }
}

// ---------------------------------------------------------------- codebook lookup

constexpr int kDacMaxCb = 16;

__global__ void __launch_bounds__(256) dac_rvq_kernel(const int32_t* __restrict__ codes, int n, int ncb, int csize,
                                                      int cbd, int latent, const float* __restrict__ cb,
                                                      const float* __restrict__ pw, const float* __restrict__ pb,
                                                      float* zf, __nv_bfloat16* zh, __nv_bfloat16* zl, int ld,
                                                      int S, int* err) {
  __shared__ float e[kDacMaxCb][kDacMaxCb];
  const int row = blockIdx.x, b = row / n, t = row - b * n;
  if (threadIdx.x < ncb) {
    int c = codes[(size_t)row * ncb + threadIdx.x];
    if (c < 0 || c >= csize) {
      if (err) atomicExch(err, 4);
      c = 0;
    }
    for (int j = 0; j < cbd; ++j) e[threadIdx.x][j] = cb[((size_t)threadIdx.x * csize + c) * cbd + j];
  }
  __syncthreads();
  const size_t o = ((size_t)b * S + kDacHalo + t) * ld;
  for (int c = threadIdx.x; c < latent; c += blockDim.x) {
    float z = 0.f;
    for (int k = 0; k < ncb; ++k) {
      const float* w = pw + ((size_t)k * latent + c) * cbd;
      float s = 0.f;
      for (int j = 0; j < cbd; ++j) s += w[j] * e[k][j];
      z += s + pb[(size_t)k * latent + c];
    }
    zf[o + c] = z;
    st_bf16_split(zh, zl, o + c, z);
  }
}

cudaError_t launch_dac_rvq(const int32_t* codes, int batch, int n, int ncb, int csize, int cbd, int latent,
                           const float* codebook, const float* proj_w, const float* proj_b, float* z_f32,
                           __nv_bfloat16* z_hi, __nv_bfloat16* z_lo, int ld, int S, int* err, cudaStream_t st) {
  if (ncb < 1 || ncb > kDacMaxCb || cbd < 1 || cbd > kDacMaxCb || latent > ld || batch <= 0 || n <= 0)
    return cudaErrorInvalidValue;
  dac_rvq_kernel<<<batch * n, 256, 0, st>>>(codes, n, ncb, csize, cbd, latent, codebook, proj_w, proj_b, z_f32,
                                            z_hi, z_lo, ld, S, err);
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

__global__ void __launch_bounds__(128) dac_out_kernel(const __nv_bfloat16* __restrict__ xh,
                                                      const __nv_bfloat16* __restrict__ xl, int ld, int C,
                                                      const float* __restrict__ w, const float* __restrict__ bias,
                                                      int T, int S, int tiles_per_seq, float* audio) {
  extern __shared__ float xs[];   // [(128 + 6) * C] then w [7 * C]
  float* ws = xs + (kDacBM + 6) * C;
  const int b = blockIdx.x / tiles_per_seq, t0 = (blockIdx.x - b * tiles_per_seq) * kDacBM;
  const size_t r0 = (size_t)b * S + kDacHalo + t0 - 3;
  for (int e = threadIdx.x; e < (kDacBM + 6) * C; e += blockDim.x) {
    const int i = e / C, c = e - i * C;
    const size_t o = (r0 + i) * ld + c;
    xs[e] = __bfloat162float(xh[o]) + __bfloat162float(xl[o]);
  }
  for (int e = threadIdx.x; e < 7 * C; e += blockDim.x) ws[e] = w[e];
  __syncthreads();
  const int t = t0 + threadIdx.x;
  if (t < T) {
    float acc = bias[0];
    for (int j = 0; j < 7; ++j) {
      const float* xr = xs + (threadIdx.x + j) * C;
      const float* wr = ws + j * C;
      float s = 0.f;
      for (int c = 0; c < C; ++c) s += wr[c] * xr[c];
      acc += s;
    }
    audio[(size_t)b * T + t] = tanhf(acc);
  }
}

cudaError_t launch_dac_out(const __nv_bfloat16* x_hi, const __nv_bfloat16* x_lo, int ld, int C, const float* w,
                           const float* bias, int batch, int T, int S, float* audio, cudaStream_t st) {
  if (C < 1 || C > ld || C > 256 || batch <= 0 || T <= 0) return cudaErrorInvalidValue;
  const int tiles = (T + kDacBM - 1) / kDacBM;
  const size_t smem = (size_t)((kDacBM + 6) * C + 7 * C) * sizeof(float);
  if (smem > 48 * 1024) {
    static bool attr_set = false;
    if (!attr_set) {
      cudaError_t e = cudaFuncSetAttribute(dac_out_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
      if (e != cudaSuccess) return e;
      attr_set = true;
    }
  }
  dac_out_kernel<<<batch * tiles, 128, smem, st>>>(x_hi, x_lo, ld, C, w, bias, T, S, tiles, audio);
  ++g_launch_count;
  return cudaGetLastError();
}

}  // namespace s2
