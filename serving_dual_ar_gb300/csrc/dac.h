// Internal declarations of the DAC vocoder kernels (k_dac.cu) and their host
// launchers, used by the vocoder runtime (s2_vocoder.cu).
//
// Activation layout: every tensor of one rate ("level") is [rows, ld] row-
// major with channels contiguous, ld a multiple of 64 (padding channels stay
// 0); sequence b occupies rows [b*S, (b+1)*S), S = T + 2*H, its time step t
// at row b*S + H + t.  The H rows before and after each sequence are kept at
// 0 in the bf16 planes the convolutions read, which makes them the zero
// padding of every convolution (H covers the widest reach, 3 * 9 = 27).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace s2 {

constexpr int kDacHalo = 32;        // H
constexpr int kDacMaxTaps = 7;

// One convolution as an implicit GEMM over time rows:
//   out[row(m), col(n)] = epilogue( sum_tap sum_c X[row_in(m) + tap_off[g][tap], c] * W[g][tap][n][c] )
// with X given as bf16 planes hi + lo (the fp32 activation split in two).
// A transposed convolution of stride s is run polyphase: output phase r of
// input row q is y[q*s + r]; the phases split into two groups (r < s/2 reads
// x[q] and x[q-1], r >= s/2 reads x[q+1] and x[q]), each a 2-tap GEMM whose
// columns are (phase within the group, output channel).
struct DacConvParams {
  int taps;                       // taps per group
  int tap_off[2][kDacMaxTaps];    // input-row offset of each tap, per group
  int kchunks;                    // input channels / 64 (padded)
  int n_group;                    // GEMM columns per group (a multiple of the N tile)
  int phases;                     // output phases per group (1: plain conv)
  int cphase;                     // columns per phase = padded output channels
  int up;                         // output rows per input row (stride s, or 1)
  int T_in, S_in, S_out, tiles_per_seq;
  const float* bias;              // [cphase]
  const float* alpha;             // [cphase] Snake alpha for the planes out, or null
  const float* inv_alpha;         // [cphase] 1 / (alpha + 1e-9)
  const float* resid;             // fp32 [rows_out, cphase] added before the stores, or null
  float* out_f32;                 // fp32 [rows_out, cphase] (pre-Snake value), or null
  __nv_bfloat16* out_hi;          // planes of Snake(value) (or of the value without alpha)
  __nv_bfloat16* out_lo;
  int* err;
};

// Launch the convolution: grid over (sequences x time tiles) x column tiles
// of `nt` columns (64, 128, 192 or 256; must divide n_group).  mapX{h,l}
// cover the input planes (box 128 rows), mapW the packed weights
// [groups * taps * n_group, kchunks * 64] (box nt rows).
cudaError_t launch_dac_conv(const CUtensorMap& mapXh, const CUtensorMap& mapXl, const CUtensorMap& mapW,
                            const DacConvParams& p, int groups, int nt, int batch, cudaStream_t st);
int dac_conv_smem_bytes(int nt);

// Projected codebook tables, once per vocoder: tables[k][i][:] =
// proj_w[k] @ codebook[k][i] + proj_b[k]  ([ncb, csize, latent] fp32).
cudaError_t launch_dac_project(int ncb, int csize, int cbd, int latent, const float* codebook, const float* proj_w,
                               const float* proj_b, float* tables, cudaStream_t st);
// Residual codebook lookup: z[b, t, :] = sum_k tables[k][codes[b, t, k]] (in
// codebook order), written as fp32 (ld) and as bf16 planes hi + lo (same
// ld).  Codes out of range set *err = 4 and read entry 0.
cudaError_t launch_dac_rvq(const int32_t* codes, int batch, int n, int ncb, int csize, int latent,
                           const float* tables, float* z_f32, __nv_bfloat16* z_hi, __nv_bfloat16* z_lo, int ld, int S,
                           int* err, cudaStream_t st);

// Zero the halo rows (every row outside [b*S + H, b*S + H + T)) of up to 16
// pairs of bf16 planes for `batch` sequences.
struct DacHaloJob {
  __nv_bfloat16* hi;
  __nv_bfloat16* lo;
  int ld, S, T;
};
struct DacHaloJobs {
  DacHaloJob job[16];
  int n;
};
cudaError_t launch_dac_zero_halos(const DacHaloJobs& jobs, int batch, cudaStream_t st);

// Output stage: audio[b, t] = tanh(bias + sum_{j<7, c<C} w[j][c] * X[b*S + H + t + j - 3][c]),
// X = hi + lo (the Snake-ed last level).
cudaError_t launch_dac_out(const __nv_bfloat16* x_hi, const __nv_bfloat16* x_lo, int ld, int C, const float* w,
                           const float* bias, int batch, int T, int S, float* audio, cudaStream_t st);

}  // namespace s2
