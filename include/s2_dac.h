/* DAC vocoder decode on sm_103a: residual codebook indices -> waveform.
 *
 * The codec stage of the three-stage pipeline ("SGLang Day-0 Support for
 * FishAudio S2", Architecture, Stage 3: the accumulated codebook indices are
 * decoded into a waveform by a DAC codec), at 2,048 samples per frame and
 * 44.1 kHz ("s2pro-native", What happens to a sentence).  The decoder is a
 * DAC-style stack: per codebook a table lookup and a 1x1 projection, summed;
 * a k=7 convolution; upsampling blocks (Snake, transposed convolution of
 * kernel 2s and stride s, three residual units with dilations 1, 3, 9);
 * Snake, a k=7 convolution to one channel, tanh.  Shapes come from the
 * weight file (format: the vocoder file of the seeded input generator).
 *
 * Every convolution runs as a tcgen05 implicit GEMM (bf16 weights, fp32
 * activations carried as two bf16 planes hi + lo, fp32 accumulation); the
 * codebook lookup and the one-channel output convolution run on CUDA cores.
 *
 * Status codes are those of s2.h (0 = OK, negative = error); no call throws
 * or traps.
 */
#ifndef S2_DAC_H
#define S2_DAC_H

#include <stddef.h>
#include <stdint.h>

#include "s2.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct s2_vocoder s2_vocoder;

/* Load a vocoder weight file onto the current CUDA device and size every
 * activation buffer for up to `max_seqs` sequences of `max_frames` frames.
 * `cuda_stream` (cudaStream_t, may be NULL: the legacy default stream) is
 * where all work is enqueued.  The vocoder owns its weights and buffers.
 * Returns S2_EBADFILE for a malformed file, S2_EINVAL for sizes <= 0 or a
 * decoder the kernels do not support (odd rates, more than 8 blocks, more
 * than 96 channels at the last level),
 * S2_ENOMEM when the device is out of memory, S2_ECUDA for any other CUDA
 * failure (no device); on failure nothing stays allocated. */
int s2_vocoder_create(const char* path, int32_t max_seqs, int32_t max_frames, void* cuda_stream,
                      s2_vocoder** out);
void s2_vocoder_destroy(s2_vocoder* v);

/* Samples per frame (the product of the upsampling rates), or 0 for NULL. */
int32_t s2_vocoder_hop(const s2_vocoder* v);

/* Decode `batch` sequences of `n` frames each.
 *   codes  int32 [batch, n, n_codebooks], row-major, each in
 *          [0, codebook_size); host or device memory (detected).
 *   audio  float [batch, n * hop], row-major; host or device memory.
 * Synchronous: returns after the waveform is in `audio`.  S2_EINVAL for
 * batch or n out of [1, max], NULL pointers or a code out of range (checked
 * on the host for host codes, by the lookup kernel for device codes, in
 * which case the waveform is unspecified); S2_ECUDA when a CUDA call fails;
 * S2_ETIMEOUT when a bounded device wait gave up. */
int s2_vocoder_decode(s2_vocoder* v, const int32_t* codes, int32_t batch, int32_t n, float* audio);

/* Copy an intermediate activation of the last decode to host memory as
 * float [batch, T_stage, channels] (padding channels dropped):
 *   stage -1: the summed codebook latent (frame rate, latent channels);
 *   stage  0: the input convolution's output (frame rate);
 *   stage  i: the output of upsampling block i-1 (after its residual units).
 * `bytes` must be at least the stage's size.  S2_EINVAL otherwise or before
 * any decode. */
int s2_vocoder_read_stage(s2_vocoder* v, int32_t stage, float* dst, size_t bytes);

/* Kernels launched by the last s2_vocoder_decode (for launch accounting). */
int64_t s2_vocoder_last_launches(const s2_vocoder* v);

/* Per-launch timing.  With profiling on, every decode records a CUDA event
 * on the vocoder's stream before each kernel launch and after the last one
 * (off by default: events cost a little).  s2_vocoder_profile writes the
 * last decode's per-launch durations in milliseconds, in launch order
 * (halo clear, codebook lookup, the convolutions in decode order, output
 * stage), into ms[0..max) and returns how many it wrote (0 when profiling is
 * off or nothing was decoded, S2_ECUDA when an event query fails). */
int s2_vocoder_set_profile(s2_vocoder* v, int32_t on);
int32_t s2_vocoder_profile(s2_vocoder* v, float* ms, int32_t max);

#ifdef __cplusplus
}
#endif

#endif /* S2_DAC_H */
