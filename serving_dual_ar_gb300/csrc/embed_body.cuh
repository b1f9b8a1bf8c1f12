// K8 input embedding: the per-row body shared by the stand-alone kernel
// (k_misc.cu) and the persistent decode kernel (k_persist.cu).
#pragma once

#include "s2_kernels.h"
#include "s2_common.cuh"

namespace s2 {

// e = E_tok[tok] + mask * sum_k E_vq[k, code_k]  ("SGLang Day-0 Support for
// FishAudio S2", Architecture: VQ embeddings are injected into the input
// embedding at masked positions; decoded frames re-enter the stream the same
// way, with the token being the frame's semantic id).  Summed in codebook
// order, fp32.
// Row r, elements i0 + tid, i0 + tid + step, ... (below d).
template <typename WT, class Wait>
S2_DEV void embed_body(const EmbedArgs& a, const int r, const int i0, const int step, const int tid,
                       Wait&& wait) {
  wait();
  int tok, masked;
  int code[16];
  const int nc = a.n_codebooks;
  if (a.tokens) {
    tok = a.tokens[r];
    masked = a.mask ? a.mask[r] : 0;
    for (int k = 0; k < nc; ++k) code[k] = masked ? a.codes[(size_t)k * a.codes_ld + r] : 0;
  } else {
    for (int k = 0; k < nc; ++k) code[k] = __ldcg(a.fb + (size_t)r * nc + k);
    tok = a.sem_begin + code[0];
    masked = 1;
  }
  const WT* te = reinterpret_cast<const WT*>(a.tok_emb) + (size_t)tok * a.d;
  const WT* ve = reinterpret_cast<const WT*>(a.vq_emb);
  for (int i = i0 + tid; i < a.d; i += step) {
    // all the rows' values are loaded before the sum (independent loads),
    // then added in codebook order
    float v[16];
#pragma unroll
    for (int k = 0; k < 16; ++k)
      v[k] = (masked && k < nc) ? to_f(ve[((size_t)k * a.codebook_size + code[k]) * a.d + i]) : 0.f;
    float e = to_f(te[i]);
#pragma unroll
    for (int k = 0; k < 16; ++k)
      if (masked && k < nc) e += v[k];
    a.out[(size_t)r * a.out_ld + i] = e;
  }
}

}  // namespace s2
