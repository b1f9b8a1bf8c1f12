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
template <typename WT, class Wait>
S2_DEV void embed_body(const EmbedArgs& a, const int r, const int tid, const int nthreads, Wait&& wait) {
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
  for (int i = tid; i < a.d; i += nthreads) {
    float e = to_f(te[i]);
    if (masked)
      for (int k = 0; k < nc; ++k)
        e += to_f(ve[((size_t)k * a.codebook_size + code[k]) * a.d + i]);
    a.out[(size_t)r * a.out_ld + i] = e;
  }
}

}  // namespace s2
