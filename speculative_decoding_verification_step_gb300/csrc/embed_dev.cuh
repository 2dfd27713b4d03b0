// Device side of the embedding gather, shared by the per-layer kernel
// (layers.cu) and the persistent forward kernel (persist.cu).
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace sv {

// Token t of e (one CTA): thread i owns the 16-element tiles i, i + blockDim,
// ...: it copies them into the fp32 residual stream and writes their sums of
// squares (the first RMSNorm of the forward folds them into 1/rms).
template <typename T>
SV_DEV void embed_token(const EmbedDesc& e, int t) {
  const int32_t* tok = e.tok_base + (e.tok_idx ? *e.tok_idx : 0) + e.tok_off;
  const T* row = (const T*)e.embed + (size_t)tok[t] * e.d;
  for (int tile = threadIdx.x; tile < e.d / 16; tile += blockDim.x) {
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const float v = to_f32(row[tile * 16 + q]);
      e.x[(size_t)t * e.d + tile * 16 + q] = v;
      s = fmaf(v, v, s);
    }
    e.ss[(size_t)tile * e.ss_ld + t] = s;
  }
}

}  // namespace sv
