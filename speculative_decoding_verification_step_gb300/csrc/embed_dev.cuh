// Device side of the embedding gather, shared by the per-layer kernel
// (layers.cu) and the persistent forward kernel (persist.cu).
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace sv {

// Token t of e (one CTA): thread i owns the 16-element tiles i, i + blockDim,
// ...: it copies them into the fp32 residual stream and writes their sums of
// squares (the first RMSNorm of the forward folds them into 1/rms).
// kSeqs = false: single-sequence passes only (the persistent kernel).
template <typename T, bool kSeqs = true>
SV_DEV void embed_token(const EmbedDesc& e, int t) {
  const int b = kSeqs ? seq_of_tok(e.spt, t) : 0, j = kSeqs ? idx_in_seq(e.spt, t) : t;
  const int32_t* tok = e.tok_base + (size_t)b * e.tok_ld + (e.tok_idx ? e.tok_idx[(size_t)b * e.idx_ld] : 0) + e.tok_off;
  const T* row = (const T*)e.embed + (size_t)tok[j] * e.d;
  for (int tile = threadIdx.x; tile < e.d / 16; tile += blockDim.x) {
    float v[16], gn[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) v[q] = to_f32(row[tile * 16 + q]);
    if (e.xg) {
#pragma unroll
      for (int q = 0; q < 16; q += 4) {
        const float4 g4 = __ldg(reinterpret_cast<const float4*>(e.gain + tile * 16 + q));
        gn[q] = g4.x; gn[q + 1] = g4.y; gn[q + 2] = g4.z; gn[q + 3] = g4.w;
      }
    }
    float s = 0.f;
    float* xo = e.x + (size_t)t * e.d + tile * 16;
#pragma unroll
    for (int q = 0; q < 16; q += 4) {
      *reinterpret_cast<float4*>(xo + q) = make_float4(v[q], v[q + 1], v[q + 2], v[q + 3]);
      s = fmaf(v[q], v[q], s);
      s = fmaf(v[q + 1], v[q + 1], s);
      s = fmaf(v[q + 2], v[q + 2], s);
      s = fmaf(v[q + 3], v[q + 3], s);
    }
    if (e.xg) {
      uint32_t w[8];
#pragma unroll
      for (int q = 0; q < 16; q += 2) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(v[q] * gn[q], v[q + 1] * gn[q + 1]);
        w[q / 2] = *reinterpret_cast<const uint32_t*>(&b);
      }
      uint4* xg = reinterpret_cast<uint4*>((bf16*)e.xg + (size_t)t * e.d + tile * 16);
      xg[0] = make_uint4(w[0], w[1], w[2], w[3]);
      xg[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
    e.ss[(size_t)tile * e.ss_ld + t] = s;
  }
}

}  // namespace sv
