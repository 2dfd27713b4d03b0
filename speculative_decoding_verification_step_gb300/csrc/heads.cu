// Self-draft heads: the input row of the next heads pass.
//
// "Speculative Decoding 101", Floor 6 and "Speculative decoding internals",
// 三條主流變體 (MTP): extra prediction heads on the target draft the next
// positions from its own final hidden state.  The heads read the LM head's
// input at the last position the target has scored: after a step with n
// accepted drafts that is verify row n (the row whose distribution gave the
// new pending token), after a prefill or a plain-decoding pass its only or
// last row.  This kernel copies that row -- the X row exactly as the LM head
// read it (bf16 h * gain, or the fp32 residual), its per-tile sums of
// squares -- and writes u = RMSNorm_final(h) in fp32, the residual the heads
// add to silu(W_i u).  1/rms is folded exactly as the GEMMs fold it, so the
// heads' GEMM and their residual see the same scale.
#include "gemm_dev.cuh"

namespace sv {

__global__ void __launch_bounds__(256) head_input_kernel(const __grid_constant__ HeadInDesc h) {
  __shared__ float s_inv;
  __shared__ int s_row;
  pdl_trigger();
  pdl_wait();
  if (h.err && ld_volatile_i32(h.err) != 0) return;   // a forward gave up: keep the last input
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) s_row = h.count ? min(max(*h.count - 1, 0), h.max_row) : h.row;
  __syncthreads();
  const int row = s_row;
  if (warp == 0) {
    GemmDesc g{};
    g.k = h.d;
    g.ss_in = h.ss;
    g.ss_ld = h.ss_ld;
    g.eps = h.eps;
    const float v = warp_inv_rms(g, row, lane);
    if (lane == 0) s_inv = v;
  }
  __syncthreads();
  const float inv = s_inv;
  for (int t = threadIdx.x; t < h.d / 16; t += blockDim.x) h.out_ss[t] = h.ss[(size_t)t * h.ss_ld + row];
  if (h.x_bf16) {
    const bf16* src = (const bf16*)h.x + (size_t)row * h.ldx;
    for (int j = threadIdx.x; j < h.d; j += blockDim.x) {
      const bf16 v = src[j];
      ((bf16*)h.out_x)[j] = v;
      h.out_u[j] = __bfloat162float(v) * inv;
    }
  } else {
    const float* src = (const float*)h.x + (size_t)row * h.ldx;
    for (int j = threadIdx.x; j < h.d; j += blockDim.x) {
      const float v = src[j];
      ((float*)h.out_x)[j] = v;
      h.out_u[j] = v * inv * h.gain[j];
    }
  }
}

cudaError_t launch_head_input(const HeadInDesc& h, cudaStream_t st) {
  if (!h.x || !h.ss || !h.out_x || !h.out_ss || !h.out_u || h.d < 16 || h.d % 16 || h.max_row < 0 ||
      h.row < 0 || h.ss_ld < 1 || (!h.count && h.row >= h.ss_ld) || (!h.x_bf16 && !h.gain))
    return cudaErrorInvalidValue;
  return launch_k(head_input_kernel, dim3(1), dim3(256), 0, st, h);
}

}  // namespace sv
