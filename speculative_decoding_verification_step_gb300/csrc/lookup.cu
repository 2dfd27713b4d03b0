// Prompt-lookup (n-gram) drafting ("Speculative Decoding 101", Floor 6: the
// draft is a chunk of the preceding text that is likely to repeat; the
// verification follows the same rules).  One launch per speculative step
// replaces the draft model's K passes:
//   match   the earlier position j < L (L: index of the pending token) whose
//           tokens ending at j agree with the context's last tokens for the
//           most steps, up to n_max; ties go to the largest j; no agreement
//           at all: no match;
//   drafts  d_i = ext[j + i], i = 1..K, ext = the context followed by the
//           drafts (a continuation reaching the pending token copies what it
//           has drafted); no match: K copies of the pending token;
//   q rows  the drafter is deterministic: q_i is one-hot at d_i, written as
//           logit rows (0 at d_i, -inf elsewhere) for the fused acceptance
//           kernel, which then accepts d_i with probability p_i(d_i) and
//           draws a rejection from p_i without d_i.
// Grid (vocabulary chunks, sequences): every CTA of a sequence runs the
// (cheap, L2-resident) search itself; the first writes the drafts, each
// writes its chunk of the K q rows.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace sv {

namespace {

constexpr int kLkThreads = 256;
constexpr int kLkChunk = 4096;   // q-row elements per CTA
constexpr int kLkBatch = 8;      // candidate positions per thread in flight

__global__ void __launch_bounds__(kLkThreads) lookup_kernel(const __grid_constant__ LookupDesc d) {
  __shared__ long long s_best[kLkThreads / 32];
  __shared__ int s_drafts[kLookupMaxK];
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.y;
  int32_t* ctx = d.seq + (size_t)b * d.seq_ld;
  const int L = d.lens[(size_t)b * d.st_ld];   // index of the pending token
  // the context's last n_max tokens, newest first
  int suf[kLookupMaxN];
#pragma unroll
  for (int t = 0; t < kLookupMaxN; ++t) suf[t] = (t < d.n_max && L - t >= 0) ? ctx[L - t] : -1;
  // best key = m * (L + 1) + j over candidates j = L-1, L-2, ... (m >= 1)
  long long best = -1;
  for (int j0 = L - 1 - (int)threadIdx.x; j0 >= 0; j0 -= kLkBatch * kLkThreads) {
    int c0[kLkBatch];
#pragma unroll
    for (int u = 0; u < kLkBatch; ++u) {   // first tokens of kLkBatch candidates in flight
      const int j = j0 - u * kLkThreads;
      c0[u] = j >= 0 ? __ldcg(ctx + j) : -2;
    }
#pragma unroll
    for (int u = 0; u < kLkBatch; ++u) {
      const int j = j0 - u * kLkThreads;
      if (j < 0 || c0[u] != suf[0]) continue;
      int m = 1;
      while (m < d.n_max && j - m >= 0 && __ldcg(ctx + j - m) == suf[m]) ++m;
      const long long key = (long long)m * (L + 1) + j;
      best = key > best ? key : best;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const long long o = __shfl_xor_sync(0xffffffffu, best, off);
    best = o > best ? o : best;
  }
  if ((threadIdx.x & 31) == 0) s_best[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    long long bb = -1;
    for (int w = 0; w < kLkThreads / 32; ++w) bb = s_best[w] > bb ? s_best[w] : bb;
    if (bb < 0) {
      for (int i = 0; i < d.K; ++i) s_drafts[i] = ctx[L];
    } else {
      const int j = (int)(bb % (L + 1));
      for (int i = 1; i <= d.K; ++i) {
        const int x = j + i;   // index into ctx followed by the drafts
        s_drafts[i - 1] = x <= L ? ctx[x] : s_drafts[x - L - 1];
      }
    }
    if (blockIdx.x == 0)
      for (int i = 0; i < d.K; ++i) ctx[L + 1 + i] = s_drafts[i];
  }
  __syncthreads();
  const int v0 = blockIdx.x * kLkChunk, v1 = min(d.V, v0 + kLkChunk);
  for (int i = 0; i < d.K; ++i) {
    float* row = d.q_out + (size_t)b * d.q_ld + (size_t)i * d.V;
    const int di = s_drafts[i];
    for (int v = v0 + threadIdx.x; v < v1; v += kLkThreads) row[v] = v == di ? 0.f : neg_inf();
  }
}

}  // namespace

cudaError_t launch_lookup(const LookupDesc& d, cudaStream_t st) {
  if (d.rows < 1 || d.K < 1 || d.K > kLookupMaxK || d.n_max < 1 || d.n_max > kLookupMaxN || d.V < 1)
    return cudaErrorInvalidValue;
  return launch_k(lookup_kernel, dim3((d.V + kLkChunk - 1) / kLkChunk, d.rows), dim3(kLkThreads), 0, st, d);
}

}  // namespace sv
