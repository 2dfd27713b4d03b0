// Draft sampler and the fused acceptance kernel.
//
// Acceptance rule ("Speculative decoding internals", 演算法核心 Steps 3-4;
// "Speculative Decoding 101", Floors 4-5): left to right, accept d_i iff
// r_i < min(1, p_i(d_i) / q_i(d_i)); on the first rejection draw a
// replacement from normalize((p_i - q_i)+) and stop; if all K are accepted,
// draw the bonus token from p_{K+1}.  Greedy (T = 0): accept while d_i equals
// the target's argmax, emit the target's argmax at the first mismatch, or the
// bonus argmax.
//
// Both kernels split the vocabulary into 2048-wide chunks, one CTA per
// (chunk, row): each CTA reduces its chunk to (max, sum exp) or (max,
// argmax) partials.  The last CTA to finish a row (one atomic ticket per
// row, no waiting) folds the partials in chunk order, takes the decisions,
// and runs the inverse-CDF draw as a block-wide two-pass scan:
//   pass 1: each warp sums a contiguous segment (32 lanes at a time, fp32
//           shuffle tree per group of 32, fp64 running sum);
//   pass 2: the warp whose segment holds the target u * Z rescans it with
//           the same arithmetic and an in-warp prefix scan.
// Inverse CDF: the smallest index whose running sum exceeds u * Z, in token
// id order.  Random numbers come from Philox-4x32-10 keyed by (seed;
// step, position, stream, row), identical to the host restatement.
#include "common.cuh"
#include "kernels.h"

namespace sv {

constexpr int kSampThreads = 256;
constexpr int kSampWarps = kSampThreads / 32;
constexpr int kMaxK = 16;

static inline int vocab_chunks(int V) { return (V + kVocabChunk - 1) / kVocabChunk; }
size_t sample_partial_floats(int rows, int V) { return (size_t)rows * vocab_chunks(V) * 2; }
size_t accept_partial_floats(int rows, int K, int V) {
  return (size_t)rows * vocab_chunks(V) * (2 * K + 1) * 2;
}

// (m, s) online-softmax partials: s = sum exp(z - m).
SV_DEV void ms_combine(float& m, float& s, float m2, float s2) {
  const float M = fmaxf(m, m2);
  if (M == neg_inf()) { m = M; s = 0.f; return; }
  s = s * expf(m - M) + s2 * expf(m2 - M);
  m = M;
}
// (value, index) argmax partials, lowest index on ties.
SV_DEV void am_combine(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) { v = v2; i = i2; }
}

// Block reduce of (m, s) over kSampThreads threads; result valid in thread 0.
SV_DEV void block_ms(float& m, float& s, float* sm_m, float* sm_s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    ms_combine(m, s, m2, s2);
  }
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) { sm_m[w] = m; sm_s[w] = s; }
  __syncthreads();
  if (threadIdx.x == 0) {
    m = sm_m[0]; s = sm_s[0];
    for (int k = 1; k < kSampWarps; ++k) ms_combine(m, s, sm_m[k], sm_s[k]);
  }
}
SV_DEV void block_am(float& v, int& i, float* sm_v, int* sm_i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
    am_combine(v, i, v2, i2);
  }
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) { sm_v[w] = v; sm_i[w] = i; }
  __syncthreads();
  if (threadIdx.x == 0) {
    v = sm_v[0]; i = sm_i[0];
    for (int k = 1; k < kSampWarps; ++k) am_combine(v, i, sm_v[k], sm_i[k]);
  }
}

// Block-wide inverse CDF over weights wfn(v), v in [0, V).  All threads call
// it; returns the index in every thread.  *z_out receives the total.
struct CdfShared {
  double tot[kSampWarps];
  double prefix, target, z;
  int wsel, result;
};

template <typename WFn>
SV_DEV int block_inverse_cdf(const WFn& wfn, int V, float u, CdfShared& sh, double* z_out) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int seg = (V + kSampWarps - 1) / kSampWarps;
  seg = (seg + 31) & ~31;
  const int beg = min(V, w * seg), end = min(V, beg + seg);
  double R = 0.0;
  for (int b = beg; b < end; b += 32) {
    const int v = b + lane;
    const float x = v < end ? wfn(v) : 0.f;
    R += (double)warp_sum(x);
  }
  __syncthreads();
  if (lane == 0) sh.tot[w] = R;
  __syncthreads();
  if (threadIdx.x == 0) {
    double z = 0.0;
    for (int k = 0; k < kSampWarps; ++k) z += sh.tot[k];
    const double target = (double)u * z;
    double pre = 0.0;
    int sel = -1;
    double sel_pre = 0.0;
    for (int k = 0; k < kSampWarps; ++k) {
      if (sel < 0 && pre + sh.tot[k] > target) { sel = k; sel_pre = pre; }
      pre += sh.tot[k];
    }
    if (sel < 0) {  // rounding left the target at the end: last warp with mass
      pre = 0.0;
      for (int k = 0; k < kSampWarps; ++k) {
        if (sh.tot[k] > 0.0) { sel = k; sel_pre = pre; }
        pre += sh.tot[k];
      }
      if (sel < 0) sel = 0;
    }
    sh.wsel = sel; sh.prefix = sel_pre; sh.target = target; sh.z = z;
    sh.result = -1;
  }
  __syncthreads();
  if (w == sh.wsel) {
    const double target = sh.target, pre = sh.prefix;
    double Rl = 0.0;
    int last_pos = -1;
    int found = -1;
    for (int b = beg; b < end; b += 32) {
      const int v = b + lane;
      const float x = v < end ? wfn(v) : 0.f;
      const float S = warp_sum(x);
      const unsigned pos_mask = __ballot_sync(0xffffffffu, x > 0.f);
      if (pos_mask) last_pos = b + 31 - __clz(pos_mask);
      if (pre + (Rl + (double)S) > target) {
        float scan = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, scan, o);
          if (lane >= o) scan += y;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, pre + Rl + (double)scan > target && x > 0.f);
        found = hit ? b + __ffs(hit) - 1 : last_pos;
        break;
      }
      Rl += (double)S;
    }
    if (found < 0) found = last_pos;
    if (lane == 0) sh.result = found < 0 ? 0 : found;
  }
  __syncthreads();
  if (z_out) *z_out = sh.z;
  return sh.result;
}

// Ticket: returns true in all threads of the CTA that arrives last for `row`.
SV_DEV bool last_arrival(int* tickets, int row, int nchunks, int* sm_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int old = atomicAdd(&tickets[row], 1);
    *sm_flag = (old == nchunks - 1);
  }
  __syncthreads();
  const bool last = *sm_flag != 0;
  if (last) __threadfence();
  return last;
}

// ---------------------------------------------------------------- sampler
__global__ void __launch_bounds__(kSampThreads) sample_kernel(const __grid_constant__ SampleDesc s) {
  __shared__ float sm_a[kSampWarps];
  __shared__ int sm_i[kSampWarps];
  __shared__ float sm_b[kSampWarps];
  __shared__ int sm_flag;
  __shared__ CdfShared cdf;
  const int c = blockIdx.x, r = blockIdx.y;
  const int nch = gridDim.x;
  const float* row = s.logits + (size_t)r * s.ld;
  const float* mix = s.mix_src ? s.mix_src + (size_t)r * s.mix_ld : nullptr;
  float* mixed = s.mix_src ? s.mixed_out + (size_t)r * s.mixed_ld : nullptr;
  const int v0 = c * kVocabChunk, v1 = min(s.V, v0 + kVocabChunk);
  const bool greedy = s.temperature == 0.f;

  float best = neg_inf();
  int bi = 0x7fffffff;
  for (int v = v0 + threadIdx.x; v < v1; v += kSampThreads) {
    float x = row[v];
    if (mix) {
      x = (1.f - s.lambda) * x + s.lambda * mix[v];
      mixed[v] = x;
    }
    if (x > best || (x == best && v < bi)) { best = x; bi = v; }
  }
  block_am(best, bi, sm_a, sm_i);
  float* part = s.partials + ((size_t)r * nch + c) * 2;
  if (threadIdx.x == 0) { part[0] = best; part[1] = __int_as_float(bi); }
  if (!last_arrival(s.tickets, r, nch, &sm_flag)) return;

  // ---- last CTA of this row ----
  __shared__ int tok_sh;
  __shared__ float gmax_sh;
  if (threadIdx.x == 0) {
    float bv = neg_inf();
    int bidx = 0x7fffffff;
    for (int k = 0; k < nch; ++k) {
      const float* p = s.partials + ((size_t)r * nch + k) * 2;
      am_combine(bv, bidx, __ldcg(p), __float_as_int(__ldcg(p + 1)));
    }
    tok_sh = bidx;
    gmax_sh = bv;
  }
  __syncthreads();
  int tok = tok_sh;
  const uint32_t step = (uint32_t)((s.step_dev ? (uint64_t)*s.step_dev : 0) + s.step_base + r);
  if (!greedy) {
    const float invT = 1.0f / s.temperature;
    const float mz = gmax_sh * invT;
    const float* src = mix ? mixed : row;
    auto wfn = [&](int v) { return expf(__ldcg(src + v) * invT - mz); };
    const float u = philox_uniform(s.seed, step, s.position, s.stream, 0);
    tok = block_inverse_cdf(wfn, s.V, u, cdf, nullptr);
  }
  if (threadIdx.x == 0) {
    s.out_token[(s.out_idx ? *s.out_idx : 0) + s.out_off + r] = tok;
    if (s.commit_seq) {
      const int len = *s.commit_len;
      s.commit_seq[len + 1] = tok;
      *s.commit_len = len + 1;
      *s.commit_step += 1;
    }
    s.tickets[r] = 0;
  }
}

cudaError_t launch_sample(const SampleDesc& s, cudaStream_t st) {
  if (s.rows <= 0 || s.V <= 0) return cudaErrorInvalidValue;
  sample_kernel<<<dim3(vocab_chunks(s.V), s.rows), kSampThreads, 0, st>>>(s);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- acceptance
__global__ void __launch_bounds__(kSampThreads) accept_kernel(const __grid_constant__ AcceptDesc a) {
  __shared__ float sm_a[kSampWarps];
  __shared__ float sm_b[kSampWarps];
  __shared__ int sm_i[kSampWarps];
  __shared__ int sm_flag;
  __shared__ CdfShared cdf;
  __shared__ double rowM[2 * kMaxK + 1], rowZ[2 * kMaxK + 1];
  __shared__ int argm[kMaxK + 1];
  __shared__ int dec_n, dec_kind, dec_tok;   // accepted count; 0 = residual, 1 = bonus

  const int c = blockIdx.x, r = blockIdx.y;
  const int nch = gridDim.x;
  const int K = a.K, V = a.V;
  const int nrow = 2 * K + 1;                // p_1..p_{K+1}, q_1..q_K
  const bool greedy = a.temperature == 0.f;
  const float invT = greedy ? 1.f : 1.0f / a.temperature;
  const float* P = a.p + (size_t)r * a.p_ld;
  const float* Q = a.q + (size_t)r * a.q_ld;
  const int v0 = c * kVocabChunk, v1 = min(V, v0 + kVocabChunk);
  float* part = a.partials + ((size_t)r * nch + c) * nrow * 2;

  // ---- phase A: chunk partials of every row ----
  const int nstat = greedy ? K + 1 : nrow;
  for (int j = 0; j < nstat; ++j) {
    const float* src = j <= K ? P + (size_t)j * V : Q + (size_t)(j - K - 1) * V;
    if (greedy) {
      float best = neg_inf();
      int bi = 0x7fffffff;
      for (int v = v0 + threadIdx.x; v < v1; v += kSampThreads) {
        const float x = src[v];
        if (x > best || (x == best && v < bi)) { best = x; bi = v; }
      }
      block_am(best, bi, sm_a, sm_i);
      if (threadIdx.x == 0) { part[j * 2] = best; part[j * 2 + 1] = __int_as_float(bi); }
    } else {
      float m = neg_inf(), sum = 0.f;
      for (int v = v0 + threadIdx.x; v < v1; v += kSampThreads) {
        const float z = src[v] * invT;
        if (z > m) { sum = sum * expf(m - z) + 1.f; m = z; }
        else sum += expf(z - m);
      }
      block_ms(m, sum, sm_a, sm_b);
      if (threadIdx.x == 0) { part[j * 2] = m; part[j * 2 + 1] = sum; }
    }
  }
  if (!last_arrival(a.tickets, r, nch, &sm_flag)) return;

  // ---- phase B: fold partials in chunk order, ratio tests ----
  const uint32_t step = (uint32_t)((a.step_dev ? (uint64_t)*a.step_dev : 0) + a.step_base + r);
  const int32_t* D = a.drafts + (a.drafts_idx ? *a.drafts_idx : 0) + a.drafts_off + (size_t)r * K;
  if (threadIdx.x < nstat) {
    const int j = threadIdx.x;
    if (greedy) {
      float bv = neg_inf();
      int bi = 0x7fffffff;
      for (int k = 0; k < nch; ++k) {
        const float* p = a.partials + (((size_t)r * nch + k) * nrow + j) * 2;
        am_combine(bv, bi, __ldcg(p), __float_as_int(__ldcg(p + 1)));
      }
      argm[j] = bi;
    } else {
      float M = neg_inf();
      for (int k = 0; k < nch; ++k)
        M = fmaxf(M, __ldcg(a.partials + (((size_t)r * nch + k) * nrow + j) * 2));
      double Z = 0.0;
      for (int k = 0; k < nch; ++k) {
        const float* p = a.partials + (((size_t)r * nch + k) * nrow + j) * 2;
        const float m = __ldcg(p), sm = __ldcg(p + 1);
        if (m != neg_inf()) Z += (double)sm * exp((double)m - (double)M);
      }
      rowM[j] = (double)M;
      rowZ[j] = Z;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int n = K;
    int kind = 1;
    int tok = -1;
    if (greedy) {
      for (int i = 0; i < K; ++i) {
        if (D[i] != argm[i]) { n = i; kind = 2; tok = argm[i]; break; }
      }
      if (kind == 1) tok = argm[K];
    } else {
      for (int i = 0; i < K; ++i) {
        const int d = D[i];
        const double lp = (double)(P[(size_t)i * V + d] * invT) - rowM[i] - log(rowZ[i]);
        const double lq = (double)(Q[(size_t)i * V + d] * invT) - rowM[K + 1 + i] - log(rowZ[K + 1 + i]);
        const double ratio = exp(lp - lq);
        const float rr = philox_uniform(a.seed, step, (uint32_t)(i + 1), kStreamAccept, 0);
        if (!((double)rr < fmin(1.0, ratio))) { n = i; kind = 0; break; }
      }
    }
    dec_n = n;
    dec_kind = kind;
    dec_tok = tok;
  }
  __syncthreads();
  const int n = dec_n, kind = dec_kind;
  int tok = dec_tok;
  uint32_t flags = (n == K) ? 0x2u : 0u;

  // ---- phase C: residual or bonus draw ----
  if (!greedy) {
    if (kind == 0) {
      const float* pr = P + (size_t)n * V;
      const float* qr = Q + (size_t)n * V;
      const float mp = (float)rowM[n], mq = (float)rowM[K + 1 + n];
      const float izp = (float)(1.0 / rowZ[n]), izq = (float)(1.0 / rowZ[K + 1 + n]);
      auto wres = [&](int v) {
        return fmaxf(expf(pr[v] * invT - mp) * izp - expf(qr[v] * invT - mq) * izq, 0.f);
      };
      const float u = philox_uniform(a.seed, step, (uint32_t)(n + 1), kStreamResidual, 0);
      double z = 0.0;
      tok = block_inverse_cdf(wres, V, u, cdf, &z);
      if (!(z > 0.0)) {
        flags |= 0x1u;
        auto wp = [&](int v) { return expf(pr[v] * invT - mp); };
        tok = block_inverse_cdf(wp, V, u, cdf, nullptr);
      }
    } else {
      const float* pr = P + (size_t)K * V;
      const float mp = (float)rowM[K];
      auto wp = [&](int v) { return expf(pr[v] * invT - mp); };
      const float u = philox_uniform(a.seed, step, (uint32_t)(K + 1), kStreamBonus, 0);
      tok = block_inverse_cdf(wp, V, u, cdf, nullptr);
    }
  }

  if (threadIdx.x == 0) {
    int32_t* out = a.out_tokens + (size_t)r * (K + 1);
    if (a.drafts_copy)
      for (int i = 0; i < K; ++i) a.drafts_copy[(size_t)r * K + i] = D[i];
    for (int i = 0; i < n; ++i) out[i] = D[i];
    out[n] = tok;
    for (int i = n + 1; i <= K; ++i) out[i] = -1;
    a.out_count[r] = n + 1;
    if (a.out_flags) a.out_flags[r] = flags;
    if (a.commit_seq) {
      const int len = *a.commit_len;
      for (int i = 0; i <= n; ++i) a.commit_seq[len + 1 + i] = out[i];
      *a.commit_len = len + n + 1;
      *a.commit_step += 1;
    }
    a.tickets[r] = 0;
  }
}

cudaError_t launch_accept(const AcceptDesc& a, cudaStream_t st) {
  if (a.rows <= 0 || a.K < 1 || a.K > kMaxK || a.V <= 0) return cudaErrorInvalidValue;
  accept_kernel<<<dim3(vocab_chunks(a.V), a.rows), kSampThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sv
