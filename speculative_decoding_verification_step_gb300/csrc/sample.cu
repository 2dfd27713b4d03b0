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
// Work split: the vocabulary is cut into 2048-token chunks and every (chunk,
// logit row) pair is one CTA, which reduces its chunk to (max z, sum
// exp(z - max)) -- or (max, argmax) when greedy -- with z = logit / T.  The
// last CTA to finish a verify row (one atomic ticket per row; nobody waits)
// folds the partials in chunk order in fp64 and takes every decision:
//   * softmax draws (draft token, bonus): chunk masses come straight from the
//     partials, s_c * exp(m_c - M); the chunk holding the target u * Z is
//     found by a running fp64 sum, and only that chunk is rescanned (block
//     prefix scan, token-id order);
//   * the residual draw: one block-wide pass computes the (p - q)+ mass of
//     every chunk, then the same chunk search and rescan.
// Inverse CDF: the smallest token whose running sum exceeds u * Z; if
// rounding leaves no such token in the chosen chunk, the last token of the
// chunk with positive weight.  Random numbers: Philox-4x32-10 keyed by
// (seed; step, position, stream, row), identical to the host restatement.
#include "common.cuh"
#include "kernels.h"

namespace sv {

constexpr int kSampThreads = 256;
constexpr int kSampWarps = kSampThreads / 32;
constexpr int kMaxK = 16;
constexpr int kMaxChunks = 128;          // vocabularies up to 262144 tokens
constexpr int kPerThread = kVocabChunk / kSampThreads;   // 8 contiguous tokens per thread in a rescan

__host__ __device__ inline int vocab_chunks(int V) { return (V + kVocabChunk - 1) / kVocabChunk; }
// Acceptance phase A: CTAs per logit row (one chunk per warp).
__host__ __device__ inline int accept_blocks_per_stat(int V) { return (vocab_chunks(V) + kSampWarps - 1) / kSampWarps; }
size_t sample_partial_floats(int rows, int V) { return (size_t)rows * vocab_chunks(V) * 3; }
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

// Block reductions; the result is valid in thread 0.
SV_DEV void block_ms(float& m, float& s, float* sm_m, float* sm_s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    ms_combine(m, s, m2, s2);
  }
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
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
  if (lane == 0) { sm_v[w] = v; sm_i[w] = i; }
  __syncthreads();
  if (threadIdx.x == 0) {
    v = sm_v[0]; i = sm_i[0];
    for (int k = 1; k < kSampWarps; ++k) am_combine(v, i, sm_v[k], sm_i[k]);
  }
}

// Statistics of one chunk [v0, v1) of one logit row (8 independent loads per
// thread are issued before any arithmetic).
SV_DEV void chunk_softmax_stats(const float* src, int v0, int v1, float invT, float* sm_a,
                                float* sm_b, float* m_out, float* s_out) {
  float x[kPerThread];
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    const int v = v0 + threadIdx.x + j * kSampThreads;
    x[j] = v < v1 ? src[v] * invT : neg_inf();
  }
  float m = neg_inf();
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) m = fmaxf(m, x[j]);
  float s = 0.f;
  if (m != neg_inf()) {
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) s += (x[j] == neg_inf()) ? 0.f : expf(x[j] - m);
  }
  block_ms(m, s, sm_a, sm_b);
  if (threadIdx.x == 0) { *m_out = m; *s_out = s; }
}

SV_DEV void chunk_argmax(const float* src, int v0, int v1, float* sm_a, int* sm_i, float* v_out,
                         int* i_out) {
  float best = neg_inf();
  int bi = 0x7fffffff;
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    const int v = v0 + threadIdx.x + j * kSampThreads;
    if (v < v1) {
      const float x = src[v];
      if (x > best || (x == best && v < bi)) { best = x; bi = v; }
    }
  }
  block_am(best, bi, sm_a, sm_i);
  if (threadIdx.x == 0) { *v_out = best; *i_out = bi; }
}

// One warp's statistics of one chunk [v0, v1) of a logit row: lane l reads
// tokens v0 + 4 (l + 32 i) .. +3 with 16-byte loads (element-wise when the
// chunk is short or not 16-byte aligned), then shuffle trees.  Softmax:
// m = max z, s = sum exp(z - m) with z = logit / T (the values are read
// twice, the second time from L1).  Argmax: lowest index on ties.
SV_DEV void warp_chunk_softmax(const float* src, int v0, int v1, float invT, float* m_out, float* s_out) {
  const int lane = threadIdx.x & 31;
  const bool vec = v1 - v0 == kVocabChunk && (reinterpret_cast<uintptr_t>(src + v0) & 15u) == 0;
  float m = neg_inf();
  if (vec) {
    const float4* p4 = reinterpret_cast<const float4*>(src + v0) + lane;
#pragma unroll 4
    for (int i = 0; i < kVocabChunk / 128; ++i) {
      const float4 x = p4[32 * i];
      m = fmaxf(m, fmaxf(fmaxf(x.x * invT, x.y * invT), fmaxf(x.z * invT, x.w * invT)));
    }
  } else {
    for (int v = v0 + lane; v < v1; v += 32) m = fmaxf(m, src[v] * invT);
  }
  m = warp_max(m);
  float sum = 0.f;
  if (m != neg_inf()) {
    if (vec) {
      const float4* p4 = reinterpret_cast<const float4*>(src + v0) + lane;
#pragma unroll 4
      for (int i = 0; i < kVocabChunk / 128; ++i) {
        const float4 x = p4[32 * i];
        sum += (expf(x.x * invT - m) + expf(x.y * invT - m)) + (expf(x.z * invT - m) + expf(x.w * invT - m));
      }
    } else {
      for (int v = v0 + lane; v < v1; v += 32) {
        const float z = src[v] * invT;
        sum += z == neg_inf() ? 0.f : expf(z - m);
      }
    }
  }
  *m_out = m;
  *s_out = warp_sum(sum);
}

SV_DEV void warp_chunk_argmax(const float* src, int v0, int v1, float* v_out, int* i_out) {
  const int lane = threadIdx.x & 31;
  float best = neg_inf();
  int bi = 0x7fffffff;
  for (int v = v0 + lane; v < v1; v += 32) {
    const float x = src[v];
    if (x > best || (x == best && v < bi)) { best = x; bi = v; }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, best, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
    am_combine(best, bi, v2, i2);
  }
  *v_out = best;
  *i_out = bi;
}

// Ticket: true in every thread of the CTA that arrives last for `row`.
SV_DEV bool last_arrival(int* tickets, int row, int arrivals, int* sm_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int old = atomicAdd(&tickets[row], 1);
    *sm_flag = (old == arrivals - 1);
  }
  __syncthreads();
  const bool last = *sm_flag != 0;
  if (last) __threadfence();
  return last;
}

struct DrawShared {
  double mass[kMaxChunks];
  double warp_sum[kSampWarps];
  double prefix, target;
  int chunk, result;
};

// Given per-chunk masses in sh.mass[0..nch), find the chunk holding u * Z
// (thread 0, fp64, chunk order).  Returns Z in every thread.
SV_DEV double pick_chunk(DrawShared& sh, int nch, float u) {
  __syncthreads();
  if (threadIdx.x == 0) {
    double z = 0.0;
    for (int c = 0; c < nch; ++c) z += sh.mass[c];
    const double target = (double)u * z;
    double pre = 0.0, sel_pre = 0.0;
    int sel = -1;
    for (int c = 0; c < nch; ++c) {
      if (sel < 0 && pre + sh.mass[c] > target) { sel = c; sel_pre = pre; }
      pre += sh.mass[c];
    }
    if (sel < 0) {   // rounding left the target at the end: last chunk with mass
      pre = 0.0;
      for (int c = 0; c < nch; ++c) {
        if (sh.mass[c] > 0.0) { sel = c; sel_pre = pre; }
        pre += sh.mass[c];
      }
      if (sel < 0) sel = 0;
    }
    sh.chunk = sel;
    sh.prefix = sel_pre;
    sh.target = target;
    sh.warp_sum[0] = z;
  }
  __syncthreads();
  return sh.warp_sum[0];
}

// Rescan chunk sh.chunk: thread t owns tokens [v0 + 8t, v0 + 8t + 8); block
// exclusive scan of the per-thread sums (fp64), then the owning thread walks
// its tokens.  Returns the token in every thread.
template <typename WFn>
SV_DEV int rescan_chunk(DrawShared& sh, const WFn& wfn, int V) {
  const int v0 = sh.chunk * kVocabChunk;
  const int t0 = v0 + threadIdx.x * kPerThread;
  float w[kPerThread];
  float tsum = 0.f;
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    w[j] = (t0 + j < V) ? wfn(t0 + j) : 0.f;
    tsum += w[j];
  }
  // inclusive scan over threads: warp shuffle scan, then warp offsets
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  double inc = (double)tsum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  __syncthreads();
  if (lane == 31) sh.warp_sum[wid] = inc;
  __syncthreads();
  double off = sh.prefix;
  for (int k = 0; k < wid; ++k) off += sh.warp_sum[k];
  const double excl = off + inc - (double)tsum;
  const double target = sh.target;
  // the first (lowest) thread whose range crosses the target walks its tokens
  const bool crosses = excl + (double)tsum > target && tsum > 0.f;
  __shared__ int first_thread;
  if (threadIdx.x == 0) first_thread = 0x7fffffff;
  __syncthreads();
  if (crosses) atomicMin(&first_thread, (int)threadIdx.x);
  __syncthreads();
  if ((int)threadIdx.x == first_thread) {
    double run = excl;
    int pick = -1, lastpos = -1;
    for (int j = 0; j < kPerThread; ++j) {
      if (w[j] > 0.f) lastpos = t0 + j;
      run += (double)w[j];
      if (pick < 0 && w[j] > 0.f && run > target) pick = t0 + j;
    }
    sh.result = pick >= 0 ? pick : lastpos;
  }
  __syncthreads();
  if (first_thread == 0x7fffffff) {
    // no thread crossed (rounding): last token of the chunk with positive weight
    __shared__ int lastpos_all;
    if (threadIdx.x == 0) lastpos_all = -1;
    __syncthreads();
    int lp = -1;
#pragma unroll
    for (int j = 0; j < kPerThread; ++j)
      if (w[j] > 0.f) lp = t0 + j;
    if (lp >= 0) atomicMax(&lastpos_all, lp);
    __syncthreads();
    if (threadIdx.x == 0) sh.result = lastpos_all >= 0 ? lastpos_all : v0;
    __syncthreads();
  }
  return sh.result;
}

// ---------------------------------------------------------------- sampler
__global__ void __launch_bounds__(kSampThreads) sample_kernel(const __grid_constant__ SampleDesc s) {
  __shared__ float sm_a[kSampWarps];
  __shared__ float sm_b[kSampWarps];
  __shared__ int sm_i[kSampWarps];
  __shared__ int sm_flag;
  __shared__ DrawShared sh;
  pdl_trigger();
  pdl_wait();
  const int c = blockIdx.x, r = blockIdx.y;
  const int nch = gridDim.x;
  const float* row = s.logits + (size_t)r * s.ld;
  const float* mix = s.mix_src ? s.mix_src + (size_t)r * s.mix_ld : nullptr;
  float* mixed = s.mixed_out ? s.mixed_out + (size_t)r * s.mixed_ld : nullptr;
  const int v0 = c * kVocabChunk, v1 = min(s.V, v0 + kVocabChunk);
  const bool greedy = s.temperature == 0.f;
  const float invT = greedy ? 1.f : 1.0f / s.temperature;

  const float* src = row;
  if (mix) {
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) {
      const int v = v0 + threadIdx.x + j * kSampThreads;
      if (v < v1) mixed[v] = (1.f - s.lambda) * row[v] + s.lambda * mix[v];
    }
    __syncthreads();
    src = mixed;   // this CTA's own writes: visible to its threads after the barrier
  } else if (mixed) {   // no mixing: the row itself is kept there
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) {
      const int v = v0 + threadIdx.x + j * kSampThreads;
      if (v < v1) mixed[v] = row[v];
    }
  }
  float* part = s.partials + ((size_t)r * nch + c) * 3;
  if (greedy) {
    float bv;
    int bi;
    chunk_argmax(src, v0, v1, sm_a, sm_i, &bv, &bi);
    if (threadIdx.x == 0) { part[0] = bv; part[1] = __int_as_float(bi); }
  } else {
    float m, sum;
    chunk_softmax_stats(src, v0, v1, invT, sm_a, sm_b, &m, &sum);
    if (threadIdx.x == 0) { part[0] = m; part[2] = sum; }
  }
  if (!last_arrival(s.tickets, r, nch, &sm_flag)) return;

  // ---- last CTA of this row: partials loaded in parallel into shared memory ----
  const float* P = s.partials + (size_t)r * nch * 3;
  __shared__ float pm[kMaxChunks], pz[kMaxChunks];
  __shared__ int pi[kMaxChunks];
  for (int k = threadIdx.x; k < nch; k += kSampThreads) {
    pm[k] = __ldcg(P + 3 * k);
    pi[k] = __float_as_int(__ldcg(P + 3 * k + 1));
    pz[k] = __ldcg(P + 3 * k + 2);
  }
  __syncthreads();
  int tok;
  if (greedy) {
    if (threadIdx.x == 0) {
      float bv = neg_inf();
      int bi = 0x7fffffff;
      for (int k = 0; k < nch; ++k) am_combine(bv, bi, pm[k], pi[k]);
      sh.result = bi;
    }
    __syncthreads();
    tok = sh.result;
  } else {
    __shared__ float gmax;
    if (threadIdx.x == 0) {
      float M = neg_inf();
      for (int k = 0; k < nch; ++k) M = fmaxf(M, pm[k]);
      gmax = M;
    }
    __syncthreads();
    const float M = gmax;
    for (int k = threadIdx.x; k < nch; k += kSampThreads)
      sh.mass[k] = (pm[k] == neg_inf()) ? 0.0 : (double)(pz[k] * expf(pm[k] - M));
    // batch: row r is sequence r (its own step counter, Philox row word r);
    // else rows are independent draws at steps step + r
    // row_pos: rows are the draft positions position + r of one step
    const uint64_t st0 = s.step_dev ? (uint64_t)s.step_dev[s.batch ? (size_t)r * s.st_ld : 0] : 0;
    const uint32_t step = (uint32_t)(st0 + s.step_base + (s.batch || s.row_pos ? 0 : r));
    const uint32_t pos = s.position + (s.row_pos ? (uint32_t)r : 0u);
    const float u = philox_uniform(s.seed, step, pos, s.stream, s.batch ? (uint32_t)r : 0u);
    pick_chunk(sh, nch, u);
    const float* srcall = mix ? mixed : row;
    auto wfn = [&](int v) { return expf(__ldcg(srcall + v) * invT - M); };
    tok = rescan_chunk(sh, wfn, s.V);
  }
  // rows without a finite logit (a forward that gave up) leave the scan with
  // no token: draw 0 rather than an id outside the vocabulary
  if (tok < 0 || tok >= s.V) tok = 0;
  if (threadIdx.x == 0) {
    // a forward that gave up (err raised) produced no logits to commit: the
    // draw is still written out, but the committed state stays as it was
    const bool commit = s.commit_seq && !(s.err && ld_volatile_i32(s.err) != 0);
    if (s.batch) {
      const size_t so = (size_t)r * s.seq_ld, io = (size_t)r * s.st_ld;
      s.out_token[(size_t)r * s.out_ld + (s.out_idx ? s.out_idx[io] : 0) + s.out_off] = tok;
      if (commit) {
        const int len = s.commit_len[io];
        s.commit_seq[so + len + 1] = tok;
        s.commit_len[io] = len + 1;
        s.commit_step[io] += 1;
      }
    } else {
      s.out_token[(s.out_idx ? *s.out_idx : 0) + s.out_off + r] = tok;
      if (commit) {
        const int len = *s.commit_len;
        s.commit_seq[len + 1] = tok;
        *s.commit_len = len + 1;
        *s.commit_step += 1;
      }
    }
    s.tickets[r] = 0;
  }
}

cudaError_t launch_sample(const SampleDesc& s, cudaStream_t st) {
  if (s.rows <= 0 || s.V <= 0 || vocab_chunks(s.V) > kMaxChunks) return cudaErrorInvalidValue;
  return launch_k(sample_kernel, dim3(vocab_chunks(s.V), s.rows), dim3(kSampThreads), 0, st, s);
}

// ---------------------------------------------------------------- acceptance
__global__ void __launch_bounds__(kSampThreads) accept_kernel(const __grid_constant__ AcceptDesc a) {
  __shared__ float sm_a[kSampWarps];
  __shared__ float sm_b[kSampWarps];
  __shared__ int sm_i[kSampWarps];
  __shared__ int sm_flag;
  __shared__ DrawShared sh;
  __shared__ double rowM[2 * kMaxK + 1], rowZ[2 * kMaxK + 1];
  __shared__ int argm[kMaxK + 1];
  __shared__ int dec_n, dec_kind, dec_tok;   // accepted count; kind 0 residual, 1 bonus, 2 greedy
  pdl_trigger();
  pdl_wait();

  const int r = blockIdx.y;
  const int K = a.K, V = a.V;
  const int nch = vocab_chunks(V);
  const int nrow = 2 * K + 1;                // p_1..p_{K+1}, q_1..q_K
  const bool greedy = a.temperature == 0.f;
  const int nstat = greedy ? K + 1 : nrow;
  const float invT = greedy ? 1.f : 1.0f / a.temperature;
  const float* P = a.p + (size_t)r * a.p_ld;
  const float* Q = a.q + (size_t)r * a.q_ld;
  const int nbl = accept_blocks_per_stat(V);            // CTAs per logit row
  const int j = blockIdx.x / nbl;                       // logit row
  const int c = (blockIdx.x % nbl) * kSampWarps + (threadIdx.x >> 5);   // this warp's chunk

  // ---- phase A: one (logit row, chunk) per warp, kSampWarps chunks per CTA ----
  if (c < nch) {
    const int v0 = c * kVocabChunk, v1 = min(V, v0 + kVocabChunk);
    float* part = a.partials + (((size_t)r * nrow + j) * nch + c) * 2;
    const float* src = j <= K ? P + (size_t)j * V : Q + (size_t)(j - K - 1) * V;
    if (greedy) {
      float bv;
      int bi;
      warp_chunk_argmax(src, v0, v1, &bv, &bi);
      if ((threadIdx.x & 31) == 0) { part[0] = bv; part[1] = __int_as_float(bi); }
    } else {
      float m, sum;
      warp_chunk_softmax(src, v0, v1, invT, &m, &sum);
      if ((threadIdx.x & 31) == 0) { part[0] = m; part[1] = sum; }
    }
  }
  if (!last_arrival(a.tickets, r, nstat * nbl, &sm_flag)) return;

  // ---- phase B: fold partials in chunk order, decisions ----
  // batch: row r is sequence r (its own step counter, Philox row word r,
  // drafts in its own token array); else rows are independent verify rows
  const size_t io = a.batch ? (size_t)r * a.st_ld : 0;
  const uint64_t st0 = a.step_dev ? (uint64_t)a.step_dev[io] : 0;
  const uint32_t step = (uint32_t)(st0 + a.step_base + (a.batch ? 0 : r));
  const uint32_t prow = a.batch ? (uint32_t)r : 0u;
  const int32_t* D = a.batch ? a.drafts + (size_t)r * a.seq_ld + (a.drafts_idx ? a.drafts_idx[io] : 0) + a.drafts_off
                             : a.drafts + (a.drafts_idx ? *a.drafts_idx : 0) + a.drafts_off + (size_t)r * K;
  const float* PR = a.partials + (size_t)r * nrow * nch * 2;
  // all partials of this verify row into shared memory, loaded in parallel
  __shared__ float pa_[(2 * kMaxK + 1) * kMaxChunks], pb_[(2 * kMaxK + 1) * kMaxChunks];
  for (int e = threadIdx.x; e < nstat * nch; e += kSampThreads) {
    pa_[e] = __ldcg(PR + 2 * e);
    pb_[e] = __ldcg(PR + 2 * e + 1);
  }
  __syncthreads();
  if (threadIdx.x < nstat) {
    const int jj = threadIdx.x;
    const float* ma = pa_ + jj * nch;
    const float* mb = pb_ + jj * nch;
    if (greedy) {
      float bv = neg_inf();
      int bi = 0x7fffffff;
      for (int k = 0; k < nch; ++k) am_combine(bv, bi, ma[k], __float_as_int(mb[k]));
      argm[jj] = bi;
    } else {
      float M = neg_inf();
      for (int k = 0; k < nch; ++k) M = fmaxf(M, ma[k]);
      double Z = 0.0;
      for (int k = 0; k < nch; ++k)
        if (ma[k] != neg_inf()) Z += (double)(mb[k] * expf(ma[k] - M));
      rowM[jj] = (double)M;
      rowZ[jj] = Z;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int n = K, kind = 1, tok = -1;
    if (greedy) {
      kind = 2;
      for (int i = 0; i < K; ++i) {
        if (D[i] != argm[i]) { n = i; tok = argm[i]; break; }
      }
      if (n == K) tok = argm[K];
    } else {
      for (int i = 0; i < K; ++i) {
        const int d = D[i];
        // p_i(d) / q_i(d) = exp((zp - Mp) - (zq - Mq)) * Zq / Zp, in fp32 with
        // the normaliser ratio taken in fp64
        const float lp = P[(size_t)i * V + d] * invT - (float)rowM[i];
        const float lq = Q[(size_t)i * V + d] * invT - (float)rowM[K + 1 + i];
        const float ratio = expf(lp - lq) * (float)(rowZ[K + 1 + i] / rowZ[i]);
        const float rr = philox_uniform(a.seed, step, (uint32_t)(i + 1), kStreamAccept, prow);
        if (!(rr < fminf(1.0f, ratio))) { n = i; kind = 0; break; }
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
  if (kind == 0) {
    const float* pr = P + (size_t)n * V;
    const float* qr = Q + (size_t)n * V;
    const float mp = (float)rowM[n], mq = (float)rowM[K + 1 + n];
    const float izp = (float)(1.0 / rowZ[n]), izq = (float)(1.0 / rowZ[K + 1 + n]);
    auto wres = [&](int v) {
      return fmaxf(expf(pr[v] * invT - mp) * izp - expf(qr[v] * invT - mq) * izq, 0.f);
    };
    // residual mass of every chunk: warp w takes chunks w, w + 8, ...
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int cc = wid; cc < nch; cc += kSampWarps) {
      const int b0 = cc * kVocabChunk, b1 = min(V, b0 + kVocabChunk);
      float acc = 0.f;
      for (int base = b0; base < b1; base += 32 * 16) {
        float pv[16], qv[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int v = base + lane + 32 * u;
          pv[u] = v < b1 ? pr[v] : neg_inf();
          qv[u] = v < b1 ? qr[v] : neg_inf();
        }
#pragma unroll
        for (int u = 0; u < 16; ++u)
          acc += fmaxf(expf(pv[u] * invT - mp) * izp - expf(qv[u] * invT - mq) * izq, 0.f);
      }
      acc = warp_sum(acc);
      if (lane == 0) sh.mass[cc] = (double)acc;
    }
    const float u = philox_uniform(a.seed, step, (uint32_t)(n + 1), kStreamResidual, prow);
    const double z = pick_chunk(sh, nch, u);
    if (z > 0.0) {
      tok = rescan_chunk(sh, wres, V);
    } else {   // zero residual mass (rounding): draw from p_i
      flags |= 0x1u;
      for (int k = threadIdx.x; k < nch; k += kSampThreads) {
        const float m = pa_[n * nch + k], sm = pb_[n * nch + k];
        sh.mass[k] = (m == neg_inf()) ? 0.0 : (double)(sm * expf(m - (float)rowM[n]));
      }
      pick_chunk(sh, nch, u);
      auto wp = [&](int v) { return expf(pr[v] * invT - mp); };
      tok = rescan_chunk(sh, wp, V);
    }
  } else if (kind == 1) {
    const float* pr = P + (size_t)K * V;
    const float mp = (float)rowM[K];
    for (int k = threadIdx.x; k < nch; k += kSampThreads) {
      const float m = pa_[K * nch + k], sm = pb_[K * nch + k];
      sh.mass[k] = (m == neg_inf()) ? 0.0 : (double)(sm * expf(m - (float)rowM[K]));
    }
    const float u = philox_uniform(a.seed, step, (uint32_t)(K + 1), kStreamBonus, prow);
    pick_chunk(sh, nch, u);
    auto wp = [&](int v) { return expf(pr[v] * invT - mp); };
    tok = rescan_chunk(sh, wp, V);
  }

  if (tok < 0 || tok >= V) tok = 0;   // no finite logit in the row: never an id outside the vocabulary
  if (threadIdx.x == 0) {
    int32_t* out = a.out_tokens + (size_t)r * (K + 1);
    if (a.drafts_copy)
      for (int i = 0; i < K; ++i) a.drafts_copy[(size_t)r * K + i] = D[i];
    for (int i = 0; i < n; ++i) out[i] = D[i];
    out[n] = tok;
    for (int i = n + 1; i <= K; ++i) out[i] = -1;
    a.out_count[r] = n + 1;
    if (a.out_flags) a.out_flags[r] = flags;
    // a forward that gave up (err raised) left no valid logits: nothing is
    // committed, so the context keeps its committed length and step counter
    if (a.commit_seq && !(a.err && ld_volatile_i32(a.err) != 0)) {
      int32_t* cs = a.commit_seq + (a.batch ? (size_t)r * a.seq_ld : 0);
      const int len = a.commit_len[io];
      for (int i = 0; i <= n; ++i) cs[len + 1 + i] = out[i];
      a.commit_len[io] = len + n + 1;
      a.commit_step[io] += 1;
    }
    a.tickets[r] = 0;
  }
}

cudaError_t launch_accept(const AcceptDesc& a, cudaStream_t st) {
  if (a.rows <= 0 || a.K < 1 || a.K > kMaxK || a.V <= 0) return cudaErrorInvalidValue;
  const int nch = vocab_chunks(a.V);
  if (nch > kMaxChunks) return cudaErrorInvalidValue;
  const int nstat = a.temperature == 0.f ? a.K + 1 : 2 * a.K + 1;
  return launch_k(accept_kernel, dim3(nstat * accept_blocks_per_stat(a.V), a.rows), dim3(kSampThreads), 0, st, a);
}

}  // namespace sv
