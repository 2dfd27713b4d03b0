// Per-layer kernels of the decoder forward other than the weight GEMMs:
// embedding gather, RMSNorm, RoPE + KV-cache append, and causal attention of
// the new positions over the KV cache.
//
// The target pass computes a next-token distribution at each of the K+1 new
// positions in one forward ("Speculative decoding internals", 演算法核心
// Step 2: T_1 = T(.|x) ... T_{K+1} = T(.|x, d_1..K)); position L+j attends to
// keys 0..L+j.  Rolling back a rejected suffix is a length truncation: the
// stale KV rows beyond the committed length are never read (each query only
// reads keys at or before its own position) and are overwritten later.
#include "common.cuh"
#include "kernels.h"

namespace sv {

// ---------------------------------------------------------------- embedding
template <typename T>
__global__ void embed_kernel(const int32_t* __restrict__ tok_base, const int32_t* tok_idx,
                             int tok_off, const T* __restrict__ emb, float* __restrict__ x, int d) {
  const int t = blockIdx.x;
  const int32_t* tok = tok_base + (tok_idx ? *tok_idx : 0) + tok_off;
  const T* row = emb + (size_t)tok[t] * d;
  for (int i = threadIdx.x; i < d; i += blockDim.x) x[(size_t)t * d + i] = to_f32(row[i]);
}

cudaError_t launch_embed(const int32_t* tok_base, const int32_t* tok_idx, int tok_off,
                         const void* embed, int dtype, float* x, int ntok, int d, cudaStream_t st) {
  if (dtype == 0)
    embed_kernel<float><<<ntok, 256, 0, st>>>(tok_base, tok_idx, tok_off, (const float*)embed, x, d);
  else
    embed_kernel<bf16><<<ntok, 256, 0, st>>>(tok_base, tok_idx, tok_off, (const bf16*)embed, x, d);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- RMSNorm
// One CTA per token; the sum of squares is reduced in a fixed order (per
// thread strided partials, warp shuffle tree, warps in index order).
template <typename T>
__global__ void __launch_bounds__(256) rmsnorm_kernel(const float* __restrict__ x,
                                                      const float* __restrict__ gain, float eps,
                                                      T* __restrict__ out, int d) {
  __shared__ float red[8];
  const int t = blockIdx.x;
  const float* xr = x + (size_t)t * d;
  float ss = 0.f;
  for (int i = threadIdx.x; i < d; i += 256) ss += xr[i] * xr[i];
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) tot += red[w];
  const float inv = 1.0f / sqrtf(tot / (float)d + eps);
  for (int i = threadIdx.x; i < d; i += 256)
    out[(size_t)t * d + i] = from_f32<T>(xr[i] * inv * gain[i]);
}

cudaError_t launch_rmsnorm(const float* x, const float* gain, float eps, void* out, int dtype,
                           int ntok, int d, cudaStream_t st) {
  if (dtype == 0)
    rmsnorm_kernel<float><<<ntok, 256, 0, st>>>(x, gain, eps, (float*)out, d);
  else
    rmsnorm_kernel<bf16><<<ntok, 256, 0, st>>>(x, gain, eps, (bf16*)out, d);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- RoPE tables
// cos/sin(pos * theta^(-2i/hd)) evaluated in fp64 so that the angle is exact
// enough at long contexts, stored as fp32.
__global__ void rope_table_kernel(float* cs, float* sn, int cap, int hd, double theta) {
  const int half = hd / 2;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)cap * half) return;
  const int pos = (int)(idx / half), i = (int)(idx % half);
  const double inv = pow(theta, -2.0 * i / (double)hd);
  double s, c;
  sincos((double)pos * inv, &s, &c);
  cs[idx] = (float)c;
  sn[idx] = (float)s;
}

cudaError_t launch_rope_table(float* cos_out, float* sin_out, int cap, int hd, double theta,
                              cudaStream_t st) {
  const long long n = (long long)cap * (hd / 2);
  rope_table_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(cos_out, sin_out, cap, hd, theta);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- RoPE + KV append
// Rotate-half RoPE: pairs (i, i + hd/2) rotated by pos * w_i.
template <typename T>
__global__ void rope_append_kernel(const __grid_constant__ RopeDesc r) {
  const int half = r.hd / 2;
  const int nh = r.hq + 2 * r.hkv;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)r.ntok * nh * half) return;
  const int i = (int)(idx % half);
  const int h = (int)((idx / half) % nh);
  const int t = (int)(idx / ((long long)half * nh));
  const int pos = *r.pos_base + r.pos_off + t;
  const float* src = r.qkv + (size_t)t * nh * r.hd + (size_t)h * r.hd;
  T* kc = (T*)r.kc;
  T* vc = (T*)r.vc;
  if (h >= r.hq + r.hkv) {  // value head: copy
    const int vh = h - r.hq - r.hkv;
    T* dst = vc + ((size_t)vh * r.cap + pos) * r.hd;
    dst[i] = from_f32<T>(src[i]);
    dst[i + half] = from_f32<T>(src[i + half]);
    return;
  }
  const float c = r.rope_cos[(size_t)pos * half + i], s = r.rope_sin[(size_t)pos * half + i];
  const float x1 = src[i], x2 = src[i + half];
  const float y1 = x1 * c - x2 * s, y2 = x2 * c + x1 * s;
  if (h < r.hq) {
    float* dq = r.q_out + ((size_t)t * r.hq + h) * r.hd;
    dq[i] = y1;
    dq[i + half] = y2;
  } else {
    T* dst = kc + ((size_t)(h - r.hq) * r.cap + pos) * r.hd;
    dst[i] = from_f32<T>(y1);
    dst[i + half] = from_f32<T>(y2);
  }
}

cudaError_t launch_rope_append(const RopeDesc& r, cudaStream_t st) {
  const long long n = (long long)r.ntok * (r.hq + 2 * r.hkv) * (r.hd / 2);
  const unsigned blocks = (unsigned)((n + 255) / 256);
  if (r.dtype == 0)
    rope_append_kernel<float><<<blocks, 256, 0, st>>>(r);
  else
    rope_append_kernel<bf16><<<blocks, 256, 0, st>>>(r);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- attention
// Query rows of one KV head: row r = t * G + j (token t, query head
// kvh * G + j, G = hq / hkv).  A CTA takes up to kRowsPerCta rows and one
// 64-key chunk c of absolute key positions [64c, 64c + 64), computes for each
// row the chunk partial (m = max score, l = sum exp(s - m), o = sum
// exp(s - m) v) over the keys at or before the row's position, and stores
// it.  The combine kernel folds the partials of chunks 0..pos/64 in
// ascending order.  Chunk boundaries are absolute, so a row's result does
// not depend on which other rows share the launch.
constexpr int kRowsPerCta = 32;
constexpr int kAttnThreads = 128;

size_t attn_partial_floats(int max_tok, int hq, int hd, int max_chunks) {
  return (size_t)max_tok * hq * max_chunks * (hd + 2);
}

template <int HD, typename T>
__global__ void __launch_bounds__(kAttnThreads) attn_chunk_kernel(const __grid_constant__ AttnDesc a) {
  extern __shared__ float sm[];
  float* Ks = sm;                                 // [64][HD+1]
  float* Vs = Ks + kAttnChunk * (HD + 1);         // [64][HD]
  float* Qs = Vs + kAttnChunk * HD;               // [kRowsPerCta][HD]
  float* S = Qs + kRowsPerCta * HD;               // [kRowsPerCta][64]
  float* Mx = S + kRowsPerCta * kAttnChunk;       // [kRowsPerCta]
  float* Ls = Mx + kRowsPerCta;                   // [kRowsPerCta]
  __shared__ int rowpos[kRowsPerCta];

  const int kvh = blockIdx.x;
  const int c = blockIdx.y;
  const int G = a.hq / a.hkv;
  const int nrows_all = a.ntok * G;
  const int r0 = blockIdx.z * kRowsPerCta;
  const int nrows = min(kRowsPerCta, nrows_all - r0);
  if (nrows <= 0) return;
  const int base = *a.pos_base + a.pos_off;
  const int key0 = c * kAttnChunk;
  const int pmax = base + (r0 + nrows - 1) / G;   // highest position in this row tile
  if (key0 > pmax) return;                        // chunk lies entirely in the future
  const int nkeys = min(kAttnChunk, pmax - key0 + 1);
  const int tid = threadIdx.x;

  const T* kc = (const T*)a.kc + ((size_t)kvh * a.cap + key0) * HD;
  const T* vc = (const T*)a.vc + ((size_t)kvh * a.cap + key0) * HD;
  for (int e = tid; e < kAttnChunk * HD; e += kAttnThreads) {
    const int j = e / HD, d = e % HD;
    const bool ok = j < nkeys;
    Ks[j * (HD + 1) + d] = ok ? to_f32(kc[(size_t)j * HD + d]) : 0.f;
    Vs[j * HD + d] = ok ? to_f32(vc[(size_t)j * HD + d]) : 0.f;
  }
  for (int e = tid; e < nrows * HD; e += kAttnThreads) {
    const int rr = e / HD, d = e % HD;
    const int r = r0 + rr;
    const int t = r / G, h = kvh * G + r % G;
    Qs[rr * HD + d] = a.q[((size_t)t * a.hq + h) * HD + d];
  }
  if (tid < nrows) rowpos[tid] = base + (r0 + tid) / G;
  __syncthreads();

  // scores: s = scale * q . k, -inf beyond the row's own position
  for (int e = tid; e < nrows * kAttnChunk; e += kAttnThreads) {
    const int rr = e / kAttnChunk, j = e % kAttnChunk;
    float s = neg_inf();
    if (key0 + j <= rowpos[rr]) {
      const float* q = Qs + rr * HD;
      const float* k = Ks + j * (HD + 1);
      float acc = 0.f;
#pragma unroll 8
      for (int d = 0; d < HD; ++d) acc = fmaf(q[d], k[d], acc);
      s = acc * a.scale;
    }
    S[rr * kAttnChunk + j] = s;
  }
  __syncthreads();

  // per-row max and sum of exp (warp per row, fixed shuffle tree)
  const int lane = tid & 31, warp = tid >> 5;
  for (int rr = warp; rr < nrows; rr += kAttnThreads / 32) {
    const float s0 = S[rr * kAttnChunk + lane], s1 = S[rr * kAttnChunk + lane + 32];
    const float m = warp_max(fmaxf(s0, s1));
    float p0 = 0.f, p1 = 0.f;
    if (m != neg_inf()) {
      p0 = (s0 == neg_inf()) ? 0.f : expf(s0 - m);
      p1 = (s1 == neg_inf()) ? 0.f : expf(s1 - m);
    }
    const float l = warp_sum(p0 + p1);
    S[rr * kAttnChunk + lane] = p0;
    S[rr * kAttnChunk + lane + 32] = p1;
    if (lane == 0) {
      Mx[rr] = m;
      Ls[rr] = l;
    }
  }
  __syncthreads();

  // o[row][d] = sum_j p[row][j] * v[j][d], keys in ascending order
  constexpr int kGroups = kAttnThreads / HD;      // rows handled per pass
  const int d = tid % HD, rg = tid / HD;
  for (int rr = rg; rr < nrows; rr += kGroups) {
    float acc = 0.f;
    const float* p = S + rr * kAttnChunk;
    for (int j = 0; j < nkeys; ++j) acc = fmaf(p[j], Vs[j * HD + d], acc);
    const int r = r0 + rr;
    const int t = r / G, h = kvh * G + r % G;
    float* dst = a.partials + (((size_t)t * a.hq + h) * a.max_chunks + c) * (HD + 2);
    dst[d] = acc;
    if (d == 0) {
      dst[HD] = Mx[rr];
      dst[HD + 1] = Ls[rr];
    }
  }
}

// Fold the chunk partials of one (token, query head) in ascending chunk order.
template <int HD, typename T>
__global__ void __launch_bounds__(HD) attn_combine_kernel(const __grid_constant__ AttnDesc a) {
  const int t = blockIdx.x / a.hq, h = blockIdx.x % a.hq;
  const int d = threadIdx.x;
  const int pos = *a.pos_base + a.pos_off + t;
  const int nc = pos / kAttnChunk + 1;
  const float* src = a.partials + ((size_t)t * a.hq + h) * a.max_chunks * (HD + 2);
  float M = neg_inf(), L = 0.f, O = 0.f;
  for (int c = 0; c < nc; ++c) {
    const float* p = src + (size_t)c * (HD + 2);
    const float m = p[HD], l = p[HD + 1], o = p[d];
    const float Mn = fmaxf(M, m);
    const float sa = expf(M - Mn), sb = expf(m - Mn);
    L = L * sa + l * sb;
    O = O * sa + o * sb;
    M = Mn;
  }
  ((T*)a.out)[(size_t)t * a.hq * HD + (size_t)h * HD + d] = from_f32<T>(O / L);
}

template <int HD>
static size_t attn_smem() {
  return sizeof(float) * ((size_t)kAttnChunk * (HD + 1) + (size_t)kAttnChunk * HD +
                          (size_t)kRowsPerCta * HD + (size_t)kRowsPerCta * kAttnChunk +
                          2 * kRowsPerCta);
}

template <int HD, typename T>
static cudaError_t configure_attn() {
  return cudaFuncSetAttribute(attn_chunk_kernel<HD, T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)attn_smem<HD>());
}

cudaError_t configure_kernels() {
  cudaError_t e;
  if ((e = configure_attn<32, float>()) != cudaSuccess) return e;
  if ((e = configure_attn<64, float>()) != cudaSuccess) return e;
  if ((e = configure_attn<128, float>()) != cudaSuccess) return e;
  if ((e = configure_attn<32, bf16>()) != cudaSuccess) return e;
  if ((e = configure_attn<64, bf16>()) != cudaSuccess) return e;
  return configure_attn<128, bf16>();
}

template <int HD, typename T>
static cudaError_t launch_attn_t(const AttnDesc& a, cudaStream_t st) {
  const size_t smem = attn_smem<HD>();
  const int G = a.hq / a.hkv;
  const int rtiles = (a.ntok * G + kRowsPerCta - 1) / kRowsPerCta;
  attn_chunk_kernel<HD, T><<<dim3(a.hkv, a.max_chunks, rtiles), kAttnThreads, smem, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_combine_kernel<HD, T><<<a.ntok * a.hq, HD, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_attention(const AttnDesc& a, cudaStream_t st) {
  if (a.hq % a.hkv != 0) return cudaErrorInvalidValue;
  if (a.dtype == 0) {
    if (a.hd == 32) return launch_attn_t<32, float>(a, st);
    if (a.hd == 64) return launch_attn_t<64, float>(a, st);
    if (a.hd == 128) return launch_attn_t<128, float>(a, st);
  } else {
    if (a.hd == 32) return launch_attn_t<32, bf16>(a, st);
    if (a.hd == 64) return launch_attn_t<64, bf16>(a, st);
    if (a.hd == 128) return launch_attn_t<128, bf16>(a, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace sv
