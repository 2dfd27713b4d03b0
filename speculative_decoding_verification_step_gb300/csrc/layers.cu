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
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x;
  const int32_t* tok = tok_base + (tok_idx ? *tok_idx : 0) + tok_off;
  const T* row = emb + (size_t)tok[t] * d;
  for (int i = threadIdx.x; i < d; i += blockDim.x) x[(size_t)t * d + i] = to_f32(row[i]);
}

cudaError_t launch_embed(const int32_t* tok_base, const int32_t* tok_idx, int tok_off,
                         const void* embed, int dtype, float* x, int ntok, int d, cudaStream_t st) {
  if (dtype == 0)
    return launch_k(embed_kernel<float>, dim3(ntok), dim3(256), 0, st, tok_base, tok_idx, tok_off,
                    (const float*)embed, x, d);
  return launch_k(embed_kernel<bf16>, dim3(ntok), dim3(256), 0, st, tok_base, tok_idx, tok_off,
                  (const bf16*)embed, x, d);
}

// ---------------------------------------------------------------- RMSNorm
// One CTA per token; the sum of squares is reduced in a fixed order (per
// thread strided partials, warp shuffle tree, warps in index order).
template <typename T>
__global__ void __launch_bounds__(256) rmsnorm_kernel(const float* __restrict__ x,
                                                      const float* __restrict__ gain, float eps,
                                                      T* __restrict__ out, int d) {
  __shared__ float red[8];
  pdl_trigger();
  pdl_wait();
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
    return launch_k(rmsnorm_kernel<float>, dim3(ntok), dim3(256), 0, st, x, gain, eps, (float*)out, d);
  return launch_k(rmsnorm_kernel<bf16>, dim3(ntok), dim3(256), 0, st, x, gain, eps, (bf16*)out, d);
}

// ---------------------------------------------------------------- RoPE tables
// cos/sin(pos * theta^(-2i/hd)) evaluated in fp64 so that the angle is exact
// enough at long contexts, stored as fp32.
__global__ void rope_table_kernel(float* cs, float* sn, int cap, int hd, double theta) {
  pdl_trigger();
  pdl_wait();
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
  return launch_k(rope_table_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, cos_out,
                  sin_out, cap, hd, theta);
}

// ---------------------------------------------------------------- RoPE + KV append
// Rotate-half RoPE: pairs (i, i + hd/2) rotated by pos * w_i.
template <typename T>
__global__ void rope_append_kernel(const __grid_constant__ RopeDesc r) {
  pdl_trigger();
  pdl_wait();
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
  if (r.dtype == 0) return launch_k(rope_append_kernel<float>, dim3(blocks), dim3(256), 0, st, r);
  return launch_k(rope_append_kernel<bf16>, dim3(blocks), dim3(256), 0, st, r);
}

// ---------------------------------------------------------------- attention
// Query rows of one KV head: row r = t * G + j (token t, query head
// kvh * G + j, G = hq / hkv).  A CTA takes up to 32 rows and one 64-key chunk
// c of absolute key positions [64c, 64c + 64) and computes, for each row,
// the chunk partial (m = max score, l = sum exp(s - m), o = sum exp(s - m) v)
// over the keys at or before the row's position.  The CTA that finishes a
// (KV head, row tile) last combines, for each of its rows, the partials of
// chunks 0..pos/64: M = max m_c, out = sum_c exp(m_c - M) o_c / sum_c
// exp(m_c - M) l_c, with every sum in ascending chunk order.  Chunk
// boundaries are absolute and every row's numbers depend only on its own
// partials, so a row's result does not depend on which other rows share the
// launch.
constexpr int kRowsPerCta = kAttnRowsPerCta;
constexpr int kAttnThreads = 256;

size_t attn_partial_floats(int max_tok, int hq, int hd, int max_chunks) {
  return (size_t)max_tok * hq * max_chunks * (hd + 2);
}
int attn_max_row_tiles(int max_tok, int hq, int hkv) {
  return (max_tok * (hq / hkv) + kRowsPerCta - 1) / kRowsPerCta;
}

// Shared-memory layout (floats): Ks [64][HD+4] (padded so that the 16 key
// groups of a warp hit distinct bank groups), Vs [64][HD], Qs [32][HD],
// S [32][64], Pt [64][32] (probabilities, key-major), Mx [32], Ls [32].
template <int HD>
constexpr size_t attn_layout_floats() {
  return (size_t)kAttnChunk * (HD + 4) + (size_t)kAttnChunk * HD + (size_t)kRowsPerCta * HD +
         2 * (size_t)kRowsPerCta * kAttnChunk + 2 * kRowsPerCta;
}
constexpr size_t kAttnSmemCap = 200 * 1024;

SV_DEV void to_floats(const uint4& v, float* dst, const bf16*) {
  dst[0] = bf16lo(v.x); dst[1] = bf16hi(v.x); dst[2] = bf16lo(v.y); dst[3] = bf16hi(v.y);
  dst[4] = bf16lo(v.z); dst[5] = bf16hi(v.z); dst[6] = bf16lo(v.w); dst[7] = bf16hi(v.w);
}
SV_DEV void to_floats(const uint4& v, float* dst, const float*) {
  dst[0] = __uint_as_float(v.x); dst[1] = __uint_as_float(v.y);
  dst[2] = __uint_as_float(v.z); dst[3] = __uint_as_float(v.w);
}

SV_DEV float dot4(const float4& a, const float4& b, float acc) {
  acc = fmaf(a.x, b.x, acc);
  acc = fmaf(a.y, b.y, acc);
  acc = fmaf(a.z, b.z, acc);
  return fmaf(a.w, b.w, acc);
}

template <int HD, typename T>
__global__ void __launch_bounds__(kAttnThreads) attn_chunk_kernel(const __grid_constant__ AttnDesc a) {
  constexpr int KS = HD + 4;
  extern __shared__ __align__(16) float sm[];
  float* Ks = sm;                                 // [64][KS]
  float* Vs = Ks + kAttnChunk * KS;               // [64][HD]
  float* Qs = Vs + kAttnChunk * HD;               // [32][HD]
  float* S = Qs + kRowsPerCta * HD;               // [32][64]
  float* Pt = S + kRowsPerCta * kAttnChunk;       // [64][32]
  float* Mx = Pt + kAttnChunk * kRowsPerCta;      // [32]
  float* Ls = Mx + kRowsPerCta;                   // [32]
  __shared__ int rowpos[kRowsPerCta];
  __shared__ int s_last;
  pdl_trigger();
  pdl_wait();

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
  const int lane = tid & 31, warp = tid >> 5;

  // ---- stage K, V and Q: every 16-byte load issued before any store ----
  constexpr int EPV = 16 / sizeof(T);             // elements per 16-byte vector
  constexpr int VPR = HD / EPV;                   // vectors per key row
  constexpr int PER = kAttnChunk * VPR / kAttnThreads;
  static_assert(PER >= 1, "tile too small");
  const T* kc = (const T*)a.kc + ((size_t)kvh * a.cap + key0) * HD;
  const T* vc = (const T*)a.vc + ((size_t)kvh * a.cap + key0) * HD;
  uint4 kr[PER], vr[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int idx = tid + i * kAttnThreads;
    const int j = idx / VPR, dv = idx % VPR;
    const bool ok = j < nkeys;
    kr[i] = ok ? *reinterpret_cast<const uint4*>(kc + (size_t)j * HD + dv * EPV) : make_uint4(0, 0, 0, 0);
    vr[i] = ok ? *reinterpret_cast<const uint4*>(vc + (size_t)j * HD + dv * EPV) : make_uint4(0, 0, 0, 0);
  }
  constexpr int QPER = (kRowsPerCta * HD / 4 + kAttnThreads - 1) / kAttnThreads;
  float4 qr[QPER];
#pragma unroll
  for (int i = 0; i < QPER; ++i) {
    const int idx = tid + i * kAttnThreads;
    const int rr = idx / (HD / 4), d4 = idx % (HD / 4);
    qr[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (rr < nrows) {
      const int r = r0 + rr;
      const int t = r / G, h = kvh * G + r % G;
      qr[i] = *reinterpret_cast<const float4*>(a.q + ((size_t)t * a.hq + h) * HD + d4 * 4);
    }
  }
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int idx = tid + i * kAttnThreads;
    const int j = idx / VPR, dv = idx % VPR;
    float f[EPV];
    to_floats(kr[i], f, (const T*)nullptr);
#pragma unroll
    for (int e = 0; e < EPV; e += 4)
      *reinterpret_cast<float4*>(Ks + j * KS + dv * EPV + e) = make_float4(f[e], f[e + 1], f[e + 2], f[e + 3]);
    to_floats(vr[i], f, (const T*)nullptr);
#pragma unroll
    for (int e = 0; e < EPV; e += 4)
      *reinterpret_cast<float4*>(Vs + j * HD + dv * EPV + e) = make_float4(f[e], f[e + 1], f[e + 2], f[e + 3]);
  }
#pragma unroll
  for (int i = 0; i < QPER; ++i) {
    const int idx = tid + i * kAttnThreads;
    const int rr = idx / (HD / 4), d4 = idx % (HD / 4);
    if (rr < kRowsPerCta) *reinterpret_cast<float4*>(Qs + rr * HD + d4 * 4) = qr[i];
  }
  if (tid < kRowsPerCta) rowpos[tid] = tid < nrows ? base + (r0 + tid) / G : -1;
  __syncthreads();

  // ---- scores: thread = (row pair, key quad); keys kq, kq+16, kq+32, kq+48 ----
  {
    const int kq = tid & 15, rp = tid >> 4;
    float acc[2][4];
#pragma unroll
    for (int a2 = 0; a2 < 2; ++a2)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[a2][i] = 0.f;
    const float* q0p = Qs + (2 * rp) * HD;
    const float* q1p = q0p + HD;
#pragma unroll 4
    for (int d = 0; d < HD; d += 4) {
      const float4 q0 = *reinterpret_cast<const float4*>(q0p + d);
      const float4 q1 = *reinterpret_cast<const float4*>(q1p + d);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 k = *reinterpret_cast<const float4*>(Ks + (kq + 16 * i) * KS + d);
        acc[0][i] = dot4(q0, k, acc[0][i]);
        acc[1][i] = dot4(q1, k, acc[1][i]);
      }
    }
#pragma unroll
    for (int a2 = 0; a2 < 2; ++a2) {
      const int rr = 2 * rp + a2;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int j = kq + 16 * i;
        S[rr * kAttnChunk + j] = (key0 + j <= rowpos[rr]) ? acc[a2][i] * a.scale : neg_inf();
      }
    }
  }
  __syncthreads();

  // ---- per-row max and sum of exp (warp per row, fixed shuffle tree) ----
  for (int rr = warp; rr < kRowsPerCta; rr += kAttnThreads / 32) {
    const float s0 = S[rr * kAttnChunk + lane], s1 = S[rr * kAttnChunk + lane + 32];
    const float m = warp_max(fmaxf(s0, s1));
    float p0 = 0.f, p1 = 0.f;
    if (m != neg_inf()) {
      p0 = (s0 == neg_inf()) ? 0.f : expf(s0 - m);
      p1 = (s1 == neg_inf()) ? 0.f : expf(s1 - m);
    }
    const float l = warp_sum(p0 + p1);
    Pt[lane * kRowsPerCta + rr] = p0;
    Pt[(lane + 32) * kRowsPerCta + rr] = p1;
    if (lane == 0) {
      Mx[rr] = m;
      Ls[rr] = l;
    }
  }
  __syncthreads();

  // ---- o[row][d] = sum_j p[row][j] v[j][d]: thread = (RPT rows, 4 dims) ----
  constexpr int DQ = HD / 4;                      // dim quads
  constexpr int RPT = kRowsPerCta * DQ / kAttnThreads;   // rows per thread: HD/32
  const int dq = tid % DQ, rg = tid / DQ;
  {
    float4 o[RPT];
#pragma unroll
    for (int q = 0; q < RPT; ++q) o[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < nkeys; ++j) {
      const float4 v = *reinterpret_cast<const float4*>(Vs + j * HD + dq * 4);
      const float* pj = Pt + j * kRowsPerCta + rg * RPT;
#pragma unroll
      for (int q = 0; q < RPT; ++q) {
        const float p = pj[q];
        o[q].x = fmaf(p, v.x, o[q].x);
        o[q].y = fmaf(p, v.y, o[q].y);
        o[q].z = fmaf(p, v.z, o[q].z);
        o[q].w = fmaf(p, v.w, o[q].w);
      }
    }
#pragma unroll
    for (int q = 0; q < RPT; ++q) {
      const int rr = rg * RPT + q;
      if (rr < nrows) {
        const int r = r0 + rr;
        const int t = r / G, h = kvh * G + r % G;
        float* dst = a.partials + (((size_t)t * a.hq + h) * a.max_chunks + c) * (HD + 2);
        *reinterpret_cast<float2*>(dst + dq * 4) = make_float2(o[q].x, o[q].y);
        *reinterpret_cast<float2*>(dst + dq * 4 + 2) = make_float2(o[q].z, o[q].w);
        if (dq == 0) {
          dst[HD] = Mx[rr];
          dst[HD + 1] = Ls[rr];
        }
      }
    }
  }

  // ---- the last chunk CTA of this (KV head, row tile) combines ----
  const int arrivals = pmax / kAttnChunk + 1;
  int* ticket = a.tickets + kvh * gridDim.z + blockIdx.z;
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    s_last = (atomicAdd(ticket, 1) == arrivals - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  float* W = sm;                                  // [32][max_chunks] chunk weights
  float* invL = W + (size_t)kRowsPerCta * a.max_chunks;
  for (int rr = warp; rr < nrows; rr += kAttnThreads / 32) {
    const int r = r0 + rr;
    const int t = r / G, h = kvh * G + r % G;
    const int nc = rowpos[rr] / kAttnChunk + 1;
    const float* src = a.partials + ((size_t)t * a.hq + h) * a.max_chunks * (HD + 2);
    float m = neg_inf();
    for (int cc = lane; cc < nc; cc += 32) m = fmaxf(m, __ldcg(src + (size_t)cc * (HD + 2) + HD));
    m = warp_max(m);
    float lsum = 0.f;
    for (int cc = lane; cc < nc; cc += 32) {
      const float* pp = src + (size_t)cc * (HD + 2);
      const float w = expf(__ldcg(pp + HD) - m);
      W[rr * a.max_chunks + cc] = w;
      lsum += w * __ldcg(pp + HD + 1);
    }
    lsum = warp_sum(lsum);
    if (lane == 0) invL[rr] = lsum;
  }
  __syncthreads();
  {
    // every thread folds RPT rows x 4 dims; chunk loads are batched 4 deep
    float4 o[RPT];
#pragma unroll
    for (int q = 0; q < RPT; ++q) o[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    int ncmax = 0;
#pragma unroll
    for (int q = 0; q < RPT; ++q) {
      const int rr = rg * RPT + q;
      if (rr < nrows) ncmax = max(ncmax, rowpos[rr] / kAttnChunk + 1);
    }
    for (int c0 = 0; c0 < ncmax; c0 += 4) {
      float2 lo[4][RPT], hi[4][RPT];
#pragma unroll
      for (int b = 0; b < 4; ++b)
#pragma unroll
        for (int q = 0; q < RPT; ++q) {
          const int rr = rg * RPT + q;
          const int cc = c0 + b;
          lo[b][q] = hi[b][q] = make_float2(0.f, 0.f);
          if (rr < nrows && cc <= rowpos[rr] / kAttnChunk) {
            const int r = r0 + rr;
            const int t = r / G, h = kvh * G + r % G;
            const float* pp = a.partials + (((size_t)t * a.hq + h) * a.max_chunks + cc) * (HD + 2) + dq * 4;
            lo[b][q] = __ldcg(reinterpret_cast<const float2*>(pp));
            hi[b][q] = __ldcg(reinterpret_cast<const float2*>(pp + 2));
          }
        }
#pragma unroll
      for (int b = 0; b < 4; ++b)
#pragma unroll
        for (int q = 0; q < RPT; ++q) {
          const int rr = rg * RPT + q;
          const int cc = c0 + b;
          if (rr < nrows && cc <= rowpos[rr] / kAttnChunk) {
            const float w = W[rr * a.max_chunks + cc];
            o[q].x = fmaf(w, lo[b][q].x, o[q].x);
            o[q].y = fmaf(w, lo[b][q].y, o[q].y);
            o[q].z = fmaf(w, hi[b][q].x, o[q].z);
            o[q].w = fmaf(w, hi[b][q].y, o[q].w);
          }
        }
    }
#pragma unroll
    for (int q = 0; q < RPT; ++q) {
      const int rr = rg * RPT + q;
      if (rr < nrows) {
        const int r = r0 + rr;
        const int t = r / G, h = kvh * G + r % G;
        const float L = invL[rr];
        T* dst = (T*)a.out + (size_t)t * a.hq * HD + (size_t)h * HD + dq * 4;
        dst[0] = from_f32<T>(o[q].x / L);
        dst[1] = from_f32<T>(o[q].y / L);
        dst[2] = from_f32<T>(o[q].z / L);
        dst[3] = from_f32<T>(o[q].w / L);
      }
    }
  }
  if (tid == 0) *ticket = 0;
}

template <int HD, typename T>
static cudaError_t configure_attn() {
  return cudaFuncSetAttribute(attn_chunk_kernel<HD, T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)kAttnSmemCap);
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
  const size_t combine = (size_t)kRowsPerCta * a.max_chunks + kRowsPerCta;
  const size_t smem = sizeof(float) * (attn_layout_floats<HD>() > combine ? attn_layout_floats<HD>() : combine);
  if (smem > kAttnSmemCap) return cudaErrorInvalidValue;
  const int G = a.hq / a.hkv;
  const int rtiles = (a.ntok * G + kRowsPerCta - 1) / kRowsPerCta;
  return launch_k(attn_chunk_kernel<HD, T>, dim3(a.hkv, a.max_chunks, rtiles), dim3(kAttnThreads), smem,
                  st, a);
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
