// Device side of the chunked causal attention, shared by the per-layer
// kernel (layers.cu) and the persistent forward kernel (persist.cu).  See
// layers.cu for the design.
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace sv {

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
// Barrier over the attention threads (the first 256 of the CTA: all of a
// per-layer attention CTA; the consumer warps of the persistent kernel).
SV_DEV void attn_sync() { named_sync(1, kAttnThreads); }


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

// One work item: (KV head kvh, chunk c, row tile rz of nrz).  Every thread
// of the CTA calls it; sm is the CTA's dynamic shared memory, rowpos/s_last
// static shared scratch of the caller.
template <int HD, typename T>
SV_DEV void attn_item(const AttnDesc& a, int kvh, int c, int rz, int nrz, float* sm, int* rowpos,
                      int* s_last) {
  constexpr int KS = HD + 4;
  float* Ks = sm;                                 // [64][KS]
  float* Vs = Ks + kAttnChunk * KS;               // [64][HD]
  float* Qs = Vs + kAttnChunk * HD;               // [32][HD]
  float* S = Qs + kRowsPerCta * HD;               // [32][64]
  float* Pt = S + kRowsPerCta * kAttnChunk;       // [64][32]
  float* Mx = Pt + kAttnChunk * kRowsPerCta;      // [32]
  float* Ls = Mx + kRowsPerCta;                   // [32]
  const int G = a.hq / a.hkv;
  const int nrows_all = a.ntok * G;
  const int r0 = rz * kRowsPerCta;
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
    kr[i] = ok ? __ldcg(reinterpret_cast<const uint4*>(kc + (size_t)j * HD + dv * EPV)) : make_uint4(0, 0, 0, 0);
    vr[i] = ok ? __ldcg(reinterpret_cast<const uint4*>(vc + (size_t)j * HD + dv * EPV)) : make_uint4(0, 0, 0, 0);
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
      qr[i] = __ldcg(reinterpret_cast<const float4*>(a.q + ((size_t)t * a.hq + h) * HD + d4 * 4));
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
  attn_sync();

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
  attn_sync();

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
  attn_sync();

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
  int* ticket = a.tickets + kvh * nrz + rz;
  attn_sync();
  if (tid == 0) {
    __threadfence();
    *s_last = (atomicAdd(ticket, 1) == arrivals - 1);
  }
  attn_sync();
  if (!*s_last) return;
  __threadfence();
  // (m, l) of every (row, chunk) of the tile into shared memory, 4 loads in
  // flight per thread; then per row: M = max m_c, w_c = exp(m_c - M),
  // L = sum_c w_c l_c (lane-strided, fixed tree)
  const int mc = a.max_chunks;
  float* W = sm;                                  // [32][mc]: m_c, then w_c
  float* Lc = W + (size_t)kRowsPerCta * mc;       // [32][mc]: l_c
  float* invL = Lc + (size_t)kRowsPerCta * mc;    // [32]
  const int ncmax_tile = pmax / kAttnChunk + 1;
  const int npairs = nrows * ncmax_tile;
  for (int e0 = tid; e0 < npairs; e0 += 4 * kAttnThreads) {
    float mv[4], lv[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int e = e0 + b * kAttnThreads;
      mv[b] = lv[b] = 0.f;
      if (e < npairs) {
        const int rr = e / ncmax_tile, cc = e % ncmax_tile;
        if (cc <= rowpos[rr] / kAttnChunk) {
          const int r = r0 + rr;
          const int t = r / G, h = kvh * G + r % G;
          const float* pp = a.partials + (((size_t)t * a.hq + h) * mc + cc) * (HD + 2);
          mv[b] = __ldcg(pp + HD);
          lv[b] = __ldcg(pp + HD + 1);
        }
      }
    }
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int e = e0 + b * kAttnThreads;
      if (e < npairs) {
        const int rr = e / ncmax_tile, cc = e % ncmax_tile;
        W[rr * mc + cc] = mv[b];
        Lc[rr * mc + cc] = lv[b];
      }
    }
  }
  attn_sync();
  for (int rr = warp; rr < nrows; rr += kAttnThreads / 32) {
    const int nc = rowpos[rr] / kAttnChunk + 1;
    float m = neg_inf();
    for (int cc = lane; cc < nc; cc += 32) m = fmaxf(m, W[rr * mc + cc]);
    m = warp_max(m);
    float lsum = 0.f;
    for (int cc = lane; cc < nc; cc += 32) {
      const float w = expf(W[rr * mc + cc] - m);
      W[rr * mc + cc] = w;
      lsum += w * Lc[rr * mc + cc];
    }
    lsum = warp_sum(lsum);
    if (lane == 0) invL[rr] = lsum;
  }
  attn_sync();
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


// Dynamic shared memory of one attention CTA (floats).
template <int HD>
inline size_t attn_smem_floats(int max_chunks) {
  const size_t combine = (size_t)2 * kRowsPerCta * max_chunks + kRowsPerCta;
  return attn_layout_floats<HD>() > combine ? attn_layout_floats<HD>() : combine;
}

}  // namespace sv
