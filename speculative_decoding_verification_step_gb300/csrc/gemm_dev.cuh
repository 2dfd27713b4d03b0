// Device side of the weight-streaming skinny GEMM, shared by the per-layer
// kernels (gemm.cu) and the persistent forward kernel (persist.cu).  See
// gemm.cu for the design.
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace sv {

constexpr int kStepK = 64;
constexpr int kMinStepsPerWarp = 8;

__host__ __device__ inline int gemm_tiles_of(const GemmDesc& g) {
  return g.epi == kEpiSwiglu ? g.n / 8 : (g.n + 15) / 16;
}

// Row r of the weight segments stacked along n.
template <typename E>
SV_DEV const E* seg_row(const GemmDesc& g, int row) {
  int r = row;
  if (r < g.seg_rows[0]) return (const E*)g.w[0] + (size_t)r * g.k;
  r -= g.seg_rows[0];
  if (r < g.seg_rows[1]) return (const E*)g.w[1] + (size_t)r * g.k;
  r -= g.seg_rows[1];
  return (const E*)g.w[2] + (size_t)r * g.k;
}

// Rows (lo, hi) a tile assigns to thread row g (0..7); -1 if out of range.
SV_DEV void tile_rows(const GemmDesc& g, int tile, int gi, int* lo, int* hi) {
  if (g.epi == kEpiQkvRope) {
    const int per = g.hd / 16;
    const int h = tile / per, j = tile % per;
    *lo = h * g.hd + 8 * j + gi;
    *hi = *lo + g.hd / 2;
  } else {
    *lo = tile * 16 + gi;
    *hi = *lo + 8;
    if (*lo >= g.n) *lo = -1;
    if (*hi >= g.n) *hi = -1;
  }
}

// 1 / sqrt(mean x^2 + eps) of token tok from per-16-row-tile sums of squares:
// lanes sum tiles lane, lane + 32, ... then a fixed shuffle tree (the result
// depends only on the token's own sums).
SV_DEV float warp_inv_rms(const GemmDesc& g, int tok, int lane) {
  const int tiles = g.k / 16;
  float s = 0.f;
  for (int t0 = 0; t0 < tiles; t0 += 32 * 8) {
    float v[8];   // 8 loads in flight per lane, added in ascending tile order
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int t = t0 + lane + 32 * u;
      v[u] = t < tiles ? __ldcg(g.ss_in + (size_t)t * g.ss_ld + tok) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) s += v[u];
  }
  s = warp_sum(s);
  return 1.0f / sqrtf(s / (float)g.k + g.eps);
}

// Epilogue inputs that do not depend on the sums, for one-token-group tiles
// (tokens 2ci, 2ci+1): the residual of rows lo/hi (kEpiAdd) or the RoPE
// cos/sin of the tokens' positions (q/k heads of kEpiQkvRope) in v[j] /
// v[2+j], the next RMSNorm's gains of rows lo/hi (kEpiAdd with xg_out) in gn;
// pos0 = position of token 0.  Issued together with other loads so that
// their latencies overlap.
struct EpiIn {
  float v[4];
  float gn[2];
  int pos0;
};

// Position of token tok of a q/k/v GEMM (pos0 = *pos_base + pos_off, used
// for one sequence) and the first KV row of its sequence.  kSeqs = false:
// the caller runs single-sequence passes only (the persistent kernel).
template <bool kSeqs = true>
SV_DEV int tok_pos(const GemmDesc& g, int tok, int pos0) {
  if (!kSeqs || g.spt <= 0) return pos0 + tok;
  return g.pos_base[(size_t)(tok / g.spt) * g.pos_ld] + g.pos_off + tok % g.spt;
}
template <bool kSeqs = true>
SV_DEV size_t tok_kv_row0(const GemmDesc& g, int tok) {
  return kSeqs ? (size_t)seq_of_tok(g.spt, tok) * g.hkv * g.cap : 0;
}
template <bool kSeqs = true>
SV_DEV void gemm_epi_load(const GemmDesc& g, int tile, int pos0, int gi, int ci, EpiIn& e) {
  e.pos0 = pos0;
  e.v[0] = e.v[1] = e.v[2] = e.v[3] = 0.f;
  e.gn[0] = e.gn[1] = 0.f;
  if (g.epi == kEpiAdd) {
    int lo, hi;
    tile_rows(g, tile, gi, &lo, &hi);
    if (g.xg_out) {
      if (lo >= 0) e.gn[0] = __ldg(g.gain_next + lo);
      if (hi >= 0) e.gn[1] = __ldg(g.gain_next + hi);
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int tok = 2 * ci + j;
      if (tok >= g.ntok) continue;
      const float* o = (const float*)g.out + (size_t)tok * g.ldo;
      if (lo >= 0) e.v[j] = __ldcg(o + lo);
      if (hi >= 0) e.v[2 + j] = __ldcg(o + hi);
    }
  } else if (g.epi == kEpiQkvRope) {
    const int per = g.hd / 16, half = g.hd / 2;
    const int h = tile / per, i = 8 * (tile % per) + gi;
    if (h >= g.hq + g.hkv) return;   // value head: no rotation
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int tok = 2 * ci + j;
      if (tok >= g.ntok) continue;
      const int pos = tok_pos<kSeqs>(g, tok, pos0);
      e.v[j] = __ldg(g.rope_cos + (size_t)pos * half + i);
      e.v[2 + j] = __ldg(g.rope_sin + (size_t)pos * half + i);
    }
  }
}

// ---- epilogue: thread holds rows lo/hi of the tile for tokens ng*8 + 2ci + j;
// pre (NG = 1 only): the inputs gemm_epi_load read, else they are loaded here ----
template <int NG, bool kSeqs = true>
SV_DEV void gemm_epilogue(const GemmDesc& g, int tile, const float (&acc)[NG][4], int gi, int ci,
                          const EpiIn* pre = nullptr) {
  if (g.epi == kEpiSwiglu) {
#pragma unroll
    for (int ng = 0; ng < NG; ++ng)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int tok = ng * 8 + 2 * ci + j;
        if (tok < g.ntok)
          ((bf16*)g.out)[(size_t)tok * g.ldo + tile * 8 + gi] =
              __float2bfloat16_rn(silu(acc[ng][j]) * acc[ng][2 + j]);
      }
    return;
  }
  if (g.epi == kEpiHeadRes) {
    int lo, hi;
    tile_rows(g, tile, gi, &lo, &hi);
#pragma unroll
    for (int ng = 0; ng < NG; ++ng)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int tok = ng * 8 + 2 * ci + j;
        if (tok >= g.ntok) continue;
        const float* u = g.hres + (size_t)tok * g.k;
        bf16* o = (bf16*)g.out + (size_t)tok * g.ldo;
        if (lo >= 0) o[lo] = __float2bfloat16_rn(u[lo % g.k] + silu(acc[ng][j]));
        if (hi >= 0) o[hi] = __float2bfloat16_rn(u[hi % g.k] + silu(acc[ng][2 + j]));
      }
    return;
  }
  if (g.epi == kEpiQkvRope) {
    const int per = g.hd / 16, half = g.hd / 2;
    const int h = tile / per, i = 8 * (tile % per) + gi;
#pragma unroll
    for (int ng = 0; ng < NG; ++ng)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int tok = ng * 8 + 2 * ci + j;
        if (tok >= g.ntok) continue;
        const float x1 = acc[ng][j], x2 = acc[ng][2 + j];
        const int pos = tok_pos<kSeqs>(g, tok, pre ? pre->pos0 : (kSeqs && g.spt > 0 ? 0 : *g.pos_base + g.pos_off));
        const size_t kv0 = tok_kv_row0<kSeqs>(g, tok);
        if (h >= g.hq + g.hkv) {   // value head: stored as is
          bf16* dst = (bf16*)g.vc + (kv0 + (size_t)(h - g.hq - g.hkv) * g.cap + pos) * g.hd;
          dst[i] = __float2bfloat16_rn(x1);
          dst[i + half] = __float2bfloat16_rn(x2);
          continue;
        }
        const float c = pre ? pre->v[j] : g.rope_cos[(size_t)pos * half + i];
        const float s = pre ? pre->v[2 + j] : g.rope_sin[(size_t)pos * half + i];
        const float y1 = x1 * c - x2 * s, y2 = x2 * c + x1 * s;
        if (h < g.hq) {
          float* dq = g.q_out + ((size_t)tok * g.hq + h) * g.hd;
          dq[i] = y1;
          dq[i + half] = y2;
        } else {
          bf16* dst = (bf16*)g.kc + (kv0 + (size_t)(h - g.hq) * g.cap + pos) * g.hd;
          dst[i] = __float2bfloat16_rn(y1);
          dst[i + half] = __float2bfloat16_rn(y2);
        }
      }
    return;
  }
  int lo, hi;
  tile_rows(g, tile, gi, &lo, &hi);
#pragma unroll
  for (int ng = 0; ng < NG; ++ng)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int tok = ng * 8 + 2 * ci + j;
      float ss = 0.f;
      if (tok < g.ntok) {
        float* o = (float*)g.out + (size_t)tok * g.ldo;
        if (g.epi == kEpiAdd) {
          bf16* xg = g.xg_out ? (bf16*)g.xg_out + (size_t)tok * g.ldo : nullptr;
          if (lo >= 0) {
            const float v = (pre ? pre->v[j] : __ldcg(o + lo)) + acc[ng][j];
            o[lo] = v;
            ss = v * v;
            if (xg) xg[lo] = __float2bfloat16_rn(v * (pre ? pre->gn[0] : __ldg(g.gain_next + lo)));
          }
          if (hi >= 0) {
            const float v = (pre ? pre->v[2 + j] : __ldcg(o + hi)) + acc[ng][2 + j];
            o[hi] = v;
            ss = fmaf(v, v, ss);
            if (xg) xg[hi] = __float2bfloat16_rn(v * (pre ? pre->gn[1] : __ldg(g.gain_next + hi)));
          }
        } else {
          if (lo >= 0) o[lo] = acc[ng][j];
          if (hi >= 0) o[hi] = acc[ng][2 + j];
        }
      }
      if (g.epi == kEpiAdd && g.ss_out) {
        // sum over the tile's 16 rows: rows g and g+8 per lane, then over g
        ss += __shfl_xor_sync(0xffffffffu, ss, 4);
        ss += __shfl_xor_sync(0xffffffffu, ss, 8);
        ss += __shfl_xor_sync(0xffffffffu, ss, 16);
        if (gi == 0 && tok < g.ntok) g.ss_out[(size_t)tile * g.ss_ld + tok] = ss;
      }
    }
}

// Largest warp whose range starts at or before step s (ranges are
// floor(w*T/N) .. floor((w+1)*T/N), all non-empty because N <= T).
SV_DEV int warp_of_step(long long s, long long total, long long nw) {
  return (int)(((s + 1) * nw - 1) / total);
}
SV_DEV long long first_step_of_warp(long long w, long long total, long long nw) {
  return (w * total) / nw;
}

// X fragment words of one k-step for token tok (8 bf16 pairs: x0 = words 0..3,
// x1 = words 4..7 of the thread's 16 consecutive k).
template <bool NORM>
SV_DEV void load_x(const GemmDesc& g, int tok, int off, float inv, uint4& x0, uint4& x1) {
  if (!NORM) {
    const uint4* xp = (const uint4*)((const uint16_t*)g.x + (size_t)tok * g.ldx + off);
    x0 = __ldcg(xp);   // activations: L2-coherent loads (they may have been
    x1 = __ldcg(xp + 1);   // written by other CTAs of a persistent launch)
    return;
  }
  const float4* xp = (const float4*)((const float*)g.x + (size_t)tok * g.ldx + off);
  const float4* gp = (const float4*)(g.gain + off);
  uint32_t w[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 xv = __ldcg(xp + q), gv = __ldg(gp + q);
    const __nv_bfloat162 a = __floats2bfloat162_rn(xv.x * inv * gv.x, xv.y * inv * gv.y);
    const __nv_bfloat162 b = __floats2bfloat162_rn(xv.z * inv * gv.z, xv.w * inv * gv.w);
    w[2 * q] = *reinterpret_cast<const uint32_t*>(&a);
    w[2 * q + 1] = *reinterpret_cast<const uint32_t*>(&b);
  }
  x0 = make_uint4(w[0], w[1], w[2], w[3]);
  x1 = make_uint4(w[4], w[5], w[6], w[7]);
}

template <int U>
struct WeightRing {
  uint4 a[U][2], b[U][2];
};

// Load k-steps ks .. ks+U-1 (those below ke) of rows pa / pb into the ring.
template <int U>
SV_DEV void ring_fill(WeightRing<U>& r, const uint16_t* pa, const uint16_t* pb, int ks, int ke, int ci) {
  const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int off = (ks + u) * kStepK + ci * 16;
    const bool live = ks + u < ke;
    r.a[u][0] = (live && pa) ? ld_stream(pa + off) : z;
    r.a[u][1] = (live && pa) ? ld_stream(pa + off + 8) : z;
    r.b[u][0] = (live && pb) ? ld_stream(pb + off) : z;
    r.b[u][1] = (live && pb) ? ld_stream(pb + off + 8) : z;
  }
}

SV_DEV void tile_ptrs(const GemmDesc& g, int tile, int gi, const uint16_t*& pa, const uint16_t*& pb) {
  if (g.epi == kEpiSwiglu) {
    const int r = tile * 8 + gi;
    pa = (const uint16_t*)g.w[0] + (size_t)r * g.k;
    pb = (const uint16_t*)g.w[1] + (size_t)r * g.k;
  } else {
    int lo, hi;
    tile_rows(g, tile, gi, &lo, &hi);
    pa = lo >= 0 ? seg_row<uint16_t>(g, lo) : nullptr;
    pb = hi >= 0 ? seg_row<uint16_t>(g, hi) : nullptr;
  }
}

// X source: kXGlobal = bf16 X from global memory; kXSmem = the normalised X
// of every token in shared memory, once per CTA (rows padded by 8 elements so
// the fragment loads are bank-conflict free) -- the per-kernel GEMM
// normalises the fp32 residual into it, the persistent kernel copies in the
// bf16 rows pre-multiplied by the gain (x_norm = 2); kXInline = RMSNorm
// applied while loading (large token counts, where the normalised X would not
// fit).
// (XMode: kernels.h)
constexpr int kXPad = 8;

// Per-warp state of one GEMM: its range of (tile, k-step) units and the
// weight ring of its current tile.
template <int U>
struct GemmWarp {
  WeightRing<U> ring;
  const uint16_t* pa;
  const uint16_t* pb;
  long long total, nw;
  int s, s1, tile, ks, ke, spt;
  bool has_work;
};

// Work split for warp gw of nwarps and the first weight loads of its first
// tile.  Weights are read-only, so this may run before the inputs are ready.
template <int U>
SV_DEV void gemm_begin(const GemmDesc& g, int total_steps, int spt, int gw, int nwarps,
                       GemmWarp<U>& st) {
  const int lane = threadIdx.x & 31;
  const int gi = lane >> 2, ci = lane & 3;
  st.total = total_steps;
  st.spt = spt;
  // at least kMinStepsPerWarp k-steps per warp: bounds how many warps share a
  // tile (and so the length of its reduction) for small matrices
  st.nw = max(1LL, min((long long)nwarps, st.total / kMinStepsPerWarp));
  st.has_work = gw < st.nw;
  st.s = st.has_work ? (int)first_step_of_warp(gw, st.total, st.nw) : 0;
  st.s1 = st.has_work ? (int)first_step_of_warp(gw + 1, st.total, st.nw) : 0;
  st.tile = st.s / spt;
  st.ks = st.s - st.tile * spt;
  st.ke = min(spt, st.ks + (st.s1 - st.s));
  st.pa = st.pb = nullptr;
  if (st.has_work) {
    tile_ptrs(g, st.tile, gi, st.pa, st.pb);
    ring_fill<U>(st.ring, st.pa, st.pb, st.ks, st.ke, ci);
  }
}

// CTA-wide (every thread of the CTA calls it): 1/rms of every token and, in
// kXSmem mode, the normalised bf16 X of every token in shared memory.
// Normalised bf16 x * inv_rms * gain of 8 consecutive k of one token.
SV_DEV uint4 norm_chunk(const float4& a0, const float4& a1, float iv, const float4& g0, const float4& g1) {
  const __nv_bfloat162 b0 = __floats2bfloat162_rn(a0.x * iv * g0.x, a0.y * iv * g0.y);
  const __nv_bfloat162 b1 = __floats2bfloat162_rn(a0.z * iv * g0.z, a0.w * iv * g0.w);
  const __nv_bfloat162 b2 = __floats2bfloat162_rn(a1.x * iv * g1.x, a1.y * iv * g1.y);
  const __nv_bfloat162 b3 = __floats2bfloat162_rn(a1.z * iv * g1.z, a1.w * iv * g1.w);
  return make_uint4(*reinterpret_cast<const uint32_t*>(&b0), *reinterpret_cast<const uint32_t*>(&b1),
                    *reinterpret_cast<const uint32_t*>(&b2), *reinterpret_cast<const uint32_t*>(&b3));
}

template <int XM>
SV_DEV void gemm_prepare_x(const GemmDesc& g, float* s_inv, uint16_t* s_x) {
  if (XM == kXGlobal && g.x_norm != 2) return;   // x_norm = 2: 1/rms scales the epilogue
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
  for (int tok = warp; tok < g.ntok; tok += nwarp) {
    const float v = warp_inv_rms(g, tok, lane);
    if (lane == 0) s_inv[tok] = v;
  }
  __syncthreads();
  if (XM != kXSmem) return;
  const int ld = g.k + kXPad;
  const int per_tok = g.k / 8;
  const int chunks = g.ntok * per_tok;
  for (int e0 = threadIdx.x; e0 < chunks; e0 += 2 * blockDim.x) {
    float4 a[2][2], gg[2][2];
#pragma unroll
    for (int b = 0; b < 2; ++b) {   // both chunks' loads issued before use
      const int e = e0 + b * blockDim.x;
      if (e < chunks) {
        const int tok = e / per_tok, k0 = (e % per_tok) * 8;
        const float4* xp = (const float4*)((const float*)g.x + (size_t)tok * g.ldx + k0);
        const float4* gp = (const float4*)(g.gain + k0);
        a[b][0] = __ldcg(xp);
        a[b][1] = __ldcg(xp + 1);
        gg[b][0] = __ldg(gp);
        gg[b][1] = __ldg(gp + 1);
      }
    }
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const int e = e0 + b * blockDim.x;
      if (e < chunks) {
        const int tok = e / per_tok, k0 = (e % per_tok) * 8;
        *reinterpret_cast<uint4*>(s_x + (size_t)tok * ld + k0) =
            norm_chunk(a[b][0], a[b][1], s_inv[tok], gg[b][0], gg[b][1]);
      }
    }
  }
  __syncthreads();
}

// x_norm = 2: the finished sums of token ng*8 + 2ci + j times its 1 / rms.
template <int NG>
SV_DEV void scale_by_inv_rms(const GemmDesc& g, float (&acc)[NG][4], const float* s_inv, int ci) {
  if (g.x_norm != 2) return;
#pragma unroll
  for (int ng = 0; ng < NG; ++ng)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int tok = ng * 8 + 2 * ci + j;
      const float sc = tok < g.ntok ? s_inv[tok] : 1.f;
      acc[ng][j] *= sc;
      acc[ng][2 + j] *= sc;
    }
}

// Main loop and epilogues of one warp (after gemm_begin and gemm_prepare_x).
template <int NG, int U, int XM>
SV_DEV void gemm_run(const GemmDesc& g, GemmWarp<U>& st, int gw, float* __restrict__ partials,
                     int* __restrict__ tickets, const float* s_inv, const uint16_t* s_x) {
  if (!st.has_work) return;
  const int lane = threadIdx.x & 31;
  const int gi = lane >> 2, ci = lane & 3;
  const uint4 zero4 = make_uint4(0, 0, 0, 0);
  const int spt = st.spt;
  int slot = 0;
  while (true) {
    float acc[NG][4];
#pragma unroll
    for (int ng = 0; ng < NG; ++ng)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[ng][e] = 0.f;
    float inv[NG];
#pragma unroll
    for (int ng = 0; ng < NG; ++ng) {
      const int tok = ng * 8 + gi;
      inv[ng] = (XM == kXInline && tok < g.ntok) ? s_inv[tok] : 1.f;
    }
    const int ks = st.ks, ke = st.ke, tile = st.tile;
    // Rolling prefetch: ring slot u holds k-step kk + u; right after its MMAs
    // consume it, it is refilled with step kk + u + U.
    for (int kk = ks; kk < ke; kk += U) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int stp = kk + u;
        if (stp < ke) {
          const int off = stp * kStepK + ci * 16;
#pragma unroll
          for (int ng = 0; ng < NG; ++ng) {
            const int tok = ng * 8 + gi;
            uint4 x0 = zero4, x1 = zero4;
            if (tok < g.ntok) {
              if (XM == kXSmem) {
                const uint4* xp = reinterpret_cast<const uint4*>(s_x + (size_t)tok * (g.k + kXPad) + off);
                x0 = xp[0];
                x1 = xp[1];
              } else {
                load_x<XM == kXInline>(g, tok, off, inv[ng], x0, x1);
              }
            }
            const WeightRing<U>& r = st.ring;
            mma_bf16_16816(acc[ng], r.a[u][0].x, r.b[u][0].x, r.a[u][0].y, r.b[u][0].y, x0.x, x0.y);
            mma_bf16_16816(acc[ng], r.a[u][0].z, r.b[u][0].z, r.a[u][0].w, r.b[u][0].w, x0.z, x0.w);
            mma_bf16_16816(acc[ng], r.a[u][1].x, r.b[u][1].x, r.a[u][1].y, r.b[u][1].y, x1.x, x1.y);
            mma_bf16_16816(acc[ng], r.a[u][1].z, r.b[u][1].z, r.a[u][1].w, r.b[u][1].w, x1.z, x1.w);
          }
          const int nx = stp + U;
          if (nx < ke) {
            const int noff = nx * kStepK + ci * 16;
            if (st.pa) {
              st.ring.a[u][0] = ld_stream(st.pa + noff);
              st.ring.a[u][1] = ld_stream(st.pa + noff + 8);
            }
            if (st.pb) {
              st.ring.b[u][0] = ld_stream(st.pb + noff);
              st.ring.b[u][1] = ld_stream(st.pb + noff + 8);
            }
          }
        }
      }
    }

    if (ks == 0 && ke == spt) {
      scale_by_inv_rms<NG>(g, acc, s_inv, ci);
      gemm_epilogue<NG>(g, tile, acc, gi, ci);
    } else {
      float* mine = partials + (size_t)(gw * 2 + slot) * NG * 32 * 4;
#pragma unroll
      for (int ng = 0; ng < NG; ++ng)
        *reinterpret_cast<float4*>(mine + ((size_t)ng * 32 + lane) * 4) =
            make_float4(acc[ng][0], acc[ng][1], acc[ng][2], acc[ng][3]);
      __threadfence();
      __syncwarp();
      const int wfirst = warp_of_step((long long)tile * spt, st.total, st.nw);
      const int wlast = warp_of_step((long long)(tile + 1) * spt - 1, st.total, st.nw);
      int old = 0;
      if (lane == 0) old = atomicAdd(&tickets[tile], 1);
      old = __shfl_sync(0xffffffffu, old, 0);
      if (old == wlast - wfirst) {
        __threadfence();
        float tot[NG][4];
#pragma unroll
        for (int ng = 0; ng < NG; ++ng)
#pragma unroll
          for (int e = 0; e < 4; ++e) tot[ng][e] = 0.f;
        // partials are loaded kBatch at a time, then added in ascending warp order
        constexpr int kBatch = NG >= 8 ? 1 : 8 / NG;
        for (int w0 = wfirst; w0 <= wlast; w0 += kBatch) {
          float4 v[kBatch][NG];
#pragma unroll
          for (int b = 0; b < kBatch; ++b) {
            const int w = w0 + b;
            if (w <= wlast) {
              const int sl = (first_step_of_warp(w, st.total, st.nw) / spt == tile) ? 0 : 1;
              const float* src = partials + (size_t)(w * 2 + sl) * NG * 32 * 4;
#pragma unroll
              for (int ng = 0; ng < NG; ++ng)
                v[b][ng] = __ldcg(reinterpret_cast<const float4*>(src + ((size_t)ng * 32 + lane) * 4));
            }
          }
#pragma unroll
          for (int b = 0; b < kBatch; ++b) {
            if (w0 + b <= wlast) {
#pragma unroll
              for (int ng = 0; ng < NG; ++ng) {
                tot[ng][0] += v[b][ng].x;
                tot[ng][1] += v[b][ng].y;
                tot[ng][2] += v[b][ng].z;
                tot[ng][3] += v[b][ng].w;
              }
            }
          }
        }
        scale_by_inv_rms<NG>(g, tot, s_inv, ci);
        gemm_epilogue<NG>(g, tile, tot, gi, ci);
        if (lane == 0) tickets[tile] = 0;
      }
    }
    slot = 1;
    st.s += ke - ks;
    if (st.s >= st.s1) break;
    st.tile = st.s / spt;
    st.ks = st.s - st.tile * spt;
    st.ke = min(spt, st.ks + (st.s1 - st.s));
    tile_ptrs(g, st.tile, gi, st.pa, st.pb);
    ring_fill<U>(st.ring, st.pa, st.pb, st.ks, st.ke, ci);
  }
}

}  // namespace sv
