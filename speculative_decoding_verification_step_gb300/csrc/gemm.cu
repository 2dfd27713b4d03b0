// Weight-streaming "skinny" GEMM of the verification step: Y[ntok][n] = X . W^T
// with ntok = K+1 (or a prefill chunk) and W read from HBM exactly once.
//
// The target pass scores all K+1 positions with one read of every weight
// ("Speculative decoding internals", 為什麼能加速 and 演算法核心 Step 2;
// "Speculative Decoding 101", Floor 3): the positions are the N side of the
// product, the weight rows the M side.
//
// bf16 models (tensor cores, mma.sync m16n8k16):
//  * Work is a list of (16-row tile, 64-wide k step) units in tile-major
//    order, split into equal contiguous ranges, one per warp of a fixed grid
//    (2 CTAs of 8 warps per SM): every SM streams the same number of bytes
//    whatever the matrix shape (stream-K at warp granularity).
//  * Each lane loads 2 x 32 contiguous bytes (rows g and g+8 of the tile)
//    per step with 128-bit streaming loads; the loaded words are used as the
//    A fragments directly.  The k order inside a step is permuted
//    identically for the weights and the activations, which leaves every
//    dot product unchanged, so no shared-memory staging or shuffles are
//    needed.  The activations (tiny, L1-resident) are loaded the same way.
//  * A tile split between warps is reduced by its last-arriving warp, in
//    ascending warp order, from a global scratch buffer (arrival counted
//    with one atomic per partial; no waiting).  The split points depend only
//    on (n, k), never on ntok, so each output element is computed with the
//    same operations in the same order for any number of tokens: the pass
//    is batch-invariant (greedy speculative output equals greedy plain
//    decoding bit for bit on the GPU too).
// fp32 models (tiny workloads): one warp per output row on CUDA cores, with a
// fixed per-lane order and shuffle tree (also batch-invariant).
#include "common.cuh"
#include "kernels.h"

namespace sv {

constexpr int kStepK = 64;
constexpr int kMinStepsPerWarp = 8;

static bool g_pdl = false;
bool pdl_enabled() { return g_pdl; }
void set_pdl_enabled(bool on) { g_pdl = on; }

int gemm_grid(int num_sms) { return 2 * num_sms; }

size_t gemm_partial_floats(int num_sms) {
  // [warp][2 slots][8 token groups][32 lanes][4]
  return (size_t)gemm_grid(num_sms) * kGemmWarpsPerCta * 2 * 8 * 32 * 4;
}

int gemm_tiles(const GemmDesc& g) { return g.epi == kEpiSwiglu ? g.n / 8 : (g.n + 15) / 16; }

SV_DEV const uint16_t* seg_row_bf16(const GemmDesc& g, int row) {
  int r = row;
  if (r < g.seg_rows[0]) return (const uint16_t*)g.w[0] + (size_t)r * g.k;
  r -= g.seg_rows[0];
  if (r < g.seg_rows[1]) return (const uint16_t*)g.w[1] + (size_t)r * g.k;
  r -= g.seg_rows[1];
  return (const uint16_t*)g.w[2] + (size_t)r * g.k;
}

SV_DEV const float* seg_row_f32(const GemmDesc& g, int row) {
  int r = row;
  if (r < g.seg_rows[0]) return (const float*)g.w[0] + (size_t)r * g.k;
  r -= g.seg_rows[0];
  if (r < g.seg_rows[1]) return (const float*)g.w[1] + (size_t)r * g.k;
  r -= g.seg_rows[1];
  return (const float*)g.w[2] + (size_t)r * g.k;
}

// Largest warp whose range starts at or before step s (ranges are
// floor(w*T/N) .. floor((w+1)*T/N), all non-empty because N <= T).
SV_DEV int warp_of_step(long long s, long long total, long long nw) {
  return (int)(((s + 1) * nw - 1) / total);
}
SV_DEV long long first_step_of_warp(long long w, long long total, long long nw) {
  return (w * total) / nw;
}

template <int NG>
SV_DEV void gemm_epilogue(const GemmDesc& g, int tile, const float (&acc)[NG][4], int gi, int ci) {
#pragma unroll
  for (int ng = 0; ng < NG; ++ng) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int tok = ng * 8 + 2 * ci + j;
      if (tok >= g.ntok) continue;
      const float lo = acc[ng][j], hi = acc[ng][2 + j];
      if (g.epi == kEpiSwiglu) {
        const int row = tile * 8 + gi;
        ((bf16*)g.out)[(size_t)tok * g.ldo + row] = __float2bfloat16_rn(silu(lo) * hi);
      } else {
        float* o = (float*)g.out + (size_t)tok * g.ldo;
        const int ra = tile * 16 + gi, rb = ra + 8;
        if (g.epi == kEpiAdd) {
          if (ra < g.n) o[ra] += lo;
          if (rb < g.n) o[rb] += hi;
        } else {
          if (ra < g.n) o[ra] = lo;
          if (rb < g.n) o[rb] = hi;
        }
      }
    }
  }
}

template <int NG, int U>
__global__ void __launch_bounds__(256, 2)
gemm_bf16_streamk(const __grid_constant__ GemmDesc g, float* __restrict__ partials,
                  int* __restrict__ tickets, int total_steps, int spt) {
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kGemmWarpsPerCta + (threadIdx.x >> 5);
  const long long total = total_steps;
  // at least kMinStepsPerWarp k-steps per warp: bounds how many warps share a
  // tile (and so the length of its reduction) for small matrices
  const long long nw = max(1LL, min((long long)gridDim.x * kGemmWarpsPerCta, total / kMinStepsPerWarp));
  if (gw >= nw) return;
  const int gi = lane >> 2, ci = lane & 3;
  int s = (int)first_step_of_warp(gw, total, nw);
  const int s1 = (int)first_step_of_warp(gw + 1, total, nw);
  const bool swiglu = g.epi == kEpiSwiglu;
  const uint16_t* xbase = (const uint16_t*)g.x;
  int slot = 0;
  bool waited = false;
  if (!g.early_prefetch) {
    pdl_wait();
    waited = true;
  }
  while (s < s1) {
    const int tile = s / spt;
    const int ks = s - tile * spt;
    const int ke = min(spt, ks + (s1 - s));
    const uint16_t* pa;
    const uint16_t* pb;
    bool va = true, vb = true;
    if (swiglu) {
      const int r = tile * 8 + gi;
      pa = (const uint16_t*)g.w[0] + (size_t)r * g.k;
      pb = (const uint16_t*)g.w[1] + (size_t)r * g.k;
    } else {
      const int ra = tile * 16 + gi, rb = ra + 8;
      va = ra < g.n;
      vb = rb < g.n;
      pa = va ? seg_row_bf16(g, ra) : nullptr;
      pb = vb ? seg_row_bf16(g, rb) : nullptr;
    }
    float acc[NG][4];
#pragma unroll
    for (int ng = 0; ng < NG; ++ng)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[ng][e] = 0.f;

    // Rolling prefetch: buffer u holds k-step kk + u; right after its MMAs
    // consume it, it is refilled with step kk + u + U, so every warp keeps U
    // steps (U x 2 KB) of weights in flight for its whole range.
    uint4 wa[U][2], wb[U][2];
    const uint4 zero4 = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int off = (ks + u) * kStepK + ci * 16;
      const bool live = ks + u < ke;
      wa[u][0] = (live && va) ? ld_stream(pa + off) : zero4;
      wa[u][1] = (live && va) ? ld_stream(pa + off + 8) : zero4;
      wb[u][0] = (live && vb) ? ld_stream(pb + off) : zero4;
      wb[u][1] = (live && vb) ? ld_stream(pb + off + 8) : zero4;
    }
    if (!waited) {   // weights are read-only: prefetched before the predecessor finishes
      pdl_wait();
      waited = true;
    }
    for (int kk = ks; kk < ke; kk += U) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int st = kk + u;
        if (st < ke) {
          const int off = st * kStepK + ci * 16;
#pragma unroll
          for (int ng = 0; ng < NG; ++ng) {
            const int tok = ng * 8 + gi;
            uint4 x0 = zero4, x1 = zero4;
            if (tok < g.ntok) {
              const uint4* xp = (const uint4*)(xbase + (size_t)tok * g.ldx + off);
              x0 = __ldg(xp);
              x1 = __ldg(xp + 1);
            }
            mma_bf16_16816(acc[ng], wa[u][0].x, wb[u][0].x, wa[u][0].y, wb[u][0].y, x0.x, x0.y);
            mma_bf16_16816(acc[ng], wa[u][0].z, wb[u][0].z, wa[u][0].w, wb[u][0].w, x0.z, x0.w);
            mma_bf16_16816(acc[ng], wa[u][1].x, wb[u][1].x, wa[u][1].y, wb[u][1].y, x1.x, x1.y);
            mma_bf16_16816(acc[ng], wa[u][1].z, wb[u][1].z, wa[u][1].w, wb[u][1].w, x1.z, x1.w);
          }
          const int nx = st + U;
          if (nx < ke) {
            const int noff = nx * kStepK + ci * 16;
            if (va) {
              wa[u][0] = ld_stream(pa + noff);
              wa[u][1] = ld_stream(pa + noff + 8);
            }
            if (vb) {
              wb[u][0] = ld_stream(pb + noff);
              wb[u][1] = ld_stream(pb + noff + 8);
            }
          }
        }
      }
    }

    if (ks == 0 && ke == spt) {
      gemm_epilogue<NG>(g, tile, acc, gi, ci);
    } else {
      float* mine = partials + (size_t)(gw * 2 + slot) * NG * 32 * 4;
#pragma unroll
      for (int ng = 0; ng < NG; ++ng)
        *reinterpret_cast<float4*>(mine + ((size_t)ng * 32 + lane) * 4) =
            make_float4(acc[ng][0], acc[ng][1], acc[ng][2], acc[ng][3]);
      __threadfence();
      __syncwarp();
      const int wfirst = warp_of_step((long long)tile * spt, total, nw);
      const int wlast = warp_of_step((long long)(tile + 1) * spt - 1, total, nw);
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
              const int sl = (first_step_of_warp(w, total, nw) / spt == tile) ? 0 : 1;
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
        gemm_epilogue<NG>(g, tile, tot, gi, ci);
        if (lane == 0) tickets[tile] = 0;
      }
    }
    slot = 1;
    s += ke - ks;
  }
}

// fp32 models: one warp per output row (per gate/up pair for SwiGLU).
__global__ void __launch_bounds__(256) gemv_f32(const __grid_constant__ GemmDesc g) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= g.n) return;
  const bool swiglu = g.epi == kEpiSwiglu;
  const float* wa = swiglu ? (const float*)g.w[0] + (size_t)row * g.k : seg_row_f32(g, row);
  const float* wb = swiglu ? (const float*)g.w[1] + (size_t)row * g.k : nullptr;
  const float* x = (const float*)g.x;
  for (int t0 = 0; t0 < g.ntok; t0 += 8) {
    float acc[8], accb[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) acc[t] = accb[t] = 0.f;
    for (int kk = lane * 4; kk < g.k; kk += 128) {
      const float4 w = *reinterpret_cast<const float4*>(wa + kk);
      float4 w2 = make_float4(0.f, 0.f, 0.f, 0.f);
      if (swiglu) w2 = *reinterpret_cast<const float4*>(wb + kk);
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        if (t0 + t < g.ntok) {
          const float4 xv = *reinterpret_cast<const float4*>(x + (size_t)(t0 + t) * g.ldx + kk);
          acc[t] += w.x * xv.x + w.y * xv.y + w.z * xv.z + w.w * xv.w;
          if (swiglu) accb[t] += w2.x * xv.x + w2.y * xv.y + w2.z * xv.z + w2.w * xv.w;
        }
      }
    }
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      acc[t] = warp_sum(acc[t]);
      if (swiglu) accb[t] = warp_sum(accb[t]);
    }
    if (lane == 0) {
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int tok = t0 + t;
        if (tok >= g.ntok) break;
        if (swiglu) {
          ((float*)g.out)[(size_t)tok * g.ldo + row] = silu(acc[t]) * accb[t];
        } else if (g.epi == kEpiAdd) {
          ((float*)g.out)[(size_t)tok * g.ldo + row] += acc[t];
        } else {
          ((float*)g.out)[(size_t)tok * g.ldo + row] = acc[t];
        }
      }
    }
  }
}

template <int NG, int U>
static cudaError_t launch_sk(const GemmDesc& g, const GemmScratch& s, int num_sms, cudaStream_t st,
                             bool pdl) {
  const int spt = g.k / kStepK;
  const int tiles = gemm_tiles(g);
  const long long total = (long long)tiles * spt;
  if (total <= 0 || total > 0x7fffffffLL) return cudaErrorInvalidValue;
  (void)pdl;
  return launch_k(gemm_bf16_streamk<NG, U>, dim3(gemm_grid(num_sms)), dim3(256), 0, st, g,
                  s.partials, s.tickets, (int)total, spt);
}

cudaError_t launch_gemm(const GemmDesc& g, int dtype, const GemmScratch& s, int num_sms,
                        cudaStream_t st, bool pdl) {
  if (g.ntok <= 0 || g.ntok > kGemmMaxTok) return cudaErrorInvalidValue;
  if (dtype == 0) {
    const int rows = g.n;
    return launch_k(gemv_f32, dim3((rows + 7) / 8), dim3(256), 0, st, g);
  }
  if (g.k % kStepK != 0) return cudaErrorInvalidValue;
  if (gemm_tiles(g) > s.max_tiles) return cudaErrorInvalidValue;
  const int groups = (g.ntok + 7) / 8;
  if (groups == 1) return launch_sk<1, 4>(g, s, num_sms, st, pdl);
  if (groups == 2) return launch_sk<2, 4>(g, s, num_sms, st, pdl);
  if (groups <= 4) return launch_sk<4, 2>(g, s, num_sms, st, pdl);
  return launch_sk<8, 2>(g, s, num_sms, st, pdl);
}

}  // namespace sv
