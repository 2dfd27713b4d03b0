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
//    needed.  A rolling buffer keeps 4 steps (8 KB) per warp in flight.
//  * A tile split between warps is reduced by its last-arriving warp, in
//    ascending warp order, from a global scratch buffer (arrival counted
//    with one atomic per partial; no waiting).  The split points depend only
//    on (n, k), never on ntok, so each output element is computed with the
//    same operations in the same order for any number of tokens: the pass
//    is batch-invariant (greedy speculative output equals greedy plain
//    decoding bit for bit on the GPU too).
//  * Fusions: the input RMSNorm is applied while loading X (fp32 residual x
//    gain x 1/rms, the 1/rms of each token folded from per-tile sums of
//    squares written by the previous residual update); the residual-add
//    epilogue writes those sums of squares for its 16 rows; the q/k/v
//    epilogue applies RoPE (a tile holds rotation pairs i, i + hd/2) and
//    writes k, v straight into the KV cache.
// fp32 models (tiny workloads): one warp per 16-row tile on CUDA cores, with
// the same row pairing, fusions and fixed reduction orders.
#include "gemm_dev.cuh"

namespace sv {

static bool g_pdl = false;
bool pdl_enabled() { return g_pdl; }
void set_pdl_enabled(bool on) { g_pdl = on; }

int gemm_grid(int num_sms) { return 2 * num_sms; }

size_t gemm_partial_floats(int num_sms) {
  // [warp][2 slots][8 token groups][32 lanes][4]
  return (size_t)gemm_grid(num_sms) * kGemmWarpsPerCta * 2 * 8 * 32 * 4;
}

int gemm_tiles(const GemmDesc& g) { return gemm_tiles_of(g); }

template <int NG, int U, int XM>
__global__ void __launch_bounds__(256, 2)
gemm_bf16_streamk(const __grid_constant__ GemmDesc g, float* __restrict__ partials,
                  int* __restrict__ tickets, int total_steps, int spt) {
  __shared__ float s_inv[kGemmMaxTok];
  extern __shared__ __align__(16) uint16_t s_x[];   // kXSmem: [ntok][k + kXPad] bf16
  pdl_trigger();
  const int gw = blockIdx.x * kGemmWarpsPerCta + (threadIdx.x >> 5);
  const int nwarps = gridDim.x * kGemmWarpsPerCta;
  GemmWarp<U> st;
  if (g.early_prefetch) {   // read-only weights, before the predecessor has finished
    gemm_begin<U>(g, total_steps, spt, gw, nwarps, st);
    pdl_wait();
  } else {
    pdl_wait();
    gemm_begin<U>(g, total_steps, spt, gw, nwarps, st);
  }
  gemm_prepare_x<XM>(g, s_inv, s_x);
  gemm_run<NG, U, XM>(g, st, gw, partials, tickets, s_inv, s_x);
}

// fp32 models: one warp per 16-row tile on CUDA cores.  For each of the 8
// (lo, hi) row pairs and each token the two dot products are lane-strided
// over k with a fixed shuffle tree; the epilogue then sees the same pairs
// (and the same per-tile sums of squares) as the tensor-core kernel.
__global__ void __launch_bounds__(256) gemv_f32(const __grid_constant__ GemmDesc g) {
  __shared__ float s_inv[kGemmMaxTok];
  __shared__ float s_val[8][2][kGemmMaxTok];   // per warp: the current pair's dot products
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (g.x_norm) {
    for (int tok = warp; tok < g.ntok; tok += 8) {
      const float v = warp_inv_rms(g, tok, lane);
      if (lane == 0) s_inv[tok] = v;
    }
  }
  __syncthreads();
  const int tile = blockIdx.x * 8 + warp;
  if (tile >= gemm_tiles_of(g)) return;
  const float* x = (const float*)g.x;
  float tile_ss[2] = {0.f, 0.f};   // tokens lane and lane + 32
  for (int gi = 0; gi < 8; ++gi) {
    const float* wa;
    const float* wb;
    if (g.epi == kEpiSwiglu) {
      wa = (const float*)g.w[0] + (size_t)(tile * 8 + gi) * g.k;
      wb = (const float*)g.w[1] + (size_t)(tile * 8 + gi) * g.k;
    } else {
      int lo, hi;
      tile_rows(g, tile, gi, &lo, &hi);
      wa = lo >= 0 ? seg_row<float>(g, lo) : nullptr;
      wb = hi >= 0 ? seg_row<float>(g, hi) : nullptr;
    }
    for (int t0 = 0; t0 < g.ntok; t0 += 8) {
      float aa[8], ab[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) aa[t] = ab[t] = 0.f;
      for (int kk = lane * 4; kk < g.k; kk += 128) {
        const float4 zf = make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 w1 = wa ? *reinterpret_cast<const float4*>(wa + kk) : zf;
        const float4 w2 = wb ? *reinterpret_cast<const float4*>(wb + kk) : zf;
        float4 gv = make_float4(1.f, 1.f, 1.f, 1.f);
        if (g.x_norm) gv = *reinterpret_cast<const float4*>(g.gain + kk);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int tok = t0 + t;
          if (tok < g.ntok) {
            float4 xv = *reinterpret_cast<const float4*>(x + (size_t)tok * g.ldx + kk);
            if (g.x_norm) {
              const float iv = s_inv[tok];
              xv = make_float4(xv.x * iv * gv.x, xv.y * iv * gv.y, xv.z * iv * gv.z, xv.w * iv * gv.w);
            }
            aa[t] += w1.x * xv.x + w1.y * xv.y + w1.z * xv.z + w1.w * xv.w;
            ab[t] += w2.x * xv.x + w2.y * xv.y + w2.z * xv.z + w2.w * xv.w;
          }
        }
      }
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        aa[t] = warp_sum(aa[t]);
        ab[t] = warp_sum(ab[t]);
      }
      if (lane == 0) {
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          if (t0 + t < g.ntok) {
            s_val[warp][0][t0 + t] = aa[t];
            s_val[warp][1][t0 + t] = ab[t];
          }
        }
      }
    }
    __syncwarp();
    // epilogue of pair gi for tokens lane and lane + 32
    for (int q = 0; q < 2; ++q) {
      const int tok = lane + 32 * q;
      if (tok >= g.ntok) continue;
      const float v1 = s_val[warp][0][tok], v2 = s_val[warp][1][tok];
      if (g.epi == kEpiSwiglu) {
        ((float*)g.out)[(size_t)tok * g.ldo + tile * 8 + gi] = silu(v1) * v2;
      } else if (g.epi == kEpiHeadRes) {
        int lo, hi;
        tile_rows(g, tile, gi, &lo, &hi);
        const float* u = g.hres + (size_t)tok * g.k;
        float* o = (float*)g.out + (size_t)tok * g.ldo;
        if (lo >= 0) o[lo] = u[lo % g.k] + silu(v1);
        if (hi >= 0) o[hi] = u[hi % g.k] + silu(v2);
      } else if (g.epi == kEpiQkvRope) {
        const int per = g.hd / 16, half = g.hd / 2;
        const int h = tile / per, i = 8 * (tile % per) + gi;
        const int pos = *g.pos_base + g.pos_off + tok;
        if (h >= g.hq + g.hkv) {
          float* dst = (float*)g.vc + ((size_t)(h - g.hq - g.hkv) * g.cap + pos) * g.hd;
          dst[i] = v1;
          dst[i + half] = v2;
        } else {
          const float c = g.rope_cos[(size_t)pos * half + i], sn = g.rope_sin[(size_t)pos * half + i];
          const float y1 = v1 * c - v2 * sn, y2 = v2 * c + v1 * sn;
          if (h < g.hq) {
            float* dq = g.q_out + ((size_t)tok * g.hq + h) * g.hd;
            dq[i] = y1;
            dq[i + half] = y2;
          } else {
            float* dst = (float*)g.kc + ((size_t)(h - g.hq) * g.cap + pos) * g.hd;
            dst[i] = y1;
            dst[i + half] = y2;
          }
        }
      } else {
        int lo, hi;
        tile_rows(g, tile, gi, &lo, &hi);
        float* o = (float*)g.out + (size_t)tok * g.ldo;
        if (g.epi == kEpiAdd) {
          if (lo >= 0) { const float v = o[lo] + v1; o[lo] = v; tile_ss[q] += v * v; }
          if (hi >= 0) { const float v = o[hi] + v2; o[hi] = v; tile_ss[q] += v * v; }
        } else {
          if (lo >= 0) o[lo] = v1;
          if (hi >= 0) o[hi] = v2;
        }
      }
    }
    __syncwarp();
  }
  if (g.epi == kEpiAdd && g.ss_out) {
    for (int q = 0; q < 2; ++q) {
      const int tok = lane + 32 * q;
      if (tok < g.ntok) g.ss_out[(size_t)tile * g.ss_ld + tok] = tile_ss[q];
    }
  }
}

constexpr size_t kXSmemMax = 80 * 1024;

size_t gemm_xsmem_bytes(const GemmDesc& g) { return (size_t)g.ntok * (g.k + kXPad) * 2; }

template <int NG, int U, int XM>
static cudaError_t launch_sk(const GemmDesc& g, const GemmScratch& s, int num_sms, cudaStream_t st) {
  const int spt = g.k / kStepK;
  const int tiles = gemm_tiles(g);
  const long long total = (long long)tiles * spt;
  if (total <= 0 || total > 0x7fffffffLL) return cudaErrorInvalidValue;
  const size_t smem = XM == kXSmem ? gemm_xsmem_bytes(g) : 0;
  return launch_k(gemm_bf16_streamk<NG, U, XM>, dim3(gemm_grid(num_sms)), dim3(256), smem, st, g,
                  s.partials, s.tickets, (int)total, spt);
}

template <int NG, int U>
static cudaError_t launch_sk_x(const GemmDesc& g, const GemmScratch& s, int num_sms, cudaStream_t st) {
  if (g.x_norm != 1) return launch_sk<NG, U, kXGlobal>(g, s, num_sms, st);   // bf16 X (x_norm = 2: x * gain)
  if (NG == 1 && gemm_xsmem_bytes(g) <= kXSmemMax) return launch_sk<NG, U, kXSmem>(g, s, num_sms, st);
  return launch_sk<NG, U, kXInline>(g, s, num_sms, st);
}

cudaError_t configure_gemm() {
  return cudaFuncSetAttribute(gemm_bf16_streamk<1, 4, kXSmem>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kXSmemMax);
}

cudaError_t launch_gemm(const GemmDesc& g, int dtype, const GemmScratch& s, int num_sms,
                        cudaStream_t st, bool pdl) {
  (void)pdl;
  if (g.ntok <= 0 || g.ntok > kGemmMaxTok) return cudaErrorInvalidValue;
  if (g.epi == kEpiQkvRope && (g.hd % 16 != 0 || g.n != (g.hq + 2 * g.hkv) * g.hd))
    return cudaErrorInvalidValue;
  if (g.x_norm && g.k % 16 != 0) return cudaErrorInvalidValue;
  if (g.epi == kEpiQkvRope && g.spt > 0 && (g.ntok % g.spt != 0 || (dtype == 0 && g.spt != g.ntok)))
    return cudaErrorInvalidValue;   // whole sequences; fp32 models: one sequence per pass
  if (dtype == 0) {
    if (g.k % 4 != 0) return cudaErrorInvalidValue;
    return launch_k(gemv_f32, dim3((gemm_tiles(g) + 7) / 8), dim3(256), 0, st, g);
  }
  if (g.k % kStepK != 0) return cudaErrorInvalidValue;
  if (gemm_tiles(g) > s.max_tiles) return cudaErrorInvalidValue;
  const int groups = (g.ntok + 7) / 8;
  if (groups == 1) return launch_sk_x<1, 4>(g, s, num_sms, st);
  if (groups == 2) return launch_sk_x<2, 4>(g, s, num_sms, st);
  if (groups <= 4) return launch_sk_x<4, 2>(g, s, num_sms, st);
  return launch_sk_x<8, 2>(g, s, num_sms, st);
}

}  // namespace sv
