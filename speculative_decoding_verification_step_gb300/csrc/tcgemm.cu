// Tensor-core GEMM on the fifth-generation tensor cores for passes of many
// tokens (a batch of sequences' K+1 verify positions): Y = X . W^T with the
// weights W [n][k] bf16 (the q/k/v segments, or the gate/up pair) and
// X [ntok][k] bf16, 16 < ntok <= 512, fp32 accumulation in tensor memory.
//
// Work unit = (row tile, k split).  A row tile is 128 output rows (gate/up:
// 64 gate rows then the same 64 up rows); the k range of the GEMM is cut into
// `splits` contiguous runs of 64-element blocks, fixed by n, k and the grid
// (not by ntok); a unit walks its run from a tile-dependent block so that the
// CTAs read different blocks of X at a time.  Persistent: one CTA per SM
// takes units blockIdx.x, blockIdx.x + gridDim.x, ...
//   warp 0, lane 0   producer: tensor copies of each 64-k block of a unit's
//                    weight rows (128 x 128 B) and of X (npad x 128 B) into
//                    one ring of stages running across the CTA's units,
//                    128-byte swizzled;
//   warp 1, lane 0   MMA issuer: four 128 x npad x 16 tcgen05.mma per stage
//                    (A = weights, B = X, both K-major) into one of two
//                    tensor-memory accumulators (unit i: buffer i mod 2);
//                    tcgen05.commit frees the stage, a last commit per unit
//                    signals its accumulator complete.  Past 256 tokens (the
//                    largest MMA N) every 16-k slice is two MMAs, one per
//                    half of the tokens, on the same weight tile, and the
//                    npad columns leave room for one accumulator only: a
//                    unit's MMAs then wait for the previous unit's readout,
//                    but the weights are still read once per pass;
//   warps 2..5       read a finished accumulator (one TMEM lane quarter each)
//                    while the next unit accumulates in the other buffer --
//                    into the unit's fp32 partial [128][npad], or through the
//                    fused epilogue below -- then free it;
//   warp 6           allocates and frees the tensor-memory columns.
// The epilogue (store / residual add with the next norm's sums of squares and
// x * gain / SwiGLU / RoPE + KV append, after scaling by 1/rms of the token:
// normalised inputs arrive as x * gain in bf16, as in the skinny GEMM) runs
//  * fused, when the tiles are not split in k (the LM heads, GEMMs with at
//    least about a wave of tiles): warps 2..5 move each finished accumulator,
//    32 tokens at a time, through a shared-memory tile into the epilogue;
//  * else in a second kernel, one CTA per (tile, 32-token block), that sums
//    the tile's partials in split order first, so that reductions and
//    epilogues are spread over the whole GPU.
// A normalised input's 1/rms per token is folded once per GEMM by a first
// small kernel (tc_rms_kernel).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "gemm_dev.cuh"
#include "kernels.h"

namespace sv {

namespace {

constexpr int kTcM = 128;           // weight rows per tile (MMA M)
constexpr int kTcKb = 64;           // k elements per stage (one 128-byte swizzle row)
constexpr int kTcThreads = 256;
constexpr int kTcABytes = kTcM * kTcKb * 2;   // 16 KB
constexpr long long kTcWaitLimit = 1LL << 26;

struct TcArgs {
  TensorMap128 wmap[3];   // weight segments: boxes of 64 k x 128 rows (gate/up: 64 rows)
  TensorMap128 xmap;      // X [ntok][k]: boxes of 64 k x npad rows
  GemmDesc g;
  int npad, tiles, splits, nkb, stages, tmem_cols;
  int halves;             // token halves per stage (npad > 256: 2, MMA N = npad / 2)
  int nbuf;               // tensor-memory accumulators (2, or 1 when two do not fit)
  float* partials;        // [tiles * splits][128][npad] (unfused)
  float* inv;             // [ntok] 1/rms of a normalised input's tokens
  int fused;              // 1: epilogue from tensor memory (splits == 1)
  int* err;
};

// ---- tcgen05 / descriptor helpers ----
// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart; start address in 16-byte units (advanced by 2 per 16-k
// slice inside the 128-byte row).
SV_DEV uint64_t smem_desc_sw128(const void* p) {
  const uint64_t a = (smem_u32(p) >> 4) & 0x3FFFu;
  return a | (1ull << 16) | (64ull << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, M = 128, N = n.
SV_DEV uint32_t idesc_bf16(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kTcM >> 4) << 24);
}
SV_DEV void tc_mma(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
      ::"r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
}
SV_DEV void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(smem_u32(bar)) : "memory");
}
SV_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
SV_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// 16 consecutive 32-bit columns of this thread's TMEM lane.
SV_DEV void tc_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Bounded wait; false (after raising the abort flag) on timeout.
SV_DEV bool tc_wait(uint64_t* bar, unsigned parity, volatile int* abort) {
  long long spins = 0;
  while (!mbar_test(bar, parity)) {
    if (*abort || ++spins > kTcWaitLimit) {
      *abort = 1;
      return false;
    }
  }
  return true;
}

// Weight row of tile-local row r of tile `tile`, as (segment, row in segment).
SV_DEV void tc_tile_src(const GemmDesc& g, int tile, int r, int* seg, int* row) {
  if (g.epi == kEpiSwiglu) {   // rows 0..63: gate rows, 64..127: the same up rows
    *seg = r < 64 ? 0 : 1;
    *row = tile * 64 + (r & 63);
    return;
  }
  int R = tile * kTcM + r, s = 0;
  while (s < 2 && g.seg_rows[s] > 0 && R >= g.seg_rows[s]) R -= g.seg_rows[s++];
  *seg = s;
  *row = R;
}

// Epilogue of tile `tile` for tokens t0 .. t0 + nt - 1: Y[(t - t0) * ld + r]
// holds the finished sum of tile row r for token t (scaled by 1/rms for
// normalised inputs).  Elements are spread over threads tid = 0 .. nth - 1,
// consecutive threads on consecutive rows of one token (coalesced global
// accesses), kEb elements per thread in flight where global loads are needed.
SV_DEV void tc_epilogue(const GemmDesc& g, int tile, const float* Y, int ld, int t0, int nt, int tid, int nth) {
  constexpr int kEb = 8;
  if (g.epi == kEpiSwiglu) {
    const int total = nt * 64;   // (token, ffn index of the tile)
    for (int e = tid; e < total; e += nth) {
      const int tl = e / 64, t = t0 + tl, j = e % 64, f = tile * 64 + j;
      if (f < g.n)
        ((bf16*)g.out)[(size_t)t * g.ldo + f] =
            __float2bfloat16_rn(silu(Y[tl * ld + j]) * Y[tl * ld + 64 + j]);
    }
  } else if (g.epi == kEpiQkvRope) {
    const int half = g.hd / 2;
    const int pos0 = g.spt > 0 ? 0 : *g.pos_base + g.pos_off;
    const int total = nt * (kTcM / 2);   // (token, rotation pair of the tile)
    for (int e0 = tid; e0 < total; e0 += kEb * nth) {
      float cs[kEb], sn[kEb];
      int pos[kEb];
#pragma unroll
      for (int u = 0; u < kEb; ++u) {   // positions and rotations first: kEb loads in flight
        const int e = e0 + u * nth;
        cs[u] = 1.f; sn[u] = 0.f; pos[u] = 0;
        if (e >= total) continue;
        const int t = t0 + e / (kTcM / 2), pr = e % (kTcM / 2), i = pr % half;
        pos[u] = tok_pos(g, t, pos0);
        const int h = (tile * kTcM) / g.hd + pr / half;
        if (h < g.hq + g.hkv) {
          cs[u] = __ldg(g.rope_cos + (size_t)pos[u] * half + i);
          sn[u] = __ldg(g.rope_sin + (size_t)pos[u] * half + i);
        }
      }
#pragma unroll
      for (int u = 0; u < kEb; ++u) {
        const int e = e0 + u * nth;
        if (e >= total) continue;
        const int tl = e / (kTcM / 2), t = t0 + tl, pr = e % (kTcM / 2);
        const int hl = pr / half, i = pr % half;
        const int h = (tile * kTcM) / g.hd + hl;          // head of the fused q/k/v rows
        if (h >= g.hq + 2 * g.hkv) continue;
        const float x1 = Y[tl * ld + hl * g.hd + i], x2 = Y[tl * ld + hl * g.hd + i + half];
        const size_t kv0 = tok_kv_row0(g, t);
        if (h >= g.hq + g.hkv) {   // value head: stored as is
          bf16* dst = (bf16*)g.vc + (kv0 + (size_t)(h - g.hq - g.hkv) * g.cap + pos[u]) * g.hd;
          dst[i] = __float2bfloat16_rn(x1);
          dst[i + half] = __float2bfloat16_rn(x2);
          continue;
        }
        const float y1 = x1 * cs[u] - x2 * sn[u], y2 = x2 * cs[u] + x1 * sn[u];
        if (h < g.hq) {
          float* dq = g.q_out + ((size_t)t * g.hq + h) * g.hd;
          dq[i] = y1;
          dq[i + half] = y2;
        } else {
          bf16* dst = (bf16*)g.kc + (kv0 + (size_t)(h - g.hq) * g.cap + pos[u]) * g.hd;
          dst[i] = __float2bfloat16_rn(y1);
          dst[i + half] = __float2bfloat16_rn(y2);
        }
      }
    }
  } else if (g.epi == kEpiStore) {
    const int total = nt * kTcM;   // (token, row of the tile)
    for (int e = tid; e < total; e += nth) {
      const int tl = e / kTcM, t = t0 + tl, r = e % kTcM, R = tile * kTcM + r;
      if (R < g.n) ((float*)g.out)[(size_t)t * g.ldo + R] = Y[tl * ld + r];
    }
  } else {
    // residual add; a warp holds 32 consecutive rows of one token, i.e. two
    // 16-row tiles of the next norm's sums of squares
    const int total = nt * kTcM;
    for (int e0 = tid; e0 < total; e0 += kEb * nth) {
      float ov[kEb];
#pragma unroll
      for (int u = 0; u < kEb; ++u) {   // residual loads first: kEb in flight
        const int e = e0 + u * nth;
        const int t = t0 + e / kTcM, R = tile * kTcM + e % kTcM;
        ov[u] = (e < total && R < g.n) ? __ldcg((const float*)g.out + (size_t)t * g.ldo + R) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kEb; ++u) {
        const int e = e0 + u * nth;
        if (e >= total) break;   // uniform across the warp (totals are multiples of 32)
        const int tl = e / kTcM, t = t0 + tl, r = e % kTcM, R = tile * kTcM + r;
        const bool in = R < g.n;
        const float v = ov[u] + Y[tl * ld + r];
        if (in) {
          ((float*)g.out)[(size_t)t * g.ldo + R] = v;
          if (g.xg_out) ((bf16*)g.xg_out)[(size_t)t * g.ldo + R] = __float2bfloat16_rn(v * __ldg(g.gain_next + R));
        }
        float ss = in ? v * v : 0.f;
        ss += __shfl_xor_sync(0xffffffffu, ss, 8);
        ss += __shfl_xor_sync(0xffffffffu, ss, 4);
        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        if (g.ss_out && (tid & 15) == 0 && in) g.ss_out[(size_t)(R / 16) * g.ss_ld + t] = ss;
      }
    }
  }
}

// Epilogue tile of the fused path and of the reduction: [32 tokens][129] fp32
// (odd stride: conflict-free transposed writes).
constexpr int kTcRedTok = 32;
constexpr int kTcRedLd = kTcM + 1;
constexpr int kTcYBytes = kTcRedTok * kTcRedLd * 4;
constexpr int kTcEpiBar = 1;   // named barrier of the four readout warps

__global__ void __launch_bounds__(kTcThreads, 1) tc_gemm_kernel(const __grid_constant__ TcArgs a) {
  extern __shared__ __align__(1024) unsigned char tsm[];
  // stage ring barriers; per accumulator buffer: MMAs done, readout done
  __shared__ uint64_t full[8], empty[8], done[2], tfree[2];
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ int s_issued, s_consumed, s_units_done;
  const GemmDesc& g = a.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int units = a.tiles * a.splits;
  // this CTA's units: blockIdx.x, blockIdx.x + gridDim.x, ...
  const int my_n = units > (int)blockIdx.x ? (units - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
  // unit u = (tile, split): its k blocks kb0 .. kb0 + nk - 1, walked from a
  // tile-dependent first block so that the CTAs read different blocks of X
  // at a time (fixed by the grid, not by ntok)
  auto unit_of = [&](int i, int* tile, int* kb0, int* nk, int* rot) {
    const int u = (int)blockIdx.x + i * (int)gridDim.x;
    *tile = u / a.splits;
    const int split = u % a.splits;
    *kb0 = (int)((long long)split * a.nkb / a.splits);
    *nk = (int)((long long)(split + 1) * a.nkb / a.splits) - *kb0;
    *rot = (int)(((long long)*tile * 5) % *nk);
  };
  const int npad = a.npad, nh = a.npad / a.halves, nbuf = a.nbuf;
  const unsigned stage_bytes = (unsigned)(kTcABytes + npad * kTcKb * 2);
  // 1024-aligned stage bases (the swizzle pattern repeats every 1024 bytes)
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(tsm) + 1023) & ~uintptr_t(1023));
  auto stage_a = [&](int s) { return base + (size_t)s * stage_bytes; };
  auto stage_b = [&](int s) { return base + (size_t)s * stage_bytes + kTcABytes; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&done[b], 1);
      mbar_init(&tfree[b], 4);   // one arrival per readout warp
    }
    s_abort = 0;
    s_issued = s_consumed = s_units_done = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 6) {   // tensor-memory columns: two accumulators of npad (one warp allocates and frees)
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(&s_tmem)), "r"(a.tmem_cols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  pdl_trigger();
  pdl_wait();

  if (warp == 0 && lane == 0) {
    // ---- producer: one continuous ring over all of this CTA's units ----
    const uint64_t pol_w = l2_evict_first(), pol_x = l2_evict_last();
    int q = 0;   // stage fills issued
    for (int i = 0; i < my_n && !s_abort; ++i) {
      int tile, kb0, nk, rot;
      unit_of(i, &tile, &kb0, &nk, &rot);
      int seg = 0, row = 0;
      if (g.epi != kEpiSwiglu) tc_tile_src(g, tile, 0, &seg, &row);
      for (int j = 0; j < nk; ++j, ++q) {
        const int s = q % a.stages;
        if (q >= a.stages && !tc_wait(&empty[s], (unsigned)((q / a.stages - 1) & 1), &s_abort)) break;
        const int kb = kb0 + (j + rot) % nk;
        mbar_arrive_expect_tx(&full[s], stage_bytes);
        if (g.epi == kEpiSwiglu) {
          tma_load_2d_hint(stage_a(s), &a.wmap[0], kb * kTcKb, tile * 64, &full[s], pol_w);
          tma_load_2d_hint(stage_a(s) + kTcABytes / 2, &a.wmap[1], kb * kTcKb, tile * 64, &full[s], pol_w);
        } else {
          tma_load_2d_hint(stage_a(s), &a.wmap[seg], kb * kTcKb, row, &full[s], pol_w);
        }
        for (int h = 0; h < a.halves; ++h)   // one box per token half (a box holds at most 256 rows)
          tma_load_2d_hint(stage_b(s) + (size_t)h * nh * (kTcKb * 2), &a.xmap, kb * kTcKb, h * nh, &full[s], pol_x);
        s_issued = q + 1;
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer: unit i accumulates into buffer i mod nbuf ----
    const uint32_t idesc = idesc_bf16(nh);
    int q = 0;   // stage fills consumed
    for (int i = 0; i < my_n && !s_abort; ++i) {
      int tile, kb0, nk, rot;
      unit_of(i, &tile, &kb0, &nk, &rot);
      const int bi = i % nbuf;
      // the readout of unit i - nbuf has emptied this buffer
      if (i >= nbuf && !tc_wait(&tfree[bi], (unsigned)((i / nbuf - 1) & 1), &s_abort)) break;
      tc_fence_after();
      const uint32_t acc = tmem + (uint32_t)(bi * npad);
      bool ok = true;
      for (int j = 0; j < nk; ++j, ++q) {
        const int s = q % a.stages;
        if (!tc_wait(&full[s], (unsigned)((q / a.stages) & 1), &s_abort)) {
          ok = false;
          break;
        }
        s_consumed = q + 1;
        tc_fence_after();
        const uint64_t ad = smem_desc_sw128(stage_a(s));
        for (int h = 0; h < a.halves; ++h) {   // token half h: columns h * nh .. of the accumulator
          const uint64_t bd = smem_desc_sw128(stage_b(s) + (size_t)h * nh * (kTcKb * 2));
#pragma unroll
          for (int kk = 0; kk < kTcKb / 16; ++kk)   // 16-k slices: +32 bytes = +2 in the start field
            tc_mma(acc + (uint32_t)(h * nh), ad + 2 * kk, bd + 2 * kk, idesc, (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&empty[s]);
      }
      tc_commit(&done[bi]);   // completes when every MMA issued above has
      if (!ok) break;
    }
  } else if (warp >= 2 && warp <= 5 && !a.fused) {
    // ---- accumulator -> partial [128][npad] of unit blockIdx.x + i gridDim.x ----
    const int q = warp & 3;                       // TMEM lane quarter of this warp
    const int r = q * 32 + lane;                  // tile row
    for (int i = 0; i < my_n; ++i) {
      const int bi = i % nbuf;
      if (!tc_wait(&done[bi], (unsigned)((i / nbuf) & 1), &s_abort)) break;
      tc_fence_after();
      const int u = (int)blockIdx.x + i * (int)gridDim.x;
      float* part = a.partials + ((size_t)u * kTcM + r) * npad;
      const uint32_t acc = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(bi * npad);
      for (int c = 0; c < npad; c += 16) {
        float v[16];
        tc_ld16(acc + (uint32_t)c, v);
#pragma unroll
        for (int e = 0; e < 16; e += 4)
          *reinterpret_cast<float4*>(part + c + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tfree[bi]);
      if (threadIdx.x == 64) s_units_done = i + 1;
    }
  } else if (warp >= 2 && warp <= 5) {
    // ---- fused: accumulator -> epilogue, 32 tokens at a time (unit = tile) ----
    // Every readout warp runs the same units and blocks and meets both
    // barriers of every block, also after an abort (it then skips the work).
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int tid = (int)threadIdx.x - 64;        // 0..127 over the four warps
    float* Y = reinterpret_cast<float*>(base + (size_t)a.stages * stage_bytes);
    for (int i = 0; i < my_n; ++i) {
      const int bi = i % nbuf;
      const bool ok = tc_wait(&done[bi], (unsigned)((i / nbuf) & 1), &s_abort);
      tc_fence_after();
      const int tile = (int)blockIdx.x + i * (int)gridDim.x;
      const uint32_t acc = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(bi * npad);
      for (int t0 = 0; t0 < g.ntok; t0 += kTcRedTok) {
        const int nt = min(kTcRedTok, g.ntok - t0);
        if (ok) {
#pragma unroll
          for (int c = 0; c < kTcRedTok; c += 16) {
            if (t0 + c >= npad) break;   // npad is a multiple of 16: no column past the buffer is read
            float v[16];
            tc_ld16(acc + (uint32_t)(t0 + c), v);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int tl = c + e;
              if (tl < nt) {
                float y = 0.f;   // the reduction's arithmetic for one split
                y += v[e];
                Y[tl * kTcRedLd + r] = g.x_norm == 2 ? y * a.inv[t0 + tl] : y;
              }
            }
          }
        }
        named_sync(kTcEpiBar, 128);
        if (ok) tc_epilogue(g, tile, Y, kTcRedLd, t0, nt, tid, 128);
        named_sync(kTcEpiBar, 128);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tfree[bi]);
      if (ok && threadIdx.x == 64) s_units_done = i + 1;
    }
  }
  __syncthreads();
  if (s_abort && threadIdx.x == 0) {
    // a wait gave up: let the copies issued but not consumed land and the
    // MMAs issued finish (bounded), before the space and the columns go
    atomicExch(a.err, 1);
    for (int q = s_consumed; q < s_issued; ++q) {
      long long spins = 0;
      while (!mbar_test(&full[q % a.stages], (unsigned)((q / a.stages) & 1)) && ++spins < (1LL << 20)) {
      }
    }
    for (int i = s_units_done; i < my_n && i < s_units_done + nbuf; ++i) {
      long long spins = 0;
      while (!mbar_test(&done[i % nbuf], (unsigned)((i / nbuf) & 1)) && ++spins < (1LL << 20)) {
      }
    }
  }
  __syncthreads();
  if (warp == 6) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(a.tmem_cols) : "memory");
  }
}

// 1/rms of every token of a normalised input, once per GEMM: 8 threads per
// token sum its k/16 per-tile sums of squares (tiles strided by 8, then a
// shuffle sum in the group of 8).
__global__ void __launch_bounds__(kTcThreads) tc_rms_kernel(const __grid_constant__ TcArgs a) {
  const GemmDesc& g = a.g;
  pdl_trigger();
  pdl_wait();
  const int tl = threadIdx.x / 8, sub = threadIdx.x % 8, nkt = g.k / 16;
  const int t = (int)blockIdx.x * kTcRedTok + tl;
  float sum = 0.f;
  if (t < g.ntok)
    for (int i = sub; i < nkt; i += 8) sum += __ldcg(g.ss_in + (size_t)i * g.ss_ld + t);
  sum += __shfl_xor_sync(0xffffffffu, sum, 4);
  sum += __shfl_xor_sync(0xffffffffu, sum, 2);
  sum += __shfl_xor_sync(0xffffffffu, sum, 1);
  if (sub == 0 && t < g.ntok) a.inv[t] = 1.0f / sqrtf(sum / (float)g.k + g.eps);
}

// Reduction and epilogue of a split GEMM: one CTA per (row tile, block of
// kTcRedTok tokens) sums the splits' partials in split order (x 1/rms) and
// runs the epilogue for those tokens.
__global__ void __launch_bounds__(kTcThreads) tc_reduce_kernel(const __grid_constant__ TcArgs a) {
  __shared__ float Y[kTcRedTok * kTcRedLd];
  __shared__ float s_inv[kTcRedTok];
  const GemmDesc& g = a.g;
  const int tile = blockIdx.x, t0 = blockIdx.y * kTcRedTok;
  const int nt = min(kTcRedTok, g.ntok - t0), npad = a.npad;
  pdl_trigger();
  pdl_wait();
  if (g.x_norm == 2 && threadIdx.x < nt) s_inv[threadIdx.x] = __ldcg(a.inv + t0 + threadIdx.x);
  __syncthreads();
  const float* P = a.partials + (size_t)tile * a.splits * kTcM * npad + t0;
  // 4 elements per thread at a time, their partial loads in flight together;
  // each element's splits are added in split order
  constexpr int kRb = 4;
  for (int e0 = threadIdx.x; e0 < kTcM * kTcRedTok; e0 += kRb * kTcThreads) {
    float acc[kRb];
#pragma unroll
    for (int u = 0; u < kRb; ++u) acc[u] = 0.f;
#pragma unroll 2
    for (int sp = 0; sp < a.splits; ++sp) {
      float v[kRb];
#pragma unroll
      for (int u = 0; u < kRb; ++u) {
        const int e = e0 + u * kTcThreads, r = e / kTcRedTok, tl = e % kTcRedTok;
        v[u] = tl < nt ? __ldcg(P + ((size_t)sp * kTcM + r) * npad + tl) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kRb; ++u) acc[u] += v[u];
    }
#pragma unroll
    for (int u = 0; u < kRb; ++u) {
      const int e = e0 + u * kTcThreads, r = e / kTcRedTok, tl = e % kTcRedTok;
      if (tl < nt) Y[tl * kTcRedLd + r] = g.x_norm == 2 ? acc[u] * s_inv[tl] : acc[u];
    }
  }
  __syncthreads();
  tc_epilogue(g, tile, Y, kTcRedLd, t0, nt, threadIdx.x, kTcThreads);
}

}  // namespace

// ---- host side ----
static PFN_cuTensorMapEncodeTiled_v12000 tc_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess || q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// Row-major bf16 matrix [rows][k], row stride ld elements, boxes of 64 k x
// box_rows with the 128-byte swizzle; rows past the end read as zero.
static bool tc_encode_rows(TensorMap128& m, const void* base, int k, long long rows, long long ld, int box_rows) {
  static_assert(sizeof(CUtensorMap) == sizeof(TensorMap128), "tensor map size");
  PFN_cuTensorMapEncodeTiled_v12000 enc = tc_encoder();
  if (!enc || !base || rows < 1 || box_rows < 1 || box_rows > 256 || (reinterpret_cast<uintptr_t>(base) & 15u) ||
      (ld * 2) % 16 != 0)
    return false;
  cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)kTcKb, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(reinterpret_cast<CUtensorMap*>(&m), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
             dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t tc_gemm_partial_floats(int num_sms, int max_n) {
  // every work unit writes one [128][npad] partial: the LM head's tiles (one
  // split), or up to eight splits of fewer tiles
  return std::max<size_t>((size_t)(max_n + kTcM - 1) / kTcM, 8 * (size_t)num_sms) * kTcM * kTcMaxTok;
}

bool tc_gemm_supported(const GemmDesc& g) {
  if (g.ntok <= kTcMinTok || g.ntok > kTcMaxTok || g.k % kTcKb != 0 || g.ldx % 8 != 0) return false;
  if (g.x_norm == 1) return false;   // normalised inputs arrive as x * gain in bf16
  if (g.x_norm == 2 && ((reinterpret_cast<uintptr_t>(g.ss_in) & 15u) || g.ss_ld % 4 != 0 || g.ss_ld < kTcMaxTok))
    return false;                    // 1/rms reads float4 columns of up to kTcMaxTok tokens
  if (g.epi == kEpiSwiglu) return g.n % 64 == 0;
  for (int s = 0; s < 3; ++s)
    if (g.seg_rows[s] > 0 && g.seg_rows[s] % kTcM != 0 && !(s == 0 && g.seg_rows[1] == 0)) return false;
  if (g.epi == kEpiQkvRope) return g.hd % 2 == 0 && kTcM % g.hd == 0 && g.n % kTcM == 0;
  return true;
}

cudaError_t launch_tc_gemm(const GemmDesc& g, float* partials, float* inv, int* err, int num_sms,
                           long long max_units, cudaStream_t st) {
  if (!tc_gemm_supported(g)) return cudaErrorInvalidValue;
  TcArgs a{};
  a.g = g;
  // tokens padded to 16 (one MMA N), past 256 to 32 (two MMAs of N = npad / 2)
  a.npad = g.ntok <= 256 ? (g.ntok + 15) / 16 * 16 : (g.ntok + 31) / 32 * 32;
  a.halves = a.npad > 256 ? 2 : 1;
  a.nkb = g.k / kTcKb;
  a.tiles = g.epi == kEpiSwiglu ? g.n / 64 : (g.n + kTcM - 1) / kTcM;
  // splits (at most 8, at least two k blocks each): the least modelled time
  // -- rounds of units per CTA times the k blocks of a unit, each block a
  // stage of weights and X at ~50 GB/s per SM, plus for split tiles the
  // partials written and read again (~50 GB/s per SM) and the reduction's
  // launch -- fewest splits on ties, within the partials.  The model is
  // evaluated at a fixed 256-token width, so that the split, and with it the
  // order in which a tile's k range is summed, depends on n, k and the grid
  // only, never on the pass's token count.
  constexpr int kModelTok = 256;
  const double kb_us = (double)(kTcABytes + kModelTok * kTcKb * 2) / 50e3;
  a.splits = 1;
  double best = -1.0;
  for (int sp = 1; sp <= std::max(1, std::min(8, a.nkb / 2)); ++sp) {
    const long long units = (long long)a.tiles * sp;
    if (units > max_units) break;
    double cost = (double)((units + num_sms - 1) / num_sms) * ((a.nkb + sp - 1) / sp) * kb_us;
    if (sp > 1) cost += (double)units * kTcM * kModelTok * 8.0 / (50e3 * num_sms) + 5.0;
    if (best < 0 || cost < best) {
      best = cost;
      a.splits = sp;
    }
  }
  a.fused = a.splits == 1 ? 1 : 0;
  const int stage_bytes = kTcABytes + a.npad * kTcKb * 2;
  a.stages = std::min(8, (kTcSmemBytes - 1024 - (a.fused ? kTcYBytes : 0)) / stage_bytes);
  if (a.stages < 2) return cudaErrorInvalidValue;
  // two accumulators of npad columns where they fit the 512 columns, else one
  a.nbuf = 2 * a.npad <= 512 ? 2 : 1;
  int cols = 32;
  while (cols < a.nbuf * a.npad) cols *= 2;
  a.tmem_cols = cols;
  if ((long long)a.tiles * a.splits > max_units) return cudaErrorInvalidValue;
  a.partials = partials;
  a.inv = inv;
  a.err = err;
  if (g.x_norm == 2 && !inv) return cudaErrorInvalidValue;
  const int box_rows = g.epi == kEpiSwiglu ? 64 : kTcM;
  for (int s = 0; s < 3; ++s) {
    if (!g.w[s]) continue;
    const long long rows = g.epi == kEpiSwiglu ? g.n : (g.seg_rows[s] > 0 ? g.seg_rows[s] : g.n);
    if (!tc_encode_rows(a.wmap[s], g.w[s], g.k, rows, g.k, box_rows)) return cudaErrorInvalidValue;
  }
  if (!tc_encode_rows(a.xmap, g.x, g.k, g.ntok, g.ldx, a.npad / a.halves)) return cudaErrorInvalidValue;
  const int grid = std::min(a.tiles * a.splits, num_sms);   // persistent: one CTA per SM
  cudaError_t e = cudaSuccess;
  if (g.x_norm == 2) {
    e = launch_k(tc_rms_kernel, dim3((g.ntok + kTcRedTok - 1) / kTcRedTok), dim3(kTcThreads), 0, st, a);
    if (e != cudaSuccess) return e;
  }
  e = launch_k(tc_gemm_kernel, dim3(grid), dim3(kTcThreads), (size_t)kTcSmemBytes, st, a);
  if (e != cudaSuccess || a.fused) return e;
  return launch_k(tc_reduce_kernel, dim3(a.tiles, (g.ntok + kTcRedTok - 1) / kTcRedTok), dim3(kTcThreads), 0, st, a);
}

cudaError_t configure_tc_gemm() {
  return cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemBytes);
}

}  // namespace sv
