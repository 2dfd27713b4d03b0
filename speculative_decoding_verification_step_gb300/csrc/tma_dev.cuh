// Tensor-copy (TMA) weight streaming of the persistent forward kernel.
//
// A GEMM phase is cut into units of one row group x 256 k.  A row group is
// two boxes of R rows (R = 16 or 32) of the weight matrix, each box one
// 2-D tensor copy of R x 256 bf16 into shared memory:
//   * plain matrices: one box of 2R consecutive rows, MMA tile t = rows
//     16t + g and 16t + 8 + g of the box;
//   * q/k/v with RoPE: rows h*hd + j*R + [0, R) and the rotation partners
//     hd/2 further, MMA tile t = row 8t + g of each box;
//   * SwiGLU: the same R rows of the gate and of the up matrix.
// So an MMA tile is exactly a 16-row tile of the per-kernel path (same
// epilogue, same tile index).  A CTA owns a contiguous range of units (split
// by shape and grid only, never by token count).  One producer thread streams
// the units through a ring of S stages (S x 2R x 512 bytes, S <= 8): per unit
// one or two weight boxes and, in phases whose X comes from global memory,
// one 8-row X box, all completing on the stage's transaction barrier.  In an
// RMSNorm'd phase the producer first copies the X columns the CTA's units
// read -- bf16 rows already multiplied by the norm's gain -- into shared
// memory with bulk copies, and 1/rms scales the finished sums.  The
// warp t < T = R/8 owns MMA tile t of every unit (its four 64-k
// steps, one accumulator chain each, added in step order).  A tile split
// between CTAs is finished by the last-arriving CTA, which adds the CTA
// partials in CTA order; no consumer warp ever waits for another.  Results
// do not depend on timing or on the token count.
//
// Every wait is bounded.  A wait that gives up raises the CTA's abort flag;
// from then on every wait of the CTA returns at once and the warps run
// through their remaining iterations without touching the data (named
// barrier counts stay identical); the kernel reports the failure and leaves
// after waiting, again with a bound, for its copies still in flight.
#pragma once
#include "gemm_dev.cuh"

namespace sv {

constexpr int kTmaK = 256;                        // k per unit (box inner extent)
constexpr int kTmaRowBytes = kTmaK * 2;           // row pitch of a box in shared memory
constexpr int kTmaSteps = kTmaK / kStepK;         // 64-k MMA steps per unit
constexpr int kCWarps = 8;                        // warps of the CTA (attention uses all)
constexpr int kProducerWarp = kCWarps - 1;        // lane 0 issues the tensor copies
constexpr int kPersistThreads = kCWarps * 32;     // 2 warps per SM sub-partition: 255 registers
constexpr int kMaxStages = 8;
constexpr int kXBoxRows = 8;
constexpr int kXStageBytes = kXBoxRows * kTmaRowBytes;
constexpr size_t kRingBytes = 160 * 1024;         // weight ring: 5 stages of 32 KB
constexpr int kMinUnitsPerCta = 2;
constexpr int kMaxMmaTiles = 4;                   // R / 8 for R <= 32
constexpr long long kWaitLimit = 1LL << 22;
constexpr long long kDrainLimit = 1LL << 16;
constexpr int kPersistMaxTok = 8;
constexpr size_t kTensorMapBytes = 128;

struct TmaPipe {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t xfull;               // the bulk X copies of an x_norm = 2 phase
  unsigned fills[kMaxStages];   // fills issued per slot (producer)
  unsigned xfills;              // X loads issued (their barrier's phase count)
  int abort;
};

SV_DEV void tma_init(TmaPipe& tp) {
  if (threadIdx.x == 0) {
    for (int i = 0; i < kMaxStages; ++i) {
      mbar_init(&tp.full[i], 1);
      mbar_init(&tp.empty[i], kMaxMmaTiles);   // released by the tile-owner warps
      tp.fills[i] = 0;
    }
    mbar_init(&tp.xfull, 1);
    tp.xfills = 0;
    tp.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
}

// Wait for the completion of the phase of `parity`; false once the CTA has
// aborted (raising the flag when this wait is the one that gives up).
SV_DEV bool tma_wait(uint64_t* bar, unsigned parity, TmaPipe& tp) {
  volatile int* ab = &tp.abort;
  long long spins = 0;
  while (true) {
    if (*ab) return false;
    if (mbar_test(bar, parity)) return true;
    if (++spins > kWaitLimit) {
      *ab = 1;
      return false;
    }
  }
}

struct TmaRange {
  long long total, nc;
  int u0, u1, kbpt;
};

SV_DEV TmaRange tma_range(const PhaseDesc& d) {
  TmaRange r;
  r.kbpt = (d.g.k + kTmaK - 1) / kTmaK;
  r.total = (long long)d.groups * r.kbpt;
  if (d.whole) {   // whole row groups per CTA, as evenly as groups allow
    r.nc = min((long long)gridDim.x, (long long)d.groups);
    const bool has = blockIdx.x < r.nc;
    r.u0 = has ? (int)first_step_of_warp(blockIdx.x, d.groups, r.nc) * r.kbpt : 0;
    r.u1 = has ? (int)first_step_of_warp(blockIdx.x + 1, d.groups, r.nc) * r.kbpt : 0;
    return r;
  }
  r.nc = max(1LL, min((long long)gridDim.x, r.total / kMinUnitsPerCta));
  const bool has = blockIdx.x < r.nc;
  r.u0 = has ? (int)first_step_of_warp(blockIdx.x, r.total, r.nc) : 0;
  r.u1 = has ? (int)first_step_of_warp(blockIdx.x + 1, r.total, r.nc) : 0;
  return r;
}

// Tensor-map index and first row of box A / box B of row group grp.
struct GroupBoxes {
  int ma, ra, mb, rb;
};
SV_DEV GroupBoxes group_boxes(const PhaseDesc& d, int grp) {
  const GemmDesc& g = d.g;
  const int R = d.R;
  if (g.epi == kEpiQkvRope) {
    const int per = g.hd / (2 * R);
    int row = (grp / per) * g.hd + (grp % per) * R;
    int seg = 0;
    if (row >= g.seg_rows[0]) {
      row -= g.seg_rows[0];
      seg = 1;
      if (row >= g.seg_rows[1]) {
        row -= g.seg_rows[1];
        seg = 2;
      }
    }
    return {seg, row, seg, row + g.hd / 2};
  }
  if (g.epi == kEpiSwiglu) return {0, grp * R, 1, grp * R};
  return {0, grp * 2 * R, 0, 0};   // one box of 2R rows
}
// Index of MMA tile t of group grp among the 16-row tiles of the matrix.
SV_DEV int group_tile(const PhaseDesc& d, int grp, int t) {
  const GemmDesc& g = d.g;
  const int R = d.R;
  if (g.epi == kEpiQkvRope) {
    const int per = g.hd / (2 * R);
    return (grp / per) * (g.hd / 16) + (grp % per) * (R / 8) + t;
  }
  return grp * (R / 8) + t;
}

// x_norm = 2 phase, before its units: the producer thread copies the k-blocks
// of X that the CTA's units read (the whole row once they span a row group,
// else one or two runs of blocks) into the X region with one bulk copy per
// token and run, completing on tp.xfull; every warp meanwhile folds the
// per-tile sums of squares into s_inv[tok] = 1 / rms.  Ends with a CTA barrier.
SV_DEV void tma_prepare_xg(const PhaseDesc& d, TmaPipe& tp, float* s_inv, unsigned char* xreg) {
  const GemmDesc& g = d.g;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp == kProducerWarp && lane == 0) {
    const TmaRange r = tma_range(d);
    const int n = r.u1 - r.u0;
    int run[2][2] = {{0, 0}, {0, 0}}, nrun = 0;   // [kb begin, kb end)
    if (n >= r.kbpt) {
      run[0][0] = 0; run[0][1] = r.kbpt; nrun = 1;
    } else if (n > 0) {
      const int kb0 = r.u0 % r.kbpt, kb1 = (r.u1 - 1) % r.kbpt;
      if (kb0 <= kb1) {
        run[0][0] = kb0; run[0][1] = kb1 + 1; nrun = 1;
      } else {
        run[0][0] = kb0; run[0][1] = r.kbpt; run[1][0] = 0; run[1][1] = kb1 + 1; nrun = 2;
      }
    }
    unsigned bytes = 0;
    for (int q = 0; q < nrun; ++q) bytes += (unsigned)(min(run[q][1] * kTmaK, g.k) - run[q][0] * kTmaK) * 2u;
    mbar_arrive_expect_tx(&tp.xfull, bytes * (unsigned)g.ntok);
    const size_t pitch = (size_t)(g.k + kXPad) * 2;
    for (int t = 0; t < g.ntok; ++t)
      for (int q = 0; q < nrun; ++q) {
        const int c0 = run[q][0] * kTmaK, c1 = min(run[q][1] * kTmaK, g.k);
        bulk_g2s(xreg + t * pitch + (size_t)c0 * 2, (const bf16*)g.x + (size_t)t * g.ldx + c0,
                 (unsigned)(c1 - c0) * 2u, &tp.xfull);
      }
    tp.xfills += 1;
  }
  for (int tok = warp; tok < g.ntok; tok += kPersistThreads / 32) {
    const float v = warp_inv_rms(g, tok, lane);
    if (lane == 0) s_inv[tok] = v;
  }
  __syncthreads();
}

// Producer thread: issue unit i of the CTA's range into slot i mod S --
// wait for the consumers to release the slot, announce the bytes, copy the
// weight boxes and, when with_x, the X box.
SV_DEV void tma_issue(const PhaseDesc& d, const TmaRange& r, int i, bool with_x, TmaPipe& tp,
                      unsigned char* ring, unsigned char* xreg, const unsigned char* maps) {
  const int slot = i % d.stages;
  const unsigned f = tp.fills[slot];
  if (!tma_wait(&tp.empty[slot], (f & 1u) ^ 1u, tp)) return;
  const int u = r.u0 + i;
  const int grp = u / r.kbpt, kb = u - grp * r.kbpt;
  const GroupBoxes b = group_boxes(d, grp);
  const bool xg = d.xm == kXGlobal;
  mbar_arrive_expect_tx(&tp.full[slot], (unsigned)d.stage_bytes + (xg ? (unsigned)kXStageBytes : 0u));
  unsigned char* st = ring + (size_t)slot * d.stage_bytes;
  const int kc = kb * kTmaK;
  const uint64_t pol = l2_evict_first();   // weights are read once per pass
  if (d.paired) {
    tma_load_2d_hint(st, maps + (size_t)d.tm[b.ma] * kTensorMapBytes, kc, b.ra, &tp.full[slot], pol);
    tma_load_2d_hint(st + (size_t)d.R * kTmaRowBytes, maps + (size_t)d.tm[b.mb] * kTensorMapBytes, kc, b.rb,
                     &tp.full[slot], pol);
  } else {
    tma_load_2d_hint(st, maps + (size_t)d.tm[0] * kTensorMapBytes, kc, b.ra, &tp.full[slot], pol);
  }
  if (with_x)
    tma_load_2d(xreg + (size_t)slot * kXStageBytes, maps + (size_t)d.tm[3] * kTensorMapBytes, kc, 0,
                &tp.full[slot]);
  tp.fills[slot] = f + 1;
}

// Producer thread: the X box of an already announced unit.
SV_DEV void tma_issue_x(const PhaseDesc& d, const TmaRange& r, int i, TmaPipe& tp, unsigned char* xreg,
                        const unsigned char* maps) {
  if (tp.abort) return;
  const int slot = i % d.stages;
  const int u = r.u0 + i;
  const int kb = u % r.kbpt;
  tma_load_2d(xreg + (size_t)slot * kXStageBytes, maps + (size_t)d.tm[3] * kTensorMapBytes, kb * kTmaK, 0,
              &tp.full[slot]);
}

// Producer thread, between arriving at the grid barrier that precedes GEMM
// phase d and waiting on it: the weight boxes of its first units (weights
// are read-only; X is not ready yet).  Returns how many units were issued.
SV_DEV int tma_prefetch(const PhaseDesc& d, TmaPipe& tp, unsigned char* ring, unsigned char* xreg,
                        const unsigned char* maps) {
  const TmaRange r = tma_range(d);
  // a phase whose X is bulk-copied after the barrier, with few units per CTA,
  // takes only 3 units ahead, so that fewer weight copies are in flight when
  // its X copies are issued (the 8B q/k/v phase's X arrives ~1 us sooner)
  const int n = r.u1 - r.u0;
  const int npre = min(n, d.xm == kXSmem && n <= 16 ? min(d.stages, 3) : d.stages);
  for (int i = 0; i < npre; ++i) tma_issue(d, r, i, false, tp, ring, xreg, maps);
  return npre;
}

// Producer thread during GEMM phase d: X boxes of the npre prefetched units,
// then every remaining unit.
SV_DEV void tma_produce(const PhaseDesc& d, int npre, TmaPipe& tp, unsigned char* ring, unsigned char* xreg,
                        const unsigned char* maps) {
  const TmaRange r = tma_range(d);
  const int n = r.u1 - r.u0;
  const bool xg = d.xm == kXGlobal;
  fence_proxy_async_global();   // X was written by other CTAs before the grid barrier
  if (xg)
    for (int i = 0; i < npre; ++i) tma_issue_x(d, r, i, tp, xreg, maps);
  for (int i = npre; i < n; ++i) tma_issue(d, r, i, xg, tp, ring, xreg, maps);
}

// Consumer warp t at the end of a row group: finish MMA tile t -- the
// epilogue when this CTA covered every k of the group, else its CTA partial
// and, for the last-arriving CTA of the group, the sum of the CTA partials in
// CTA order and the epilogue.  s_inv (x_norm = 2, else null): 1 / rms per
// token, applied to the finished sums of tokens 2ci, 2ci+1.  The last CTA
// issues the epilogue's own input loads (residual or RoPE factors at token
// 0's position pos0) together with the partial loads.  No other warp takes
// part.
SV_DEV void tma_tile_end(const PhaseDesc& d, const TmaRange& r, int grp, int kbs, int kbe, int pslot,
                         const float (&tot)[1][4], float* __restrict__ partials, int* __restrict__ tickets,
                         const float* s_inv, int pos0) {
  const GemmDesc& g = d.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gi = lane >> 2, ci = lane & 3;
  const int tile = group_tile(d, grp, warp);
  if (tile >= gemm_tiles_of(g)) return;
  const float sc0 = s_inv ? s_inv[2 * ci] : 1.f, sc1 = s_inv ? s_inv[2 * ci + 1] : 1.f;
  if (kbs == 0 && kbe == r.kbpt) {
    const float y[1][4] = {{tot[0][0] * sc0, tot[0][1] * sc1, tot[0][2] * sc0, tot[0][3] * sc1}};
    gemm_epilogue<1, false>(g, tile, y, gi, ci);
    return;
  }
  float* mine = partials + (((size_t)blockIdx.x * 2 + pslot) * kMaxMmaTiles + warp) * 32 * 4;
  *reinterpret_cast<float4*>(mine + (size_t)lane * 4) = make_float4(tot[0][0], tot[0][1], tot[0][2], tot[0][3]);
  __syncwarp();
  const int cfirst = warp_of_step((long long)grp * r.kbpt, r.total, r.nc);
  const int clast = warp_of_step((long long)(grp + 1) * r.kbpt - 1, r.total, r.nc);
  int old = 0;   // the acq_rel ticket publishes this partial and acquires the earlier ones
  if (lane == 0) old = (int)atom_add_acq_rel_gpu(reinterpret_cast<unsigned*>(&tickets[tile]), 1u);
  old = __shfl_sync(0xffffffffu, old, 0);
  if (old != clast - cfirst) return;
  __syncwarp();
  // the epilogue's own inputs are loaded together with the first partials
  EpiIn pre;
  gemm_epi_load<false>(g, tile, pos0, gi, ci, pre);
  float4 pv[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int c = cfirst + q;
    pv[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c <= clast) {
      const int sl = (first_step_of_warp(c, r.total, r.nc) / r.kbpt == grp) ? 0 : 1;
      pv[q] = __ldcg(reinterpret_cast<const float4*>(
          partials + (((size_t)c * 2 + sl) * kMaxMmaTiles + warp) * 32 * 4 + (size_t)lane * 4));
    }
  }
  float sum[1][4] = {{0.f, 0.f, 0.f, 0.f}};   // CTA order
  for (int c = cfirst; c <= clast; ++c) {
    float4 v;
    if (c - cfirst < 2) {
      v = c == cfirst ? pv[0] : pv[1];
    } else {
      const int sl = (first_step_of_warp(c, r.total, r.nc) / r.kbpt == grp) ? 0 : 1;
      v = __ldcg(reinterpret_cast<const float4*>(
          partials + (((size_t)c * 2 + sl) * kMaxMmaTiles + warp) * 32 * 4 + (size_t)lane * 4));
    }
    sum[0][0] += v.x;
    sum[0][1] += v.y;
    sum[0][2] += v.z;
    sum[0][3] += v.w;
  }
  sum[0][0] *= sc0;
  sum[0][1] *= sc1;
  sum[0][2] *= sc0;
  sum[0][3] *= sc1;
  gemm_epilogue<1, false>(g, tile, sum, gi, ci, &pre);
  if (lane == 0) tickets[tile] = 0;
}

// Consumer warps during GEMM phase d.  Warp t < T = R/8 owns MMA tile t of
// every unit and runs its four 64-k steps, each into its own accumulator
// chain (added in step order at the end of the group); warps t >= T only
// keep the ring bookkeeping.  cpar: per-slot parity of the next completion
// of each stage's full barrier (identical in every consumer warp).
// stamp (optional): atomicMax of the globaltimer when the last unit arrived.
template <int XM>
SV_DEV void tma_consume(const PhaseDesc& d, TmaPipe& tp, unsigned& cpar, const unsigned char* ring,
                        const unsigned char* xreg, const float* s_inv, float* __restrict__ partials,
                        int* __restrict__ tickets, unsigned long long* stamp) {
  const GemmDesc& g = d.g;
  const TmaRange r = tma_range(d);
  const int n = r.u1 - r.u0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gi = lane >> 2, ci = lane & 3;
  const int R = d.R, T = R / 8, S = d.stages, sb = d.stage_bytes;
  if (warp >= T) {   // not a tile owner in this phase (the producer warp never gets here)
    for (int i = 0; i < n; ++i) cpar ^= 1u << (i % S);
    return;
  }
  const uint4 zero4 = make_uint4(0, 0, 0, 0);
  const int t = warp;
  const int arow = d.paired ? 8 * t + gi : 16 * t + gi;
  const int brow = d.paired ? R + 8 * t + gi : 16 * t + 8 + gi;
  const bool has_tok = gi < g.ntok;
  const int k = g.k;
  const size_t xs_pitch = (size_t)(k + kXPad) * 2;
  const unsigned arrivals = (unsigned)(kMaxMmaTiles / T);   // the empty barrier expects kMaxMmaTiles
  float acc[kTmaSteps][4];
#pragma unroll
  for (int s = 0; s < kTmaSteps; ++s) acc[s][0] = acc[s][1] = acc[s][2] = acc[s][3] = 0.f;
  int pslot = 0;
  int kbs = n > 0 ? r.u0 % r.kbpt : 0;
  const bool xg = XM == kXSmem && g.x_norm == 2;
  const int pos0 = g.epi == kEpiQkvRope ? __ldcg(g.pos_base) + g.pos_off : 0;
  bool xok = true;
  if (xg && n > 0) xok = tma_wait(&tp.xfull, (tp.xfills - 1) & 1u, tp);   // X copied in

#pragma unroll 1
  for (int i = 0; i < n; ++i) {
    const int slot = i % S;
    const int u = r.u0 + i;
    const int grp = u / r.kbpt, kb = u - grp * r.kbpt;
    const bool ok = tma_wait(&tp.full[slot], (cpar >> slot) & 1u, tp) && xok;
    cpar ^= 1u << slot;
    if (stamp && i == n - 1 && threadIdx.x == 0) {
      unsigned long long tm;
      asm volatile("mov.u64 %0, %globaltimer;" : "=l"(tm));
      atomicMax(stamp, tm);
    }
    if (ok) {
      const unsigned char* st = ring + (size_t)slot * sb + ci * 32;
#pragma unroll
      for (int s = 0; s < kTmaSteps; ++s) {
        const int kg = kb * kTmaK + s * kStepK;
        if (kg < k) {
          const unsigned char* ap = st + arow * kTmaRowBytes + s * (kStepK * 2);
          const unsigned char* bp = st + brow * kTmaRowBytes + s * (kStepK * 2);
          const uint4 a0 = *reinterpret_cast<const uint4*>(ap);
          const uint4 a1 = *reinterpret_cast<const uint4*>(ap + 16);
          const uint4 b0 = *reinterpret_cast<const uint4*>(bp);
          const uint4 b1 = *reinterpret_cast<const uint4*>(bp + 16);
          uint4 x0 = zero4, x1 = zero4;
          if (has_tok) {
            const unsigned char* xp =
                XM == kXSmem ? xreg + gi * xs_pitch + (size_t)(kg + ci * 16) * 2
                             : xreg + (size_t)slot * kXStageBytes + gi * kTmaRowBytes + s * (kStepK * 2) + ci * 32;
            x0 = *reinterpret_cast<const uint4*>(xp);
            x1 = *reinterpret_cast<const uint4*>(xp + 16);
          }
          mma_bf16_16816(acc[s], a0.x, b0.x, a0.y, b0.y, x0.x, x0.y);
          mma_bf16_16816(acc[s], a0.z, b0.z, a0.w, b0.w, x0.z, x0.w);
          mma_bf16_16816(acc[s], a1.x, b1.x, a1.y, b1.y, x1.x, x1.y);
          mma_bf16_16816(acc[s], a1.z, b1.z, a1.w, b1.w, x1.z, x1.w);
        }
      }
    }
    __syncwarp();
    if (lane == 0 && ok) mbar_arrive_count(&tp.empty[slot], arrivals);
    if (kb == r.kbpt - 1 || i == n - 1) {
      float tot[1][4];
#pragma unroll
      for (int e = 0; e < 4; ++e) tot[0][e] = ((acc[0][e] + acc[1][e]) + acc[2][e]) + acc[3][e];
      if (!tp.abort) tma_tile_end(d, r, grp, kbs, kb + 1, pslot, tot, partials, tickets, xg ? s_inv : nullptr, pos0);
#pragma unroll
      for (int s = 0; s < kTmaSteps; ++s) acc[s][0] = acc[s][1] = acc[s][2] = acc[s][3] = 0.f;
      pslot = 1;
      kbs = 0;
    }
  }
}

// After an abort: wait (bounded) for the latest fill of every slot, so that
// no copy lands after the CTA has left.  A fill whose bytes were never all
// issued does not complete; its wait gives up after kDrainLimit probes.
SV_DEV void tma_drain(TmaPipe& tp) {
  if (threadIdx.x != 0) return;
  if (tp.xfills) {
    long long spins = 0;
    while (!mbar_test(&tp.xfull, (tp.xfills - 1) & 1u) && ++spins < kDrainLimit) {
    }
  }
  for (int s = 0; s < kMaxStages; ++s) {
    const unsigned f = tp.fills[s];
    if (f == 0) continue;
    long long spins = 0;
    while (!mbar_test(&tp.full[s], (f - 1) & 1u) && ++spins < kDrainLimit) {
    }
  }
}

}  // namespace sv

namespace sv {
static_assert(kProducerWarp >= kMaxMmaTiles, "the producer warp must not own an MMA tile");
}  // namespace sv
