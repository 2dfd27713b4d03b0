// Tensor-copy (TMA) weight streaming of the persistent forward kernel.
//
// A GEMM phase's output rows come in MMA tiles of 16 rows (gemm_dev.cuh:
// plain tiles are rows 16t .. 16t+15; q/k/v tiles pair 8 rows with their
// RoPE partners hd/2 further; SwiGLU tiles pair 8 gate rows with the same 8
// up rows).  Each CTA owns a contiguous range of whole tiles -- every k of
// them -- so no tile is split between CTAs: a tile's sum is finished inside
// the CTA that streamed it, with no partial sums in global memory, no
// tickets and no last-arriving CTA on the way to the grid barrier.  The
// ranges are as even as whole tiles allow; when some CTAs own one tile
// fewer, they finish early and the busier ones, sharing HBM with fewer
// streams, run faster (one SM ingests ~44 GB/s when all 152 stream, up to
// ~80 GB/s when few do), so uneven ranges cost far less than their byte
// imbalance.
//
// Stages.  A stage holds gt tiles x kc columns of weights (32 KB): per tile
// and 256-k block one tensor copy of 16 rows (plain) or two of 8 rows
// (paired).  The input X (ntok rows) is either resident -- copied into
// shared memory once per phase, one bulk copy per token, when ntok x k fits
// the X region -- or streamed: per 256-k block one box of the ntok rows,
// behind the stage's weights (the 14336-wide input of a 6-token 8B
// down-projection).  Resident phases take one tile per stage group (gt = 1,
// kc = 1024); streamed phases group two tiles (gt = 2, kc = 512) so that
// each X box serves both.
//
// Warps.  One producer thread (warp kProducerWarp) issues the copies through
// a ring of S stages.  The eight consumer warps split every stage by k: warp
// w takes the stage's 64-k steps w and w + 8 (16 steps per stage: with
// gt = 2 the first eight belong to the group's first tile, the last eight to
// its second), each into its own accumulator chain.  At the end of a group
// every warp leaves its partial sums in shared memory; after a barrier of
// the consumer warps one warp per tile adds the eight partials in warp
// order, applies 1/rms (RMSNorm'd inputs) and runs the tile's epilogue while
// the other warps go on with the next stages (resident phases alternate two
// partial buffers, so the next group's partials never overwrite ones still
// being read).  The summation order depends on k and the warp count only, so
// every pass is batch-invariant.  (Handing the partials to the epilogue warp
// through mbarriers instead of the barrier measured no faster.)
//
// Phase boundaries.  Between arriving at the grid barrier before a GEMM
// phase and leaving it, the producer already fills the ring with the
// phase's first units (weights are read-only), so HBM keeps streaming while
// the grid waits; after the barrier it copies X (and, streamed, the X boxes
// of those units) and streams the rest.
//
// Every wait is bounded.  A wait that gives up raises the CTA's abort flag;
// from then on every wait of the CTA returns at once and the warps run
// through their remaining iterations without touching the data (barrier
// counts stay identical); the kernel reports the failure and leaves after
// waiting, again with a bound, for its copies still in flight.
#pragma once
#include "gemm_dev.cuh"

namespace sv {

constexpr int kTmaK = 256;                        // k per box (box inner extent)
constexpr int kTmaRowBytes = kTmaK * 2;           // row pitch of a box in shared memory
constexpr int kTileRows = 16;
constexpr int kTileBlockBytes = kTileRows * kTmaRowBytes;   // one tile x 256 k: 8 KB
constexpr int kStageWeightBytes = 4 * kTileBlockBytes;       // 32 KB of weights per stage
constexpr int kStageSteps = kStageWeightBytes / (kTileRows * kStepK * 2);   // 64-k steps per stage: 16
constexpr int kCWarps = 8;                        // consumer warps (attention uses them all)
constexpr int kConsumerThreads = kCWarps * 32;
constexpr int kProducerWarp = kCWarps;            // lane 0 issues the tensor copies
constexpr int kPersistThreads = (kCWarps + 1) * 32;
constexpr int kMaxStages = 8;
constexpr int kMaxGroupTiles = 2;
constexpr size_t kRingMaxBytes = 160 * 1024;      // weight ring (5 stages of 32 KB)
// group partials: [2 buffers or kMaxGroupTiles tiles][8 warps][32 lanes] float4
constexpr size_t kRedBytes = (size_t)2 * kCWarps * 32 * 16;
constexpr size_t kXMinBytes = 36 * 1024;          // X region: at least a 2-token 8192-wide input
constexpr long long kWaitLimit = 1LL << 22;
constexpr long long kDrainLimit = 1LL << 16;
constexpr int kPersistMaxTok = 8;
constexpr size_t kTensorMapBytes = 128;
constexpr int kGemmBarrier = 2;                   // named barrier of the consumer warps (1: attention)

struct TmaPipe {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t xfull;               // the bulk X copies of a resident-X phase
  unsigned fills[kMaxStages];   // fills issued per slot (producer)
  unsigned xfills;              // X loads issued (their barrier's phase count)
  int abort;
};

SV_DEV void tma_init(TmaPipe& tp) {
  if (threadIdx.x == 0) {
    for (int i = 0; i < kMaxStages; ++i) {
      mbar_init(&tp.full[i], 1);
      mbar_init(&tp.empty[i], kCWarps);   // released by every consumer warp
      tp.fills[i] = 0;
    }
    mbar_init(&tp.xfull, 1);
    tp.xfills = 0;
    tp.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
}

// Wait for the completion of the phase of `parity`; false once the CTA has
// aborted (raising the flag when this wait is the one that gives up).  The
// abort flag is read every 64 probes only: a shared-memory read in every
// probe of the eight polling consumer warps slowed the weight stream by ~7%.
SV_DEV bool tma_wait(uint64_t* bar, unsigned parity, TmaPipe& tp) {
  volatile int* ab = &tp.abort;
  long long spins = 0;
  while (true) {
    if (mbar_test(bar, parity)) return true;
    if ((++spins & 63) == 0) {
      if (*ab) return false;
      if (spins > kWaitLimit) {
        *ab = 1;
        return false;
      }
    }
  }
}

// The phase's streaming geometry and this CTA's tiles [t0, t1), copied out
// of the shared-memory phase descriptor into registers once per phase: the
// copy and MMA loops run between asm statements that act as compiler memory
// barriers, so fields read from the descriptor inside them would be loaded
// again and again on the issue path.
struct TmaGeo {
  const unsigned char* maps;
  const void* x;                 // streamed X's tensor map is tm[3]
  int S, sb, kc, k, gt, paired, ntok, xoff, xs;
  int epi, hd, seg0, seg1;
  int tm0, tm1, tm2, tmx;        // weight segments 0..2, streamed X
  int t0, t1, nchunks, ngroups, n;
};

SV_DEV TmaGeo tma_geo(const PhaseDesc& d, const unsigned char* maps) {
  TmaGeo q;
  q.maps = maps;
  q.x = d.g.x;
  q.S = d.stages;
  q.sb = d.stage_bytes;
  q.kc = d.kc;
  q.k = d.g.k;
  q.gt = d.gt;
  q.paired = d.paired;
  q.ntok = d.g.ntok;
  q.xoff = d.xoff;
  q.xs = d.xm == kXGlobal;
  q.epi = d.g.epi;
  q.hd = d.g.hd;
  q.seg0 = d.g.seg_rows[0];
  q.seg1 = d.g.seg_rows[1];
  q.tm0 = d.tm[0];
  q.tm1 = d.tm[1];
  q.tm2 = d.tm[2];
  q.tmx = d.tm[3];
  const int tiles = d.tiles;
  const int G = min((int)gridDim.x, tiles);
  const bool has = (int)blockIdx.x < G;
  q.t0 = has ? (int)first_step_of_warp(blockIdx.x, tiles, G) : 0;
  q.t1 = has ? (int)first_step_of_warp(blockIdx.x + 1, tiles, G) : 0;
  q.nchunks = (q.k + q.kc - 1) / q.kc;
  q.ngroups = (q.t1 - q.t0 + q.gt - 1) / q.gt;
  q.n = q.ngroups * q.nchunks;
  return q;
}

// Tensor-map index and first row of box A (and box B when paired) of tile t.
struct TileBoxes {
  int ma, ra, mb, rb;
};
SV_DEV TileBoxes tile_boxes(const TmaGeo& q, int t) {
  if (q.epi == kEpiQkvRope) {
    const int per = q.hd / 16;
    int row = (t / per) * q.hd + 8 * (t % per);
    int seg = 0;
    if (row >= q.seg0) {
      row -= q.seg0;
      seg = 1;
      if (row >= q.seg1) {
        row -= q.seg1;
        seg = 2;
      }
    }
    const int m = seg == 0 ? q.tm0 : seg == 1 ? q.tm1 : q.tm2;
    return {m, row, m, row + q.hd / 2};
  }
  if (q.epi == kEpiSwiglu) return {q.tm0, 8 * t, q.tm1, 8 * t};
  return {q.tm0, 16 * t, q.tm0, 16 * t};   // one box of 16 rows
}

// 256-k blocks of chunk c (the last chunk may be short).
SV_DEV int chunk_blocks(const TmaGeo& q, int c) {
  return min(q.kc / kTmaK, (q.k - c * q.kc + kTmaK - 1) / kTmaK);
}

// Resident-X phase, before its units: the producer thread copies the ntok
// input rows (k bf16 each; for an RMSNorm'd input the rows already carry the
// norm's gain) into the X region with one bulk copy per token, completing on
// tp.xfull; every warp meanwhile folds the per-tile sums of squares into
// s_inv[tok] = 1 / rms (RMSNorm'd inputs only).  Ends with a CTA barrier.
SV_DEV void tma_prepare_x(const PhaseDesc& d, TmaPipe& tp, float* s_inv, unsigned char* xreg) {
  const GemmDesc& g = d.g;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp == kProducerWarp && lane == 0 && tma_geo(d, nullptr).n > 0) {
    const int k = g.k, ntok = g.ntok, ldx = g.ldx;
    const bf16* x = (const bf16*)g.x;
    fence_proxy_async_global();   // X was written by other CTAs before the grid barrier
    mbar_arrive_expect_tx(&tp.xfull, (unsigned)k * 2u * (unsigned)ntok);
    const size_t pitch = (size_t)(k + kXPad) * 2;
    for (int t = 0; t < ntok; ++t) bulk_g2s(xreg + t * pitch, x + (size_t)t * ldx, (unsigned)k * 2u, &tp.xfull);
    tp.xfills += 1;
  }
  if (g.x_norm == 2)
    for (int tok = warp; tok < g.ntok; tok += kPersistThreads / 32) {
      const float v = warp_inv_rms(g, tok, lane);
      if (lane == 0) s_inv[tok] = v;
    }
  __syncthreads();
}

// Producer thread: walks the CTA's units (tile group, chunk) in order,
// issuing units [i, end) into the ring -- per unit: wait for the consumers
// to release the slot, announce the bytes (the weights and, for streamed X,
// the X boxes, even when those are issued later), copy the weight boxes
// and, when with_x, the X boxes.  The walk keeps its position in registers;
// no division on the way.
struct TmaWalk {
  int i, slot, grp, c, ng;
  TileBoxes b0, b1;   // the group's tiles (kMaxGroupTiles = 2)
};
static_assert(kMaxGroupTiles == 2, "TmaWalk holds two tiles");

SV_DEV void walk_group(const TmaGeo& q, TmaWalk& w) {
  const int tb = q.t0 + w.grp * q.gt;
  w.ng = min(q.gt, q.t1 - tb);
  w.b0 = tile_boxes(q, tb);
  if (w.ng > 1) w.b1 = tile_boxes(q, tb + 1);
}

SV_DEV TmaWalk walk_start(const TmaGeo& q) {
  TmaWalk w;
  w.i = 0;
  w.slot = 0;
  w.grp = 0;
  w.c = 0;
  w.ng = 0;
  if (q.n > 0) walk_group(q, w);
  return w;
}

SV_DEV void walk_next(const TmaGeo& q, TmaWalk& w) {
  ++w.i;
  if (++w.slot == q.S) w.slot = 0;
  if (++w.c == q.nchunks) {
    w.c = 0;
    ++w.grp;
    if (w.i < q.n) walk_group(q, w);
  }
}

SV_DEV void tma_issue_units(const TmaGeo& q, TmaWalk& w, int end, bool with_x, TmaPipe& tp, unsigned char* ring) {
  const uint64_t pol = l2_evict_first();   // weights are read once per pass
  const int kbs = q.kc / kTmaK;
  const unsigned char* maps = q.maps;
  for (; w.i < end; walk_next(q, w)) {
    const int slot = w.slot;
    const unsigned f = tp.fills[slot];
    if (!tma_wait(&tp.empty[slot], (f & 1u) ^ 1u, tp)) return;
    const int nkb = chunk_blocks(q, w.c);
    const int k0 = w.c * q.kc;
    const unsigned xbytes = q.xs ? (unsigned)(nkb * q.ntok * kTmaRowBytes) : 0u;
    mbar_arrive_expect_tx(&tp.full[slot], (unsigned)(w.ng * nkb * kTileBlockBytes) + xbytes);
    unsigned char* st = ring + (size_t)slot * q.sb;
#pragma unroll
    for (int gq = 0; gq < kMaxGroupTiles; ++gq) {
      if (gq >= w.ng) break;
      const TileBoxes b = gq ? w.b1 : w.b0;
      const unsigned char* mapA = maps + (size_t)b.ma * kTensorMapBytes;
      const unsigned char* mapB = maps + (size_t)b.mb * kTensorMapBytes;
      unsigned char* dst = st + (size_t)gq * kbs * kTileBlockBytes;
      for (int kb = 0; kb < nkb; ++kb, dst += kTileBlockBytes) {
        tma_load_2d_hint(dst, mapA, k0 + kb * kTmaK, b.ra, &tp.full[slot], pol);
        if (q.paired) tma_load_2d_hint(dst + 8 * kTmaRowBytes, mapB, k0 + kb * kTmaK, b.rb, &tp.full[slot], pol);
      }
    }
    if (with_x) {
      const unsigned char* mapX = maps + (size_t)q.tmx * kTensorMapBytes;
      for (int kb = 0; kb < nkb; ++kb)
        tma_load_2d(st + q.xoff + (size_t)kb * q.ntok * kTmaRowBytes, mapX, k0 + kb * kTmaK, 0, &tp.full[slot]);
    }
    tp.fills[slot] = f + 1;
  }
}

// Producer thread, between arriving at the grid barrier that precedes GEMM
// phase d and waiting on it: the weight boxes of its first d.prefetch units
// (weights are read-only; X is not ready yet).  Returns how many units were
// issued.
SV_DEV int tma_prefetch(const PhaseDesc& d, TmaPipe& tp, unsigned char* ring, const unsigned char* maps) {
  const TmaGeo q = tma_geo(d, maps);
  TmaWalk w = walk_start(q);
  const int npre = min(q.n, d.prefetch);
  tma_issue_units(q, w, npre, false, tp, ring);
  return npre;
}

// Producer thread during GEMM phase d: the X boxes of the npre prefetched
// units (streamed X), then every remaining unit.
SV_DEV void tma_produce(const PhaseDesc& d, int npre, TmaPipe& tp, unsigned char* ring, const unsigned char* maps) {
  const TmaGeo q = tma_geo(d, maps);
  TmaWalk w = walk_start(q);
  if (q.xs) {
    fence_proxy_async_global();   // X was written by other CTAs before the grid barrier
    const unsigned char* mapX = maps + (size_t)q.tmx * kTensorMapBytes;
    for (; w.i < npre; walk_next(q, w)) {
      if (tp.abort) return;
      const int nkb = chunk_blocks(q, w.c);
      unsigned char* st = ring + (size_t)w.slot * q.sb;
      for (int kb = 0; kb < nkb; ++kb)
        tma_load_2d(st + q.xoff + (size_t)kb * q.ntok * kTmaRowBytes, mapX, w.c * q.kc + kb * kTmaK, 0,
                    &tp.full[w.slot]);
    }
  } else {
    while (w.i < npre) walk_next(q, w);
  }
  tma_issue_units(q, w, q.n, q.xs != 0, tp, ring);
}

// One 64-k step of a tile: rows gi / gi + 8 of the tile's 16-row block at
// byte offset boff (the step's 128-byte column) -- the thread's 16
// consecutive k at ci * 16 -- against the X words of token gi.
SV_DEV void tma_step(float (&acc)[4], const unsigned char* blk, const uint4& x0, const uint4& x1, int gi) {
  const uint4 a0 = *reinterpret_cast<const uint4*>(blk + gi * kTmaRowBytes);
  const uint4 a1 = *reinterpret_cast<const uint4*>(blk + gi * kTmaRowBytes + 16);
  const uint4 b0 = *reinterpret_cast<const uint4*>(blk + (gi + 8) * kTmaRowBytes);
  const uint4 b1 = *reinterpret_cast<const uint4*>(blk + (gi + 8) * kTmaRowBytes + 16);
  mma_bf16_16816(acc, a0.x, b0.x, a0.y, b0.y, x0.x, x0.y);
  mma_bf16_16816(acc, a0.z, b0.z, a0.w, b0.w, x0.z, x0.w);
  mma_bf16_16816(acc, a1.x, b1.x, a1.y, b1.y, x1.x, x1.y);
  mma_bf16_16816(acc, a1.z, b1.z, a1.w, b1.w, x1.z, x1.w);
}

// Consumer warps during GEMM phase d (see the file comment).  cpar: per-slot
// parity of the next completion of each stage's full barrier (identical in
// every consumer warp).  red: the group-partial area (kRedBytes).  s_inv:
// 1 / rms per token (RMSNorm'd inputs).  stamp (optional): atomicMax of the
// globaltimer when the last unit arrived.
template <bool kResident>
SV_DEV void tma_consume(const PhaseDesc& d, TmaPipe& tp, unsigned& cpar, const unsigned char* ring,
                        const unsigned char* xreg, float4* red, const float* s_inv, unsigned long long* stamp) {
  const GemmDesc& g = d.g;
  const TmaGeo q = tma_geo(d, nullptr);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gi = lane >> 2, ci = lane & 3;
  const int spt = q.kc / kStepK;            // 64-k steps per tile in a stage (16 or 8)
  const int kbs = q.kc / kTmaK;             // 256-k blocks per tile in a stage
  // this warp's two steps of every stage: tile (within the group), byte
  // offset of the step's 128-byte column in the stage, its k and, streamed,
  // its X column
  const int sA = warp, sB = warp + kCWarps;
  const int gA = sA / spt, kA = sA % spt, gB = sB / spt, kB = sB % spt;
  const int offA = (gA * kbs + kA / 4) * kTileBlockBytes + (kA % 4) * (kStepK * 2) + ci * 32;
  const int offB = (gB * kbs + kB / 4) * kTileBlockBytes + (kB % 4) * (kStepK * 2) + ci * 32;
  const bool has_tok = gi < q.ntok;
  const size_t xs_pitch = (size_t)(q.k + kXPad) * 2;
  const int xoffA = q.xoff + ((kA / 4) * q.ntok + gi) * kTmaRowBytes + (kA % 4) * (kStepK * 2) + ci * 32;
  const int xoffB = q.xoff + ((kB / 4) * q.ntok + gi) * kTmaRowBytes + (kB % 4) * (kStepK * 2) + ci * 32;
  const unsigned char* xrow = xreg + gi * xs_pitch + ci * 32;
  const uint4 zero4 = make_uint4(0, 0, 0, 0);
  const bool xn = g.x_norm == 2;
  const int pos0 = q.epi == kEpiQkvRope ? __ldcg(g.pos_base) + g.pos_off : 0;
  const int tiles_all = gemm_tiles_of(g);
  bool xok = true;
  if (kResident && q.n > 0) xok = tma_wait(&tp.xfull, (tp.xfills - 1) & 1u, tp);   // X copied in
  int i = 0, slot = 0;
#pragma unroll 1
  for (int grp = 0; grp < q.ngroups; ++grp) {
    const int tb = q.t0 + grp * q.gt, ng = min(q.gt, q.t1 - tb);
    const bool liveA = gA < ng, liveB = gB < ng;
    float accA[4] = {0.f, 0.f, 0.f, 0.f}, accB[4] = {0.f, 0.f, 0.f, 0.f};
    int kgA = kA * kStepK, kgB = kB * kStepK;   // the steps' k in this chunk
#pragma unroll 1
    for (int c = 0; c < q.nchunks; ++c, ++i, kgA += q.kc, kgB += q.kc) {
      const bool ok = tma_wait(&tp.full[slot], (cpar >> slot) & 1u, tp) && xok;
      cpar ^= 1u << slot;
      if (stamp && i == q.n - 1 && threadIdx.x == 0) {
        unsigned long long tm;
        asm volatile("mov.u64 %0, %globaltimer;" : "=l"(tm));
        atomicMax(stamp, tm);
      }
      if (ok) {
        const unsigned char* st = ring + (size_t)slot * q.sb;
        if (liveA && kgA < q.k) {
          uint4 x0 = zero4, x1 = zero4;
          if (has_tok) {
            const unsigned char* xp = kResident ? xrow + (size_t)kgA * 2 : st + xoffA;
            x0 = *reinterpret_cast<const uint4*>(xp);
            x1 = *reinterpret_cast<const uint4*>(xp + 16);
          }
          tma_step(accA, st + offA, x0, x1, gi);
        }
        if (liveB && kgB < q.k) {
          uint4 x0 = zero4, x1 = zero4;
          if (has_tok) {
            const unsigned char* xp = kResident ? xrow + (size_t)kgB * 2 : st + xoffB;
            x0 = *reinterpret_cast<const uint4*>(xp);
            x1 = *reinterpret_cast<const uint4*>(xp + 16);
          }
          tma_step(accB, st + offB, x0, x1, gi);
        }
      }
      __syncwarp();
      if (lane == 0 && ok) mbar_arrive(&tp.empty[slot]);
      if (++slot == q.S) slot = 0;
    }
    // end of the group: partials of every warp, then one warp per tile adds
    // them in warp order and runs the epilogue
    float4* rb = red + (size_t)(kResident ? (grp & 1) : 0) * kCWarps * 32;   // buffer (resident) or tile 0
    if (q.gt == 1) {
      rb[warp * 32 + lane] = make_float4(accA[0] + accB[0], accA[1] + accB[1], accA[2] + accB[2], accA[3] + accB[3]);
    } else {
      rb[warp * 32 + lane] = make_float4(accA[0], accA[1], accA[2], accA[3]);
      rb[(kCWarps + warp) * 32 + lane] = make_float4(accB[0], accB[1], accB[2], accB[3]);
    }
    named_sync(kGemmBarrier, kConsumerThreads);
    for (int gq = 0; gq < ng; ++gq) {
      const int ew = kResident ? grp % kCWarps : gq;   // the tile's epilogue warp
      if (warp != ew || tp.abort) continue;
      const int tile = tb + gq;
      if (tile >= tiles_all) continue;
      const float4* pt = rb + (size_t)gq * kCWarps * 32 + lane;
      float y[1][4] = {{0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int w = 0; w < kCWarps; ++w) {
        const float4 v = pt[w * 32];
        y[0][0] += v.x;
        y[0][1] += v.y;
        y[0][2] += v.z;
        y[0][3] += v.w;
      }
      if (xn) {
        const float sc0 = s_inv[2 * ci], sc1 = s_inv[2 * ci + 1];
        y[0][0] *= sc0;
        y[0][1] *= sc1;
        y[0][2] *= sc0;
        y[0][3] *= sc1;
      }
      EpiIn pre;
      gemm_epi_load<false>(g, tile, pos0, gi, ci, pre);
      gemm_epilogue<1, false>(g, tile, y, gi, ci, &pre);
    }
    // streamed X: the partial area is not double-buffered -- the next
    // group's partials wait until the epilogue warps have read these
    if (!kResident && grp + 1 < q.ngroups) named_sync(kGemmBarrier, kConsumerThreads);
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
