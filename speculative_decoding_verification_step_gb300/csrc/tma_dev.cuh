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
// every warp leaves its partial sums in shared memory and the group's tiles
// are finished -- the eight partials added in warp order, 1/rms applied
// (RMSNorm'd inputs), the epilogue run -- in one of two ways:
//  * bf16 phases (a group spans several stages): after a barrier of the
//    consumer warps, by one of them per tile while the others go on with the
//    next stages (resident phases alternate two partial buffers, so the next
//    group's partials never overwrite ones still being read);
//  * 4-bit phases (a whole tile per stage, so a group ends at every stage):
//    by a warp of its own (kEpiWarp), which waits on an mbarrier for the
//    eight partials, frees the buffer and runs the epilogue; the consumer
//    warps then share no barrier and never wait for an epilogue.  (On the
//    bf16 phases this hand-off measured ~1.5% slower than the barrier.)  The summation order depends on k and the warp
// count only, so every pass is batch-invariant.
//
// Phase boundaries.  Between arriving at the grid barrier before a GEMM
// phase and leaving it, the producer already fills the ring with the
// phase's first units (weights are read-only), so HBM keeps streaming while
// the grid waits; after the barrier it copies X (and, streamed, the X boxes
// of those units) and streams the rest.
//
// 4-bit weights (q4).  A matrix is stored as packed signed nibbles [n][k/2]
// (element 2b in the low nibble of byte b) followed by bf16 scales, one per
// 64-k group, group-major [k/64][n]; weight = scale x code.  A tile's stage
// block holds, per 8-row half, the codes as [k/256 blocks][8 rows][128 B]
// (one 3-D tensor copy with the 128-byte swizzle, so eight rows read at the
// same k hit distinct banks), then per half the scales [groups][8 rows] (one
// 2-D copy; a row's scale of a group is one 2-byte read).  A 64-k step is
// one group: the codes become bf16 (136 + v) by one lop3 per pair and exact
// v by one bf16x2 subtraction; four MMAs give the group's code . X sum,
// which the row's scale weights into the tile's fp32 total.  The code pairs
// come out as elements (i, i + 4) of each 8-code word, so the X operand
// takes the same pairs: resident X rows are permuted into that order once
// per phase, streamed X per step.
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
constexpr int kEpiWarp = kCWarps + 1;             // adds the partials and runs the epilogues
// (ten warps: an SM partition holds at most three, as with nine, so the
// register budget per thread is the same)
constexpr int kPersistThreads = (kCWarps + 2) * 32;
constexpr int kMaxStages = 8;
constexpr int kMaxGroupTiles = 2;
constexpr size_t kRingMaxBytes = 160 * 1024;      // weight ring (5 stages of 32 KB)
// group partials: [kMaxGroupTiles tiles][8 warps][32 lanes] float4
constexpr size_t kRedBytes = (size_t)kMaxGroupTiles * kCWarps * 32 * 16;
constexpr size_t kXMinBytes = 36 * 1024;          // X region: at least a 2-token 8192-wide input
constexpr long long kWaitLimit = 1LL << 22;
constexpr long long kDrainLimit = 1LL << 16;
constexpr int kPersistMaxTok = 8;
constexpr int kGemmBarrier = 2;                   // named barrier of the consumer warps (1: attention)
constexpr size_t kTensorMapBytes = 128;

struct TmaPipe {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t rfull;               // a group's partials written (every consumer warp)
  uint64_t rfree;               // ... and read (the epilogue warp)
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
    mbar_init(&tp.rfull, kCWarps);
    mbar_init(&tp.rfree, 1);
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

// The same for a warp with nothing else to do (the epilogue warp): each
// failed probe backs off 64 ns, so that its polling takes few issue slots
// from the consumer warps sharing its SM partition.
SV_DEV bool tma_wait_idle(uint64_t* bar, unsigned parity, TmaPipe& tp) {
  volatile int* ab = &tp.abort;
  long long spins = 0;
  while (true) {
    if (mbar_test(bar, parity)) return true;
    __nanosleep(64);
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
  int q4, tile_bytes, tms0, tms1, tms2;
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
  q.q4 = d.q4;
  q.tile_bytes = d.q4 ? d.tile_bytes : (d.kc / kTmaK) * kTileBlockBytes;
  q.tms0 = d.tms[0];
  q.tms1 = d.tms[1];
  q.tms2 = d.tms[2];
  // contiguous tile ranges, the larger shares first; counted from the last
  // CTA down when d.rev (see PhaseDesc::rev)
  const int tiles = d.tiles;
  const int G = min((int)gridDim.x, tiles);
  const int c = d.rev ? (int)gridDim.x - 1 - (int)blockIdx.x : (int)blockIdx.x;
  const bool has = c < G;
  const int base = tiles / G, rem = tiles - base * G;
  q.t0 = has ? c * base + min(c, rem) : 0;
  q.t1 = has ? q.t0 + base + (c < rem ? 1 : 0) : 0;
  q.nchunks = (q.k + q.kc - 1) / q.kc;
  q.ngroups = (q.t1 - q.t0 + q.gt - 1) / q.gt;
  q.n = q.ngroups * q.nchunks;
  return q;
}

// Tensor-map index and first row of box A (and box B when paired) of tile t.
struct TileBoxes {
  int ma, ra, mb, rb;
  int sa, sb;   // q4: scale maps of box A / B
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
    const int ms = seg == 0 ? q.tms0 : seg == 1 ? q.tms1 : q.tms2;
    return {m, row, m, row + q.hd / 2, ms, ms};
  }
  if (q.epi == kEpiSwiglu) return {q.tm0, 8 * t, q.tm1, 8 * t, q.tms0, q.tms1};
  // plain: one box of 16 rows (bf16); q4 always copies two 8-row halves
  return {q.tm0, 16 * t, q.tm0, 16 * t + 8, q.tms0, q.tms0};
}

// 256-k blocks of chunk c (the last chunk may be short).
SV_DEV int chunk_blocks(const TmaGeo& q, int c) {
  return min(q.kc / kTmaK, (q.k - c * q.kc + kTmaK - 1) / kTmaK);
}

// Before a resident-X or RMSNorm'd phase's units: for resident X the
// producer thread copies the ntok input rows (k bf16 each; for an RMSNorm'd
// input the rows already carry the norm's gain) into the X region with one
// bulk copy per token, completing on tp.xfull; every warp meanwhile folds the
// per-tile sums of squares into s_inv[tok] = 1 / rms (RMSNorm'd inputs,
// resident or streamed).  Ends with a CTA barrier.
SV_DEV void tma_prepare_x(const PhaseDesc& d, TmaPipe& tp, float* s_inv, unsigned char* xreg) {
  const GemmDesc& g = d.g;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (d.xm == kXSmem && warp == kProducerWarp && lane == 0 && tma_geo(d, nullptr).n > 0) {
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
  const unsigned char* maps = q.maps;
  for (; w.i < end; walk_next(q, w)) {
    const int slot = w.slot;
    const unsigned f = tp.fills[slot];
    if (!tma_wait(&tp.empty[slot], (f & 1u) ^ 1u, tp)) return;
    const int nkb = chunk_blocks(q, w.c);
    const int k0 = w.c * q.kc;
    const unsigned xbytes = q.xs ? (unsigned)(nkb * q.ntok * kTmaRowBytes) : 0u;
    // q4: full boxes every chunk (a short last chunk reads zeros past k):
    // per tile two code boxes of 8 rows x kc/2 bytes and two scale boxes of
    // 8 rows x kc/64 bf16 -- 8.5 kc bytes (the tile's block is padded to 1 KB)
    const unsigned wbytes =
        q.q4 ? (unsigned)(w.ng * (q.kc * 8 + q.kc / 2)) : (unsigned)(w.ng * nkb * kTileBlockBytes);
    mbar_arrive_expect_tx(&tp.full[slot], wbytes + xbytes);
    unsigned char* st = ring + (size_t)slot * q.sb;
#pragma unroll
    for (int gq = 0; gq < kMaxGroupTiles; ++gq) {
      if (gq >= w.ng) break;
      const TileBoxes b = gq ? w.b1 : w.b0;
      const unsigned char* mapA = maps + (size_t)b.ma * kTensorMapBytes;
      const unsigned char* mapB = maps + (size_t)b.mb * kTensorMapBytes;
      unsigned char* dst = st + (size_t)gq * q.tile_bytes;
      if (q.q4) {
        const int half = (q.kc / kTmaK) * 1024;   // codes of one 8-row half
        tma_load_3d_hint(dst, mapA, 0, b.ra, k0 / kTmaK, &tp.full[slot], pol);
        tma_load_3d_hint(dst + half, mapB, 0, b.rb, k0 / kTmaK, &tp.full[slot], pol);
        unsigned char* sd = dst + 2 * half;
        tma_load_2d_hint(sd, maps + (size_t)b.sa * kTensorMapBytes, b.ra, k0 / 64, &tp.full[slot], pol);
        tma_load_2d_hint(sd + (q.kc / 64) * 16, maps + (size_t)b.sb * kTensorMapBytes, b.rb, k0 / 64, &tp.full[slot],
                         pol);
        continue;
      }
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

// End of a tile group of a bf16 phase (every consumer warp): each warp's
// partial sums of the group's tiles (gt = 1: a + b, the warp's two chains;
// gt = 2: a for the first tile, b for the second) go to shared memory; after
// a barrier of the consumer warps one warp per tile adds the eight partials
// in warp order, applies 1/rms (RMSNorm'd inputs) and runs the tile's
// epilogue.  Resident phases alternate two partial buffers (the next group's
// partials never overwrite ones still being read); streamed phases use both
// halves for their two tiles and wait for the readers before the next group.
SV_DEV void tma_group_end(const TmaGeo& q, const GemmDesc& g, TmaPipe& tp, float4* red, const float* s_inv,
                          const float (&a)[4], const float (&b)[4], bool resident, int grp, int tb, int ng, int pos0,
                          int tiles_all) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gi = lane >> 2, ci = lane & 3;
  float4* rb = red + (size_t)(resident ? (grp & 1) : 0) * kCWarps * 32;   // buffer (resident) or tile 0
  if (q.gt == 1) {
    rb[warp * 32 + lane] = make_float4(a[0] + b[0], a[1] + b[1], a[2] + b[2], a[3] + b[3]);
  } else {
    rb[warp * 32 + lane] = make_float4(a[0], a[1], a[2], a[3]);
    rb[(kCWarps + warp) * 32 + lane] = make_float4(b[0], b[1], b[2], b[3]);
  }
  named_sync(kGemmBarrier, kConsumerThreads);
  for (int gq = 0; gq < ng; ++gq) {
    const int ew = resident ? grp % kCWarps : gq;   // the tile's epilogue warp
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
    if (g.x_norm == 2) {
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
  // streamed X: the partial area is not double-buffered -- the next group's
  // partials wait until the epilogue warps have read these
  if (!resident && grp + 1 < q.ngroups) named_sync(kGemmBarrier, kConsumerThreads);
}

// End of a tile group of a 4-bit phase (every consumer warp): the warp's partial sums of the
// group's tiles (gt = 1: a + b, its two chains; gt = 2: a for the first
// tile, b for the second) go to the partial buffer -- once the epilogue warp
// has read the previous group's -- and the warp arrives on its barrier.
// gcount counts the groups of the launch (every consumer warp runs the same
// groups).
SV_DEV void tma_group_put(const TmaGeo& q, TmaPipe& tp, float4* red, const float (&a)[4], const float (&b)[4],
                          unsigned& gcount) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (gcount > 0) tma_wait(&tp.rfree, (gcount - 1) & 1u, tp);
  float4* rb = red;
  if (q.gt == 1) {
    rb[warp * 32 + lane] = make_float4(a[0] + b[0], a[1] + b[1], a[2] + b[2], a[3] + b[3]);
  } else {
    rb[warp * 32 + lane] = make_float4(a[0], a[1], a[2], a[3]);
    rb[(kCWarps + warp) * 32 + lane] = make_float4(b[0], b[1], b[2], b[3]);
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(&tp.rfull);
  ++gcount;
}

// The epilogue warp during a 4-bit GEMM phase d: for every tile group of the CTA, in
// order, wait for the eight partials (ecount counts the groups of the launch,
// as gcount does), add them in warp order, free the buffer, apply 1/rms
// (RMSNorm'd inputs) and run the tiles' epilogues.
SV_DEV void tma_epilogue(const PhaseDesc& d, TmaPipe& tp, const float4* red, const float* s_inv, unsigned& ecount) {
  static_assert(kMaxGroupTiles == 2, "the epilogue warp holds two tiles' sums");
  const GemmDesc& g = d.g;
  const TmaGeo q = tma_geo(d, nullptr);
  const int lane = threadIdx.x & 31, gi = lane >> 2, ci = lane & 3;
  const int pos0 = q.epi == kEpiQkvRope ? __ldcg(g.pos_base) + g.pos_off : 0;
  const int tiles_all = gemm_tiles_of(g);
#pragma unroll 1
  for (int grp = 0; grp < q.ngroups; ++grp) {
    const int tb = q.t0 + grp * q.gt, ng = min(q.gt, q.t1 - tb);
    const bool ok = tma_wait_idle(&tp.rfull, ecount & 1u, tp);
    float y0[1][4] = {{0.f, 0.f, 0.f, 0.f}}, y1[1][4] = {{0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int w = 0; w < kCWarps; ++w) {
      const float4 v = red[w * 32 + lane];
      y0[0][0] += v.x;
      y0[0][1] += v.y;
      y0[0][2] += v.z;
      y0[0][3] += v.w;
    }
    if (ng > 1) {
#pragma unroll
      for (int w = 0; w < kCWarps; ++w) {
        const float4 v = red[(kCWarps + w) * 32 + lane];
        y1[0][0] += v.x;
        y1[0][1] += v.y;
        y1[0][2] += v.z;
        y1[0][3] += v.w;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&tp.rfree);   // the consumers may write the next group's partials
    ++ecount;
    for (int gq = 0; gq < ng; ++gq) {
      const int tile = tb + gq;
      if (!ok || tp.abort || tile >= tiles_all) continue;
      float (&y)[1][4] = gq ? y1 : y0;
      if (g.x_norm == 2) {
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
  }
}

// One 64-k group of a q4 tile for rows gi (half 0) and gi + 8 (half 1):
// the thread's 16 codes per row (bytes ci*8 .. ci*8+7 of the group's 32, at
// their swizzled place), the rows' scales, and the 16 X values x0, x1 of
// token gi at the same k; adds scale x (codes . X) to tot.
SV_DEV uint32_t q4_pair(uint32_t t) {   // nibbles 0 and 4 of t (offset binary) -> bf16 (136 + v) x 2
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(t), "r"(0x000F000Fu), "r"(0x43004300u));
  return r;
}
SV_DEV uint32_t q4_exact(uint32_t p) {   // (136 + v) x 2 -> v x 2, exactly (0x4308 = bf16 136)
  uint32_t r;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(p), "r"(0x43084308u));
  return r;
}
SV_DEV uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
// Two chained MMAs over the 8 codes (one word) of each row of a pair against
// the thread's X pairs for them.
SV_DEV void q4_mma(float (&acc)[4], uint32_t wa, uint32_t wb, uint32_t xa, uint32_t xb, uint32_t xc, uint32_t xd,
                   bool first) {
  const uint32_t ta = wa ^ 0x88888888u, tb = wb ^ 0x88888888u;
  const uint32_t a0 = q4_exact(q4_pair(ta)), b0 = q4_exact(q4_pair(tb));
  const uint32_t a1 = q4_exact(q4_pair(ta >> 4)), b1 = q4_exact(q4_pair(tb >> 4));
  const uint32_t a2 = q4_exact(q4_pair(ta >> 8)), b2 = q4_exact(q4_pair(tb >> 8));
  const uint32_t a3 = q4_exact(q4_pair(ta >> 12)), b3 = q4_exact(q4_pair(tb >> 12));
  if (first)
    mma_bf16_16816_z(acc, a0, b0, a1, b1, xa, xb);
  else
    mma_bf16_16816_acc(acc, a0, b0, a1, b1, xa, xb);
  mma_bf16_16816_acc(acc, a2, b2, a3, b3, xc, xd);
}
// The thread's 8 code bytes of group ks in row gi of a half: block ks / 4,
// logical 16-byte chunk 2 (ks mod 4) + ci / 2 of the row, swizzled by the
// row (rbase = gi * 128 + (ci mod 2) * 8).
// kResident: x0, x1 are already in the codes' pair order; else they are
// natural X and permuted here.
template <bool kResident>
SV_DEV void q4_step(float (&tot)[4], const unsigned char* tile, int half, int ngrp, int ks, int rbase, int ci,
                    const uint4& x0, const uint4& x1, int gi, float w) {
  const int off = (ks >> 2) * 1024 + rbase + (((((ks & 3) << 1) + (ci >> 1)) ^ gi) & 7) * 16;
  const uint2 ca = *reinterpret_cast<const uint2*>(tile + off);
  const uint2 cb = *reinterpret_cast<const uint2*>(tile + half + off);
  const unsigned char* sc = tile + 2 * half + ks * 16 + gi * 2;
  const float sa = w * __uint_as_float((uint32_t)*reinterpret_cast<const unsigned short*>(sc) << 16);
  const float sb = w * __uint_as_float((uint32_t)*reinterpret_cast<const unsigned short*>(sc + ngrp * 16) << 16);
  float acc[4], acd[4];
  // codes 0..7 of the row pair, then 8..15 (two independent chains)
  if (kResident) {
    q4_mma(acc, ca.x, cb.x, x0.x, x0.y, x0.z, x0.w, true);
    q4_mma(acd, ca.y, cb.y, x1.x, x1.y, x1.z, x1.w, true);
  } else {
    q4_mma(acc, ca.x, cb.x, prmt(x0.x, x0.z, 0x5410u), prmt(x0.x, x0.z, 0x7632u), prmt(x0.y, x0.w, 0x5410u),
           prmt(x0.y, x0.w, 0x7632u), true);
    q4_mma(acd, ca.y, cb.y, prmt(x1.x, x1.z, 0x5410u), prmt(x1.x, x1.z, 0x7632u), prmt(x1.y, x1.w, 0x5410u),
           prmt(x1.y, x1.w, 0x7632u), true);
  }
  tot[0] = fmaf(sa, acc[0] + acd[0], tot[0]);
  tot[1] = fmaf(sa, acc[1] + acd[1], tot[1]);
  tot[2] = fmaf(sb, acc[2] + acd[2], tot[2]);
  tot[3] = fmaf(sb, acc[3] + acd[3], tot[3]);
}

// Consumer warps of a q4 GEMM phase: every stage holds gt tiles x kc k as
// gt tile blocks; its (tile, group) steps are dealt to the warps round robin
// (step s to warp s mod 8), each tile's sum kept in its own accumulator.
template <bool kResident>
SV_DEV void tma_consume_q4(const PhaseDesc& d, TmaPipe& tp, unsigned& cpar, unsigned& gcount,
                           const unsigned char* ring, const unsigned char* xreg, float4* red,
                           unsigned long long* stamp) {
  const TmaGeo q = tma_geo(d, nullptr);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gi = lane >> 2, ci = lane & 3;
  const int ngrp = q.kc / 64;               // 64-k groups per tile in a stage (a power of two)
  const int lgn = 31 - __clz(ngrp);
  const int half = (q.kc / kTmaK) * 1024;   // codes of one 8-row half
  const int steps = q.gt * ngrp;
  const int nj = (steps + kCWarps - 1) / kCWarps;   // steps per warp per stage
  const bool has_tok = gi < q.ntok;
  const int gx = min(gi, q.ntok - 1);       // X row read (rows past ntok are read as 0)
  const size_t xs_pitch = (size_t)(q.k + kXPad) * 2;
  const unsigned char* xrow = xreg + gx * xs_pitch + ci * 32;
  const int rbase = gi * 128 + (ci & 1) * 8;
  const uint4 zero4 = make_uint4(0, 0, 0, 0);
  bool xok = true;
  if (kResident && q.n > 0) {
    xok = tma_wait(&tp.xfull, (tp.xfills - 1) & 1u, tp);   // X copied in
    // every 8-element block of the rows permuted once into the codes' pair
    // order (0,4) (1,5) (2,6) (3,7)
    const int nb = q.k / 8;
    for (int e = threadIdx.x; xok && e < q.ntok * nb; e += kConsumerThreads) {
      const int t = e / nb, bq = e - t * nb;
      uint4* blk = reinterpret_cast<uint4*>(const_cast<unsigned char*>(xreg) + t * xs_pitch) + bq;
      const uint4 v = *blk;
      *blk = make_uint4(prmt(v.x, v.z, 0x5410u), prmt(v.x, v.z, 0x7632u), prmt(v.y, v.w, 0x5410u),
                        prmt(v.y, v.w, 0x7632u));
    }
    named_sync(kGemmBarrier, kConsumerThreads);
  }
  int i = 0, slot = 0;
#pragma unroll 1
  for (int grp = 0; grp < q.ngroups; ++grp) {
    const int tb = q.t0 + grp * q.gt, ng = min(q.gt, q.t1 - tb);
    float accA[4] = {0.f, 0.f, 0.f, 0.f}, accB[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
    for (int c = 0; c < q.nchunks; ++c, ++i) {
      const bool ok = tma_wait(&tp.full[slot], (cpar >> slot) & 1u, tp) && xok;
      cpar ^= 1u << slot;
      if (stamp && i == q.n - 1 && threadIdx.x == 0) {
        unsigned long long tm;
        asm volatile("mov.u64 %0, %globaltimer;" : "=l"(tm));
        atomicMax(stamp, tm);
      }
      if (ok) {
        const unsigned char* st = ring + (size_t)slot * q.sb;
        const int kc0 = c * q.kc;
        // branch-free steps (so that the compiler can overlap them): a step
        // past the stage's work reads group 0 of tile 0 and weighs it by 0
#pragma unroll 2
        for (int j = 0; j < nj; ++j) {
          const int s = warp + kCWarps * j;
          int gq = s >> lgn, ks = s & (ngrp - 1);
          int kg = kc0 + ks * 64;
          const bool live = s < steps && gq < ng && kg < q.k;
          gq = live ? gq : 0;
          ks = live ? ks : 0;
          kg = live ? kg : kc0;
          const unsigned char* xp =
              kResident ? xrow + (size_t)kg * 2
                        : st + q.xoff + ((size_t)(ks >> 2) * q.ntok + gx) * kTmaRowBytes + (ks & 3) * 128 + ci * 32;
          uint4 x0 = *reinterpret_cast<const uint4*>(xp);
          uint4 x1 = *reinterpret_cast<const uint4*>(xp + 16);
          x0 = has_tok ? x0 : zero4;
          x1 = has_tok ? x1 : zero4;
          const float w = live ? 1.f : 0.f;
          if (kResident || gq == 0)   // resident phases hold one tile per group
            q4_step<kResident>(accA, st, half, ngrp, ks, rbase, ci, x0, x1, gi, w);
          else
            q4_step<kResident>(accB, st + (size_t)q.tile_bytes, half, ngrp, ks, rbase, ci, x0, x1, gi, w);
        }
      }
      __syncwarp();
      if (lane == 0 && ok) mbar_arrive(&tp.empty[slot]);
      if (++slot == q.S) slot = 0;
    }
    if (q.gt == 1) {   // one tile: the warp's sum is accA alone
#pragma unroll
      for (int e = 0; e < 4; ++e) accB[e] = 0.f;
    }
    tma_group_put(q, tp, red, accA, accB, gcount);
  }
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
  const int pos0 = q.epi == kEpiQkvRope ? __ldcg(g.pos_base) + g.pos_off : 0;
  const int tiles_all = gemm_tiles_of(g);
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
    tma_group_end(q, g, tp, red, s_inv, accA, accB, kResident, grp, tb, ng, pos0, tiles_all);
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
