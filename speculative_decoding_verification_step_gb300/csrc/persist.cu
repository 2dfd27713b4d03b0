// Persistent forward kernel (bf16 models).
//
// A batch-1 decode or verify pass is a chain of ~5 dependent phases per layer
// (q/k/v GEMM with RoPE + KV append, attention, o-projection, gate/up GEMM,
// down-projection), each of which must see the whole output of the previous
// one.  Launched one kernel per phase, every weight-streaming GEMM pays its
// ramp-up and tail (the HBM pipe drains at each kernel boundary), which for
// the 8-50 MB matrices of a decoder layer costs as much as the streaming
// itself.  Here one cooperative launch runs all phases of a forward:
//   * one CTA per SM stays resident; phases are separated by a grid barrier
//     split in an arrive and a wait half;
//   * GEMM phases stream weights with 2-D tensor copies (TMA) through a
//     shared-memory ring (tma_dev.cuh): each CTA owns whole 16-row output
//     tiles, one producer warp copies, eight consumer warps split every
//     stage by k and finish their tiles inside the CTA;
//   * between arriving at a barrier and waiting on it, the producer already
//     issues the weight copies of the next GEMM phase's first units (weights
//     are read-only), so HBM keeps streaming across phase boundaries;
//   * attention phases run the tensor-core decode attention (dattn_dev.cuh)
//     on the eight consumer warps; the embedding reuses embed_dev.cuh.
// The work split depends only on the matrix shapes and the SM count, never
// on the token count, so every pass is batch-invariant.  Every wait is
// bounded: a grid-barrier wait that gives up, or a pipeline wait (see
// tma_dev.cuh), sets the error flag and the kernel leaves; the host reports
// a timeout.  Activations written by other CTAs are read through L2.
#include "dattn_dev.cuh"
#include "embed_dev.cuh"
#include "tma_dev.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <algorithm>

namespace sv {

constexpr long long kBarrierSpinLimit = 1LL << 22;

SV_DEV unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

SV_DEV unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barrier of a co-resident launch, split in two halves so that
// the next phase's weight copies can be issued in between.  bar[0] counts
// arrivals since the launch began: every CTA arrives once at each barrier
// (after phase ph the count to wait for is (ph + 1) * gridDim.x) and once
// more on leaving, and the CTA whose leaving arrival completes the count
// resets it for the next launch -- by then every CTA has passed its last
// wait.  grid_arrive (every thread, after the phase's last shared-memory use)
// publishes this CTA's writes with a release add; grid_wait returns once the
// count is reached, false (in every thread of the CTA) when the wait gave up
// or another CTA reported an error.
SV_DEV void grid_arrive(unsigned* bar) {
  __syncthreads();
  if (threadIdx.x == 0) red_add_release_gpu(bar, 1u);
}

// The error flag is read only while still waiting -- every 64 polls -- so a
// completed wait costs no extra round trip: a CTA that gave up stops
// arriving, and the others notice its flag within 64 polls.  A launch that
// starts with the flag raised (a pass before it in the same step gave up and
// left the arrival count unbalanced) leaves before its first arrival, so no
// wait ever completes on a stale count.
SV_DEV bool grid_wait(unsigned* bar, unsigned target, int* err, int* s_ok, long long limit) {
  if (threadIdx.x == 0) {
    int ok = 1;
    long long spins = 0;
    while (ld_acquire_u32(bar) < target) {
      ++spins;
      if (spins > limit) {
        atomicExch(err, 1);
        ok = 0;
        break;
      }
      if ((spins & 63) == 0 && ld_volatile_i32(err) != 0) {
        ok = 0;
        break;
      }
    }
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok != 0;
}

SV_DEV void grid_leave(unsigned* bar, unsigned total) {
  __syncthreads();
  if (threadIdx.x == 0 && atom_add_acq_rel_gpu(bar, 1u) == total - 1) st_relaxed_gpu(bar, 0u);
}

template <int HD, bool kGroup>
__global__ void __launch_bounds__(kPersistThreads, 1) persist_forward(const __grid_constant__ PersistDesc p) {
  // dynamic shared memory: [group partials, kRedBytes][weight ring,
  // p.ring_bytes][X region: resident GEMM inputs]; a streamed-X GEMM phase,
  // which has no resident input, runs its ring on into the X region;
  // attention phases reuse it all from offset 0
  extern __shared__ __align__(1024) unsigned char dsm[];
  __shared__ TmaPipe tp;
  __shared__ uint64_t dbars[kDWarps * kDMaxDepth];   // attention stage barriers
  __shared__ float s_inv[kGemmMaxTok];
  __shared__ int s_last, s_ok;
  // the current and the next phase descriptor, staged in shared memory
  __shared__ __align__(16) PhaseDesc s_ph[2];
  float4* red = reinterpret_cast<float4*>(dsm);
  unsigned char* ring = dsm + kRedBytes;
  unsigned char* xreg = dsm + kRedBytes + p.ring_bytes;
  const unsigned char* maps = reinterpret_cast<const unsigned char*>(p.tmaps);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool producer = warp == kProducerWarp;
  const bool epiw = warp == kEpiWarp;
  // phase descriptors: one word per thread, read at the start of the
  // previous phase and stored into its shared-memory slot at that phase's
  // end, so that the load's latency is not on the way to the grid barrier
  constexpr int kDescWords = (int)(sizeof(PhaseDesc) / 4);
  static_assert(sizeof(PhaseDesc) % 4 == 0 && kDescWords <= kPersistThreads, "one word per thread");
  auto load_desc = [&](int ph) {
    return threadIdx.x < kDescWords ? __ldg(reinterpret_cast<const int*>(p.phases + ph) + threadIdx.x) : 0;
  };
  auto store_desc = [&](int slot, int word) {
    if (threadIdx.x < kDescWords) reinterpret_cast<int*>(&s_ph[slot])[threadIdx.x] = word;
  };
  unsigned long long* const times = p.times;
  if (times && blockIdx.x == 0 && threadIdx.x == 0) times[0] = global_ns();
  // fault injection (tests): extra arrivals to wait for, and the probe bound
  unsigned bar_extra = 0;
  long long bar_limit = kBarrierSpinLimit;
  if (p.ctl && threadIdx.x == 0) {
    bar_extra = (unsigned)max(0, ld_volatile_i32(p.ctl));
    const int lim = ld_volatile_i32(p.ctl + 1);
    if (lim > 0) bar_limit = lim;
  }
  tma_init(tp);
  dattn_init_bars(dbars);
  unsigned dpar = 0;   // attention: per-warp stage parities
  store_desc(0, load_desc(0));
  if (threadIdx.x == 0) s_ok = ld_volatile_i32(p.err) == 0;
  __syncthreads();
  if (!s_ok) return;   // an earlier pass gave up: nothing arrived, nothing issued
  unsigned cpar = 0;   // consumers: parity of each stage's next full-barrier completion
  unsigned gcount = 0, ecount = 0;   // tile groups handed over / finished (consumers / epilogue warp)
  int npre = 0;        // units of the current GEMM phase issued before its barrier
  for (int ph = 0; ph < p.nphases; ++ph) {
    const PhaseDesc& d = s_ph[ph & 1];
    const int next_word = ph + 1 < p.nphases ? load_desc(ph + 1) : 0;
    unsigned long long* const st = times ? times + 1 + kPhaseStamps * ph : nullptr;
    if (d.kind == kPhaseEmbed) {
      for (int t = blockIdx.x; t < d.e.ntok; t += gridDim.x) embed_token<bf16, false>(d.e, t);
    } else if (d.kind == kPhaseGemm) {
      // resident X copied in; 1/rms of an RMSNorm'd input (resident or streamed)
      if (d.xm == kXSmem || d.g.x_norm == 2) tma_prepare_x(d, tp, s_inv, xreg);
      if (st && threadIdx.x == 0) atomicMax(st + 3, global_ns());
      if (producer) {
        if (lane == 0) tma_produce(d, npre, tp, ring, maps);
        __syncwarp();
      } else if (epiw) {
        if (d.q4) tma_epilogue(d, tp, red, s_inv, ecount);
      } else if (d.q4) {
        if (d.xm == kXSmem)
          tma_consume_q4<true>(d, tp, cpar, gcount, ring, xreg, red, st ? st + 4 : nullptr);
        else
          tma_consume_q4<false>(d, tp, cpar, gcount, ring, xreg, red, st ? st + 4 : nullptr);
      } else if (d.xm == kXSmem) {
        tma_consume<true>(d, tp, cpar, ring, xreg, red, s_inv, st ? st + 4 : nullptr);
      } else {
        tma_consume<false>(d, tp, cpar, ring, xreg, red, s_inv, st ? st + 4 : nullptr);
      }
    } else if (warp < kCWarps) {   // attention: the eight consumer warps
      for (int it = blockIdx.x; it < d.attn_items; it += gridDim.x)
        dattn_item_mode<HD, kGroup, false>(d.a, it, dsm, &s_last, dbars, dpar, st ? st + 3 : nullptr);
      if (st && threadIdx.x == 0) atomicMax(st + 4, global_ns());
    }
    // this thread's global writes and shared-memory accesses are ordered
    // before later tensor copies (other CTAs' copies of X; this CTA's ring)
    npre = 0;
    fence_proxy_async_global();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (times) {   // arrival of this CTA (its threads are done with the phase)
      __syncthreads();
      if (threadIdx.x == 0) {
        const unsigned long long t = global_ns();
        atomicMax(st, ~t);
        atomicMax(st + 1, t);
      }
    }
    if (ph + 1 < p.nphases) {
      store_desc((ph + 1) & 1, next_word);
      grid_arrive(p.bar);   // its __syncthreads also ends this phase's shared-memory use
      if (threadIdx.x == 0 && tp.abort) atomicExch(p.err, 1);
      const PhaseDesc& nx = s_ph[(ph + 1) & 1];
      if (nx.kind == kPhaseGemm && producer) {   // weights of the next GEMM: issued while waiting
        if (lane == 0) npre = tma_prefetch(nx, tp, ring, maps);
        npre = __shfl_sync(0xffffffffu, npre, 0);
      }
      if (!grid_wait(p.bar, (unsigned)(ph + 1) * gridDim.x + bar_extra, p.err, &s_ok, bar_limit)) {
        tma_drain(tp);
        return;
      }
      if (st && blockIdx.x == 0 && threadIdx.x == 0) st[2] = global_ns();
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && tp.abort) atomicExch(p.err, 1);
  if (tp.abort) tma_drain(tp);
  grid_leave(p.bar, (unsigned)p.nphases * gridDim.x);
}

// ---- host side ----

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// Row-major bf16 matrix [rows][k] with row stride ld elements, boxes of
// box_rows x kTmaK; elements outside the matrix read as zero.
static bool encode_rows(TensorMap128& m, const void* base, int k, long long rows, long long ld, int box_rows) {
  static_assert(sizeof(CUtensorMap) == sizeof(TensorMap128), "tensor map size");
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc || !base || rows < 1 || (reinterpret_cast<uintptr_t>(base) & 15u) || (ld * 2) % 16 != 0) return false;
  cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)kTmaK, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(reinterpret_cast<CUtensorMap*>(&m), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
             dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-bit codes of a [rows][k] matrix (k/2 bytes per row), viewed as
// [k/256 blocks][rows][128 bytes]: boxes of 128 bytes x 8 rows x nblk blocks
// with the 128-byte swizzle (shared-memory layout [block][row][128 B]).
static bool encode_q4_codes(TensorMap128& m, const void* base, int k, long long rows, int nblk) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc || !base || rows < 1 || k % kTmaK || (reinterpret_cast<uintptr_t>(base) & 15u)) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)rows, (cuuint64_t)(k / kTmaK)};
  cuuint64_t strides[2] = {(cuuint64_t)k / 2, 128};
  cuuint32_t box[3] = {128, 8, (cuuint32_t)nblk};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(reinterpret_cast<CUtensorMap*>(&m), CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims,
             strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 scales of a [rows][k] q4 matrix stored group-major [k/64][rows]:
// boxes of 8 rows x ngrp groups (shared-memory layout [group][row]).
static bool encode_q4_scales(TensorMap128& m, const void* base, int k, long long rows, int ngrp) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc || !base || rows < 8 || rows % 8 || (reinterpret_cast<uintptr_t>(base) & 15u)) return false;
  cuuint64_t dims[2] = {(cuuint64_t)rows, (cuuint64_t)(k / 64)};
  cuuint64_t strides[1] = {(cuuint64_t)rows * 2};
  cuuint32_t box[2] = {8, (cuuint32_t)ngrp};
  cuuint32_t es[2] = {1, 1};
  return enc(reinterpret_cast<CUtensorMap*>(&m), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
             dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_kv_map(TensorMap128& m, const void* base, int hd, long long rows, int box_cols) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc || !base || rows < 1 || (hd != 32 && hd != 64 && hd != 128) ||
      (reinterpret_cast<uintptr_t>(base) & 15u))
    return false;
  const int cols = box_cols > 0 ? box_cols : (hd < 64 ? hd : 64);
  if (cols != 32 && cols != 64) return false;
  cuuint64_t dims[2] = {(cuuint64_t)hd, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)hd * 2};
  cuuint32_t box[2] = {(cuuint32_t)cols, (cuuint32_t)kDStepKeys};
  cuuint32_t es[2] = {1, 1};
  return enc(reinterpret_cast<CUtensorMap*>(&m), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
             dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             cols < 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Shared memory a GEMM phase's ring may fill: the ring region, and for a
// streamed-X phase the X region behind it as well (it holds no input then).
static size_t persist_ring_bytes(const PhaseDesc& p, const PersistLayout& lay) {
  return lay.ring + (p.xm == kXGlobal ? lay.xreg : 0);
}

// q4 phase (see tma_dev.cuh): tiles of two 8-row halves (plain matrices
// too); X resident when it fits (one tile x 4096 k per stage), else
// streamed (two tiles x 1024 k per stage).
static bool persist_phase_q4(PhaseDesc& p, const GemmDesc& g, std::vector<TensorMap128>& maps, int grid,
                             const PersistLayout& lay) {
  if (g.k % kTmaK) return false;
  p.q4 = 1;
  p.paired = 1;
  const size_t xbytes = (size_t)g.ntok * (g.k + kXPad) * 2;
  p.xm = xbytes <= lay.xreg ? kXSmem : kXGlobal;
  const int nct = std::min(grid, p.tiles);
  const int tiles_max = (p.tiles + nct - 1) / nct;
  p.gt = p.xm == kXSmem ? 1 : std::min(kMaxGroupTiles, tiles_max);
  // k per stage: a power of two (the steps split by shifts), at most 4096
  // (resident X) or 1024 (streamed X), at most k
  p.kc = p.xm == kXSmem ? 16 * kTmaK : 4 * kTmaK;
  while (p.kc > g.k) p.kc /= 2;
  if (p.kc < kTmaK) return false;
  const int nblk = p.kc / kTmaK, ngrp = p.kc / 64;
  p.tile_bytes = (2 * nblk * 1024 + 2 * ngrp * 16 + 1023) / 1024 * 1024;
  auto add2 = [&](const void* base, long long rows, int* mc, int* ms) {
    // codes [rows][k/2], then the scales, 16-byte aligned
    TensorMap128 a{}, b{};
    const unsigned char* sc = (const unsigned char*)base + (size_t)rows * g.k / 2;
    if (!encode_q4_codes(a, base, g.k, rows, nblk) || !encode_q4_scales(b, sc, g.k, rows, ngrp)) return false;
    maps.push_back(a);
    *mc = (int)maps.size() - 1;
    maps.push_back(b);
    *ms = (int)maps.size() - 1;
    return true;
  };
  bool ok = true;
  if (g.epi == kEpiQkvRope) {
    if (g.hd % 16 != 0) return false;
    for (int s = 0; s < 3; ++s) ok = ok && add2(g.w[s], g.seg_rows[s], &p.tm[s], &p.tms[s]);
  } else if (g.epi == kEpiSwiglu) {
    if (g.n % 8 != 0) return false;
    ok = add2(g.w[0], g.n, &p.tm[0], &p.tms[0]) && add2(g.w[1], g.n, &p.tm[1], &p.tms[1]);
    p.tm[2] = p.tm[0];
    p.tms[2] = p.tms[0];
  } else {
    if (g.n % 8 != 0) return false;
    ok = add2(g.w[0], g.n, &p.tm[0], &p.tms[0]);
    p.tm[1] = p.tm[2] = p.tm[0];
    p.tms[1] = p.tms[2] = p.tms[0];
  }
  if (!ok) return false;
  if (p.xm == kXGlobal) {
    TensorMap128 m{};
    if (!encode_rows(m, g.x, g.k, g.ntok, g.ldx, g.ntok)) return false;
    maps.push_back(m);
    p.tm[3] = (int)maps.size() - 1;
  }
  const int xstage = p.xm == kXGlobal ? nblk * g.ntok * kTmaRowBytes : 0;
  p.xoff = p.gt * p.tile_bytes;
  p.stage_bytes = (p.gt * p.tile_bytes + xstage + 1023) / 1024 * 1024;
  p.stages = std::min<int>(kMaxStages, (int)(persist_ring_bytes(p, lay) / (size_t)p.stage_bytes));
  if (p.stages < 2) return false;
  const int units_max = ((tiles_max + p.gt - 1) / p.gt) * ((g.k + p.kc - 1) / p.kc);
  p.prefetch = p.xm == kXSmem && units_max <= 8 ? std::min(p.stages, 2) : p.stages;
  return true;
}

bool persist_phase_from_gemm(PhaseDesc& p, const GemmDesc& g, std::vector<TensorMap128>& maps, int grid,
                             const PersistLayout& lay) {
  p = PhaseDesc{};
  p.kind = kPhaseGemm;
  p.g = g;
  if (g.k % 8 != 0 || g.ntok < 1 || g.ntok > kPersistMaxTok) return false;
  // an RMSNorm'd input comes pre-multiplied by its gain (x_norm = 2)
  if (g.x_norm == 1) return false;
  if (g.ldx % 8 != 0 || reinterpret_cast<uintptr_t>(g.x) % 16 != 0) return false;
  auto add = [&](const void* base, long long rows, long long ld, int box_rows) {
    TensorMap128 m{};
    if (!encode_rows(m, base, g.k, rows, ld, box_rows)) return -1;
    maps.push_back(m);
    return (int)maps.size() - 1;
  };
  p.tiles = gemm_tiles_of(g);
  if (g.q4) return persist_phase_q4(p, g, maps, grid, lay);
  if (g.epi == kEpiQkvRope) {
    if (g.hd % 16 != 0) return false;
    p.paired = 1;
    for (int s = 0; s < 3; ++s) p.tm[s] = add(g.w[s], g.seg_rows[s], g.k, 8);
  } else if (g.epi == kEpiSwiglu) {
    if (g.n % 8 != 0) return false;
    p.paired = 1;
    p.tm[0] = add(g.w[0], g.n, g.k, 8);
    p.tm[1] = add(g.w[1], g.n, g.k, 8);
    p.tm[2] = p.tm[0];
  } else {
    p.paired = 0;
    p.tm[0] = add(g.w[0], g.n, g.k, kTileRows);
    p.tm[1] = p.tm[2] = p.tm[0];
  }
  // X resident in shared memory when the ntok input rows fit the X region,
  // else streamed with the weights, one box of the ntok rows per 256 k
  const size_t xbytes = (size_t)g.ntok * (g.k + kXPad) * 2;
  p.xm = xbytes <= lay.xreg ? kXSmem : kXGlobal;
  const int nct = std::min(grid, p.tiles);
  const int tiles_max = (p.tiles + nct - 1) / nct;
  if (p.xm == kXSmem) {
    p.gt = 1;
    p.kc = 4 * kTmaK;
    p.tm[3] = 0;
  } else {
    p.gt = std::min(kMaxGroupTiles, tiles_max);
    p.kc = 4 * kTmaK / p.gt;
    p.tm[3] = add(g.x, g.ntok, g.ldx, g.ntok);
  }
  for (int i = 0; i < 4; ++i)
    if (p.tm[i] < 0) return false;
  const int xstage = p.xm == kXGlobal ? (p.kc / kTmaK) * g.ntok * kTmaRowBytes : 0;
  p.xoff = kStageWeightBytes;
  p.stage_bytes = (kStageWeightBytes + xstage + 1023) / 1024 * 1024;
  p.stages = std::min<int>(kMaxStages, (int)(persist_ring_bytes(p, lay) / (size_t)p.stage_bytes));
  if (p.stages < 2) return false;
  // units issued before the phase's barrier: a full ring, except that a
  // resident-X phase with few units per CTA takes only 3 ahead, so that its
  // X copies are not queued behind a ring of weight copies
  const int units_max = ((tiles_max + p.gt - 1) / p.gt) * ((g.k + p.kc - 1) / p.kc);
  p.prefetch = p.xm == kXSmem && units_max <= 16 ? std::min(p.stages, 3) : p.stages;
  return true;
}

bool persist_phase_from_attn(PhaseDesc& p, const AttnDesc& a) {
  p = PhaseDesc{};
  p.kind = kPhaseAttn;
  p.a = a;
  p.attn_items = dattn_items(a.ntok, a.hq, a.hkv, a.cap, a.hd);
  return a.dtype == 1 && a.ntok <= kPersistMaxTok && a.hq % a.hkv == 0 && a.tmk && a.tmv &&
         (a.hd == 32 || a.hd == 64 || a.hd == 128);
}

size_t persist_attn_partial_floats(int max_tok, int hq, int hd, int cap) {
  return (size_t)max_tok * hq * dattn_splits(cap) * (hd + 4);
}

void persist_phase_from_embed(PhaseDesc& p, const EmbedDesc& e) {
  p = PhaseDesc{};
  p.kind = kPhaseEmbed;
  p.e = e;
}

bool persist_layout(int hd, int max_tok, int d_model, PersistLayout* out) {
  size_t attn = 0;
  if (hd == 32) attn = DAttnSmem<32>::kBytes;
  if (hd == 64) attn = DAttnSmem<64>::kBytes;
  if (hd == 128) attn = DAttnSmem<128>::kBytes;
  if (!attn) return false;
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return false;
  // static shared memory of the kernel (the largest of its instances)
  size_t stat = 0;
  const void* fns[] = {(const void*)persist_forward<32, false>, (const void*)persist_forward<64, false>,
                       (const void*)persist_forward<128, false>, (const void*)persist_forward<32, true>,
                       (const void*)persist_forward<64, true>, (const void*)persist_forward<128, true>};
  for (const void* fn : fns) {
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) return false;
    stat = std::max(stat, fa.sharedSizeBytes);
  }
  const size_t budget = (size_t)optin > stat + 1024 ? (size_t)optin - stat - 1024 : 0;
  size_t xreg = ((size_t)max_tok * (d_model + kXPad) * 2 + 1023) / 1024 * 1024;
  xreg = std::max(xreg, kXMinBytes);
  if (budget < kRedBytes + xreg + 2 * (size_t)kStageWeightBytes) return false;
  const size_t ring = std::min(kRingMaxBytes, budget - kRedBytes - xreg) / 1024 * 1024;
  out->ring = ring;
  out->xreg = xreg;
  out->total = std::max(ring + kRedBytes + xreg, attn);
  return out->total <= budget;
}

// The dynamic shared-memory limit is a per-function attribute shared by
// every context of the process (a draft and a target with the same head
// dimension use the same instance): it only ever grows here.
template <int HD, bool kGroup>
static bool persist_fits_mode(size_t smem) {
  cudaFuncAttributes fa{};
  if (cudaFuncGetAttributes(&fa, persist_forward<HD, kGroup>) != cudaSuccess) return false;
  if ((size_t)fa.maxDynamicSharedSizeBytes < smem &&
      cudaFuncSetAttribute(persist_forward<HD, kGroup>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return false;
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, persist_forward<HD, kGroup>, kPersistThreads,
                                                    smem) != cudaSuccess)
    return false;
  return blocks >= 1;
}
template <int HD>
static bool persist_fits(size_t smem) {
  return persist_fits_mode<HD, false>(smem) && persist_fits_mode<HD, true>(smem);
}

bool persist_supported(int hd, size_t smem, int num_sms, int max_tok) {
  (void)num_sms;
  if (max_tok > kPersistMaxTok || !tensor_map_encoder()) return false;
  if (hd == 32) return persist_fits<32>(smem);
  if (hd == 64) return persist_fits<64>(smem);
  if (hd == 128) return persist_fits<128>(smem);
  return false;
}

template <int HD, bool kGroup>
static cudaError_t launch_persist_t(const PersistDesc& p, size_t smem, int num_sms, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);   // one CTA per SM, all co-resident
  cfg.blockDim = dim3(kPersistThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, persist_forward<HD, kGroup>, p);
}

template <int HD>
static cudaError_t launch_persist_hd(const PersistDesc& p, bool group, size_t smem, int num_sms, cudaStream_t st) {
  return group ? launch_persist_t<HD, true>(p, smem, num_sms, st) : launch_persist_t<HD, false>(p, smem, num_sms, st);
}

cudaError_t launch_persist(const PersistDesc& p, int hd, bool group, size_t smem, int num_sms, cudaStream_t st) {
  if (hd == 32) return launch_persist_hd<32>(p, group, smem, num_sms, st);
  if (hd == 64) return launch_persist_hd<64>(p, group, smem, num_sms, st);
  if (hd == 128) return launch_persist_hd<128>(p, group, smem, num_sms, st);
  return cudaErrorInvalidValue;
}

}  // namespace sv
