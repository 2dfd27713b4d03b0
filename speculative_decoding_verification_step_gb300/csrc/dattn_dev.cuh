// Decode / verify attention of the persistent forward kernel (at most 8
// query tokens, bf16 KV cache), on tensor cores.
//
// Work item = (KV head, token group, group of up to 8 of the KV head's
// query heads, key split, V part).  Its at most 8 rows are (token, head)
// pairs, tokens outer: min(G, 8) heads (G query heads per KV head) of one
// token, or -- once the pass's last position reaches 1024, where the keys
// no longer sit in L2 and re-reading them per token costs HBM bytes -- of
// 8 / min(G, 8) consecutive tokens (2 tokens x 4 heads for the 8B and 1B
// shapes), so one walk over the KV head's keys serves all of them.  Row r sees keys
// 0..p_r of its own position; keys past it are masked.  With head dim 64 or
// 128 an item reads all of K (the scores need every dim) but only its half
// of V, and writes its half of the output dims: each 16-dim block of P.V is
// its own MMA, so the two items of a row produce exactly the bits one item
// would, with 25% fewer bytes per CTA.  Keys are walked in absolute 16-key
// steps; step s belongs to consumer warp s mod 8.  A warp keeps, per row, an
// online softmax state over its steps (running max m, sum l, output o):
//   scores  S = K_step Q^T              (mma m16n8k16: keys x rows, k = dims)
//   m' = max(m, max_j S_j), scale = exp(m - m'), p_j = exp(S_j - m')
//   l  = l * scale + sum_j p_j,  o = o * scale + V_step^T p   (bf16 p)
// with K, Q, V and p in bf16 and fp32 accumulation; a step holding no key of
// a row leaves the row's state as it is (scale 1, p = 0).  The eight warp
// states are then merged in warp order: M = max_w m_w, out = sum_w e^(m_w -
// M) o_w / sum_w e^(m_w - M) l_w.  Keys are split in absolute 1024-key
// ranges; a row whose position spans several splits writes one (M, L, O)
// partial per split and the last split item of its token group to finish
// merges each row's splits in split order.  Every step of a row's
// arithmetic is fixed by its own position, so a row gets the same bits
// whichever rows share the item or the pass (batch invariance).
//
// Memory: per warp a pipeline of 3 (head dim 128) or 6 stages of 16-key K/V
// tiles, each filled by 2-D tensor copies (hardware-swizzled so the fragment
// loads and ldmatrix rows hit distinct banks) issued by the warp's lane 0 and
// completing on the stage's barrier, and a 16x8 probability tile; the warp
// merge reuses the same space.
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace sv {

constexpr int kDStepKeys = 16;
constexpr int kDSplitKeys = 1024;
constexpr int kDWarps = 8;
constexpr int kDRows = 8;                          // rows per item (MMA n)

template <int HD, int NT = 1>
struct DAttnSmem {
  // per warp: kDepth stages of a 16-key K tile and V tile, each tile written
  // by 2-D tensor copies of 16 keys x kBoxCols dims with the hardware 128-byte
  // (64-byte for head dim 32) swizzle, then the probability tile
  // [8 rows][16 keys]; warp regions stay 1 KB aligned (swizzle atoms)
  static constexpr int kDepth = HD >= 128 ? 3 : 6;
  static constexpr int kTileElems = kDStepKeys * HD;   // K tile
  static constexpr int kTileBytes = kTileElems * 2;
  static constexpr int kBoxCols = HD < 64 ? HD : 64;
  static constexpr int kBoxes = HD / kBoxCols;
  // V is read in kVParts column parts, one per item (head dim 128 / 64:
  // halves, copied as boxes of 64 / 32 dims with the 128- / 64-byte swizzle
  // -- every 16-dim block of the output is its own MMA, so an item needs all
  // of K for the scores but only its part of V)
  static constexpr int kVParts = HD >= 64 ? 2 : 1;
  static constexpr int kVDims = HD / kVParts;
  static constexpr int kVTileElems = kDStepKeys * kVDims;
  static constexpr int kVBoxCols = kVDims < 64 ? kVDims : 64;
  static constexpr int kVBoxes = kVDims / kVBoxCols;
  static constexpr int kStageElems = kTileElems + kVTileElems;   // K tile, then V tile
  // (the probabilities as a bf16 pair, high then low parts: 2 x NT tiles of
  // [8 rows][16 keys]; wide items have NT x 8 rows)
  static constexpr size_t kWarpRaw = (size_t)kDepth * kStageElems * 2 + 2 * NT * kDRows * kDStepKeys * 2;
  static constexpr size_t kWarpBytes = (kWarpRaw + 1023) / 1024 * 1024;
  // merge area: m, l [8 warps][8 NT rows], o [8 warps][8 NT rows][kVDims] (fp32)
  static constexpr size_t kMergeBytes = (size_t)kDWarps * NT * kDRows * (2 + kVDims) * 4;
  static constexpr size_t kBytes = kDWarps * kWarpBytes > kMergeBytes ? kDWarps * kWarpBytes : kMergeBytes;
  // element offset of logical 16-byte chunk c of key row r in a tile: box
  // c / 8 (64 dims), row r, chunk (c mod 8) XOR (r mod 8) -- the tensor
  // copy's 128-byte swizzle; for head dim 32, (c XOR (r / 2 mod 4)) in 64-byte
  // rows -- the 64-byte swizzle.  Eight consecutive rows read at one logical
  // chunk land in eight distinct bank groups.
  static __device__ __forceinline__ int at(int r, int c) {
    if (HD >= 64) return (c >> 3) * (kDStepKeys * 64) + r * 64 + (((c & 7) ^ (r & 7)) << 3);
    return r * HD + ((c ^ ((r >> 1) & 3)) << 3);
  }
  // the same for a V tile of kVDims dims
  static __device__ __forceinline__ int at_v(int r, int c) {
    if (kVDims >= 64) return (c >> 3) * (kDStepKeys * 64) + r * 64 + (((c & 7) ^ (r & 7)) << 3);
    return r * kVDims + ((c ^ ((r >> 1) & 3)) << 3);
  }
};
constexpr int kDMaxDepth = 6;
constexpr long long kDWaitLimit = 1LL << 22;

SV_DEV void ldmatrix_x4_trans(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(smem_u32(p)));
}

SV_DEV uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// A probability p as the bf16 pair (h, l) = (bf16(p), bf16(p - h)): h + l
// equals p to about 2^-17 relative, so P.V over both parts (two MMAs) keeps
// the probabilities at nearly fp32 precision -- rounding them to one bf16
// moves the logits of a 4096-wide model by up to ~0.05, and by an amount that
// depends on the running maximum each key was scaled by.
SV_DEV void store_prob(bf16* hi_tile, bf16* lo_tile, int idx, float p) {
  const bf16 h = __float2bfloat16_rn(p);
  hi_tile[idx] = h;
  lo_tile[idx] = __float2bfloat16_rn(p - __bfloat162float(h));
}

// Item geometry.
// Rows of an item are (token, head) pairs, tokens outer: hpi = min(G, 8)
// heads (G = query heads per KV head) of tpi consecutive tokens, tpi = 1 or
// 8 / hpi (see kDGroupMinPos), so one K/V walk serves every token of the group.
struct DItem {
  int kvh, tg, hg, split;
};
__host__ __device__ inline int dattn_hgroups(int hq, int hkv) { return (hq / hkv + kDRows - 1) / kDRows; }
__host__ __device__ inline int dattn_hpi(int hq, int hkv) { return hq / hkv < kDRows ? hq / hkv : kDRows; }
SV_DEV DItem dattn_item_of(const AttnDesc& a, int it, int hgroups, int tgroups) {
  DItem d;
  d.hg = it % hgroups;
  it /= hgroups;
  d.kvh = it % a.hkv;
  it /= a.hkv;
  d.tg = it % tgroups;
  d.split = it / tgroups;
  return d;
}
__host__ __device__ inline int dattn_splits(int cap) { return (cap + kDSplitKeys - 1) / kDSplitKeys; }
__host__ __device__ inline int dattn_vparts(int hd) { return hd >= 64 ? 2 : 1; }
// Columns of a V tensor-map box (its swizzle: 2 bytes x this).
__host__ __device__ inline int dattn_vbox_cols(int hd) {
  const int vd = hd / dattn_vparts(hd);
  return vd < 64 ? vd : 64;
}
// Items are enumerated as for one token per item (ntok token slots); with
// token groups the slots past the last group return at once.
__host__ __device__ inline int dattn_items(int ntok, int hq, int hkv, int cap, int hd) {
  return dattn_splits(cap) * ntok * hkv * dattn_hgroups(hq, hkv) * dattn_vparts(hd);
}

// Lane 0: the tensor copies of K step s (keys 16s .. 16s+15 of the rows of
// KV head row0 / cap; keys beyond the row's position are masked later, rows
// past the cache read as zero) and of V part vp of it into one stage,
// completing on bar.
template <int HD>
SV_DEV void dattn_fetch(const AttnDesc& a, int row0, int s, int vp, bf16* kt, bf16* vt, uint64_t* bar) {
  using L = DAttnSmem<HD>;
  mbar_arrive_expect_tx(bar, (unsigned)(L::kTileElems + L::kVTileElems) * 2u);
  const int r = row0 + s * kDStepKeys;
  const uint64_t pol = l2_evict_last();   // the cache is read again by every later pass
#pragma unroll
  for (int b = 0; b < L::kBoxes; ++b)
    tma_load_2d_hint(kt + b * kDStepKeys * L::kBoxCols, a.tmk, b * L::kBoxCols, r, bar, pol);
#pragma unroll
  for (int b = 0; b < L::kVBoxes; ++b)
    tma_load_2d_hint(vt + b * kDStepKeys * L::kVBoxCols, a.tmv, vp * L::kVDims + b * L::kVBoxCols, r, bar, pol);
}

// Bounded wait on a stage barrier; false (after raising *a.err) on timeout.
SV_DEV bool dattn_wait(const AttnDesc& a, uint64_t* bar, unsigned parity) {
  long long spins = 0;
  while (!mbar_test(bar, parity)) {
    if (++spins > kDWaitLimit) {
      if (a.err) atomicExch(a.err, 1);
      return false;
    }
  }
  return true;
}

// Stage barriers of the eight warps (kDMaxDepth each), initialised once per
// kernel by thread 0 before any item; dpar: per-warp parity bitmask of the
// next completion of each stage, carried from item to item.
SV_DEV void dattn_init_bars(uint64_t* bars) {
  if (threadIdx.x == 0) {
    for (int i = 0; i < kDWarps * kDMaxDepth; ++i) mbar_init(&bars[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
}

// One item; kGroup: token groups (8 / hpi tokens per item) rather than one
// token per item.  stamp (optional): atomicMax of the globaltimer when the
// key walk ended.
// kSeqs = false: single-sequence passes only (the persistent kernel).
template <int HD, bool kGroup, bool kSeqs>
SV_DEV void dattn_item_rows(const AttnDesc& a, int it, unsigned char* sm, int* s_last, uint64_t* bars,
                            unsigned& dpar, unsigned long long* stamp) {
  using L = DAttnSmem<HD>;
  constexpr int VD = L::kVDims;                       // output dims of this item
  const int vp = it % L::kVParts;                     // V part (fastest in the item order)
  const int hgroups = dattn_hgroups(a.hq, a.hkv);
  const DItem d = dattn_item_of(a, it / L::kVParts, hgroups, a.ntok);
  const int G = a.hq / a.hkv, hpi = dattn_hpi(a.hq, a.hkv);
  const int S = kSeqs && a.spt > 0 ? a.spt : a.ntok;  // tokens per sequence
  const int b = kSeqs ? d.tg / S : 0;                 // the item's sequence
  const int tpi = kGroup ? kDRows / hpi : 1;          // tokens per item
  const int j0 = (kSeqs ? d.tg % S : d.tg) * tpi;     // its first token within the sequence
  if (kGroup && j0 >= S) return;                      // token slot past the last group
  const int t0 = b * S + j0;                          // ... and within the pass
  // position of pass token t (of this sequence)
  const int pbase = kSeqs ? a.pos_base[(size_t)b * a.pos_ld] + a.pos_off - b * S : *a.pos_base + a.pos_off;
  // rows 0 .. nrows-1 are valid: row r = (token t0 + r / hpi, head h0 + r % hpi)
  const int nrows = kGroup ? min(tpi, S - j0) * min(hpi, G - d.hg * kDRows) : min(kDRows, G - d.hg * kDRows);
  const int pmax = pbase + t0 + (kGroup ? min(tpi, S - j0) - 1 : 0);
  const int k0 = d.split * kDSplitKeys;
  if (k0 > pmax) return;                              // split entirely in the future
  const int last = min(pmax, k0 + kDSplitKeys - 1);   // last key of this split
  const int nsplit = pmax / kDSplitKeys + 1;          // splits of the token group
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gi = lane >> 2, ci = lane & 3;
  const int h0 = d.kvh * G + d.hg * kDRows;           // first query head of the item
  const int row0 = ((kSeqs ? a.seq0 + b : 0) * a.hkv + d.kvh) * a.cap;   // first cache row of the KV head
  uint64_t* wbar = bars + warp * kDMaxDepth;
  // token of valid item row r, and its head
  auto row_tok = [&](int r) { return kGroup ? t0 + r / hpi : t0; };
  auto row_head = [&](int r) { return h0 + (kGroup ? r % hpi : r); };

  // Q fragments (rows = (token, head) pairs; dims in groups of GD, k-permuted
  // as in the GEMM): thread (g, c) holds row g, dims j*GD + c*GD/4 .. +GD/4-1
  // of every group j as TW bf16 pairs; MMA i of a group takes pairs 2i, 2i+1.
  constexpr int GD = HD < 64 ? HD : 64;
  constexpr int NG = HD / GD, TW = GD / 8, NM = GD / 16;
  uint32_t qf[NG][TW];
  {
    const bool ok = gi < nrows;
    const float* qp = a.q + ((size_t)(ok ? row_tok(gi) : t0) * a.hq + (ok ? row_head(gi) : h0)) * HD + ci * (GD / 4);
#pragma unroll
    for (int j = 0; j < NG; ++j) {
#pragma unroll
      for (int e = 0; e < TW / 2; ++e) {
        const float4 v = ok ? __ldcg(reinterpret_cast<const float4*>(qp + j * GD + 4 * e)) : make_float4(0.f, 0.f, 0.f, 0.f);
        qf[j][2 * e] = pack_bf16(v.x, v.y);
        qf[j][2 * e + 1] = pack_bf16(v.z, v.w);
      }
    }
  }

  // stage b of the warp: K tile at wb + b * kStageElems, V tile after it
  constexpr int D = L::kDepth;
  bf16* wb = reinterpret_cast<bf16*>(sm + (size_t)warp * L::kWarpBytes);
  bf16* ps = wb + D * L::kStageElems;                 // [8 rows][16 keys], high parts
  bf16* pl = ps + kDRows * kDStepKeys;                // low parts

  // this warp's steps: s = first + 8j, j < nst, kept D steps ahead in flight
  const int s_begin = k0 / kDStepKeys, s_end = last / kDStepKeys;
  const int first = s_begin + warp;
  const int nst = first <= s_end ? (s_end - first) / kDWarps + 1 : 0;
  float m_r[2] = {neg_inf(), neg_inf()}, l_r[2] = {0.f, 0.f};   // rows 2c, 2c+1
  float o[VD / 16][4];
#pragma unroll
  for (int mt = 0; mt < VD / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  // positions of rows 2c, 2c+1 (-1: empty row); keys past them are masked
  const bool rv0 = 2 * ci < nrows, rv1 = 2 * ci + 1 < nrows;
  const int p0 = rv0 ? pbase + row_tok(2 * ci) : -1;
  const int p1 = rv1 ? pbase + row_tok(2 * ci + 1) : -1;
  if (lane == 0) {
    // the region was last read and written through the generic proxy (the
    // previous item's merge, the previous phase)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    for (int j = 0; j < D && j < nst; ++j)
      dattn_fetch<HD>(a, row0, first + kDWarps * j, vp, wb + j * L::kStageElems,
                      wb + j * L::kStageElems + L::kTileElems, &wbar[j]);
  }
  // per-lane element offsets of the fragments (fixed for the whole walk)
  int koff_lo[NG][TW / 4], koff_hi[NG][TW / 4], voff[VD / 16];
#pragma unroll
  for (int jg = 0; jg < NG; ++jg)
#pragma unroll
    for (int e = 0; e < TW / 4; ++e) {
      const int c = jg * (GD / 8) + ci * (GD / 32) + e;   // logical 16-byte chunk
      koff_lo[jg][e] = L::at(gi, c);
      koff_hi[jg][e] = L::at(gi + 8, c);
    }
  {
    const int lrow = (lane & 7) + ((lane >> 4) << 3);   // key of this lane's ldmatrix row
    const int lchk = (lane >> 3) & 1;                   // 8-dim half of a 16-dim tile
#pragma unroll
    for (int mt = 0; mt < VD / 16; ++mt) voff[mt] = L::at_v(lrow, 2 * mt + lchk);
  }
  bool live = true;
  for (int j = 0; j < nst; ++j) {
    const int s = first + kDWarps * j;
    const int buf = j % D;
    const bf16* kt = wb + buf * L::kStageElems;
    const bf16* vt = kt + L::kTileElems;
    live = __all_sync(0xffffffffu, live && dattn_wait(a, &wbar[buf], (dpar >> buf) & 1u));
    dpar ^= 1u << buf;
    if (!live) continue;   // timed out: the rows of this item are not computed
    // scores: D[key g / g+8][row 2c / 2c+1]
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int jg = 0; jg < NG; ++jg) {
      uint32_t lo[TW], hi[TW];   // key rows g and g+8
#pragma unroll
      for (int e = 0; e < TW / 4; ++e) {
        const uint4 x = *reinterpret_cast<const uint4*>(kt + koff_lo[jg][e]);
        const uint4 y = *reinterpret_cast<const uint4*>(kt + koff_hi[jg][e]);
        lo[4 * e] = x.x; lo[4 * e + 1] = x.y; lo[4 * e + 2] = x.z; lo[4 * e + 3] = x.w;
        hi[4 * e] = y.x; hi[4 * e + 1] = y.y; hi[4 * e + 2] = y.z; hi[4 * e + 3] = y.w;
      }
#pragma unroll
      for (int i = 0; i < NM; ++i)
        mma_bf16_16816(sc, lo[2 * i], hi[2 * i], lo[2 * i + 1], hi[2 * i + 1], qf[jg][2 * i], qf[jg][2 * i + 1]);
    }
    const int key_lo = s * kDStepKeys + gi, key_hi = key_lo + 8;
    // one token per item: every row's last key is `last`
    const bool kl0 = kGroup ? key_lo <= p0 : rv0 && key_lo <= last;
    const bool kl1 = kGroup ? key_lo <= p1 : rv1 && key_lo <= last;
    const bool kh0 = kGroup ? key_hi <= p0 : rv0 && key_hi <= last;
    const bool kh1 = kGroup ? key_hi <= p1 : rv1 && key_hi <= last;
    float v00 = kl0 ? sc[0] * a.scale : neg_inf();   // row 2c, key g
    float v01 = kl1 ? sc[1] * a.scale : neg_inf();   // row 2c+1, key g
    float v10 = kh0 ? sc[2] * a.scale : neg_inf();   // row 2c, key g+8
    float v11 = kh1 ? sc[3] * a.scale : neg_inf();   // row 2c+1, key g+8
    // step max per row over the 16 keys (lanes sharing c)
    float mx0 = fmaxf(v00, v10), mx1 = fmaxf(v01, v11);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(m_r[0], mx0), mn1 = fmaxf(m_r[1], mx1);
    // no key of the row yet: its state stays (0, 0); a step past the row's
    // position has scale exp(0) = 1 and p = 0, so it leaves the state as is
    // (one token per item: a valid row has a key in every step, and
    // exp(-inf - finite) = 0 on its first)
    const float sc0 = (kGroup ? mn0 == neg_inf() : !rv0) ? 0.f : expf(m_r[0] - mn0);
    const float sc1 = (kGroup ? mn1 == neg_inf() : !rv1) ? 0.f : expf(m_r[1] - mn1);
    const float p00 = v00 == neg_inf() ? 0.f : expf(v00 - mn0);
    const float p10 = v10 == neg_inf() ? 0.f : expf(v10 - mn0);
    const float p01 = v01 == neg_inf() ? 0.f : expf(v01 - mn1);
    const float p11 = v11 == neg_inf() ? 0.f : expf(v11 - mn1);
    float ls0 = p00 + p10, ls1 = p01 + p11;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      ls0 += __shfl_xor_sync(0xffffffffu, ls0, off);
      ls1 += __shfl_xor_sync(0xffffffffu, ls1, off);
    }
    if (kGroup || rv0) {
      l_r[0] = l_r[0] * sc0 + ls0;
      m_r[0] = mn0;
    }
    if (kGroup || rv1) {
      l_r[1] = l_r[1] * sc1 + ls1;
      m_r[1] = mn1;
    }
    // probabilities as bf16 pairs, [row][key]
    store_prob(ps, pl, (2 * ci) * kDStepKeys + gi, p00);
    store_prob(ps, pl, (2 * ci + 1) * kDStepKeys + gi, p01);
    store_prob(ps, pl, (2 * ci) * kDStepKeys + gi + 8, p10);
    store_prob(ps, pl, (2 * ci + 1) * kDStepKeys + gi + 8, p11);
    __syncwarp();
    const uint32_t pb0 = *reinterpret_cast<const uint32_t*>(ps + gi * kDStepKeys + 2 * ci);
    const uint32_t pb1 = *reinterpret_cast<const uint32_t*>(ps + gi * kDStepKeys + 2 * ci + 8);
    const uint32_t pc0 = *reinterpret_cast<const uint32_t*>(pl + gi * kDStepKeys + 2 * ci);
    const uint32_t pc1 = *reinterpret_cast<const uint32_t*>(pl + gi * kDStepKeys + 2 * ci + 8);
    // o^T[dim][row] = o^T * scale + V^T p: A = V^T via transposing ldmatrix
#pragma unroll
    for (int mt = 0; mt < VD / 16; ++mt) {
      uint32_t va[4];
      ldmatrix_x4_trans(va, vt + voff[mt]);
      o[mt][0] *= sc0;
      o[mt][1] *= sc1;
      o[mt][2] *= sc0;
      o[mt][3] *= sc1;
      mma_bf16_16816(o[mt], va[0], va[1], va[2], va[3], pb0, pb1);
      mma_bf16_16816(o[mt], va[0], va[1], va[2], va[3], pc0, pc1);
    }
    __syncwarp();   // the stage and the probability tile are reused
    if (lane == 0 && j + D < nst) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // our reads before the copy's writes
      dattn_fetch<HD>(a, row0, s + kDWarps * D, vp, wb + buf * L::kStageElems,
                      wb + buf * L::kStageElems + L::kTileElems, &wbar[buf]);
    }
  }
  // after a timeout: let the copies still in flight land before the space is reused
  if (!live && lane == 0)
    for (int j = nst - D > 0 ? nst - D : 0; j < nst; ++j) {
      long long spins = 0;
      while (!mbar_test(&wbar[j % D], ((dpar >> (j % D)) & 1u) ^ 1u) && ++spins < (1LL << 16)) {
      }
    }
  __syncwarp();

  // ---- merge the eight warps (warp order) ----
  named_sync(1, kDWarps * 32);   // every warp is done with its buffers
  if (stamp && threadIdx.x == 0) {
    unsigned long long tm;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(tm));
    atomicMax(stamp, tm);
  }
  float* mm = reinterpret_cast<float*>(sm);          // [8 warps][8 rows]
  float* ll = mm + kDWarps * kDRows;                 // [8 warps][8 rows]
  float* oo = ll + kDWarps * kDRows;                 // [8 warps][8 rows][VD]
  if (gi == 0) {
    mm[warp * kDRows + 2 * ci] = m_r[0];
    mm[warp * kDRows + 2 * ci + 1] = m_r[1];
    ll[warp * kDRows + 2 * ci] = l_r[0];
    ll[warp * kDRows + 2 * ci + 1] = l_r[1];
  }
#pragma unroll
  for (int mt = 0; mt < VD / 16; ++mt) {
    float* ow = oo + (size_t)warp * kDRows * VD;
    ow[(2 * ci) * VD + mt * 16 + gi] = o[mt][0];
    ow[(2 * ci + 1) * VD + mt * 16 + gi] = o[mt][1];
    ow[(2 * ci) * VD + mt * 16 + gi + 8] = o[mt][2];
    ow[(2 * ci + 1) * VD + mt * 16 + gi + 8] = o[mt][3];
  }
  named_sync(1, kDWarps * 32);
  const int tid = threadIdx.x;
  const int dv0 = vp * VD;                           // first output dim of this item
  const int ns = dattn_splits(a.cap);
  // a split partial: [HD dims][M, L of V part 0][M, L of V part 1]
  for (int e = tid; e < nrows * VD; e += kDWarps * 32) {
    const int r = e / VD, dm = e % VD;
    const int t = row_tok(r);
    if (kGroup && pbase + t < k0) continue;          // no key of the row in this split
    float M = neg_inf();
#pragma unroll
    for (int w = 0; w < kDWarps; ++w) M = fmaxf(M, mm[w * kDRows + r]);
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int w = 0; w < kDWarps; ++w) {
      const float mw = mm[w * kDRows + r];
      const float f = mw == neg_inf() ? 0.f : expf(mw - M);
      num = fmaf(f, oo[((size_t)w * kDRows + r) * VD + dm], num);
      den = fmaf(f, ll[w * kDRows + r], den);
    }
    const int h = row_head(r);
    if (nsplit == 1) {
      ((bf16*)a.out)[(size_t)t * a.hq * HD + (size_t)h * HD + dv0 + dm] = __float2bfloat16_rn(num / den);
    } else {
      float* pp = a.partials + (((size_t)t * a.hq + h) * ns + d.split) * (HD + 4);
      pp[dv0 + dm] = num;
      if (dm == 0) {
        pp[HD + 2 * vp] = M;
        pp[HD + 2 * vp + 1] = den;
      }
    }
  }
  if (nsplit == 1) {
    named_sync(1, kDWarps * 32);   // the merge area is reused by the next item
    return;
  }
  // ---- several splits: the last one of the token group (and V part) to
  // finish merges each row's splits 0 .. p_r / 1024 in split order ----
  int* ticket = a.tickets + (((size_t)d.tg * a.hkv + d.kvh) * hgroups + d.hg) * L::kVParts + vp;
  named_sync(1, kDWarps * 32);
  if (tid == 0)   // acq_rel: publishes this split's partial, acquires the earlier ones
    *s_last = (atom_add_acq_rel_gpu(reinterpret_cast<unsigned*>(ticket), 1u) == (unsigned)nsplit - 1);
  named_sync(1, kDWarps * 32);
  if (!*s_last) return;
  for (int e = tid; e < nrows * VD; e += kDWarps * 32) {
    const int r = e / VD, dm = e % VD;
    const int t = row_tok(r);
    const int nr = (pbase + t) / kDSplitKeys + 1;    // the row's own splits
    const int h = row_head(r);
    const float* base = a.partials + ((size_t)t * a.hq + h) * ns * (HD + 4);
    float M = neg_inf();
    for (int sp = 0; sp < nr; ++sp) M = fmaxf(M, __ldcg(base + (size_t)sp * (HD + 4) + HD + 2 * vp));
    float num = 0.f, den = 0.f;
    for (int sp = 0; sp < nr; ++sp) {
      const float* pp = base + (size_t)sp * (HD + 4);
      const float f = expf(__ldcg(pp + HD + 2 * vp) - M);
      num = fmaf(f, __ldcg(pp + dv0 + dm), num);
      den = fmaf(f, __ldcg(pp + HD + 2 * vp + 1), den);
    }
    ((bf16*)a.out)[(size_t)t * a.hq * HD + (size_t)h * HD + dv0 + dm] = __float2bfloat16_rn(num / den);
  }
  named_sync(1, kDWarps * 32);
  if (tid == 0) *ticket = 0;
}

// Item it of an attention phase in a fixed grouping mode (the persistent
// kernel is instantiated per mode and the host picks it per pass).
template <int HD, bool kGroup, bool kSeqs>
SV_DEV void dattn_item_mode(const AttnDesc& a, int it, unsigned char* sm, int* s_last, uint64_t* bars,
                            unsigned& dpar, unsigned long long* stamp = nullptr) {
  dattn_item_rows<HD, kGroup, kSeqs>(a, it, sm, s_last, bars, dpar, stamp);
}

// Item it of an attention phase: token groups once the last position of the
// item's sequence in the pass reaches kDGroupMinPos, or when the pass asks for
// them (a.group: batched passes with items for several waves of CTAs, where
// half as many walks beats more parallel ones), else one token per item (the
// items of a sequence all take the same mode).
template <int HD>
SV_DEV void dattn_item(const AttnDesc& a, int it, unsigned char* sm, int* s_last, uint64_t* bars,
                       unsigned& dpar, unsigned long long* stamp = nullptr) {
  using L = DAttnSmem<HD>;
  const int S = a.spt > 0 ? a.spt : a.ntok;
  const int b = dattn_item_of(a, it / L::kVParts, dattn_hgroups(a.hq, a.hkv), a.ntok).tg / S;
  if (a.group || a.pos_base[(size_t)b * a.pos_ld] + a.pos_off + S - 1 >= kDGroupMinPos)
    dattn_item_rows<HD, true, true>(a, it, sm, s_last, bars, dpar, stamp);
  else
    dattn_item_rows<HD, false, true>(a, it, sm, s_last, bars, dpar, stamp);
}

// ---- wide items (batched passes of the per-operation kernel) ----
// Item = (sequence, group of tpi = 8 NT / G of its tokens, KV head, 1024-key
// split, V part) with NT n-tiles of 8 rows: all G query heads of tpi tokens
// (G <= 8), so one K/V tile in shared memory serves 8 NT rows -- each step's
// K fragments feed NT score MMAs and each V fragment NT P.V MMAs.  A row's
// arithmetic is step for step that of the one-tile items (the same MMAs,
// softmax updates and merges on its own column), so its bits do not depend
// on the item width.
__host__ __device__ inline int dattn_wide_tpi(int nt, int hq, int hkv) { return nt * kDRows / (hq / hkv); }
__host__ __device__ inline int dattn_items_wide(int nt, int ntok, int spt, int hq, int hkv, int cap, int hd) {
  const int S = spt > 0 ? spt : ntok, tpi = dattn_wide_tpi(nt, hq, hkv);
  return dattn_splits(cap) * (ntok / S) * ((S + tpi - 1) / tpi) * hkv * dattn_vparts(hd);
}

template <int HD, int NT>
SV_DEV void dattn_item_wide(const AttnDesc& a, int it, unsigned char* sm, int* s_last, uint64_t* bars,
                            unsigned& dpar) {
  using L = DAttnSmem<HD, NT>;
  constexpr int VD = L::kVDims;                       // output dims of this item
  constexpr int R = NT * kDRows;                      // rows of the item
  const int vp = it % L::kVParts;
  const int G = a.hq / a.hkv;                         // heads per KV head (<= 8): hpi
  const int S = a.spt > 0 ? a.spt : a.ntok;           // tokens per sequence
  const int tpi = R / G, gps = (S + tpi - 1) / tpi;   // tokens per item, groups per sequence
  const DItem d = dattn_item_of(a, it / L::kVParts, 1, (a.ntok / S) * gps);
  const int b = d.tg / gps, j0 = (d.tg % gps) * tpi;
  const int t0 = b * S + j0, ntk = min(tpi, S - j0);
  const int pbase = a.pos_base[(size_t)b * a.pos_ld] + a.pos_off - b * S;
  const int nrows = ntk * G;
  const int pmax = pbase + t0 + ntk - 1;
  const int k0 = d.split * kDSplitKeys;
  if (k0 > pmax) return;                              // split entirely in the future
  const int last = min(pmax, k0 + kDSplitKeys - 1);
  const int nsplit = pmax / kDSplitKeys + 1;          // splits of the token group
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gi = lane >> 2, ci = lane & 3;
  const int h0 = d.kvh * G;
  const int row0 = ((a.seq0 + b) * a.hkv + d.kvh) * a.cap;
  uint64_t* wbar = bars + warp * kDMaxDepth;
  auto row_tok = [&](int r) { return t0 + r / G; };
  auto row_head = [&](int r) { return h0 + r % G; };

  constexpr int GD = HD < 64 ? HD : 64;
  constexpr int NG = HD / GD, TW = GD / 8, NM = GD / 16;
  uint32_t qf[NT][NG][TW];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int r = nt * kDRows + gi;
    const bool ok = r < nrows;
    const float* qp = a.q + ((size_t)(ok ? row_tok(r) : t0) * a.hq + (ok ? row_head(r) : h0)) * HD + ci * (GD / 4);
#pragma unroll
    for (int j = 0; j < NG; ++j) {
#pragma unroll
      for (int e = 0; e < TW / 2; ++e) {
        const float4 v = ok ? __ldcg(reinterpret_cast<const float4*>(qp + j * GD + 4 * e)) : make_float4(0.f, 0.f, 0.f, 0.f);
        qf[nt][j][2 * e] = pack_bf16(v.x, v.y);
        qf[nt][j][2 * e + 1] = pack_bf16(v.z, v.w);
      }
    }
  }

  constexpr int D = L::kDepth;
  bf16* wb = reinterpret_cast<bf16*>(sm + (size_t)warp * L::kWarpBytes);
  bf16* ps = wb + D * L::kStageElems;                 // [NT][8 rows][16 keys], high parts
  bf16* pl = ps + NT * kDRows * kDStepKeys;           // low parts
  const int s_begin = k0 / kDStepKeys, s_end = last / kDStepKeys;
  const int first = s_begin + warp;
  const int nst = first <= s_end ? (s_end - first) / kDWarps + 1 : 0;
  float m_r[NT][2], l_r[NT][2], o[VD / 16][NT][4];
  int p0[NT], p1[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_r[nt][0] = m_r[nt][1] = neg_inf();
    l_r[nt][0] = l_r[nt][1] = 0.f;
    const int ra = nt * kDRows + 2 * ci;
    p0[nt] = ra < nrows ? pbase + row_tok(ra) : -1;
    p1[nt] = ra + 1 < nrows ? pbase + row_tok(ra + 1) : -1;
#pragma unroll
    for (int mt = 0; mt < VD / 16; ++mt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
  }
  if (lane == 0) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // after generic-proxy use
    for (int j = 0; j < D && j < nst; ++j)
      dattn_fetch<HD>(a, row0, first + kDWarps * j, vp, wb + j * L::kStageElems,
                      wb + j * L::kStageElems + L::kTileElems, &wbar[j]);
  }
  int koff_lo[NG][TW / 4], koff_hi[NG][TW / 4], voff[VD / 16];
#pragma unroll
  for (int jg = 0; jg < NG; ++jg)
#pragma unroll
    for (int e = 0; e < TW / 4; ++e) {
      const int c = jg * (GD / 8) + ci * (GD / 32) + e;
      koff_lo[jg][e] = L::at(gi, c);
      koff_hi[jg][e] = L::at(gi + 8, c);
    }
  {
    const int lrow = (lane & 7) + ((lane >> 4) << 3);
    const int lchk = (lane >> 3) & 1;
#pragma unroll
    for (int mt = 0; mt < VD / 16; ++mt) voff[mt] = L::at_v(lrow, 2 * mt + lchk);
  }
  bool live = true;
  for (int j = 0; j < nst; ++j) {
    const int s = first + kDWarps * j;
    const int buf = j % D;
    const bf16* kt = wb + buf * L::kStageElems;
    const bf16* vt = kt + L::kTileElems;
    live = __all_sync(0xffffffffu, live && dattn_wait(a, &wbar[buf], (dpar >> buf) & 1u));
    dpar ^= 1u << buf;
    if (!live) continue;
    float sc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int jg = 0; jg < NG; ++jg) {
      uint32_t lo[TW], hi[TW];
#pragma unroll
      for (int e = 0; e < TW / 4; ++e) {
        const uint4 x = *reinterpret_cast<const uint4*>(kt + koff_lo[jg][e]);
        const uint4 y = *reinterpret_cast<const uint4*>(kt + koff_hi[jg][e]);
        lo[4 * e] = x.x; lo[4 * e + 1] = x.y; lo[4 * e + 2] = x.z; lo[4 * e + 3] = x.w;
        hi[4 * e] = y.x; hi[4 * e + 1] = y.y; hi[4 * e + 2] = y.z; hi[4 * e + 3] = y.w;
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < NM; ++i)
          mma_bf16_16816(sc[nt], lo[2 * i], hi[2 * i], lo[2 * i + 1], hi[2 * i + 1], qf[nt][jg][2 * i],
                         qf[nt][jg][2 * i + 1]);
    }
    const int key_lo = s * kDStepKeys + gi, key_hi = key_lo + 8;
    float scl[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float v00 = key_lo <= p0[nt] ? sc[nt][0] * a.scale : neg_inf();
      const float v01 = key_lo <= p1[nt] ? sc[nt][1] * a.scale : neg_inf();
      const float v10 = key_hi <= p0[nt] ? sc[nt][2] * a.scale : neg_inf();
      const float v11 = key_hi <= p1[nt] ? sc[nt][3] * a.scale : neg_inf();
      float mx0 = fmaxf(v00, v10), mx1 = fmaxf(v01, v11);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      const float mn0 = fmaxf(m_r[nt][0], mx0), mn1 = fmaxf(m_r[nt][1], mx1);
      const float sc0 = mn0 == neg_inf() ? 0.f : expf(m_r[nt][0] - mn0);
      const float sc1 = mn1 == neg_inf() ? 0.f : expf(m_r[nt][1] - mn1);
      const float p00 = v00 == neg_inf() ? 0.f : expf(v00 - mn0);
      const float p10 = v10 == neg_inf() ? 0.f : expf(v10 - mn0);
      const float p01 = v01 == neg_inf() ? 0.f : expf(v01 - mn1);
      const float p11 = v11 == neg_inf() ? 0.f : expf(v11 - mn1);
      float ls0 = p00 + p10, ls1 = p01 + p11;
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        ls0 += __shfl_xor_sync(0xffffffffu, ls0, off);
        ls1 += __shfl_xor_sync(0xffffffffu, ls1, off);
      }
      l_r[nt][0] = l_r[nt][0] * sc0 + ls0;
      m_r[nt][0] = mn0;
      l_r[nt][1] = l_r[nt][1] * sc1 + ls1;
      m_r[nt][1] = mn1;
      scl[nt][0] = sc0;
      scl[nt][1] = sc1;
      bf16* pt = ps + nt * kDRows * kDStepKeys;
      bf16* qt = pl + nt * kDRows * kDStepKeys;
      store_prob(pt, qt, (2 * ci) * kDStepKeys + gi, p00);
      store_prob(pt, qt, (2 * ci + 1) * kDStepKeys + gi, p01);
      store_prob(pt, qt, (2 * ci) * kDStepKeys + gi + 8, p10);
      store_prob(pt, qt, (2 * ci + 1) * kDStepKeys + gi + 8, p11);
    }
    __syncwarp();
    uint32_t pb0[NT], pb1[NT], pc0[NT], pc1[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const bf16* pt = ps + nt * kDRows * kDStepKeys;
      const bf16* qt = pl + nt * kDRows * kDStepKeys;
      pb0[nt] = *reinterpret_cast<const uint32_t*>(pt + gi * kDStepKeys + 2 * ci);
      pb1[nt] = *reinterpret_cast<const uint32_t*>(pt + gi * kDStepKeys + 2 * ci + 8);
      pc0[nt] = *reinterpret_cast<const uint32_t*>(qt + gi * kDStepKeys + 2 * ci);
      pc1[nt] = *reinterpret_cast<const uint32_t*>(qt + gi * kDStepKeys + 2 * ci + 8);
    }
#pragma unroll
    for (int mt = 0; mt < VD / 16; ++mt) {
      uint32_t va[4];
      ldmatrix_x4_trans(va, vt + voff[mt]);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        o[mt][nt][0] *= scl[nt][0];
        o[mt][nt][1] *= scl[nt][1];
        o[mt][nt][2] *= scl[nt][0];
        o[mt][nt][3] *= scl[nt][1];
        mma_bf16_16816(o[mt][nt], va[0], va[1], va[2], va[3], pb0[nt], pb1[nt]);
        mma_bf16_16816(o[mt][nt], va[0], va[1], va[2], va[3], pc0[nt], pc1[nt]);
      }
    }
    __syncwarp();
    if (lane == 0 && j + D < nst) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      dattn_fetch<HD>(a, row0, s + kDWarps * D, vp, wb + buf * L::kStageElems,
                      wb + buf * L::kStageElems + L::kTileElems, &wbar[buf]);
    }
  }
  if (!live && lane == 0)
    for (int j = nst - D > 0 ? nst - D : 0; j < nst; ++j) {
      long long spins = 0;
      while (!mbar_test(&wbar[j % D], ((dpar >> (j % D)) & 1u) ^ 1u) && ++spins < (1LL << 16)) {
      }
    }
  __syncwarp();

  // ---- merge the eight warps (warp order) ----
  named_sync(1, kDWarps * 32);
  float* mm = reinterpret_cast<float*>(sm);          // [8 warps][R rows]
  float* ll = mm + kDWarps * R;                      // [8 warps][R rows]
  float* oo = ll + kDWarps * R;                      // [8 warps][R rows][VD]
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int ra = nt * kDRows + 2 * ci;
    if (gi == 0) {
      mm[warp * R + ra] = m_r[nt][0];
      mm[warp * R + ra + 1] = m_r[nt][1];
      ll[warp * R + ra] = l_r[nt][0];
      ll[warp * R + ra + 1] = l_r[nt][1];
    }
    float* ow = oo + (size_t)warp * R * VD;
#pragma unroll
    for (int mt = 0; mt < VD / 16; ++mt) {
      ow[ra * VD + mt * 16 + gi] = o[mt][nt][0];
      ow[(ra + 1) * VD + mt * 16 + gi] = o[mt][nt][1];
      ow[ra * VD + mt * 16 + gi + 8] = o[mt][nt][2];
      ow[(ra + 1) * VD + mt * 16 + gi + 8] = o[mt][nt][3];
    }
  }
  named_sync(1, kDWarps * 32);
  const int tid = threadIdx.x;
  const int dv0 = vp * VD;
  const int ns = dattn_splits(a.cap);
  for (int e = tid; e < nrows * VD; e += kDWarps * 32) {
    const int r = e / VD, dm = e % VD;
    const int t = row_tok(r);
    if (pbase + t < k0) continue;                    // no key of the row in this split
    float M = neg_inf();
#pragma unroll
    for (int w = 0; w < kDWarps; ++w) M = fmaxf(M, mm[w * R + r]);
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int w = 0; w < kDWarps; ++w) {
      const float mw = mm[w * R + r];
      const float f = mw == neg_inf() ? 0.f : expf(mw - M);
      num = fmaf(f, oo[((size_t)w * R + r) * VD + dm], num);
      den = fmaf(f, ll[w * R + r], den);
    }
    const int h = row_head(r);
    if (nsplit == 1) {
      ((bf16*)a.out)[(size_t)t * a.hq * HD + (size_t)h * HD + dv0 + dm] = __float2bfloat16_rn(num / den);
    } else {
      float* pp = a.partials + (((size_t)t * a.hq + h) * ns + d.split) * (HD + 4);
      pp[dv0 + dm] = num;
      if (dm == 0) {
        pp[HD + 2 * vp] = M;
        pp[HD + 2 * vp + 1] = den;
      }
    }
  }
  if (nsplit == 1) {
    named_sync(1, kDWarps * 32);
    return;
  }
  int* ticket = a.tickets + ((size_t)d.tg * a.hkv + d.kvh) * L::kVParts + vp;
  named_sync(1, kDWarps * 32);
  if (tid == 0)
    *s_last = (atom_add_acq_rel_gpu(reinterpret_cast<unsigned*>(ticket), 1u) == (unsigned)nsplit - 1);
  named_sync(1, kDWarps * 32);
  if (!*s_last) return;
  for (int e = tid; e < nrows * VD; e += kDWarps * 32) {
    const int r = e / VD, dm = e % VD;
    const int t = row_tok(r);
    const int nr = (pbase + t) / kDSplitKeys + 1;
    const int h = row_head(r);
    const float* base = a.partials + ((size_t)t * a.hq + h) * ns * (HD + 4);
    float M = neg_inf();
    for (int sp = 0; sp < nr; ++sp) M = fmaxf(M, __ldcg(base + (size_t)sp * (HD + 4) + HD + 2 * vp));
    float num = 0.f, den = 0.f;
    for (int sp = 0; sp < nr; ++sp) {
      const float* pp = base + (size_t)sp * (HD + 4);
      const float f = expf(__ldcg(pp + HD + 2 * vp) - M);
      num = fmaf(f, __ldcg(pp + dv0 + dm), num);
      den = fmaf(f, __ldcg(pp + HD + 2 * vp + 1), den);
    }
    ((bf16*)a.out)[(size_t)t * a.hq * HD + (size_t)h * HD + dv0 + dm] = __float2bfloat16_rn(num / den);
  }
  named_sync(1, kDWarps * 32);
  if (tid == 0) *ticket = 0;
}

}  // namespace sv
