// Shared device helpers of the GB300 speculative-verification library.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>

#define SV_DEV __device__ __forceinline__

namespace sv {

typedef __nv_bfloat16 bf16;

constexpr int kWarp = 32;
SV_DEV float neg_inf() { return __int_as_float(0xff800000u); }

// ---------------------------------------------------------------------------
// Philox-4x32-10, restated from its published definition (Salmon, Moraes,
// Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11): ten
// rounds; each multiplies counter words 0 and 2 by two odd constants, XORs
// the high halves with words 1 and 3 and the round key, keeps the low halves,
// and bumps the key by two Weyl increments.
//
// Draw layout of the speculative step: key = (seed lo, seed hi), counter =
// (step, position, stream, row), uniform = (word0 >> 8) * 2^-24 in [0, 1).
// ---------------------------------------------------------------------------
enum Stream : uint32_t { kStreamDraft = 0, kStreamAccept = 1, kStreamResidual = 2,
                         kStreamBonus = 3, kStreamAR = 4 };

SV_DEV uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
    k.x += 0x9E3779B9u;
    k.y += 0xBB67AE85u;
  }
  return c;
}

SV_DEV float philox_uniform(uint64_t seed, uint32_t step, uint32_t position, uint32_t stream,
                            uint32_t row) {
  const uint4 o = philox4x32_10(make_uint4(step, position, stream, row),
                                make_uint2((uint32_t)seed, (uint32_t)(seed >> 32)));
  return (float)(o.x >> 8) * (1.0f / 16777216.0f);
}

// ---------------------------------------------------------------------------
// Element helpers
// ---------------------------------------------------------------------------
SV_DEV float to_f32(float x) { return x; }
SV_DEV float to_f32(bf16 x) { return __bfloat162float(x); }
template <typename T> SV_DEV T from_f32(float x);
template <> SV_DEV float from_f32<float>(float x) { return x; }
template <> SV_DEV bf16 from_f32<bf16>(float x) { return __float2bfloat16_rn(x); }

// Two bf16 packed in one 32-bit word (low half first) -> floats.
SV_DEV float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
SV_DEV float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Streaming 128-bit load of weights: read once per launch, do not keep in L1.
SV_DEV uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// Warp-level tensor-core MMA m16n8k16, bf16 inputs, fp32 accumulate.
SV_DEV void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                           uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The same, not volatile (a pure function of its operands: the compiler may
// interleave independent MMA chains), with the accumulator (_acc) or a zero
// accumulator input (_z, d = A.B).
SV_DEV void mma_bf16_16816_acc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                               uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
SV_DEV void mma_bf16_16816_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                             uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

SV_DEV float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
SV_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

SV_DEV float silu(float x) { return x / (1.0f + expf(-x)); }

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel is launched with programmatic
// stream serialisation, so it may start while its predecessor in the stream
// is still running.  pdl_trigger() (called on entry) lets the successor
// launch; pdl_wait() blocks until the predecessor grid has completed and its
// memory is visible.  A kernel touches no output of an earlier kernel, and
// writes nothing, before pdl_wait(); the weight GEMM issues its first
// read-only weight loads before it, overlapping its ramp-up with the tail of
// the previous kernel.  Both are no-ops without a programmatic dependency.
// ---------------------------------------------------------------------------
SV_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
SV_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

bool pdl_enabled();
void set_pdl_enabled(bool on);

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------------------
// GPU-scope atomics with explicit ordering (cheaper than a full fence plus a
// relaxed atomic).  An acq_rel add publishes the calling thread's earlier
// writes (and, through a preceding CTA or warp barrier, those of its peers)
// and makes the writes published by earlier adders visible to it.
// ---------------------------------------------------------------------------
SV_DEV unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
SV_DEV void red_add_release_gpu(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
SV_DEV void st_relaxed_gpu(unsigned* p, unsigned v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---------------------------------------------------------------------------
// Asynchronous bulk copies and shared-memory barriers (sm_90 and later).
// A transaction barrier completes its phase when its expected arrivals have
// arrived and the bytes announced with expect_tx have landed.
// ---------------------------------------------------------------------------
SV_DEV unsigned smem_u32(const void* p) { return (unsigned)__cvta_generic_to_shared(p); }

SV_DEV void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// One arrival that also announces `bytes` of copies completing on the barrier.
SV_DEV void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
SV_DEV void mbar_arrive_count(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
SV_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// True once the phase of the given parity has completed (one bounded probe).
SV_DEV bool mbar_test(uint64_t* bar, unsigned parity) {
  unsigned done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(done) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return done != 0;
}
// Contiguous global -> shared copy of `bytes` (multiple of 16, both addresses
// 16-byte aligned) through the asynchronous copy engine, completing on bar.
SV_DEV void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
// Tensor copy of one 3-D box (coordinates innermost first) into shared
// memory, completing on bar, with an L2 cache policy.
SV_DEV void tma_load_3d_hint(void* dst, const void* tmap, int c0, int c1, int c2, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)),
        "l"(policy)
      : "memory");
}
// Tensor copy of one 2-D box (coordinates: inner element, row) described by
// the tensor map at global address tmap into shared memory (128-byte
// aligned), completing on bar.  Elements outside the tensor are zero-filled;
// the barrier is credited with the full box size.
SV_DEV void tma_load_2d(void* dst, const void* tmap, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}
// L2 eviction-priority policies for the cache_hint form below: data read once
// per pass (streamed weights) is evicted first, data read again soon (the KV
// cache, activations) last.
SV_DEV uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
SV_DEV uint64_t l2_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// tma_load_2d with an L2 cache policy.
SV_DEV void tma_load_2d_hint(void* dst, const void* tmap, int c0, int c1, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(smem_u32(bar)),
        "l"(policy)
      : "memory");
}
// Prefetch of one 2-D box of the tensor map at tmap into L2 (no shared
// memory, no barrier; completes on its own).
SV_DEV void tma_prefetch_l2_2d(const void* tmap, int c0, int c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
               ::"l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1) : "memory");
}
// 16-byte asynchronous global -> shared copy (L2 only); with valid = false
// nothing is read and the destination is zero-filled.
SV_DEV void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0) : "memory");
}
SV_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
SV_DEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
// Load that bypasses the L1 and any earlier cached copy (a flag written by
// an earlier kernel or another CTA).
SV_DEV int ld_volatile_i32(const int32_t* p) { return *reinterpret_cast<const volatile int32_t*>(p); }
// Orders this thread's earlier generic-proxy global accesses with its later
// bulk-copy (async-proxy) accesses, and the reverse.
SV_DEV void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
// Barrier over the first `threads` threads of the CTA (id 1..15).
SV_DEV void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace sv
