// Per-layer kernels of the decoder forward other than the weight GEMMs:
// embedding gather, RMSNorm, RoPE + KV-cache append, and causal attention of
// the new positions over the KV cache.
//
// The target pass computes a next-token distribution at each of the K+1 new
// positions in one forward ("Speculative decoding internals", 演算法核心
// Step 2: T_1 = T(.|x) ... T_{K+1} = T(.|x, d_1..K)); position L+j attends to
// keys 0..L+j.  Rolling back a rejected suffix is a length truncation: the
// stale KV rows beyond the committed length are never read (each query only
// reads keys at or before its own position) and are overwritten later.
#include "attn_dev.cuh"
#include "dattn_dev.cuh"
#include "embed_dev.cuh"

namespace sv {

// ---------------------------------------------------------------- embedding
// One CTA per token (device code: embed_dev.cuh).
template <typename T>
__global__ void embed_kernel(const __grid_constant__ EmbedDesc e) {
  pdl_trigger();
  pdl_wait();
  embed_token<T>(e, blockIdx.x);
}

cudaError_t launch_embed(const EmbedDesc& e, cudaStream_t st) {
  if (e.d % 16 != 0) return cudaErrorInvalidValue;
  if (e.dtype == 0) return launch_k(embed_kernel<float>, dim3(e.ntok), dim3(256), 0, st, e);
  return launch_k(embed_kernel<bf16>, dim3(e.ntok), dim3(256), 0, st, e);
}

// ---------------------------------------------------------------- RoPE tables
// cos/sin(pos * theta^(-2i/hd)) evaluated in fp64 so that the angle is exact
// enough at long contexts, stored as fp32.
__global__ void rope_table_kernel(float* cs, float* sn, int cap, int hd, double theta) {
  pdl_trigger();
  pdl_wait();
  const int half = hd / 2;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)cap * half) return;
  const int pos = (int)(idx / half), i = (int)(idx % half);
  const double inv = pow(theta, -2.0 * i / (double)hd);
  double s, c;
  sincos((double)pos * inv, &s, &c);
  cs[idx] = (float)c;
  sn[idx] = (float)s;
}

cudaError_t launch_rope_table(float* cos_out, float* sin_out, int cap, int hd, double theta,
                              cudaStream_t st) {
  const long long n = (long long)cap * (hd / 2);
  return launch_k(rope_table_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, cos_out,
                  sin_out, cap, hd, theta);
}

// ---------------------------------------------------------------- synthetic state
// SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
// generators", 2014): one 64-bit word per (seed, index).
__device__ __forceinline__ unsigned long long splitmix64(unsigned long long z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void fill_tokens_kernel(int32_t* p, size_t n, int V, unsigned long long seed) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    p[i] = (int32_t)(splitmix64(seed ^ splitmix64(i)) % (unsigned long long)V);
}

// Box-Muller on two 24-bit uniforms of one word: u1 in (0, 1], u2 in [0, 1).
template <typename T>
__global__ void fill_normal_kernel(T* p, size_t n, unsigned long long seed) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const unsigned long long w = splitmix64(seed ^ splitmix64(i));
    const float u1 = ((float)(w >> 40) + 1.0f) * (1.0f / 16777216.0f);
    const float u2 = (float)((w >> 16) & 0xFFFFFFull) * (1.0f / 16777216.0f);
    const float z = sqrtf(-2.0f * logf(u1)) * cospif(2.0f * u2);
    p[i] = from_f32<T>(z);
  }
}

static unsigned fill_grid(size_t n) {
  const size_t blocks = (n + 255) / 256;
  return (unsigned)(blocks < 65536 ? (blocks ? blocks : 1) : 65536);
}

cudaError_t launch_fill_tokens(int32_t* p, size_t n, int V, uint64_t seed, cudaStream_t st) {
  if (V < 1) return cudaErrorInvalidValue;
  return launch_k(fill_tokens_kernel, dim3(fill_grid(n)), dim3(256), 0, st, p, n, V, (unsigned long long)seed);
}

cudaError_t launch_fill_normal(void* p, size_t n, int dtype, uint64_t seed, cudaStream_t st) {
  if (dtype == 1)
    return launch_k(fill_normal_kernel<bf16>, dim3(fill_grid(n)), dim3(256), 0, st, (bf16*)p, n,
                    (unsigned long long)seed);
  return launch_k(fill_normal_kernel<float>, dim3(fill_grid(n)), dim3(256), 0, st, (float*)p, n,
                  (unsigned long long)seed);
}

// ---------------------------------------------------------------- attention
// Query rows of one KV head: row r = t * G + j (token t, query head
// kvh * G + j, G = hq / hkv).  A CTA takes up to 32 rows and one 64-key chunk
// c of absolute key positions [64c, 64c + 64) and computes, for each row,
// the chunk partial (m = max score, l = sum exp(s - m), o = sum exp(s - m) v)
// over the keys at or before the row's position.  The CTA that finishes a
// (KV head, row tile) last combines, for each of its rows, the partials of
// chunks 0..pos/64: M = max m_c, out = sum_c exp(m_c - M) o_c / sum_c
// exp(m_c - M) l_c, with every sum in ascending chunk order.  Chunk
// boundaries are absolute and every row's numbers depend only on its own
// partials, so a row's result does not depend on which other rows share the
// launch.  (Device code: attn_dev.cuh.)
size_t attn_partial_floats(int max_tok, int hq, int hd, int max_chunks) {
  return (size_t)max_tok * hq * max_chunks * (hd + 2);
}
int attn_max_row_tiles(int max_tok, int hq, int hkv) {
  return (max_tok * (hq / hkv) + kRowsPerCta - 1) / kRowsPerCta;
}

template <int HD, typename T>
__global__ void __launch_bounds__(kAttnThreads) attn_chunk_kernel(const __grid_constant__ AttnDesc a) {
  extern __shared__ __align__(16) float sm[];
  __shared__ int rowpos[kRowsPerCta];
  __shared__ int s_last;
  pdl_trigger();
  pdl_wait();
  attn_item<HD, T>(a, blockIdx.x, blockIdx.y, blockIdx.z, gridDim.z, sm, rowpos, &s_last);
}

template <int HD, typename T>
static cudaError_t configure_attn() {
  return cudaFuncSetAttribute(attn_chunk_kernel<HD, T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)kAttnSmemCap);
}

// Tensor-core attention with one item per (KV head, token, head group, key
// split) -- the device code of the persistent kernel as its own launch.
template <int HD>
__global__ void __launch_bounds__(kDWarps * 32) dattn_kernel(const __grid_constant__ AttnDesc a) {
  extern __shared__ __align__(1024) unsigned char dsm_attn[];
  __shared__ int s_last;
  __shared__ uint64_t bars[kDWarps * kDMaxDepth];
  dattn_init_bars(bars);
  __syncthreads();
  pdl_trigger();
  pdl_wait();
  unsigned dpar = 0;
  dattn_item<HD>(a, blockIdx.x, dsm_attn, &s_last, bars, dpar);
}

// Wide items (batched passes): NT 8-row tiles per item.
template <int HD, int NT>
__global__ void __launch_bounds__(kDWarps * 32) dattn_wide_kernel(const __grid_constant__ AttnDesc a) {
  extern __shared__ __align__(1024) unsigned char dsm_attn[];
  __shared__ int s_last;
  __shared__ uint64_t bars[kDWarps * kDMaxDepth];
  dattn_init_bars(bars);
  __syncthreads();
  pdl_trigger();
  pdl_wait();
  unsigned dpar = 0;
  dattn_item_wide<HD, NT>(a, blockIdx.x, dsm_attn, &s_last, bars, dpar);
}

template <int HD>
static cudaError_t configure_dattn() {
  cudaError_t e = cudaFuncSetAttribute(dattn_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)DAttnSmem<HD>::kBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(dattn_wide_kernel<HD, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)DAttnSmem<HD, 2>::kBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(dattn_wide_kernel<HD, 3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)DAttnSmem<HD, 3>::kBytes);
  return e;
}

template <int HD>
static cudaError_t launch_dattn_wide(const AttnDesc& a, cudaStream_t st) {
  const int items = dattn_items_wide(a.wide, a.ntok, a.spt, a.hq, a.hkv, a.cap, a.hd);
  if (a.wide == 2)
    return launch_k(dattn_wide_kernel<HD, 2>, dim3(items), dim3(kDWarps * 32), DAttnSmem<HD, 2>::kBytes, st, a);
  return launch_k(dattn_wide_kernel<HD, 3>, dim3(items), dim3(kDWarps * 32), DAttnSmem<HD, 3>::kBytes, st, a);
}

int dattn_v_box_cols(int hd) { return dattn_vbox_cols(hd); }

int dattn_tickets(int max_tok, int hq, int hkv) { return max_tok * hkv * dattn_hgroups(hq, hkv) * 2; }

cudaError_t launch_dattn(const AttnDesc& a, cudaStream_t st) {
  if (a.dtype != 1 || a.hq % a.hkv != 0 || !a.tmk || !a.tmv) return cudaErrorInvalidValue;
  if (a.spt > 0 && a.ntok % a.spt != 0) return cudaErrorInvalidValue;
  if (a.wide == 2 || a.wide == 3) {
    if (a.hq / a.hkv > kDRows) return cudaErrorInvalidValue;   // one head group per KV head
    if (a.hd == 32) return launch_dattn_wide<32>(a, st);
    if (a.hd == 64) return launch_dattn_wide<64>(a, st);
    if (a.hd == 128) return launch_dattn_wide<128>(a, st);
    return cudaErrorInvalidValue;
  }
  const int items = dattn_items(a.ntok, a.hq, a.hkv, a.cap, a.hd);
  if (a.hd == 32) return launch_k(dattn_kernel<32>, dim3(items), dim3(kDWarps * 32), DAttnSmem<32>::kBytes, st, a);
  if (a.hd == 64) return launch_k(dattn_kernel<64>, dim3(items), dim3(kDWarps * 32), DAttnSmem<64>::kBytes, st, a);
  if (a.hd == 128)
    return launch_k(dattn_kernel<128>, dim3(items), dim3(kDWarps * 32), DAttnSmem<128>::kBytes, st, a);
  return cudaErrorInvalidValue;
}

cudaError_t configure_kernels() {
  cudaError_t e;
  if ((e = configure_gemm()) != cudaSuccess) return e;
  if ((e = configure_tc_gemm()) != cudaSuccess) return e;
  if ((e = configure_attn<32, float>()) != cudaSuccess) return e;
  if ((e = configure_attn<64, float>()) != cudaSuccess) return e;
  if ((e = configure_attn<128, float>()) != cudaSuccess) return e;
  if ((e = configure_attn<32, bf16>()) != cudaSuccess) return e;
  if ((e = configure_attn<64, bf16>()) != cudaSuccess) return e;
  if ((e = configure_attn<128, bf16>()) != cudaSuccess) return e;
  if ((e = configure_dattn<32>()) != cudaSuccess) return e;
  if ((e = configure_dattn<64>()) != cudaSuccess) return e;
  return configure_dattn<128>();
}

template <int HD, typename T>
static cudaError_t launch_attn_t(const AttnDesc& a, cudaStream_t st) {
  const size_t smem = sizeof(float) * attn_smem_floats<HD>(a.max_chunks);
  if (smem > kAttnSmemCap) return cudaErrorInvalidValue;
  const int G = a.hq / a.hkv;
  const int rtiles = (a.ntok * G + kRowsPerCta - 1) / kRowsPerCta;
  return launch_k(attn_chunk_kernel<HD, T>, dim3(a.hkv, a.max_chunks, rtiles), dim3(kAttnThreads), smem,
                  st, a);
}

cudaError_t launch_attention(const AttnDesc& a, cudaStream_t st) {
  if (a.hq % a.hkv != 0) return cudaErrorInvalidValue;
  if (a.spt > 0 && a.spt != a.ntok) return cudaErrorInvalidValue;   // one sequence per pass
  if (a.dtype == 0) {
    if (a.hd == 32) return launch_attn_t<32, float>(a, st);
    if (a.hd == 64) return launch_attn_t<64, float>(a, st);
    if (a.hd == 128) return launch_attn_t<128, float>(a, st);
  } else {
    if (a.hd == 32) return launch_attn_t<32, bf16>(a, st);
    if (a.hd == 64) return launch_attn_t<64, bf16>(a, st);
    if (a.hd == 128) return launch_attn_t<128, bf16>(a, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace sv
