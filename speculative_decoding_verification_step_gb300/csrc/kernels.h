// Internal launch interface between the kernels and the engine.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace sv {

enum Epi : int {
  kEpiStore = 0,   // out_f32[tok][row] = y
  kEpiAdd = 1,     // out_f32[tok][row] += y          (residual add)
  kEpiSwiglu = 2,  // out[tok][j] = silu(gate_j) * up_j, model dtype (gate/up tiles)
};

// Y = X . W^T for a "skinny" X (ntok rows), W stacked from up to three
// row-major [rows][k] segments (q/k/v), or the gate/up pair for kEpiSwiglu.
struct GemmDesc {
  const void* w[3];
  int seg_rows[3];
  int n;          // total output rows (kEpiSwiglu: ffn, the number of gate rows)
  int k;
  const void* x;  // [ntok][ldx], bf16 for bf16 models, fp32 for fp32 models
  int ldx;
  int ntok;
  int epi;
  void* out;      // see Epi
  int ldo;
  int early_prefetch;  // 1: issue the first weight loads before waiting for the
                       // previous kernel (only when that kernel is itself a
                       // bandwidth-bound GEMM; a latency-bound predecessor would
                       // be slowed by the extra traffic)
};

// Cross-warp partial sums and per-tile arrival counters of the bf16 GEMM.
// Tickets must be zero before the first launch; every launch leaves them zero.
struct GemmScratch {
  float* partials;
  size_t partial_floats;
  int* tickets;
  int max_tiles;
};

constexpr int kGemmWarpsPerCta = 8;
constexpr int kGemmMaxTok = 64;      // tokens per GEMM pass (8 groups of 8)

int gemm_grid(int num_sms);
size_t gemm_partial_floats(int num_sms);
int gemm_tiles(const GemmDesc& g);
// dtype: 0 = fp32 model (CUDA-core GEMV), 1 = bf16 model (tensor-core stream-K).
cudaError_t launch_gemm(const GemmDesc& g, int dtype, const GemmScratch& s, int num_sms,
                        cudaStream_t st, bool pdl);

// x[t][:] = embed[tok[t]][:] (fp32 residual stream), with
// tok = tok_base + (tok_idx ? *tok_idx : 0) + tok_off (device-resident index).
cudaError_t launch_embed(const int32_t* tok_base, const int32_t* tok_idx, int tok_off,
                         const void* embed, int dtype, float* x, int ntok, int d, cudaStream_t st);
// out[t][:] = x[t][:] / sqrt(mean(x^2) + eps) * gain   (out in model dtype)
cudaError_t launch_rmsnorm(const float* x, const float* gain, float eps, void* out, int dtype,
                           int ntok, int d, cudaStream_t st);

// Rotate q and k of the fused qkv rows (fp32 [ntok][(hq+2hkv)*hd]) at
// positions *pos_base + t; q -> q_out fp32 [ntok][hq][hd], k,v -> KV cache
// [hkv][cap][hd] (model dtype) at those positions.
struct RopeDesc {
  const float* qkv;
  const int32_t* pos_base;  // position of token t = *pos_base + pos_off + t
  int pos_off;
  const float* rope_cos;  // [cap][hd/2]
  const float* rope_sin;
  float* q_out;
  void* kc;
  void* vc;
  int ntok, hq, hkv, hd, cap, dtype;
};
cudaError_t launch_rope_append(const RopeDesc& r, cudaStream_t st);

// Causal GQA attention of ntok new query rows over the KV cache, split by
// fixed 64-key chunks of absolute position; the last CTA of each (KV head,
// row tile) combines the chunk partials of its rows (the result of a row
// depends only on its own position and partials).
constexpr int kAttnChunk = 64;
constexpr int kAttnRowsPerCta = 32;
struct AttnDesc {
  const float* q;          // [ntok][hq][hd] fp32 (rotated)
  const void* kc;          // [hkv][cap][hd]
  const void* vc;
  const int32_t* pos_base; // query t sits at *pos_base + pos_off + t
  int pos_off;
  float* partials;         // [ntok*hq][max_chunks][hd+2]
  int* tickets;            // [hkv][row tiles], zero before and after
  void* out;               // [ntok][hq*hd] model dtype
  int ntok, hq, hkv, hd, cap, max_chunks, dtype;
  float scale;
};
size_t attn_partial_floats(int max_tok, int hq, int hd, int max_chunks);
int attn_max_row_tiles(int max_tok, int hq, int hkv);
cudaError_t launch_attention(const AttnDesc& a, cudaStream_t st);
// One-time kernel attributes (dynamic shared memory); call before any capture.
cudaError_t configure_kernels();

// ---- sampling / acceptance ----
constexpr int kVocabChunk = 2048;
struct SampleDesc {
  const float* logits;      // rows of V fp32 (row stride ld)
  int64_t ld;
  const float* mix_src;     // optional second row set (same layout), mixed in at weight lambda
  int64_t mix_ld;
  float lambda;
  float* mixed_out;         // where the mixed row is written (needed when mix_src != null)
  int64_t mixed_ld;
  int rows, V;
  float temperature;
  uint64_t seed;
  const int32_t* step_dev;  // if non-null, step = *step_dev + step_base + row
  uint64_t step_base;
  uint32_t position;        // Philox position (draft index i; 0 for AR)
  uint32_t stream;          // Philox stream id
  int32_t* out_token;       // [rows]; row r goes to out_token[(out_idx ? *out_idx : 0) + out_off + r]
  const int32_t* out_idx;
  int out_off;
  // optional commit of an autoregressive draw: seq[*len + 1] = tok, *len += 1
  int32_t* commit_seq;
  int32_t* commit_len;
  int32_t* commit_step;     // incremented when committing
  float* partials;          // scratch [rows][chunks][2]
  int* tickets;             // [rows], zero before and after
};
size_t sample_partial_floats(int rows, int V);
cudaError_t launch_sample(const SampleDesc& s, cudaStream_t st);

struct AcceptDesc {
  const float* p;           // [rows] x [K+1][V], row stride p_ld floats
  int64_t p_ld;
  const float* q;           // [rows] x [K][V]
  int64_t q_ld;
  const int32_t* drafts;    // [rows][K], offset by (drafts_idx ? *drafts_idx : 0) + drafts_off
  const int32_t* drafts_idx;
  int drafts_off;
  int32_t* drafts_copy;     // optional [rows][K] copy of the drafts read
  int rows, K, V;
  float temperature;
  uint64_t seed;
  const int32_t* step_dev;  // if non-null, step = *step_dev (+ row)
  uint64_t step_base;
  int32_t* out_tokens;      // [rows][K+1]
  int32_t* out_count;       // [rows]
  uint32_t* out_flags;      // [rows] or null
  // optional commit (rows == 1): seq[len+1..len+n+1] = emitted; len += n+1; step += 1
  int32_t* commit_seq;
  int32_t* commit_len;
  int32_t* commit_step;
  float* partials;          // scratch [rows][chunks][2K+1][2]
  int* tickets;             // [rows]
};
size_t accept_partial_floats(int rows, int K, int V);
cudaError_t launch_accept(const AcceptDesc& a, cudaStream_t st);

// RoPE tables: cos/sin of pos * theta^(-2i/hd) for pos < cap, computed in fp64.
cudaError_t launch_rope_table(float* cos_out, float* sin_out, int cap, int hd, double theta,
                              cudaStream_t st);

}  // namespace sv
