// Internal launch interface between the kernels and the engine.
#pragma once
#include <cuda_runtime.h>
#include <vector>
#include <stddef.h>
#include <stdint.h>

namespace sv {

// Batched passes: the tokens of a pass are the sequences' tokens in sequence
// order, spt per sequence (token t is token t % spt of sequence t / spt;
// spt <= 0: one sequence).  Per-sequence device state (committed length L,
// step counters, ...) is kStateLd int32 apart; sequence b's KV rows are
// those of KV heads b * hkv .. b * hkv + hkv - 1 of a [B * hkv][cap][hd] cache.
constexpr int kStateLd = 4;
__host__ __device__ inline int seq_of_tok(int spt, int t) { return spt > 0 ? t / spt : 0; }
__host__ __device__ inline int idx_in_seq(int spt, int t) { return spt > 0 ? t % spt : t; }

enum Epi : int {
  kEpiStore = 0,    // out_f32[tok][row] = y
  kEpiAdd = 1,      // out_f32[tok][row] += y (residual add); optionally per-tile sums of
                    // squares of the updated rows -> ss_out (the next RMSNorm's input)
  kEpiSwiglu = 2,   // out[tok][j] = silu(gate_j) * up_j, model dtype (gate/up tiles)
  kEpiQkvRope = 3,  // fused q/k/v: rotate q, k at their positions; q -> q_out (fp32),
                    // k, v -> KV cache (model dtype)
  kEpiHeadRes = 4,  // self-draft heads: out[tok][row] = hres[tok][row mod k] + silu(y),
                    // model dtype (the rows of K stacked d x d heads, k = d)
};

// Y = X . W^T for a "skinny" X (ntok rows), W stacked from up to three
// row-major [rows][k] segments (q/k/v), or the gate/up pair for kEpiSwiglu.
//
// Output tiles are 16 rows.  Row pairing per tile (thread rows g and g+8):
//   plain:        rows 16t + g, 16t + g + 8
//   kEpiSwiglu:   gate row 8t + g, up row 8t + g
//   kEpiQkvRope:  head h = t / (hd/16), j = t % (hd/16): rows h*hd + 8j + g and
//                 h*hd + 8j + g + hd/2 (a RoPE rotation pair)
struct GemmDesc {
  const void* w[3];
  int seg_rows[3];
  int n;          // total output rows (kEpiSwiglu: ffn, the number of gate rows)
  int k;
  // X operand: [ntok][ldx]; bf16 (fp32 models: fp32), or with x_norm = 1 the fp32
  // residual, normalised on load: X = x * inv_rms(tok) * gain, inv_rms from the
  // per-16-row-tile sums of squares ss_in[(k/16) tiles][ss_ld].  x_norm = 2
  // (persistent kernel only): X is the bf16 product x * gain written by the
  // producer of x (xg_out below), and inv_rms(tok) scales the finished sums
  // before the epilogue.
  const void* x;
  int ldx;
  int ntok;
  int x_norm;
  const float* gain;
  const float* ss_in;
  int ss_ld;
  float eps;
  // epilogue
  int epi;
  void* out;      // kEpiStore/kEpiAdd: fp32 [ntok][ldo]; kEpiSwiglu: model dtype [ntok][ldo]
  int ldo;
  float* ss_out;  // kEpiAdd: per-tile sums of squares [tiles][ss_ld] (may be null)
  void* xg_out;            // kEpiAdd (may be null): bf16 [ntok][ldo] updated rows x gain_next,
  const float* gain_next;  // the next RMSNorm's x_norm = 2 input
  // kEpiQkvRope
  int hq, hkv, hd, cap;
  const int32_t* pos_base;   // position of token t = *pos_base + pos_off + t, or with
  int pos_off;               // spt > 0: pos_base[b * pos_ld] + pos_off + j (token j of sequence b)
  int spt, pos_ld;
  const float* rope_cos;     // [cap][hd/2]
  const float* rope_sin;
  float* q_out;              // [ntok][hq][hd]
  void* kc;                  // [hkv][cap][hd] of this layer
  void* vc;
  const float* hres;   // kEpiHeadRes: fp32 [ntok][k] residual added to silu(y)
  int q4;              // 1: 4-bit group-quantized weights (persistent kernel only): each
                       // segment is packed codes [rows][k/2] followed by bf16 scales
                       // [k/64][rows] (group-major), 16-byte aligned
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

// Tensor-core (tcgen05) GEMM for batched passes of kTcMinTok < ntok <=
// kTcMaxTok tokens (tcgemm.cu): work units of 128 weight rows x a k split,
// taken by one persistent CTA per SM.  A GEMM whose tiles are not split runs
// its epilogue straight from tensor memory; otherwise every unit writes an
// fp32 partial ([units][128][npad], at most max_units units,
// tc_gemm_partial_floats) that a second launch sums and finishes.  inv:
// scratch of kTcMaxTok floats (1/rms per token of a normalised input, folded
// by a first launch).  err raised when a bounded wait gives up.
constexpr int kTcMinTok = 16;    // the tensor-memory GEMM takes passes of more tokens
constexpr int kTcMaxTok = 512;
// stage ring: 4 stages at 256 tokens, 3 up to 448, 2 at 512 (+ 1 KB alignment)
constexpr int kTcSmemBytes = 3 * (128 * 64 * 2 + 448 * 64 * 2) + 1024;
bool tc_gemm_supported(const GemmDesc& g);
size_t tc_gemm_partial_floats(int num_sms, int max_n);
cudaError_t launch_tc_gemm(const GemmDesc& g, float* partials, float* inv, int* err, int num_sms,
                           long long max_units, cudaStream_t st);
cudaError_t configure_tc_gemm();

int gemm_grid(int num_sms);
size_t gemm_partial_floats(int num_sms);
int gemm_tiles(const GemmDesc& g);
// dtype: 0 = fp32 model (CUDA-core GEMV), 1 = bf16 model (tensor-core stream-K).
cudaError_t launch_gemm(const GemmDesc& g, int dtype, const GemmScratch& s, int num_sms,
                        cudaStream_t st, bool pdl);
cudaError_t configure_gemm();

// x[t][:] = embed[tok[t]][:] (fp32 residual stream), with
// tok = tok_base + (tok_idx ? *tok_idx : 0) + tok_off (device-resident index);
// with spt > 0 token j of sequence b is tok_base[b * tok_ld + (tok_idx ?
// tok_idx[b * idx_ld] : 0) + tok_off + j];
// ss[i][t] = sum of x[t][16i .. 16i+15]^2 (the first RMSNorm's input);
// optionally xg[t][:] = bf16(x[t][:] * gain) (its x_norm = 2 input).
struct EmbedDesc {
  const int32_t* tok_base;
  const int32_t* tok_idx;
  int tok_off;
  int spt, idx_ld;
  int64_t tok_ld;
  const void* embed;
  int dtype;
  float* x;
  void* xg;
  const float* gain;
  float* ss;
  int ss_ld;
  int ntok, d;
};
cudaError_t launch_embed(const EmbedDesc& e, cudaStream_t st);
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
  const int32_t* pos_base; // query t sits at *pos_base + pos_off + t, or with spt > 0
  int pos_off;             // (bf16 path only) at pos_base[b * pos_ld] + pos_off + j
  int spt, pos_ld;
  int seq0;                // bf16 path: sequence b of the pass is cache sequence seq0 + b
  int group;               // bf16 per-operation path: 1 = token-group items at any position
  int wide;                // bf16 per-operation path: 2 or 3 = wide items of that many 8-row
                           // tiles (all heads of several tokens of one sequence; G <= 8)
  float* partials;         // [ntok*hq][max_chunks][hd+2]
  int* tickets;            // [hkv][row tiles], zero before and after
  void* out;               // [ntok][hq*hd] model dtype
  int ntok, hq, hkv, hd, cap, max_chunks, dtype;
  float scale;
  // tensor-core path (bf16): 2-D tensor maps of this layer's K and V cache
  // ([hkv * cap][hd], see encode_kv_map) and the flag raised when a wait for
  // their copies gives up
  const void* tmk;
  const void* tmv;
  int* err;
};
size_t attn_partial_floats(int max_tok, int hq, int hd, int max_chunks);
int attn_max_row_tiles(int max_tok, int hq, int hkv);
cudaError_t launch_attention(const AttnDesc& a, cudaStream_t st);
// Tensor-core attention (bf16 cache, head dim 32/64/128, any token count):
// items per (KV head, token group, group of 8 query heads, 1024-key split,
// V column part -- two for head dims 64 and 128); its
// tickets are dattn_tickets(tokens, hq, hkv) zeroed counters, its partials
// persist_attn_partial_floats floats.
cudaError_t launch_dattn(const AttnDesc& a, cudaStream_t st);
struct TensorMap128;
// Tensor map of a bf16 KV cache [rows][hd] for launch_dattn (head dim 32, 64
// or 128; boxes of 16 rows x box_cols dims, 0: min(hd, 64)); false when the
// map cannot be encoded.
bool encode_kv_map(TensorMap128& m, const void* base, int hd, long long rows, int box_cols = 0);
// Box columns of the V map launch_dattn expects (head dim 64: 32 -- items
// read V in halves).
int dattn_v_box_cols(int hd);
// Attention items of a pass whose last position is at least this take token
// groups (8 / min(G, 8) tokens share one walk over the KV head's keys);
// earlier passes give each token its own items, since the keys are then few
// and L2-resident and more, shorter items finish sooner.  Grouping changes
// no row's arithmetic.
constexpr int kDGroupMinPos = 1024;
int dattn_tickets(int max_tok, int hq, int hkv);
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
  float* mixed_out;         // where the mixed row (or, without mix_src, the row) is written;
                            // needed when mix_src != null
  int64_t mixed_ld;
  int rows, V;
  float temperature;
  uint64_t seed;
  const int32_t* step_dev;  // if non-null, step = *step_dev + step_base + row
  uint64_t step_base;
  uint32_t position;        // Philox position (draft index i; 0 for AR)
  uint32_t stream;          // Philox stream id
  int row_pos;              // batch = 0 only: row r is the draft at position position + r of
                            // one step (step = *step_dev + step_base), not a draw at step + r
  int32_t* out_token;       // [rows]; row r goes to out_token[(out_idx ? *out_idx : 0) + out_off + r]
  const int32_t* out_idx;
  int out_off;
  // optional commit of an autoregressive draw: seq[*len + 1] = tok, *len += 1
  int32_t* commit_seq;
  int32_t* commit_len;
  int32_t* commit_step;     // incremented when committing
  const int32_t* err;       // optional: the commit is skipped while *err != 0 (a forward gave up)
  // batch = 1: row r is sequence r of a batch -- step = step_dev[r * st_ld] +
  // step_base with Philox row word r, the token goes to out_token[r * out_ld +
  // (out_idx ? out_idx[r * st_ld] : 0) + out_off], and the commit uses
  // commit_seq + r * seq_ld, commit_len[r * st_ld], commit_step[r * st_ld]
  int batch, st_ld;
  int64_t out_ld, seq_ld;
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
  // optional commit (rows == 1, or batch): seq[len+1..len+n+1] = emitted; len += n+1; step += 1
  int32_t* commit_seq;
  int32_t* commit_len;
  int32_t* commit_step;
  const int32_t* err;       // optional: the commit is skipped while *err != 0 (a forward gave up)
  // batch = 1: row r is sequence r -- step = step_dev[r * st_ld] + step_base
  // with Philox row word r, drafts at drafts + r * seq_ld + (drafts_idx ?
  // drafts_idx[r * st_ld] : 0) + drafts_off, commit into commit_seq + r * seq_ld,
  // commit_len[r * st_ld], commit_step[r * st_ld]
  int batch, st_ld;
  int64_t seq_ld;
  float* partials;          // scratch [rows][chunks][2K+1][2]
  int* tickets;             // [rows]
};
size_t accept_partial_floats(int rows, int K, int V);
cudaError_t launch_accept(const AcceptDesc& a, cudaStream_t st);

// Prompt-lookup drafting (lookup.cu): per sequence b, drafts d_1..d_K of the
// most recent longest suffix match (up to n_max tokens) written to
// seq[b * seq_ld + L_b + 1 ..], L_b = lens[b * st_ld], and one-hot q logit
// rows (0 at d_i, -inf elsewhere) to q_out + b * q_ld + (i-1) * V.
constexpr int kLookupMaxK = 16;
constexpr int kLookupMaxN = 8;
struct LookupDesc {
  int32_t* seq;
  int64_t seq_ld;
  const int32_t* lens;
  int st_ld;
  int rows, K, n_max, V;
  float* q_out;
  int64_t q_ld;
};
cudaError_t launch_lookup(const LookupDesc& d, cudaStream_t st);

// Self-draft heads' input: copies one row of the LM head's input of a pass
// (its X row and its per-tile sums of squares) and writes the normalised
// row u = RMSNorm_final(h) in fp32, for the next heads pass (heads.cu).
struct HeadInDesc {
  const void* x;           // the pass's LM-head input rows: bf16 h * gain (x_bf16) or fp32 h
  int x_bf16;
  int64_t ldx;             // elements between rows
  const float* ss;         // per-16-row-tile sums of squares of h, [d/16][ss_ld]
  int ss_ld;
  const int32_t* count;    // non-null: row = *count - 1, clamped to [0, max_row]
  int row, max_row;        // else row `row` (a host-checked index)
  int d;
  const float* gain;       // the final RMSNorm's gain (fp32 rows; bf16 rows carry it)
  float eps;
  const int32_t* err;      // optional: nothing is copied while *err != 0
  void* out_x;             // [d], the row's dtype
  float* out_ss;           // [d/16]
  float* out_u;            // [d]
};
cudaError_t launch_head_input(const HeadInDesc& h, cudaStream_t st);

// ---- persistent forward (bf16 models) ----
// One cooperative launch runs the phases of a whole forward (embedding, the
// per-layer GEMMs and attention, the LM head), separated by a bounded grid
// barrier.  GEMM phases stream their weights with 2-D tensor copies (see
// tma_dev.cuh); results agree with the per-kernel path up to the order of
// fp32 partial sums, and are batch-invariant like it.
enum PhaseKind : int { kPhaseEmbed = 0, kPhaseGemm = 1, kPhaseAttn = 2 };
// GEMM X source: from global memory (per-operation GEMM; the persistent
// kernel's streamed X), kept in shared memory (the persistent kernel's
// resident X), or normalised while loading (per-operation GEMM).
enum XMode : int { kXGlobal = 0, kXSmem = 1, kXInline = 2 };
constexpr int kPhaseStamps = 5;
constexpr int kPrefillChunk = 8;   // positions per persistent prefill pass (4-bit models)
struct PhaseDesc {
  int kind;
  // GEMM streaming geometry (tma_dev.cuh): X resident in shared memory
  // (kXSmem) or streamed beside the weights (kXGlobal); paired boxes (RoPE /
  // SwiGLU: two 8-row boxes per tile) or one 16-row box; 16-row tiles; tiles
  // per stage group and k per stage; ring stages, bytes per stage and the
  // offset of the stage's X boxes; units issued before the phase's barrier;
  // tensor-map indices of the weight segments (0..2) and of X (3)
  int xm, paired, tiles, gt, kc;
  int stages, stage_bytes, xoff, prefetch;
  int tm[4];
  // 4-bit group-quantized weights (q4 = 1): tensor maps of the segments'
  // codes (tm[0..2]) and group-major scales (tms[0..2]); bytes per tile in
  // a stage (codes of both 8-row halves, then their scales)
  int q4, tile_bytes;
  int tms[3];
  // GEMM: tile ranges counted from the last CTA down (1) or from CTA 0 (0);
  // the CTAs with the larger shares of tiles are then the ones that finished
  // the previous phase early (no attention item, or a smaller share) and
  // streamed this phase's first weights while waiting at its barrier
  int rev;
  int attn_items;
  GemmDesc g;
  AttnDesc a;
  EmbedDesc e;
};
// 2-D tensor-map descriptors (opaque, 128 bytes, 64-byte aligned in memory).
struct alignas(64) TensorMap128 {
  unsigned char bytes[128];
};
struct PersistDesc {
  const PhaseDesc* phases;   // device array
  int nphases;
  const TensorMap128* tmaps; // device array indexed by PhaseDesc::tm
  int ring_bytes;            // dynamic shared memory: [group partials][ring][X region]
  unsigned* bar;             // [1] arrival count (zero at start; the kernel leaves it zero)
  int* err;                  // set to 1 when a wait gives up
  // optional fault injection (null: off): [0] arrivals added to every grid-
  // barrier target (> 0: a barrier that cannot complete), [1] grid-barrier
  // probe limit (0: the default bound); read once at kernel start
  const int* ctl;
  // optional (null: off): [1 + kPhaseStamps * nphases] globaltimer stamps,
  // zeroed before the launch -- start, then per phase the earliest arrival
  // (stored as ~t, atomicMax), the latest arrival (atomicMax), CTA 0's
  // release, the latest end of X preparation (GEMM) or of a key walk
  // (attention), and the latest delivery of a CTA's last weight unit (GEMM)
  // or end of its items (attention)
  unsigned long long* times;
};
// Shared-memory layout of one persistent kernel instance: the weight ring,
// the group-partial area and the X region (resident GEMM inputs) -- the
// attention tiles reuse the whole of it.
struct PersistLayout {
  size_t ring, xreg, total;
};
// Layout for head dim hd and passes of at most max_tok tokens of a model of
// width d_model (X region: at least max_tok rows of d_model); false when it
// does not fit one CTA per SM.
bool persist_layout(int hd, int max_tok, int d_model, PersistLayout* out);
// Fill the kernel-side fields of a phase.  The GEMM variant also encodes the
// phase's tensor maps, appending them to maps; false when the phase does not
// meet the tensor-copy rules (16-byte aligned rows, k and the X stride
// multiples of 8, at most 8 tokens, RoPE head dim a multiple of 32).
bool persist_phase_from_gemm(PhaseDesc& p, const GemmDesc& g, std::vector<TensorMap128>& maps, int grid,
                             const PersistLayout& lay);
// Attention phases need a bf16 cache, at most 8 tokens and head dim 32, 64
// or 128; their scratch is persist_attn_partial_floats floats and
// dattn_tickets zeroed counters (a.partials, a.tickets).
bool persist_phase_from_attn(PhaseDesc& p, const AttnDesc& a);
size_t persist_attn_partial_floats(int max_tok, int hq, int hd, int cap);
void persist_phase_from_embed(PhaseDesc& p, const EmbedDesc& e);
// True when one CTA per SM of the persistent kernel fits, for passes of at
// most max_tok tokens.
bool persist_supported(int hd, size_t smem, int num_sms, int max_tok);
// group: attention items take token groups (kDGroupMinPos); either mode gives
// the same bits, the caller picks the faster one for the pass's positions.
cudaError_t launch_persist(const PersistDesc& p, int hd, bool group, size_t smem, int num_sms, cudaStream_t st);

// Synthetic state: token ids uniform in [0, V) (up to a modulo bias below
// 2^-40) and normally distributed values (dtype 0 fp32, 1 bf16), both from a
// counter-based generator keyed by seed.
cudaError_t launch_fill_tokens(int32_t* p, size_t n, int V, uint64_t seed, cudaStream_t st);
cudaError_t launch_fill_normal(void* p, size_t n, int dtype, uint64_t seed, cudaStream_t st);

// RoPE tables: cos/sin of pos * theta^(-2i/hd) for pos < cap, computed in fp64.
cudaError_t launch_rope_table(float* cos_out, float* sin_out, int cap, int hd, double theta,
                              cudaStream_t st);

}  // namespace sv
