// Context, forward orchestration and the C ABI (include/specverify.h).
//
// One speculative step ("Speculative decoding internals", 演算法核心 Steps
// 1-4; "Speculative Decoding 101", Floors 3-5 and the Boss Level replay):
//
//   state on the device: seq[0..L] committed tokens (seq[L] = pending token,
//   not yet scored), L, the step counters.
//   draft pass 1 : tokens seq[L-1], seq[L] at positions L-1, L (the first
//                  row rewrites an identical KV entry unless the previous step
//                  accepted all K drafts, in which case the draft has not yet
//                  seen d_K); its last row gives q_1, d_1 -> seq[L+1]
//   draft pass i : token seq[L+i-1] at position L+i-1 -> q_i, d_i -> seq[L+i]
//   verify       : target over seq[L..L+K] at positions L..L+K -> p_1..p_{K+1}
//   accept       : fused kernel; writes the emitted tokens over seq[L+1..],
//                  L += n+1, step += 1 (KV rollback = the new L; no copies)
//   readback     : one small device-to-host copy of (tokens, count, flags).
// Every position and index is read from device memory, so the whole step is
// captured once as a CUDA graph and replayed.
//
// Self-draft heads (opts.draft_heads; "Speculative Decoding 101", Floor 6,
// "Speculative decoding internals", 三條主流變體 MTP) replace the draft passes
// by one heads pass over the target's LM-head input at the last scored
// position: z_i = u + silu(W_i u) for the K heads in one GEMM, the target's
// LM head over the K rows z_i, then the K drafts in one sampler launch.
// After the acceptance a one-block kernel keeps verify row n (n accepted) as
// the next heads pass's input.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "specverify.h"

using namespace sv;

namespace {

thread_local std::string g_err = "no error";

// Test hooks (spec_inject_fault): the n-th device allocation of the next
// spec_init fails (0: off), and the bytes every context holds in device
// allocations.
std::atomic<int> g_fail_alloc_at{0};
std::atomic<long long> g_device_bytes{0};

struct ModelState {
  // d.dtype is the arithmetic dtype (a 4-bit model computes like a bf16
  // model, with q4 set: its GEMMs stream packed codes and scales)
  spec_model_desc d{};
  bool q4 = false;
  std::vector<spec_layer_weights> layers;
  void* kc = nullptr;   // [n_layers][hkv][cap][hd]
  void* vc = nullptr;
  float* rope_cos = nullptr;
  float* rope_sin = nullptr;
  TensorMap128* kv_maps = nullptr;   // bf16: [layer][K, V] tensor maps of the cache
  int esize = 4;
  int qkv_rows() const { return (d.n_heads + 2 * d.n_kv_heads) * d.head_dim; }
  size_t layer_kv_elems(int cap) const { return (size_t)d.n_kv_heads * cap * d.head_dim; }
  // bytes one weight costs in a pass: 4-bit codes plus a bf16 scale per 64
  double wbytes() const { return q4 ? 0.5 + 2.0 / 64.0 : esize; }
  double matrix_bytes_layer() const {
    const double hd = d.head_dim, dm = d.d_model;
    return ((2.0 * d.n_heads + 2.0 * d.n_kv_heads) * hd * dm + 3.0 * dm * d.ffn_dim) * wbytes();
  }
  double head_bytes() const { return (double)d.vocab * d.d_model * wbytes(); }
  double weight_bytes() const { return d.n_layers * matrix_bytes_layer() + head_bytes(); }
  double kv_bytes_per_token() const { return 2.0 * d.n_layers * d.n_kv_heads * d.head_dim * esize; }
};

}  // namespace

namespace sv {
// Error message of a failed stateless call, read by spec_last_error(NULL).
void set_thread_error(const std::string& msg) { g_err = msg; }
}  // namespace sv

struct PersistFwd {
  PersistDesc desc{};
  int hd = 0;
  size_t smem = 0;
  std::vector<PhaseDesc> host;   // the phase list (for spec_phase_times)
};

struct spec_ctx {
  ModelState tgt, drf;
  bool persist = false;            // persistent forward kernels (bf16 models)
  // draft passes 1..K (0..K-1), verify (K), plain decoding (K+1), the last
  // scored prompt position of the draft (K+2) and of the target (K+3), and
  // for 4-bit models the prefill chunks of kPrefillChunk positions at the
  // host-set position: target (K+4), target with its LM-head rows (K+5),
  // draft (K+6)
  PersistFwd pforward[24];
  bool q4 = false;                 // a 4-bit model: prefill runs the persistent chunks
  float* logits_chunk = nullptr;   // [kPrefillChunk][V] LM-head rows of the last target chunk
  PhaseDesc* phase_dev = nullptr;
  unsigned* bar = nullptr;
  int K = 0;
  int B = 1;                       // sequences (batch > 1: per-operation path, bf16 models)
  int lookup = 0;                  // > 0: prompt-lookup drafting with suffix matches up to this
  // self-draft heads: [K][d][d] in the target's arithmetic dtype (null: none)
  const void* heads = nullptr;
  int heads_pass = -1;             // its persistent pass (index into pforward)
  void* hin_x = nullptr;           // the heads' input row: the LM head's X row of the last scored position,
  float* hin_ss = nullptr;         // its per-tile sums of squares,
  float* hin_u = nullptr;          // and the normalised row u (fp32)
  void* zbuf = nullptr;            // [K][d] u + silu(W_i u), the LM head's input of the heads pass
  bool draft_model() const { return !lookup && !heads; }
  int64_t seq_ld = 0;              // int32 stride between the sequences' token arrays
  int tok_max = kGemmMaxTok;       // tokens per forward pass (batch > 1: up to kTcMaxTok)
  float* tc_part = nullptr;        // tensor-core GEMM partials (batch > 1), tc_units work units
  float* tc_inv = nullptr;         // tensor-core GEMM: 1/rms per token of a normalised input
  long long tc_units = 0;
  spec_opts opts{};
  cudaStream_t stream = nullptr;
  bool own_stream = false;
  int num_sms = 0;
  int cap = 0;
  int max_chunks = 0;
  // device state
  // per sequence b, kStateLd apart: [0] L, [1] spec step, [2] ar step,
  // [3] eager position scratch
  int32_t* st = nullptr;
  int32_t* seq = nullptr;   // [B][seq_ld], seq_ld = cap + K + 2
  int32_t* fwd_tok = nullptr;  // [kGemmMaxTok] host-supplied tokens of spec_model_forward
  // activations
  float* x = nullptr;
  void* xg = nullptr;   // bf16 x * gain of the next RMSNorm (persistent forward: x_norm = 2 input)
  void* hbuf = nullptr;
  float* q = nullptr;
  void* attn = nullptr;
  float* attn_part = nullptr;
  int* attn_tick = nullptr;
  int* dattn_tick = nullptr;       // tensor-core attention (bf16 models)
  int dattn_nt = 0;
  float* ss = nullptr;         // [d_max/16][tok_max] per-tile sums of squares
  float* logits_p = nullptr;  // [K+1][V]
  float* logits_q = nullptr;  // [B][K][V]
  float* logits_d = nullptr;  // batch > 1: [2B][V] draft-pass logits before sampling
  GemmScratch gs{};
  float* samp_part = nullptr;
  int* samp_tick = nullptr;
  float* acc_part = nullptr;
  int* acc_tick = nullptr;
  // device [B][K+1 tokens][B counts][B flags][B][K drafts][wait-timeout flag]
  int32_t* result = nullptr;
  int32_t* h_result = nullptr;  // pinned host mirror
  int32_t* h_pos = nullptr;     // pinned host scratch for eager positions
  std::vector<std::pair<void*, size_t>> allocs;
  int* fault_ctl = nullptr;   // persistent kernels' fault-injection words (PersistDesc::ctl)
  // graphs
  // step and profiling graphs per attention mode (index: grp)
  cudaGraphExec_t step_exec[2] = {nullptr, nullptr};
  cudaGraphExec_t ar_exec = nullptr;
  // draft loop, verify, ar, verify forward alone
  cudaGraphExec_t prof_exec[4][2] = {};
  int prof_kernels[4] = {0, 0, 0, 0};
  // attention mode of the persistent launches being enqueued: token groups
  // (the passes' last position reaches kDGroupMinPos) or one token per item
  bool grp = false;
  // host mirror of the state
  bool prefilled = false;
  bool draft_stale = false;
  int host_L = 0;                  // sequence 0 (batch 1: the sequence)
  std::vector<int> host_Ls;        // every sequence's L
  int kernels_step = 0, kernels_ar = 0, gemms_verify = 0;
  int64_t steps = 0, ar_steps = 0, emitted = 0, accepted = 0;
  int64_t hist[17] = {0};
  // timing (SPEC_OPT_TIMING)
  std::vector<cudaEvent_t> ev;
  std::vector<double> ev_bytes;
  int ev_used = 0;
  bool timing_verify = false;
  double timed_ms = 0.0, timed_bytes = 0.0;
  int64_t timed_launches = 0;
  int launch_count = 0;
  std::string err = "no error";
};

namespace {

int fail(spec_ctx* c, int code, const std::string& msg) {
  if (c) c->err = msg;
  g_err = msg;
  return code;
}

#define CUDA_TRY(c, expr)                                                                   \
  do {                                                                                      \
    cudaError_t e__ = (expr);                                                               \
    if (e__ != cudaSuccess)                                                                 \
      return fail((c), SPEC_E_CUDA, std::string(#expr) + ": " + cudaGetErrorString(e__));   \
  } while (0)

template <typename T>
cudaError_t dalloc(spec_ctx* c, T** p, size_t bytes) {
  void* v = nullptr;
  const size_t b = bytes < 16 ? 16 : bytes;
  // an injected allocation failure (tests) behaves like an exhausted device
  if (g_fail_alloc_at.load() > 0 && g_fail_alloc_at.fetch_sub(1) == 1) return cudaErrorMemoryAllocation;
  cudaError_t e = cudaMalloc(&v, b);
  if (e != cudaSuccess) return e;
  c->allocs.emplace_back(v, b);
  g_device_bytes += (long long)b;
  *p = (T*)v;
  return cudaSuccess;
}

bool valid_hd(int hd) { return hd == 32 || hd == 64 || hd == 128; }

int check_model(const spec_model_desc* m, const char* which, std::string* why) {
  char buf[256];
  if (!m) { *why = std::string(which) + ": null model"; return SPEC_E_ARG; }
  if (m->n_layers < 1 || m->d_model < 1 || m->n_heads < 1 || m->n_kv_heads < 1 ||
      m->ffn_dim < 1 || m->vocab < 2 || !(m->rms_eps > 0.f) || !(m->rope_theta > 0.f)) {
    *why = std::string(which) + ": non-positive dimension or parameter";
    return SPEC_E_SHAPE;
  }
  if (m->dtype != SPEC_DTYPE_F32 && m->dtype != SPEC_DTYPE_BF16 && m->dtype != SPEC_DTYPE_Q4) {
    *why = std::string(which) + ": unknown dtype";
    return SPEC_E_SHAPE;
  }
  if (m->dtype == SPEC_DTYPE_Q4 &&
      (m->d_model % 256 || m->ffn_dim % 256 || (m->n_heads * m->head_dim) % 256 || m->vocab % 8 ||
       (m->n_kv_heads * m->head_dim) % 8)) {
    *why = std::string(which) +
           ": 4-bit models need d_model, ffn_dim and n_heads*head_dim multiples of 256, vocab and "
           "n_kv_heads*head_dim multiples of 8";
    return SPEC_E_SHAPE;
  }
  if (!valid_hd(m->head_dim) || m->n_heads % m->n_kv_heads != 0) {
    snprintf(buf, sizeof buf, "%s: head_dim %d must be 32/64/128 and n_heads %% n_kv_heads == 0",
             which, m->head_dim);
    *why = buf;
    return SPEC_E_SHAPE;
  }
  const int kmul = m->dtype == SPEC_DTYPE_F32 ? 4 : 64;
  if (m->d_model % kmul || m->ffn_dim % kmul || (m->n_heads * m->head_dim) % kmul ||
      m->ffn_dim % 8) {
    snprintf(buf, sizeof buf, "%s: d_model, ffn_dim and n_heads*head_dim must be multiples of %d",
             which, kmul);
    *why = buf;
    return SPEC_E_SHAPE;
  }
  if (!m->embed || !m->final_norm || !m->lm_head || !m->layers) {
    *why = std::string(which) + ": null weight pointer";
    return SPEC_E_ARG;
  }
  for (int l = 0; l < m->n_layers; ++l) {
    const spec_layer_weights& w = m->layers[l];
    if (!w.attn_norm || !w.wq || !w.wk || !w.wv || !w.wo || !w.ffn_norm || !w.w_gate ||
        !w.w_up || !w.w_down) {
      snprintf(buf, sizeof buf, "%s: null weight pointer in layer %d", which, l);
      *why = buf;
      return SPEC_E_ARG;
    }
  }
  return SPEC_OK;
}

// Result words of the device result buffer (see spec_ctx::result).
int32_t* res_err(spec_ctx* c) { return c->result + (size_t)c->B * (2 * c->K + 3); }
int res_words(const spec_ctx* c) { return c->B * (2 * c->K + 3) + 1; }

// ---------------------------------------------------------------- launches
struct Launch {
  spec_ctx* c;
  cudaError_t e = cudaSuccess;
  void note(cudaError_t r) {
    if (e == cudaSuccess && r != cudaSuccess) e = r;
    c->launch_count++;
  }
};

void gemm(Launch& L, const GemmDesc& g, int dtype) {
  spec_ctx* c = L.c;
  if (c->tok_max > kGemmMaxTok && g.ntok > kTcMinTok && tc_gemm_supported(g)) {   // batched passes
    L.note(launch_tc_gemm(g, c->tc_part, c->tc_inv, res_err(c), c->num_sms, c->tc_units, c->stream));
    return;
  }
  const bool timed = c->timing_verify && c->ev_used + 2 <= (int)c->ev.size();
  if (timed) cudaEventRecord(c->ev[c->ev_used], c->stream);
  L.note(launch_gemm(g, dtype, c->gs, c->num_sms, c->stream, false));
  if (timed) {
    cudaEventRecord(c->ev[c->ev_used + 1], c->stream);
    const double es = dtype == SPEC_DTYPE_BF16 ? 2.0 : 4.0;
    const double rows = g.epi == kEpiSwiglu ? 2.0 * g.n : (double)g.n;
    c->ev_bytes[c->ev_used / 2] = rows * g.k * es;
    c->ev_used += 2;
  }
}

// One kernel-level operation of a forward.
struct Op {
  int kind;   // PhaseKind
  GemmDesc g;
  AttnDesc a;
  EmbedDesc e;
};

// Operations of one model's forward over ntok tokens.  tokens = tok_base +
// *tok_idx + tok_off; positions = *pos_idx + pos_off + t.  LM-head logits of
// rows [lrow0, lrow0 + lrows) go to logits ([lrows][V]).  Per layer: q/k/v
// GEMM (input RMSNorm on load, RoPE + KV append in its epilogue), attention,
// o-projection + residual (writes the next norm's sums of squares), gate/up
// GEMM (RMSNorm on load, SwiGLU epilogue), down-projection + residual.
// pregain (bf16 models): the residual producers also write x times the next
// RMSNorm's gain in bf16 (c->xg), which the normalised GEMMs read (x_norm =
// 2) and scale by 1/rms after the sums.
// Sequences of a batched pass (batch > 1, per-operation path): the pass's
// tokens are spt per sequence for sequences seq0 .. seq0 + n - 1 of the
// context; tok_base / tok_idx / pos_idx then point at sequence seq0's token
// array and state, and sequence b's are tok_ld / kStateLd further.  spt = 0:
// one sequence (the batch-1 layout).
struct Seqs {
  int spt = 0;
  int64_t tok_ld = 0;
  int seq0 = 0;
};

std::vector<Op> forward_ops(spec_ctx* c, ModelState& m, int ntok, const int32_t* tok_base,
                            const int32_t* tok_idx, int tok_off, const int32_t* pos_idx,
                            int pos_off, int lrow0, int lrows, float* logits, bool pregain = false,
                            const Seqs& sq = Seqs()) {
  const spec_model_desc& d = m.d;
  const int dm = d.d_model, hq = d.n_heads, hkv = d.n_kv_heads, hd = d.head_dim;
  const int qkvr = m.qkv_rows();
  const int dt = d.dtype;
  const int q4 = m.q4 ? 1 : 0;
  std::vector<Op> ops;
  Op op{};
  op.kind = kPhaseEmbed;
  op.e.tok_base = tok_base; op.e.tok_idx = tok_idx; op.e.tok_off = tok_off; op.e.embed = d.embed;
  op.e.dtype = dt; op.e.x = c->x; op.e.ss = c->ss; op.e.ss_ld = c->tok_max; op.e.ntok = ntok;
  op.e.d = dm;
  op.e.spt = sq.spt; op.e.idx_ld = kStateLd; op.e.tok_ld = sq.tok_ld;
  if (pregain) {
    op.e.xg = c->xg;
    op.e.gain = (const float*)m.layers[0].attn_norm;
  }
  ops.push_back(op);
  // a normalised GEMM's X: the fp32 residual normalised on load, or its
  // pre-multiplied bf16 copy
  auto norm_x = [&](GemmDesc& g, const void* gain, int row0) {
    g.ldx = dm;
    g.gain = (const float*)gain;
    if (pregain) {
      g.x = (const uint16_t*)c->xg + (size_t)row0 * dm;
      g.x_norm = 2;
    } else {
      g.x = c->x + (size_t)row0 * dm;
      g.x_norm = 1;
    }
  };
  for (int l = 0; l < d.n_layers; ++l) {
    const spec_layer_weights& w = m.layers[l];
    const size_t kvoff = ((size_t)l * c->B + sq.seq0) * m.layer_kv_elems(c->cap) * m.esize;
    void* kc = (char*)m.kc + kvoff;
    void* vc = (char*)m.vc + kvoff;
    Op q{};
    q.kind = kPhaseGemm;
    GemmDesc& g = q.g;
    g.w[0] = w.wq; g.w[1] = w.wk; g.w[2] = w.wv;
    g.seg_rows[0] = hq * hd; g.seg_rows[1] = hkv * hd; g.seg_rows[2] = hkv * hd;
    g.n = qkvr; g.k = dm; g.ntok = ntok;
    norm_x(g, w.attn_norm, 0);
    g.ss_in = c->ss; g.ss_ld = c->tok_max; g.eps = d.rms_eps;
    g.epi = kEpiQkvRope; g.hq = hq; g.hkv = hkv; g.hd = hd; g.cap = c->cap;
    g.pos_base = pos_idx; g.pos_off = pos_off; g.rope_cos = m.rope_cos; g.rope_sin = m.rope_sin;
    g.spt = sq.spt; g.pos_ld = kStateLd;
    g.q_out = c->q; g.kc = kc; g.vc = vc;
    g.q4 = q4;
    ops.push_back(q);
    Op at{};
    at.kind = kPhaseAttn;
    AttnDesc& a = at.a;
    a.q = c->q; a.kc = kc; a.vc = vc; a.pos_base = pos_idx; a.pos_off = pos_off;
    a.spt = sq.spt; a.pos_ld = kStateLd; a.seq0 = sq.seq0;
    // batched passes of several tokens per sequence with one-token items for
    // at least two waves: token-group items (the same bits, half the walks)
    a.group = sq.spt >= 2 && (long long)ntok * hkv * (hd >= 64 ? 2 : 1) >= 2LL * c->num_sms;
    // batched passes of 3+ tokens per sequence with at least one wave of
    // (sequence, KV head, V part) items: wide items, all G heads of 2 x tiles
    // tokens per K/V walk (the same bits; K/V read up to 3x less often)
    if (sq.spt >= 3 && hq / hkv <= 8 && (long long)(ntok / sq.spt) * hkv * (hd >= 64 ? 2 : 1) >= c->num_sms)
      a.wide = sq.spt <= 4 ? 2 : 3;
    a.partials = c->attn_part; a.tickets = c->attn_tick; a.out = c->attn;
    a.ntok = ntok; a.hq = hq; a.hkv = hkv; a.hd = hd; a.cap = c->cap;
    a.max_chunks = c->max_chunks; a.dtype = dt;
    a.scale = 1.0f / sqrtf((float)hd);
    if (m.kv_maps) {
      a.tmk = m.kv_maps + 2 * l;
      a.tmv = m.kv_maps + 2 * l + 1;
    }
    a.err = res_err(c);
    ops.push_back(at);
    Op o{};
    o.kind = kPhaseGemm;
    o.g.w[0] = w.wo; o.g.seg_rows[0] = dm; o.g.n = dm; o.g.k = hq * hd; o.g.x = c->attn;
    o.g.ldx = hq * hd; o.g.ntok = ntok; o.g.epi = kEpiAdd; o.g.out = c->x; o.g.ldo = dm;
    if (pregain) {
      o.g.xg_out = c->xg;
      o.g.gain_next = (const float*)w.ffn_norm;
    }
    o.g.ss_out = c->ss; o.g.ss_ld = c->tok_max;
    o.g.q4 = q4;
    ops.push_back(o);
    Op gu{};
    gu.kind = kPhaseGemm;
    gu.g.w[0] = w.w_gate; gu.g.w[1] = w.w_up; gu.g.n = d.ffn_dim; gu.g.k = dm; gu.g.ntok = ntok;
    norm_x(gu.g, w.ffn_norm, 0);
    gu.g.ss_in = c->ss; gu.g.ss_ld = c->tok_max; gu.g.eps = d.rms_eps;
    gu.g.epi = kEpiSwiglu; gu.g.out = c->hbuf; gu.g.ldo = d.ffn_dim;
    gu.g.q4 = q4;
    ops.push_back(gu);
    Op dn{};
    dn.kind = kPhaseGemm;
    dn.g.w[0] = w.w_down; dn.g.seg_rows[0] = dm; dn.g.n = dm; dn.g.k = d.ffn_dim; dn.g.x = c->hbuf;
    dn.g.ldx = d.ffn_dim; dn.g.ntok = ntok; dn.g.epi = kEpiAdd; dn.g.out = c->x; dn.g.ldo = dm;
    if (pregain) {
      dn.g.xg_out = c->xg;
      dn.g.gain_next = (const float*)(l + 1 < d.n_layers ? m.layers[l + 1].attn_norm : d.final_norm);
    }
    dn.g.ss_out = c->ss; dn.g.ss_ld = c->tok_max;
    dn.g.early_prefetch = 1;   // follows the gate/up GEMM
    dn.g.q4 = q4;
    ops.push_back(dn);
  }
  if (lrows > 0) {
    Op h{};
    h.kind = kPhaseGemm;
    h.g.w[0] = d.lm_head; h.g.seg_rows[0] = d.vocab; h.g.n = d.vocab; h.g.k = dm; h.g.ntok = lrows;
    norm_x(h.g, d.final_norm, lrow0);
    h.g.ss_in = c->ss + lrow0; h.g.ss_ld = c->tok_max; h.g.eps = d.rms_eps;
    h.g.epi = kEpiStore; h.g.out = logits; h.g.ldo = d.vocab;
    h.g.q4 = q4;
    ops.push_back(h);
  }
  return ops;
}

// The heads pass: z_i = u + silu(W_i u) for the K stacked heads (one GEMM
// over the kept input row), then the target's LM head over the K rows z_i
// into the q rows.
std::vector<Op> heads_ops(spec_ctx* c) {
  const ModelState& m = c->tgt;
  const spec_model_desc& d = m.d;
  const int dm = d.d_model, K = c->K;
  std::vector<Op> ops;
  Op a{};
  a.kind = kPhaseGemm;
  GemmDesc& g = a.g;
  g.w[0] = c->heads; g.seg_rows[0] = K * dm; g.n = K * dm; g.k = dm; g.ntok = 1;
  g.x = c->hin_x; g.ldx = dm; g.x_norm = d.dtype == SPEC_DTYPE_BF16 ? 2 : 1;
  g.gain = (const float*)d.final_norm; g.ss_in = c->hin_ss; g.ss_ld = 1; g.eps = d.rms_eps;
  g.epi = kEpiHeadRes; g.hres = c->hin_u; g.out = c->zbuf; g.ldo = K * dm;
  ops.push_back(a);
  Op h{};
  h.kind = kPhaseGemm;
  h.g.w[0] = d.lm_head; h.g.seg_rows[0] = d.vocab; h.g.n = d.vocab; h.g.k = dm; h.g.ntok = K;
  h.g.x = c->zbuf; h.g.ldx = dm; h.g.x_norm = 0;
  h.g.epi = kEpiStore; h.g.out = c->logits_q; h.g.ldo = d.vocab;
  h.g.q4 = m.q4 ? 1 : 0;
  ops.push_back(h);
  return ops;
}

// Keeps the LM-head input row of the last scored position as the next heads
// pass's input: row *count - 1 of the verify pass (count = emitted tokens),
// or row `row` of a prefill / plain-decoding pass.
void keep_head_input(Launch& L, const int32_t* count, int row) {
  spec_ctx* c = L.c;
  if (!c->heads) return;
  const ModelState& m = c->tgt;
  const bool bf = m.d.dtype == SPEC_DTYPE_BF16;
  HeadInDesc h{};
  h.x = bf ? c->xg : (const void*)c->x; h.x_bf16 = bf ? 1 : 0; h.ldx = m.d.d_model;
  h.ss = c->ss; h.ss_ld = c->tok_max;
  h.count = count; h.row = row; h.max_row = c->K;
  h.d = m.d.d_model; h.gain = (const float*)m.d.final_norm; h.eps = m.d.rms_eps;
  h.err = res_err(c);
  h.out_x = c->hin_x; h.out_ss = c->hin_ss; h.out_u = c->hin_u;
  L.note(launch_head_input(h, c->stream));
}

// Per-kernel path: one launch per operation.
void forward(Launch& L, ModelState& m, int ntok, const int32_t* tok_base, const int32_t* tok_idx,
             int tok_off, const int32_t* pos_idx, int pos_off, int lrow0, int lrows,
             float* logits, const Seqs& sq = Seqs()) {
  spec_ctx* c = L.c;
  // bf16 models: normalised GEMM inputs as x * gain in bf16 (as in the
  // persistent kernel), 1/rms applied after the sums
  const std::vector<Op> ops = forward_ops(c, m, ntok, tok_base, tok_idx, tok_off, pos_idx, pos_off, lrow0,
                                          lrows, logits, m.d.dtype == SPEC_DTYPE_BF16, sq);
  for (const Op& op : ops) {
    if (op.kind == kPhaseEmbed) L.note(launch_embed(op.e, c->stream));
    else if (op.kind == kPhaseAttn) {
      if (m.d.dtype == SPEC_DTYPE_BF16) {   // same attention arithmetic as the persistent kernel
        AttnDesc a = op.a;
        a.tickets = c->dattn_tick;
        L.note(launch_dattn(a, c->stream));
      } else {
        L.note(launch_attention(op.a, c->stream));
      }
    }
    else gemm(L, op.g, m.d.dtype);
  }
}

// True when every GEMM of the model meets the tensor-memory GEMM's tiling
// (128-row tiles of the q/k/v segments and of d_model, 64-row gate/up
// tiles, k in 64-element blocks).
bool tc_model_ok(const ModelState& m) {
  const spec_model_desc& d = m.d;
  const int hd = d.head_dim, q = d.n_heads * hd, kv = d.n_kv_heads * hd;
  return d.dtype == SPEC_DTYPE_BF16 && d.d_model % 128 == 0 && q % 128 == 0 && kv % 128 == 0 &&
         128 % hd == 0 && d.ffn_dim % 64 == 0;
}

// Batched per-operation forward: spt tokens of every sequence, token j of
// sequence b taken from seq[b][L_b + tok_off + j] at position L_b + pos_off
// + j; the LM-head logits of all B * spt rows go to logits ([B][spt][V]).
// Sequences are processed in groups of at most c->tok_max tokens (each group
// streams the weights once; groups of more than kGemmMaxTok tokens run their
// GEMMs on the tensor-memory GEMM, when the model's shapes allow it); the
// fewest groups, as even as whole sequences allow.
void forward_batch(Launch& L, ModelState& m, int spt, int tok_off, int pos_off, float* logits) {
  spec_ctx* c = L.c;
  const int cap = std::max(1, (tc_model_ok(m) ? c->tok_max : kGemmMaxTok) / spt);
  const int ngroups = (c->B + cap - 1) / cap;
  const int per = (c->B + ngroups - 1) / ngroups;
  const size_t V = (size_t)m.d.vocab;
  for (int b0 = 0; b0 < c->B; b0 += per) {
    const int n = std::min(per, c->B - b0);
    Seqs sq;
    sq.spt = spt; sq.tok_ld = c->seq_ld; sq.seq0 = b0;
    const int32_t* stb = c->st + (size_t)b0 * kStateLd;
    forward(L, m, n * spt, c->seq + (size_t)b0 * c->seq_ld, stb, tok_off, stb, pos_off, 0, n * spt,
            logits + (size_t)b0 * spt * V, sq);
  }
}

// Persistent path: one cooperative launch for the whole forward, from a
// phase list prepared at init (index into c->pforward).
void forward_persist(Launch& L, int which) {
  spec_ctx* c = L.c;
  const PersistFwd& f = c->pforward[which];
  if (f.desc.times)
    L.note(cudaMemsetAsync(f.desc.times, 0,
                           sizeof(unsigned long long) * (1 + (size_t)kPhaseStamps * f.desc.nphases), c->stream));
  L.note(launch_persist(f.desc, f.hd, c->grp, f.smem, c->num_sms, c->stream));
}

// Sampler rows of a context: row b is sequence b (its step counter at
// st[b][which], Philox row word b), drawing into out_token[b * out_ld +
// (out_idx ? L_b : 0) + out_off].
SampleDesc sampler(spec_ctx* c, int which, int32_t* out_token, int64_t out_ld, const int32_t* out_idx,
                   int out_off) {
  SampleDesc sd{};
  sd.rows = c->B; sd.V = c->tgt.d.vocab; sd.temperature = c->opts.temperature; sd.seed = c->opts.seed;
  sd.batch = 1; sd.st_ld = kStateLd; sd.seq_ld = c->seq_ld;
  sd.step_dev = c->st + which; sd.step_base = 0;
  sd.out_token = out_token; sd.out_ld = out_ld; sd.out_idx = out_idx; sd.out_off = out_off;
  sd.partials = c->samp_part; sd.tickets = c->samp_tick;
  return sd;
}

void enqueue_draft(Launch& L) {
  spec_ctx* c = L.c;
  const int K = c->K, V = c->tgt.d.vocab;
  if (c->heads) {   // one heads pass, then the K drafts in one sampler launch
    if (c->persist) {
      forward_persist(L, c->heads_pass);
    } else {
      for (const Op& op : heads_ops(c)) gemm(L, op.g, c->tgt.d.dtype);
    }
    SampleDesc sd = sampler(c, 1, c->seq, 0, c->st, 1);   // draft i -> seq[L + i]
    sd.batch = 0; sd.rows = K; sd.row_pos = 1;
    sd.position = 1; sd.stream = kStreamDraft;
    sd.logits = c->logits_q; sd.ld = V;
    L.note(launch_sample(sd, c->stream));
    return;
  }
  if (c->lookup) {   // prompt lookup: drafts and one-hot q rows in one launch
    LookupDesc ld{};
    ld.seq = c->seq; ld.seq_ld = c->seq_ld; ld.lens = c->st; ld.st_ld = kStateLd;
    ld.rows = c->B; ld.K = K; ld.n_max = c->lookup; ld.V = V;
    ld.q_out = c->logits_q; ld.q_ld = (int64_t)K * V;
    L.note(launch_lookup(ld, c->stream));
    return;
  }
  const int32_t* Lp = c->st;  // committed length index (position of the pending token)
  const bool mix = c->opts.draft_mix_lambda != 0.f;
  for (int i = 1; i <= K; ++i) {
    float* qrow = c->logits_q + (size_t)(i - 1) * V;   // q row i of sequence b: qrow + b * K * V
    const int S = i == 1 ? 2 : 1;                        // tokens per sequence of this pass
    if (c->persist)
      forward_persist(L, i - 1);
    else if (c->B == 1 && i == 1)
      forward(L, c->drf, 2, c->seq, Lp, -1, Lp, -1, 1, 1, qrow);
    else if (c->B == 1)
      forward(L, c->drf, 1, c->seq, Lp, i - 1, Lp, i - 1, 0, 1, qrow);
    else
      forward_batch(L, c->drf, S, i == 1 ? -1 : i - 1, i == 1 ? -1 : i - 1, c->logits_d);
    SampleDesc sd = sampler(c, 1, c->seq, c->seq_ld, Lp, i);
    sd.position = (uint32_t)i; sd.stream = kStreamDraft;
    if (c->B == 1) {
      sd.logits = qrow; sd.ld = V;
    } else {   // the last row of each sequence; the row is kept as q_i
      sd.logits = c->logits_d + (size_t)(S - 1) * V; sd.ld = (int64_t)S * V;
      sd.mixed_out = qrow; sd.mixed_ld = (int64_t)K * V;
    }
    if (mix) {   // batch 1 only
      sd.mix_src = c->logits_p + (size_t)(i - 1) * V; sd.mix_ld = V;
      sd.lambda = c->opts.draft_mix_lambda; sd.mixed_out = qrow; sd.mixed_ld = V;
    }
    L.note(launch_sample(sd, c->stream));
  }
}

void enqueue_verify(Launch& L, bool commit) {
  spec_ctx* c = L.c;
  const int K = c->K, V = c->tgt.d.vocab, B = c->B;
  const int32_t* Lp = c->st;
  const bool was = c->timing_verify;
  c->timing_verify = commit && (c->opts.flags & SPEC_OPT_TIMING) != 0;
  if (c->persist)
    forward_persist(L, K);
  else if (B == 1)
    forward(L, c->tgt, K + 1, c->seq, Lp, 0, Lp, 0, 0, K + 1, c->logits_p);
  else
    forward_batch(L, c->tgt, K + 1, 0, 0, c->logits_p);
  c->timing_verify = was;
  AcceptDesc ad{};
  ad.p = c->logits_p; ad.p_ld = (int64_t)(K + 1) * V; ad.q = c->logits_q; ad.q_ld = (int64_t)K * V;
  ad.batch = 1; ad.st_ld = kStateLd; ad.seq_ld = c->seq_ld;
  ad.drafts = c->seq; ad.drafts_idx = Lp; ad.drafts_off = 1;
  ad.drafts_copy = c->result + (size_t)B * (K + 3);
  ad.rows = B; ad.K = K; ad.V = V; ad.temperature = c->opts.temperature; ad.seed = c->opts.seed;
  ad.step_dev = c->st + 1; ad.step_base = 0;
  ad.out_tokens = c->result; ad.out_count = c->result + (size_t)B * (K + 1);
  ad.out_flags = (uint32_t*)(c->result + (size_t)B * (K + 2));
  if (commit) {
    ad.commit_seq = c->seq; ad.commit_len = c->st; ad.commit_step = c->st + 1;
    ad.err = res_err(c);   // no commit after a forward that gave up
  }
  ad.partials = c->acc_part; ad.tickets = c->acc_tick;
  L.note(launch_accept(ad, c->stream));
}

void enqueue_step(Launch& L) {
  spec_ctx* c = L.c;
  enqueue_draft(L);
  enqueue_verify(L, true);
  keep_head_input(L, c->result + (size_t)c->B * (c->K + 1), 0);   // verify row n = count - 1
  L.note(cudaMemcpyAsync(c->h_result, c->result, sizeof(int32_t) * res_words(c),
                         cudaMemcpyDeviceToHost, c->stream));
  c->launch_count--;  // the copy is not a kernel
}

void enqueue_verify_only(Launch& L) { enqueue_verify(L, false); }

// The verify forward alone (the target over the K+1 positions, no acceptance).
void enqueue_verify_forward(Launch& L) {
  spec_ctx* c = L.c;
  const int32_t* Lp = c->st;
  if (c->persist)
    forward_persist(L, c->K);
  else if (c->B == 1)
    forward(L, c->tgt, c->K + 1, c->seq, Lp, 0, Lp, 0, 0, c->K + 1, c->logits_p);
  else
    forward_batch(L, c->tgt, c->K + 1, 0, 0, c->logits_p);
}

void enqueue_ar_pass(Launch& L, bool commit) {
  spec_ctx* c = L.c;
  const int V = c->tgt.d.vocab;
  const int32_t* Lp = c->st;
  if (c->persist)
    forward_persist(L, c->K + 1);
  else if (c->B == 1)
    forward(L, c->tgt, 1, c->seq, Lp, 0, Lp, 0, 0, 1, c->logits_p);
  else
    forward_batch(L, c->tgt, 1, 0, 0, c->logits_p);
  SampleDesc sd = sampler(c, 2, c->result, 1, nullptr, 0);   // token of sequence b -> result[b]
  sd.logits = c->logits_p; sd.ld = V;
  sd.position = 0; sd.stream = kStreamAR;
  if (commit) {
    sd.commit_seq = c->seq; sd.commit_len = c->st; sd.commit_step = c->st + 2;
    sd.err = res_err(c);
  }
  L.note(launch_sample(sd, c->stream));
}

void enqueue_ar(Launch& L) {
  spec_ctx* c = L.c;
  enqueue_ar_pass(L, true);
  keep_head_input(L, nullptr, 0);
  L.note(cudaMemcpyAsync(c->h_result, c->result, sizeof(int32_t) * res_words(c),
                         cudaMemcpyDeviceToHost, c->stream));
  c->launch_count--;
}

void enqueue_ar_only(Launch& L) { enqueue_ar_pass(L, false); }

int capture(spec_ctx* c, cudaGraphExec_t* exec, void (*enq)(Launch&), int* nkern) {
  CUDA_TRY(c, cudaStreamBeginCapture(c->stream, cudaStreamCaptureModeRelaxed));
  Launch L{c};
  c->launch_count = 0;
  enq(L);
  cudaGraph_t g = nullptr;
  cudaError_t e2 = cudaStreamEndCapture(c->stream, &g);
  CUDA_TRY(c, L.e);
  CUDA_TRY(c, e2);
  *nkern = c->launch_count;
  cudaError_t e3 = cudaGraphInstantiate(exec, g, 0);
  cudaGraphDestroy(g);
  CUDA_TRY(c, e3);
  return SPEC_OK;
}

bool use_graph(const spec_ctx* c) {
  return !(c->opts.flags & (SPEC_OPT_NO_GRAPH | SPEC_OPT_TIMING));
}

int run_captured(spec_ctx* c, cudaGraphExec_t* exec, void (*enq)(Launch&), int* nkern) {
  if (!use_graph(c)) {
    Launch L{c};
    c->launch_count = 0;
    enq(L);
    *nkern = c->launch_count;
    CUDA_TRY(c, L.e);
    return SPEC_OK;
  }
  if (!*exec) {
    int rc = capture(c, exec, enq, nkern);
    if (rc) return rc;
  }
  CUDA_TRY(c, cudaGraphLaunch(*exec, c->stream));
  return SPEC_OK;
}

void free_ctx(spec_ctx* c) {
  if (!c) return;
  for (cudaGraphExec_t g : c->step_exec)
    if (g) cudaGraphExecDestroy(g);
  if (c->ar_exec) cudaGraphExecDestroy(c->ar_exec);
  for (auto& pe : c->prof_exec)
    for (cudaGraphExec_t g : pe)
      if (g) cudaGraphExecDestroy(g);
  for (cudaEvent_t e : c->ev) cudaEventDestroy(e);
  for (auto& a : c->allocs) {
    cudaFree(a.first);
    g_device_bytes -= (long long)a.second;
  }
  if (c->h_result) cudaFreeHost(c->h_result);
  if (c->h_pos) cudaFreeHost(c->h_pos);
  if (c->own_stream && c->stream) cudaStreamDestroy(c->stream);
  delete c;
}

// A grid-barrier wait of a persistent kernel gave up: clear the flag and the
// barrier state so that the context stays usable, and report the timeout.
int persist_timeout(spec_ctx* c) {
  cudaMemsetAsync(res_err(c), 0, sizeof(int32_t), c->stream);
  if (c->bar) cudaMemsetAsync(c->bar, 0, sizeof(unsigned) * 4, c->stream);
  // kernels that left mid-phase may hold split-tile or attention tickets
  cudaMemsetAsync(c->gs.tickets, 0, sizeof(int) * c->gs.max_tiles, c->stream);
  cudaMemsetAsync(c->dattn_tick, 0, sizeof(int) * c->dattn_nt, c->stream);
  cudaStreamSynchronize(c->stream);
  return fail(c, SPEC_E_TIMEOUT, "a bounded wait of a forward kernel (grid barrier or copy) timed out");
}

// Position of a host-driven forward of sequence b: st[b][3] = pos.
int set_eager_pos(spec_ctx* c, int pos, int b = 0) {
  *c->h_pos = pos;
  CUDA_TRY(c, cudaMemcpyAsync(c->st + (size_t)b * kStateLd + 3, c->h_pos, sizeof(int32_t),
                              cudaMemcpyHostToDevice, c->stream));
  return SPEC_OK;
}

}  // namespace

extern "C" {

const char* spec_version(void) { return "specverify-gb300 0.1 (sm_103a)"; }

const char* spec_last_error(const spec_ctx* ctx) {
  return ctx ? ctx->err.c_str() : g_err.c_str();
}

void spec_free(spec_ctx* ctx) { free_ctx(ctx); }

int spec_init(const spec_model_desc* target, const spec_model_desc* draft, int K,
              const spec_opts* opts, spec_ctx** out) {
  // an injected allocation failure applies to this call only, fired or not
  struct Disarm {
    ~Disarm() { g_fail_alloc_at = 0; }
  } disarm;
  if (!out) return fail(nullptr, SPEC_E_ARG, "spec_init: null output pointer");
  *out = nullptr;
  std::string why;
  int rc;
  if (!opts) return fail(nullptr, SPEC_E_ARG, "spec_init: null opts");
  if ((rc = check_model(target, "target", &why)) != SPEC_OK) return fail(nullptr, rc, why);
  // self-draft heads: no draft model (the target's shape sizes the draft-side buffers)
  const bool heads = opts->draft_heads != nullptr;
  if (heads && draft && draft != target)
    return fail(nullptr, SPEC_E_ARG, "self-draft heads replace the draft model: pass draft = NULL (or the target)");
  if (heads) draft = target;
  if ((rc = check_model(draft, "draft", &why)) != SPEC_OK) return fail(nullptr, rc, why);
  if (heads && (opts->batch != 1 || opts->draft_lookup != 0 || opts->draft_mix_lambda != 0.f))
    return fail(nullptr, SPEC_E_ARG, "self-draft heads need batch 1, no prompt lookup and draft_mix_lambda 0");
  if (heads && (K > 8 || (reinterpret_cast<uintptr_t>(opts->draft_heads) & 15u)))
    return fail(nullptr, SPEC_E_ARG, "self-draft heads need K <= 8 and 16-byte aligned head weights");
  if (target->vocab != draft->vocab)
    return fail(nullptr, SPEC_E_VOCAB, "draft and target vocabularies differ (" +
                                           std::to_string(draft->vocab) + " vs " +
                                           std::to_string(target->vocab) + ")");
  if (K < 1 || K > 16) return fail(nullptr, SPEC_E_ARG, "K must be in 1..16");
  if (opts->batch < 1 || opts->batch > SPEC_MAX_BATCH)
    return fail(nullptr, SPEC_E_ARG, "batch must be in 1..SPEC_MAX_BATCH");
  if (opts->batch > 1 && (target->dtype != SPEC_DTYPE_BF16 || draft->dtype != SPEC_DTYPE_BF16))
    return fail(nullptr, SPEC_E_ARG, "batch > 1 needs bf16 target and draft models");
  const bool any_q4 = target->dtype == SPEC_DTYPE_Q4 || draft->dtype == SPEC_DTYPE_Q4;
  if (any_q4 && (opts->flags & (SPEC_OPT_NO_PERSIST | SPEC_OPT_TIMING)))
    return fail(nullptr, SPEC_E_ARG, "4-bit models run only on the persistent kernel (no NO_PERSIST / TIMING)");
  if (any_q4 && K + 1 > kPrefillChunk) return fail(nullptr, SPEC_E_ARG, "4-bit models need K <= 7");
  if (opts->batch > 1 && opts->draft_mix_lambda != 0.f)
    return fail(nullptr, SPEC_E_ARG, "batch > 1 does not support draft_mix_lambda");
  if (opts->draft_lookup < 0 || opts->draft_lookup > kLookupMaxN)
    return fail(nullptr, SPEC_E_ARG, "draft_lookup must be in 0..8");
  if (opts->draft_lookup > 0 && opts->draft_mix_lambda != 0.f)
    return fail(nullptr, SPEC_E_ARG, "prompt lookup has no draft logits to mix (draft_mix_lambda must be 0)");
  if (opts->max_ctx < K + 3) return fail(nullptr, SPEC_E_ARG, "max_ctx must be at least K + 3");
  if (!(opts->temperature >= 0.f)) return fail(nullptr, SPEC_E_ARG, "temperature must be >= 0");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(nullptr, SPEC_E_CUDA, std::string("no CUDA device: ") + cudaGetErrorString(e));

  spec_ctx* c = new spec_ctx();
  c->K = K;
  c->B = opts->batch;
  c->lookup = opts->draft_lookup;
  c->heads = opts->draft_heads;
  c->opts = *opts;
  c->cap = opts->max_ctx;
  c->seq_ld = (int64_t)c->cap + K + 2;
  c->host_Ls.assign(c->B, 0);
  c->max_chunks = (c->cap + kAttnChunk - 1) / kAttnChunk;
  auto setup_model = [&](ModelState& m, const spec_model_desc* d) {
    m.d = *d;
    m.q4 = d->dtype == SPEC_DTYPE_Q4;
    if (m.q4) m.d.dtype = SPEC_DTYPE_BF16;   // the arithmetic and the KV cache are bf16
    m.layers.assign(d->layers, d->layers + d->n_layers);
    m.d.layers = m.layers.data();
    m.esize = m.d.dtype == SPEC_DTYPE_BF16 ? 2 : 4;
  };
  setup_model(c->tgt, target);
  setup_model(c->drf, draft);
#define INIT_TRY(expr)                                                                      \
  do {                                                                                      \
    cudaError_t e__ = (expr);                                                               \
    if (e__ != cudaSuccess) {                                                               \
      const int code__ = (e__ == cudaErrorMemoryAllocation) ? SPEC_E_OOM : SPEC_E_CUDA;     \
      std::string m__ = std::string(#expr) + ": " + cudaGetErrorString(e__);                \
      free_ctx(c);                                                                          \
      return fail(nullptr, code__, m__);                                                    \
    }                                                                                       \
  } while (0)
  INIT_TRY(cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, dev));
  set_pdl_enabled((opts->flags & SPEC_OPT_PDL) != 0);
  INIT_TRY(configure_kernels());
  if (opts->cuda_stream) {
    c->stream = (cudaStream_t)opts->cuda_stream;
  } else {
    INIT_TRY(cudaStreamCreateWithFlags(&c->stream, cudaStreamNonBlocking));
    c->own_stream = true;
  }
  const int V = target->vocab;
  c->tok_max = opts->batch > 1 ? kTcMaxTok : kGemmMaxTok;
  const int maxN = c->tok_max;
  auto mx = [&](auto f) { return std::max(f(c->tgt.d), f(c->drf.d)); };
  const size_t dmax = mx([](const spec_model_desc& d) { return (size_t)d.d_model; });
  const size_t fmax = mx([](const spec_model_desc& d) { return (size_t)d.ffn_dim; });
  const size_t qkvmax = mx([](const spec_model_desc& d) {
    return (size_t)(d.n_heads + 2 * d.n_kv_heads) * d.head_dim; });
  const size_t hqd = mx([](const spec_model_desc& d) { return (size_t)d.n_heads * d.head_dim; });
  const size_t hqmax = mx([](const spec_model_desc& d) { return (size_t)d.n_heads; });
  const size_t hdmax = mx([](const spec_model_desc& d) { return (size_t)d.head_dim; });
  const int B = c->B;
  const size_t stw = std::max<size_t>(16, (size_t)kStateLd * B);
  INIT_TRY(dalloc(c, &c->st, stw * sizeof(int32_t)));
  INIT_TRY(cudaMemset(c->st, 0, stw * sizeof(int32_t)));
  INIT_TRY(dalloc(c, &c->seq, sizeof(int32_t) * B * c->seq_ld));
  INIT_TRY(cudaMemset(c->seq, 0, sizeof(int32_t) * B * c->seq_ld));
  INIT_TRY(dalloc(c, &c->fwd_tok, sizeof(int32_t) * maxN));
  INIT_TRY(dalloc(c, &c->x, sizeof(float) * maxN * dmax));
  INIT_TRY(dalloc(c, &c->xg, 2 * maxN * dmax));
  INIT_TRY(dalloc(c, &c->hbuf, 4 * maxN * fmax));
  INIT_TRY(dalloc(c, &c->ss, sizeof(float) * maxN * (dmax / 16 + 1)));
  INIT_TRY(dalloc(c, &c->q, sizeof(float) * maxN * hqd));
  INIT_TRY(dalloc(c, &c->attn, 4 * maxN * hqd));
  INIT_TRY(dalloc(c, &c->attn_part,
                  sizeof(float) * attn_partial_floats(maxN, (int)hqmax, (int)hdmax, c->max_chunks)));
  {
    const int hkvmax = std::max(c->tgt.d.n_kv_heads, c->drf.d.n_kv_heads);
    const int rt = std::max(attn_max_row_tiles(maxN, c->tgt.d.n_heads, c->tgt.d.n_kv_heads),
                            attn_max_row_tiles(maxN, c->drf.d.n_heads, c->drf.d.n_kv_heads));
    const size_t nt = (size_t)hkvmax * rt;
    INIT_TRY(dalloc(c, &c->attn_tick, sizeof(int) * nt));
    INIT_TRY(cudaMemset(c->attn_tick, 0, sizeof(int) * nt));
    const int dnt = std::max(dattn_tickets(maxN, c->tgt.d.n_heads, c->tgt.d.n_kv_heads),
                             dattn_tickets(maxN, c->drf.d.n_heads, c->drf.d.n_kv_heads));
    c->dattn_nt = dnt;
    INIT_TRY(dalloc(c, &c->dattn_tick, sizeof(int) * dnt));
    INIT_TRY(cudaMemset(c->dattn_tick, 0, sizeof(int) * dnt));
  }
  INIT_TRY(dalloc(c, &c->logits_p, sizeof(float) * (size_t)B * (K + 1) * V));
  INIT_TRY(dalloc(c, &c->logits_q, sizeof(float) * (size_t)B * K * V));
  if (B > 1) INIT_TRY(dalloc(c, &c->logits_d, sizeof(float) * (size_t)2 * B * V));
  c->gs.partial_floats = gemm_partial_floats(c->num_sms);
  c->gs.max_tiles = (int)std::max<size_t>(
      (V + 15) / 16, std::max(fmax / 8, (std::max(qkvmax, dmax) + 15) / 16));
  if (heads) c->gs.max_tiles = std::max(c->gs.max_tiles, (int)((size_t)K * dmax / 16));   // the stacked heads
  INIT_TRY(dalloc(c, &c->gs.partials, sizeof(float) * c->gs.partial_floats));
  INIT_TRY(dalloc(c, &c->gs.tickets, sizeof(int) * c->gs.max_tiles));
  INIT_TRY(cudaMemset(c->gs.tickets, 0, sizeof(int) * c->gs.max_tiles));
  if (c->tok_max > kGemmMaxTok) {
    const int maxn = (int)std::max<size_t>((size_t)V, std::max(2 * fmax, std::max(qkvmax, dmax)));
    const size_t tpf = tc_gemm_partial_floats(c->num_sms, maxn);
    c->tc_units = (long long)(tpf / ((size_t)128 * kTcMaxTok));
    INIT_TRY(dalloc(c, &c->tc_part, sizeof(float) * tpf));
    INIT_TRY(dalloc(c, &c->tc_inv, sizeof(float) * kTcMaxTok));
  }
  const size_t nt = std::max(std::max(4, B), K);   // sampler rows: sequences, or the K head drafts
  INIT_TRY(dalloc(c, &c->samp_part, sizeof(float) * sample_partial_floats(std::max(B, K), V)));
  INIT_TRY(dalloc(c, &c->samp_tick, sizeof(int) * nt));
  INIT_TRY(cudaMemset(c->samp_tick, 0, sizeof(int) * nt));
  INIT_TRY(dalloc(c, &c->acc_part, sizeof(float) * accept_partial_floats(B, K, V)));
  INIT_TRY(dalloc(c, &c->acc_tick, sizeof(int) * nt));
  INIT_TRY(cudaMemset(c->acc_tick, 0, sizeof(int) * nt));
  const size_t rw = (size_t)res_words(c) + 7;
  INIT_TRY(dalloc(c, &c->result, sizeof(int32_t) * rw));
  INIT_TRY(cudaMallocHost(&c->h_result, sizeof(int32_t) * rw));
  INIT_TRY(cudaMallocHost(&c->h_pos, sizeof(int32_t) * 4));
  if (heads) {   // the heads' input row and the LM-head input of the heads pass
    const size_t es = (size_t)c->tgt.esize;
    INIT_TRY(dalloc(c, &c->hin_x, es * dmax));
    INIT_TRY(dalloc(c, &c->hin_ss, sizeof(float) * (dmax / 16 + 1)));
    INIT_TRY(dalloc(c, &c->hin_u, sizeof(float) * dmax));
    INIT_TRY(dalloc(c, &c->zbuf, es * (size_t)K * dmax));
    INIT_TRY(cudaMemset(c->hin_x, 0, es * dmax));
    INIT_TRY(cudaMemset(c->hin_ss, 0, sizeof(float) * (dmax / 16 + 1)));
    INIT_TRY(cudaMemset(c->hin_u, 0, sizeof(float) * dmax));
  }
  for (ModelState* m : {&c->tgt, &c->drf}) {
    if (m == &c->drf && heads) continue;   // no draft model, no draft cache
    const size_t kvb = (size_t)m->d.n_layers * B * m->layer_kv_elems(c->cap) * m->esize;
    INIT_TRY(dalloc(c, &m->kc, kvb));
    INIT_TRY(dalloc(c, &m->vc, kvb));
    INIT_TRY(cudaMemset(m->kc, 0, kvb));
    INIT_TRY(cudaMemset(m->vc, 0, kvb));
    const size_t tb = sizeof(float) * (size_t)c->cap * (m->d.head_dim / 2);
    INIT_TRY(dalloc(c, &m->rope_cos, tb));
    INIT_TRY(dalloc(c, &m->rope_sin, tb));
    INIT_TRY(launch_rope_table(m->rope_cos, m->rope_sin, c->cap, m->d.head_dim,
                               (double)m->d.rope_theta, c->stream));
    if (m->d.dtype == SPEC_DTYPE_BF16) {   // tensor maps of every layer's K and V cache
      std::vector<TensorMap128> maps(2 * (size_t)m->d.n_layers);
      const long long rows = (long long)B * m->d.n_kv_heads * c->cap;   // every sequence of the layer
      bool ok = true;
      for (int l = 0; l < m->d.n_layers && ok; ++l) {
        const size_t off = (size_t)l * B * m->layer_kv_elems(c->cap) * m->esize;
        ok = encode_kv_map(maps[2 * l], (char*)m->kc + off, m->d.head_dim, rows) &&
             encode_kv_map(maps[2 * l + 1], (char*)m->vc + off, m->d.head_dim, rows,
                           dattn_v_box_cols(m->d.head_dim));
      }
      if (!ok) {
        free_ctx(c);
        return fail(nullptr, SPEC_E_CUDA, "could not encode the KV-cache tensor maps");
      }
      INIT_TRY(dalloc(c, &m->kv_maps, sizeof(TensorMap128) * maps.size()));
      INIT_TRY(cudaMemcpy(m->kv_maps, maps.data(), sizeof(TensorMap128) * maps.size(), cudaMemcpyHostToDevice));
    }
  }
  INIT_TRY(cudaMemset(c->result, 0, sizeof(int32_t) * rw));
  // Persistent forward kernels: both models bf16, and the weight ring plus
  // K+1 tokens of normalised input (or the attention tile) fit one CTA's
  // shared memory.
  if (B == 1 && c->tgt.d.dtype == SPEC_DTYPE_BF16 && c->drf.d.dtype == SPEC_DTYPE_BF16 &&
      !(opts->flags & (SPEC_OPT_TIMING | SPEC_OPT_NO_PERSIST))) {
    PersistLayout lay_t{}, lay_d{};
    const bool lay_ok = persist_layout(target->head_dim, K + 1, target->d_model, &lay_t) &&
                        persist_layout(draft->head_dim, 2, draft->d_model, &lay_d);
    if (lay_ok && persist_supported(target->head_dim, lay_t.total, c->num_sms, K + 1) &&
        persist_supported(draft->head_dim, lay_d.total, c->num_sms, 2)) {
      std::vector<PhaseDesc> all;
      std::vector<TensorMap128> maps;
      size_t start[24] = {}, count[24] = {};
      bool encodable = true;
      // decode-attention scratch: partials in the attention buffer, own tickets
      for (const spec_model_desc* m : {target, draft})
        encodable = encodable && persist_attn_partial_floats(K + 1, m->n_heads, m->head_dim, c->cap) <=
                                     attn_partial_floats(maxN, (int)hqmax, (int)hdmax, c->max_chunks);
      int* const dattn_tick = c->dattn_tick;   // sized for kGemmMaxTok >= K + 1 tokens
      auto add = [&](int idx, const std::vector<Op>& ops) {
        const bool drf = (idx < K || idx == K + 2 || idx == K + 6) && !heads;
        const PersistLayout& lay = drf ? lay_d : lay_t;
        start[idx] = all.size();
        int rev = 1, prev = kPhaseEmbed;
        for (const Op& op : ops) {
          PhaseDesc p{};
          if (op.kind == kPhaseEmbed) {
            persist_phase_from_embed(p, op.e);
          } else if (op.kind == kPhaseAttn) {
            encodable = persist_phase_from_attn(p, op.a) && encodable;
            p.a.tickets = dattn_tick;
          } else {
            encodable = persist_phase_from_gemm(p, op.g, maps, c->num_sms, lay) && encodable;
            // GEMM tile ranges alternate direction; after attention (whose
            // items run on the first CTAs) they are counted from the last CTA
            rev = prev == kPhaseAttn ? 1 : 1 - rev;
            p.rev = rev;
          }
          prev = op.kind;
          all.push_back(p);
        }
        count[idx] = ops.size();
      };
      for (int i = 1; i <= K && !heads; ++i) {
        float* qrow = c->logits_q + (size_t)(i - 1) * V;
        if (i == 1)
          add(0, forward_ops(c, c->drf, 2, c->seq, c->st, -1, c->st, -1, 1, 1, qrow, true));
        else
          add(i - 1, forward_ops(c, c->drf, 1, c->seq, c->st, i - 1, c->st, i - 1, 0, 1, qrow, true));
      }
      add(K, forward_ops(c, c->tgt, K + 1, c->seq, c->st, 0, c->st, 0, 0, K + 1, c->logits_p, true));
      add(K + 1, forward_ops(c, c->tgt, 1, c->seq, c->st, 0, c->st, 0, 0, 1, c->logits_p, true));
      // last scored prompt position (st[0] - 1) of both models, run by
      // spec_prefill so that its KV rows carry the step passes' arithmetic
      if (!heads) add(K + 2, forward_ops(c, c->drf, 1, c->seq, c->st, -1, c->st, -1, 0, 0, nullptr, true));
      add(K + 3, forward_ops(c, c->tgt, 1, c->seq, c->st, -1, c->st, -1, 0,
                             opts->draft_mix_lambda != 0.f ? 1 : 0, c->logits_p + (size_t)K * V, true));
      int nf = K + 4;
      if (any_q4) {   // prefill chunks at the host-set position st[3]
        INIT_TRY(dalloc(c, &c->logits_chunk, sizeof(float) * (size_t)kPrefillChunk * V));
        const int32_t* ep = c->st + 3;
        add(K + 4, forward_ops(c, c->tgt, kPrefillChunk, c->seq, ep, 0, ep, 0, 0, 0, nullptr, true));
        add(K + 5, forward_ops(c, c->tgt, kPrefillChunk, c->seq, ep, 0, ep, 0, 0, kPrefillChunk, c->logits_chunk,
                               true));
        if (!heads) add(K + 6, forward_ops(c, c->drf, kPrefillChunk, c->seq, ep, 0, ep, 0, 0, 0, nullptr, true));
        nf = K + 7;
      }
      if (heads) {   // the heads pass (the target's layout)
        c->heads_pass = nf;
        add(nf, heads_ops(c));
        nf += 1;
      }
      if (encodable) {
        INIT_TRY(dalloc(c, &c->phase_dev, sizeof(PhaseDesc) * all.size()));
        INIT_TRY(cudaMemcpy(c->phase_dev, all.data(), sizeof(PhaseDesc) * all.size(), cudaMemcpyHostToDevice));
        TensorMap128* tmaps_dev = nullptr;
        INIT_TRY(dalloc(c, &tmaps_dev, sizeof(TensorMap128) * maps.size()));
        INIT_TRY(cudaMemcpy(tmaps_dev, maps.data(), sizeof(TensorMap128) * maps.size(), cudaMemcpyHostToDevice));
        INIT_TRY(dalloc(c, &c->bar, sizeof(unsigned) * 4));
        INIT_TRY(cudaMemset(c->bar, 0, sizeof(unsigned) * 4));
        INIT_TRY(dalloc(c, &c->fault_ctl, sizeof(int) * 4));
        INIT_TRY(cudaMemset(c->fault_ctl, 0, sizeof(int) * 4));
        unsigned long long* times = nullptr;
        if (opts->flags & SPEC_OPT_PHASE_TIMES) {
          const size_t words = (size_t)nf + (size_t)kPhaseStamps * all.size();   // a start word per forward
          INIT_TRY(dalloc(c, &times, sizeof(unsigned long long) * words));
          INIT_TRY(cudaMemset(times, 0, sizeof(unsigned long long) * words));
        }
        for (int f = 0; f < nf; ++f) {
          PersistFwd& pf = c->pforward[f];
          pf.host.assign(all.begin() + start[f], all.begin() + start[f] + count[f]);
          if (times) pf.desc.times = times + f + (size_t)kPhaseStamps * start[f];
          pf.desc.phases = c->phase_dev + start[f];
          pf.desc.nphases = (int)count[f];
          pf.desc.tmaps = tmaps_dev;
          const bool drf = (f < K || f == K + 2 || f == K + 6) && !heads;
          pf.desc.ring_bytes = (int)(drf ? lay_d.ring : lay_t.ring);
          pf.desc.bar = c->bar;
          pf.desc.err = res_err(c);
          pf.desc.ctl = c->fault_ctl;
          pf.hd = drf ? draft->head_dim : target->head_dim;
          pf.smem = drf ? lay_d.total : lay_t.total;
        }
        c->persist = true;
      }
    }
  }
  if (any_q4 && !c->persist) {
    free_ctx(c);
    return fail(nullptr, SPEC_E_SHAPE,
                "4-bit models need the persistent kernel, which this pair does not fit (batch 1, K <= 7, "
                "head dims 32/64/128)");
  }
  c->q4 = any_q4;
  if (opts->flags & SPEC_OPT_TIMING) {
    const int n = 2 * (4 * target->n_layers + 1);
    c->ev.resize(n);
    c->ev_bytes.assign(n / 2, 0.0);
    for (auto& ev : c->ev) INIT_TRY(cudaEventCreate(&ev));
  }
  INIT_TRY(cudaStreamSynchronize(c->stream));
#undef INIT_TRY
  *out = c;
  return SPEC_OK;
}

// Step state of every sequence after a prefill of L tokens: L_b = L - 1
// (position of the pending token), step counters 0.
int reset_state(spec_ctx* c, int L) {
  for (int b = 0; b < c->B; ++b) {
    int32_t* w = c->h_result + (size_t)b * kStateLd;
    w[0] = L - 1; w[1] = 0; w[2] = 0; w[3] = 0;
  }
  CUDA_TRY(c, cudaMemcpyAsync(c->st, c->h_result, sizeof(int32_t) * kStateLd * c->B, cudaMemcpyHostToDevice,
                              c->stream));
  CUDA_TRY(c, cudaStreamSynchronize(c->stream));   // h_result is reused by the step read-back
  return SPEC_OK;
}

void mark_prefilled(spec_ctx* c, int L) {
  c->host_L = L - 1;
  c->host_Ls.assign(c->B, L - 1);
  c->prefilled = true;
  c->draft_stale = false;
  c->steps = c->ar_steps = c->emitted = c->accepted = 0;
  std::fill(std::begin(c->hist), std::end(c->hist), 0);
}

int max_host_L(const spec_ctx* c) { return *std::max_element(c->host_Ls.begin(), c->host_Ls.end()); }

int spec_prefill(spec_ctx* c, const int32_t* tokens, int L) {
  if (!c) return fail(nullptr, SPEC_E_ARG, "null context");
  if (!tokens || L < 2) return fail(c, SPEC_E_ARG, "prefill needs at least 2 tokens");
  if (L + c->K + 1 > c->cap) return fail(c, SPEC_E_CAPACITY, "prompt + K + 1 exceeds max_ctx");
  const bool mix = c->opts.draft_mix_lambda != 0.f;
  if (mix && L < c->K + 2) return fail(c, SPEC_E_ARG, "mixed draft needs a prompt of at least K + 2 tokens");
  const int V = c->tgt.d.vocab;
  for (size_t i = 0; i < (size_t)c->B * L; ++i)
    if (tokens[i] < 0 || tokens[i] >= V) return fail(c, SPEC_E_ARG, "token id out of range");
  c->prefilled = false;
  CUDA_TRY(c, cudaMemcpy2DAsync(c->seq, sizeof(int32_t) * c->seq_ld, tokens, sizeof(int32_t) * L,
                                sizeof(int32_t) * L, c->B, cudaMemcpyHostToDevice, c->stream));
  int rc = reset_state(c, L);
  if (rc) return rc;
  const int n = L - 1;   // positions 0..L-2 are scored; token L-1 is pending
  const int K = c->K;
  const int lo = n - (K + 1);  // rows of the previous-step logits before step 0
  // The first draft pass of a step recomputes position st[0] - 1.  On the
  // persistent path that position is scored here by the persistent kernel
  // too (both models), so that both KV caches hold the same bits for it.
  const int nk = c->persist ? n - 1 : n;   // positions scored one kernel per operation
  Launch Lc{c};
  if (c->q4) {   // 4-bit models: persistent chunks of kPrefillChunk positions (the last one overlapping)
    if (nk < kPrefillChunk) return fail(c, SPEC_E_ARG, "4-bit models need prompts of at least 10 tokens");
    for (int p0 = 0; p0 < nk; p0 += kPrefillChunk) {
      const int s0 = std::min(p0, nk - kPrefillChunk);
      const bool last = p0 + kPrefillChunk >= nk;
      rc = set_eager_pos(c, s0);
      if (rc) return rc;
      if (c->draft_model()) forward_persist(Lc, K + 6);
      forward_persist(Lc, last && mix ? K + 5 : K + 4);
      CUDA_TRY(c, Lc.e);
      CUDA_TRY(c, cudaStreamSynchronize(c->stream));   // the pinned position slot is reused
    }
    if (mix) {   // previous-step rows at positions lo .. n-2 from the last chunk (row n-1: pass K+3)
      const int r0 = lo - (nk - kPrefillChunk);
      CUDA_TRY(c, cudaMemcpyAsync(c->logits_p, c->logits_chunk + (size_t)r0 * V, sizeof(float) * (size_t)K * V,
                                  cudaMemcpyDeviceToDevice, c->stream));
    }
  }
  for (int b = 0; b < c->B && !c->q4; ++b) {   // sequence by sequence, in chunks of positions
    Seqs sq;
    sq.seq0 = b;
    const int32_t* sb = c->seq + (size_t)b * c->seq_ld;
    const int32_t* pb = c->st + (size_t)b * kStateLd + 3;
    for (int p0 = 0; p0 < nk; p0 += kGemmMaxTok) {
      const int nt = std::min(kGemmMaxTok, nk - p0);
      rc = set_eager_pos(c, p0, b);
      if (rc) return rc;
      if (c->draft_model()) forward(Lc, c->drf, nt, sb, nullptr, p0, pb, 0, 0, 0, nullptr, sq);
      int r0 = 0, rn = 0;
      if (mix) {
        r0 = std::max(lo, p0) - p0;
        rn = std::min(n, p0 + nt) - p0 - r0;
        if (rn < 0) rn = 0;
      }
      float* dst = c->logits_p + (size_t)std::max(0, p0 + r0 - lo) * V;
      forward(Lc, c->tgt, nt, sb, nullptr, p0, pb, 0, r0, rn, dst, sq);
      if (!c->persist && p0 + nt >= nk) keep_head_input(Lc, nullptr, nt - 1);   // position L-2
      CUDA_TRY(c, Lc.e);
      // the pinned position slot is reused by the next chunk
      CUDA_TRY(c, cudaStreamSynchronize(c->stream));
    }
  }
  if (c->persist) {
    c->grp = false;   // one token per pass
    if (c->draft_model()) forward_persist(Lc, K + 2);
    forward_persist(Lc, K + 3);
    keep_head_input(Lc, nullptr, 0);   // position L-2
    CUDA_TRY(c, Lc.e);
  }
  CUDA_TRY(c, cudaMemcpyAsync(c->h_result, c->result, sizeof(int32_t) * res_words(c), cudaMemcpyDeviceToHost,
                              c->stream));
  CUDA_TRY(c, cudaStreamSynchronize(c->stream));
  if (c->h_result[res_words(c) - 1]) return persist_timeout(c);
  mark_prefilled(c, L);
  return SPEC_OK;
}

int spec_prefill_synthetic(spec_ctx* c, int L, uint64_t seed) {
  if (!c) return fail(nullptr, SPEC_E_ARG, "null context");
  if (L < 2) return fail(c, SPEC_E_ARG, "need at least 2 positions");
  if (L + c->K + 1 > c->cap) return fail(c, SPEC_E_CAPACITY, "L + K + 1 exceeds max_ctx");
  c->prefilled = false;
  const int V = c->tgt.d.vocab;
  CUDA_TRY(c, launch_fill_tokens(c->seq, (size_t)c->B * c->seq_ld, V, seed, c->stream));
  uint64_t sub = 1;
  for (ModelState* m : {&c->tgt, &c->drf}) {
    const size_t elems = (size_t)m->d.n_layers * c->B * m->layer_kv_elems(c->cap);
    CUDA_TRY(c, launch_fill_normal(m->kc, elems, m->d.dtype, seed ^ (0x9E3779B97F4A7C15ull * sub++), c->stream));
    CUDA_TRY(c, launch_fill_normal(m->vc, elems, m->d.dtype, seed ^ (0x9E3779B97F4A7C15ull * sub++), c->stream));
  }
  int rc = reset_state(c, L);
  if (rc) return rc;
  mark_prefilled(c, L);
  return SPEC_OK;
}

int spec_seq_context(spec_ctx* c, int b, int32_t* context, int32_t* len) {
  if (!c) return fail(nullptr, SPEC_E_ARG, "null context");
  if (b < 0 || b >= c->B || !len) return fail(c, SPEC_E_ARG, "bad sequence index or null length");
  const int n = c->host_Ls[b] + 1;
  if (context) {   // on the context's stream, after anything still queued there
    CUDA_TRY(c, cudaMemcpyAsync(context, c->seq + (size_t)b * c->seq_ld, sizeof(int32_t) * n,
                                cudaMemcpyDeviceToHost, c->stream));
    CUDA_TRY(c, cudaStreamSynchronize(c->stream));
  }
  *len = n;
  return SPEC_OK;
}

int spec_step(spec_ctx* c, int32_t* out_tokens, int32_t* out_count, uint32_t* out_flags) {
  if (!c) return fail(nullptr, SPEC_E_ARG, "null context");
  if (!out_tokens || !out_count) return fail(c, SPEC_E_ARG, "null output buffer");
  if (!c->prefilled) return fail(c, SPEC_E_STATE, "spec_step before spec_prefill");
  if (c->draft_stale && c->draft_model())   // (prompt lookup and the heads keep no draft cache)
    return fail(c, SPEC_E_STATE, "draft cache is stale after spec_ar_step; prefill again");
  if (max_host_L(c) + c->K + 2 > c->cap) return fail(c, SPEC_E_CAPACITY, "context would exceed max_ctx");
  const int K = c->K, B = c->B;
  c->ev_used = 0;
  c->grp = c->host_L + K >= kDGroupMinPos;   // last verify position (persistent path: batch 1)
  int rc = run_captured(c, &c->step_exec[c->grp], enqueue_step, &c->kernels_step);
  if (rc) return rc;
  CUDA_TRY(c, cudaStreamSynchronize(c->stream));
  const int32_t* h = c->h_result;
  if (h[res_words(c) - 1]) return persist_timeout(c);
  for (int b = 0; b < B; ++b) {
    const int cnt = h[(size_t)B * (K + 1) + b];
    if (cnt < 1 || cnt > K + 1) return fail(c, SPEC_E_CUDA, "acceptance kernel returned an invalid count");
  }
  for (int b = 0; b < B; ++b) {
    const int cnt = h[(size_t)B * (K + 1) + b];
    for (int i = 0; i <= K; ++i) out_tokens[(size_t)b * (K + 1) + i] = h[(size_t)b * (K + 1) + i];
    out_count[b] = cnt;
    if (out_flags) out_flags[b] = (uint32_t)h[(size_t)B * (K + 2) + b];
    c->host_Ls[b] += cnt;
    c->emitted += cnt;
    c->accepted += cnt - 1;
    c->hist[cnt - 1]++;
  }
  c->host_L = c->host_Ls[0];
  c->steps++;
  if (c->opts.flags & SPEC_OPT_TIMING) {
    for (int i = 0; i + 1 < c->ev_used; i += 2) {
      float ms = 0.f;
      CUDA_TRY(c, cudaEventElapsedTime(&ms, c->ev[i], c->ev[i + 1]));
      c->timed_ms += ms;
      c->timed_bytes += c->ev_bytes[i / 2];
      c->timed_launches++;
    }
  }
  return SPEC_OK;
}

int spec_generate(spec_ctx* c, int n_new, int32_t* out, int32_t* out_n) {
  if (!c) return fail(nullptr, SPEC_E_ARG, "null context");
  if (n_new < 0 || (!out && n_new > 0) || !out_n) return fail(c, SPEC_E_ARG, "bad output buffer");
  if (c->B != 1) return fail(c, SPEC_E_ARG, "spec_generate is for batch 1; call spec_step");
  std::vector<int32_t> buf(c->K + 1);
  int got = 0;
  while (got < n_new) {
    int32_t cnt = 0;
    int rc = spec_step(c, buf.data(), &cnt, nullptr);
    if (rc) return rc;
    for (int i = 0; i < cnt && got < n_new; ++i) out[got++] = buf[i];
  }
  *out_n = got;
  return SPEC_OK;
}

int spec_ar_step(spec_ctx* c, int32_t* out_token) {
  if (!c) return fail(nullptr, SPEC_E_ARG, "null context");
  if (!out_token) return fail(c, SPEC_E_ARG, "null output buffer");
  if (!c->prefilled) return fail(c, SPEC_E_STATE, "spec_ar_step before spec_prefill");
  if (max_host_L(c) + 2 > c->cap) return fail(c, SPEC_E_CAPACITY, "context would exceed max_ctx");
  c->grp = false;   // one token: nothing to share
  int rc = run_captured(c, &c->ar_exec, enqueue_ar, &c->kernels_ar);
  if (rc) return rc;
  CUDA_TRY(c, cudaStreamSynchronize(c->stream));
  if (c->h_result[res_words(c) - 1]) return persist_timeout(c);
  for (int b = 0; b < c->B; ++b) {
    out_token[b] = c->h_result[b];
    c->host_Ls[b] += 1;
  }
  c->host_L = c->host_Ls[0];
  c->ar_steps++;
  c->draft_stale = c->draft_model();
  return SPEC_OK;
}

int spec_get_stats(const spec_ctx* c, spec_stats* o) {
  if (!c || !o) return fail(const_cast<spec_ctx*>(c), SPEC_E_ARG, "null argument");
  memset(o, 0, sizeof *o);
  o->steps = c->steps;
  o->ar_steps = c->ar_steps;
  o->tokens_emitted = c->emitted;
  o->drafts_accepted = c->accepted;
  for (int i = 0; i < 17; ++i) o->accept_hist[i] = c->hist[i];
  o->context_len = c->host_L + 1;
  o->kernels_per_step = c->kernels_step;
  o->kernels_per_ar_step = c->kernels_ar;
  o->gemm_launches_per_verify = 4 * c->tgt.d.n_layers + 1;
  o->verify_weight_bytes = c->tgt.weight_bytes();
  // heads: the K heads plus the LM head's second read per step
  o->draft_weight_bytes = c->heads ? (double)c->K * c->tgt.d.d_model * c->tgt.d.d_model * c->tgt.esize +
                                         c->tgt.head_bytes()
                                   : c->drf.weight_bytes();
  o->kv_bytes_per_token_target = c->tgt.kv_bytes_per_token();
  o->kv_bytes_per_token_draft = c->drf.kv_bytes_per_token();
  o->timed_gemm_ms = c->timed_ms;
  o->timed_gemm_bytes = c->timed_bytes;
  o->timed_gemm_launches = c->timed_launches;
  return SPEC_OK;
}

int spec_last_step_debug(spec_ctx* c, float* p_logits, float* q_logits, int32_t* drafts,
                         int32_t* context, int32_t* context_len) {
  if (!c) return fail(nullptr, SPEC_E_ARG, "null context");
  const int K = c->K, V = c->tgt.d.vocab, B = c->B;
  if (p_logits)
    CUDA_TRY(c, cudaMemcpyAsync(p_logits, c->logits_p, sizeof(float) * (size_t)B * (K + 1) * V,
                                cudaMemcpyDeviceToHost, c->stream));
  if (q_logits)
    CUDA_TRY(c, cudaMemcpyAsync(q_logits, c->logits_q, sizeof(float) * (size_t)B * K * V,
                                cudaMemcpyDeviceToHost, c->stream));
  if (drafts)
    CUDA_TRY(c, cudaMemcpyAsync(drafts, c->result + (size_t)B * (K + 3), sizeof(int32_t) * B * K,
                                cudaMemcpyDeviceToHost, c->stream));
  if (context)
    CUDA_TRY(c, cudaMemcpyAsync(context, c->seq, sizeof(int32_t) * (c->host_L + 1),
                                cudaMemcpyDeviceToHost, c->stream));
  if (context_len) *context_len = c->host_L + 1;
  CUDA_TRY(c, cudaStreamSynchronize(c->stream));
  return SPEC_OK;
}

int spec_profile(spec_ctx* c, int iters, spec_profile_t* out) {
  if (!c || !out) return fail(c, SPEC_E_ARG, "null argument");
  if (iters < 1) return fail(c, SPEC_E_ARG, "iters must be >= 1");
  if (!c->prefilled) return fail(c, SPEC_E_STATE, "spec_profile before spec_prefill");
  if (c->draft_stale && c->draft_model())
    return fail(c, SPEC_E_STATE, "draft cache is stale after spec_ar_step; prefill again");
  if (max_host_L(c) + c->K + 2 > c->cap) return fail(c, SPEC_E_CAPACITY, "context would exceed max_ctx");
  void (*enq[4])(Launch&) = {enqueue_draft, enqueue_verify_only, enqueue_ar_only, enqueue_verify_forward};
  double ms[4];
  cudaEvent_t e0, e1;
  CUDA_TRY(c, cudaEventCreate(&e0));
  CUDA_TRY(c, cudaEventCreate(&e1));
  for (int k = 0; k < 4; ++k) {
    c->grp = k != 2 && c->host_L + c->K >= kDGroupMinPos;   // as spec_step / spec_ar_step pick it
    cudaGraphExec_t& ex = c->prof_exec[k][c->grp];
    if (!ex) {
      int rc = capture(c, &ex, enq[k], &c->prof_kernels[k]);
      if (rc) { cudaEventDestroy(e0); cudaEventDestroy(e1); return rc; }
    }
    for (int w = 0; w < 2; ++w) CUDA_TRY(c, cudaGraphLaunch(ex, c->stream));
    CUDA_TRY(c, cudaEventRecord(e0, c->stream));
    for (int i = 0; i < iters; ++i) CUDA_TRY(c, cudaGraphLaunch(ex, c->stream));
    CUDA_TRY(c, cudaEventRecord(e1, c->stream));
    CUDA_TRY(c, cudaEventSynchronize(e1));
    float t = 0.f;
    CUDA_TRY(c, cudaEventElapsedTime(&t, e0, e1));
    ms[k] = (double)t / iters;
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  {
    int32_t flag = 0;
    CUDA_TRY(c, cudaMemcpy(&flag, res_err(c), sizeof flag, cudaMemcpyDeviceToHost));
    if (flag) return persist_timeout(c);
  }
  out->draft_loop_ms = ms[0];
  out->verify_ms = ms[1];
  out->ar_ms = ms[2];
  out->iters = iters;
  out->kernels_draft_loop = c->prof_kernels[0];
  out->kernels_verify = c->prof_kernels[1];
  out->kernels_ar = c->prof_kernels[2];
  out->verify_forward_ms = ms[3];
  out->kernels_verify_forward = c->prof_kernels[3];
  return SPEC_OK;
}

int spec_phase_times(spec_ctx* c, int which, int64_t* out, int max_phases, int* nphases) {
  if (!c || !out || !nphases) return fail(c, SPEC_E_ARG, "null argument");
  if (!c->persist) return fail(c, SPEC_E_STATE, "no persistent forward kernel in this context");
  if (which < 0 || which > c->K + 1) return fail(c, SPEC_E_ARG, "which must be in [0, K+1]");
  const PersistFwd& f = c->pforward[c->heads && which < c->K ? c->heads_pass : which];
  if (!f.desc.times) return fail(c, SPEC_E_STATE, "context created without SPEC_OPT_PHASE_TIMES");
  const int n = f.desc.nphases;
  *nphases = n;
  if (max_phases < n) return fail(c, SPEC_E_ARG, "max_phases below the number of phases");
  std::vector<unsigned long long> t(1 + (size_t)kPhaseStamps * n);
  CUDA_TRY(c, cudaStreamSynchronize(c->stream));
  CUDA_TRY(c, cudaMemcpy(t.data(), f.desc.times, sizeof(unsigned long long) * t.size(),
                         cudaMemcpyDeviceToHost));
  const unsigned long long t0 = t[0];
  auto rel = [&](unsigned long long v) { return v ? (int64_t)(v - t0) : (int64_t)-1; };
  for (int i = 0; i < n; ++i) {
    const PhaseDesc& d = f.host[i];
    const unsigned long long* st = t.data() + 1 + (size_t)kPhaseStamps * i;
    int64_t* o = out + 8 * (size_t)i;
    o[0] = d.kind;
    o[1] = d.kind == kPhaseGemm ? d.g.n : d.kind == kPhaseAttn ? d.a.hq : d.e.ntok;
    o[2] = d.kind == kPhaseGemm ? d.g.k : d.kind == kPhaseAttn ? d.a.ntok : 0;
    o[3] = st[0] ? rel(~st[0]) : -1;
    o[4] = rel(st[1]);
    o[5] = rel(st[2]);
    o[6] = rel(st[3]);
    o[7] = rel(st[4]);
  }
  return SPEC_OK;
}

int spec_phase_list(spec_ctx* c, int which, int64_t* out, int max_phases, int* nphases) {
  if (!c || !out || !nphases) return fail(c, SPEC_E_ARG, "null argument");
  if (!c->persist) return fail(c, SPEC_E_STATE, "no persistent forward kernel in this context");
  if (which < 0 || which > c->K + 1) return fail(c, SPEC_E_ARG, "which must be in [0, K+1]");
  const PersistFwd& f = c->pforward[c->heads && which < c->K ? c->heads_pass : which];
  const int n = (int)f.host.size();
  *nphases = n;
  if (max_phases < n) return fail(c, SPEC_E_ARG, "max_phases below the number of phases");
  for (int i = 0; i < n; ++i) {
    const PhaseDesc& d = f.host[i];
    int64_t* o = out + 8 * (size_t)i;
    o[0] = d.kind;
    if (d.kind == kPhaseGemm) {
      o[1] = d.g.n; o[2] = d.g.k; o[3] = d.g.ntok;
      o[4] = d.tiles;
      o[5] = 0;   // CTAs own whole tiles: no tile's k range is split between CTAs
      o[6] = d.stages;
      o[7] = d.xm == kXSmem ? 1 : 0;
    } else if (d.kind == kPhaseAttn) {
      o[1] = d.a.hq; o[2] = d.a.hkv; o[3] = d.a.ntok; o[4] = d.attn_items;
      o[5] = o[6] = 0; o[7] = d.a.hd;
    } else {
      o[1] = d.e.ntok; o[2] = d.e.d; o[3] = d.e.ntok;
      o[4] = o[5] = o[6] = o[7] = 0;
    }
  }
  return SPEC_OK;
}

int spec_model_forward(spec_ctx* c, int which, const int32_t* tokens, int n, int pos0,
                       float* logits_dev) {
  if (!c) return fail(nullptr, SPEC_E_ARG, "null context");
  if (which != 0 && which != 1) return fail(c, SPEC_E_ARG, "which must be 0 (target) or 1 (draft)");
  if (!tokens || n < 1 || pos0 < 0) return fail(c, SPEC_E_ARG, "bad tokens");
  if (pos0 + n > c->cap) return fail(c, SPEC_E_CAPACITY, "positions exceed max_ctx");
  if (which == 1 && c->heads) return fail(c, SPEC_E_ARG, "a context with self-draft heads has no draft model");
  ModelState& m = which == 0 ? c->tgt : c->drf;
  if (m.q4) return fail(c, SPEC_E_STATE, "spec_model_forward runs one kernel per operation: not for 4-bit models");
  for (int i = 0; i < n; ++i)
    if (tokens[i] < 0 || tokens[i] >= m.d.vocab) return fail(c, SPEC_E_ARG, "token id out of range");
  c->prefilled = false;
  Launch L{c};
  for (int p = 0; p < n; p += kGemmMaxTok) {
    const int nt = std::min(kGemmMaxTok, n - p);
    CUDA_TRY(c, cudaMemcpyAsync(c->fwd_tok, tokens + p, sizeof(int32_t) * nt,
                                cudaMemcpyHostToDevice, c->stream));
    int rc = set_eager_pos(c, pos0 + p);
    if (rc) return rc;
    forward(L, m, nt, c->fwd_tok, nullptr, 0, c->st + 3, 0, 0, logits_dev ? nt : 0,
            logits_dev ? logits_dev + (size_t)p * m.d.vocab : nullptr);
    CUDA_TRY(c, L.e);
    CUDA_TRY(c, cudaStreamSynchronize(c->stream));
  }
  int32_t flag = 0;
  CUDA_TRY(c, cudaMemcpy(&flag, res_err(c), sizeof flag, cudaMemcpyDeviceToHost));
  if (flag) return persist_timeout(c);
  return SPEC_OK;
}

int spec_accept_rows(const float* p_logits, int64_t p_row_stride, const float* q_logits,
                     int64_t q_row_stride, const int32_t* drafts, int rows, int K, int V,
                     float temperature, uint64_t seed, uint64_t step_base, int32_t* tokens,
                     int32_t* counts, uint32_t* flags, void* stream) {
  if (!p_logits || !q_logits || !drafts || !tokens || !counts)
    return fail(nullptr, SPEC_E_ARG, "spec_accept_rows: null pointer");
  if (rows < 1 || K < 1 || K > 16 || V < 2 || !(temperature >= 0.f))
    return fail(nullptr, SPEC_E_ARG, "spec_accept_rows: bad size or temperature");
  if (rows > 65535) return fail(nullptr, SPEC_E_ARG, "spec_accept_rows: at most 65535 rows per call");
  cudaStream_t st = (cudaStream_t)stream;
  const size_t pf = accept_partial_floats(rows, K, V);
  void* scratch = nullptr;
  const size_t bytes = pf * sizeof(float) + (size_t)rows * sizeof(int);
  cudaError_t e = cudaMallocAsync(&scratch, bytes, st);
  if (e != cudaSuccess) return fail(nullptr, SPEC_E_OOM, std::string("spec_accept_rows: ") + cudaGetErrorString(e));
  int* tick = (int*)((float*)scratch + pf);
  e = cudaMemsetAsync(tick, 0, (size_t)rows * sizeof(int), st);
  AcceptDesc a{};
  a.p = p_logits; a.p_ld = p_row_stride; a.q = q_logits; a.q_ld = q_row_stride;
  a.drafts = drafts; a.rows = rows; a.K = K; a.V = V; a.temperature = temperature;
  a.seed = seed; a.step_base = step_base; a.out_tokens = tokens; a.out_count = counts;
  a.out_flags = flags; a.partials = (float*)scratch; a.tickets = tick;
  if (e == cudaSuccess) e = launch_accept(a, st);
  cudaError_t e2 = cudaFreeAsync(scratch, st);
  if (e != cudaSuccess) return fail(nullptr, SPEC_E_CUDA, std::string("spec_accept_rows: ") + cudaGetErrorString(e));
  if (e2 != cudaSuccess) return fail(nullptr, SPEC_E_CUDA, std::string("spec_accept_rows: ") + cudaGetErrorString(e2));
  return SPEC_OK;
}

int spec_sample_rows(const float* logits, int64_t row_stride, int rows, int V, float temperature,
                     uint64_t seed, uint64_t step_base, int position, int32_t* tokens,
                     void* stream) {
  if (!logits || !tokens) return fail(nullptr, SPEC_E_ARG, "spec_sample_rows: null pointer");
  if (rows < 1 || rows > 65535 || V < 2 || !(temperature >= 0.f) || position < 0)
    return fail(nullptr, SPEC_E_ARG, "spec_sample_rows: bad size or temperature");
  cudaStream_t st = (cudaStream_t)stream;
  const size_t pf = sample_partial_floats(rows, V);
  void* scratch = nullptr;
  const size_t bytes = pf * sizeof(float) + (size_t)rows * sizeof(int);
  cudaError_t e = cudaMallocAsync(&scratch, bytes, st);
  if (e != cudaSuccess) return fail(nullptr, SPEC_E_OOM, std::string("spec_sample_rows: ") + cudaGetErrorString(e));
  int* tick = (int*)((float*)scratch + pf);
  e = cudaMemsetAsync(tick, 0, (size_t)rows * sizeof(int), st);
  SampleDesc s{};
  s.logits = logits; s.ld = row_stride; s.rows = rows; s.V = V; s.temperature = temperature;
  s.seed = seed; s.step_base = step_base; s.position = (uint32_t)position;
  s.stream = kStreamDraft; s.out_token = tokens; s.partials = (float*)scratch; s.tickets = tick;
  if (e == cudaSuccess) e = launch_sample(s, st);
  cudaError_t e2 = cudaFreeAsync(scratch, st);
  if (e != cudaSuccess) return fail(nullptr, SPEC_E_CUDA, std::string("spec_sample_rows: ") + cudaGetErrorString(e));
  if (e2 != cudaSuccess) return fail(nullptr, SPEC_E_CUDA, std::string("spec_sample_rows: ") + cudaGetErrorString(e2));
  return SPEC_OK;
}

int spec_inject_fault(spec_ctx* c, int kind, int arg) {
  if (kind == SPEC_FAULT_CLEAR) {
    g_fail_alloc_at = 0;
    if (c && c->fault_ctl) {
      const int z[2] = {0, 0};
      CUDA_TRY(c, cudaMemcpyAsync(c->fault_ctl, z, sizeof z, cudaMemcpyHostToDevice, c->stream));
      CUDA_TRY(c, cudaStreamSynchronize(c->stream));
    }
    return SPEC_OK;
  }
  if (kind == SPEC_FAULT_ALLOC) {
    if (c) return fail(c, SPEC_E_ARG, "SPEC_FAULT_ALLOC applies to the next spec_init: pass a NULL context");
    if (arg < 1) return fail(nullptr, SPEC_E_ARG, "SPEC_FAULT_ALLOC needs arg >= 1");
    g_fail_alloc_at = arg;
    return SPEC_OK;
  }
  if (kind == SPEC_FAULT_WAIT_TIMEOUT) {
    if (!c) return fail(nullptr, SPEC_E_ARG, "SPEC_FAULT_WAIT_TIMEOUT needs a context");
    if (!c->fault_ctl) return fail(c, SPEC_E_STATE, "no persistent forward kernel in this context");
    if (arg < 0) return fail(c, SPEC_E_ARG, "SPEC_FAULT_WAIT_TIMEOUT needs arg >= 0");
    // arg > 0: every grid barrier waits for one arrival more than will come,
    // giving up after arg probes; 0: disarmed
    const int w[2] = {arg > 0 ? 1 : 0, arg};
    CUDA_TRY(c, cudaMemcpyAsync(c->fault_ctl, w, sizeof w, cudaMemcpyHostToDevice, c->stream));
    CUDA_TRY(c, cudaStreamSynchronize(c->stream));
    return SPEC_OK;
  }
  return fail(c, SPEC_E_ARG, "unknown fault kind");
}

int64_t spec_device_bytes_held(void) { return (int64_t)g_device_bytes.load(); }

}  // extern "C"
