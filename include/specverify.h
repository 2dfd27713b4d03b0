/*
 * specverify.h -- C ABI of the GB300 speculative-decoding verification step.
 *
 * One draft model proposes K tokens; one forward of the target model scores
 * the pending token plus the K drafts (K+1 positions, weights read once);
 * a fused kernel applies the acceptance rule and commits the result.
 *
 * Sources for the operations declared here (restated, not copied):
 *  [INT]  "Speculative decoding internals" (tarrragon LLM notes):
 *         section "演算法核心：sampling 階段的接受邏輯", Steps 1-4;
 *         section "為什麼能加速：memory bandwidth bound 的縫隙";
 *         section "怎麼挑 drafter" (draft and target share one vocabulary).
 *  [101]  "Speculative Decoding 101" (gu-log, English): Floor 3 (one pass
 *         scores every position), Floor 4 (greedy rule, 1..K+1 tokens per
 *         round), Floor 5 (acceptance rule, residual draw, bonus token).
 *
 * Conventions shared by every entry point:
 *  - Return value: SPEC_OK (0) or a negative SPEC_E_* code.  After an error
 *    spec_last_error() returns a message; a failed call leaves a context's
 *    committed state unchanged.
 *  - Weights are caller-owned DEVICE memory and must outlive the context.
 *    Matrices are row-major [out_features][in_features] (the nn.Linear
 *    convention), in the model's dtype; RMSNorm gains are fp32.
 *  - KV caches, activations, scratch and RNG state are library-owned device
 *    memory allocated by spec_init and released by spec_free.
 *  - Token buffers of the context API are caller-owned HOST memory; every
 *    context call returns only after its outputs are written.
 *  - A context holds `batch` independent sequences (1..SPEC_MAX_BATCH).
 *    Batch 1 runs each forward as one persistent kernel (bf16 models);
 *    batch > 1 needs bf16 models and runs one kernel per operation, with
 *    the sequences' tokens in one pass (groups of at most 512 tokens, each
 *    group streaming the weights once; passes of more than 16 tokens on the
 *    tensor-memory GEMM).  Sequences advance independently
 *    (ragged acceptance): every sequence has its own committed length, step
 *    counters, KV rows and Philox row word (its index b).
 *  - All work runs on one GPU, on the stream given in spec_opts (or a
 *    stream the library creates).  There is no CPU fallback: without a
 *    usable GPU every call fails with SPEC_E_CUDA.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SPEC_API __attribute__((visibility("default")))
#else
#define SPEC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---- */
#define SPEC_OK             0
#define SPEC_E_ARG         -1   /* bad pointer, size or option */
#define SPEC_E_VOCAB       -2   /* draft and target vocabularies differ [INT 怎麼挑 drafter] */
#define SPEC_E_SHAPE       -3   /* unsupported model shape */
#define SPEC_E_CAPACITY    -4   /* context would exceed max_ctx */
#define SPEC_E_CUDA        -5   /* CUDA runtime error (no GPU, launch failure ...) */
#define SPEC_E_OOM         -6   /* device allocation failed */
#define SPEC_E_TIMEOUT     -7   /* a bounded device-side wait gave up */
#define SPEC_E_STATE       -8   /* call out of order (e.g. step before prefill) */

/* ---- model dtypes ---- */
#define SPEC_MAX_BATCH     64

#define SPEC_DTYPE_F32      0
#define SPEC_DTYPE_BF16     1
/* 4-bit group-quantized weights ("Speculative decoding internals",
 * section "怎麼測自己的加速倍率": the measured models are Q4 files).  Every
 * weight matrix [n][k] (wq, wk, wv, wo, w_gate, w_up, w_down, lm_head) is
 * one buffer: packed signed 4-bit codes [n][k/2] (byte b of a row holds
 * element 2b in its low nibble and 2b+1 in its high nibble, two's
 * complement, codes -8..7), immediately followed by bf16 scales stored
 * group-major [k/64][n] (scale of row r, 64-k group j at index j*n + r);
 * weight = scale x code.  The embedding is bf16, norm gains fp32, and the
 * model computes in bf16 with fp32 accumulation like a bf16 model (KV cache
 * bf16).  4-bit models run only on the persistent kernel: batch 1, K <= 7,
 * d_model, ffn_dim and n_heads*head_dim multiples of 256, vocab and
 * n_kv_heads*head_dim multiples of 8, prompts of at least 10 tokens. */
#define SPEC_DTYPE_Q4       2

/* ---- per-step flags (spec_step out_flags) ---- */
#define SPEC_FLAG_RESID_ZERO   0x1u  /* rejection with zero residual mass; drew from p */
#define SPEC_FLAG_ALL_ACCEPTED 0x2u  /* all K drafts accepted; last token is the bonus */

/* ---- option flags (spec_opts.flags) ---- */
#define SPEC_OPT_NO_GRAPH      0x1   /* launch the step kernel by kernel (no CUDA graph) */
#define SPEC_OPT_TIMING        0x2   /* record CUDA events around every weight-streaming
                                        GEMM of the verify pass (implies NO_GRAPH) */
#define SPEC_OPT_PDL           0x4   /* launch kernels with programmatic dependent launch
                                        (process-wide; off by default: measured slower on
                                        the verify pass) */
#define SPEC_OPT_NO_PERSIST    0x8   /* run each forward as one kernel per operation
                                        instead of one persistent kernel (bf16 models).
                                        The two paths sum in different orders: their
                                        logits agree to rounding, not bit for bit; each
                                        is batch-invariant on its own */
#define SPEC_OPT_PHASE_TIMES   0x10  /* persistent kernel records per-phase timestamps
                                        (read with spec_phase_times) */

typedef struct spec_ctx spec_ctx;

/* Weights of one decoder layer (device pointers). */
typedef struct spec_layer_weights {
    const void* attn_norm;   /* [d_model] fp32 */
    const void* wq;          /* [n_heads*head_dim][d_model] */
    const void* wk;          /* [n_kv_heads*head_dim][d_model] */
    const void* wv;          /* [n_kv_heads*head_dim][d_model] */
    const void* wo;          /* [d_model][n_heads*head_dim] */
    const void* ffn_norm;    /* [d_model] fp32 */
    const void* w_gate;      /* [ffn_dim][d_model] */
    const void* w_up;        /* [ffn_dim][d_model] */
    const void* w_down;      /* [d_model][ffn_dim] */
} spec_layer_weights;

/* A Llama-style decoder: pre-norm RMSNorm blocks, rotate-half RoPE,
 * grouped-query causal attention (query head h reads KV head
 * h*n_kv_heads/n_heads), SwiGLU MLP, untied LM head. */
typedef struct spec_model_desc {
    int   n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn_dim, vocab;
    float rope_theta, rms_eps;
    int   dtype;                        /* SPEC_DTYPE_F32, SPEC_DTYPE_BF16 or SPEC_DTYPE_Q4 */
    const void* embed;                  /* [vocab][d_model] */
    const void* final_norm;             /* [d_model] fp32 */
    const void* lm_head;                /* [vocab][d_model] */
    const spec_layer_weights* layers;   /* host array [n_layers]; copied by spec_init */
} spec_model_desc;

typedef struct spec_opts {
    int      batch;             /* sequences, 1..SPEC_MAX_BATCH (> 1: bf16 models,
                                   draft_mix_lambda 0) */
    int      max_ctx;           /* KV capacity in positions (prompt + generated + K + 1) */
    float    temperature;       /* 0 = greedy; >0 scales target and draft logits */
    uint64_t seed;              /* Philox key of every random draw */
    float    draft_mix_lambda;  /* 0 = off; else q-logits = (1-l)*draft + l*target's
                                   previous-step logits (same row index) */
    void*    cuda_stream;       /* cudaStream_t to run on; NULL = library-created stream */
    int      flags;             /* SPEC_OPT_* */
    int      draft_lookup;      /* 0 = the draft model drafts; n in 1..8 = prompt lookup
                                   ([101 Floor 6] n-gram drafting): the drafts continue the
                                   most recent longest (up to n tokens) earlier match of the
                                   context's end, q is one-hot at each draft, and the draft
                                   model is not run (draft_mix_lambda must be 0) */
    const void* draft_heads;    /* NULL = off; else self-draft heads ([101 Floor 6], [INT
                                   三條主流變體] MTP: extra prediction heads on the target):
                                   device pointer to K stacked row-major d_model x d_model
                                   matrices W_1..W_K in the target's arithmetic dtype (bf16
                                   for bf16 and 4-bit targets, fp32 for fp32 targets),
                                   16-byte aligned, caller-owned.  Head i drafts position
                                   L + i from the target's LM-head input u at the last
                                   scored position: q_i logits = W_head (u + silu(W_i u)).
                                   The draft model is not used (pass draft = NULL); needs
                                   batch 1, K <= 8, draft_lookup 0, draft_mix_lambda 0 */
} spec_opts;

typedef struct spec_stats {
    int64_t steps;              /* speculative steps run since prefill */
    int64_t ar_steps;           /* plain autoregressive steps run since prefill */
    int64_t tokens_emitted;     /* by speculative steps */
    int64_t drafts_accepted;    /* sum of n (accepted drafts) over steps */
    int64_t accept_hist[17];    /* steps with n = 0..K accepted drafts (K <= 16) */
    int32_t context_len;        /* committed tokens including the pending one */
    int32_t kernels_per_step;   /* kernel launches of one spec_step */
    int32_t kernels_per_ar_step;
    int32_t gemm_launches_per_verify;
    double  verify_weight_bytes;  /* matrix bytes one target pass streams */
    double  draft_weight_bytes;   /* matrix bytes one draft pass streams */
    double  kv_bytes_per_token_target;
    double  kv_bytes_per_token_draft;
    double  timed_gemm_ms;      /* SPEC_OPT_TIMING: summed event time of verify GEMMs */
    double  timed_gemm_bytes;   /* SPEC_OPT_TIMING: weight bytes of those GEMMs */
    int64_t timed_gemm_launches;
} spec_stats;

/* Create a context for one target/draft pair and K drafts per step (with
 * opts->draft_heads the target drafts for itself and draft may be NULL).
 * Checks shapes (head_dim in {32, 64, 128}; n_heads a multiple of
 * n_kv_heads; d_model, ffn_dim and n_heads*head_dim multiples of 64 for
 * bf16 models, of 4 for fp32 models), equal vocabularies
 * (SPEC_E_VOCAB, [INT 怎麼挑 drafter]) and 1 <= K <= 16; allocates the KV
 * caches for max_ctx positions, activations and scratch.  *out receives the
 * context (NULL on error; spec_last_error(NULL) then has the message). */
SPEC_API int spec_init(const spec_model_desc* target, const spec_model_desc* draft, int K,
              const spec_opts* opts, spec_ctx** out);

/* Release everything spec_init allocated.  NULL is a no-op. */
SPEC_API void spec_free(spec_ctx* ctx);

/* Message of the last error on ctx (or of the last failed spec_init /
 * stateless call on this thread when ctx is NULL).  Never NULL. */
SPEC_API const char* spec_last_error(const spec_ctx* ctx);

/* Prefill: tokens[b][0..L-1] (host, int32 [batch][L], 0 <= id < vocab),
 * the same length L for every sequence.  Both models score positions
 * 0..L-2 into their KV caches; tokens[b][L-1] becomes the pending token of
 * sequence b's first step (it is the x of [INT 演算法核心] Step 2's
 * T(.|x)).  Resets the step counters.  Requires 2 <= L and
 * L + K + 1 <= max_ctx; with draft_mix_lambda != 0 also L >= K + 2. */
SPEC_API int spec_prefill(spec_ctx* ctx, const int32_t* tokens, int L);

/* Benchmark state without a prefill: every sequence gets L committed
 * positions (L - 1 cached, token L-1 pending) with token ids drawn uniformly
 * from [0, vocab) and both models' KV caches filled with synthetic
 * normally distributed bf16 / fp32 values (a counter-based generator keyed
 * by seed), not with the models' own keys and values.  Steps then run the
 * same kernels and read the same bytes as after a real prefill of L tokens;
 * their tokens carry no meaning.  Resets the step counters.  Requires
 * 2 <= L and L + K + 1 <= max_ctx. */
SPEC_API int spec_prefill_synthetic(spec_ctx* ctx, int L, uint64_t seed);

/* Committed tokens of sequence b (host, capacity max_ctx): context[0 ..
 * *len - 1], the last one being the pending token. */
SPEC_API int spec_seq_context(spec_ctx* ctx, int b, int32_t* context, int32_t* len);

/* One speculative step [INT 演算法核心 Steps 1-4; 101 Floors 4-5]:
 *  1. draft loop: K draft forwards, d_i ~ softmax(q_i / T) (argmax at T=0);
 *  2. one target forward over [pending, d_1..d_K] -> K+1 distributions;
 *  3. left to right, accept d_i iff r_i < min(1, p_i(d_i)/q_i(d_i)); on the
 *     first reject draw from normalize((p_i - q_i)+) and stop; if all K are
 *     accepted draw the bonus from p_{K+1} (greedy: match / first mismatch
 *     emits the target's argmax / bonus argmax);
 *  4. commit: the emitted tokens extend the context, the last one becomes
 *     the pending token; KV entries past the accepted prefix are dropped by
 *     length truncation (no copies).
 * For every sequence b: out_tokens (host, [batch][K+1]) row b receives its
 * n_b+1 emitted tokens (the rest of the row is -1), out_count[b] = n_b+1
 * (1 <= n_b+1 <= K+1, [101 Floor 4]); out_flags ([batch]) may be NULL.
 * Fails with SPEC_E_STATE before prefill, SPEC_E_CAPACITY when a sequence's
 * context plus K+1 would exceed max_ctx. */
SPEC_API int spec_step(spec_ctx* ctx, int32_t* out_tokens, int32_t* out_count, uint32_t* out_flags);

/* Speculative generation of n_new tokens (batch 1): spec_step until at
 * least n_new tokens are emitted; out (host, capacity n_new) receives the
 * first n_new, *out_n = n_new.  Extra emitted tokens of the last step stay
 * committed.  Batched contexts call spec_step directly. */
SPEC_API int spec_generate(spec_ctx* ctx, int n_new, int32_t* out, int32_t* out_n);

/* Plain autoregressive decoding on the same kernels [101 Floor 1]: one
 * target forward over the pending token of every sequence, one draw per
 * sequence from softmax(p / T) (argmax at T=0), committed like a step.
 * out_token[b] (host, [batch]) receives sequence b's token. */
SPEC_API int spec_ar_step(spec_ctx* ctx, int32_t* out_token);

/* Counters and byte accounting of the context. */
SPEC_API int spec_get_stats(const spec_ctx* ctx, spec_stats* out);

/* Copy the internals of the last spec_step to host buffers (any may be
 * NULL): target logits [batch][K+1][vocab] fp32, draft q logits after
 * mixing [batch][K][vocab] fp32, draft tokens [batch][K], and sequence 0's
 * committed context tokens [context_len] (capacity max_ctx; other
 * sequences: spec_seq_context).  For verification against a reference. */
SPEC_API int spec_last_step_debug(spec_ctx* ctx, float* p_logits, float* q_logits,
                         int32_t* drafts, int32_t* context, int32_t* context_len);

/* Run one model's forward over n tokens (host ids) at positions pos0 ..
 * pos0+n-1 of its own KV cache (sequence 0; pos0 <= its current valid length; the valid
 * length becomes pos0+n) and write fp32 logits of all n positions to
 * logits_dev ([n][vocab], device).  which: 0 = target, 1 = draft.  This is
 * the forward the step uses [101 Floor 3]; it does not touch the step state
 * (call spec_prefill again before stepping). */
SPEC_API int spec_model_forward(spec_ctx* ctx, int which, const int32_t* tokens, int n, int pos0,
                       float* logits_dev);

/* Stateless fused acceptance over `rows` independent verify rows
 * [INT 演算法核心 Step 3-4]: row r has target logits p[r] ([K+1][V] fp32,
 * device, row stride p_row_stride floats between verify rows), draft logits
 * q[r] ([K][V], stride q_row_stride) and drafts d[r] ([K] int32, device).
 * Random draws use Philox key `seed` and step counter step_base + r.
 * Writes tokens[r][0..K] (int32, device, K+1 per row), counts[r] and
 * flags[r] (may be NULL).  temperature 0 = greedy rule.  Scratch comes from
 * the stream-ordered allocator of the current device.  Asynchronous on
 * `stream` (cudaStream_t; NULL = default stream). */
SPEC_API int spec_accept_rows(const float* p_logits, int64_t p_row_stride,
                     const float* q_logits, int64_t q_row_stride,
                     const int32_t* drafts, int rows, int K, int V, float temperature,
                     uint64_t seed, uint64_t step_base, int32_t* tokens, int32_t* counts,
                     uint32_t* flags, void* stream);

/* Same as spec_accept_rows, but allocates nothing.  The pages have no
 * counterpart: this exists for callers that cannot allocate device memory
 * when they verify drafts -- e.g. a serving process whose memory pool has
 * already reserved (nearly) all of HBM, or a latency-critical loop that must
 * not trigger the device synchronisation an allocation can cause.  Scratch
 * comes from one fixed 4 MiB array compiled into the library (present on
 * every GPU that loads it, until the process exits); calls needing more
 * (about 750 rows at K=5, V=128256) fail with SPEC_E_ARG and a message.
 * Every call looks up the array's device address on the current device
 * (nothing is cached, so a device reset that reloads the module is
 * harmless); the first call on a device may load the module, so make it
 * before any stream capture.  All calls share the array: calls that overlap on the GPU race, so order
 * them (one stream, or events).  Asynchronous on `stream`. */
SPEC_API int spec_accept_rows_noalloc(const float* p_logits, int64_t p_row_stride,
                     const float* q_logits, int64_t q_row_stride,
                     const int32_t* drafts, int rows, int K, int V, float temperature,
                     uint64_t seed, uint64_t step_base, int32_t* tokens, int32_t* counts,
                     uint32_t* flags, void* stream);

/* Stateless draft sampler: one token per row from softmax(logits[r] / T)
 * by inverse CDF (argmax at T=0), with the Philox draw (seed; step_base+r,
 * position, stream 0, row 0).  logits: [rows] rows of V fp32 (device,
 * stride row_stride floats).  tokens: [rows] int32 device.  Asynchronous. */
SPEC_API int spec_sample_rows(const float* logits, int64_t row_stride, int rows, int V,
                     float temperature, uint64_t seed, uint64_t step_base, int position,
                     int32_t* tokens, void* stream);

/* Phase timing of the step as run in production (CUDA graphs, CUDA events
 * on the context's stream), averaged over `iters` replays after two
 * warm-up replays: the draft loop (K draft passes + samplers), the verify
 * pass (target over the K+1 positions + fused acceptance, not committed)
 * and one plain-decoding pass (target over 1 position + sampler, not
 * committed), and the verify pass's target forward alone (the one
 * persistent kernel launch, or its per-operation kernels).  Requires a
 * prefilled context; the committed state is left
 * unchanged (only uncommitted KV rows and draft slots are rewritten, with
 * the values the next step computes anyway).  Measures the quantities of
 * [INT 加速倍率 = K × acceptance rate 的限制]: T_draft, T_target and C. */
typedef struct spec_profile_t {
    double draft_loop_ms;
    double verify_ms;
    double ar_ms;
    int32_t iters;
    int32_t kernels_draft_loop;
    int32_t kernels_verify;
    int32_t kernels_ar;
    double verify_forward_ms;     /* the verify pass's target forward alone */
    int32_t kernels_verify_forward;
} spec_profile_t;
SPEC_API int spec_profile(spec_ctx* ctx, int iters, spec_profile_t* out);

/* Per-phase timing of the last run of one persistent forward pass
 * (context created with SPEC_OPT_PHASE_TIMES on the persistent path).
 * which: 0..K-1 the K draft passes of a step, K the verify pass, K+1 the
 * plain-decoding pass.  Writes *nphases and, per phase i, eight int64 at
 * out[8 i ..]: kind (0 embedding, 1 GEMM, 2 attention), rows n (GEMM) or
 * query heads (attention) or tokens (embedding), k (GEMM) or tokens
 * (attention), then %globaltimer offsets in ns from CTA 0's start: the
 * earliest and the latest CTA's arrival at the end of the phase, CTA 0's
 * release from the grid barrier after it (-1 for the last phase), the latest
 * CTA's end of X preparation (GEMM) or end of its key walk (attention),
 * and the latest CTA's delivery of its last weight unit (GEMM) or end of
 * its items (attention); -1 where a stamp was not taken.  out holds max_phases * 8
 * int64 (host).  Synchronises the context's stream.  Errors: SPEC_E_STATE
 * without the option or the persistent path, SPEC_E_ARG when max_phases is
 * too small (after setting *nphases). */
SPEC_API int spec_phase_times(spec_ctx* ctx, int which, int64_t* out, int max_phases, int* nphases);

/* ---- failure injection (test hooks) ----
 * The pages describe no failure handling; these hooks let tests drive the
 * library's own error paths without faulting or hanging a GPU.
 *
 * SPEC_FAULT_ALLOC (ctx must be NULL, arg = n >= 1): the n-th device
 *   allocation of the next spec_init call fails as if the device were out
 *   of memory; that spec_init returns SPEC_E_OOM after releasing everything
 *   it had allocated.  The injection applies to that one call (it is
 *   cleared when the call returns, whether or not it fired).
 * SPEC_FAULT_WAIT_TIMEOUT (persistent-path context, arg >= 0): with
 *   arg > 0 every grid barrier of the context's forward kernels waits for
 *   one arrival more than will ever come and gives up after arg probes,
 *   raising the context's error flag; the kernels then leave at their first
 *   barrier, nothing is committed, and the step returns SPEC_E_TIMEOUT with
 *   the committed state unchanged.  arg = 0 disarms it.  The bound keeps
 *   every wait finite: no kernel hangs and the context stays usable.
 * SPEC_FAULT_CLEAR: disarm both (ctx may be NULL).
 * Errors: SPEC_E_ARG for an unknown kind or a bad argument, SPEC_E_STATE for
 * SPEC_FAULT_WAIT_TIMEOUT on a context without persistent kernels. */
#define SPEC_FAULT_CLEAR         0
#define SPEC_FAULT_ALLOC         1
#define SPEC_FAULT_WAIT_TIMEOUT  2
SPEC_API int spec_inject_fault(spec_ctx* ctx, int kind, int arg);

/* Bytes of device memory held by every live context of the process (the
 * allocations spec_init made and spec_free releases). */
SPEC_API int64_t spec_device_bytes_held(void);

/* Phase list of one persistent forward pass, for inspection (no device
 * work): which = 0..K-1 the draft passes of a step, K the verify pass, K+1
 * the plain-decoding pass.  Writes *nphases and, per phase i, eight int64 at
 * out[8 i ..]: kind (0 embedding, 1 GEMM, 2 attention), then
 *   GEMM:      rows n, k, tokens, 16-row output tiles, 1 if a tile's k range
 *              is split between CTAs (else 0), ring stages, 1 if the input
 *              rows are resident in shared memory (else streamed);
 *   attention: query heads, KV heads, tokens, work items, 0, 0, head dim;
 *   embedding: tokens, d_model, tokens, 0, 0, 0, 0.
 * The geometry depends only on the shapes and the SM count, so a model cut
 * to fewer layers runs the same per-layer phases as the full-depth model.
 * out holds max_phases * 8 int64 (host).  Errors: SPEC_E_STATE without the
 * persistent path, SPEC_E_ARG when max_phases is too small (after setting
 * *nphases). */
SPEC_API int spec_phase_list(spec_ctx* ctx, int which, int64_t* out, int max_phases, int* nphases);

/* Library version string. */
SPEC_API const char* spec_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SPECVERIFY_H */
