"""Batched contexts (several sequences per step) through the C ABI.

A batched context runs every forward once over all sequences' tokens (the
per-operation path, groups of at most 512 tokens), samples and accepts one row
per sequence, and commits each sequence by its own count (ragged
acceptance).  The pages describe one sequence; a batch is that algorithm per
sequence, with sequence b's Philox draws at row word b.

* Each sequence advances exactly as it would alone: greedy steps of a
  3-sequence batch (passes of at most 16 tokens, the skinny GEMM) give
  bit-identical tokens and counts to three batch-1 contexts on the
  per-operation path (every split point is independent of the number of
  tokens in a pass), and so does sequence 0 at T = 1 (row word 0 in both).
* Teacher-forced parity per sequence against the fp64 oracle: stage (i)
  logits within the bf16 tolerance, stage (ii) the oracle's acceptance with
  row word b on the GPU's logits reproduces sequence b's emitted tokens.
* Passes of more than 16 tokens (6 or 16 sequences x 5 positions; 64 x 5 in
  one pass whose MMAs take the tokens in two halves of 160; 64 x 9 in two
  passes of 32 sequences, halves of 144) run their GEMMs on the tensor-memory
  (tcgen05) GEMM; the teacher-forced parity above
  covers every GEMM kind on that path (q/k/v + RoPE + KV append, residual
  adds, gate/up + SwiGLU, LM head).  With enough sequences for a wave of
  (sequence, KV head) items, attention items carry 2 or 3 eight-row tiles
  (all heads of several tokens per K/V walk): 48 x 3 and 40 x 5 tokens.
* Sequences whose contexts cross the first 1024-key split (token-group
  attention items, split merges), after a synthetic prefill, step with valid
  counts and ragged lengths; spec_ar_step and spec_profile run on batches.
"""
import numpy as np
import pytest
import torch

import helpers
import speculative_decoding_verification_step_gb300 as sv
import workloads
from oracle import generate as gen

pytestmark = pytest.mark.gpu

SHAPE = workloads.small_shape(name="hd64", dtype="bf16", n_heads=4, n_kv_heads=2, head_dim=64)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sv.build()
    sv.lib()


def _pair(seed=1):
    w = workloads.make_weights(SHAPE, seed=seed)
    dshape, dw = workloads.noisy_layer0_draft(SHAPE, w, seed=seed + 1)
    return w, dshape, dw


def _dec(w, dshape, dw, k, max_ctx, temp, batch, flags=0, seed=0):
    return sv.SpecDecoder(SHAPE, helpers.to_device(w), dshape, helpers.to_device(dw), k, max_ctx,
                          temperature=temp, seed=seed, flags=flags, batch=batch)


@pytest.mark.parametrize("temp", [0.0, 1.0])
def test_batch_sequences_match_single(temp):
    k, max_ctx, nseq, steps = 4, 128, 3, 6
    w, dshape, dw = _pair()
    prompts = workloads.make_prompt(SHAPE.vocab, 20, seed=5, batch=nseq).tolist()
    dec = _dec(w, dshape, dw, k, max_ctx, temp, nseq)
    dec.prefill(prompts)
    got = [dec.step() for _ in range(steps)]
    ctxs = [dec.seq_context(b).tolist() for b in range(nseq)]
    dec.close()
    # at T = 1 only sequence 0 shares its Philox row word with a batch-1 context
    check = range(nseq) if temp == 0.0 else range(1)
    for b in check:
        one = _dec(w, dshape, dw, k, max_ctx, temp, 1, flags=sv.SPEC_OPT_NO_PERSIST)
        one.prefill(prompts[b])
        for s in range(steps):
            toks, _ = one.step()
            assert toks == got[s][0][b], (b, s, toks, got[s][0][b])
        assert one.seq_context(0).tolist() == ctxs[b]
        one.close()
    # ragged: the sequences' lengths are their own
    for b in range(nseq):
        assert len(ctxs[b]) == 20 + sum(len(got[s][0][b]) for s in range(steps))


@pytest.mark.parametrize("nseq,k", [(3, 3), (6, 4), (16, 4), (48, 2), (40, 4), (64, 4), (64, 8)],
                         ids=["3x4tok", "6x5tok-tensor-memory-gemm", "16x5tok-tensor-memory-gemm",
                              "48x3tok-wide2-attention", "40x5tok-wide3-attention", "64x5tok-token-halves",
                              "64x9tok-two-passes"])
@pytest.mark.parametrize("temp", [0.0, 1.0])
def test_batch_teacher_forced(temp, nseq, k):
    # 6 x 5 and 16 x 5 tokens per verify pass: the GEMMs run on the
    # tensor-memory (tcgen05) GEMM; 48 x 3 and 40 x 5 tokens (with 152 SMs):
    # attention items of 2 and 3 eight-row tiles; 64 x 5 = 320 tokens: one
    # pass, two MMAs (token halves) per weight tile; 64 x 9 = 576 tokens: two
    # passes of 288 (sequence groups of at most 512 tokens)
    max_ctx, steps, seed = 128, 5, 7
    w, dshape, dw = _pair(seed=3)
    prompts = workloads.make_prompt(SHAPE.vocab, 12, seed=9, batch=nseq).tolist()
    dec = _dec(w, dshape, dw, k, max_ctx, temp, nseq, seed=seed)
    dec.prefill(prompts)
    T, D = gen.Model(SHAPE, w), gen.Model(dshape, dw)
    tol = helpers.logit_tol(SHAPE)
    ctxs = [list(p) for p in prompts]
    skipped = 0
    for step in range(steps):
        rows, _ = dec.step()
        p, q, d, _ = dec.last_step_debug(max_ctx)
        for b in range(nseq):
            toks = rows[b]
            assert 1 <= len(toks) <= k + 1
            ref = gen.spec_step(T, D, ctxs[b], k, temp, seed, step, row=b, tie_eps=helpers.tie_eps(SHAPE))
            same = 0
            while same < k and ref.drafts[same] == int(d[b, same]):
                same += 1
            upto = min(k, same + 1)
            assert np.abs(q[b, :upto] - ref.q_logits[:upto]).max() < tol
            if same == k:
                assert np.abs(p[b] - ref.p_logits).max() < tol
            for i in range(k):
                dg, fl = gen.draft_token(q[b, i], temp, seed, step, i + 1, row=b, tie_eps=0.0)
                if not fl & helpers.SKIP_FLAGS:
                    assert dg == int(d[b, i]), (step, b, i, dg, int(d[b, i]))
            em, _, fl = gen.verify(p[b], q[b], list(d[b]), temp, seed, step, row=b, tie_eps=0.0)
            if fl & helpers.SKIP_FLAGS:
                skipped += 1
            else:
                assert em == toks, (step, b, em, toks)
            ctx = dec.seq_context(b).tolist()
            assert ctx[len(ctxs[b]):] == toks
            ctxs[b] = ctx
    assert skipped <= steps * nseq // 4
    dec.close()


@pytest.mark.parametrize("nseq", [4, 16, 40])
def test_batch_long_context_synthetic(nseq):
    # last verify position past 1024: token-group items, split merges; 16
    # sequences: 96-token verify passes on the tensor-memory GEMM; 40: wide
    # attention items across key splits
    k, L = 5, 1100
    w, dshape, dw = _pair(seed=4)
    dec = _dec(w, dshape, dw, k, 1200, 1.0, nseq)
    dec.prefill_synthetic(L, seed=11)
    lens = [L] * nseq
    for _ in range(3):
        rows, _ = dec.step()
        for b in range(nseq):
            assert 1 <= len(rows[b]) <= k + 1
            assert all(0 <= t < SHAPE.vocab for t in rows[b])
            lens[b] += len(rows[b])
            ctx = dec.seq_context(b)
            assert len(ctx) == lens[b]
            assert ctx[-len(rows[b]):].tolist() == rows[b]
    prof = dec.profile(iters=2)
    assert prof["verify_ms"] > 0 and prof["draft_loop_ms"] > 0
    toks = dec.ar_step()
    assert len(toks) == nseq and all(0 <= t < SHAPE.vocab for t in toks)
    for b in range(nseq):
        assert dec.seq_context(b)[-1] == toks[b]
    dec.close()


def test_batch_greedy_long_context_matches_single():
    # contexts across the 1024-key split: the batch and the batch-1 contexts
    # take the same attention mode per sequence, so tokens stay bit-identical
    k, nseq, L = 3, 2, 1030
    w, dshape, dw = _pair(seed=6)
    prompts = workloads.make_prompt(SHAPE.vocab, L, seed=13, batch=nseq).tolist()
    dec = _dec(w, dshape, dw, k, 1100, 0.0, nseq)
    dec.prefill(prompts)
    got = [dec.step()[0] for _ in range(3)]
    dec.close()
    for b in range(nseq):
        one = _dec(w, dshape, dw, k, 1100, 0.0, 1, flags=sv.SPEC_OPT_NO_PERSIST)
        one.prefill(prompts[b])
        for s in range(3):
            assert one.step()[0] == got[s][b], (b, s)
        one.close()
